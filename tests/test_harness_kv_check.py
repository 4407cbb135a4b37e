"""The K/V check of the GPU parity tests, exercised on the CPU.

The check compares the GPU's K/V appends with the fp32 C oracle's and, where an element
misses the bar and both sides started the step from the same pool, lets the float64
twin decide. These tests run the check on a stand-in for the GPU side: a pool holding
the twin's own appends. A mistake planted in the ORACLE's pool must be forgiven by the
twin; the same mistake in the stand-in's pool must fail, and so must the oracle-side
mistake when the step did not start from a common pool (the twin then has no history).
"""
import numpy as np
import pytest

import oracle
import synth

harness = pytest.importorskip("harness")

B = 2
NPAGES = 16


class _HostPair(harness.Pair):
    """Pair without the GPU: its "GPU pool" is whatever the test writes into ``gpu_pool``."""

    def __init__(self, cfg, seed):
        self.cfg = cfg
        self.W = synth.make_weights(cfg, seed, device="cpu", gain_noise=0.02)
        pool = torch_empty_pool(cfg)
        synth.fill_normal_bf16_(pool, seed + 1)
        self.orc = oracle.OracleModel(cfg, self.W)
        self.kv_host = synth.bf16_bits(pool).copy()
        self.kv_start = self.kv_host.copy()
        self.num_pages = NPAGES
        self.start_is_common = True
        self.last_inputs = None
        self._twin = None
        self.gpu_pool = self.kv_start.copy()

    def oracle_step(self, tokens, positions, page_table):
        self.last_inputs = (tokens, positions, page_table, self.start_is_common)
        self.start_is_common = False
        self.orc.decode_step(self.kv_host, tokens, positions, page_table, positions + 1)

    def gpu_kv_bits(self):
        return self.gpu_pool


def torch_empty_pool(cfg):
    import torch
    return torch.empty(synth.kv_pool_shape(cfg, NPAGES), dtype=torch.bfloat16)


def _bits(v):
    return (np.asarray(v, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _setup(start_common=True):
    cfg = synth.TINY
    pair = _HostPair(cfg, seed=3)
    rng = np.random.default_rng(3)
    positions = np.array([21, 37], np.int32)
    pages = [int(p) // 16 + 1 for p in positions]
    page_table = synth.random_page_tables(rng, NPAGES, pages, max(pages))
    tokens = synth.random_tokens(rng, cfg.vocab, B)
    pair.start_is_common = start_common
    pair.oracle_step(tokens, positions, page_table)
    # the stand-in GPU pool: the twin's appends at the oracle's slots, run from its own
    # appends (layer l's rows depend only on the appends of the layers before it, so
    # n_layers passes make them consistent)
    for b in range(B):
        page, slot = page_table[b][positions[b] // 16], positions[b] % 16
        for _ in range(cfg.n_layers):
            t = pair.twin_appends(b, pair.gpu_pool)
            for l in range(cfg.n_layers):
                for kv in (0, 1):
                    pair.gpu_pool[l, page, kv, :, slot, :] = _bits(t[l, kv])
    return pair, (int(page_table[1][positions[1] // 16]), int(positions[1] % 16))


def _largest(pool, page, slot):
    """Index (layer 1, V, head 0, slot, dim) of the largest-magnitude element of that row."""
    row = pool[1, page, 1, 0, slot].astype(np.int32) & 0x7FFF
    return (1, page, 1, 0, slot, int(np.argmax(row)))


def test_twin_stand_in_passes_as_is():
    pair, _ = _setup()
    twin_before = harness.KV_STATS["twin"]
    assert harness.check_kv(pair) == B * 2 * 2 * 2
    assert harness.KV_STATS["twin"] == twin_before


def test_oracle_side_mistake_is_forgiven_by_the_twin():
    pair, (page, slot) = _setup()
    i = _largest(pair.kv_host, page, slot)
    pair.kv_host[i] += 5  # five BF16 ulps away from the fp32 oracle's own value
    twin_before = harness.KV_STATS["twin"]
    harness.check_kv(pair)
    assert harness.KV_STATS["twin"] == twin_before + 1


def test_gpu_side_mistake_fails():
    pair, (page, slot) = _setup()
    i = _largest(pair.gpu_pool, page, slot)
    pair.gpu_pool[i] += 5
    with pytest.raises(AssertionError, match="differ by more than 1 BF16 ulp"):
        harness.check_kv(pair)


def test_no_twin_without_a_common_start():
    pair, (page, slot) = _setup(start_common=False)
    i = _largest(pair.kv_host, page, slot)
    pair.kv_host[i] += 5
    with pytest.raises(AssertionError, match="differ by more than 1 BF16 ulp"):
        harness.check_kv(pair)

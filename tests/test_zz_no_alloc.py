"""mk_decode_step_noalloc: the decode step for callers that cannot allocate device
memory (a memory plan that owns all of HBM, allocator-free or sandboxed runtimes,
paths where cudaMalloc would synchronise the device). Its scratch lives in the
library's static device array; the caller passes every input and output, including
the KV pool.

Checked here, on two consecutive calls each (the second one finds the array holding the
first call's contents): the result matches the CPU oracle at the parity bar (logits,
tokens where the oracle's margin is clear, K/V appends at the oracle's addresses and
within 1 BF16 ulp), at batch 1 and 2 (tagged-word hand-off, which relies on the
per-call clearing of the array) and batch 3 and 8 (counters), for a small dense model, a
small MoE and the 2B shapes cut to two layers; and it matches the handle-based
mk_decode_step on the same inputs.

This file is collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
import synth
import persistent_megakernel_05_b300 as mk
from harness import check_logits, check_kv

pytestmark = pytest.mark.gpu


def _addr(t):
    return t.data_ptr()


class _NoAllocPair:
    """The no-allocation entry point on a caller-owned pool, beside the oracle with its
    own copy of the same seeded pool (the attributes check_kv reads)."""

    def __init__(self, cfg, seed, num_pages, kv_seed):
        self.cfg = cfg
        self.W = synth.make_weights(cfg, seed, device="cuda", gain_noise=0.02)
        # a handle only to build the descriptor and weight structs the call takes (the
        # entry point itself allocates nothing)
        self.model = mk.DecodeModel(cfg, self.W, 8)
        self.pool = torch.empty(synth.kv_pool_shape(cfg, num_pages), dtype=torch.bfloat16, device="cuda")
        synth.fill_normal_bf16_(self.pool, kv_seed)
        torch.cuda.synchronize()
        self.num_pages = num_pages
        self.orc = oracle.OracleModel(cfg, self.W)
        self.kv_host = synth.bf16_bits(self.pool).copy()
        self.kv_start = self.kv_host.copy()
        self.status = torch.full((2,), -1, dtype=torch.int32, device="cuda")

    def call(self, toks, pos, pt):
        B = len(toks)
        t = torch.tensor(np.asarray(toks, np.int32), device="cuda")
        p = torch.tensor(np.asarray(pos, np.int32), device="cuda")
        ptd = torch.tensor(np.asarray(pt, np.int32), device="cuda")
        sl = p + 1
        nx = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        lg = torch.full((B, self.cfg.vocab), float("nan"), device="cuda")
        stream = torch.cuda.current_stream().cuda_stream
        rc = mk.mk_decode_step_noalloc(self.model.desc, self.model.w, _addr(self.pool), self.num_pages,
                                       _addr(t), _addr(p), _addr(ptd), ptd.shape[1], _addr(sl), B,
                                       _addr(nx), _addr(lg), _addr(self.status), stream)
        assert rc == mk.MK_OK, mk.status_string(rc)
        torch.cuda.synchronize()
        assert self.status.tolist()[0] == mk.MK_OK, self.status.tolist()
        o_lg, o_nx = self.orc.decode_step(self.kv_host, np.asarray(toks), np.asarray(pos),
                                          np.asarray(pt), np.asarray(pos) + 1)
        return lg.cpu().numpy(), nx.cpu().numpy(), o_lg, o_nx

    def gpu_kv_bits(self):
        torch.cuda.synchronize()
        return synth.bf16_bits(self.pool)

    def close(self):
        self.model.close()


# a small MoE (8 experts of width 128, top-2) and the 2B shapes cut to two layers, with
# max_batch 2 and 1,024 positions so that their scratch fits the static array
_TINY_MOE = synth.ModelConfig("tiny-moe", n_layers=2, d_model=256, n_q_heads=4, n_kv_heads=2,
                              head_dim=64, ffn_dim=0, vocab=4096, n_experts=8, top_k=2,
                              expert_ffn_dim=128, max_positions=512)
_DENSE_2B_SMALL = synth.DENSE_2B.with_(n_layers=2, max_batch=2, max_positions=1024)
_CASES = [(synth.TINY, 1), (synth.TINY, 3), (synth.TINY, 8), (_TINY_MOE, 1), (_TINY_MOE, 3),
          (_DENSE_2B_SMALL, 1), (_DENSE_2B_SMALL, 2)]


@pytest.mark.parametrize("cfg,B", _CASES, ids=[f"{c.name}-B{b}" for c, b in _CASES])
def test_noalloc_matches_the_oracle_on_two_consecutive_calls(cfg, B):
    from persistent_megakernel_05_b300 import build
    build.build()
    rng = np.random.default_rng(21 + B)
    pos = np.array([3, 15, 16, 40, 77, 100, 129, 200], np.int32)[:B]
    if cfg.d_model > 256:
        pos = pos + 700  # 45+ pages per row: the attention runs split over several CTAs
    pages = [int(p) // 16 + 2 for p in pos]
    npages = max(64, sum(pages) + 4)
    pair = _NoAllocPair(cfg, seed=21 + B, num_pages=npages, kv_seed=4)
    pt = synth.random_page_tables(rng, npages, pages, max(pages))
    toks = synth.random_tokens(rng, cfg.vocab, B)
    for call in range(2):
        g_lg, g_nx, o_lg, o_nx = pair.call(toks, pos + call, pt)
        check_logits(g_lg, g_nx, o_lg, o_nx, what=f"no-alloc B={B} call {call}")
        toks = g_nx
    assert check_kv(pair) == 2 * B * cfg.n_layers * 2 * cfg.n_kv_heads
    pair.close()


def test_noalloc_matches_the_handle_path():
    """The same kernel as mk_decode_step: same tokens, logits equal to within the float
    rounding of the RoPE table (made on the device here, on the host by mk_create), the
    same appends to the two pools; and the cost of a call beside a handle step."""
    cfg = synth.TINY
    npages = 64
    W = synth.make_weights(cfg, 21, device="cuda", gain_noise=0.02)
    model = mk.DecodeModel(cfg, W, npages)
    synth.fill_normal_bf16_(model.kv(), 4)
    pool2 = model.kv().clone()  # the caller owns the second pool
    rng = np.random.default_rng(21)
    B = 3
    pos = np.array([3, 40, 129], np.int32)
    pages = [int(p) // 16 + 2 for p in pos]
    pt = torch.tensor(synth.random_page_tables(rng, npages, pages, max(pages)), device="cuda")
    toks = torch.tensor(synth.random_tokens(rng, cfg.vocab, B), device="cuda")
    status = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        p = torch.tensor(pos + call, device="cuda")
        sl = p + 1
        nx_a = torch.empty(B, dtype=torch.int32, device="cuda")
        nx_b = torch.empty(B, dtype=torch.int32, device="cuda")
        lg_a = torch.empty((B, cfg.vocab), device="cuda")
        lg_b = torch.empty((B, cfg.vocab), device="cuda")
        model.step(toks, p, pt, sl, nx_a, lg_a)
        assert model.status()[0] == mk.MK_OK
        rc = mk.mk_decode_step_noalloc(model.desc, model.w, _addr(pool2), npages, _addr(toks),
                                       _addr(p), _addr(pt), pt.shape[1], _addr(sl), B,
                                       _addr(nx_b), _addr(lg_b), _addr(status), stream)
        assert rc == mk.MK_OK, mk.status_string(rc)
        torch.cuda.synchronize()
        assert status.tolist()[0] == mk.MK_OK, status.tolist()
        a, b = lg_a.cpu().numpy(), lg_b.cpu().numpy()
        assert np.abs(a - b).max() <= 1e-4 * max(1.0, np.abs(a).max()), f"call {call}"
        assert np.array_equal(nx_a.cpu().numpy(), nx_b.cpu().numpy())
        toks = nx_a.clone()
    ka = synth.bf16_bits(model.kv())
    kb = synth.bf16_bits(pool2)
    from harness import bf16_ulp_diff
    assert bf16_ulp_diff(ka, kb).max() <= 1
    # cost per call (the RoPE table is already in the array; warm both paths first)
    p = torch.tensor(pos + 2, device="cuda")
    sl, nx = p + 1, torch.empty(B, dtype=torch.int32, device="cuda")

    def timed(fn, n=20):
        fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            fn()
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / n * 1e6

    t_handle = timed(lambda: model.step(toks, p, pt, sl, nx, None))
    t_noalloc = timed(lambda: mk.mk_decode_step_noalloc(
        model.desc, model.w, _addr(pool2), npages, _addr(toks), _addr(p), _addr(pt), pt.shape[1],
        _addr(sl), B, _addr(nx), None, _addr(status), stream))
    print(f"\nper call, tiny model batch {B}: handle path {t_handle:.1f} us, no-allocation path "
          f"{t_noalloc:.1f} us (set-up kernel + step)")
    model.close()


def test_noalloc_rejects_a_descriptor_whose_scratch_does_not_fit():
    cfg = synth.TINY
    W = synth.make_weights(cfg, 22, device="cuda")
    model = mk.DecodeModel(cfg, W, 8)
    big = mk.mk_model_desc()
    ctypes.memmove(ctypes.byref(big), ctypes.byref(model.desc), ctypes.sizeof(big))
    big.max_positions = 1 << 20  # RoPE table alone: 1M * 32 * 8 B = 256 MiB > 8 MiB
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    rc = mk.mk_decode_step_noalloc(big, model.w, _addr(model.kv()), 8, _addr(dummy), _addr(dummy),
                                   _addr(dummy), 1, _addr(dummy), 1, _addr(dummy), None,
                                   _addr(dummy), None)
    assert rc == mk.MK_ERR_INVALID_ARG
    model.close()

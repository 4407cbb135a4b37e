"""GPU parity at the contexts the benchmark lines run: the 8B shapes at a 32,768-token
context (the attention partition with 2,048 pages per kv head), the MoE shapes (head
dim 64, 8 query heads per kv head) at a 4,096-token context at batch 1 and 8, and a
batch-8 run that crosses a continuous-batching replacement event, where the finished
rows' pages are handed to the new rows. Both sides are fed the GPU's tokens."""
import numpy as np
import pytest
import torch

import synth
import persistent_megakernel_05_b300 as mk
from harness import Pair, check_kv, check_kv_and_share, check_logits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from persistent_megakernel_05_b300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")


def test_dense_8b_two_layers_32k_context():
    """8B shapes (d 4096, 32/8 heads of 128, ffn 14336, vocab 128256), two layers, batch
    1 at positions 32768 and 32769 over 2,050 randomly permuted pages."""
    cfg = synth.DENSE_8B.with_(n_layers=2)
    ctx = 32768
    pages = (ctx + 2) // 16 + 1
    npages = pages + 6
    pair = Pair(cfg, seed=24, num_pages=npages, kv_seed=9)
    rng = np.random.default_rng(24)
    pt = synth.random_page_tables(rng, npages, [pages], max_pages=pages)
    tok = [int(synth.random_tokens(rng, cfg.vocab, 1)[0])]
    for s in range(2):
        g_lg, g_nx, o_lg, o_nx = pair.step(tok, [ctx + s], pt)
        check_logits(g_lg, g_nx, o_lg, o_nx, what=f"8B 32K step {s}")
        tok = [int(g_nx[0])]
    assert check_kv(pair) == 2 * cfg.n_layers * 2 * cfg.n_kv_heads
    pair.close()


@pytest.mark.parametrize("B", [1, 8])
def test_moe_two_layers_4k_context(B):
    """MoE shapes (d 2048, 32/4 heads of 64, 64 experts of 768, top-8) with two layers at
    a 4,096-token context per row (batch 8: ragged around it)."""
    cfg = synth.MOE.with_(n_layers=2)
    rng = np.random.default_rng(25 + B)
    pos = (4096 - rng.integers(0, 64, size=B)).astype(np.int32) if B > 1 else np.array([4096], np.int32)
    pages = [int(p + 2) // 16 + 1 for p in pos]
    npages = sum(pages) + 4
    pair = Pair(cfg, seed=25, num_pages=npages, kv_seed=10)
    pt = synth.random_page_tables(rng, npages, pages, max_pages=max(pages))
    toks = synth.random_tokens(rng, cfg.vocab, B)
    for s in range(2):
        g_lg, g_nx, o_lg, o_nx = pair.step(toks, pos + s, pt)
        check_logits(g_lg, g_nx, o_lg, o_nx, what=f"MoE 4K B={B} step {s}")
        u = pair.gpu.buffer(mk.MK_BUF_MOE_UNION)
        assert (u >= cfg.top_k).all() and (u <= min(cfg.n_experts, B * cfg.top_k)).all(), u
        toks = g_nx
    assert check_kv(pair) == 2 * B * cfg.n_layers * 2 * cfg.n_kv_heads
    pair.close()


def _refill_pages(pair, pages, seed):
    """Fresh seeded N(0, 1) K/V history in `pages` of both pools (a new sequence's
    prefilled context); it becomes the starting state the K/V check compares against."""
    cfg = pair.cfg
    shape = (cfg.n_layers, len(pages), 2, cfg.n_kv_heads, cfg.page_size, cfg.head_dim)
    fresh = synth.normal_bf16(shape, 1.0, seed)
    bits = synth.bf16_bits(fresh)
    idx = np.asarray(pages, np.int64)
    pair.kv_host[:, idx] = bits
    pair.kv_start[:, idx] = bits
    kv = pair.gpu.kv()
    kv[:, torch.as_tensor(idx, device=kv.device)] = fresh.to(kv.device)
    torch.cuda.synchronize()


def test_tiny_batch8_continuous_batching_crosses_a_replacement():
    """Batch 8 for 72 steps. At step 64 the rows of the first replacement event finish;
    their pages go back to the pool and the new rows (fresh 48-token contexts) draw those
    freed pages first, so the new rows attend over and append into pages that other
    sequences wrote earlier in the run. Every step is compared from a common K/V history
    (the GPU's, handed to the oracle after the step's appends are checked)."""
    cfg = synth.TINY
    B, steps, event, fresh_len = 8, 72, 64, 48
    rng = np.random.default_rng(26)
    lens = rng.integers(40, 200, size=B).astype(np.int32)
    maxp = (200 + steps) // 16 + 2
    need = [int(n + steps) // 16 + 1 for n in lens]
    npages = sum(need) + 8
    pair = Pair(cfg, seed=26, num_pages=npages, kv_seed=13)
    free = [int(x) for x in rng.permutation(npages)]
    pt = np.full((B, maxp), -1, np.int32)
    for b in range(B):
        pt[b, :need[b]] = [free.pop() for _ in range(need[b])]
    pos = lens.copy()
    toks = synth.random_tokens(rng, cfg.vocab, B)
    reused = 0
    for t in range(steps):
        if t == event:
            for slot in synth.replacement_slots(0, B):
                freed = [int(x) for x in pt[slot] if x >= 0]
                free = freed + free  # the pool hands out the freed pages first
                n = (fresh_len + steps - event) // 16 + 1
                new = [free.pop(0) for _ in range(n)]
                reused += len(set(new) & set(freed))
                pt[slot] = -1
                pt[slot, :n] = new
                _refill_pages(pair, new, seed=1000 + slot)
                pos[slot] = fresh_len
                toks[slot] = int(synth.random_tokens(rng, cfg.vocab, 1)[0])
        g_lg, g_nx, o_lg, o_nx = pair.step(toks, pos, pt)
        check_logits(g_lg, g_nx, o_lg, o_nx, what=f"step {t}")
        # this step's appends at the oracle's slots and values; then both sides go on
        # from the same K/V history
        assert check_kv_and_share(pair) == B * cfg.n_layers * 2 * cfg.n_kv_heads
        toks = g_nx.copy()
        pos = pos + 1
    assert reused > 0
    pair.close()

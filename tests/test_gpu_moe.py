"""GPU parity of the MoE layers (softmax top-k routing over the router logits, routed
experts' SwiGLU, routing-weighted sum; "Kog Inference Engine" MoE paragraphs) against the
CPU oracle, through the C ABI, at batch 1 and 2 (tagged-word hand-off) and batches 3 and 8
(fp32 + counters), over the union of the rows' routes."""
import numpy as np
import pytest
import torch

import synth
import persistent_megakernel_05_b300 as mk
from harness import Pair, check_kv, check_logits

pytestmark = pytest.mark.gpu

# a small MoE: 8 experts of width 128, top-2
TINY_MOE = synth.ModelConfig("tiny-moe", n_layers=2, d_model=256, n_q_heads=4, n_kv_heads=2,
                             head_dim=64, ffn_dim=0, vocab=4096, n_experts=8, top_k=2,
                             expert_ffn_dim=128, max_positions=512)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from persistent_megakernel_05_b300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")


def _union_ok(pair, cfg, B):
    u = pair.gpu.buffer(mk.MK_BUF_MOE_UNION)
    assert u.shape == (cfg.n_layers,)
    assert (u >= cfg.top_k).all() and (u <= min(cfg.n_experts, B * cfg.top_k)).all(), u
    return u


@pytest.mark.parametrize("gain_noise", [0.0, 0.02])
def test_tiny_moe_prompt_then_greedy(gain_noise):
    cfg = TINY_MOE
    pair = Pair(cfg, seed=11, num_pages=8, gain_noise=gain_noise)
    rng = np.random.default_rng(11)
    prompt = synth.random_tokens(rng, cfg.vocab, 20)
    pt = synth.random_page_tables(rng, 8, [3], max_pages=4)
    tok = int(prompt[0])
    for t in range(30):
        g_lg, g_nx, o_lg, o_nx = pair.step([tok], [t], pt)
        check_logits(g_lg, g_nx, o_lg, o_nx, what=f"step {t}")
        u = _union_ok(pair, cfg, 1)
        assert (u == cfg.top_k).all()  # one row: exactly its k experts
        tok = int(prompt[t + 1]) if t + 1 < 20 else int(g_nx[0])
    assert check_kv(pair) == 30 * cfg.n_layers * 2 * cfg.n_kv_heads
    pair.close()


@pytest.mark.parametrize("B", [2, 3, 8])
def test_tiny_moe_batch_ragged(B):
    """Batch 2 (tagged words), 3 and 8 (fp32 + counters): each row routes on its own; the
    expert stages run over the union of the rows' routes."""
    cfg = TINY_MOE
    pair = Pair(cfg, seed=12, num_pages=96, kv_seed=3)
    rng = np.random.default_rng(12)
    pos = np.array([0, 15, 16, 17, 100, 31, 200, 63], np.int32)[:B]
    pages = [(int(p) + 4) // 16 + 1 for p in pos]
    pt = synth.random_page_tables(rng, 96, pages, max_pages=max(pages) + 1)
    toks = synth.random_tokens(rng, cfg.vocab, B)
    for s in range(4):
        g_lg, g_nx, o_lg, o_nx = pair.step(toks, pos + s, pt)
        check_logits(g_lg, g_nx, o_lg, o_nx, what=f"B={B} step {s}")
        _union_ok(pair, cfg, B)
        toks = g_nx
    check_kv(pair)
    pair.close()


@pytest.mark.parametrize("B", [1, 8])
def test_moe_64x768_top8_two_layers(B):
    """The MoE decoder's own shapes (d 2048, 32/4 heads of 64, 64 experts of 768, top-8,
    vocab 128256) with two layers, so the oracle stays fast."""
    cfg = synth.MOE.with_(n_layers=2, max_positions=1024)
    npages = 48 * B
    pair = Pair(cfg, seed=13, num_pages=npages, kv_seed=5)
    rng = np.random.default_rng(13)
    pos = rng.integers(1, 400, size=B).astype(np.int32)
    pages = [int(p) // 16 + 1 for p in pos]
    pt = synth.random_page_tables(rng, npages, pages, max_pages=max(pages) + 1)
    toks = synth.random_tokens(rng, cfg.vocab, B)
    for s in range(2):
        g_lg, g_nx, o_lg, o_nx = pair.step(toks, pos + s, pt)
        check_logits(g_lg, g_nx, o_lg, o_nx, what=f"B={B} step {s}")
        u = _union_ok(pair, cfg, B)
        if B == 1:
            assert (u == 8).all()
        toks = g_nx
    check_kv(pair)
    pair.close()

"""Temperature sampling limited to the top-k logits (the limited top-k of the sampling
modes: "Cohere, Megakernel sunum sistemini acik kaynak yapti", section "Sinirlar acikca
yazilmis"). The kernel keeps each row's running top-k list in the LM-head epilogue,
publishes every CTA's list, merges them and draws by Gumbel-max over the merged list;
the CPU oracle draws from the same rule (oracle.sample_gumbel_topk)."""
import numpy as np
import pytest
import torch

import oracle
import synth
import persistent_megakernel_05_b300 as mk
from harness import Pair, check_kv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from persistent_megakernel_05_b300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")


def _topk_scores(logits, T, k, seed, pos, row):
    """The scores of the candidate set (others -inf), to find the oracle's margin."""
    order = np.lexsort((np.arange(len(logits)), -logits.astype(np.float64)))
    keep = np.full(len(logits), False)
    keep[order[:k]] = True
    z = oracle.gumbel_scores(logits, T, seed, pos, row)
    return np.where(keep, z, -np.inf)


@pytest.mark.parametrize("k", [1, 5, 32])
def test_topk_draws_match_the_oracle(k):
    cfg = synth.TINY
    T, seed = 1.5, 0x5EED0000 + k
    pair = Pair(cfg, seed=40 + k, num_pages=32, kv_seed=4)
    pair.gpu.set_sampling(T, seed, top_k=k)
    rng = np.random.default_rng(40 + k)
    B = 3
    pos = np.array([5, 40, 77], np.int32)
    pages = [int(p) // 16 + 2 for p in pos]
    pt = synth.random_page_tables(rng, 32, pages, max_pages=max(pages))
    toks = synth.random_tokens(rng, cfg.vocab, B)
    compared = 0
    for s in range(10):
        g_lg, g_nx, o_lg, o_nx = pair.step(toks, pos + s, pt)
        assert np.abs(g_lg - o_lg).max() <= 3e-2
        for b in range(B):
            z = _topk_scores(o_lg[b], T, k, seed, int(pos[b] + s), b)
            ref = oracle.sample_gumbel_topk(o_lg[b], T, k, seed, int(pos[b] + s), b)
            assert int(np.argmax(z)) == ref
            # the GPU's token is in the GPU's own top k
            ahead = np.sum((g_lg[b] > g_lg[b][g_nx[b]]) |
                           ((g_lg[b] == g_lg[b][g_nx[b]]) & (np.arange(cfg.vocab) < g_nx[b])))
            assert ahead < k, (s, b, ahead)
            top2 = np.sort(z)[-2:]
            if k == 1 or top2[1] - top2[0] > 0.1:
                assert g_nx[b] == ref, (s, b, k)
                compared += 1
        toks = g_nx
    assert compared >= 15
    pair.close()


def test_topk_over_a_full_vocabulary_row():
    """The MoE shapes' 128256-token head over 148 CTAs' lists, batch 1 and 2 layers."""
    cfg = synth.MOE.with_(n_layers=2, max_positions=1024)
    T, k, seed = 0.7, 8, 77
    pair = Pair(cfg, seed=46, num_pages=48, kv_seed=5)
    pair.gpu.set_sampling(T, seed, top_k=k)
    rng = np.random.default_rng(46)
    pos = np.array([300], np.int32)
    pt = synth.random_page_tables(rng, 48, [20], max_pages=20)
    toks = synth.random_tokens(rng, cfg.vocab, 1)
    compared = 0
    for s in range(4):
        g_lg, g_nx, o_lg, o_nx = pair.step(toks, pos + s, pt)
        z = _topk_scores(o_lg[0], T, k, seed, int(pos[0] + s), 0)
        top2 = np.sort(z)[-2:]
        if top2[1] - top2[0] > 0.1:
            assert g_nx[0] == oracle.sample_gumbel_topk(o_lg[0], T, k, seed, int(pos[0] + s), 0)
            compared += 1
        toks = g_nx
    assert compared >= 2
    check_kv(pair)
    pair.close()


def test_topk_multi_step_launch_equals_single_steps():
    cfg = synth.TINY
    B, n = 3, 6
    W = synth.make_weights(cfg, 47, device="cuda")
    ms = []
    for _ in range(2):
        m = mk.DecodeModel(cfg, W, 40)
        synth.fill_normal_bf16_(m.kv(), 6)
        m.set_sampling(1.1, seed=99, top_k=4)
        ms.append(m)
    torch.cuda.synchronize()
    a, b = ms
    rng = np.random.default_rng(47)
    pt = torch.tensor(synth.random_page_tables(rng, 40, [10] * B, 10), device="cuda")
    pos = torch.tensor([5, 70, 120], dtype=torch.int32, device="cuda")
    toks = torch.tensor(synth.random_tokens(rng, cfg.vocab, B), device="cuda")
    ref = torch.empty((n, B), dtype=torch.int32, device="cuda")
    cur = toks.clone()
    for s in range(n):
        p = pos + s
        a.step(cur, p, pt, p + 1, ref[s])
        cur = ref[s].clone()
    out = torch.empty((n, B), dtype=torch.int32, device="cuda")
    b.steps(n, toks, pos, pt, pos + 1, out)
    assert a.status()[0] == mk.MK_OK and b.status()[0] == mk.MK_OK
    assert torch.equal(out, ref)
    a.close()
    b.close()


def test_topk_argument_checks():
    cfg = synth.TINY
    W = synth.make_weights(cfg, 48, device="cuda")
    m = mk.DecodeModel(cfg, W, 8)
    for bad in (-1, 33):
        with pytest.raises(RuntimeError):
            m.set_sampling(1.0, seed=1, top_k=bad)
    m.set_sampling(1.0, seed=1, top_k=32)
    m.close()

"""Several decode steps in one launch (mk_decode_steps): each step's token is fed back on
the device ("Kog AI: standart GPU'larda 3,000 token/s", on kernel boundaries and on
sampling kept on the GPU). A launch of n steps must give exactly what n single-step
launches give when each step's tokens are fed to the next (the arithmetic is the same),
and must match the CPU oracle, which replays the steps with the GPU's tokens."""
import numpy as np
import pytest
import torch

import synth
import persistent_megakernel_05_b300 as mk
from harness import check_kv, Pair, MARGIN, LOGIT_ATOL

pytestmark = pytest.mark.gpu

TINY_MOE = synth.ModelConfig("tiny-moe", n_layers=2, d_model=256, n_q_heads=4, n_kv_heads=2,
                             head_dim=64, ffn_dim=0, vocab=4096, n_experts=8, top_k=2,
                             expert_ffn_dim=128, max_positions=512)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from persistent_megakernel_05_b300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")


def _twin_models(cfg, W, npages, kv_seed):
    """Two handles on the same weights, each with its own copy of one seeded KV pool."""
    ms = []
    for _ in range(2):
        m = mk.DecodeModel(cfg, W, npages)
        synth.fill_normal_bf16_(m.kv(), kv_seed)
        ms.append(m)
    torch.cuda.synchronize()
    return ms


def _single_steps(m, toks, pos, pt, n, with_logits):
    B = toks.numel()
    dev = toks.device
    out = torch.empty((n, B), dtype=torch.int32, device=dev)
    lg = torch.empty((B, m.cfg.vocab), dtype=torch.float32, device=dev) if with_logits else None
    cur = toks.clone()
    for s in range(n):
        p = pos + s
        m.step(cur, p, pt, p + 1, out[s], lg if s == n - 1 else None)
        cur = out[s].clone()
    return out, lg


CASES = {
    "tiny-b1": (synth.TINY, 1, None),
    "tiny-b3": (synth.TINY, 3, None),
    "tiny-swa-b6": (synth.TINY.with_(sliding_window=48), 6, None),
    "tiny-b4-prefix": (synth.TINY, 4, ([0, 0, 0, 3], [3, 3, 3, 0])),
    "moe-b1": (TINY_MOE, 1, None),
    "moe-b8": (TINY_MOE, 8, None),
}


@pytest.mark.parametrize("case", list(CASES))
def test_launch_of_n_steps_equals_n_launches(case):
    cfg, B, groups = CASES[case]
    n = 9
    npages = 16 * B + 8
    W = synth.make_weights(cfg, 31, device="cuda")
    a, b = _twin_models(cfg, W, npages, kv_seed=4)
    rng = np.random.default_rng(31)
    if groups:  # rows 0-2 share a 3-page prefix run, row 3 has pages of its own
        perm = rng.permutation(npages)
        pt = np.full((B, 12), -1, np.int32)
        pt[:3, :3] = perm[:3]
        for r in range(3):
            pt[r, 3:12] = perm[3 + 9 * r:12 + 9 * r]
        pt[3, :12] = perm[30:42]
        a.set_shared_prefix(*groups)
        b.set_shared_prefix(*groups)
        pos = np.array([48 + 3, 48 + 20, 48 + 40, 30], np.int32)
    else:
        pt = synth.random_page_tables(rng, npages, [12] * B, 12)
        pos = rng.integers(10, 150, size=B).astype(np.int32)
    dev = "cuda"
    ptd = torch.tensor(pt, device=dev)
    posd = torch.tensor(pos, device=dev)
    toks = torch.tensor(synth.random_tokens(rng, cfg.vocab, B), device=dev)
    ref, ref_lg = _single_steps(a, toks, posd, ptd, n, True)
    out = torch.full((n, B), -1, dtype=torch.int32, device=dev)
    lg = torch.full((B, cfg.vocab), float("nan"), device=dev)
    b.steps(n, toks, posd, ptd, posd + 1, out, lg)
    assert a.status()[0] == mk.MK_OK and b.status()[0] == mk.MK_OK
    assert torch.equal(out, ref), (out, ref)
    assert torch.equal(lg, ref_lg)
    assert torch.equal(a.kv().view(torch.int16), b.kv().view(torch.int16))
    # a second launch continues from where the first ended (epochs, counters)
    nxt = out[-1].clone()
    out2 = torch.empty((3, B), dtype=torch.int32, device=dev)
    b.steps(3, nxt, posd + n, ptd, posd + n + 1, out2)
    ref2, _ = _single_steps(a, nxt, posd + n, ptd, 3, False)
    assert b.status()[0] == mk.MK_OK
    assert torch.equal(out2, ref2)
    a.close()
    b.close()


def test_multi_step_matches_the_oracle():
    """Tiny decoder, batch 2, 7 steps in one launch: the oracle replays them with the
    GPU's tokens; tokens agree where the oracle's top-2 margin exceeds 0.1, the last
    step's logits within the parity bar, and the K/V rows written are the oracle's."""
    cfg = synth.TINY
    B, n = 2, 7
    pair = Pair(cfg, seed=32, num_pages=24, kv_seed=5)
    rng = np.random.default_rng(32)
    pt = synth.random_page_tables(rng, 24, [10, 10], 10)
    pos = np.array([17, 60], np.int32)
    toks = synth.random_tokens(rng, cfg.vocab, B)
    dev = "cuda"
    out = torch.empty((n, B), dtype=torch.int32, device=dev)
    lg = torch.empty((B, cfg.vocab), dtype=torch.float32, device=dev)
    posd = torch.tensor(pos, device=dev)
    pair.gpu.steps(n, torch.tensor(toks, device=dev), posd, torch.tensor(pt, device=dev), posd + 1,
                   out, lg)
    assert pair.gpu.status()[0] == mk.MK_OK
    g_tok = out.cpu().numpy()
    cur = toks.copy()
    for s in range(n):
        o_lg, o_nx = pair.orc.decode_step(pair.kv_host, cur, pos + s, pt, pos + s + 1)
        for r in range(B):
            top2 = np.partition(o_lg[r], -2)[-2:]
            if top2[1] - top2[0] > MARGIN:
                assert g_tok[s, r] == o_nx[r], (s, r)
        cur = g_tok[s]
    err = np.abs(lg.cpu().numpy() - o_lg).max()
    assert err <= LOGIT_ATOL, err
    assert check_kv(pair) == n * B * cfg.n_layers * 2 * cfg.n_kv_heads
    pair.close()


def test_multi_step_sampling_equals_single_steps():
    cfg = synth.TINY
    B, n = 3, 6
    W = synth.make_weights(cfg, 33, device="cuda")
    a, b = _twin_models(cfg, W, 40, kv_seed=6)
    for m in (a, b):
        m.set_sampling(0.8, seed=1234)
    rng = np.random.default_rng(33)
    pt = torch.tensor(synth.random_page_tables(rng, 40, [10] * B, 10), device="cuda")
    pos = torch.tensor([5, 70, 120], dtype=torch.int32, device="cuda")
    toks = torch.tensor(synth.random_tokens(rng, cfg.vocab, B), device="cuda")
    ref, _ = _single_steps(a, toks, pos, pt, n, False)
    out = torch.empty((n, B), dtype=torch.int32, device="cuda")
    b.steps(n, toks, pos, pt, pos + 1, out)
    assert b.status()[0] == mk.MK_OK
    assert torch.equal(out, ref)
    a.close()
    b.close()


def test_multi_step_errors():
    cfg = synth.TINY
    W = synth.make_weights(cfg, 34, device="cuda")
    m = mk.DecodeModel(cfg, W, 8)
    synth.fill_normal_bf16_(m.kv(), 1)
    t = torch.zeros(1, dtype=torch.int32, device="cuda")
    p = torch.tensor([20], dtype=torch.int32, device="cuda")
    pt = torch.tensor([[0, 1, 2]], dtype=torch.int32, device="cuda")
    out = torch.empty((40, 1), dtype=torch.int32, device="cuda")
    with pytest.raises(RuntimeError):
        m.steps(0, t, p, pt, p + 1, out)
    # the last step's position (20 + 39) lies past the 3 mapped pages: rejected on the
    # device before any work, and the handle recovers
    m.steps(40, t, p, pt, p + 1, out)
    assert m.status()[0] == mk.MK_ERR_INVALID_ARG
    m.reset()
    m.steps(20, t, p, pt, p + 1, out)  # positions 20..39 fit
    assert m.status()[0] == mk.MK_OK
    m.close()


def test_full_size_2b_sixteen_steps_equal_sixteen_launches():
    """The 2B decoder at its 8192-token context, as the benchmark runs it."""
    cfg = synth.DENSE_2B
    npages = (8192 + 64) // 16 + 2
    W = synth.make_weights(cfg, 1, device="cuda")
    a, b = _twin_models(cfg, W, npages, kv_seed=11)
    rng = np.random.default_rng(1)
    pt = torch.tensor(synth.random_page_tables(rng, npages, [npages - 2], npages - 2), device="cuda")
    pos = torch.tensor([8192], dtype=torch.int32, device="cuda")
    toks = torch.tensor(synth.random_tokens(rng, cfg.vocab, 1), device="cuda")
    n = 16
    ref, ref_lg = _single_steps(a, toks, pos, pt, n, True)
    out = torch.empty((n, 1), dtype=torch.int32, device="cuda")
    lg = torch.empty((1, cfg.vocab), dtype=torch.float32, device="cuda")
    b.steps(n, toks, pos, pt, pos + 1, out, lg)
    assert a.status()[0] == mk.MK_OK and b.status()[0] == mk.MK_OK
    assert torch.equal(out, ref)
    assert torch.equal(lg, ref_lg)
    a.close()
    b.close()

"""GPU parity of shared-prefix (cascade) attention against the CPU oracle, through the
C ABI. Rows that share a prefix-cached page run ("Cohere, Megakernel sunum sistemini
acik kaynak yapti", section "Sinirlar acikca yazilmis": prefix cache) have their prefix
K/V read once per kv head for the group; the oracle attends every row over its own page
table, so equal results show the shared read changes nothing but summation order."""
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


def grouped_page_tables(rng, num_pages, B, groups, private_pages, max_pages):
    """Page tables in which each group (rows, prefix pages) shares one prefix page run;
    every row then has `private_pages` pages of its own. Returns the table and the
    leader / shared-pages lists that declare the groups."""
    perm = list(rng.permutation(num_pages))
    pt = np.full((B, max_pages), -1, np.int32)
    leader, shared = list(range(B)), [0] * B
    for rows, P in groups:
        run = [perm.pop() for _ in range(P)]
        for r in rows:
            pt[r, :P] = run
            leader[r] = min(rows)
            shared[r] = P
    for b in range(B):
        start = shared[b]
        pt[b, start:start + private_pages] = [perm.pop() for _ in range(private_pages)]
    return pt, leader, shared


def test_8b_shapes_batch4_one_group_two_column_tiles():
    """8B shapes (G = 4, head dim 128): 4 rows x 4 heads = 16 query columns in two MMA
    tiles, two finish passes per piece; the prefix spans several splits. Each step's K/V
    appends are checked from a common history (with the 8B shapes, one side's rounding of
    an earlier append shifts the next layers' inputs enough to move small K/V elements
    past the bar)."""
    cfg = synth.DENSE_8B.with_(n_layers=2, max_positions=2048)
    B, P = 4, 24
    npages = P + 4 * B + 8
    pair = Pair(cfg, seed=21, num_pages=npages, kv_seed=7)
    rng = np.random.default_rng(21)
    pt, leader, shared = grouped_page_tables(rng, npages, B, [((0, 1, 2, 3), P)], 4, P + 4)
    pair.gpu.set_shared_prefix(leader, shared)
    pos = (P * 16 + rng.integers(0, 40, size=B)).astype(np.int32)
    toks = synth.random_tokens(rng, cfg.vocab, B)
    for s in range(3):
        g_lg, g_nx, o_lg, o_nx = pair.step(toks, pos + s, pt)
        check_logits(g_lg, g_nx, o_lg, o_nx, what=f"step {s}")
        assert check_kv_and_share(pair) == B * cfg.n_layers * 2 * cfg.n_kv_heads
        toks = g_nx
    pair.close()


@pytest.mark.parametrize("B,groups", [
    (2, [((0, 1), 4)]),                          # tagged words, one tile (4 columns)
    (3, [((0, 1, 2), 4)]),                       # fp32 + counters, one tile (6 columns)
    (6, [((0, 2, 3), 4), ((1, 5), 3)]),          # fp32 + counters; row 4 alone
    (8, [((0, 1, 2, 3, 4, 5, 6, 7), 5)]),        # 16 columns of head dim 64
])
def test_tiny_groups_with_sliding_layers(B, groups):
    """Tiny decoder (G = 2, head dim 64) with a 96-token window on layer 1: there the
    window cuts into the prefix, so the rows attend on their own; layer 0 shares."""
    cfg = synth.TINY.with_(sliding_window=96)
    npages = 8 + 8 * B + 16
    pair = Pair(cfg, seed=22, num_pages=npages, kv_seed=8)
    rng = np.random.default_rng(22 + B)
    pt, leader, shared = grouped_page_tables(rng, npages, B, groups, 6, 16)
    pair.gpu.set_shared_prefix(leader, shared)
    pos = np.array([s * 16 + int(rng.integers(0, 60)) for s in shared], np.int32)
    toks = synth.random_tokens(rng, cfg.vocab, B)
    for s in range(4):
        g_lg, g_nx, o_lg, o_nx = pair.step(toks, pos + s, pt)
        check_logits(g_lg, g_nx, o_lg, o_nx, what=f"B={B} step {s}")
        toks = g_nx
    check_kv(pair)
    pair.close()


def test_moe_shapes_two_rows_share():
    """The MoE decoder's attention shapes (G = 8, head dim 64): two rows fill both column
    tiles; a third row attends alone."""
    cfg = synth.MOE.with_(n_layers=2, max_positions=1024)
    B, P = 3, 20
    npages = P + 6 * B + 8
    pair = Pair(cfg, seed=23, num_pages=npages, kv_seed=9)
    rng = np.random.default_rng(23)
    pt, leader, shared = grouped_page_tables(rng, npages, B, [((0, 1), P)], 6, P + 6)
    pair.gpu.set_shared_prefix(leader, shared)
    pos = np.array([P * 16 + 5, P * 16 + 33, 50], np.int32)
    toks = synth.random_tokens(rng, cfg.vocab, B)
    for s in range(2):
        g_lg, g_nx, o_lg, o_nx = pair.step(toks, pos + s, pt)
        check_logits(g_lg, g_nx, o_lg, o_nx, what=f"step {s}")
        toks = g_nx
    check_kv(pair)
    pair.close()


def test_declaration_rules():
    cfg = synth.TINY
    W = synth.make_weights(cfg, 24, device="cuda")
    m = mk.DecodeModel(cfg, W, 16)
    for leader, shared in (([0, 2], [1, 1]),    # leader after the row
                           ([0, 0], [2, 1]),    # shared pages differ within the group
                           ([-1, 0], [1, 1])):  # no leader
        with pytest.raises(RuntimeError):
            m.set_shared_prefix(leader, shared)
    m.set_shared_prefix([0, 1, 1], [0, 1, 1])  # row 0 alone; rows 1 and 2 share a page
    with pytest.raises(RuntimeError):  # 9 rows > max batch
        m.set_shared_prefix([0] * 9, [1] * 9)
    with pytest.raises(RuntimeError):  # leader's own leader must be itself
        m.set_shared_prefix([0, 0, 1], [1, 1, 1])
    # groups declared for batch 3: a batch-2 step is refused on the host
    t = torch.zeros(2, dtype=torch.int32, device="cuda")
    p = torch.tensor([20, 20], dtype=torch.int32, device="cuda")
    pt = torch.tensor([[0, 1, 2, 3], [4, 5, 6, 7]], dtype=torch.int32, device="cuda")
    nx = torch.empty(2, dtype=torch.int32, device="cuda")
    with pytest.raises(RuntimeError):
        m.step(t, p, pt, p + 1, nx)
    m.set_shared_prefix()  # cleared: the step runs
    m.step(t, p, pt, p + 1, nx)
    assert m.status()[0] == mk.MK_OK
    m.close()
    # 8B shapes (G = 4): at most 4 rows per group
    cfg8 = synth.DENSE_8B.with_(n_layers=1, d_model=512, ffn_dim=512, vocab=1024,
                               max_positions=256)
    W8 = synth.make_weights(cfg8, 25, device="cuda")
    m8 = mk.DecodeModel(cfg8, W8, 16)
    m8.set_shared_prefix([0, 0, 0, 0], [2, 2, 2, 2])
    with pytest.raises(RuntimeError):
        m8.set_shared_prefix([0] * 5, [2] * 5)
    m8.close()


def test_full_size_8b_prefix_equals_unshared():
    """The 8B decoder at full size with a 16384-token shared prefix and 1024-token private
    runs (batch 4), as the benchmark runs it: the step with the group declared equals the
    step without it (the same launch reads the prefix per row) to fp32 summation order,
    and both give the same tokens."""
    cfg = synth.DENSE_8B
    B, P, priv = 4, 1024, 64
    npages = P + B * priv + 2
    W = synth.make_weights(cfg, 26, device="cuda")
    m = mk.DecodeModel(cfg, W, npages)
    synth.fill_normal_bf16_(m.kv(), 10)
    rng = np.random.default_rng(26)
    pt_np = synth.prefix_shared_page_tables(rng, npages, B, P, priv, P + priv)
    dev = "cuda"
    pt = torch.tensor(pt_np, device=dev)
    pos = torch.tensor([P * 16 + 256 + 100 * b for b in range(B)], dtype=torch.int32, device=dev)
    toks = torch.tensor(synth.random_tokens(rng, cfg.vocab, B), device=dev)
    outs = []
    for share in (True, False):
        if share:
            m.set_shared_prefix([0] * B, [P] * B)
        else:
            m.set_shared_prefix()
        lg = torch.empty((B, cfg.vocab), dtype=torch.float32, device=dev)
        nx = torch.empty(B, dtype=torch.int32, device=dev)
        m.step(toks, pos, pt, pos + 1, nx, lg)  # the same K/V append both times
        assert m.status()[0] == mk.MK_OK
        outs.append((lg.cpu().numpy(), nx.cpu().numpy()))
    (a, ta), (b, tb) = outs
    err = float(np.abs(a - b).max())
    assert err <= 5e-3, err
    for r in range(B):
        top2 = np.partition(b[r], -2)[-2:]
        if top2[1] - top2[0] > 1e-2:
            assert ta[r] == tb[r]
    m.close()

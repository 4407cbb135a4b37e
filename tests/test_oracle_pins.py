"""Pins for the CPU oracle (no GPU).

The pages print no equations and no worked example of the decode step, so the
oracle is pinned to things other than itself: closed forms (RMSNorm of a constant
vector, RoPE as a complex rotation, single-key attention), textbook/library routines
(torch rms_norm, scaled_dot_product_attention with GQA, silu, stable sort), an
independently written float64 NumPy twin, and structural invariants (cached decode
equals a full causal recompute; paged equals contiguous; page permutations and
batch composition change nothing; MoE with one expert is the dense MLP).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth
from oracle.twin import Twin, bf16_bits_to_f64, round_to_bf16

TINY = synth.TINY
TINY_MOE = synth.ModelConfig("tiny-moe", n_layers=2, d_model=256, n_q_heads=4, n_kv_heads=2,
                             head_dim=64, ffn_dim=0, vocab=512, n_experts=8, top_k=2,
                             expert_ffn_dim=128, max_positions=512)


def bits(t):
    return synth.bf16_bits(t)


# ---------------------------------------------------------------- BF16 rounding
def test_bf16_round_to_nearest_even_cases():
    one = 1.0
    ulp = 2.0 ** -7  # BF16 spacing at 1.0 (8 significant bits)
    cases = {
        one: 0x3F80,
        one + ulp / 2: 0x3F80,          # tie -> even (1.0)
        one + 3 * ulp / 2: 0x3F82,      # tie -> even (1 + 2 ulp)
        one + ulp / 2 + 2 ** -20: 0x3F81,  # just above the tie -> up
        -2.0: 0xC000,
        0.0: 0x0000,
    }
    for x, want in cases.items():
        assert oracle.lib().or_f32_to_bf16(x) == want, x


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(4000) * np.exp(rng.uniform(-20, 20, 4000))).astype(np.float32)
    got = oracle.f32_to_bf16_bits(x)
    want = bits(torch.from_numpy(x).to(torch.bfloat16))
    assert np.array_equal(got, want)
    assert np.array_equal(bits(torch.from_numpy(x).to(torch.bfloat16)),
                          (round_to_bf16(x).astype(np.float32).view(np.uint32) >> 16)
                          .astype(np.uint16))


# ---------------------------------------------------------------- RMSNorm
def test_rmsnorm_constant_vector_closed_form():
    n, eps = 256, 1e-5
    g = torch.ones(n, dtype=torch.bfloat16)
    for c in (3.0, -0.25, 1e-3):
        out = oracle.rmsnorm(np.full(n, c, np.float32), bits(g), eps)
        want = c / math.sqrt(c * c + eps)
        np.testing.assert_allclose(out, want, rtol=1e-6)


def test_rmsnorm_matches_torch_and_uses_gain():
    rng = np.random.default_rng(1)
    n, eps = 2048, 1e-5
    x = rng.standard_normal(n).astype(np.float32) * 0.3
    g = (1 + 0.1 * torch.from_numpy(rng.standard_normal(n).astype(np.float32))).to(torch.bfloat16)
    out = oracle.rmsnorm(x, bits(g), eps)
    want = F.rms_norm(torch.from_numpy(x).double(), (n,), g.double(), eps).numpy()
    np.testing.assert_allclose(out, want, rtol=2e-6, atol=1e-6)
    ms = float(np.mean(x.astype(np.float64) ** 2))
    assert np.sqrt(np.mean((out / g.float().numpy()) ** 2)) == pytest.approx(
        math.sqrt(ms / (ms + eps)), abs=1e-6)


# ---------------------------------------------------------------- RoPE
def test_rope_position_zero_is_identity():
    v = np.random.default_rng(2).standard_normal(128).astype(np.float32)
    assert np.array_equal(oracle.rope(v, 0, 1e4), v)


def test_rope_single_pair_is_rotation_by_pos_radians():
    # hd = 2: one pair, inv_freq = theta^0 = 1, so position p rotates by p radians
    for p in (1, 2, 7):
        out = oracle.rope(np.array([1.0, 0.0], np.float32), p, 1e4)
        np.testing.assert_allclose(out, [math.cos(p), math.sin(p)], atol=1e-6)


def test_rope_is_complex_rotation_and_keeps_pair_norms():
    rng = np.random.default_rng(3)
    hd, theta = 128, 1e4
    v = rng.standard_normal(hd).astype(np.float32)
    for pos in (1, 17, 4095, 8191):
        out = oracle.rope(v, pos, theta)
        i = np.arange(hd // 2)
        z = (v[:64] + 1j * v[64:]) * np.exp(1j * pos * theta ** (-2.0 * i / hd))
        np.testing.assert_allclose(out, np.concatenate([z.real, z.imag]), atol=2e-5)
        np.testing.assert_allclose(np.hypot(out[:64], out[64:]), np.hypot(v[:64], v[64:]),
                                   rtol=1e-5)


def test_rope_scores_depend_only_on_relative_position():
    rng = np.random.default_rng(4)
    q = rng.standard_normal(64).astype(np.float32)
    k = rng.standard_normal(64).astype(np.float32)
    a = np.dot(oracle.rope(q, 40, 1e4), oracle.rope(k, 33, 1e4))
    b = np.dot(oracle.rope(q, 1007, 1e4), oracle.rope(k, 1000, 1e4))
    assert a == pytest.approx(b, rel=1e-4, abs=1e-4)


# ---------------------------------------------------------------- attention
def test_attention_single_key_returns_v_exactly():
    rng = np.random.default_rng(5)
    q = rng.standard_normal(128).astype(np.float32)
    K = rng.standard_normal((1, 128)).astype(np.float32)
    V = rng.standard_normal((1, 128)).astype(np.float32)
    assert np.array_equal(oracle.attend(q, K, V), V[0])


def test_attention_uniform_scores_give_mean_and_onehot_selects():
    rng = np.random.default_rng(6)
    K = rng.standard_normal((37, 64)).astype(np.float32)
    V = rng.standard_normal((37, 64)).astype(np.float32)
    np.testing.assert_allclose(oracle.attend(np.zeros(64, np.float32), K, V), V.mean(0),
                               rtol=1e-5, atol=1e-6)
    K2 = np.zeros((37, 64), np.float32)
    K2[11, 0] = 1.0
    q = np.zeros(64, np.float32)
    q[0] = 1e4  # score 1e4/8 for key 11, 0 for the others
    np.testing.assert_allclose(oracle.attend(q, K2, V), V[11], rtol=1e-6)


def test_attention_matches_torch_sdpa():
    rng = np.random.default_rng(7)
    q = rng.standard_normal(128).astype(np.float32)
    K = rng.standard_normal((300, 128)).astype(np.float32)
    V = rng.standard_normal((300, 128)).astype(np.float32)
    want = F.scaled_dot_product_attention(torch.from_numpy(q).double()[None, None, None],
                                          torch.from_numpy(K).double()[None, None],
                                          torch.from_numpy(V).double()[None, None])[0, 0, 0]
    np.testing.assert_allclose(oracle.attend(q, K, V), want.numpy(), rtol=1e-5, atol=1e-6)


def test_matvec_matches_float64_matmul():
    rng = np.random.default_rng(8)
    W = torch.from_numpy(rng.standard_normal((64, 2048)).astype(np.float32) * 0.02).to(torch.bfloat16)
    x = rng.standard_normal(2048).astype(np.float32)
    np.testing.assert_allclose(oracle.matvec(bits(W), x), W.double().numpy() @ x,
                               rtol=1e-4, atol=1e-5)


# ---------------------------------------------------------------- routing / argmax
def test_route_matches_brute_force_sort():
    rng = np.random.default_rng(9)
    for _ in range(20):
        lg = rng.standard_normal(64).astype(np.float32)
        ids, w = oracle.route(lg, 8)
        p = np.exp(lg.astype(np.float64) - lg.max())
        p /= p.sum()
        order = sorted(range(64), key=lambda e: (-p[e], e))[:8]
        assert ids.tolist() == order
        np.testing.assert_allclose(w, p[order] / p[order].sum(), rtol=1e-5)
        assert w.sum() == pytest.approx(1.0, abs=1e-6)


def test_route_ties_take_lower_index_and_uniform_gives_equal_weights():
    ids, w = oracle.route(np.zeros(64, np.float32), 8)
    assert ids.tolist() == list(range(8))
    np.testing.assert_allclose(w, 1 / 8, rtol=1e-6)
    ids, w = oracle.route(np.zeros(8, np.float32), 8)  # k = E: all experts, mean
    np.testing.assert_allclose(w, 1 / 8, rtol=1e-6)


def test_argmax_ties_lowest_index():
    v = np.array([0.5, 2.0, -1.0, 2.0, 2.0], np.float32)
    assert oracle.argmax(v) == 1
    assert oracle.argmax(np.zeros(10, np.float32)) == 0


# ---------------------------------------------------------------- whole model helpers
def _model(cfg, seed, gain_noise=0.0):
    W = synth.make_weights(cfg, seed, gain_noise=gain_noise)
    return W, oracle.OracleModel(cfg, W)


def _decode_sequence(om, cfg, tokens, num_pages=8, perm_seed=0, window=None):
    """Teacher-forced decode of one sequence through the paged cache; returns the
    logits of every step and the final pool."""
    T = len(tokens)
    rng = np.random.default_rng(perm_seed)
    pages = (T + cfg.page_size - 1) // cfg.page_size
    pt = synth.random_page_tables(rng, num_pages, [pages], max_pages=pages + 1)
    kv = np.zeros(synth.kv_pool_shape(cfg, num_pages), np.uint16)
    out = []
    for t in range(T):
        lg, _ = om.decode_step(kv, [tokens[t]], [t], pt, [t + 1], nthreads=2)
        out.append(lg[0])
    return np.stack(out), kv, pt


def _torch_reference_forward(cfg, W, tokens):
    """Full causal forward in float64 from torch library routines (rms_norm, sdpa
    with GQA and a causal/window mask, silu); RoPE as a complex rotation; the K/V
    the cache would hold rounded to BF16."""
    f = lambda t: t.double()  # noqa: E731
    T, hd = len(tokens), cfg.head_dim
    tok = torch.tensor(tokens)
    x = f(W["embed"])[tok]
    i = torch.arange(hd // 2, dtype=torch.float64)
    ang = torch.arange(T, dtype=torch.float64)[:, None] * cfg.rope_theta ** (-2.0 * i / hd)
    rot = torch.polar(torch.ones_like(ang), ang)
    rot = torch.complex(rot.real.float().double(), rot.imag.float().double())

    def rope(v):  # [T, H, hd]
        z = torch.complex(v[..., : hd // 2], v[..., hd // 2:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], -1)

    def bf(v):
        return v.float().to(torch.bfloat16).double()

    pos = torch.arange(T)
    for l, L in enumerate(W["layers"]):
        xn = F.rms_norm(x, (cfg.d_model,), f(L["attn_norm"]), cfg.rms_eps)
        q = rope((xn @ f(L["wq"]).T).view(T, cfg.n_q_heads, hd))
        k = bf(rope((xn @ f(L["wk"]).T).view(T, cfg.n_kv_heads, hd)))
        v = bf((xn @ f(L["wv"]).T).view(T, cfg.n_kv_heads, hd))
        mask = pos[None, :] <= pos[:, None]
        if cfg.sliding_window > 0 and cfg.layer_is_sliding()[l]:
            mask &= pos[None, :] > pos[:, None] - cfg.sliding_window
        o = F.scaled_dot_product_attention(q.transpose(0, 1), k.transpose(0, 1),
                                           v.transpose(0, 1), attn_mask=mask, enable_gqa=True)
        x = x + o.transpose(0, 1).reshape(T, -1) @ f(L["wo"]).T
        xn = F.rms_norm(x, (cfg.d_model,), f(L["mlp_norm"]), cfg.rms_eps)
        if cfg.is_moe:
            r = torch.softmax(xn @ f(L["router"]).T, -1)
            top = torch.topk(r, cfg.top_k, dim=-1, sorted=True)
            wts = top.values / top.values.sum(-1, keepdim=True)
            mo = torch.zeros_like(x)
            for t in range(T):
                for e, we in zip(top.indices[t].tolist(), wts[t].tolist()):
                    h = F.silu(xn[t] @ f(L["exp_gate"][e]).T) * (xn[t] @ f(L["exp_up"][e]).T)
                    mo[t] += we * (h @ f(L["exp_down"][e]).T)
            x = x + mo
        else:
            h = F.silu(xn @ f(L["w_gate"]).T) * (xn @ f(L["w_up"]).T)
            x = x + h @ f(L["w_down"]).T
    xn = F.rms_norm(x, (cfg.d_model,), f(W["final_norm"]), cfg.rms_eps)
    return (xn @ f(W["lm_head"]).T).numpy()


@pytest.fixture(scope="module")
def tiny_run():
    cfg = TINY
    W, om = _model(cfg, 0, gain_noise=0.02)
    rng = np.random.default_rng(0)
    tokens = synth.random_tokens(rng, cfg.vocab, 48).tolist()
    logits, kv, pt = _decode_sequence(om, cfg, tokens, num_pages=8, perm_seed=1)
    return cfg, W, om, tokens, logits, kv, pt


def test_cached_decode_equals_full_recompute(tiny_run):
    cfg, W, om, tokens, logits, _, _ = tiny_run
    full = om.forward_full(tokens, nthreads=2)
    np.testing.assert_allclose(logits, full, rtol=0, atol=1e-5)


def test_oracle_matches_float64_twin(tiny_run):
    cfg, W, om, tokens, logits, _, _ = tiny_run
    tw = Twin(cfg, W)
    cache = tw.new_cache()
    for t in (0, 1, 15, 16, 17, 31, 47):
        while cache[0]["k"].shape[0] < t:
            tw.step(cache, tokens[cache[0]["k"].shape[0]], cache[0]["k"].shape[0])
        np.testing.assert_allclose(logits[t], tw.step(cache, tokens[t], t), rtol=0, atol=1e-4)


def test_oracle_matches_torch_library_forward(tiny_run):
    cfg, W, om, tokens, logits, _, _ = tiny_run
    ref = _torch_reference_forward(cfg, W, tokens)
    np.testing.assert_allclose(logits, ref, rtol=0, atol=1e-4)


def test_norm_gains_are_used(tiny_run):
    cfg, W, om, tokens, logits, _, _ = tiny_run
    W1 = synth.make_weights(cfg, 0, gain_noise=0.0)
    lg1, _, _ = _decode_sequence(oracle.OracleModel(cfg, W1), cfg, tokens[:4], perm_seed=1)
    assert np.abs(lg1 - logits[:4]).max() > 1e-3


def test_paged_equals_contiguous_and_permutation_invariant(tiny_run):
    cfg, W, om, tokens, logits, _, _ = tiny_run
    T = 20
    # contiguous: pages 0,1 in order; permuted: a 16-page pool, two other permutations
    ref = None
    for num_pages, seed in ((2, None), (16, 5), (16, 9)):
        kv = np.zeros(synth.kv_pool_shape(cfg, num_pages), np.uint16)
        if seed is None:
            pt = np.array([[0, 1]], np.int32)
        else:
            pt = synth.random_page_tables(np.random.default_rng(seed), num_pages, [2], 2)
        out = [om.decode_step(kv, [tokens[t]], [t], pt, [t + 1], nthreads=2)[0][0]
               for t in range(T)]
        out = np.stack(out)
        if ref is None:
            ref = out
        assert np.array_equal(out, ref)
    assert np.array_equal(ref, logits[:T])


def test_kv_append_writes_exactly_one_slot_per_layer_head(tiny_run):
    cfg, W, om, tokens, _, _, _ = tiny_run
    num_pages = 6
    kv = np.full(synth.kv_pool_shape(cfg, num_pages), 0xABCD, np.uint16)
    pt = np.array([[4, 1, 3]], np.int32)
    pos = 21  # page index 1 -> physical page 1, slot 5
    before = kv.copy()
    om.decode_step(kv, [tokens[0]], [pos], pt, [pos + 1], nthreads=2)
    changed = np.argwhere(np.any(kv != before, axis=-1))
    want = {(l, 1, kvi, g, 5) for l in range(cfg.n_layers) for kvi in (0, 1)
            for g in range(cfg.n_kv_heads)}
    assert {tuple(c) for c in changed.tolist()} == want


def test_batch_rows_are_independent(tiny_run):
    cfg, W, om, tokens, _, _, _ = tiny_run
    rng = np.random.default_rng(11)
    num_pages = 24
    lens = [5, 37, 20]
    pt = synth.random_page_tables(rng, num_pages, [(n + 15) // 16 + 1 for n in lens], 4)
    kv = np.zeros(synth.kv_pool_shape(cfg, num_pages), np.uint16)
    kv[:] = synth.bf16_bits(torch.randn(kv.shape, generator=torch.Generator().manual_seed(3))
                            .to(torch.bfloat16))
    kv0 = kv.copy()
    toks = [7, 99, 4000]
    lg_b, nt_b = om.decode_step(kv, toks, lens, pt, [n + 1 for n in lens], nthreads=2)
    for b in range(3):
        kv1 = kv0.copy()
        lg1, nt1 = om.decode_step(kv1, toks[b:b + 1], lens[b:b + 1], pt[b:b + 1],
                                  [lens[b] + 1], nthreads=2)
        assert np.array_equal(lg1[0], lg_b[b]) and nt1[0] == nt_b[b]
    assert np.array_equal(nt_b, np.argmax(lg_b, axis=1))


def test_sliding_window_wider_than_context_is_full_attention(tiny_run):
    cfg, W, om, tokens, logits, _, _ = tiny_run
    cfg_w = cfg.with_(sliding_window=1000)
    om_w = oracle.OracleModel(cfg_w, W)
    lg, _, _ = _decode_sequence(om_w, cfg_w, tokens, perm_seed=1)
    assert np.array_equal(lg, logits)


def test_sliding_window_matches_twin_and_torch():
    cfg = TINY.with_(sliding_window=8)
    W, om = _model(cfg, 2)
    tokens = synth.random_tokens(np.random.default_rng(2), cfg.vocab, 30).tolist()
    lg, _, _ = _decode_sequence(om, cfg, tokens, perm_seed=3)
    np.testing.assert_allclose(lg, _torch_reference_forward(cfg, W, tokens), atol=1e-4, rtol=0)
    full = oracle.OracleModel(TINY, W)
    lg_full, _, _ = _decode_sequence(full, TINY, tokens, perm_seed=3)
    assert np.abs(lg_full[-1] - lg[-1]).max() > 1e-3  # the window changed something
    tw = Twin(cfg, W)
    cache = tw.new_cache()
    for t in range(30):
        out = tw.step(cache, tokens[t], t)
    np.testing.assert_allclose(lg[-1], out, atol=1e-4, rtol=0)


def test_moe_with_one_expert_is_dense_swiglu():
    dense_cfg = TINY.with_(vocab=512)
    W = synth.make_weights(dense_cfg, 4)
    moe_cfg = dense_cfg.with_(name="moe1", ffn_dim=0, n_experts=1, top_k=1,
                              expert_ffn_dim=dense_cfg.ffn_dim)
    Wm = {k: v for k, v in W.items() if k != "layers"}
    Wm["layers"] = []
    for L in W["layers"]:
        M = {k: v for k, v in L.items() if k not in ("w_gate", "w_up", "w_down")}
        M["router"] = synth.normal_bf16((1, dense_cfg.d_model), 0.02, 1)
        M["exp_gate"], M["exp_up"], M["exp_down"] = (L["w_gate"][None], L["w_up"][None],
                                                     L["w_down"][None])
        Wm["layers"].append(M)
    toks = [3, 50, 7, 400]
    a, _, _ = _decode_sequence(oracle.OracleModel(dense_cfg, W), dense_cfg, toks)
    b, _, _ = _decode_sequence(oracle.OracleModel(moe_cfg, Wm), moe_cfg, toks)
    assert np.array_equal(a, b)


def test_moe_matches_twin_and_torch():
    cfg = TINY_MOE
    W, om = _model(cfg, 5)
    tokens = synth.random_tokens(np.random.default_rng(5), cfg.vocab, 20).tolist()
    lg, _, _ = _decode_sequence(om, cfg, tokens, perm_seed=4)
    np.testing.assert_allclose(lg, _torch_reference_forward(cfg, W, tokens), atol=1e-4, rtol=0)
    tw = Twin(cfg, W)
    cache = tw.new_cache()
    for t in range(20):
        out = tw.step(cache, tokens[t], t)
    np.testing.assert_allclose(lg[-1], out, atol=1e-4, rtol=0)


def test_oracle_rejects_bad_inputs(tiny_run):
    cfg, W, om, tokens, _, _, _ = tiny_run
    kv = np.zeros(synth.kv_pool_shape(cfg, 4), np.uint16)
    pt = np.array([[0, 1]], np.int32)
    with pytest.raises(ValueError):
        om.decode_step(kv, [cfg.vocab], [0], pt, [1])       # token out of range
    with pytest.raises(ValueError):
        om.decode_step(kv, [1], [3], pt, [3])               # seq_len != pos + 1
    with pytest.raises(ValueError):
        om.decode_step(kv, [1], [3], np.array([[9, 1]], np.int32), [4])  # bad page id


# ---------------------------------------------------------------- temperature sampling
def test_philox4x32_10_known_answer_vectors():
    """Philox4x32-10 (Salmon et al., SC 2011): the published known-answer vectors."""
    assert oracle.philox4x32_10([0, 0, 0, 0], [0, 0]) == [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]
    f = 0xFFFFFFFF
    assert oracle.philox4x32_10([f, f, f, f], [f, f]) == [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]
    assert oracle.philox4x32_10([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344],
                                [0xA4093822, 0x299F31D0]) == [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]


def test_gumbel_draws_have_the_standard_gumbel_moments():
    """mean = Euler-Mascheroni constant, variance = pi^2 / 6."""
    g = np.array([oracle.gumbel(7, t, 3, 0) for t in range(40000)])
    assert abs(g.mean() - 0.5772156649) < 0.03
    assert abs(g.var() - np.pi ** 2 / 6) < 0.08


def test_gumbel_max_samples_follow_softmax_over_temperature():
    """argmax(z / T + Gumbel) is an exact draw from softmax(z / T): empirical frequencies
    over many counters match it."""
    z = np.array([1.0, 0.2, -0.5, 0.9, 0.0], np.float32)
    for T in (0.7, 1.5):
        n = 20000
        counts = np.zeros(len(z))
        for pos in range(n):
            counts[oracle.sample_gumbel(z, T, 11, pos, 2)] += 1
        p = np.exp(z / T) / np.exp(z / T).sum()
        assert np.abs(counts / n - p).max() < 0.015, (T, counts / n, p)


def test_gumbel_max_at_tiny_temperature_is_the_argmax():
    rng = np.random.default_rng(5)
    for _ in range(20):
        z = rng.normal(size=300).astype(np.float32)
        assert oracle.sample_gumbel(z, 1e-4, 3, 17, 0) == int(np.argmax(z))


def _gumbel_from_philox(seed: int, token: int, pos: int, row: int) -> float:
    """The noise as the sampling rule defines it, from the known-answer-pinned generator:
    counter (token, position, row, 0), key = seed (low word first), u from the top 24 bits
    of word 0 plus one half, g = -log(-log u), evaluated here in float64."""
    w0 = oracle.philox4x32_10([token, pos, row, 0], [seed & 0xFFFFFFFF, seed >> 32])[0]
    u = ((w0 >> 8) + 0.5) / 16777216.0
    return -np.log(-np.log(u))


def test_gumbel_scores_use_the_documented_counter_layout():
    """gumbel_scores(z)[i] = z_i / T + the noise of counter (i, pos, row, 0) under key =
    seed: a swapped position / row, a wrong token index or a wrong key word fails."""
    rng = np.random.default_rng(21)
    for seed, pos, row in ((0, 0, 0), (3, 17, 2), ((5 << 32) | 9, 8193, 7), (123456789, 40000, 1)):
        z = rng.normal(size=64).astype(np.float32)
        T = 0.8
        sc = oracle.gumbel_scores(z, T, seed, pos, row)
        ref = np.array([z[i] / T + _gumbel_from_philox(seed, i, pos, row) for i in range(len(z))])
        np.testing.assert_allclose(sc, ref, rtol=2e-6, atol=2e-5)
        if pos != row:  # the counter is not symmetric in (position, row)
            sw = oracle.gumbel_scores(z, T, seed, row, pos)
            assert np.abs(sw - sc).max() > 1e-3


def test_gumbel_scores_are_affine_in_the_logits_with_slope_one_over_t():
    """The scores of z minus those of zero logits are exactly z / T (the noise does not
    depend on the logits): a T * z or a dropped 1/T fails for T != 1."""
    rng = np.random.default_rng(22)
    z = rng.normal(size=500).astype(np.float32)
    for T in (0.25, 0.5, 2.0, 3.0):
        d = oracle.gumbel_scores(z, T, 7, 100, 3) - oracle.gumbel_scores(np.zeros_like(z), T, 7, 100, 3)
        np.testing.assert_allclose(d, z.astype(np.float64) / T, rtol=1e-5, atol=2e-6)


def test_sampled_token_is_the_argmax_of_the_scores():
    """sample_gumbel picks the largest score (lowest index on ties) over many counters."""
    rng = np.random.default_rng(23)
    for k in range(200):
        z = rng.normal(size=257).astype(np.float32)
        pos, row, seed = int(rng.integers(0, 1 << 20)), int(rng.integers(0, 8)), int(rng.integers(0, 1 << 62))
        sc = oracle.gumbel_scores(z, 0.9, seed, pos, row)
        assert oracle.sample_gumbel(z, 0.9, seed, pos, row) == int(np.argmax(sc))


# ---------------------------------------------------------------- limited top-k sampling
def test_topk_one_is_the_greedy_token():
    """k = 1 leaves one candidate, the largest logit (lowest index among equal ones),
    whatever the temperature and the draw."""
    rng = np.random.default_rng(31)
    for t in range(50):
        z = rng.normal(size=300).astype(np.float32)
        if t % 5 == 0:
            z[rng.integers(0, 300, size=3)] = z.max()  # tied maxima
        for T in (0.3, 1.0, 4.0):
            assert oracle.sample_gumbel_topk(z, T, 1, t, 1000 + t, 2) == int(np.argmax(z))


def test_topk_of_the_whole_vocabulary_is_the_unrestricted_draw():
    rng = np.random.default_rng(32)
    for t in range(50):
        z = rng.normal(size=257).astype(np.float32)
        for k in (0, 257, 300):
            assert oracle.sample_gumbel_topk(z, 0.9, k, 5, t, 1) == oracle.sample_gumbel(z, 0.9, 5, t, 1)


def test_topk_draws_stay_in_the_candidate_set():
    """The drawn token has fewer than k tokens ahead of it (larger logit, or equal logit
    and a lower index); ties at the boundary keep the lower indices."""
    rng = np.random.default_rng(33)
    for t in range(200):
        z = np.round(rng.normal(size=64), 1).astype(np.float32)  # many equal logits
        k = int(rng.integers(1, 20))
        i = oracle.sample_gumbel_topk(z, 1.3, k, 77, t, 0)
        ahead = int(np.sum((z > z[i]) | ((z == z[i]) & (np.arange(64) < i))))
        assert ahead < k, (k, i, ahead)


def test_topk_frequencies_are_the_renormalised_softmax():
    """Over many counters, draws restricted to the top k follow softmax(z / T) over those
    k tokens; the tied boundary token with the higher index is never drawn."""
    z = np.array([0.5, 2.0, 1.0, 1.0, -1.0, 1.5], np.float32)  # order: 1, 5, 2, 3, 0, 4
    k, T, n = 3, 0.8, 30000
    counts = np.zeros(len(z))
    for pos in range(n):
        counts[oracle.sample_gumbel_topk(z, T, k, 19, pos, 4)] += 1
    cand = [1, 5, 2]
    p = np.zeros(len(z))
    p[cand] = np.exp(z[cand] / T) / np.exp(z[cand] / T).sum()
    assert counts[3] == 0 and counts[0] == 0 and counts[4] == 0
    assert np.abs(counts / n - p).max() < 0.012, (counts / n, p)


# ---------------------------------------------------------------- K/V appends at 8B shapes
def _bf16_ulps_apart(a, b):
    """Distance in BF16 steps between arrays of BF16 values (sign-magnitude order)."""
    def key(x):
        u = (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.int64)
        return np.where(u & 0x8000, -(u & 0x7FFF), u & 0x7FFF)
    return np.abs(key(a) - key(b))


def test_oracle_appends_at_8b_shapes_match_the_twin_run_from_them():
    """The C oracle's K/V appends of one batch-8 step with the 8B decoder's shapes (d 4096,
    32/8 heads of 128, ffn 14336, vocabulary 128256; two layers) against the float64 twin
    run over the same pool and from the oracle's own appends of the earlier layer: every
    element within 1 BF16 ulp or 1/4096 of its row's RMS. Run from its own appends
    instead, the twin lands beyond that bar on dozens of second-layer elements of row 4
    (one of its first-layer roundings falls the other way, and the current token attends
    to its own K/V), which is why the GPU parity checks condition the twin the same way."""
    cfg = synth.DENSE_8B.with_(n_layers=2, max_positions=1024)
    B, npages = 8, 104
    W = synth.make_weights(cfg, 102, device="cpu")
    pool = torch.empty(synth.kv_pool_shape(cfg, npages), dtype=torch.bfloat16)
    synth.fill_normal_bf16_(pool, 8)
    start = bits(pool).copy()
    kv = start.copy()
    rng = np.random.default_rng(102)
    pt = synth.prefix_shared_page_tables(rng, npages, B, 24, 4, max_pages=28)
    pos = (24 * 16 + rng.integers(0, 48, size=B)).astype(np.int32)
    toks = synth.random_tokens(rng, cfg.vocab, B)
    oracle.OracleModel(cfg, W).decode_step(kv, toks, pos, pt, pos + 1)
    # the logits are not compared: embedding and LM head cut to the rows used
    tw = Twin(cfg, dict(W, embed=W["embed"][:1], lm_head=W["lm_head"][:1]))
    misses = {}
    for conditioned in (True, False):
        for b in range(B):
            p = int(pos[b])
            keys = np.arange(p)
            pages = pt[b][keys // 16]
            cache = [{"k": bf16_bits_to_f64(start[l, pages, 0, :, keys % 16]),
                      "v": bf16_bits_to_f64(start[l, pages, 1, :, keys % 16])} for l in range(2)]
            page, slot = pt[b][p // 16], p % 16
            theirs = [(bf16_bits_to_f64(kv[l, page, 0, :, slot]), bf16_bits_to_f64(kv[l, page, 1, :, slot]))
                      for l in range(2)]
            tw.embed = bf16_bits_to_f64(bits(W["embed"][int(toks[b]):int(toks[b]) + 1]))
            tw.step(cache, 0, p, appended=theirs if conditioned else None)
            for l in range(2):
                for which in (0, 1):
                    o = theirs[l][which]
                    t = tw.own_appends[l][which]
                    rms = np.sqrt(np.mean(t ** 2, axis=-1, keepdims=True))
                    ok = (np.abs(o - t) <= rms * 2.0 ** -12) | (_bf16_ulps_apart(o, t) <= 1)
                    misses[(conditioned, b, l)] = misses.get((conditioned, b, l), 0) + int((~ok).sum())
    assert sum(n for (c, _, _), n in misses.items() if c) == 0, misses
    assert misses[(False, 4, 0)] == 0 and misses[(False, 4, 1)] >= 20, misses

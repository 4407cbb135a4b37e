"""Shared helpers for the GPU parity tests: run the CUDA path (through the C ABI) and
the CPU oracle on the same seeded inputs and compare them.

Parity bar (stated by the task's target): logits max-abs error <= 3e-2 (fp32
accumulation), greedy tokens equal wherever the oracle's top-2 margin exceeds 0.1,
KV slot writes at exactly the oracle's addresses, and every written value within 1
BF16 ulp of the oracle's (the two sides round K/V computed with different fp32
summation orders; elements much smaller than their row's scale are held to 1/4096 of
the row RMS instead, see check_kv).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
from oracle.twin import Twin, bf16_bits_to_f64
import persistent_megakernel_05_b300 as mk

LOGIT_ATOL = 3e-2
MARGIN = 0.1


class Pair:
    """A model on the GPU (DecodeModel) and the same model in the oracle, each with its
    own copy of one seeded KV pool."""

    def __init__(self, cfg, seed: int, num_pages: int, kv_seed: int = 1, gain_noise: float = 0.0,
                 weights=None):
        self.cfg = cfg
        self.W = weights if weights is not None else synth.make_weights(
            cfg, seed, device="cuda", gain_noise=gain_noise)
        self.gpu = mk.DecodeModel(cfg, self.W, num_pages)
        kv = self.gpu.kv()
        synth.fill_normal_bf16_(kv, kv_seed)
        torch.cuda.synchronize()
        self.orc = oracle.OracleModel(cfg, self.W)
        self.kv_host = synth.bf16_bits(kv).copy()
        self.kv_start = self.kv_host.copy()
        self.num_pages = num_pages
        # kv_start is the pool both sides start the next step from (true until a step
        # appends without check_kv_and_share handing the GPU's pool back)
        self.start_is_common = True
        self.last_inputs = None  # (tokens, positions, page_table, start_is_common) of the last step
        self._twin = None

    def step(self, tokens, positions, page_table, with_logits=True):
        B = len(tokens)
        dev = "cuda"
        t = torch.tensor(np.asarray(tokens, np.int32), device=dev)
        p = torch.tensor(np.asarray(positions, np.int32), device=dev)
        pt = torch.tensor(np.asarray(page_table, np.int32), device=dev)
        sl = p + 1
        nxt = torch.full((B,), -1, dtype=torch.int32, device=dev)
        lg = torch.full((B, self.cfg.vocab), float("nan"), device=dev) if with_logits else None
        self.last_inputs = (np.asarray(tokens, np.int32).copy(), np.asarray(positions, np.int32).copy(),
                            np.asarray(page_table, np.int32).copy(), self.start_is_common)
        self.start_is_common = False
        self.gpu.step(t, p, pt, sl, nxt, lg)
        code, task = self.gpu.status()
        assert code == mk.MK_OK, (mk.status_string(code), task)
        o_lg, o_nx = self.orc.decode_step(self.kv_host, np.asarray(tokens), np.asarray(positions),
                                          np.asarray(page_table), np.asarray(positions) + 1)
        return (lg.cpu().numpy() if lg is not None else None), nxt.cpu().numpy(), o_lg, o_nx

    def twin_appends(self, b: int, pool: np.ndarray) -> np.ndarray:
        """The K/V rows that batch row ``b`` of the last step appends per the float64 twin,
        run over the common pre-step pool and from ``pool``'s own appends of this step
        (each layer's current-token K/V as ``pool`` holds them feed the later layers):
        [layer, K/V, kv head, head_dim], BF16 values."""
        cfg = self.cfg
        tokens, positions, page_table, _ = self.last_inputs
        if self._twin is None:
            # the logits are not needed: the twin's embedding and LM head are cut to one row
            ws = dict(self.W)
            ws["embed"] = self.W["embed"][:1]
            ws["lm_head"] = self.W["lm_head"][:1]
            self._twin = Twin(cfg, ws)
        tw = self._twin
        tok, p = int(tokens[b]), int(positions[b])
        e = self.W["embed"][tok:tok + 1]
        tw.embed = bf16_bits_to_f64(e if isinstance(e, np.ndarray) else synth.bf16_bits(e))
        keys = np.arange(p)
        pages = page_table[b][keys // cfg.page_size]
        mapped = (pages >= 0)[:, None, None]  # keys a sliding window dropped may be unmapped
        cache = []
        for l in range(cfg.n_layers):
            hist = [np.where(mapped, bf16_bits_to_f64(self.kv_start[l, np.maximum(pages, 0), kv, :,
                                                                    keys % cfg.page_size]), 0.0)
                    for kv in (0, 1)]
            cache.append({"k": hist[0], "v": hist[1]})
        page, slot = page_table[b][p // cfg.page_size], p % cfg.page_size
        theirs = [(bf16_bits_to_f64(pool[l, page, 0, :, slot]), bf16_bits_to_f64(pool[l, page, 1, :, slot]))
                  for l in range(cfg.n_layers)]
        tw.step(cache, 0, p, appended=theirs)
        return np.stack([np.stack(kv) for kv in tw.own_appends])

    def gpu_kv_bits(self):
        torch.cuda.synchronize()
        return synth.bf16_bits(self.gpu.kv())

    def close(self):
        self.gpu.close()


def check_logits(g_lg, g_nx, o_lg, o_nx, atol=LOGIT_ATOL, what=""):
    assert np.isfinite(g_lg).all(), f"{what}: non-finite GPU logits"
    err = np.abs(g_lg - o_lg).max()
    assert err <= atol, f"{what}: logits max-abs error {err:.4g} > {atol}"
    for b in range(o_lg.shape[0]):
        top2 = np.partition(o_lg[b], -2)[-2:]
        if top2[1] - top2[0] > MARGIN:
            assert g_nx[b] == o_nx[b], f"{what}: row {b} token {g_nx[b]} != oracle {o_nx[b]}"
        # the GPU token is always the argmax of the GPU's own logits
        assert g_lg[b, g_nx[b]] == g_lg[b].max()
        assert g_nx[b] == int(np.argmax(g_lg[b]))
    return err


def bf16_ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """|a - b| in units of BF16 ulps for BF16 bit patterns (monotone integer mapping)."""
    def key(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x & 0x7FFF)
    return np.abs(key(a) - key(b))


# Every written K/V element must be within 1 BF16 ulp of the oracle's element, or within
# 1/4096 of its row's RMS (a sixteenth of one ulp at the row's scale). The two sides
# compute the same fp32 projection in different summation orders (and, past the first
# layer, from fp32 inputs that differ in the last bits) and round it to BF16 once; that
# fp32 difference is far below a BF16 ulp of any element of ordinary size, so those
# round to the same or the neighbouring BF16 value. Only elements much smaller than
# their row's scale have an ulp finer than the fp32 difference; they are held to the
# absolute bound instead. KV_STATS collects the histogram of every check for the report.
#
# Past the first layer a second effect appears: the current token attends to its own key
# and value, so where one side's BF16 rounding of an early layer's append falls the other
# way (an allowed 1-ulp difference) every later layer starts from a slightly different
# input. With the 8B shapes that moves some second-layer K/V elements by ~1e-4 of the
# row RMS, beyond the bar, on either side. So where the GPU misses the bar against the
# oracle and both sides started the step from the same pool, the float64 twin decides,
# run from the GPU's own earlier-layer appends: the element passes if the GPU meets the
# same bar against the twin's value.
SMALL = 2.0 ** -12
KV_STATS = {"elements": 0, "ulp0": 0, "ulp1": 0, "small": 0, "twin": 0}


def _f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def check_kv(pair: Pair):
    """The GPU wrote exactly the slots the oracle wrote (bit-exact addresses: every other
    byte of the pool is unchanged), and every written element is within 1 BF16 ulp of the
    oracle's, or within 1/4096 of its row's RMS. Returns the number of written rows."""
    g = pair.gpu_kv_bits()
    o = pair.kv_host
    s = pair.kv_start
    g_changed = np.any(g != s, axis=-1)
    o_changed = np.any(o != s, axis=-1)
    # a slot may be written with an identical value by chance only with vanishing odds
    assert np.array_equal(g_changed, o_changed), "KV slot writes differ from the oracle's"
    assert np.array_equal(g[~g_changed], s[~g_changed])
    gb, ob = g[g_changed], o[g_changed]
    if gb.size:
        ulp = bf16_ulp_diff(gb, ob)
        gv, ov = _f32(gb).astype(np.float64), _f32(ob).astype(np.float64)
        rms = np.sqrt(np.mean(ov ** 2, axis=-1, keepdims=True))
        small = np.abs(gv - ov) <= SMALL * rms
        bad = (ulp > 1) & ~small
        rows = np.argwhere(g_changed)  # (layer, page, K/V, head, slot) of each written row
        last = getattr(pair, "last_inputs", None)
        if bad.any() and last is not None and last[3]:
            twin_ok = _twin_arbitration(pair, rows, g, gb, bad)
            KV_STATS["twin"] += int(twin_ok.sum())
            bad &= ~twin_ok
        if bad.any():
            where = [f"(layer, page, kv, head, slot) {tuple(int(v) for v in rows[r])} dim {int(d)}: "
                     f"gpu {gv[r, d]:.6g} oracle {ov[r, d]:.6g} row rms {rms[r, 0]:.3g}"
                     for r, d in np.argwhere(bad)[:6]]
            raise AssertionError(f"{int(bad.sum())} K/V elements differ by more than 1 BF16 ulp and more "
                                 f"than 1/4096 of their row's RMS (max {int(ulp[bad].max())} ulp); "
                                 + "; ".join(where))
        KV_STATS["elements"] += int(ulp.size)
        KV_STATS["ulp0"] += int((ulp == 0).sum())
        KV_STATS["ulp1"] += int((ulp == 1).sum())
        KV_STATS["small"] += int(((ulp > 1) & small).sum())
    return int(g_changed.sum())


def _twin_arbitration(pair: Pair, rows: np.ndarray, g: np.ndarray, gb: np.ndarray,
                      bad: np.ndarray) -> np.ndarray:
    """For the written rows holding elements in ``bad``: True where the GPU's element is
    within 1 BF16 ulp, or 1/4096 of the row RMS, of the float64 twin's value (the twin run
    from the GPU's own appends of the earlier layers, ``g`` being the GPU's pool)."""
    cfg = pair.cfg
    _, positions, page_table, _ = pair.last_inputs
    ok = np.zeros_like(bad)
    twins = {}
    for r in np.unique(np.argwhere(bad)[:, 0]):
        l, page, kv, head, slot = (int(v) for v in rows[r])
        b = [i for i in range(len(positions))
             if page_table[i][positions[i] // cfg.page_size] == page
             and positions[i] % cfg.page_size == slot]
        if len(b) != 1:
            continue
        if b[0] not in twins:
            twins[b[0]] = pair.twin_appends(b[0], g)
        tv = twins[b[0]][l, kv, head]
        tbits = (tv.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        trms = np.sqrt(np.mean(tv ** 2))
        gv = _f32(gb[r]).astype(np.float64)
        ok[r] = bad[r] & ((bf16_ulp_diff(gb[r], tbits) <= 1) | (np.abs(gv - tv) <= SMALL * trms))
    return ok


def check_kv_and_share(pair) -> int:
    """check_kv, then hand the GPU's pool to the oracle as the new common history (and as
    the new starting state): the next step is compared from identical K/V on both sides.
    Long runs use it, since each side otherwise attends over its own rounding of every
    earlier append and the two histories drift apart step by step."""
    n = check_kv(pair)
    g = pair.gpu_kv_bits()
    pair.kv_host[...] = g
    pair.kv_start[...] = g
    pair.start_is_common = True
    return n


def kv_stats_line() -> str:
    n = max(KV_STATS["elements"], 1)
    return (f"K/V elements checked {KV_STATS['elements']}: identical {KV_STATS['ulp0'] / n:.4%}, "
            f"1 ulp apart {KV_STATS['ulp1'] / n:.4%}, more than 1 ulp apart but within 1/4096 of "
            f"the row RMS {KV_STATS['small'] / n:.4%}; further than that from the fp32 oracle but "
            f"within the bar of the float64 twin: {KV_STATS['twin']}")

"""Shared helpers for the GPU parity tests: run the CUDA path (through the C ABI) and
the CPU oracle on the same seeded inputs and compare them.

Parity bar (stated by the task's target): logits max-abs error <= 3e-2 (fp32
accumulation), greedy tokens equal wherever the oracle's top-2 margin exceeds 0.1,
KV slot writes at exactly the oracle's addresses (values within 1 BF16 ulp, since
the two sides round K/V computed with different fp32 summation orders).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
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

    def step(self, tokens, positions, page_table, with_logits=True):
        B = len(tokens)
        dev = "cuda"
        t = torch.tensor(np.asarray(tokens, np.int32), device=dev)
        p = torch.tensor(np.asarray(positions, np.int32), device=dev)
        pt = torch.tensor(np.asarray(page_table, np.int32), device=dev)
        sl = p + 1
        nxt = torch.full((B,), -1, dtype=torch.int32, device=dev)
        lg = torch.full((B, self.cfg.vocab), float("nan"), device=dev) if with_logits else None
        self.gpu.step(t, p, pt, sl, nxt, lg)
        code, task = self.gpu.status()
        assert code == mk.MK_OK, (mk.status_string(code), task)
        o_lg, o_nx = self.orc.decode_step(self.kv_host, np.asarray(tokens), np.asarray(positions),
                                          np.asarray(page_table), np.asarray(positions) + 1)
        return (lg.cpu().numpy() if lg is not None else None), nxt.cpu().numpy(), o_lg, o_nx

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


KV_REL = 2e-2


def _f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def check_kv(pair: Pair):
    """The GPU wrote exactly the slots the oracle wrote (bit-exact addresses: every other
    byte of the pool is unchanged), and each written row agrees with the oracle's row
    to KV_REL of the row's largest magnitude (the rows are fp32 projections computed in
    a different summation order, then rounded to BF16)."""
    g = pair.gpu_kv_bits()
    o = pair.kv_host
    s = pair.kv_start
    g_changed = np.any(g != s, axis=-1)
    o_changed = np.any(o != s, axis=-1)
    # a slot may be written with an identical value by chance only with vanishing odds
    assert np.array_equal(g_changed, o_changed), "KV slot writes differ from the oracle's"
    assert np.array_equal(g[~g_changed], s[~g_changed])
    gv, ov = _f32(g[g_changed]), _f32(o[g_changed])
    scale = np.abs(ov).max(axis=-1, keepdims=True)
    err = (np.abs(gv - ov) / np.maximum(scale, 1e-6)).max() if gv.size else 0.0
    assert err <= KV_REL, f"KV rows differ by {err:.3g} of their scale"
    return int(g_changed.sum())

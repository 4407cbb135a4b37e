"""Float64 NumPy twin of the CPU oracle (TEST INFRASTRUCTURE ONLY).

A second, separately written implementation of the same decode step, used to pin
the C oracle: it keeps the KV cache as contiguous per-sequence arrays (no pages),
does every product and sum in float64 with NumPy's matmul, and shares no code with
oracle.c. The model is the plainest pre-norm reading of the "Cohere Megakernel"
page (section "Megakernel ne demek": the whole decode step of an LM) with the
limits listed in its section "Sinirlar acikca yazilmis" (BF16 weights, batch 1..8,
sliding window, greedy sampling).

The only values it rounds are the cached K and V rows, which the cache stores as
BF16 (the fp32 value rounded to nearest-even), exactly as the pages' BF16-only
contract implies.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    u = (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16)
    return u.view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """float64 -> float32 -> nearest-even BF16, returned as float64 values."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) & 0xFFFF
    nan = np.isnan(f)
    r = np.where(nan, (u >> 16) | 0x40, r).astype(np.uint32)
    return (r << 16).view(np.float32).astype(np.float64)


class Twin:
    def __init__(self, cfg, weights: dict):
        from synth import bf16_bits
        conv = lambda t: bf16_bits_to_f64(t if isinstance(t, np.ndarray) else bf16_bits(t))  # noqa
        self.cfg = cfg
        self.embed = conv(weights["embed"])
        self.final_norm = conv(weights["final_norm"])
        self.lm_head = conv(weights["lm_head"])
        self.layers = [{k: conv(v) for k, v in L.items()} for L in weights["layers"]]
        hd = cfg.head_dim
        half = hd // 2
        i = np.arange(half, dtype=np.float64)
        self.inv_freq = float(cfg.rope_theta) ** (-2.0 * i / hd)

    # --- pieces ---
    def rmsnorm(self, x, g):
        return x / np.sqrt(np.mean(x * x) + self.cfg.rms_eps) * g

    def rope(self, v, pos):
        """v [..., hd]; rotate-half with complex numbers z_i = v_i + i v_{i+hd/2}."""
        half = v.shape[-1] // 2
        ang = pos * self.inv_freq
        # the oracle rounds cos/sin to fp32; the angle rounding is part of the definition
        c = np.cos(ang).astype(np.float32).astype(np.float64)
        s = np.sin(ang).astype(np.float32).astype(np.float64)
        z = v[..., :half] + 1j * v[..., half:]
        z = z * (c + 1j * s)
        return np.concatenate([z.real, z.imag], axis=-1)

    def mlp(self, l, xn):
        L = self.layers[l]
        silu = lambda z: z / (1.0 + np.exp(-z))  # noqa: E731
        if not self.cfg.is_moe:
            return L["w_down"] @ (silu(L["w_gate"] @ xn) * (L["w_up"] @ xn))
        r = L["router"] @ xn
        p = np.exp(r - r.max())
        p = p / p.sum()
        sel = np.argsort(-p, kind="stable")[: self.cfg.top_k]
        w = p[sel] / p[sel].sum()
        out = np.zeros_like(xn)
        for e, we in sorted(zip(sel.tolist(), w.tolist())):
            h = silu(L["exp_gate"][e] @ xn) * (L["exp_up"][e] @ xn)
            out = out + we * (L["exp_down"][e] @ h)
        return out

    # --- one sequence, one step ---
    def new_cache(self):
        cfg = self.cfg
        return [{"k": np.zeros((0, cfg.n_kv_heads, cfg.head_dim)),
                 "v": np.zeros((0, cfg.n_kv_heads, cfg.head_dim))} for _ in range(cfg.n_layers)]

    def step(self, cache, token: int, pos: int, appended=None):
        """Appends the step's K/V rows to ``cache`` (which must hold exactly ``pos`` rows)
        and returns the logits (float64 [vocab]).

        The step's own BF16-rounded K/V rows are also kept in ``self.own_appends`` (one
        (K, V) pair of [kv heads, head_dim] arrays per layer). ``appended``, if given,
        holds one such pair per layer from another implementation of the same step: the
        cache then stores those rows instead of the step's own, so every later layer
        runs from that implementation's rounding of the current token's K/V (the current
        token attends to its own key and value, so one BF16 rounding that falls the
        other way in an early layer shifts every later layer's input)."""
        cfg = self.cfg
        hd, Hq, Hkv = cfg.head_dim, cfg.n_q_heads, cfg.n_kv_heads
        G = Hq // Hkv
        x = self.embed[token].copy()
        self.own_appends = []
        for l, L in enumerate(self.layers):
            c = cache[l]
            assert c["k"].shape[0] == pos
            xn = self.rmsnorm(x, L["attn_norm"])
            q = self.rope((L["wq"] @ xn).reshape(Hq, hd), pos)
            k = self.rope((L["wk"] @ xn).reshape(Hkv, hd), pos)
            v = (L["wv"] @ xn).reshape(Hkv, hd)
            kr, vr = round_to_bf16(k), round_to_bf16(v)
            self.own_appends.append((kr, vr))
            if appended is not None:
                kr, vr = appended[l]
            c["k"] = np.concatenate([c["k"], kr[None]], 0)
            c["v"] = np.concatenate([c["v"], vr[None]], 0)
            slides = cfg.sliding_window > 0 and cfg.layer_is_sliding()[l]
            lo = max(0, pos - cfg.sliding_window + 1) if slides else 0
            o = np.empty((Hq, hd))
            for h in range(Hq):
                K = c["k"][lo:pos + 1, h // G]
                V = c["v"][lo:pos + 1, h // G]
                s = K @ q[h] / np.sqrt(hd)
                p = np.exp(s - s.max())
                o[h] = (p / p.sum()) @ V
            x = x + L["wo"] @ o.reshape(-1)
            x = x + self.mlp(l, self.rmsnorm(x, L["mlp_norm"]))
        return self.lm_head @ self.rmsnorm(x, self.final_norm)

"""CPU oracle for the paged-KV decode step.

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and bench.py's CPU
baseline / reference arm may import this package. The product package never does.

Two independent implementations live here:
  * ``liboracle.so`` (oracle.c): plain C, fp32 arithmetic in natural index order,
    the reference the CUDA path is compared against;
  * ``twin`` (twin.py): a float64 NumPy restatement written separately, used only to
    pin the C oracle.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liboracle.so")
SRC_PATH = os.path.join(HERE, "oracle.c")
CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-Wall"]

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc)."""
    if (not force and os.path.exists(LIB_PATH)
            and os.path.getmtime(LIB_PATH) >= os.path.getmtime(SRC_PATH)):
        return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, SRC_PATH, "-lm"])
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


_P = ctypes.POINTER
_u16p = _P(ctypes.c_uint16)
_f32p = _P(ctypes.c_float)
_i32p = _P(ctypes.c_int32)


class _Model(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32), ("d_model", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("ffn_dim", ctypes.c_int32),
        ("vocab", ctypes.c_int32), ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
        ("expert_ffn_dim", ctypes.c_int32), ("rms_eps", ctypes.c_float),
        ("rope_theta", ctypes.c_float), ("sliding_window", ctypes.c_int32),
        ("layer_is_sliding", _P(ctypes.c_uint8)), ("page_size", ctypes.c_int32),
        ("embed", _u16p), ("final_norm", _u16p), ("lm_head", _u16p),
        ("attn_norm", _P(_u16p)), ("wq", _P(_u16p)), ("wk", _P(_u16p)), ("wv", _P(_u16p)),
        ("wo", _P(_u16p)), ("mlp_norm", _P(_u16p)), ("w_gate", _P(_u16p)), ("w_up", _P(_u16p)),
        ("w_down", _P(_u16p)), ("router", _P(_u16p)), ("exp_gate", _P(_u16p)),
        ("exp_up", _P(_u16p)), ("exp_down", _P(_u16p)),
    ]


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB_PATH)
        L.or_decode_step.restype = ctypes.c_int
        L.or_decode_step.argtypes = [_P(_Model), _u16p, ctypes.c_int32, _i32p, _i32p, _i32p,
                                     ctypes.c_int32, _i32p, ctypes.c_int32, _f32p, _i32p,
                                     ctypes.c_int32]
        L.or_forward_full.restype = ctypes.c_int
        L.or_forward_full.argtypes = [_P(_Model), _i32p, ctypes.c_int32, _f32p, ctypes.c_int32]
        L.or_rmsnorm.argtypes = [_f32p, _u16p, ctypes.c_int32, ctypes.c_float, _f32p]
        L.or_rope.argtypes = [_f32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_float]
        L.or_attend.argtypes = [_f32p, _f32p, _f32p, ctypes.c_int32, ctypes.c_int32, _f32p]
        L.or_route.argtypes = [_f32p, ctypes.c_int32, ctypes.c_int32, _i32p, _f32p]
        L.or_argmax.restype = ctypes.c_int32
        L.or_argmax.argtypes = [_f32p, ctypes.c_int32]
        L.or_philox4x32_10.argtypes = [_P(ctypes.c_uint32), _P(ctypes.c_uint32), _P(ctypes.c_uint32)]
        L.or_gumbel.restype = ctypes.c_float
        L.or_gumbel.argtypes = [ctypes.c_uint64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]
        L.or_gumbel_scores.argtypes = [_f32p, ctypes.c_int32, ctypes.c_float, ctypes.c_uint64,
                                       ctypes.c_int32, ctypes.c_int32, _f32p]
        L.or_sample_gumbel_topk.restype = ctypes.c_int32
        L.or_sample_gumbel_topk.argtypes = [_f32p, ctypes.c_int32, ctypes.c_float, ctypes.c_int32,
                                            ctypes.c_uint64, ctypes.c_int32, ctypes.c_int32]
        L.or_sample_gumbel.restype = ctypes.c_int32
        L.or_sample_gumbel.argtypes = [_f32p, ctypes.c_int32, ctypes.c_float, ctypes.c_uint64,
                                       ctypes.c_int32, ctypes.c_int32]
        L.or_matvec.argtypes = [_u16p, _f32p, ctypes.c_int32, ctypes.c_int32, _f32p]
        L.or_f32_to_bf16.restype = ctypes.c_uint16
        L.or_f32_to_bf16.argtypes = [ctypes.c_float]
        L.or_bf16_to_f32.restype = ctypes.c_float
        L.or_bf16_to_f32.argtypes = [ctypes.c_uint16]
        _lib = L
    return _lib


def _ptr(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


class OracleModel:
    """Holds host copies (uint16 BF16 bits) of a model's weights and the C descriptor.

    ``weights`` is the dict produced by ``synth.make_weights`` (torch BF16 tensors on
    any device) or an equivalent dict of numpy uint16 arrays.
    """

    def __init__(self, cfg, weights: dict):
        from synth import bf16_bits  # seeded-input helper; holds no decode arithmetic
        self.cfg = cfg
        conv = lambda t: _c(t if isinstance(t, np.ndarray) else bf16_bits(t), np.uint16)  # noqa
        self._keep = []
        self.embed = conv(weights["embed"])
        self.final_norm = conv(weights["final_norm"])
        self.lm_head = conv(weights["lm_head"])
        names = ["attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down",
                 "router", "exp_gate", "exp_up", "exp_down"]
        self.layers = []
        arrays = {n: [] for n in names}
        for L in weights["layers"]:
            hostL = {}
            for n in names:
                if n in L:
                    hostL[n] = conv(L[n])
                    arrays[n].append(_ptr(hostL[n], _u16p))
                else:
                    arrays[n].append(_u16p())
            self.layers.append(hostL)
        self.sliding = _c(cfg.layer_is_sliding(), np.uint8)
        m = _Model()
        m.n_layers, m.d_model, m.n_q_heads = cfg.n_layers, cfg.d_model, cfg.n_q_heads
        m.n_kv_heads, m.head_dim, m.ffn_dim, m.vocab = (cfg.n_kv_heads, cfg.head_dim,
                                                        cfg.ffn_dim, cfg.vocab)
        m.n_experts, m.top_k, m.expert_ffn_dim = cfg.n_experts, cfg.top_k, cfg.expert_ffn_dim
        m.rms_eps, m.rope_theta = cfg.rms_eps, cfg.rope_theta
        m.sliding_window = cfg.sliding_window
        m.layer_is_sliding = _ptr(self.sliding, _P(ctypes.c_uint8))
        m.page_size = cfg.page_size
        m.embed = _ptr(self.embed, _u16p)
        m.final_norm = _ptr(self.final_norm, _u16p)
        m.lm_head = _ptr(self.lm_head, _u16p)
        for n in names:
            arr = (_u16p * cfg.n_layers)(*arrays[n])
            self._keep.append(arr)
            setattr(m, n, ctypes.cast(arr, _P(_u16p)))
        self.m = m

    def decode_step(self, kv: np.ndarray, tokens, positions, page_table, seq_lens,
                    nthreads: Optional[int] = None, temperature: float = 0.0, seed: int = 0,
                    top_k: int = 0):
        """One decode step; appends into ``kv`` (uint16, pool layout) in place.
        Returns (logits [B, vocab] float32, next_tokens [B] int32). temperature > 0
        samples the next tokens from softmax(logits / T) (Gumbel-max, Philox draws keyed
        by ``seed``, counter (token, position, row)), restricted to the ``top_k`` largest
        logits when top_k > 0; else greedy."""
        cfg = self.cfg
        assert kv.dtype == np.uint16 and kv.flags.c_contiguous
        num_pages = kv.shape[1]
        tokens = _c(tokens, np.int32)
        positions = _c(positions, np.int32)
        seq_lens = _c(seq_lens, np.int32)
        page_table = _c(page_table, np.int32)
        B = tokens.shape[0]
        logits = np.empty((B, cfg.vocab), np.float32)
        nxt = np.empty(B, np.int32)
        rc = lib().or_decode_step(ctypes.byref(self.m), _ptr(kv, _u16p), num_pages,
                                  _ptr(tokens, _i32p), _ptr(positions, _i32p),
                                  _ptr(page_table, _i32p), page_table.shape[1],
                                  _ptr(seq_lens, _i32p), B, _ptr(logits, _f32p),
                                  _ptr(nxt, _i32p), nthreads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle decode_step returned {rc}")
        if temperature > 0.0:  # Gumbel-max sampling from softmax(logits / T), optionally top-k
            for b in range(B):
                nxt[b] = sample_gumbel_topk(logits[b], temperature, top_k, seed, int(positions[b]), b)
        return logits, nxt

    def forward_full(self, tokens, nthreads: Optional[int] = None) -> np.ndarray:
        """Logits at every position of ``tokens`` from a full causal recompute (no cache)."""
        tokens = _c(tokens, np.int32)
        T = tokens.shape[0]
        logits = np.empty((T, self.cfg.vocab), np.float32)
        rc = lib().or_forward_full(ctypes.byref(self.m), _ptr(tokens, _i32p), T,
                                   _ptr(logits, _f32p), nthreads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle forward_full returned {rc}")
        return logits


# ---- thin wrappers over the exported building blocks (for the unit pins) ----

def rmsnorm(x, g_bits, eps):
    x = _c(x, np.float32)
    g = _c(g_bits, np.uint16)
    out = np.empty_like(x)
    lib().or_rmsnorm(_ptr(x, _f32p), _ptr(g, _u16p), x.size, eps, _ptr(out, _f32p))
    return out


def rope(v, pos, theta):
    v = _c(v, np.float32).copy()
    lib().or_rope(_ptr(v, _f32p), v.size, int(pos), float(theta))
    return v


def attend(q, K, V):
    q = _c(q, np.float32)
    K = _c(K, np.float32)
    V = _c(V, np.float32)
    out = np.empty(q.shape[0], np.float32)
    lib().or_attend(_ptr(q, _f32p), _ptr(K, _f32p), _ptr(V, _f32p), K.shape[0], q.shape[0],
                    _ptr(out, _f32p))
    return out


def route(logits, k):
    logits = _c(logits, np.float32)
    ids = np.empty(k, np.int32)
    w = np.empty(k, np.float32)
    lib().or_route(_ptr(logits, _f32p), logits.size, k, _ptr(ids, _i32p), _ptr(w, _f32p))
    return ids, w


def argmax(v):
    v = _c(v, np.float32)
    return int(lib().or_argmax(_ptr(v, _f32p), v.size))


def matvec(W_bits, x):
    W = _c(W_bits, np.uint16)
    x = _c(x, np.float32)
    y = np.empty(W.shape[0], np.float32)
    lib().or_matvec(_ptr(W, _u16p), _ptr(x, _f32p), W.shape[0], W.shape[1], _ptr(y, _f32p))
    return y


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Vectorised call of the oracle's RNE rounding (used only in tests)."""
    x = _c(x, np.float32).ravel()
    f = lib().or_f32_to_bf16
    return np.array([f(float(v)) for v in x], np.uint16)


def philox4x32_10(ctr, key):
    """Philox4x32-10 block: four 32-bit counter words, two key words -> four words."""
    c = (ctypes.c_uint32 * 4)(*[int(x) & 0xFFFFFFFF for x in ctr])
    k = (ctypes.c_uint32 * 2)(*[int(x) & 0xFFFFFFFF for x in key])
    o = (ctypes.c_uint32 * 4)()
    lib().or_philox4x32_10(c, k, o)
    return [int(x) for x in o]


def gumbel(seed: int, token: int, pos: int, row: int) -> float:
    return float(lib().or_gumbel(seed, token, pos, row))


def gumbel_scores(logits, temperature: float, seed: int, pos: int, row: int) -> np.ndarray:
    """logits / T + the Gumbel draw of every token (their argmax is the sampled token)."""
    v = _c(logits, np.float32)
    z = np.empty_like(v)
    lib().or_gumbel_scores(_ptr(v, _f32p), v.shape[0], temperature, seed, pos, row, _ptr(z, _f32p))
    return z


def sample_gumbel_topk(logits, temperature: float, top_k: int, seed: int, pos: int, row: int) -> int:
    """A draw from softmax(logits / T) over the top_k largest logits (lower index first
    among equal logits); top_k 0 or >= vocab: no cut."""
    v = _c(logits, np.float32)
    r = int(lib().or_sample_gumbel_topk(_ptr(v, _f32p), v.shape[0], temperature, int(top_k), seed, pos, row))
    if r < 0:
        raise MemoryError("or_sample_gumbel_topk")
    return r


def sample_gumbel(logits, temperature: float, seed: int, pos: int, row: int) -> int:
    v = _c(logits, np.float32)
    return int(lib().or_sample_gumbel(_ptr(v, _f32p), v.shape[0], temperature, seed, pos, row))

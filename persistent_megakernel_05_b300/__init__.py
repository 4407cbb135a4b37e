"""B300 persistent decode megakernel: Python binding of the C ABI in include/mk.h.

The binding only marshals arguments (ctypes); every step of the decode path runs in
the CUDA kernel of ``libmk.so``. PyTorch is used for device memory and streams only.
There is no CPU fallback: importing the binding without the built library, or
calling it without a CUDA device, raises.

Names mirror the C ABI (``mk_create``, ``mk_kv_alloc``, ``mk_decode_step``, ...);
``DecodeModel`` bundles them for a model whose weights are torch BF16 tensors.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmk.so")

MK_OK = 0
MK_ERR_INVALID_ARG = 1
MK_ERR_UNSUPPORTED_DEVICE = 2
MK_ERR_OOM = 3
MK_ERR_LAUNCH = 4
MK_ERR_BAD_PAGE = 5
MK_ERR_TIMEOUT = 6
MK_ERR_INTERNAL = 7
MK_ERR_NO_DEVICE = 8
MK_OPT_TIMEOUT_NS = 1
MK_OPT_SKIP_PUBLISH = 2
MK_OPT_PREFETCH_SLOTS = 3

# exported symbols of include/mk.h
ABI_SYMBOLS = ("mk_create", "mk_kv_alloc", "mk_kv_free", "mk_decode_step", "mk_status_sync",
               "mk_status_reset", "mk_set_option", "mk_get_info", "mk_debug_buffer",
               "mk_status_string", "mk_destroy", "mk_decode_step_noalloc", "mk_set_sampling",
               "mk_set_shared_prefix", "mk_decode_steps", "mk_decode_step_host")
MK_NOALLOC_SCRATCH_BYTES = 8 << 20
MK_BUF_X, MK_BUF_QKV, MK_BUF_ATTN, MK_BUF_H, MK_BUF_ROUTE, MK_BUF_MOE_UNION = 1, 2, 3, 4, 5, 6


class MkError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} ({code})" if what else status_string(code))


_P = ctypes.POINTER
_vp = ctypes.c_void_p


class mk_model_desc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("d_model", ctypes.c_int32),
                ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("ffn_dim", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("expert_ffn_dim", ctypes.c_int32),
                ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
                ("sliding_window", ctypes.c_int32), ("layer_is_sliding", _P(ctypes.c_uint8)),
                ("max_batch", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("max_positions", ctypes.c_int32)]


LAYER_FIELDS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down",
                "router", "exp_gate", "exp_up", "exp_down")


class mk_layer_weights(ctypes.Structure):
    _fields_ = [(n, _vp) for n in LAYER_FIELDS]


class mk_weights(ctypes.Structure):
    _fields_ = [("embed", _vp), ("final_norm", _vp), ("lm_head", _vp),
                ("layers", _P(mk_layer_weights))]


class mk_kv_pool(ctypes.Structure):
    _fields_ = [("base", _vp), ("num_pages", ctypes.c_int32), ("layer_stride", ctypes.c_int64),
                ("page_stride", ctypes.c_int64), ("kv_stride", ctypes.c_int64),
                ("head_stride", ctypes.c_int64), ("slot_stride", ctypes.c_int64),
                ("bytes", ctypes.c_int64)]


class mk_info(ctypes.Structure):
    _fields_ = [("num_ctas", ctypes.c_int32), ("threads_per_cta", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int32), ("ring_stages", ctypes.c_int32),
                ("weight_bytes", ctypes.c_int64), ("scratch_bytes", ctypes.c_int64)]


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libmk.so (raises if it has not been built: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing; build it with "
                          "`python -m persistent_megakernel_05_b300.build`")
    L = ctypes.CDLL(path)
    i32, i64 = ctypes.c_int32, ctypes.c_int64
    L.mk_create.restype = ctypes.c_int
    L.mk_create.argtypes = [_P(mk_model_desc), _P(mk_weights), ctypes.c_int, _P(_vp)]
    L.mk_kv_alloc.restype = ctypes.c_int
    L.mk_kv_alloc.argtypes = [_vp, i32, _P(mk_kv_pool)]
    L.mk_kv_free.restype = ctypes.c_int
    L.mk_kv_free.argtypes = [_vp, _P(mk_kv_pool)]
    L.mk_decode_step.restype = ctypes.c_int
    L.mk_decode_step.argtypes = [_vp, _vp, _vp, _vp, i32, _vp, i32, _vp, _vp, _vp]
    L.mk_decode_step_host.restype = ctypes.c_int
    L.mk_decode_step_host.argtypes = [_vp, _vp, _vp, _vp, i32, _vp, i32, _vp, _vp, _vp]
    L.mk_decode_steps.restype = ctypes.c_int
    L.mk_decode_steps.argtypes = [_vp, i32, _vp, _vp, _vp, i32, _vp, i32, _vp, _vp, _vp]
    L.mk_status_sync.restype = ctypes.c_int
    L.mk_status_sync.argtypes = [_vp, _vp, _P(i32)]
    L.mk_status_reset.restype = ctypes.c_int
    L.mk_status_reset.argtypes = [_vp]
    L.mk_set_option.restype = ctypes.c_int
    L.mk_set_option.argtypes = [_vp, ctypes.c_int, i64]
    L.mk_set_sampling.restype = ctypes.c_int
    L.mk_set_sampling.argtypes = [_vp, ctypes.c_float, ctypes.c_int32, ctypes.c_uint64]
    L.mk_set_shared_prefix.restype = ctypes.c_int
    L.mk_set_shared_prefix.argtypes = [_vp, i32, _P(i32), _P(i32)]
    L.mk_get_info.restype = ctypes.c_int
    L.mk_get_info.argtypes = [_vp, _P(mk_info)]
    L.mk_debug_buffer.restype = ctypes.c_int
    L.mk_debug_buffer.argtypes = [_vp, ctypes.c_int32, _P(_vp), _P(i64)]
    L.mk_decode_step_noalloc.restype = ctypes.c_int
    L.mk_decode_step_noalloc.argtypes = [_P(mk_model_desc), _P(mk_weights), _vp, i32, _vp, _vp,
                                         _vp, i32, _vp, i32, _vp, _vp, _vp, _vp]
    L.mk_status_string.restype = ctypes.c_char_p
    L.mk_status_string.argtypes = [ctypes.c_int]
    L.mk_destroy.restype = None
    L.mk_destroy.argtypes = [_vp]
    _lib = L
    return L


def status_string(code: int) -> str:
    try:
        return load().mk_status_string(int(code)).decode()
    except ImportError:
        return f"status {code}"


def _check(code: int, what: str):
    if code != MK_OK:
        raise MkError(code, what)


# ---- thin wrappers with the C names -------------------------------------------------
def mk_create(desc: mk_model_desc, weights: mk_weights, device: int = 0) -> int:
    h = _vp()
    _check(load().mk_create(ctypes.byref(desc), ctypes.byref(weights), device, ctypes.byref(h)),
           "mk_create")
    return h.value


def mk_kv_alloc(handle: int, num_pages: int) -> mk_kv_pool:
    pool = mk_kv_pool()
    _check(load().mk_kv_alloc(handle, num_pages, ctypes.byref(pool)), "mk_kv_alloc")
    return pool


def mk_kv_free(handle: int, pool: Optional[mk_kv_pool] = None):
    _check(load().mk_kv_free(handle, ctypes.byref(pool) if pool is not None else None),
           "mk_kv_free")


def mk_decode_step(handle: int, tokens: int, positions: int, page_table: int,
                   max_pages_per_seq: int, seq_lens: int, batch: int, next_tokens: int,
                   logits: Optional[int], stream: Optional[int] = None) -> int:
    """Raw call with device addresses (ints). Returns the mk_status code."""
    return load().mk_decode_step(handle, tokens, positions, page_table, max_pages_per_seq,
                                 seq_lens, batch, next_tokens, logits, stream)


def mk_decode_step_host(handle: int, tokens: int, positions: int, page_table: int,
                        max_pages_per_seq: int, seq_lens: int, batch: int, next_tokens: int,
                        logits: Optional[int], stream: Optional[int] = None) -> int:
    """Raw call with HOST addresses (ints); synchronous. Returns the mk_status code (the
    step's device status when the call itself succeeded)."""
    return load().mk_decode_step_host(handle, tokens, positions, page_table, max_pages_per_seq,
                                      seq_lens, batch, next_tokens, logits, stream)


def mk_decode_steps(handle: int, n_steps: int, tokens: int, positions: int, page_table: int,
                    max_pages_per_seq: int, seq_lens: int, batch: int, next_tokens: int,
                    logits: Optional[int], stream: Optional[int] = None) -> int:
    """Raw call with device addresses (ints): n_steps steps in one launch. Returns the
    mk_status code."""
    return load().mk_decode_steps(handle, n_steps, tokens, positions, page_table,
                                  max_pages_per_seq, seq_lens, batch, next_tokens, logits, stream)


def mk_status_sync(handle: int, stream: Optional[int] = None):
    task = ctypes.c_int32(-1)
    code = load().mk_status_sync(handle, stream, ctypes.byref(task))
    return code, task.value


def mk_status_reset(handle: int):
    _check(load().mk_status_reset(handle), "mk_status_reset")


def mk_set_option(handle: int, opt: int, value: int):
    _check(load().mk_set_option(handle, opt, int(value)), "mk_set_option")


def mk_set_sampling(handle: int, temperature: float, seed: int, top_k: int = 0):
    _check(load().mk_set_sampling(handle, float(temperature), int(top_k), int(seed) & (2 ** 64 - 1)),
           "mk_set_sampling")


def mk_set_shared_prefix(handle: int, leader, shared_pages):
    """leader[b], shared_pages[b] for each row of the batch (host lists); empty lists
    clear the groups."""
    B = len(leader)
    if len(shared_pages) != B:
        raise ValueError("leader and shared_pages differ in length")
    if B == 0:
        _check(load().mk_set_shared_prefix(handle, 0, None, None), "mk_set_shared_prefix")
        return
    arr = ctypes.c_int32 * B
    _check(load().mk_set_shared_prefix(handle, B, arr(*[int(x) for x in leader]),
                                       arr(*[int(x) for x in shared_pages])),
           "mk_set_shared_prefix")


def mk_get_info(handle: int) -> mk_info:
    info = mk_info()
    _check(load().mk_get_info(handle, ctypes.byref(info)), "mk_get_info")
    return info


def mk_debug_buffer(handle: int, which: int):
    ptr, nbytes = _vp(), ctypes.c_int64()
    _check(load().mk_debug_buffer(handle, which, ctypes.byref(ptr), ctypes.byref(nbytes)),
           "mk_debug_buffer")
    return ptr.value, nbytes.value


def perm_col(k):
    """Storage column of logical column k in the permuted activation layouts."""
    return (k & ~63) | (((k & 7) >> 1) << 4) | (((k & 63) >> 3) << 1) | (k & 1)


def mk_decode_step_noalloc(desc: mk_model_desc, weights: mk_weights, kv_pool: int,
                           num_pages: int, tokens: int, positions: int, page_table: int,
                           max_pages_per_seq: int, seq_lens: int, batch: int, next_tokens: int,
                           logits: Optional[int], status_out: int,
                           stream: Optional[int] = None) -> int:
    """Decode step without a handle and without any device allocation (all scratch in
    the library's static device array); raw device addresses. Returns the mk_status of
    the host-side checks; the device status lands in status_out (int32[2])."""
    return load().mk_decode_step_noalloc(ctypes.byref(desc), ctypes.byref(weights), kv_pool,
                                         num_pages, tokens, positions, page_table,
                                         max_pages_per_seq, seq_lens, batch, next_tokens,
                                         logits, status_out, stream)


def mk_destroy(handle: int):
    load().mk_destroy(handle)


# ---- model wrapper --------------------------------------------------------------------
def _desc_from_cfg(cfg, sliding_buf) -> mk_model_desc:
    d = mk_model_desc()
    d.n_layers, d.d_model = cfg.n_layers, cfg.d_model
    d.n_q_heads, d.n_kv_heads, d.head_dim = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    d.ffn_dim, d.vocab = cfg.ffn_dim, cfg.vocab
    d.n_experts, d.top_k, d.expert_ffn_dim = cfg.n_experts, cfg.top_k, cfg.expert_ffn_dim
    d.rms_eps, d.rope_theta, d.sliding_window = cfg.rms_eps, cfg.rope_theta, cfg.sliding_window
    d.layer_is_sliding = ctypes.cast(sliding_buf, _P(ctypes.c_uint8))
    d.max_batch, d.page_size, d.max_positions = cfg.max_batch, cfg.page_size, cfg.max_positions
    return d


class _CudaArray:
    """Exposes raw device memory to torch through __cuda_array_interface__."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"data": (ptr, False), "shape": tuple(shape),
                                         "typestr": typestr, "version": 3, "strides": None}


class DecodeModel:
    """One handle: a model (borrowed torch BF16 weights on a CUDA device) plus the
    library-owned paged KV pool."""

    def __init__(self, cfg, weights: dict, num_pages: int, device: int = 0):
        import torch
        if not torch.cuda.is_available():
            raise MkError(MK_ERR_NO_DEVICE, "DecodeModel")
        self.cfg = cfg
        self.weights = weights  # keep the borrowed tensors alive
        self._sliding = (ctypes.c_uint8 * cfg.n_layers)(*cfg.layer_is_sliding())
        self.desc = _desc_from_cfg(cfg, self._sliding)
        layers = (mk_layer_weights * cfg.n_layers)()
        for i, L in enumerate(weights["layers"]):
            for n in LAYER_FIELDS:
                t = L.get(n)
                if t is not None:
                    assert t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous(), n
                    setattr(layers[i], n, t.data_ptr())
        self._layers = layers
        self.w = mk_weights(weights["embed"].data_ptr(), weights["final_norm"].data_ptr(),
                            weights["lm_head"].data_ptr(),
                            ctypes.cast(layers, _P(mk_layer_weights)))
        self.device = device
        self.handle = mk_create(self.desc, self.w, device)
        try:
            self.pool = mk_kv_alloc(self.handle, num_pages)
        except Exception:
            mk_destroy(self.handle)
            self.handle = None
            raise
        self.num_pages = num_pages
        self.info = mk_get_info(self.handle)

    def kv(self):
        """The pool as a torch BF16 tensor view [L, pages, 2, Hkv, 16, hd] (no copy)."""
        import torch
        c = self.cfg
        shape = (c.n_layers, self.num_pages, 2, c.n_kv_heads, c.page_size, c.head_dim)
        t = torch.as_tensor(_CudaArray(self.pool.base, shape, "<i2"), device=f"cuda:{self.device}")
        return t.view(torch.bfloat16)

    def buffer(self, which: int):
        """Copy of a last-layer activation buffer as fp32 [max_batch, width], logical
        column order (see mk_debug_buffer)."""
        import numpy as np
        import torch
        ptr, nbytes = mk_debug_buffer(self.handle, which)
        cfg = self.cfg
        if which == MK_BUF_MOE_UNION:
            t = torch.as_tensor(_CudaArray(ptr, (nbytes // 4,), "<i4"), device=f"cuda:{self.device}")
            return t.cpu().numpy().copy()
        h_width = cfg.n_experts * cfg.expert_ffn_dim if cfg.is_moe else cfg.ffn_dim
        width = {MK_BUF_X: cfg.d_model, MK_BUF_QKV: (cfg.n_q_heads + 2 * cfg.n_kv_heads) * cfg.head_dim,
                 MK_BUF_ATTN: cfg.n_q_heads * cfg.head_dim, MK_BUF_H: h_width,
                 MK_BUF_ROUTE: cfg.n_experts}[which]
        step = nbytes // (cfg.max_batch * width * 4)  # 2: tagged words (value in the low half)
        t = torch.as_tensor(_CudaArray(ptr, (nbytes // 4,), "<f4"), device=f"cuda:{self.device}")
        a = t.cpu().numpy()[0::step].reshape(cfg.max_batch, -1).copy()
        if which not in (MK_BUF_QKV, MK_BUF_ROUTE):
            idx = np.array([perm_col(k) for k in range(a.shape[1])])
            a = a[:, idx]
        return a

    def step(self, tokens, positions, page_table, seq_lens, next_tokens, logits=None,
             stream=None):
        """Enqueues one decode step. All tensors are int32 / fp32 CUDA tensors."""
        import torch
        for t in (tokens, positions, page_table, seq_lens, next_tokens):
            assert t.is_cuda and t.dtype == torch.int32 and t.is_contiguous()
        if logits is not None:
            assert logits.is_cuda and logits.dtype == torch.float32 and logits.is_contiguous()
        B = tokens.shape[0]
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        code = mk_decode_step(self.handle, tokens.data_ptr(), positions.data_ptr(),
                              page_table.data_ptr(), page_table.shape[1], seq_lens.data_ptr(), B,
                              next_tokens.data_ptr(),
                              logits.data_ptr() if logits is not None else None, s.cuda_stream)
        _check(code, "mk_decode_step")

    def step_host(self, tokens, positions, page_table, seq_lens, next_tokens, logits=None,
                  stream=None):
        """One decode step from and to host memory (numpy arrays, C-contiguous: int32
        inputs and next_tokens, fp32 logits [B][vocab] or None); returns when next_tokens
        (and logits) hold the step's results. Raises on a host or device error."""
        import numpy as np
        import torch
        for a in (tokens, positions, page_table, seq_lens, next_tokens):
            assert isinstance(a, np.ndarray) and a.dtype == np.int32 and a.flags.c_contiguous
        if logits is not None:
            assert logits.dtype == np.float32 and logits.flags.c_contiguous
        B = tokens.shape[0]
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        code = mk_decode_step_host(self.handle, tokens.ctypes.data, positions.ctypes.data,
                                   page_table.ctypes.data, page_table.shape[1], seq_lens.ctypes.data,
                                   B, next_tokens.ctypes.data,
                                   logits.ctypes.data if logits is not None else None, s.cuda_stream)
        _check(code, "mk_decode_step_host")

    def steps(self, n_steps, tokens, positions, page_table, seq_lens, next_tokens, logits=None,
              stream=None):
        """Enqueues n_steps decode steps as one launch: step s > 0 takes step s-1's tokens
        at positions + s. next_tokens is [n_steps][B] int32; logits (optional) receives the
        last step's [B][vocab] fp32."""
        import torch
        for t in (tokens, positions, page_table, seq_lens, next_tokens):
            assert t.is_cuda and t.dtype == torch.int32 and t.is_contiguous()
        B = tokens.shape[0]
        assert next_tokens.numel() >= n_steps * B
        if logits is not None:
            assert logits.is_cuda and logits.dtype == torch.float32 and logits.is_contiguous()
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        code = mk_decode_steps(self.handle, int(n_steps), tokens.data_ptr(), positions.data_ptr(),
                               page_table.data_ptr(), page_table.shape[1], seq_lens.data_ptr(), B,
                               next_tokens.data_ptr(),
                               logits.data_ptr() if logits is not None else None, s.cuda_stream)
        _check(code, "mk_decode_steps")

    def status(self, stream=None):
        import torch
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        return mk_status_sync(self.handle, s.cuda_stream)

    def reset(self):
        mk_status_reset(self.handle)

    def set_option(self, opt: int, value: int):
        mk_set_option(self.handle, opt, value)

    def set_sampling(self, temperature: float, seed: int = 0, top_k: int = 0):
        """temperature 0: greedy; > 0: draw from softmax(logits / temperature), over the
        top_k largest logits when top_k > 0."""
        mk_set_sampling(self.handle, temperature, seed, top_k)

    def set_shared_prefix(self, leader=(), shared_pages=()):
        """Rows b with the same leader[b] share logical pages [0, shared_pages[b]) of their
        page tables; their prefix K/V is read once per kv head for the group. No
        arguments: clear."""
        mk_set_shared_prefix(self.handle, list(leader), list(shared_pages))

    def close(self):
        if getattr(self, "handle", None):
            mk_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

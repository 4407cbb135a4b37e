"""mk_decode_step_noalloc: the decode step for callers that cannot allocate device
memory (a memory plan that owns all of HBM, allocator-free or sandboxed runtimes,
paths where cudaMalloc would synchronise the device). It must give the same result
as the handle-based mk_decode_step while its scratch lives in the library's static
device array.

This file is collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
import persistent_megakernel_05_b300 as mk
from harness import LOGIT_ATOL, MARGIN

pytestmark = pytest.mark.gpu


def _addr(t):
    return t.data_ptr()


def test_noalloc_matches_handle_path_on_two_consecutive_calls():
    from persistent_megakernel_05_b300 import build
    build.build()
    cfg = synth.TINY
    W = synth.make_weights(cfg, 21, device="cuda", gain_noise=0.02)
    npages = 64
    model = mk.DecodeModel(cfg, W, npages)
    synth.fill_normal_bf16_(model.kv(), 4)
    # the caller owns the second pool: a plain torch allocation, same contents
    pool2 = model.kv().clone()
    rng = np.random.default_rng(21)
    B = 8
    pos = np.array([3, 15, 16, 40, 77, 100, 129, 200], np.int32)
    pages = [int(p) // 16 + 2 for p in pos]
    pt = torch.tensor(synth.random_page_tables(rng, npages, pages, max(pages)), device="cuda")
    toks = torch.tensor(synth.random_tokens(rng, cfg.vocab, B), device="cuda")
    status = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        p = torch.tensor(pos + call, device="cuda")
        sl = p + 1
        nx_a = torch.empty(B, dtype=torch.int32, device="cuda")
        nx_b = torch.empty(B, dtype=torch.int32, device="cuda")
        lg_a = torch.empty((B, cfg.vocab), device="cuda")
        lg_b = torch.empty((B, cfg.vocab), device="cuda")
        model.step(toks, p, pt, sl, nx_a, lg_a)
        assert model.status()[0] == mk.MK_OK
        stream = torch.cuda.current_stream().cuda_stream
        rc = mk.mk_decode_step_noalloc(model.desc, model.w, _addr(pool2), npages, _addr(toks),
                                       _addr(p), _addr(pt), pt.shape[1], _addr(sl), B,
                                       _addr(nx_b), _addr(lg_b), _addr(status), stream)
        assert rc == mk.MK_OK, mk.status_string(rc)
        torch.cuda.synchronize()
        assert status.tolist()[0] == mk.MK_OK, status.tolist()
        a, b = lg_a.cpu().numpy(), lg_b.cpu().numpy()
        assert np.isfinite(b).all()
        assert np.abs(a - b).max() <= LOGIT_ATOL, f"call {call}: {np.abs(a - b).max()}"
        na, nb = nx_a.cpu().numpy(), nx_b.cpu().numpy()
        for r in range(B):
            top2 = np.partition(a[r], -2)[-2:]
            if top2[1] - top2[0] > MARGIN:
                assert na[r] == nb[r], (call, r)
        toks = nx_a.clone()
    # both pools received the same appends
    ka = synth.bf16_bits(model.kv()).astype(np.int32)
    kb = synth.bf16_bits(pool2).astype(np.int32)
    f = lambda x: ((x.astype(np.uint32) << 16).view(np.float32))  # noqa: E731
    assert np.abs(f(ka) - f(kb)).max() <= 2e-2 * max(np.abs(f(ka)).max(), 1.0)
    model.close()


def test_noalloc_rejects_a_descriptor_whose_scratch_does_not_fit():
    cfg = synth.TINY
    W = synth.make_weights(cfg, 22, device="cuda")
    model = mk.DecodeModel(cfg, W, 8)
    big = mk.mk_model_desc()
    ctypes.memmove(ctypes.byref(big), ctypes.byref(model.desc), ctypes.sizeof(big))
    big.max_positions = 1 << 20  # RoPE table alone: 1M * 32 * 8 B = 256 MiB > 8 MiB
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    rc = mk.mk_decode_step_noalloc(big, model.w, _addr(model.kv()), 8, _addr(dummy), _addr(dummy),
                                   _addr(dummy), 1, _addr(dummy), 1, _addr(dummy), None,
                                   _addr(dummy), None)
    assert rc == mk.MK_ERR_INVALID_ARG
    model.close()

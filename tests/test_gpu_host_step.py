"""mk_decode_step_host: the decode step from and to host memory. The arithmetic is the
device-buffer step's, so tokens, logits and K/V appends must equal it bit for bit; the
call must also hand back the step's device status (a latched error, then recovery)."""
import numpy as np
import pytest
import torch

import synth
import persistent_megakernel_05_b300 as mk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from persistent_megakernel_05_b300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")


def _twin_models(cfg, W, npages, kv_seed):
    ms = []
    for _ in range(2):
        m = mk.DecodeModel(cfg, W, npages)
        synth.fill_normal_bf16_(m.kv(), kv_seed)
        ms.append(m)
    torch.cuda.synchronize()
    return ms


CASES = {
    "tiny-b1": (synth.TINY, 1),
    "tiny-b3": (synth.TINY, 3),
    "tiny-b8": (synth.TINY, 8),
    "2b-2layers-b2": (synth.DENSE_2B.with_(n_layers=2, max_batch=2, max_positions=2048), 2),
}


@pytest.mark.parametrize("case", list(CASES))
def test_host_step_equals_device_step(case):
    cfg, B = CASES[case]
    W = synth.make_weights(cfg, 41, device="cuda")
    per = 6 if cfg.d_model <= 256 else 40
    npages = per * B + 4
    dev_m, host_m = _twin_models(cfg, W, npages, kv_seed=5)
    rng = np.random.default_rng(41 + B)
    pt = synth.random_page_tables(rng, npages, [per] * B, per).astype(np.int32)
    pos0 = (rng.integers(0, 16 * (per - 2), size=B)).astype(np.int32)
    tok = synth.random_tokens(rng, cfg.vocab, B).astype(np.int32)
    d_pt = torch.tensor(pt, device="cuda")
    d_tok = torch.tensor(tok, device="cuda")
    d_next = torch.empty(B, dtype=torch.int32, device="cuda")
    d_lg = torch.empty((B, cfg.vocab), dtype=torch.float32, device="cuda")
    h_tok = tok.copy()
    h_next = np.empty(B, np.int32)
    h_lg = np.empty((B, cfg.vocab), np.float32)
    for s in range(3):
        pos = pos0 + s
        d_pos = torch.tensor(pos, device="cuda")
        dev_m.step(d_tok, d_pos, d_pt, d_pos + 1, d_next, d_lg)
        assert dev_m.status()[0] == mk.MK_OK
        # every other step without logits (the host call then copies only status + tokens)
        want_lg = s != 1
        host_m.step_host(h_tok, pos.copy(), pt, pos + 1, h_next, h_lg if want_lg else None)
        assert np.array_equal(h_next, d_next.cpu().numpy()), s
        if want_lg:
            assert np.array_equal(h_lg, d_lg.cpu().numpy()), s
        d_tok = d_next.clone()
        h_tok = h_next.copy()
    torch.cuda.synchronize()
    assert torch.equal(dev_m.kv(), host_m.kv())
    dev_m.close()
    host_m.close()


def test_host_step_returns_the_device_status():
    cfg = synth.TINY
    W = synth.make_weights(cfg, 42, device="cuda")
    m = mk.DecodeModel(cfg, W, 8)
    synth.fill_normal_bf16_(m.kv(), 2)
    torch.cuda.synchronize()
    nxt = np.zeros(1, np.int32)
    tok, pos, sl = np.array([5], np.int32), np.array([20], np.int32), np.array([21], np.int32)
    bad_pt = np.array([[0, 99]], np.int32)  # page 99 does not exist: the kernel's check latches
    code = mk.mk_decode_step_host(m.handle, tok.ctypes.data, pos.ctypes.data, bad_pt.ctypes.data, 2,
                                  sl.ctypes.data, 1, nxt.ctypes.data, None,
                                  torch.cuda.current_stream().cuda_stream)
    assert code == mk.MK_ERR_BAD_PAGE
    m.reset()
    m.step_host(tok, pos, np.array([[0, 1]], np.int32), sl, nxt)
    assert 0 <= nxt[0] < cfg.vocab
    # host-side argument errors come back before any copy
    assert mk.mk_decode_step_host(m.handle, tok.ctypes.data, pos.ctypes.data, bad_pt.ctypes.data, 2,
                                  sl.ctypes.data, 0, nxt.ctypes.data, None, None) == mk.MK_ERR_INVALID_ARG
    m.close()

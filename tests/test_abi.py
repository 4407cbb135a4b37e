"""The C-ABI library loads and exports every symbol include/mk.h declares; host-side
argument checks return errors without touching a GPU (no GPU needed)."""
import ctypes
import os
import re

import pytest

import persistent_megakernel_05_b300 as mk
from persistent_megakernel_05_b300 import build as mkbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mkbuild.build()
    return mk.load()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "mk.h")).read()
    return re.findall(r"MK_API\s+[\w\s\*]+?\b(mk_\w+)\s*\(", src)


def test_header_declares_the_abi():
    assert sorted(declared_symbols()) == sorted(mk.ABI_SYMBOLS)


@pytest.mark.parametrize("lang,std", [("c", "-std=c99"), ("c++", "-std=c++17")])
def test_header_compiles_as_plain_c_and_cpp(tmp_path, lang, std):
    """The ABI header is usable from C (no C++ or torch types leak into it)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / "use_mk.c"
    src.write_text('#include "mk.h"\nint main(void) { return (int)sizeof(mk_model_desc) > 0 ? 0 : 1; }\n')
    subprocess.run([cc, "-x", lang, std, "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), "-c", str(src), "-o", str(tmp_path / "use_mk.o")],
                   check=True)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    # nothing else leaks out of the library's C namespace
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", mkbuild.LIB], capture_output=True,
                         text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert {s for s in exported if s.startswith("mk_")} == set(mk.ABI_SYMBOLS)


def test_status_strings(lib):
    for code in range(9):
        assert mk.status_string(code)
    assert mk.status_string(0) == "ok"


def test_host_side_argument_errors_need_no_gpu(lib):
    h = ctypes.c_void_p()
    assert lib.mk_create(None, None, 0, ctypes.byref(h)) == mk.MK_ERR_INVALID_ARG
    assert h.value is None
    d = mk.mk_model_desc()
    d.n_layers, d.d_model, d.n_q_heads, d.n_kv_heads, d.head_dim = 2, 100, 4, 2, 64  # d % 64
    d.ffn_dim, d.vocab, d.rms_eps, d.rope_theta = 768, 4096, 1e-5, 1e4
    d.max_batch, d.page_size, d.max_positions = 8, 16, 64
    w = mk.mk_weights()
    assert lib.mk_create(ctypes.byref(d), ctypes.byref(w), 0, ctypes.byref(h)) == mk.MK_ERR_INVALID_ARG
    d.d_model = 256
    d.head_dim = 96
    assert lib.mk_create(ctypes.byref(d), ctypes.byref(w), 0, ctypes.byref(h)) == mk.MK_ERR_INVALID_ARG
    d.head_dim = 64
    d.page_size = 32
    assert lib.mk_create(ctypes.byref(d), ctypes.byref(w), 0, ctypes.byref(h)) == mk.MK_ERR_INVALID_ARG
    d.page_size = 16
    d.max_batch = 9
    assert lib.mk_create(ctypes.byref(d), ctypes.byref(w), 0, ctypes.byref(h)) == mk.MK_ERR_INVALID_ARG
    d.max_batch = 8
    # valid shape, but null weight pointers
    assert lib.mk_create(ctypes.byref(d), ctypes.byref(w), 0, ctypes.byref(h)) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_decode_step(None, None, None, None, 1, None, 1, None, None, None) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_decode_step_host(None, None, None, None, 1, None, 1, None, None, None) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_kv_alloc(None, 4, None) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_status_reset(None) == mk.MK_ERR_INVALID_ARG
    assert lib.mk_set_option(None, mk.MK_OPT_TIMEOUT_NS, 10**9) == mk.MK_ERR_INVALID_ARG
    lib.mk_destroy(None)  # allowed


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(ImportError):
        mk._lib_backup = mk._lib
        try:
            mk._lib = None
            mk.load(str(tmp_path / "missing.so"))
        finally:
            mk._lib = mk._lib_backup

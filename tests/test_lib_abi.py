"""The C-ABI library builds, loads and exports every declared symbol; host-side
argument validation rejects bad calls before any launch (CPU only: no compute
call is made)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdv.h")


@pytest.fixture(scope="module")
def lib():
    from speculative_decode_verify_sdv_gb300 import build, sdv
    build.build()
    return sdv.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sdv_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("sdv_qlinear", "sdv_qlinear_swiglu", "sdv_verify_head", "sdv_greedy_accept",
                 "sdv_moe_gather_qmm", "sdv_quantize_block32", "sdv_workspace_bytes"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in sdv.h but not exported"


def test_binding_names_match_the_header(lib):
    from speculative_decode_verify_sdv_gb300 import sdv
    for name in declared_functions():
        assert callable(getattr(sdv, name, None)), f"binding lacks {name}"


def test_no_unexpected_exports(lib):
    # only the sdv_ API is visible (kernels and helpers are hidden)
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True).stdout
    syms = {l.split()[-1] for l in out.splitlines() if " T " in l}
    api = {s for s in syms if s.startswith("sdv_")}
    assert api == set(declared_functions())


def test_version_and_status_strings(lib):
    assert lib.sdv_version() >= 100
    assert lib.sdv_status_string(0) == b"SDV_OK"
    assert lib.sdv_status_string(4) == b"SDV_ERR_TIMEOUT"


def _qw(lib, qtype=8, n=64, k=64, codes=16, scales=16):
    from speculative_decode_verify_sdv_gb300.sdv import sdv_qweight
    return sdv_qweight(qtype, n, k, ctypes.c_void_p(codes), ctypes.c_void_p(scales))


def test_host_validation_rejects_bad_arguments(lib):
    from speculative_decode_verify_sdv_gb300 import sdv
    p16 = ctypes.c_void_p(16)
    # bad weights: k not a multiple of 32, unknown qtype, null codes, misaligned scales
    for qw in (_qw(lib, k=48), _qw(lib, qtype=5), _qw(lib, codes=0), _qw(lib, scales=18)):
        st = lib.sdv_verify_head(ctypes.byref(qw), p16, 9, p16, 8, None, p16, p16, p16, p16, 1 << 20, None)
        assert st == sdv.SDV_ERR_INVALID_ARG
    qw = _qw(lib)
    # n_valid outside [0, S-1]
    assert lib.sdv_verify_head(ctypes.byref(qw), p16, 9, p16, 9, None, p16, p16, p16, p16, 1 << 20, None) \
        == sdv.SDV_ERR_INVALID_ARG
    assert lib.sdv_verify_head(ctypes.byref(qw), p16, 9, p16, -1, None, p16, p16, p16, p16, 1 << 20, None) \
        == sdv.SDV_ERR_INVALID_ARG
    # S = 0 is invalid, S > 32 unsupported
    assert lib.sdv_verify_head(ctypes.byref(qw), p16, 0, p16, 0, None, p16, p16, p16, p16, 1 << 20, None) \
        == sdv.SDV_ERR_INVALID_ARG
    assert lib.sdv_verify_head(ctypes.byref(qw), p16, 33, p16, 0, None, p16, p16, p16, p16, 1 << 20, None) \
        == sdv.SDV_ERR_UNSUPPORTED
    # drafts required when n_valid > 0; misaligned activations
    assert lib.sdv_verify_head(ctypes.byref(qw), p16, 9, None, 3, None, p16, p16, p16, p16, 1 << 20, None) \
        == sdv.SDV_ERR_INVALID_ARG
    assert lib.sdv_verify_head(ctypes.byref(qw), ctypes.c_void_p(8), 9, p16, 3, None, p16, p16, p16, p16,
                               1 << 20, None) == sdv.SDV_ERR_INVALID_ARG
    # qlinear: null output; accept: bad n_valid; quantize: bad k
    assert lib.sdv_qlinear(ctypes.byref(qw), p16, 4, None, p16, 1 << 20, None) == sdv.SDV_ERR_INVALID_ARG
    assert lib.sdv_greedy_accept(p16, 4, p16, 4, p16, p16, None) == sdv.SDV_ERR_INVALID_ARG
    assert lib.sdv_quantize_block32(p16, 4, 40, 8, p16, p16, None) == sdv.SDV_ERR_INVALID_ARG
    assert lib.sdv_quantize_block32(p16, 4, 64, 3, p16, p16, None) == sdv.SDV_ERR_INVALID_ARG
    assert lib.sdv_workspace_init(None, 1024, None) == sdv.SDV_ERR_WORKSPACE


def test_sampling_verify_validation(lib):
    from speculative_decode_verify_sdv_gb300 import sdv
    p16 = ctypes.c_void_p(16)
    qw = _qw(lib)

    def call(S=9, n_valid=8, T=1.0, drafts=p16, x=p16, ws_bytes=1 << 20):
        return lib.sdv_verify_sample(ctypes.byref(qw), x, S, drafts, n_valid, T, 1, 2, None, p16, p16, p16,
                                     p16, ws_bytes, None)
    for T in (0.0, -1.0, float("nan"), float("inf")):
        assert call(T=T) == sdv.SDV_ERR_INVALID_ARG
    assert call(n_valid=9) == sdv.SDV_ERR_INVALID_ARG
    assert call(S=0, n_valid=0) == sdv.SDV_ERR_INVALID_ARG
    assert call(S=33, n_valid=0) == sdv.SDV_ERR_UNSUPPORTED
    assert call(drafts=None, n_valid=3) == sdv.SDV_ERR_INVALID_ARG
    assert call(x=ctypes.c_void_p(8)) == sdv.SDV_ERR_INVALID_ARG
    assert lib.sdv_workspace_bytes(sdv.SDV_OP_VERIFY_SAMPLE, 4096, 256, 9, 0, 0) > 0
    assert lib.sdv_workspace_bytes(sdv.SDV_OP_VERIFY_SAMPLE, 4096, 256, 33, 0, 0) == 0


def test_workspace_bytes_rejects_bad_window(lib):
    assert lib.sdv_workspace_bytes(3, 4096, 256, 0, 0, 0) == 0
    assert lib.sdv_workspace_bytes(3, 4096, 256, 33, 0, 0) == 0
    assert lib.sdv_workspace_bytes(99, 4096, 256, 9, 0, 0) == 0


@pytest.mark.parametrize("op", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("n,k", [(0, 256), (-5, 256), (4096, 0), (4096, 48), (4096, -256), (2**31 - 1, 256)])
def test_workspace_bytes_rejects_bad_shapes(lib, op, n, k):
    # answered before any device query, so no GPU is needed
    assert lib.sdv_workspace_bytes(op, n, k, 9, 8, 2) == 0


def test_moe_shape_products_do_not_wrap(lib):
    # E * I = 2**32 + 32768 wraps to 32768 in 32-bit arithmetic: must not match gate/up of 32768 rows
    from speculative_decode_verify_sdv_gb300 import sdv
    p16 = ctypes.c_void_p(16)
    E, I, H = 1024, 2**22 + 32, 256
    gate, up = _qw(lib, n=32768, k=H), _qw(lib, n=32768, k=H)
    down = _qw(lib, n=E * H, k=I)
    st = lib.sdv_moe_gather_qmm(ctypes.byref(gate), ctypes.byref(up), ctypes.byref(down), E, I, H, 8, p16, p16, 9,
                                p16, None, None, p16, 1 << 20, None)
    assert st == sdv.SDV_ERR_INVALID_ARG
    big = _qw(lib, n=2**31 - 1)
    assert lib.sdv_qlinear(ctypes.byref(big), p16, 4, p16, p16, 1 << 20, None) == sdv.SDV_ERR_INVALID_ARG

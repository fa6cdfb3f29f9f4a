"""The C ABI without a GPU: the library loads, exports every function the
header declares, and rejects invalid calls on the host before any launch."""
import ctypes
import subprocess

import numpy as np
import pytest

import implicit_gemm_convolution_gb300 as om
import oracle

E = om.STATUS_NAMES
INV, NUL, ALIAS, UNS, ALIGN, BIG = 1, 2, 3, 4, 7, 8


@pytest.fixture(scope="module")
def L():
    om.build()
    return om.lib()


def test_every_header_function_is_exported(L):
    names = om.header_functions()
    assert len(names) >= 8
    out = subprocess.run(["nm", "-D", "--defined-only", om.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for n in names:
        assert n in exported, n
        assert hasattr(L, n)
    # nothing else escapes the library's C namespace
    assert {e for e in exported if e.startswith("om_")} == set(names)


def test_version_and_status_strings(L):
    assert L.om_version() == 10000
    for code, name in E.items():
        assert L.om_status_string(code).decode() == name
    assert L.om_status_string(99).decode() == "OM_UNKNOWN"


def test_out_dim_matches_oracle(L):
    rng = np.random.default_rng(0)
    for _ in range(500):
        size, k = int(rng.integers(0, 70)), int(rng.integers(1, 8))
        s, p, d = int(rng.integers(1, 5)), int(rng.integers(0, 4)), int(rng.integers(1, 4))
        assert L.om_conv_out_dim(size, k, s, p, d) == oracle.conv_out_dim(size, k, s, p, p, d)
    for bad in [(-1, 3, 1, 0, 1), (5, 0, 1, 0, 1), (5, 3, 0, 0, 1), (5, 3, 1, -1, 1), (5, 3, 1, 0, 0)]:
        assert L.om_conv_out_dim(*bad) == -1


P = 0x10000  # an aligned non-null stand-in pointer: validation fails before any use


def gemm(L, m, n, k, A=P, lda=None, B=P * 16, ldb=None, C=P * 256, ldc=None, mode=0):
    lda = k if lda is None else lda
    ldb = n if ldb is None else ldb
    ldc = n if ldc is None else ldc
    return L.om_gemm_f32(m, n, k, A, lda, B, ldb, C, ldc, mode, None)


def test_gemm_validation(L):
    assert gemm(L, -1, 2, 2) == INV
    assert gemm(L, 2, 2, -3) == INV
    assert gemm(L, 2, 2, 2, mode=7) == UNS
    assert gemm(L, 0, 5, 5, A=None, B=None, C=None) == 0  # empty: success, nothing launched
    assert gemm(L, 5, 0, 5, A=None, B=None, C=None) == 0
    assert gemm(L, 4, 4, 4, lda=3) == INV
    assert gemm(L, 4, 4, 4, ldb=3) == INV
    assert gemm(L, 4, 4, 4, ldc=3) == INV
    assert gemm(L, 4, 4, 4, A=None) == NUL
    assert gemm(L, 4, 4, 4, B=None) == NUL
    assert gemm(L, 4, 4, 4, C=None) == NUL
    assert gemm(L, 4, 4, 4, A=P + 2) == ALIGN
    assert gemm(L, 4, 4, 4, C=P + 4) == ALIAS       # C inside A's rows
    assert gemm(L, 4, 4, 4, C=P * 16 + 8) == ALIAS  # C inside B


def test_gemm_alias_edges(L):
    # A occupies [P, P + (3*4+4)*4) = [P, P+64): C starting at P+64 does not overlap.
    assert gemm(L, 4, 4, 4, C=P + 60) == ALIAS
    assert gemm(L, 4, 4, 4, lda=4, C=P + 64, B=P * 1024) not in (ALIAS, INV, NUL, ALIGN)


def conv(L, N=1, Cin=4, H=5, W=5, Cout=4, G=1, KH=3, KW=3, s=1, p=1, d=1, x=P, w=P * 64,
         y=P * 256, mode=0, packed=False):
    f = L.om_conv2d_f32_packed if packed else L.om_conv2d_f32
    return f(N, Cin, H, W, Cout, G, KH, KW, s, p, d, x, w, y, mode, None)


def test_conv_validation(L):
    assert conv(L, N=-1) == INV
    assert conv(L, G=0) == INV
    assert conv(L, Cin=6, G=4) == INV
    assert conv(L, Cout=6, G=4, Cin=8) == INV
    assert conv(L, KH=0) == INV
    assert conv(L, s=0) == INV
    assert conv(L, d=0) == INV
    assert conv(L, p=-1) == INV
    assert conv(L, mode=2) == UNS
    assert conv(L, mode=9) == UNS
    assert conv(L, N=0, x=None, w=None, y=None) == 0
    assert conv(L, H=1, W=1, KH=3, KW=3, p=0, x=None, w=None, y=None) == 0  # empty output
    assert conv(L, x=None) == NUL
    assert conv(L, w=None) == NUL
    assert conv(L, y=None) == NUL
    assert conv(L, y=P + 4) == ALIAS
    assert conv(L, x=P + 1) == ALIGN
    assert conv(L, packed=True, w=P * 64 + 4) == ALIGN
    assert conv(L, KH=70000) == BIG


def test_pack_size_query(L):
    size = ctypes.c_size_t(0)
    assert L.om_pack_conv_weights(64, 64, 1, 3, 3, None, None, ctypes.byref(size), None) == 0
    assert size.value == 64 * 576 * 4
    assert L.om_pack_conv_weights(256, 256, 32, 3, 3, None, None, ctypes.byref(size), None) == 0
    assert size.value == 256 * 72 * 4
    assert L.om_pack_conv_weights(8, 3, 1, 3, 3, None, None, ctypes.byref(size), None) == 0
    assert size.value == 8 * 28 * 4  # K = 27 padded to 28
    assert L.om_pack_conv_weights(8, 3, 1, 3, 3, None, None, None, None) == NUL
    assert L.om_pack_conv_weights(8, 6, 4, 3, 3, None, None, ctypes.byref(size), None) == INV
    assert L.om_pack_conv_weights(8, 4, 1, 3, 3, P, P * 64 + 4, ctypes.byref(size), None) == ALIGN


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import implicit_gemm_convolution_gb300._build as b
    monkeypatch.setattr(b, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(om, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        om.lib()


def test_epilogue_entry_points_validate_on_host(L):
    # unknown activation, residual aliasing the output, short residual stride
    assert L.om_gemm_f32_ex(4, 4, 4, P, 4, P * 16, 4, P * 256, 4, None, None, 0, 5, 0, None, 0,
                            None) == INV
    assert L.om_gemm_f32_ex(4, 4, 4, P, 4, P * 16, 4, P * 256, 4, None, P * 256, 4, 1, 0, None, 0,
                            None) == ALIAS
    assert L.om_gemm_f32_ex(4, 4, 4, P, 4, P * 16, 4, P * 256, 4, None, P * 512, 2, 1, 0, None, 0,
                            None) == INV
    assert L.om_conv2d_f32_ex(1, 4, 5, 5, 4, 1, 3, 3, 1, 1, 1, P, P * 64, 0, None, None, 9,
                              P * 256, 0, None, 0, None) == INV
    assert L.om_conv2d_f32_ex(1, 4, 5, 5, 4, 1, 3, 3, 1, 1, 1, P, P * 64, 0, None, P * 256, 1,
                              P * 256, 0, None, 0, None) == ALIAS


def test_selftest_hook_rejects_bad_arguments_before_launch(L):
    for which, limit in ((2, 20), (-1, 20), (0, 0), (1, 1001)):
        assert L.om_selftest_wait_timeout(which, limit, None) == INV

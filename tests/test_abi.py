"""C-ABI library on the host (no GPU): it loads, exports every function that
``include/kq.h`` declares, its host helpers agree with the oracle, and its
argument checks reject bad calls before touching CUDA."""
import ctypes
import os
import re

import numpy as np
import pytest

from conftest import ROOT
from w4a4_mxfp4_activation_gb300 import kq, synth

HEADER = os.path.join(ROOT, "include", "kq.h")
TESTING_HEADER = os.path.join(ROOT, "include", "kq_testing.h")


@pytest.fixture(scope="module")
def L():
    from w4a4_mxfp4_activation_gb300 import build
    build.build()
    return kq.lib()


def declared_functions(header=HEADER):
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"KQ_API\s+[\w\s\*]+?\b(kq_\w+)\s*\(", text)))


def test_header_declares_the_api():
    names = declared_functions()
    for required in ("kq_expand_blocks", "kq_quantize_mxfp4", "kq_smooth_quantize_mxfp4",
                     "kq_hadamard_quantize_mxfp4", "kq_dequantize"):
        assert required in names
    assert set(names) == set(kq.EXPORTS)
    # the verification hooks stay out of the public header
    hooks = declared_functions(TESTING_HEADER)
    assert set(hooks) == set(kq.TESTING_EXPORTS)
    assert not set(hooks) & set(names)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions() + declared_functions(TESTING_HEADER):
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_mma_sync_variant_is_not_built(L):
    """The warp-level mma.sync transform lost to both other implementations
    and is no longer in the library: its variant number is rejected before
    anything runs."""
    vp = ctypes.c_void_p
    assert L.kq_quantize_mxfp4_variant(vp(4096), 4, 64, 64, vp(8192), vp(8192), vp(12288), 32,
                                       vp(16384), 0, None, 1, None) == 4


def test_status_strings(L):
    for s in range(7):
        assert kq.status_string(s)
    assert kq.status_string(99) == "unknown status"


def test_sf_bytes_matches_oracle(L, oracle_lib):
    for m in (0, 1, 127, 128, 129, 4608):
        for d in (32, 1152, 2240, 5600, 12288):
            for layout in (0, 1):
                assert kq.kq_sf_bytes(m, d, layout) == oracle_lib.sf_bytes(m, d // 32, layout)
    assert kq.kq_sf_bytes(4, 33, 0) == 0 and kq.kq_sf_bytes(-1, 32, 0) == 0
    assert kq.kq_sf_bytes(4, 32, 7) == 0


def test_expanded_bytes(L):
    assert kq.kq_expanded_bytes(36, kq.KQ_K_FP32) == 36 * 4096
    assert kq.kq_expanded_bytes(36, kq.KQ_K_BF16X3) == 36 * 6144
    assert kq.kq_expanded_bytes(0, kq.KQ_K_FP32) == 0


@pytest.mark.parametrize("sign", [-1, 1])
def test_lu_to_factors_matches_oracle_bitwise(L, oracle_lib, sign):
    """Library helper and oracle both evaluate eq. (6) in fp64 and round once
    to fp32: the entries must be identical."""
    lu = synth.lu_params(384, 2003)
    got = kq.kq_lu_to_factors(lu, sign)
    ref = oracle_lib.lu_to_factors(lu.astype(np.float64), sign).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_invert_transpose_factors(L):
    F = kq.kq_lu_to_factors(synth.lu_params(20, 5), 1)
    Finv = kq.kq_invert_transpose_factors(F)
    for j in range(20):
        for k in range(5):
            ref = np.linalg.inv(F[j, k].astype(np.float64)).T
            assert np.allclose(Finv[j, k], ref, rtol=2 ** -23, atol=0)
    with pytest.raises(kq.KqError):
        kq.kq_invert_transpose_factors(np.zeros((1, 5, 2, 2), np.float32))


def test_lu_to_factors_rejects(L):
    with pytest.raises(kq.KqError):
        kq.kq_lu_to_factors(np.zeros((1, 5, 3), np.float32), 1)   # a = 0
    with pytest.raises(kq.KqError):
        kq.kq_lu_to_factors(synth.lu_params(1, 0), 2)             # bad sign


# --- argument checks: each call fails validation before any CUDA call ----------------

FAKE = 1 << 20          # a 16-byte aligned, never dereferenced address


def _q(L, A=FAKE, m=4, d=64, lda=64, f=FAKE, K=None, q=FAKE, ldq=32, sf=FAKE, layout=0, y=None,
       variant=None):
    if variant is None:
        return L.kq_quantize_mxfp4(A, m, d, lda, f, K, q, ldq, sf, layout, y, None)
    return L.kq_quantize_mxfp4_variant(A, m, d, lda, f, K, q, ldq, sf, layout, y, variant, None)


def test_quantize_argument_checks(L):
    assert _q(L, d=48) == 2                       # d % 32
    assert _q(L, d=0) == 2
    assert _q(L, m=-1) == 2
    assert _q(L, lda=32) == 2                     # lda < d
    assert _q(L, ldq=16) == 2                     # ldq < d/2
    assert _q(L, layout=5) == 4
    assert _q(L, A=None) == 1
    assert _q(L, q=None) == 1
    assert _q(L, sf=None) == 1
    assert _q(L, A=FAKE + 2) == 3                 # A misaligned
    assert _q(L, q=FAKE + 8) == 3
    assert _q(L, lda=68) == 3                     # row pitch not 16-byte multiple
    assert _q(L, ldq=40) == 3
    assert _q(L, y=FAKE + 4) == 3
    assert _q(L, f=FAKE + 4) == 3                 # factors misaligned
    assert _q(L, m=0) == 0                        # empty: no-op
    assert _q(L, m=0, A=None, q=None, sf=None) == 0
    assert _q(L, variant=5) == 4
    assert _q(L, variant=4, f=None) == 1          # K2 builds from the factors
    assert _q(L, variant=4, f=FAKE + 4) == 3
    assert _q(L, variant=3, K=None) == 1
    assert _q(L, variant=1, K=FAKE) == 4         # the mma.sync variant is not built
    assert _q(L, variant=0, f=None) == 1


def test_baseline_argument_checks(L):
    assert L.kq_smooth_quantize_mxfp4(FAKE, 4, 64, 64, None, FAKE, 32, FAKE, 0, None, None) == 1
    assert L.kq_smooth_quantize_mxfp4(FAKE, 4, 64, 64, FAKE + 4, FAKE, 32, FAKE, 0, None, None) == 3
    assert L.kq_smooth_quantize_mxfp4(FAKE, 4, 60, 64, FAKE, FAKE, 32, FAKE, 0, None, None) == 2
    assert L.kq_hadamard_quantize_mxfp4(FAKE, 4, 64, 64, FAKE, 32, None, 0, None, None) == 1
    assert L.kq_hadamard_quantize_mxfp4(FAKE, 0, 64, 64, FAKE, 32, FAKE, 0, None, None) == 0


def test_aux_argument_checks(L):
    assert L.kq_dequantize(FAKE, 32, FAKE, 0, 4, 63, FAKE, None) == 2
    assert L.kq_dequantize(None, 32, FAKE, 0, 4, 64, FAKE, None) == 1
    assert L.kq_dequantize(FAKE, 32, FAKE, 2, 4, 64, FAKE, None) == 4
    assert L.kq_dequantize(FAKE, 32, FAKE, 0, 4, 64, FAKE + 4, None) == 3
    assert L.kq_expand_blocks(FAKE, 0, 0, FAKE, None) == 2
    assert L.kq_expand_blocks(FAKE, 4, 9, FAKE, None) == 4
    assert L.kq_expand_blocks(None, 4, 0, FAKE, None) == 1
    assert L.kq_test_encode_e2m1(0, 7, FAKE, None) == 2
    assert L.kq_test_encode_e2m1(0xFFFFFFF8, 16, FAKE, None) == 2
    assert L.kq_test_encode_e2m1(0, 0, None, None) == 0


def test_dual_argument_checks(L):
    """kq_quantize_mxfp4_dual validates before launching: the side output and
    the expanded blocks are required, 16-byte aligned, ldat >= d, ldat % 8 == 0.
    Every call here fails a check (or has m = 0), so nothing is launched."""
    vp = ctypes.c_void_p
    A, K, q, sf, at = vp(4096), vp(8192), vp(12288), vp(16384), vp(20480)
    f = L.kq_quantize_mxfp4_dual
    assert f(A, 4, 64, 64, K, q, 32, sf, 0, at, 32, None, None) == 2          # ldat < d
    assert f(A, 4, 64, 64, None, q, 32, sf, 0, at, 64, None, None) == 1       # no blocks
    assert f(A, 4, 64, 64, K, q, 32, sf, 0, None, 64, None, None) == 1        # no side output
    assert f(A, 4, 64, 64, K, q, 32, sf, 0, vp(20488), 64, None, None) == 3   # misaligned
    assert f(A, 4, 64, 64, K, q, 32, sf, 0, at, 68, None, None) == 3          # ldat % 8
    assert f(A, 0, 64, 64, None, None, 32, None, 0, None, 64, None, None) == 0  # m = 0


def test_fwht_argument_checks(L):
    """The full-row transform needs a power-of-two d in [128, 16384]; nothing
    is launched when a check fails."""
    vp = ctypes.c_void_p
    A, q, sf = vp(4096), vp(8192), vp(12288)
    f = L.kq_fwht_quantize_mxfp4
    for d in (96, 64, 3072, 32768):
        assert f(A, 4, d, d, q, d // 2, sf, 0, None, None) == 2, d
    assert f(A, 0, 1024, 1024, None, 512, None, 0, None, None) == 0


def test_gemm_argument_checks(L):
    """The W4A4 / bf16 products and the error sums validate before launching;
    every call here fails a check (or is empty), so nothing is launched."""
    vp = ctypes.c_void_p
    qa, sa, qw, sw, c = vp(4096), vp(8192), vp(12288), vp(16384), vp(20480)
    g = L.kq_w4a4_gemm
    assert g(qa, 32, sa, qw, 32, sw, 4, 8, 48, c, 8, None) == 2          # k % 32
    assert g(qa, 32, sa, qw, 32, sw, 4, 8, 0, c, 8, None) == 2           # k = 0
    assert g(qa, 16, sa, qw, 32, sw, 4, 8, 64, c, 8, None) == 2          # ldqa < k/2
    assert g(qa, 32, sa, qw, 32, sw, 4, 8, 64, c, 4, None) == 2          # ldc < n
    assert g(qa, 32, sa, qw, 32, sw, -1, 8, 64, c, 8, None) == 2
    assert g(None, 32, sa, qw, 32, sw, 4, 8, 64, c, 8, None) == 1
    assert g(qa, 32, None, qw, 32, sw, 4, 8, 64, c, 8, None) == 1
    assert g(qa, 32, sa, qw, 32, sw, 4, 8, 64, None, 8, None) == 1
    assert g(vp(4104), 32, sa, qw, 32, sw, 4, 8, 64, c, 8, None) == 3    # misaligned
    assert g(qa, 40, sa, qw, 32, sw, 4, 8, 64, c, 8, None) == 3          # ldqa % 16
    assert g(qa, 32, sa, qw, 32, sw, 4, 8, 64, c, 10, None) == 3         # ldc % 4
    assert L.kq_w4a4_gemm_variant(qa, 32, sa, qw, 32, sw, 4, 8, 64, c, 8, 4, None) == 4
    assert g(None, 32, None, None, 32, None, 0, 8, 64, None, 8, None) == 0   # m = 0
    assert g(None, 32, None, None, 32, None, 4, 0, 64, None, 0, None) == 0   # n = 0
    b = L.kq_bf16_gemm
    assert b(qa, 64, qw, 64, 4, 8, 0, c, 8, None) == 2
    assert b(qa, 32, qw, 64, 4, 8, 64, c, 8, None) == 2                  # lda < k
    assert b(qa, 68, qw, 64, 4, 8, 64, c, 8, None) == 3                  # lda % 8
    assert b(qa, 64, None, 64, 4, 8, 64, c, 8, None) == 1
    assert b(None, 64, None, 64, 0, 8, 64, None, 8, None) == 0
    e = L.kq_layer_error
    assert e(c, 8, c, 8, 4, 8, None, None) == 1                          # no out
    assert e(c, 8, c, 8, 4, 8, vp(4100), None) == 3                      # out misaligned
    assert e(c, 4, c, 8, 4, 8, vp(4096), None) == 2                      # ldc < n
    assert e(None, 8, c, 8, 4, 8, vp(4096), None) == 1
    assert e(c, 8, vp(20484), 8, 4, 8, vp(4096), None) == 3


def test_shared_argument_checks(L):
    """kq_quantize_mxfp4_shared needs the shared factors or their record;
    nothing is launched when a check fails."""
    vp = ctypes.c_void_p
    A, q, sf, F = vp(4096), vp(8192), vp(12288), vp(16384)
    f = L.kq_quantize_mxfp4_shared
    assert f(A, 4, 64, 64, None, None, q, 32, sf, 0, None, None) == 1
    assert f(A, 4, 64, 64, vp(16388), None, q, 32, sf, 0, None, None) == 3
    assert f(A, 4, 64, 64, None, vp(16392), q, 32, sf, 0, None, None) == 3
    assert f(A, 4, 48, 64, F, None, q, 32, sf, 0, None, None) == 2
    assert f(A, 0, 64, 64, None, None, q, 32, sf, 0, None, None) == 0


def test_ex_argument_checks(L):
    """kq_quantize_mxfp4_ex: format, transform and parameter checks, before
    any launch."""
    vp = ctypes.c_void_p
    A, q, sf, P = vp(4096), vp(8192), vp(12288), vp(16384)
    f = L.kq_quantize_mxfp4_ex
    assert f(A, 2, 4, 64, 64, 0, P, q, 32, sf, 0, None, None) == 4          # format
    assert f(A, 1, 4, 64, 64, 5, P, q, 32, sf, 0, None, None) == 4          # transform
    assert f(A, 1, 4, 64, 64, 0, None, q, 32, sf, 0, None, None) == 1       # kron needs factors
    assert f(A, 1, 4, 64, 64, 1, None, q, 32, sf, 0, None, None) == 1       # diag needs s
    assert f(A, 1, 4, 64, 64, 0, vp(16388), q, 32, sf, 0, None, None) == 3
    assert f(A, 1, 4, 64, 64, 4, None, q, 32, sf, 0, None, None) == 2       # fwht: d < 128
    assert f(A, 1, 4, 96, 96, 2, None, q, 56, sf, 0, None, None) == 3       # ldq % 16
    assert f(A, 1, 0, 64, 64, 0, None, q, 32, sf, 0, None, None) == 0       # m = 0


def test_stall_hook_argument_checks(L):
    """kq_test_quantize_stall takes a wait limit between 1 ms and 1 s and the
    checks of the tensor-core path; nothing launches when one fails."""
    vp = ctypes.c_void_p
    A, K, q, sf = vp(4096), vp(8192), vp(12288), vp(16384)
    h = L.kq_test_quantize_stall
    assert h(A, 4, 64, 64, K, q, 32, sf, 0, 0, 999_999, None) == 2          # limit < 1 ms
    assert h(A, 4, 64, 64, K, q, 32, sf, 0, 0, 2_000_000_000, None) == 2    # limit > 1 s
    assert h(A, 4, 64, 64, None, q, 32, sf, 0, 0, 10_000_000, None) == 1    # no blocks
    assert h(A, 4, 64, 64, vp(8200), q, 32, sf, 0, 0, 10_000_000, None) == 3  # blocks alignment
    assert h(A, 0, 64, 64, K, q, 32, sf, 0, 0, 10_000_000, None) == 0       # m = 0

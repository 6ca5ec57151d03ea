"""Thin Python binding of the C ABI in ``include/kq.h`` (ctypes).

Argument marshalling only: every step of the quantizer runs in the CUDA
library ``libkq_gb300.so``.  PyTorch provides device memory and streams.  The
functions keep the C names; tensor arguments are CUDA tensors, results are
written into caller-provided tensors or into tensors allocated here with
``torch.empty``.  A non-OK status raises :class:`KqError`.  If the library
has not been built, loading raises -- there is no other implementation to
fall back on.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkq_gb300.so")

KQ_OK = 0
KQ_SF_ROWMAJOR = 0
KQ_SF_BLOCKED_128x4 = 1
KQ_K_FP32 = 0
KQ_K_BF16X3 = 1
KQ_IN_BF16 = 0
KQ_IN_F16 = 1
KQ_TRANSFORM = {"kron": 0, "diag": 1, "hadamard": 2, "identity": 3, "fwht": 4}
VARIANT_BUTTERFLY = 0
VARIANT_IDENTITY = 2
VARIANT_UMMA = 3
VARIANT_K2 = 4          # tensor cores, operand records built in the kernel from the factors

# the functions include/kq.h declares, then those of include/kq_testing.h
EXPORTS = (
    "kq_quantize_mxfp4", "kq_smooth_quantize_mxfp4", "kq_hadamard_quantize_mxfp4",
    "kq_expand_blocks", "kq_expanded_bytes", "kq_dequantize", "kq_sf_bytes",
    "kq_status_string", "kq_lu_to_factors", "kq_invert_transpose_factors",
    "kq_quantize_mxfp4_dual",
    "kq_fwht_quantize_mxfp4", "kq_w4a4_gemm", "kq_bf16_gemm",
    "kq_layer_error", "kq_quantize_mxfp4_shared", "kq_quantize_mxfp4_ex",
)
TESTING_EXPORTS = (
    "kq_quantize_mxfp4_variant", "kq_w4a4_gemm_variant", "kq_test_encode_e2m1",
    "kq_test_quantize_stall",
)


class KqError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({status_string(status)})")


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """Load the library (once).  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                    "g.build()'` (nvcc, sm_103a)")
            L = ctypes.CDLL(LIB_PATH)
            i64, vp, u32, f32p = ctypes.c_int64, ctypes.c_void_p, ctypes.c_uint32, ctypes.c_void_p
            st = ctypes.c_int
            L.kq_quantize_mxfp4.argtypes = [vp, i64, i64, i64, vp, vp, vp, i64, vp, st, vp, vp]
            L.kq_quantize_mxfp4.restype = st
            L.kq_quantize_mxfp4_variant.argtypes = [vp, i64, i64, i64, vp, vp, vp, i64, vp, st, vp,
                                                    st, vp]
            L.kq_quantize_mxfp4_variant.restype = st
            L.kq_quantize_mxfp4_dual.argtypes = [vp, i64, i64, i64, vp, vp, i64, vp, st, vp, i64,
                                                 vp, vp]
            L.kq_quantize_mxfp4_dual.restype = st
            L.kq_test_quantize_stall.argtypes = [vp, i64, i64, i64, vp, vp, i64, vp, st, i64,
                                                 ctypes.c_uint64, vp]
            L.kq_test_quantize_stall.restype = st
            L.kq_quantize_mxfp4_shared.argtypes = [vp, i64, i64, i64, vp, vp, vp, i64, vp, st, vp,
                                                   vp]
            L.kq_quantize_mxfp4_shared.restype = st
            L.kq_quantize_mxfp4_ex.argtypes = [vp, st, i64, i64, i64, st, vp, vp, i64, vp, st, vp,
                                               vp]
            L.kq_quantize_mxfp4_ex.restype = st
            L.kq_smooth_quantize_mxfp4.argtypes = [vp, i64, i64, i64, vp, vp, i64, vp, st, vp, vp]
            L.kq_smooth_quantize_mxfp4.restype = st
            L.kq_hadamard_quantize_mxfp4.argtypes = [vp, i64, i64, i64, vp, i64, vp, st, vp, vp]
            L.kq_fwht_quantize_mxfp4.argtypes = [vp, i64, i64, i64, vp, i64, vp, st, vp, vp]
            L.kq_fwht_quantize_mxfp4.restype = st
            L.kq_hadamard_quantize_mxfp4.restype = st
            L.kq_expand_blocks.argtypes = [vp, i64, st, vp, vp]
            L.kq_expand_blocks.restype = st
            L.kq_expanded_bytes.argtypes = [i64, st]
            L.kq_expanded_bytes.restype = ctypes.c_size_t
            L.kq_dequantize.argtypes = [vp, i64, vp, st, i64, i64, vp, vp]
            L.kq_dequantize.restype = st
            L.kq_sf_bytes.argtypes = [i64, i64, st]
            L.kq_sf_bytes.restype = ctypes.c_size_t
            L.kq_status_string.argtypes = [st]
            L.kq_status_string.restype = ctypes.c_char_p
            L.kq_lu_to_factors.argtypes = [f32p, i64, st, f32p]
            L.kq_lu_to_factors.restype = st
            L.kq_invert_transpose_factors.argtypes = [f32p, i64, f32p]
            L.kq_invert_transpose_factors.restype = st
            L.kq_test_encode_e2m1.argtypes = [u32, i64, vp, vp]
            L.kq_test_encode_e2m1.restype = st
            L.kq_w4a4_gemm.argtypes = [vp, i64, vp, vp, i64, vp, i64, i64, i64, vp, i64, vp]
            L.kq_w4a4_gemm.restype = st
            L.kq_w4a4_gemm_variant.argtypes = [vp, i64, vp, vp, i64, vp, i64, i64, i64, vp, i64, st,
                                               vp]
            L.kq_w4a4_gemm_variant.restype = st
            L.kq_bf16_gemm.argtypes = [vp, i64, vp, i64, i64, i64, i64, vp, i64, vp]
            L.kq_bf16_gemm.restype = st
            L.kq_layer_error.argtypes = [vp, i64, vp, i64, i64, i64, vp, vp]
            L.kq_layer_error.restype = st
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().kq_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != KQ_OK:
        raise KqError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _bf16_bits(A):
    import torch
    if A.dtype == torch.bfloat16:
        return A
    if A.dtype in (torch.int16, torch.uint16):
        return A
    raise TypeError("A must be bfloat16 (or its 16-bit patterns)")


# --- sizes and host helpers ------------------------------------------------------

def kq_sf_bytes(m: int, d: int, layout: int = KQ_SF_ROWMAJOR) -> int:
    return int(lib().kq_sf_bytes(m, d, layout))


def kq_expanded_bytes(nb: int, fmt: int) -> int:
    return int(lib().kq_expanded_bytes(nb, fmt))


def kq_lu_to_factors(lu: np.ndarray, det_sign: int) -> np.ndarray:
    """Host: LU parameters fp32 [nb, 5, 3] -> raw factors fp32 [nb, 5, 2, 2]."""
    lu = np.ascontiguousarray(lu, dtype=np.float32)
    nb = lu.shape[0]
    out = np.empty((nb, 5, 2, 2), np.float32)
    _check(lib().kq_lu_to_factors(lu.ctypes.data, nb, det_sign, out.ctypes.data),
           "kq_lu_to_factors")
    return out


def kq_invert_transpose_factors(factors: np.ndarray) -> np.ndarray:
    """Host: factors of K^{-T} (for the weight side W T^{-T})."""
    f = np.ascontiguousarray(factors, dtype=np.float32)
    nb = f.shape[0]
    out = np.empty_like(f)
    _check(lib().kq_invert_transpose_factors(f.ctypes.data, nb, out.ctypes.data),
           "kq_invert_transpose_factors")
    return out


# --- device entry points -------------------------------------------------------------

def _outputs(A, m, d, layout, q, sf, y_debug):
    import torch
    dev = A.device
    if q is None:
        q = torch.empty((m, d // 2), dtype=torch.uint8, device=dev)
    if sf is None:
        sf = torch.empty(max(kq_sf_bytes(m, d, layout), 16), dtype=torch.uint8, device=dev)
    if y_debug is True:
        y_debug = torch.empty((m, d), dtype=torch.float32, device=dev)
    elif y_debug is False:
        y_debug = None
    return q, sf, y_debug


def kq_quantize_mxfp4(A, d: int | None = None, factors=None, K_expanded=None,
                      layout: int = KQ_SF_ROWMAJOR, q=None, sf=None, y_debug=None,
                      variant: int | None = None, stream=None):
    """Quantize A (bf16 [m, lda] CUDA tensor, first d columns).  Returns
    (q, sf, y_debug).  ``y_debug=True`` allocates the fp32 debug output."""
    A = _bf16_bits(A)
    m, lda = A.shape
    d = lda if d is None else d
    q, sf, y_debug = _outputs(A, m, d, layout, q, sf, y_debug)
    ldq = q.shape[1] if q.dim() == 2 else d // 2
    args = (_ptr(A), m, d, A.stride(0), _ptr(factors), _ptr(K_expanded), _ptr(q), ldq, _ptr(sf),
            layout, _ptr(y_debug))
    if variant is None:
        _check(lib().kq_quantize_mxfp4(*args, _stream(stream)), "kq_quantize_mxfp4")
    else:
        _check(lib().kq_quantize_mxfp4_variant(*args, variant, _stream(stream)),
               "kq_quantize_mxfp4_variant")
    return q, sf, y_debug


def kq_quantize_mxfp4_dual(A, K_expanded, d: int | None = None, layout: int = KQ_SF_ROWMAJOR,
                           q=None, sf=None, at=None, y_debug=None, stream=None):
    """Quantize A on the tensor-core path and also write the bf16 side output
    A T.  Returns (q, sf, at, y_debug); ``at`` is allocated as bf16 [m, d]
    when not given."""
    import torch
    A = _bf16_bits(A)
    m, lda = A.shape
    d = lda if d is None else d
    q, sf, y_debug = _outputs(A, m, d, layout, q, sf, y_debug)
    if at is None:
        at = torch.empty((m, d), dtype=torch.bfloat16, device=A.device)
    ldq = q.shape[1] if q.dim() == 2 else d // 2
    ldat = at.stride(0) if at.dim() == 2 else d
    _check(lib().kq_quantize_mxfp4_dual(_ptr(A), m, d, A.stride(0), _ptr(K_expanded), _ptr(q), ldq,
                                        _ptr(sf), layout, _ptr(at), ldat, _ptr(y_debug),
                                        _stream(stream)),
           "kq_quantize_mxfp4_dual")
    return q, sf, at, y_debug


def kq_test_quantize_stall(A, K_expanded, d: int, skip_tile: int, wait_limit_ns: int,
                           layout: int = KQ_SF_ROWMAJOR, q=None, sf=None, stream=None):
    """Verification hook: the tensor-core quantizer with tile ``skip_tile``'s
    loads never issued and every wait bounded by ``wait_limit_ns``.
    Returns (q, sf)."""
    A = _bf16_bits(A)
    m, lda = A.shape
    q, sf, _ = _outputs(A, m, d, layout, q, sf, None)
    ldq = q.shape[1] if q.dim() == 2 else d // 2
    _check(lib().kq_test_quantize_stall(_ptr(A), m, d, A.stride(0), _ptr(K_expanded), _ptr(q), ldq,
                                        _ptr(sf), layout, skip_tile, wait_limit_ns,
                                        _stream(stream)),
           "kq_test_quantize_stall")
    return q, sf


def kq_quantize_mxfp4_shared(A, d: int | None = None, factors=None, K_expanded=None,
                             layout: int = KQ_SF_ROWMAJOR, q=None, sf=None, y_debug=None,
                             stream=None):
    """Quantize A with one factor set ([5, 2, 2] fp32 CUDA tensor, or its
    expanded record from kq_expand_blocks(factors[None], KQ_K_BF16X3)) shared
    by every block.  Returns (q, sf, y_debug)."""
    A = _bf16_bits(A)
    m, lda = A.shape
    d = lda if d is None else d
    q, sf, y_debug = _outputs(A, m, d, layout, q, sf, y_debug)
    ldq = q.shape[1] if q.dim() == 2 else d // 2
    _check(lib().kq_quantize_mxfp4_shared(_ptr(A), m, d, A.stride(0), _ptr(factors),
                                          _ptr(K_expanded), _ptr(q), ldq, _ptr(sf), layout,
                                          _ptr(y_debug), _stream(stream)),
           "kq_quantize_mxfp4_shared")
    return q, sf, y_debug


def kq_quantize_mxfp4_ex(A, transform: str, param=None, d: int | None = None,
                         in_format: int = KQ_IN_BF16, layout: int = KQ_SF_ROWMAJOR, q=None,
                         sf=None, y_debug=None, stream=None):
    """CUDA-core quantizer with the input format chosen: A holds bf16 or
    fp16 16-bit patterns ([m, lda] CUDA tensor of dtype bfloat16, float16,
    int16 or uint16); transform in KQ_TRANSFORM.  Returns (q, sf, y_debug)."""
    import torch
    if A.dtype not in (torch.bfloat16, torch.float16, torch.int16, torch.uint16):
        raise TypeError("A must hold 16-bit patterns")
    m, lda = A.shape
    d = lda if d is None else d
    q, sf, y_debug = _outputs(A, m, d, layout, q, sf, y_debug)
    ldq = q.shape[1] if q.dim() == 2 else d // 2
    _check(lib().kq_quantize_mxfp4_ex(_ptr(A), in_format, m, d, A.stride(0),
                                      KQ_TRANSFORM[transform], _ptr(param), _ptr(q), ldq,
                                      _ptr(sf), layout, _ptr(y_debug), _stream(stream)),
           "kq_quantize_mxfp4_ex")
    return q, sf, y_debug


def kq_smooth_quantize_mxfp4(A, s, d: int | None = None, layout: int = KQ_SF_ROWMAJOR, q=None,
                             sf=None, y_debug=None, stream=None):
    A = _bf16_bits(A)
    m, lda = A.shape
    d = lda if d is None else d
    q, sf, y_debug = _outputs(A, m, d, layout, q, sf, y_debug)
    ldq = q.shape[1] if q.dim() == 2 else d // 2
    _check(lib().kq_smooth_quantize_mxfp4(_ptr(A), m, d, A.stride(0), _ptr(s), _ptr(q), ldq,
                                          _ptr(sf), layout, _ptr(y_debug), _stream(stream)),
           "kq_smooth_quantize_mxfp4")
    return q, sf, y_debug


def kq_hadamard_quantize_mxfp4(A, d: int | None = None, layout: int = KQ_SF_ROWMAJOR, q=None,
                               sf=None, y_debug=None, stream=None):
    A = _bf16_bits(A)
    m, lda = A.shape
    d = lda if d is None else d
    q, sf, y_debug = _outputs(A, m, d, layout, q, sf, y_debug)
    ldq = q.shape[1] if q.dim() == 2 else d // 2
    _check(lib().kq_hadamard_quantize_mxfp4(_ptr(A), m, d, A.stride(0), _ptr(q), ldq, _ptr(sf),
                                            layout, _ptr(y_debug), _stream(stream)),
           "kq_hadamard_quantize_mxfp4")
    return q, sf, y_debug


def kq_fwht_quantize_mxfp4(A, d: int | None = None, layout: int = KQ_SF_ROWMAJOR, q=None,
                           sf=None, y_debug=None, stream=None):
    """Full-row Walsh-Hadamard baseline (d a power of two, 128..16384)."""
    A = _bf16_bits(A)
    m, lda = A.shape
    d = lda if d is None else d
    q, sf, y_debug = _outputs(A, m, d, layout, q, sf, y_debug)
    ldq = q.shape[1] if q.dim() == 2 else d // 2
    _check(lib().kq_fwht_quantize_mxfp4(_ptr(A), m, d, A.stride(0), _ptr(q), ldq, _ptr(sf),
                                        layout, _ptr(y_debug), _stream(stream)),
           "kq_fwht_quantize_mxfp4")
    return q, sf, y_debug


def kq_expand_blocks(factors, fmt: int = KQ_K_FP32, out=None, stream=None):
    """factors: fp32 CUDA tensor [nb, 5, 2, 2] -> expanded blocks (uint8 bytes
    tensor of kq_expanded_bytes, or the caller's ``out``)."""
    import torch
    nb = factors.shape[0]
    if out is None:
        out = torch.empty(kq_expanded_bytes(nb, fmt), dtype=torch.uint8, device=factors.device)
    _check(lib().kq_expand_blocks(_ptr(factors), nb, fmt, _ptr(out), _stream(stream)),
           "kq_expand_blocks")
    return out


def kq_dequantize(q, sf, m: int, d: int, layout: int = KQ_SF_ROWMAJOR, out=None, stream=None):
    import torch
    if out is None:
        out = torch.empty((m, d), dtype=torch.float32, device=q.device)
    ldq = q.shape[1] if q.dim() == 2 else d // 2
    _check(lib().kq_dequantize(_ptr(q), ldq, _ptr(sf), layout, m, d, _ptr(out), _stream(stream)),
           "kq_dequantize")
    return out


def kq_test_encode_e2m1(first: int, count: int, out=None, stream=None):
    import torch
    if out is None:
        out = torch.empty(count // 2, dtype=torch.uint8, device="cuda")
    _check(lib().kq_test_encode_e2m1(first, count, _ptr(out), _stream(stream)),
           "kq_test_encode_e2m1")
    return out


# --- the consumer product of eq. (11) and the layer error of eq. (2) ---------------

def _ld(t, default):
    return t.stride(0) if t.dim() == 2 else default


def _gemm_out(m, n, device):
    """fp32 [m, n] view of a buffer whose row pitch is a multiple of 4."""
    import torch
    ldc = n + (-n) % 4
    return torch.empty((m, ldc), dtype=torch.float32, device=device)[:, :n]


GEMM_MXF4 = 0
GEMM_DEQUANT_BF16 = 1
GEMM_MXF4_NARROW = 2
GEMM_MXF4_WIDE = 3


def kq_w4a4_gemm(qa, sfa, qw, sfw, m: int, n: int, k: int, c=None, variant: int | None = None,
                 stream=None):
    """C = deq(qa) deq(qw)^T (fp32 [m, n]) from packed codes and 128x4 tiled
    scales, on the tensor cores (``variant``: GEMM_MXF4, GEMM_DEQUANT_BF16,
    GEMM_MXF4_NARROW or GEMM_MXF4_WIDE; None = the library's default)."""
    if c is None:
        c = _gemm_out(m, n, qa.device)
    args = (_ptr(qa), _ld(qa, k // 2), _ptr(sfa), _ptr(qw), _ld(qw, k // 2), _ptr(sfw), m, n, k,
            _ptr(c), _ld(c, n))
    if variant is None:
        _check(lib().kq_w4a4_gemm(*args, _stream(stream)), "kq_w4a4_gemm")
    else:
        _check(lib().kq_w4a4_gemm_variant(*args, variant, _stream(stream)), "kq_w4a4_gemm_variant")
    return c


def kq_bf16_gemm(a, w, k: int | None = None, c=None, stream=None):
    """C = A W^T (fp32 [m, n]) for bf16 A [m, k] and W [n, k]."""
    a, w = _bf16_bits(a), _bf16_bits(w)
    m, n = a.shape[0], w.shape[0]
    k = a.shape[1] if k is None else k
    if c is None:
        c = _gemm_out(m, n, a.device)
    _check(lib().kq_bf16_gemm(_ptr(a), a.stride(0), _ptr(w), w.stride(0), m, n, k, _ptr(c),
                              _ld(c, n), _stream(stream)),
           "kq_bf16_gemm")
    return c


def kq_layer_error(c, c_ref, out=None, stream=None):
    """fp64 device [sum (c - c_ref)^2, sum c_ref^2] for fp32 [m, n] c, c_ref."""
    import torch
    m, n = c_ref.shape
    if out is None:
        out = torch.empty(2, dtype=torch.float64, device=c_ref.device)
    _check(lib().kq_layer_error(_ptr(c), c.stride(0), _ptr(c_ref), c_ref.stride(0), m, n,
                                _ptr(out), _stream(stream)),
           "kq_layer_error")
    return out

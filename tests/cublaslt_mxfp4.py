"""Test-only consumer of the quantizer's output: the MX block-scaled GEMM of
cuBLASLt (a library routine), called through ctypes.

It computes C[m][n] = sum_k A[m][k] * B[n][k] with A and B given as K-major
elements -- packed E2M1 codes ([rows][k/2] bytes, two per byte) or E4M3
bytes ([rows][k]) -- and E8M0 scales of 32-element blocks in the 128x4 tiled
layout of block-scaled MMA (cuBLASLt's CUBLASLT_MATMUL_MATRIX_SCALE_VEC32_UE8M0;
the same layout for MXFP4 and MXFP8).  The tests hand it the library's own
scales, so NVIDIA's reading of the tiled layout checks ours.  Enum values are
those of the CUDA 13 headers (library_types.h, cublasLt.h).
"""
import ctypes
import ctypes.util
import glob
import os

CUDA_R_32F, CUDA_R_16BF, CUDA_R_8F_E4M3, CUDA_R_4F_E2M1 = 0, 14, 28, 33
CUBLAS_COMPUTE_32F = 68
DESC_TRANSA, DESC_TRANSB = 3, 4
DESC_A_SCALE_POINTER, DESC_B_SCALE_POINTER = 17, 18
DESC_A_SCALE_MODE, DESC_B_SCALE_MODE = 31, 32
SCALE_VEC32_UE8M0 = 2
PREF_MAX_WORKSPACE_BYTES = 1
OP_N, OP_T = 0, 1


class _Heuristic(ctypes.Structure):
    _fields_ = [("algo", ctypes.c_uint64 * 8), ("workspaceSize", ctypes.c_size_t),
                ("state", ctypes.c_int), ("wavesCount", ctypes.c_float),
                ("reserved", ctypes.c_int * 4)]


def _load():
    names = [ctypes.util.find_library("cublasLt")]
    names += sorted(glob.glob("/usr/local/cuda/lib64/libcublasLt.so*"))
    try:
        import torch
        names += sorted(glob.glob(os.path.join(os.path.dirname(torch.__file__), "lib",
                                               "libcublasLt.so*")))
    except ImportError:
        pass
    for n in names:
        if not n:
            continue
        try:
            L = ctypes.CDLL(n)
        except OSError:
            continue
        vp, i32, u64, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_int64
        L.cublasLtCreate.argtypes = [ctypes.POINTER(vp)]
        L.cublasLtDestroy.argtypes = [vp]
        L.cublasLtMatmulDescCreate.argtypes = [ctypes.POINTER(vp), i32, i32]
        L.cublasLtMatmulDescDestroy.argtypes = [vp]
        L.cublasLtMatmulDescSetAttribute.argtypes = [vp, i32, vp, ctypes.c_size_t]
        L.cublasLtMatrixLayoutCreate.argtypes = [ctypes.POINTER(vp), i32, u64, u64, i64]
        L.cublasLtMatrixLayoutDestroy.argtypes = [vp]
        L.cublasLtMatmulPreferenceCreate.argtypes = [ctypes.POINTER(vp)]
        L.cublasLtMatmulPreferenceDestroy.argtypes = [vp]
        L.cublasLtMatmulPreferenceSetAttribute.argtypes = [vp, i32, vp, ctypes.c_size_t]
        L.cublasLtMatmulAlgoGetHeuristic.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32,
                                                     ctypes.POINTER(_Heuristic),
                                                     ctypes.POINTER(i32)]
        L.cublasLtMatmul.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                     ctypes.POINTER(_Heuristic), vp, ctypes.c_size_t, vp]
        return L
    return None


def mx_gemm(qa, sfa, m, qb, sfb, n, k, out, out_type, workspace, ws_bytes, stream,
            elem_type=CUDA_R_4F_E2M1):
    """C = A . B^T into out (row-major [m][n] of out_type); every pointer is a
    device address (int), elements of elem_type.  Returns None on success,
    else the reason the library declined (nothing is launched then)."""
    L = _load()
    if L is None:
        return "libcublasLt not found"
    vp = ctypes.c_void_p
    h, desc, pref = vp(), vp(), vp()
    lay = [vp() for _ in range(3)]
    try:
        if L.cublasLtCreate(ctypes.byref(h)) != 0:
            return "cublasLtCreate failed"
        if L.cublasLtMatmulDescCreate(ctypes.byref(desc), CUBLAS_COMPUTE_32F, CUDA_R_32F) != 0:
            return "cublasLtMatmulDescCreate failed"

        def setattr_(attr, cval):
            return L.cublasLtMatmulDescSetAttribute(desc, attr, ctypes.cast(ctypes.byref(cval), vp),
                                                    ctypes.sizeof(cval))
        # column-major view: D (n x m) = Bw^T (n x k) . Aa (k x m); both stored K-contiguous
        for attr, val in ((DESC_TRANSA, ctypes.c_int32(OP_T)), (DESC_TRANSB, ctypes.c_int32(OP_N)),
                          (DESC_A_SCALE_MODE, ctypes.c_int32(SCALE_VEC32_UE8M0)),
                          (DESC_B_SCALE_MODE, ctypes.c_int32(SCALE_VEC32_UE8M0)),
                          (DESC_A_SCALE_POINTER, vp(sfb)), (DESC_B_SCALE_POINTER, vp(sfa))):
            if setattr_(attr, val) != 0:
                return f"matmul attribute {attr} rejected"
        if (L.cublasLtMatrixLayoutCreate(ctypes.byref(lay[0]), elem_type, k, n, k) or
                L.cublasLtMatrixLayoutCreate(ctypes.byref(lay[1]), elem_type, k, m, k) or
                L.cublasLtMatrixLayoutCreate(ctypes.byref(lay[2]), out_type, n, m, n)):
            return "matrix layout rejected"
        if L.cublasLtMatmulPreferenceCreate(ctypes.byref(pref)) != 0:
            return "preference create failed"
        wsb = ctypes.c_uint64(ws_bytes)
        L.cublasLtMatmulPreferenceSetAttribute(pref, PREF_MAX_WORKSPACE_BYTES,
                                               ctypes.cast(ctypes.byref(wsb), vp), 8)
        res, cnt = _Heuristic(), ctypes.c_int(0)
        st = L.cublasLtMatmulAlgoGetHeuristic(h, desc, lay[0], lay[1], lay[2], lay[2], pref, 1,
                                              ctypes.byref(res), ctypes.byref(cnt))
        if st != 0 or cnt.value < 1:
            return f"no algorithm (status {st}, count {cnt.value})"
        alpha, beta = ctypes.c_float(1.0), ctypes.c_float(0.0)
        st = L.cublasLtMatmul(h, desc, ctypes.cast(ctypes.byref(alpha), vp), vp(qb), lay[0],
                              vp(qa), lay[1], ctypes.cast(ctypes.byref(beta), vp), vp(out), lay[2],
                              vp(out), lay[2], ctypes.byref(res), vp(workspace), ws_bytes,
                              vp(stream))
        return None if st == 0 else f"cublasLtMatmul status {st}"
    finally:
        for x in lay:
            if x.value:
                L.cublasLtMatrixLayoutDestroy(x)
        if pref.value:
            L.cublasLtMatmulPreferenceDestroy(pref)
        if desc.value:
            L.cublasLtMatmulDescDestroy(desc)
        if h.value:
            L.cublasLtDestroy(h)

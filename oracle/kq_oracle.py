"""KroQuant MXFP4 activation quantizer -- CPU reference ("oracle"), Python side.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It never imports the
CUDA library or its binding; the only code the two sides share is the seeded
input generator, which holds none of the method's arithmetic.

The arithmetic lives in ``kq_oracle.c`` (fp64, OpenMP over rows); this module
compiles it with gcc, loads it with ctypes and wraps it for numpy arrays.
Citations ([KQ] + section / equation) refer to "KroQuant: Kronecker-Structured
Block Transforms for Efficient Post-Training Quantization of Diffusion
Transformers" (arXiv 2607.21446v1).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libkq_oracle.so")

SF_ROWMAJOR = 0
SF_BLOCKED_128x4 = 1

FLAG_MIDPOINT = 1
FLAG_POW2_EDGE = 2
FLAG_ZERO_SIGN = 4

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build/libkq_oracle.so``.

    ``-ffp-contract=off`` keeps every fp64 operation a separately rounded IEEE
    operation on both x86-64 and aarch64 (no fused multiply-add contraction),
    so the oracle gives the same bits on every host.
    """
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-std=c11", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _bind(path: str) -> ctypes.CDLL:
    L = ctypes.CDLL(path)
    i64, dp, u8p, u16p = (ctypes.c_int64, ctypes.POINTER(ctypes.c_double),
                          ctypes.POINTER(ctypes.c_uint8), ctypes.POINTER(ctypes.c_uint16))
    L.kqo_bf16_to_f64.argtypes = [ctypes.c_uint16]
    L.kqo_bf16_to_f64.restype = ctypes.c_double
    L.kqo_f16_to_f64.argtypes = [ctypes.c_uint16]
    L.kqo_f16_to_f64.restype = ctypes.c_double
    L.kqo_set_input_format.argtypes = [ctypes.c_int]
    L.kqo_lu_to_factor.argtypes = [dp, ctypes.c_int, dp]
    L.kqo_expand_block.argtypes = [dp, dp]
    L.kqo_hadamard_block.argtypes = [dp]
    L.kqo_transform_dense.argtypes = [u16p, i64, i64, i64, dp, dp, dp]
    L.kqo_transform_kron.argtypes = [u16p, i64, i64, i64, dp, dp, dp, dp]
    L.kqo_transform_hadamard.argtypes = [u16p, i64, i64, i64, dp, dp, dp]
    L.kqo_transform_diag.argtypes = [u16p, i64, i64, i64, dp, dp, dp]
    L.kqo_transform_identity.argtypes = [u16p, i64, i64, i64, dp, dp]
    L.kqo_transform_fwht.argtypes = [u16p, i64, i64, i64, dp, dp]
    L.kqo_e8m0_exponent.argtypes = [ctypes.c_double]
    L.kqo_e8m0_exponent.restype = ctypes.c_int
    L.kqo_e2m1_value.argtypes = [ctypes.c_uint8]
    L.kqo_e2m1_value.restype = ctypes.c_double
    L.kqo_encode_e2m1.argtypes = [ctypes.c_double]
    L.kqo_encode_e2m1.restype = ctypes.c_uint8
    L.kqo_sf_offset.argtypes = [i64, i64, i64, ctypes.c_int]
    L.kqo_sf_offset.restype = i64
    L.kqo_sf_bytes.argtypes = [i64, i64, ctypes.c_int]
    L.kqo_sf_bytes.restype = i64
    L.kqo_sf_place.argtypes = [u8p, i64, i64, ctypes.c_int, ctypes.c_uint8, u8p]
    L.kqo_quantize.argtypes = [dp, dp, i64, i64, u8p, i64, u8p, ctypes.c_int, u8p]
    L.kqo_dequantize.argtypes = [u8p, i64, u8p, ctypes.c_int, i64, i64, dp]
    L.kqo_encode_f32_range.argtypes = [ctypes.c_uint32, i64, u8p]
    L.kqo_encode_e2m1_array.argtypes = [dp, i64, u8p]
    L.kqo_f64_to_bf16.argtypes = [ctypes.c_double]
    L.kqo_f64_to_bf16.restype = ctypes.c_uint16
    L.kqo_f64_to_bf16_array.argtypes = [dp, i64, u16p]
    return L


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


class swapped_library:
    """Context manager: run the oracle functions on another build of the C
    source (used by the tests that plant a mistake in a copy of the oracle
    and check that the pins catch it)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        lib()
        self._saved = _lib
        _lib = _bind(self.path)
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def build_variant(src_text: str, out_path: str) -> str:
    """Compile a modified copy of the C source (for planted-mistake tests)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                    "-shared", "-std=c11", "-o", out_path, src, "-lm"], check=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _p(a: np.ndarray, ctype):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _bits(A: np.ndarray) -> np.ndarray:
    A = np.ascontiguousarray(A)
    assert A.dtype == np.uint16 and A.ndim == 2, "A must be bf16 bit patterns [m][lda]"
    return A


# --- [KQ] Sec. 3.2 -----------------------------------------------------------

def lu_to_factors(lu: np.ndarray, det_sign: int) -> np.ndarray:
    """eq. (6): LU parameters (a, b, c) [..., 3] -> raw 2x2 entries [..., 2, 2].

    Computed in fp64 from the given parameters, returned in fp64 (round with
    ``.astype(np.float32)`` to get the fp32 entries a kernel consumes)."""
    lu = _f64(lu)
    flat = lu.reshape(-1, 3)
    out = np.empty((flat.shape[0], 4), np.float64)
    L = lib()
    for k in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[k])
        g = np.empty(4, np.float64)
        L.kqo_lu_to_factor(_p(row, ctypes.c_double), int(det_sign), _p(g, ctypes.c_double))
        out[k] = g
    return out.reshape(lu.shape[:-1] + (2, 2))


def expand_block(G: np.ndarray) -> np.ndarray:
    """eq. (12): five 2x2 factors [5, 2, 2] -> dense K [32, 32] (fp64)."""
    G = _f64(G).reshape(5, 2, 2)
    K = np.empty((32, 32), np.float64)
    lib().kqo_expand_block(_p(G, ctypes.c_double), _p(K, ctypes.c_double))
    return K


def expand_blocks(factors: np.ndarray) -> np.ndarray:
    """[nb, 5, 2, 2] -> [nb, 32, 32]."""
    f = _f64(factors).reshape(-1, 5, 2, 2)
    return np.stack([expand_block(f[j]) for j in range(f.shape[0])]) if f.shape[0] else \
        np.zeros((0, 32, 32))


def hadamard_block() -> np.ndarray:
    K = np.empty((32, 32), np.float64)
    lib().kqo_hadamard_block(_p(K, ctypes.c_double))
    return K


# --- transforms: y = a . K_j per 32-block (eq. 4) ------------------------------

_format_lock = threading.Lock()


def f16_to_f64(h: int) -> float:
    """fp16 bit pattern -> its value (IEEE 754 binary16)."""
    return float(lib().kqo_f16_to_f64(int(h)))


def transform(A: np.ndarray, d: int, kind: str, param=None, in_format: str = "bf16"):
    """Return (y, bound), both fp64 [m, d].

    kind: 'kron' (param = factors [nb, 5, 2, 2]), 'dense' (param = [nb, 32, 32]),
    'hadamard', 'diag' (param = s [d]), 'identity', 'fwht' (full-row
    Walsh-Hadamard, d a power of two).  in_format: 'bf16' or 'f16', the
    format of A's 16-bit patterns.
    ``bound[i, c] = sum_r |a_r K_rc|`` is the scale the 2^-16 rule uses."""
    if in_format not in ("bf16", "f16"):
        raise ValueError(in_format)
    with _format_lock:
        lib().kqo_set_input_format(1 if in_format == "f16" else 0)
        try:
            return _transform(A, d, kind, param)
        finally:
            lib().kqo_set_input_format(0)


def _transform(A: np.ndarray, d: int, kind: str, param=None):
    A = _bits(A)
    m, lda = A.shape
    assert d % 32 == 0 and d <= lda
    nb = d // 32
    y = np.empty((m, d), np.float64)
    bound = np.empty((m, d), np.float64)
    L = lib()
    Ap = _p(A, ctypes.c_uint16)
    yp, bp = _p(y, ctypes.c_double), _p(bound, ctypes.c_double)
    if kind == "kron":
        f = _f64(param).reshape(nb, 5, 2, 2)
        Ks = np.empty((max(nb, 1), 32, 32), np.float64)
        L.kqo_transform_kron(Ap, m, d, lda, _p(f, ctypes.c_double), _p(Ks, ctypes.c_double), yp, bp)
    elif kind == "dense":
        K = _f64(param).reshape(nb, 32, 32)
        L.kqo_transform_dense(Ap, m, d, lda, _p(K, ctypes.c_double), yp, bp)
    elif kind == "hadamard":
        Ks = np.empty((max(nb, 1), 32, 32), np.float64)
        L.kqo_transform_hadamard(Ap, m, d, lda, _p(Ks, ctypes.c_double), yp, bp)
    elif kind == "diag":
        s = _f64(param).reshape(d)
        L.kqo_transform_diag(Ap, m, d, lda, _p(s, ctypes.c_double), yp, bp)
    elif kind == "identity":
        L.kqo_transform_identity(Ap, m, d, lda, yp, bp)
    elif kind == "fwht":
        assert d & (d - 1) == 0, "the full-row transform needs a power-of-two d"
        L.kqo_transform_fwht(Ap, m, d, lda, yp, bp)
    else:
        raise ValueError(kind)
    return y, bound


# --- MXFP4 quantizer (Sec. 3.1; OCP MX) ----------------------------------------

def e8m0_exponent(amax: float) -> int:
    return int(lib().kqo_e8m0_exponent(float(amax)))


def encode_e2m1(v: float) -> int:
    return int(lib().kqo_encode_e2m1(float(v)))


def encode_e2m1_array(v: np.ndarray) -> np.ndarray:
    v = _f64(v).ravel()
    out = np.empty(v.size, np.uint8)
    lib().kqo_encode_e2m1_array(_p(v, ctypes.c_double), v.size, _p(out, ctypes.c_uint8))
    return out


def round_bf16(x) -> np.ndarray:
    """fp64 values -> bf16 bit patterns (uint16), round to nearest even: the
    cast of the transformed activations to the 16-bit input dtype ([KQ] Sec.
    3.5.1 K1, App. D "Quantization": the low-rank branch of eq. (11) takes A T
    in 16 bits)."""
    x = _f64(x)
    flat = x.ravel()
    out = np.empty(flat.size, np.uint16)
    lib().kqo_f64_to_bf16_array(_p(flat, ctypes.c_double), flat.size, _p(out, ctypes.c_uint16))
    return out.reshape(x.shape)


def e2m1_value(code: int) -> float:
    return float(lib().kqo_e2m1_value(int(code)))


def sf_offset(i: int, kb: int, nb: int, layout: int) -> int:
    return int(lib().kqo_sf_offset(i, kb, nb, layout))


def sf_bytes(m: int, nb: int, layout: int) -> int:
    return int(lib().kqo_sf_bytes(m, nb, layout))


def sf_place(sf_rowmajor: np.ndarray, layout: int, fill: int = 0) -> np.ndarray:
    """Scale bytes [m, nb] placed into the given layout; padding positions
    of the tiled layout get ``fill``."""
    rm = np.ascontiguousarray(sf_rowmajor, dtype=np.uint8)
    m, nb = rm.shape
    out = np.empty(sf_bytes(m, nb, layout), np.uint8)
    lib().kqo_sf_place(_p(rm, ctypes.c_uint8), m, nb, layout, fill, _p(out, ctypes.c_uint8))
    return out


def quantize(y: np.ndarray, bound: np.ndarray | None, layout: int = SF_ROWMAJOR,
             ldq: int | None = None):
    """Return (q [m, ldq] uint8, sf uint8, flags [m, d] uint8)."""
    y = _f64(y)
    m, d = y.shape
    assert d % 32 == 0
    ldq = d // 2 if ldq is None else ldq
    q = np.zeros((m, ldq), np.uint8)
    sf = np.zeros(sf_bytes(m, d // 32, layout), np.uint8)
    flags = np.zeros((m, d), np.uint8)
    b = None if bound is None else _f64(bound)
    lib().kqo_quantize(_p(y, ctypes.c_double), _p(b, ctypes.c_double) if b is not None else None,
                       m, d, _p(q, ctypes.c_uint8), ldq, _p(sf, ctypes.c_uint8), layout,
                       _p(flags, ctypes.c_uint8))
    return q, sf, flags


def dequantize(q: np.ndarray, sf: np.ndarray, layout: int, m: int, d: int) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    out = np.empty((m, d), np.float64)
    lib().kqo_dequantize(_p(q, ctypes.c_uint8), q.shape[1] if m else d // 2,
                         _p(sf, ctypes.c_uint8), layout, m, d, _p(out, ctypes.c_double))
    return out


def encode_f32_range(first: int, count: int) -> np.ndarray:
    """Packed codes of fp32 bit patterns first .. first+count-1 at scale 2^0."""
    assert count % 2 == 0
    out = np.empty(count // 2, np.uint8)
    lib().kqo_encode_f32_range(first, count, _p(out, ctypes.c_uint8))
    return out


# --- the whole path and the layer error of eq. (2) -------------------------------

def quantize_activations(A, d, kind, param=None, layout=SF_ROWMAJOR):
    """Transform + quantize: returns dict(y, bound, q, sf, flags)."""
    y, bound = transform(A, d, kind, param)
    q, sf, flags = quantize(y, bound, layout)
    return dict(y=y, bound=bound, q=q, sf=sf, flags=flags)


def inverse_transpose_blocks(factors: np.ndarray) -> np.ndarray:
    """Dense K_j^{-T} [nb, 32, 32] for the weight side W T^{-T} (eq. 1).

    K_j is expanded by eq. (12) and inverted as a dense matrix with
    ``numpy.linalg.inv`` (a library routine; the Kronecker inverse identity
    of eq. 5 is checked separately by the tests)."""
    K = expand_blocks(factors)
    return np.stack([np.linalg.inv(K[j]).T for j in range(K.shape[0])])


def layer_error(A, W, d, factors, layout=SF_ROWMAJOR):
    """eq. (2): E(T) = Q(AT) Q(W T^{-T})^T - A W^T, returned as (||E||_F,
    ||A W^T||_F) with everything in fp64."""
    qa = quantize_activations(A, d, "kron", factors, layout)
    yw, bw = transform(W, d, "dense", inverse_transpose_blocks(factors))
    qw, sfw, _ = quantize(yw, bw, layout)
    m, o = A.shape[0], W.shape[0]
    Aq = dequantize(qa["q"], qa["sf"], layout, m, d)
    Wq = dequantize(qw, sfw, layout, o, d)
    a = transform(A, d, "identity")[0]
    w = transform(W, d, "identity")[0]
    ref = a @ w.T
    E = Aq @ Wq.T - ref
    return float(np.linalg.norm(E)), float(np.linalg.norm(ref))

"""Seeded synthetic inputs for the KroQuant MXFP4 activation quantizer.

This module only draws random numbers and rounds them to the storage types
(fp32, bf16); it holds none of the method's arithmetic, so both the CUDA path
and the CPU reference may consume what it produces.

Stand-ins for the activations of the DiT layers named in "KroQuant:
Kronecker-Structured Block Transforms for Efficient Post-Training Quantization
of Diffusion Transformers" (arXiv 2607.21446v1), Sec. 4.1 (PixArt-Sigma, SANA,
FLUX.1-schnell) and the shapes of Tables 3-4.  No model weights, prompts or
dataset items are involved: every value is drawn from a seeded numpy
``default_rng``.

Models (``activations(..., model=...)``):
  * ``"gauss_outlier8"``: N(0,1) entries, 8 channels (drawn without
    replacement) scaled x100.
  * ``"pixart"``: N(0,1) x per-token lognormal(0, 0.5); 1 % of channels scaled
    by U[50, 200] (one factor per chosen channel).
  * ``"sana"``: N(0,1) x per-token lognormal(0, 0.5); 0.5 % of channels x100.
  * ``"flux"``: N(0,1) x per-token lognormal(0, 0.7); 1 % of channels scaled by
    U[30, 300].
"""
from __future__ import annotations

import numpy as np

SEED_A = 1000          # + config id
SEED_FACTORS = 2000    # + config id + layer
SEED_W = 3000
SEED_S = 4000


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 (round to nearest even) -> bf16 (round to nearest even),
    returned as uint16 bit patterns."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def f64_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """fp64 -> fp16 (round to nearest even, numpy) as uint16 bit patterns."""
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float16)).view(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint32) << 16).view(np.float32)


def activations(m: int, d: int, seed: int, model: str, lda: int | None = None,
                fmt: str = "bf16") -> np.ndarray:
    """bf16 (or, fmt='f16', fp16) bit patterns [m, lda] (columns d..lda-1
    are zero padding)."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((m, d))
    if model == "gauss_outlier8":
        ch = rng.choice(d, size=min(8, d), replace=False)
        x[:, ch] *= 100.0
    elif model in ("pixart", "sana", "flux"):
        sigma = 0.7 if model == "flux" else 0.5
        x *= rng.lognormal(0.0, sigma, size=(m, 1))
        frac = 0.005 if model == "sana" else 0.01
        n_out = max(1, int(round(frac * d)))
        ch = rng.choice(d, size=n_out, replace=False)
        if model == "pixart":
            x[:, ch] *= rng.uniform(50.0, 200.0, size=n_out)
        elif model == "sana":
            x[:, ch] *= 100.0
        else:
            x[:, ch] *= rng.uniform(30.0, 300.0, size=n_out)
    else:
        raise ValueError(f"unknown activation model {model!r}")
    bits = f64_to_f16_bits(x) if fmt == "f16" else f64_to_bf16_bits(x)
    if lda is not None and lda != d:
        out = np.zeros((m, lda), np.uint16)
        out[:, :d] = bits
        return out
    return bits


def weights(o: int, d: int, seed: int = SEED_W, std: float = 0.02) -> np.ndarray:
    """bf16 bit patterns [o, d], N(0, std^2)."""
    rng = np.random.default_rng(seed)
    return f64_to_bf16_bits(rng.standard_normal((o, d)) * std)


def lu_params(nb: int, seed: int) -> np.ndarray:
    """Per-block, per-factor LU parameters (a, b, c) as fp32 [nb, 5, 3]:
    a = u11 = exp(N(0, 0.2^2)), b = u12 ~ N(0, 0.3^2), c = l ~ N(0, 0.3^2)."""
    rng = np.random.default_rng(seed)
    c = rng.normal(0.0, 0.3, size=(nb, 5))
    b = rng.normal(0.0, 0.3, size=(nb, 5))
    a = np.exp(rng.normal(0.0, 0.2, size=(nb, 5)))
    return np.stack([a, b, c], axis=-1).astype(np.float32)


def hadamard_factors(nb: int) -> np.ndarray:
    """The Hadamard initial factor [[cos pi/4, sin pi/4], [sin pi/4, -cos pi/4]]
    (Sec. 3.2) for every factor of every block, fp32 [nb, 5, 2, 2]."""
    h = np.float32(np.cos(np.pi / 4))
    g = np.array([[h, h], [h, -h]], np.float32)
    return np.broadcast_to(g, (nb, 5, 2, 2)).copy()


def random_factors(nb: int, seed: int, scale: float = 1.0) -> np.ndarray:
    """Unstructured raw 2x2 entries N(0, scale^2) fp32 [nb, 5, 2, 2] (for
    tests of the raw-entry interface; no determinant constraint)."""
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((nb, 5, 2, 2)) * scale).astype(np.float32)


def smooth_scales(d: int, seed: int = SEED_S, sigma: float = 0.5) -> np.ndarray:
    """Per-channel scales s ~ lognormal(0, sigma) fp32 [d] (diagonal baseline)."""
    rng = np.random.default_rng(seed)
    return rng.lognormal(0.0, sigma, size=d).astype(np.float32)


def packed_codes(rows: int, k: int, seed: int) -> np.ndarray:
    """Uniform random bytes [rows, k/2]: two 4-bit E2M1 codes each, every
    code value equally likely (operands of the W4A4 product)."""
    rng = np.random.default_rng(seed)
    return rng.integers(0, 256, size=(rows, k // 2), dtype=np.uint8)


def scale_bytes(rows: int, nb: int, seed: int, lo: int, hi: int) -> np.ndarray:
    """Uniform random E8M0 bytes in [lo, hi], row-major [rows, nb]."""
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=(rows, nb), dtype=np.uint8)


# Workloads: (name, m, d, activation model, config id)
CONFIG0 = [("cfg0_tiny", 256, 1152, "gauss_outlier8", 0)]
CONFIG1 = [("pixart_qkv", 4096, 1152, "pixart", 1), ("pixart_ffn_down", 4096, 4608, "pixart", 1)]
CONFIG2 = [("sana_2240", 4096, 2240, "sana", 2), ("sana_5600", 4096, 5600, "sana", 2)]
CONFIG3 = [("flux_3072", 4608, 3072, "flux", 3), ("flux_ffn_down", 4608, 12288, "flux", 3)]
SWEEP_M = (256, 1024, 4096, 16384, 65536)
SWEEP_D = (1152, 3072, 12288)

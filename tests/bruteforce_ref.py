"""Brute-force restatement of the KroQuant MXFP4 quantizer for tiny inputs.

This is a pin for the C oracle, not a second copy of it: every step is
derived a different way from the same definitions, with plain Python loops,
so that a mistake in the oracle (a dropped factor, a transposed block, a
wrong bit order, a wrong tie rule, a wrong scale offset or tile layout) makes
the two disagree.

  * K_j       : nested ``numpy.kron`` (eq. 5) instead of the bit formula (eq. 12)
  * y = a.K   : explicit sums over r for every output channel c (eq. 4, K1's
                A_tile @ K orientation)
  * E8M0      : search for the largest integer k with 2^k <= amax, minus 2
  * e2m1      : arg-min over all 16 codes, whose values are decoded from the
                bit fields (sign, 2-bit exponent with bias 1, 1-bit mantissa);
                ties prefer the code whose sign matches v, then the even code;
                |v| > 6 saturates
  * packing   : loops over byte positions
  * 128x4 SF  : built by padding, reshaping and permuting an index matrix

Citations: "KroQuant: Kronecker-Structured Block Transforms for Efficient
Post-Training Quantization of Diffusion Transformers" (arXiv 2607.21446v1),
Sec. 3.1-3.2, eqs. (4), (5), (12); OCP Microscaling Formats (MX) v1.0,
E2M1 element and E8M0 scale definitions.
"""
from __future__ import annotations

import math

import numpy as np


def bf16_bits_to_float(h: int) -> float:
    return float(np.array([h << 16], dtype=np.uint32).view(np.float32)[0])


def kron_block(G) -> np.ndarray:
    G = np.asarray(G, dtype=np.float64).reshape(5, 2, 2)
    K = G[4]
    for k in (3, 2, 1, 0):
        K = np.kron(G[k], K)
    return K


def e2m1_decode(code: int) -> float:
    s = -1.0 if code & 8 else 1.0
    E = (code >> 1) & 3
    M = code & 1
    if E == 0:
        mag = M * 0.5                   # subnormal: 2^(1-bias) * M/2, bias 1
    else:
        mag = 2.0 ** (E - 1) * (1.0 + M / 2.0)
    return s * mag


def e2m1_encode(v: float) -> int:
    if abs(v) > 6.0:
        v = math.copysign(6.0, v)
    neg = math.copysign(1.0, v) < 0
    best, best_key = None, None
    for code in range(16):
        dist = abs(v - e2m1_decode(code))
        sign_mismatch = int(bool(code & 8) != neg)
        key = (dist, sign_mismatch, code & 1)
        if best_key is None or key < best_key:
            best, best_key = code, key
    return best


def e8m0_exponent(amax: float) -> int:
    if amax == 0.0:
        return -127
    k = -1100
    while math.ldexp(1.0, k + 1) <= amax:
        k += 1
    return max(-127, min(127, k - 2))


def blocked_sf_positions(m: int, nb: int) -> np.ndarray:
    """pos[i, kb] = byte position of scale (i, kb) in the 128x4 tiled layout."""
    mp = -(-m // 128) * 128
    nbp = -(-nb // 4) * 4
    idx = np.arange(mp * nbp).reshape(mp, nbp)          # row-major ids
    tiles = idx.reshape(mp // 128, 128, nbp // 4, 4).transpose(0, 2, 1, 3)
    # inside a tile: (row // 32, row % 32, col) -> (row % 32, row // 32, col)
    t = tiles.reshape(-1, 4, 32, 4).transpose(0, 2, 1, 3).reshape(-1)
    pos = np.empty(mp * nbp, np.int64)
    pos[t] = np.arange(t.size)
    return pos.reshape(mp, nbp)[:m, :nb]


def quantize_rows(A_bits: np.ndarray, d: int, Kblocks: np.ndarray, layout: int):
    """A_bits [m, d] uint16; Kblocks [nb, 32, 32] fp64.  Returns (y, q, sf)."""
    m = A_bits.shape[0]
    nb = d // 32
    y = np.zeros((m, d))
    for i in range(m):
        for j in range(nb):
            a = [bf16_bits_to_float(int(A_bits[i, 32 * j + r])) for r in range(32)]
            for c in range(32):
                acc = 0.0
                for r in range(32):
                    acc += a[r] * Kblocks[j][r][c]
                y[i, 32 * j + c] = acc
    q = np.zeros((m, d // 2), np.uint8)
    if layout == 0:
        sf = np.zeros(m * nb, np.uint8)
        pos = np.arange(m * nb).reshape(m, nb)
    else:
        sf = np.zeros((-(-m // 128)) * (-(-nb // 4)) * 512, np.uint8)
        pos = blocked_sf_positions(m, nb)
    for i in range(m):
        for j in range(nb):
            blk = y[i, 32 * j:32 * j + 32]
            amax = max(abs(x) for x in blk)
            e = e8m0_exponent(amax)
            sf[pos[i, j]] = e + 127
            codes = [e2m1_encode(x / 2.0 ** e) for x in blk]
            for k in range(16):
                q[i, 16 * j + k] = codes[2 * k] + 16 * codes[2 * k + 1]
    return y, q, sf

"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with itself: each test checks it against a
closed form, a library routine, a hand-derived golden value, an invariant or
the brute-force restatement in ``bruteforce_ref``.

Citations: [KQ] = "KroQuant: Kronecker-Structured Block Transforms for
Efficient Post-Training Quantization of Diffusion Transformers"
(arXiv 2607.21446v1); OCP MX = OCP Microscaling Formats v1.0.
"""
import ctypes
import math

import numpy as np
import pytest
import scipy.linalg

from conftest import build_c_helper, read_golden
from bruteforce_ref import (blocked_sf_positions, e2m1_decode, e8m0_exponent as bf_e8m0,
                            kron_block, quantize_rows)
from w4a4_mxfp4_activation_gb300 import synth

H2 = np.array([[1.0, 1.0], [1.0, -1.0]]) / math.sqrt(2.0)


def _factor_set(**named):
    """Five 2x2 factors, identity unless given as G1..G5."""
    G = np.tile(np.eye(2), (5, 1, 1))
    for k, v in named.items():
        G[int(k[1]) - 1] = np.asarray(v, float).reshape(2, 2)
    return G


# ---------------------------------------------------------------- eq. (6) --

def test_lu_factor_determinants(oracle_lib):
    """[KQ] eq. (6): det G = a * u22 = -1 in the paper's form; the workloads'
    form with u22 = +1/a has det +1.  np.linalg.det is the check."""
    rng = np.random.default_rng(7)
    lu = np.stack([np.exp(rng.normal(0, .2, 50)), rng.normal(0, .3, 50),
                   rng.normal(0, .3, 50)], -1)
    for sign in (-1, 1):
        G = oracle_lib.lu_to_factors(lu, sign)
        dets = np.linalg.det(G)
        assert np.allclose(dets, sign, atol=1e-13)
        # L . U multiplied by numpy
        for k in range(50):
            a, b, c = lu[k]
            L = np.array([[1, 0], [c, 1]])
            U = np.array([[a, b], [0, sign / a]])
            assert np.allclose(G[k], L @ U, rtol=0, atol=1e-15)


def test_lu_hadamard_special_case(oracle_lib):
    """[KQ] Sec. 3.2: the Hadamard initial factor [[cos, sin], [sin, -cos]]
    at pi/4 is reachable in the paper's form (det -1) with a = b = 1/sqrt2,
    c = 1."""
    r = 1 / math.sqrt(2)
    G = oracle_lib.lu_to_factors(np.array([r, r, 1.0]), -1)
    assert np.allclose(G, H2, atol=1e-15)


# ------------------------------------------------- eq. (5), (12), orientation --

def test_expand_matches_nested_kron(oracle_lib):
    """eq. (12) bit formula == eq. (5) nested numpy.kron, G1 outermost."""
    rng = np.random.default_rng(11)
    for _ in range(20):
        G = rng.standard_normal((5, 2, 2))
        assert np.allclose(oracle_lib.expand_block(G), kron_block(G), rtol=1e-15, atol=1e-15)


def test_hadamard_closed_form(oracle_lib):
    """P1: all factors H2/sqrt2 -> K = normalised 32-point Walsh-Hadamard
    (closed form and scipy.linalg.hadamard, Sylvester order)."""
    K = oracle_lib.expand_block(np.tile(H2, (5, 1, 1)))
    H = scipy.linalg.hadamard(32) / math.sqrt(32)
    assert np.max(np.abs(K - H)) <= 1e-15
    assert np.max(np.abs(oracle_lib.hadamard_block() - H)) <= 1e-15
    # the transform of random rows equals a @ H (library matmul)
    A = synth.activations(4, 128, 5, "gauss_outlier8")
    y, bound = oracle_lib.transform(A, 128, "hadamard")
    a = synth.bf16_bits_to_f32(A).astype(np.float64)
    ref = np.concatenate([a[:, 32 * j:32 * j + 32] @ H for j in range(4)], axis=1)
    assert np.allclose(y, ref, rtol=0, atol=1e-12 * np.abs(a).max())
    assert np.allclose(bound, np.concatenate(
        [np.abs(a[:, 32 * j:32 * j + 32]).sum(1, keepdims=True).repeat(32, 1) / math.sqrt(32)
         for j in range(4)], axis=1), rtol=1e-14)
    # Kronecker path with Hadamard factors == fixed Hadamard path
    yk, _ = oracle_lib.transform(A, 128, "kron", np.tile(H2, (4, 5, 1, 1)))
    assert np.allclose(yk, y, rtol=0, atol=1e-13 * np.abs(a).max())


def test_orientation_and_bit_order(oracle_lib):
    """P7: y = a . K (row vector times K, K1's A_tile @ K) and G1 on the most
    significant index bit -- hand-derived cases in golden/kron_orientation.txt."""
    for row in read_golden("kron_orientation.txt"):
        assert row[0] == "case"
        named, i = {}, 1
        while row[i].startswith("G"):
            named[row[i]] = [float(x) for x in row[i + 1:i + 5]]
            i += 5
        assert row[i] == "r"
        r = int(row[i + 1])
        assert row[i + 2] == "y"
        expect = np.zeros(32)
        for item in row[i + 3:]:
            c, v = item.split(":")
            expect[int(c)] = float(v)
        G = _factor_set(**named)
        a_bits = np.zeros((1, 32), np.uint16)
        a_bits[0, r] = 0x3F80                       # bf16 1.0
        y, _ = oracle_lib.transform(a_bits, 32, "kron", G[None])
        assert np.array_equal(y[0], expect), (named, r, y[0][:4])


def test_determinant_and_inverse(oracle_lib):
    """P2: det K = 1 for unit-|det| factors (both sign conventions, since
    det(G1 x ... x G5) = prod det(G_k)^16), and K . (x_k G_k^{-1}) = I
    ([KQ] Sec. 3.2, the Kronecker inverse identity)."""
    lu = synth.lu_params(6, 2000).astype(np.float64)
    for sign in (-1, 1):
        F = oracle_lib.lu_to_factors(lu, sign)
        for j in range(6):
            K = oracle_lib.expand_block(F[j])
            assert abs(np.linalg.det(K) - 1.0) <= 1e-9
            Kinv = kron_block(np.stack([np.linalg.inv(F[j, k]) for k in range(5)]))
            assert np.max(np.abs(K @ Kinv - np.eye(32))) <= 1e-12


def test_linear_map_invariance(oracle_lib):
    """P3: eq. (1) AT . (W T^{-T})^T = A W^T in fp64 to 1e-10 (the 256 x 1152
    correctness workload, W 1152 x 1152)."""
    m, d, o = 256, 1152, 1152
    A = synth.activations(m, d, synth.SEED_A + 0, "gauss_outlier8")
    W = synth.weights(o, d)
    F = oracle_lib.lu_to_factors(synth.lu_params(d // 32, synth.SEED_FACTORS), +1)
    F32 = F.astype(np.float32).astype(np.float64)
    yA, _ = oracle_lib.transform(A, d, "kron", F32)
    yW, _ = oracle_lib.transform(W, d, "dense", oracle_lib.inverse_transpose_blocks(F32))
    a = synth.bf16_bits_to_f32(A).astype(np.float64)
    w = synth.bf16_bits_to_f32(W).astype(np.float64)
    ref = a @ w.T
    err = np.linalg.norm(yA @ yW.T - ref) / np.linalg.norm(ref)
    assert err <= 1e-10, err


# ------------------------------------------------------------ quantizer --

def _golden_grid():
    return {int(r[0]): float(r[1]) for r in read_golden("e2m1_grid.txt")}


def test_e2m1_values_against_grid(oracle_lib):
    grid = _golden_grid()
    for code, v in grid.items():
        got = oracle_lib.e2m1_value(code)
        assert got == v and math.copysign(1, got) == math.copysign(1, v)
        assert e2m1_decode(code) == v


def test_e2m1_rounding_golden(oracle_lib):
    for v, code in read_golden("e2m1_rounding.txt"):
        assert oracle_lib.encode_e2m1(float(v)) == int(code), v


def test_e2m1_exhaustive_fp32(oracle_lib, tmp_path):
    """P4: every finite fp32 value, oracle encoder vs a scan of the E2M1
    table for the nearest magnitude (ties -> even code, |v| > 6 -> 6)."""
    pin = ctypes.CDLL(build_c_helper(tmp_path, "pin_e2m1_table_scan"))
    pin.pin_count_mismatches.restype = ctypes.c_uint64
    pin.pin_count_mismatches.argtypes = [ctypes.c_uint64, ctypes.c_uint64,
                                         ctypes.POINTER(ctypes.c_double), ctypes.c_void_p,
                                         ctypes.POINTER(ctypes.c_uint64)]
    grid = _golden_grid()
    mag = np.array([grid[k] for k in range(8)], np.float64)
    enc = ctypes.cast(oracle_lib.lib().kqo_encode_e2m1, ctypes.c_void_p)
    first_bad = ctypes.c_uint64(0)
    bad = pin.pin_count_mismatches(0, 1 << 32, mag.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                   enc, ctypes.byref(first_bad))
    assert bad == 0, f"{bad} mismatches, first at 0x{first_bad.value:08x}"


def test_e8m0_edges(oracle_lib):
    """P6: shared exponent at power-of-two edges, tiny and zero amax."""
    for mant, pw, e in read_golden("e8m0_edges.txt"):
        amax = math.ldexp(float(mant), int(pw))
        assert oracle_lib.e8m0_exponent(amax) == int(e), (mant, pw)
        assert bf_e8m0(amax) == int(e)


def test_e8m0_random_against_search(oracle_lib):
    rng = np.random.default_rng(3)
    for x in np.exp(rng.uniform(-95, 95, 400)):
        assert oracle_lib.e8m0_exponent(x) == bf_e8m0(float(x))


def test_worked_block(oracle_lib):
    """A hand-derived 32-element block (golden/worked_block.txt)."""
    g = {r[0]: r[1:] for r in read_golden("worked_block.txt")}
    y = np.array([[float(v) for v in g["y"]]])
    codes = [int(c) for c in g["codes"]]
    q, sf, _ = oracle_lib.quantize(y, None, 0)
    assert int(sf[0]) == int(g["scale"][0])
    packed = [codes[2 * k] | (codes[2 * k + 1] << 4) for k in range(16)]
    assert list(q[0]) == packed


def test_sf_blocked_offsets_golden(oracle_lib):
    for nb, i, kb, off in read_golden("sf_blocked_offsets.txt"):
        assert oracle_lib.sf_offset(int(i), int(kb), int(nb), 1) == int(off)


@pytest.mark.parametrize("m,nb", [(1, 1), (128, 4), (200, 70), (256, 36), (300, 175)])
def test_sf_blocked_bijection(oracle_lib, m, nb):
    """P8 (host part): the tiled offsets are a bijection onto the padded
    tile area and agree with the reshape/permute construction."""
    pos = blocked_sf_positions(m, nb)
    mp, nbp = -(-m // 128) * 128, -(-nb // 4) * 4
    full = np.array([[oracle_lib.sf_offset(i, k, nb, 1) for k in range(nbp)] for i in range(mp)])
    assert sorted(full.ravel().tolist()) == list(range(mp * nbp))
    assert oracle_lib.sf_bytes(m, nb, 1) == mp * nbp
    assert np.array_equal(full[:m, :nb], pos)


@pytest.mark.parametrize("m,nb", [(1, 1), (200, 70), (300, 175)])
def test_sf_place_matches_permutation(oracle_lib, m, nb):
    """sf_place scatters row-major scales to the positions of the
    reshape/permute construction and fills every other byte."""
    rm = np.random.default_rng(m + nb).integers(0, 255, size=(m, nb), dtype=np.uint8)
    out = oracle_lib.sf_place(rm, 1, fill=255)
    pos = blocked_sf_positions(m, nb)
    assert np.array_equal(out[pos], rm)
    rest = np.ones(out.size, bool)
    rest[pos.ravel()] = False
    assert np.all(out[rest] == 255)
    assert np.array_equal(oracle_lib.sf_place(rm, 0), rm.ravel())


# ------------------------------------------------- brute force (P5) --

@pytest.mark.parametrize("m,d", [(1, 32), (2, 64), (3, 128), (4, 1152)])
@pytest.mark.parametrize("kind", ["kron", "hadamard", "diag", "identity"])
@pytest.mark.parametrize("layout", [0, 1])
def test_bruteforce_agreement(oracle_lib, m, d, kind, layout):
    """P5: on 1-4 rows the brute-force restatement (nested kron, explicit
    loops, exponent search, 16-code arg-min, index-permutation SF layout)
    agrees with the oracle: y to 1e-12 of its scale, codes and scales
    exactly."""
    nb = d // 32
    A = synth.activations(m, d, 17 + m, "gauss_outlier8")
    if kind == "kron":
        F = oracle_lib.lu_to_factors(synth.lu_params(nb, 99), +1).astype(np.float32).astype(float)
        param, Kb = F, np.stack([kron_block(F[j]) for j in range(nb)])
    elif kind == "hadamard":
        param, Kb = None, np.stack([scipy.linalg.hadamard(32) / math.sqrt(32)] * nb)
    elif kind == "diag":
        s = synth.smooth_scales(d).astype(np.float64)
        param, Kb = s, np.stack([np.diag(s[32 * j:32 * j + 32]) for j in range(nb)])
    else:
        param, Kb = None, np.stack([np.eye(32)] * nb)
    y, bound = oracle_lib.transform(A, d, kind, param)
    q, sf, flags = oracle_lib.quantize(y, bound, layout)
    yb, qb, sfb = quantize_rows(A, d, Kb, layout)
    assert np.all(np.abs(y - yb) <= 1e-12 * np.maximum(bound, 1e-300))
    # codes can only differ where the two fp64 sums straddle a decision
    # point; the oracle flags those (tolerance far above fp64 rounding)
    assert np.array_equal(sf, sfb)
    codes = np.stack([q & 15, q >> 4], -1).reshape(m, d)
    codesb = np.stack([qb & 15, qb >> 4], -1).reshape(m, d)
    diff = codes != codesb
    assert not np.any(diff & (flags == 0))


def bruteforce_small_case(oracle_lib):
    """One fixed brute-force case (2 rows, d = 64, random unit-det factors)."""
    test_bruteforce_agreement(oracle_lib, 2, 64, "kron", 0)


def test_dequantize_roundtrip_exact(oracle_lib):
    """Values already on the grid x 2^e come back exactly (P9's host side):
    y = value(code) * 2^e with the block amax fixing e."""
    rng = np.random.default_rng(5)
    m, d = 8, 256
    grid = np.array([e2m1_decode(c) for c in range(16)])
    codes = rng.integers(0, 16, (m, d))
    codes[:, ::32] = 7                              # |v| = 6 in every block -> amax = 6*2^e
    e = rng.integers(-100, 100, (m, d // 32))
    y = grid[codes] * np.ldexp(1.0, np.repeat(e, 32, axis=1))
    for layout in (0, 1):
        q, sf, _ = oracle_lib.quantize(y, None, layout)
        back = oracle_lib.dequantize(q, sf, layout, m, d)
        assert np.array_equal(back, y)
        assert np.array_equal(np.signbit(back), np.signbit(y))


def test_quantize_flags(oracle_lib):
    """Flag bits: midpoint (1), power-of-two amax (2), undecided zero sign (4)."""
    y = np.zeros((1, 64))
    y[0, 0] = 4.0                     # amax exactly 4 -> edge flag on block 0
    y[0, 1] = 1.25                    # midpoint
    y[0, 32] = 5.0                    # block 1 amax 5 -> e = 0
    y[0, 33] = 2.5 * (1 + 5e-4)       # within 1e-3 of midpoint 2.5
    y[0, 34] = 2.5 * (1 + 2e-3)       # outside
    y[0, 35] = -1e-9                  # rounds to -0
    bound = np.full((1, 64), 1.0)
    _, _, fl = oracle_lib.quantize(y, bound, 0)
    assert fl[0, 0] & 2 and fl[0, 1] & 2 and fl[0, 1] & 1
    assert not fl[0, 32] & 2
    assert fl[0, 33] & 1 and not fl[0, 34] & 1
    assert fl[0, 35] & 4 and not fl[0, 32] & 4


def test_layer_error_hadamard_vs_identity_sanity(oracle_lib):
    """eq. (2) on the 256 x 1152 workload: ||E||_F is finite, positive and
    well below ||A W^T||_F for the Hadamard and the random unit-det
    factors."""
    m, d = 256, 1152
    A = synth.activations(m, d, synth.SEED_A, "gauss_outlier8")
    W = synth.weights(1152, d)
    for F in (synth.hadamard_factors(d // 32).astype(np.float64),
              oracle_lib.lu_to_factors(synth.lu_params(d // 32, synth.SEED_FACTORS), +1)
              .astype(np.float32).astype(np.float64)):
        e, ref = oracle_lib.layer_error(A, W, d, F)
        assert 0 < e < 0.5 * ref


def _golden_layer_case():
    """The hand-derived single-block case of tests/golden/layer_error.txt:
    (A bits [1, 32], W bits [1, 32], factors [1, 5, 2, 2], ||E||_F, ||A W^T||_F)."""
    g = {r[0]: r[1:] for r in read_golden("layer_error.txt")}
    F = np.array([[float(v) for v in g[f"G{k}"]] for k in range(1, 6)]).reshape(1, 5, 2, 2)
    a = np.zeros((1, 32))
    w = np.zeros((1, 32))
    a[0, :len(g["a"])] = [float(v) for v in g["a"]]
    w[0, :len(g["w"])] = [float(v) for v in g["w"]]
    return (synth.f64_to_bf16_bits(a), synth.f64_to_bf16_bits(w), F,
            float(g["error_norm"][0]), float(g["reference_norm"][0]))


def test_layer_error_golden(oracle_lib):
    """eq. (2) on the hand-derived block: a shear factor G5 makes A T leave
    the MXFP4 grid (one element on a rounding midpoint) while W T^{-T} stays
    on it, so ||E||_F = 1.5 and ||A W^T||_F = 3.5 exactly.  A dropped
    transform on either side, K^{-1} or K in place of K^{-T}, or a sign slip
    in E gives another value."""
    A, W, F, e_want, r_want = _golden_layer_case()
    for layout in (0, 1):
        e, ref = oracle_lib.layer_error(A, W, 32, F, layout=layout)
        assert e == e_want and ref == r_want, (e, ref)


# Monomial 2x2 factors with power-of-two entries and det 1 (signed
# permutations times diagonal scalings): products and inverses are exact in
# binary arithmetic, and none of P, Q is symmetric or orthogonal.
_MONOMIAL = {
    "I": [[1.0, 0.0], [0.0, 1.0]],
    "P": [[0.0, 2.0], [-0.5, 0.0]],
    "Q": [[0.0, -0.25], [4.0, 0.0]],
    "D": [[2.0, 0.0], [0.0, 0.5]],
    "S": [[0.0, 1.0], [-1.0, 0.0]],
    "N": [[-1.0, 0.0], [0.0, -1.0]],
}


def _grid_rows(rng, rows, d):
    """Rows whose every 32-block is E2M1 values x 2^e with block amax 4 or 6
    times 2^e, i.e. exactly representable in MXFP4."""
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    v = grid[rng.integers(0, 8, (rows, d))] * rng.choice([-1.0, 1.0], (rows, d))
    for j in range(d // 32):
        pos = 32 * j + rng.integers(0, 32, rows)
        v[np.arange(rows), pos] = rng.choice([-6.0, -4.0, 4.0, 6.0], rows)
        v[:, 32 * j:32 * j + 32] *= np.ldexp(1.0, rng.integers(-4, 5, (rows, 1)))
    return v


def _kron_dense(G):
    """Dense K = G1 (x) ... (x) G5 by nested numpy kron (a library routine;
    G1 outermost, so it acts on bit 4 of the channel index)."""
    K = np.array([[1.0]])
    for k in range(5):
        K = np.kron(K, G[k])
    return K


def _exact_zero_case(seed=11, m=3, d=64):
    """A and W with A T and W T^{-T} exactly on the MXFP4 grid under monomial
    factors: the quantizer is then exact on both sides and eq. (1) makes
    Q(A T) Q(W T^{-T})^T equal A W^T exactly.  Returns (A bits, W bits,
    factors, y = A T, z = W T^{-T}); W is square (o = d)."""
    rng = np.random.default_rng(seed)
    names = [["P", "I", "D", "S", "Q"], ["N", "Q", "I", "P", "D"]][: d // 32]
    F = np.array([[_MONOMIAL[n] for n in blk] for blk in names])
    y = _grid_rows(rng, m, d)
    z = _grid_rows(rng, d, d)
    A = np.zeros((m, d))
    W = np.zeros((d, d))
    for j in range(d // 32):
        K = _kron_dense(F[j])
        # K is monomial (one nonzero +-2^k per row and column), so its inverse
        # is its transpose with every nonzero entry replaced by its reciprocal
        assert ((K != 0).sum(0) == 1).all() and ((K != 0).sum(1) == 1).all()
        Kinv = np.where(K != 0, 1.0 / np.where(K != 0, K, 1.0), 0.0).T
        assert np.array_equal(K @ Kinv, np.eye(32))
        sl = slice(32 * j, 32 * j + 32)
        A[:, sl] = y[:, sl] @ Kinv                  # A T = y
        W[:, sl] = z[:, sl] @ K.T                   # W T^{-T} = z
    A_bits, W_bits = synth.f64_to_bf16_bits(A), synth.f64_to_bf16_bits(W)
    assert np.array_equal(synth.bf16_bits_to_f32(A_bits), A)      # exact in bf16
    assert np.array_equal(synth.bf16_bits_to_f32(W_bits), W)
    return A_bits, W_bits, F, y, z


def _exact_frobenius(y, z):
    """||y z^T||_F from integer arithmetic on the dyadic entries (no floating
    point in the sums)."""
    from fractions import Fraction
    sy = sz = 2 ** 12
    Y = [[int(v * sy) for v in row] for row in y]
    Z = [[int(v * sz) for v in row] for row in z]
    assert np.array_equal(np.array(Y, float) / sy, y) and np.array_equal(np.array(Z, float) / sz, z)
    tot = sum(sum(yi * zi for yi, zi in zip(r, c)) ** 2 for r in Y for c in Z)
    return math.sqrt(float(Fraction(tot, (sy * sz) ** 2)))


def test_layer_error_exact_on_grid(oracle_lib):
    """eq. (1)-(2) with nothing left to round: signed-permutation-times-
    power-of-two factors and activations / weights whose transformed blocks
    lie on the E2M1 grid times 2^e.  The quantization error is zero, so
    ||E||_F must be exactly 0 while ||A W^T||_F equals the exact integer
    computation of ||y z^T||_F (y = A T, z = W T^{-T}).  Quantizing A without
    T, using K^{-1} or K for K^{-T}, multiplying by W_q instead of W_q^T, or a
    sign slip all give a nonzero error."""
    A, W, F, y, z = _exact_zero_case()
    for layout in (0, 1):
        e, ref = oracle_lib.layer_error(A, W, 64, F, layout=layout)
        assert e == 0.0, e
        assert abs(ref - _exact_frobenius(y, z)) <= 1e-15 * ref and ref > 0


# --- the 16-bit side output: fp64 -> bf16, round to nearest even ----------------

def _bf16_decode(bits):
    """bf16 patterns -> fp64 through numpy's fp32 view (independent of the oracle)."""
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_bf16_rounding_golden(oracle_lib):
    """Hand-derived cases: ties in normal and subnormal binades, carries into
    the next binade, overflow at the top tie, signed zero."""
    for v, b in read_golden("bf16_rounding.txt"):
        got = int(oracle_lib.round_bf16(np.array([float.fromhex(v)]))[0])
        assert got == int(b, 16), (v, hex(got), b)


def test_bf16_rounding_is_nearest_even(oracle_lib):
    """Brute-force property on random doubles over the whole bf16 range
    (subnormals included) and on exact ties: the result is no farther from x
    than either adjacent bf16 value, an exact tie goes to the even pattern,
    the sign is kept, and infinity only appears at or beyond the top tie."""
    rng = np.random.default_rng(77)
    n = 200_000
    x = rng.uniform(1.0, 2.0, n) * np.exp2(rng.integers(-140, 128, n))
    # exact midpoints between adjacent bf16 values in random binades
    k = rng.integers(128, 255, n // 4).astype(np.float64)
    e = rng.integers(-126, 127, n // 4)
    ties = (k + 0.5) * np.exp2(e - 7)
    sub = (rng.integers(0, 127, n // 8) + 0.5) * 2.0 ** -133      # subnormal ties
    x = np.concatenate([x, ties, sub])
    x *= rng.choice([-1.0, 1.0], x.size)
    r = oracle_lib.round_bf16(x).astype(np.int64)
    assert np.array_equal((r >> 15) == 1, np.signbit(x))
    mag = r & 0x7FFF
    ax = np.abs(x)
    top = 2.0 ** 128
    inf = mag == 0x7F80
    assert not np.any(mag > 0x7F80)
    assert np.all(ax[inf] >= (_bf16_decode(0x7F7F) + top) / 2)
    fin = ~inf
    m, a = mag[fin], ax[fin]
    v = _bf16_decode(m)
    lo = _bf16_decode(np.maximum(m - 1, 0))
    hi = np.where(m + 1 >= 0x7F80, top, _bf16_decode(np.minimum(m + 1, 0x7F7F)))
    err = np.abs(a - v)
    assert np.all(err <= np.abs(a - lo)) and np.all(err <= np.abs(a - hi))
    tie = ((err == np.abs(a - hi)) & (hi != v)) | ((err == np.abs(a - lo)) & (lo != v))
    assert tie.sum() > n // 4
    assert np.all(m[tie] % 2 == 0)


def test_bf16_rounding_matches_torch_fp32(oracle_lib):
    """Special case reducing to a library routine: for fp32-representable x,
    rounding to bf16 is torch's fp32 -> bf16 conversion (round to nearest even)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(78)
    bits = rng.integers(0, 2 ** 32, 400_000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle_lib.round_bf16(f.astype(np.float64))
    assert np.array_equal(got, want)


# --- full-row Walsh-Hadamard baseline ------------------------------------------------

@pytest.mark.parametrize("d", [32, 64, 1024, 4096])
def test_fwht_matches_library_hadamard(oracle_lib, d):
    """Special case reducing to a library routine: y = a . H_d / sqrt(d) with
    scipy's Sylvester-order Hadamard matrix."""
    A = synth.activations(3, d, 120 + d, "flux")
    y, bound = oracle_lib.transform(A, d, "fwht")
    a = synth.bf16_bits_to_f32(A).astype(np.float64)
    H = scipy.linalg.hadamard(d).astype(np.float64)
    want = a @ H / math.sqrt(d)
    assert np.allclose(y, want, rtol=0, atol=1e-12 * np.abs(a).sum(axis=1, keepdims=True).max())
    assert np.allclose(bound, np.abs(a).sum(axis=1, keepdims=True) / math.sqrt(d), rtol=1e-15)


def test_fwht_closed_forms(oracle_lib):
    """One-hot rows give rows of H_d / sqrt(d) ((-1)^popcount(r & c)), the
    transform keeps the Euclidean norm (H_d / sqrt(d) is orthogonal), and at
    d = 32 it is the block Hadamard transform."""
    d = 2048
    rows = [0, 1, 5, 1000, 2047]
    A = np.zeros((len(rows), d), np.uint16)
    for i, r in enumerate(rows):
        A[i, r] = 0x3F80                                   # 1.0
    y, _ = oracle_lib.transform(A, d, "fwht")
    c = np.arange(d)
    for i, r in enumerate(rows):
        sign = np.array([1.0 if bin(r & cc).count("1") % 2 == 0 else -1.0 for cc in c])
        assert np.array_equal(y[i], sign / math.sqrt(d))
    B = synth.activations(4, 8192, 131, "flux")
    yb, _ = oracle_lib.transform(B, 8192, "fwht")
    b = synth.bf16_bits_to_f32(B).astype(np.float64)
    assert np.allclose(np.linalg.norm(yb, axis=1), np.linalg.norm(b, axis=1), rtol=1e-13)
    C = synth.activations(5, 32, 132, "flux")
    y32, _ = oracle_lib.transform(C, 32, "fwht")
    yh, _ = oracle_lib.transform(C, 32, "hadamard")
    assert np.allclose(y32, yh, rtol=0, atol=1e-13)


# ------------------------------------------------ fp16 input (Sec. 4.1) --

def test_f16_conversion_all_patterns(oracle_lib):
    """The oracle's binary16 decoding against numpy's float16 on all 65536
    bit patterns (a library routine: NaNs compared as NaN)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_lib.f16_to_f64(int(h)) for h in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_f16_closed_forms(oracle_lib):
    """Values of binary16 fixed by its definition (bias 15, 10-bit fraction,
    subnormals f * 2^-24)."""
    cases = {0x3C00: 1.0, 0x7BFF: 65504.0, 0x0001: 2.0 ** -24, 0x03FF: 1023 * 2.0 ** -24,
             0x0400: 2.0 ** -14, 0xC000: -2.0, 0x3555: 1365 / 4096, 0x8000: -0.0,
             0x7C00: float("inf"), 0xFC00: float("-inf")}
    for h, v in cases.items():
        got = oracle_lib.f16_to_f64(h)
        assert got == v and np.signbit(got) == np.signbit(v), (hex(h), got, v)


@pytest.mark.parametrize("kind", ["kron", "diag", "identity", "hadamard", "fwht"])
def test_f16_input_equals_bf16_input_on_shared_values(oracle_lib, kind):
    """Activations exactly representable in both formats (8 significant bits,
    exponents inside fp16's range) give the same y and bound whether they
    arrive as fp16 or as bf16 patterns."""
    rng = np.random.default_rng(11)
    m, d = 3, 256
    vals = np.ldexp(rng.integers(-255, 256, size=(m, d)).astype(np.float64),
                    rng.integers(-12, 4, size=(m, d)))
    f16 = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(f16.view(np.float16).astype(np.float64), vals)
    bf16 = (vals.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((bf16.astype(np.uint32) << 16).view(np.float32).astype(np.float64), vals)
    param = None
    if kind == "kron":
        param = rng.standard_normal((d // 32, 5, 2, 2))
    elif kind == "diag":
        param = rng.lognormal(0.0, 0.5, size=d)
    y16, b16 = oracle_lib.transform(f16, d, kind, param, in_format="f16")
    yb, bb = oracle_lib.transform(bf16, d, kind, param)
    assert np.array_equal(y16, yb) and np.array_equal(b16, bb)
    # and the format switch does not leak into the next call
    y2, _ = oracle_lib.transform(bf16, d, kind, param)
    assert np.array_equal(y2, yb)

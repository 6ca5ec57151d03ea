"""GPU parity: the CUDA quantizers, called through the C ABI, against the CPU
oracle on seeded synthetic inputs (comparison rules in ``parity.py``).

Workloads: stand-ins for the DiT layers of "KroQuant: Kronecker-Structured
Block Transforms for Efficient Post-Training Quantization of Diffusion
Transformers" (Sec. 4.1; Tables 3-4 shapes): the 256 x 1152 correctness case,
PixArt-Sigma (4096 x 1152 / 4608), SANA (4096 x 2240 / 5600), FLUX.1-schnell
(4608 x 3072 / 12288) and the m x d sweep.
"""
import ctypes
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from conftest import build_c_helper, read_golden
import parity
from oracle import kq_oracle as O
from w4a4_mxfp4_activation_gb300 import kq, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w4a4_mxfp4_activation_gb300 import build
    build.build()
    kq.lib()


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def to_bf16(bits):
    return dev(bits.view(np.int16)).view(torch.bfloat16)


def np_(t):
    return t.cpu().numpy()


def lib_factors(nb, seed, sign=+1):
    """Raw fp32 factors through the library helper (GPU side) and the
    oracle's own fp64 entries from the same LU parameters."""
    lu = synth.lu_params(nb, seed)
    return kq.kq_lu_to_factors(lu, sign), O.lu_to_factors(lu.astype(np.float64), sign) \
        .astype(np.float32).astype(np.float64)


def run_kind(kind, A_bits, d, layout, param_gpu=None, y_debug=True, variant=None, q=None, sf=None):
    A = A_bits if isinstance(A_bits, torch.Tensor) else to_bf16(A_bits)
    if kind == "kron_umma":
        records = kq.kq_expand_blocks(dev(param_gpu), kq.KQ_K_BF16X3)
        return kq.kq_quantize_mxfp4(A, d, K_expanded=records, layout=layout, y_debug=y_debug,
                                    variant=kq.VARIANT_UMMA, q=q, sf=sf)
    if kind == "kron_k2":
        # the tensor-core kernel building its operand records from the factors
        return kq.kq_quantize_mxfp4(A, d, factors=dev(param_gpu), layout=layout, y_debug=y_debug,
                                    variant=kq.VARIANT_K2, q=q, sf=sf)
    if kind == "kron":
        # the CUDA-core butterfly (the default from raw factors is K2)
        return kq.kq_quantize_mxfp4(A, d, factors=dev(param_gpu), layout=layout, y_debug=y_debug,
                                    variant=kq.VARIANT_BUTTERFLY if variant is None else variant,
                                    q=q, sf=sf)
    if kind == "identity":
        return kq.kq_quantize_mxfp4(A, d, layout=layout, y_debug=y_debug, q=q, sf=sf)
    if kind == "diag":
        return kq.kq_smooth_quantize_mxfp4(A, dev(param_gpu), d, layout=layout, y_debug=y_debug,
                                           q=q, sf=sf)
    if kind == "hadamard":
        return kq.kq_hadamard_quantize_mxfp4(A, d, layout=layout, y_debug=y_debug, q=q, sf=sf)
    raise ValueError(kind)


def oracle_kind(kind):
    return "kron" if kind in ("kron_umma", "kron_k2") else kind


def params_for(kind, nb, d, seed):
    """(gpu param, oracle param) for a transform kind."""
    if kind in ("kron", "kron_umma", "kron_k2"):
        return lib_factors(nb, seed)
    if kind == "diag":
        s = synth.smooth_scales(d)
        return s, s.astype(np.float64)
    return None, None


# ------------------------------------------------------------------ encoder --

def test_encoder_exhaustive_fp32(tmp_path):
    """P4g: every finite fp32 bit pattern through the kernels' E2M1 encoder
    (scale 2^0) equals the table scan (nearest magnitude, ties to the even
    code, |v| > 6 -> 6, sign kept) -- also pins the nibble order."""
    pin = ctypes.CDLL(build_c_helper(tmp_path, "pin_e2m1_table_scan"))
    pin.pin_table_scan_packed.argtypes = [ctypes.c_uint64, ctypes.c_uint64,
                                          ctypes.POINTER(ctypes.c_double), ctypes.c_void_p]
    grid = {int(r[0]): float(r[1]) for r in read_golden("e2m1_grid.txt")}
    mag = np.array([grid[k] for k in range(8)], np.float64)
    magp = mag.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    chunk = 1 << 28
    out = torch.empty(chunk // 2, dtype=torch.uint8, device="cuda")
    exp = np.empty(chunk // 2, np.uint8)
    per_exp = 1 << 22                                # bytes per fp32 exponent value
    for first in range(0, 1 << 32, chunk):
        kq.kq_test_encode_e2m1(first, chunk, out)
        got = np_(out)
        pin.pin_table_scan_packed(first, chunk, magp, exp.ctypes.data)
        for r in range(chunk // 2 // per_exp):
            if (((first >> 23) + r) & 0xFF) == 0xFF:
                continue                             # inf / NaN patterns: out of contract
            g, e = got[r * per_exp:(r + 1) * per_exp], exp[r * per_exp:(r + 1) * per_exp]
            if not np.array_equal(g, e):
                k = int(np.argmax(g != e))
                raise AssertionError(f"encoder mismatch at pattern 0x{first + 2 * (r * per_exp + k):08x}:"
                                     f" got {g[k]:#04x}, want {e[k]:#04x}")


def test_worked_block_bare_quantizer():
    """Hand-derived block through the identity transform (bit-exact)."""
    g = {r[0]: r[1:] for r in read_golden("worked_block.txt")}
    y = np.array([float(v) for v in g["y"]])
    bits = synth.f64_to_bf16_bits(y[None, :])
    assert np.array_equal(synth.bf16_bits_to_f32(bits)[0].astype(np.float64), y)
    q, sf, _ = run_kind("identity", bits, 32, 0)
    codes = [int(c) for c in g["codes"]]
    assert int(np_(sf)[0]) == int(g["scale"][0])
    assert list(np_(q)[0]) == [codes[2 * k] | (codes[2 * k + 1] << 4) for k in range(16)]


# ------------------------------------------------------------- configs 0-3 --

CASES = synth.CONFIG0 + synth.CONFIG1 + synth.CONFIG2 + synth.CONFIG3


@pytest.mark.parametrize("name,m,d,model,cfg", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("kind", ["kron", "kron_umma", "kron_k2", "diag", "hadamard", "identity"])
def test_config_parity(name, m, d, model, cfg, kind):
    """Configs 0-3 at full size, every row and block, both scale layouts
    (the oracle's result computed once and compared with both)."""
    nb = d // 32
    A_bits = synth.activations(m, d, synth.SEED_A + cfg, model)
    pg, po = params_for(kind, nb, d, synth.SEED_FACTORS + cfg)
    ref = parity.reference(A_bits, d, oracle_kind(kind), po)
    for layout in (0, 1):
        q, sf, y = run_kind(kind, A_bits, d, layout, pg)
        res = parity.check(A_bits, d, oracle_kind(kind), po, layout, np_(q), np_(sf), np_(y),
                           ref=ref)
        # the production launch (no debug output) writes the same bytes
        q2, sf2, _ = run_kind(kind, A_bits, d, layout, pg, y_debug=False)
        assert torch.equal(q, q2) and torch.equal(sf, sf2)
        parity.record(f"config {cfg}", name, m, d, kind, layout, res)
        print(name, kind, layout, res)


def test_umma_matches_butterfly_outside_flags():
    """The tensor-core and the butterfly implementations of the same
    transform agree on every unflagged code (both are checked against the
    oracle elsewhere)."""
    m, d = 4096, 4608
    A_bits = synth.activations(m, d, synth.SEED_A + 1, "pixart")
    Fg, Fo = lib_factors(d // 32, synth.SEED_FACTORS + 1)
    qb, sfb, _ = run_kind("kron", A_bits, d, 1, Fg, y_debug=False)
    qm, sfm, _ = run_kind("kron_umma", A_bits, d, 1, Fg, y_debug=False)
    rows = np.arange(0, m, 7)
    _, _, flags = O.quantize(*O.transform(np.ascontiguousarray(A_bits[rows]), d, "kron", Fo),
                             O.SF_ROWMAJOR)
    strict = flags == 0
    cb, cm = parity.unpack(np_(qb)[rows], d), parity.unpack(np_(qm)[rows], d)
    assert np.array_equal(cb[strict], cm[strict])


def test_hadamard_factors_config0():
    """Config 0's second run: every factor the Hadamard initial factor; the
    KroQuant kernel and the fixed block-Hadamard kernel both match the
    oracle, and each other outside the oracle's flags."""
    m, d = 256, 1152
    nb = d // 32
    A_bits = synth.activations(m, d, synth.SEED_A, "gauss_outlier8")
    F = synth.hadamard_factors(nb)
    qk, sfk, yk = run_kind("kron", A_bits, d, 0, F)
    parity.check(A_bits, d, "kron", F.astype(np.float64), 0, np_(qk), np_(sfk), np_(yk))
    qh, sfh, yh = run_kind("hadamard", A_bits, d, 0)
    _, _, flags = O.quantize(*O.transform(A_bits, d, "hadamard"), O.SF_ROWMAJOR)
    ck, ch = parity.unpack(np_(qk), d), parity.unpack(np_(qh), d)
    strict = flags == 0
    assert np.array_equal(ck[strict], ch[strict])


# ------------------------------------------------------------------ E(T) --

@pytest.mark.parametrize("factor_kind", ["random", "hadamard"])
def test_layer_error_config0(factor_kind):
    """eq. (2): ||Q(AT) Q(W T^{-T})^T - A W^T||_F from the GPU quantizer and
    dequantizer matches the oracle to 1e-3 relative."""
    m, d, o = 256, 1152, 1152
    nb = d // 32
    A_bits = synth.activations(m, d, synth.SEED_A, "gauss_outlier8")
    W_bits = synth.weights(o, d)
    if factor_kind == "random":
        Fg, Fo = lib_factors(nb, synth.SEED_FACTORS)
    else:
        Fg = synth.hadamard_factors(nb)
        Fo = Fg.astype(np.float64)
    FgT = kq.kq_invert_transpose_factors(Fg)
    qa, sfa, _ = run_kind("kron", A_bits, d, 0, Fg, y_debug=False)
    qw, sfw, _ = run_kind("kron", W_bits, d, 0, FgT, y_debug=False)
    Aq = np_(kq.kq_dequantize(qa, sfa, m, d)).astype(np.float64)
    Wq = np_(kq.kq_dequantize(qw, sfw, o, d)).astype(np.float64)
    a = synth.bf16_bits_to_f32(A_bits).astype(np.float64)
    w = synth.bf16_bits_to_f32(W_bits).astype(np.float64)
    e_gpu = np.linalg.norm(Aq @ Wq.T - a @ w.T)
    e_ref, ref = O.layer_error(A_bits, W_bits, d, Fo)
    assert abs(e_gpu - e_ref) <= 1e-3 * e_ref, (e_gpu, e_ref)
    assert e_ref < ref


@pytest.mark.parametrize("name,m,d,model,cfg", synth.CONFIG1 + synth.CONFIG2 + synth.CONFIG3,
                         ids=[c[0] for c in synth.CONFIG1 + synth.CONFIG2 + synth.CONFIG3])
def test_layer_error_configs(name, m, d, model, cfg):
    """E(T) on configs 1-3: first 512 rows of A, a square weight of o = d
    output channels (an FFN-down-like d x d projection)."""
    m, o = 512, d
    nb = d // 32
    A_bits = synth.activations(m, d, synth.SEED_A + cfg, model)
    W_bits = synth.weights(o, d, seed=synth.SEED_W + cfg)
    Fg, Fo = lib_factors(nb, synth.SEED_FACTORS + cfg)
    qa, sfa, _ = run_kind("kron", A_bits, d, 1, Fg, y_debug=False)
    qw, sfw, _ = run_kind("kron", W_bits, d, 1, kq.kq_invert_transpose_factors(Fg), y_debug=False)
    Aq = np_(kq.kq_dequantize(qa, sfa, m, d, layout=1)).astype(np.float64)
    Wq = np_(kq.kq_dequantize(qw, sfw, o, d, layout=1)).astype(np.float64)
    a = synth.bf16_bits_to_f32(A_bits).astype(np.float64)
    w = synth.bf16_bits_to_f32(W_bits).astype(np.float64)
    e_gpu = np.linalg.norm(Aq @ Wq.T - a @ w.T)
    e_ref, _ = O.layer_error(A_bits, W_bits, d, Fo, layout=1)
    assert abs(e_gpu - e_ref) <= 1e-3 * e_ref, (e_gpu, e_ref)


# ------------------------------------------------------------ config 4 --

SWEEP = [(m, d) for m in synth.SWEEP_M for d in synth.SWEEP_D]


@pytest.mark.parametrize("m,d", SWEEP, ids=[f"{m}x{d}" for m, d in SWEEP])
def test_sweep_parity(m, d):
    """Config 4: 4 layers' factor sets per point; KroQuant (butterfly, the
    tensor cores on expanded records for two layers, the tensor cores with
    the records built in the kernel), diagonal and Hadamard quantizers.  Every row up
    to m = 16384; at m = 65536 a seeded sample of 4096 rows (the first and
    last tiles always included)."""
    nb = d // 32
    A_bits = synth.activations(m, d, synth.SEED_A + 4, "flux")
    rng = np.random.default_rng(m + d)
    rows = None
    if m > 16384:
        rows = np.unique(np.concatenate([np.arange(128), np.arange(m - 128, m),
                                         rng.choice(m, 4096, replace=False)]))
    for layer in range(4):
        Fg, Fo = lib_factors(nb, synth.SEED_FACTORS + 4 + layer)
        kind = ("kron", "kron_umma", "kron_k2", "kron_umma")[layer]
        q, sf, y = run_kind(kind, A_bits, d, layer % 2, Fg)
        res = parity.check(A_bits, d, "kron", Fo, layer % 2, np_(q), np_(sf), np_(y), rows)
        parity.record("config 4", f"sweep layer {layer}", m, d, kind, layer % 2, res)
        del q, sf, y
    s = synth.smooth_scales(d)
    q, sf, y = run_kind("diag", A_bits, d, 1, s)
    res = parity.check(A_bits, d, "diag", s.astype(np.float64), 1, np_(q), np_(sf), np_(y), rows)
    parity.record("config 4", "sweep", m, d, "diag", 1, res)
    q, sf, y = run_kind("hadamard", A_bits, d, 0)
    res = parity.check(A_bits, d, "hadamard", None, 0, np_(q), np_(sf), np_(y), rows)
    parity.record("config 4", "sweep", m, d, "hadamard", 0, res)


# ------------------------------------------------------------ edge cases --

EDGE_SHAPES = [(1, 32), (7, 96), (127, 160), (129, 64), (200, 5600), (3, 2240), (300, 1152)]


@pytest.mark.parametrize("m,d", EDGE_SHAPES, ids=[f"{m}x{d}" for m, d in EDGE_SHAPES])
@pytest.mark.parametrize("kind", ["kron", "kron_umma", "kron_k2", "diag", "hadamard", "identity"])
def test_ragged_shapes_with_pitches_and_canaries(m, d, kind):
    """Ragged m and d (partial tiles and block-columns), lda > d, ldq > d/2,
    and guard bytes around every output that must stay untouched."""
    nb = d // 32
    lda, ldq = d + 64, d // 2 + 32
    A_bits = synth.activations(m, d, 77 + m, "pixart", lda=lda)
    pg, po = params_for(kind, nb, d, 55 + d)
    for layout in (0, 1):
        sfb = kq.kq_sf_bytes(m, d, layout)
        q_store = torch.full((m + 2, ldq), 0xA5, dtype=torch.uint8, device="cuda")
        sf_store = torch.full((sfb + 64,), 0xA5, dtype=torch.uint8, device="cuda")
        q = q_store[1:m + 1]
        sf = sf_store[16:16 + sfb]
        qq, ssf, y = run_kind(kind, A_bits, d, layout, pg, q=q, sf=sf)
        qs = np_(q_store)
        assert (qs[0] == 0xA5).all() and (qs[m + 1] == 0xA5).all()
        assert (qs[1:m + 1, d // 2:] == 0xA5).all(), "row padding of q overwritten"
        ss = np_(sf_store)
        assert (ss[:16] == 0xA5).all() and (ss[16 + sfb:] == 0xA5).all()
        parity.check(np.ascontiguousarray(A_bits[:, :d]), d, oracle_kind(kind), po, layout,
                     np_(q)[:, :d // 2], np_(sf), np_(y))
        if layout == 1:
            # padding of the tiled layout is written as zero
            full = np.zeros(sfb, bool)
            rows = np.arange(m)
            i, kb = np.meshgrid(rows, np.arange(nb), indexing="ij")
            ncb = (nb + 3) // 4
            off = ((i // 128) * ncb + kb // 4) * 512 + (i % 32) * 16 + ((i % 128) // 32) * 4 + kb % 4
            full[off.ravel()] = True
            assert (np_(sf)[~full] == 0).all()


@pytest.mark.parametrize("m", [2907, 4347])
def test_k2_tile_pairs(m):
    """K2 with enough tiles per CTA to walk them by pairs of row tiles of one
    column, sharing the pair's records: an odd row-tile count (23, the last
    ragged), whose last pair is completed by a tile past the last row that
    must write nothing, and an even one (34, the last ragged: 17 pairs);
    lda > d, ldq > d/2, guard bytes around every output, every row against
    the oracle, both scale layouts."""
    d = 12288
    nb = d // 32
    lda, ldq = d + 64, d // 2 + 32
    A_bits = synth.activations(m, d, 3100 + m, "flux", lda=lda)
    pg, po = params_for("kron_k2", nb, d, 3200)
    for layout in (0, 1):
        sfb = kq.kq_sf_bytes(m, d, layout)
        q_store = torch.full((m + 2, ldq), 0xA5, dtype=torch.uint8, device="cuda")
        sf_store = torch.full((sfb + 4096,), 0xA5, dtype=torch.uint8, device="cuda")
        q = q_store[1:m + 1]
        sf = sf_store[16:16 + sfb]
        qq, ssf, y = run_kind("kron_k2", A_bits, d, layout, pg, q=q, sf=sf)
        qs = np_(q_store)
        assert (qs[0] == 0xA5).all() and (qs[m + 1] == 0xA5).all()
        assert (qs[1:m + 1, d // 2:] == 0xA5).all(), "row padding of q overwritten"
        ss = np_(sf_store)
        assert (ss[:16] == 0xA5).all() and (ss[16 + sfb:] == 0xA5).all(), "bytes past the scales written"
        parity.check(np.ascontiguousarray(A_bits[:, :d]), d, "kron", po, layout,
                     np_(q)[:, :d // 2], np_(sf), np_(y))


# ------------------------------------------------------------ maximum sizes --

MAX_ROWS = 0x7FFFFFFF          # the largest m the entry points accept
PERIOD = 4096                  # rows of the seeded base that every row repeats


@pytest.fixture
def max_rows_input():
    """A bf16 [2^31 - 1, 32] input (137 GB) whose row r is row r % 4096 of a
    seeded base, built on the device."""
    d = 32
    torch.cuda.empty_cache()              # blocks the previous case released
    free, _ = torch.cuda.mem_get_info()
    if free < 200e9:
        pytest.skip(f"needs about 190 GB of free device memory, {free / 1e9:.0f} GB free")
    base_bits = synth.activations(PERIOD, d, 9100, "flux")
    A = to_bf16(base_bits).repeat(-(-MAX_ROWS // PERIOD), 1)[:MAX_ROWS]
    yield base_bits, A
    del A
    torch.cuda.empty_cache()


def _periodic_equal(got, pattern, what):
    """got (1-D uint8 device tensor) equals pattern repeated, chunk by chunk."""
    reps = max(1, (256 << 20) // pattern.numel())
    ref = pattern.repeat(reps)
    step = ref.numel()
    for s in range(0, got.numel(), step):
        e = min(got.numel(), s + step)
        assert torch.equal(got[s:e], ref[:e - s]), f"{what}: bytes {s}..{e} differ from the base"


MAX_ROW_CASES = [("kron_umma", 0), ("kron_umma", 1), ("kron_k2", 0), ("kron_k2", 1), ("kron", 0),
                 ("kron", 1), ("diag", 0), ("diag", 1), ("hadamard", 0), ("identity", 1)]


@pytest.mark.parametrize("kind,layout", MAX_ROW_CASES, ids=[f"{k}-{l}" for k, l in MAX_ROW_CASES])
def test_maximum_rows(max_rows_input, kind, layout):
    """m = 2^31 - 1 rows, the entry points' upper limit (row offsets past
    2^31 bytes in every output, 2^24 row tiles).  The 4096-row base is
    checked against the oracle under rules i-iii; every row of the full
    launch must then equal the base launch's output for row r % 4096, bit
    for bit, and in the tiled scale layout the padding row of the last
    128-row tile must read 0."""
    base_bits, A = max_rows_input
    d, nb = 32, 1
    pg, po = params_for(kind, nb, d, 9101)
    qb, sfb, yb = run_kind(kind, base_bits, d, layout, pg)
    parity.check(base_bits, d, oracle_kind(kind), po, layout, np_(qb), np_(sfb), np_(yb))
    q, sf, _ = run_kind(kind, A, d, layout, pg, y_debug=None)
    torch.cuda.synchronize()
    _periodic_equal(q.view(-1), qb.view(-1), "codes")
    if layout == 0:
        _periodic_equal(sf.view(-1), sfb.view(-1), "scales")
    else:
        # 512 bytes per 128-row tile; the base spans 32 tiles, the launch
        # 2^24, the last of which holds 127 rows and one padding row
        assert sf.numel() == (MAX_ROWS + 1) // 128 * 512
        _periodic_equal(sf.view(-1)[:-512], sfb.view(-1), "scales")
        last = sfb.view(-1)[-512:].clone()
        last[31 * 16 + 3 * 4] = 0                  # row 127 of the tile, block 0
        assert torch.equal(sf.view(-1)[-512:], last)
    del q, sf
    torch.cuda.empty_cache()


LARGE_ROWS = (1 << 28) - 3      # at d = 128: 68.7 GB of bf16 input, 2^35 input bytes past 2^31


@pytest.mark.parametrize("kind", ["fwht", "dual"])
def test_large_rows_whole_row_and_dual(kind):
    """The full-row FWHT and the dual kernel (codes, scales and the bf16 side
    output A T) at 2^28 - 3 rows of 128 channels, a ragged last tile.  Every
    row repeats row r % 4096 of a seeded base: the base launch is checked
    against the oracle, and every row of the large launch must equal the
    base launch's row bit for bit."""
    m, d = LARGE_ROWS, 128
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info()
    need = m * d * (2 + 0.5 + (2 if kind == "dual" else 0)) + m * 4 + 4e9
    if free < need:
        pytest.skip(f"needs about {need / 1e9:.0f} GB of free device memory, {free / 1e9:.0f} GB free")
    base_bits = synth.activations(PERIOD, d, 9300, "flux")
    base = to_bf16(base_bits)
    A = base.repeat(-(-m // PERIOD), 1)[:m]
    if kind == "fwht":
        qb, sfb, yb = kq.kq_fwht_quantize_mxfp4(base, d, y_debug=True)
        parity.check(base_bits, d, "fwht", None, 0, np_(qb), np_(sfb), np_(yb))
        q, sf, _ = kq.kq_fwht_quantize_mxfp4(A, d)
        pairs = [(q, qb), (sf, sfb)]
    else:
        pg, po = lib_factors(d // 32, 9301)
        records = kq.kq_expand_blocks(dev(pg), kq.KQ_K_BF16X3)
        qb, sfb, atb, yb = kq.kq_quantize_mxfp4_dual(base, records, d, y_debug=True)
        parity.check(base_bits, d, "kron", po, 0, np_(qb), np_(sfb), np_(yb))
        parity.check_side_output(base_bits, d, "kron", po,
                                 np_(atb.view(torch.int16)).view(np.uint16), np_(yb))
        q, sf, at, _ = kq.kq_quantize_mxfp4_dual(A, records, d)
        pairs = [(q, qb), (sf, sfb), (at.view(torch.uint8), atb.view(torch.uint8))]
    torch.cuda.synchronize()
    for name, (got, ref) in zip(("codes", "scales", "side output"), pairs):
        _periodic_equal(got.reshape(-1)[:m * ref.numel() // PERIOD], ref.reshape(-1), name)
    del A, q, sf, pairs
    if kind == "dual":
        del at
    torch.cuda.empty_cache()


WIDE = (300, (1 << 20) + 96)   # 2^20 + 96 channels: 32771 blocks (odd, not a multiple of 4)


@pytest.mark.parametrize("kind", ["kron_umma", "kron_k2", "kron", "diag", "hadamard", "identity"])
def test_widest_rows(kind):
    """Rows of 2^20 + 96 channels (column coordinates past 2^20, 32771
    blocks, 201 MB of operand records), every element against the oracle in
    both scale layouts."""
    m, d = WIDE
    A_bits = synth.activations(m, d, 9200, "flux")
    pg, po = params_for(kind, d // 32, d, 9201)
    ref = parity.reference(A_bits, d, oracle_kind(kind), po)
    for layout in (0, 1):
        q, sf, y = run_kind(kind, A_bits, d, layout, pg)
        parity.check(A_bits, d, oracle_kind(kind), po, layout, np_(q), np_(sf), np_(y), ref=ref)


def test_special_values():
    """Zeros, negative zeros, bf16 subnormals, the largest bf16 values and
    exact midpoints through the bare quantizer and the Kronecker kernel."""
    rows = []
    rows.append(np.zeros(32))
    rows.append(-np.zeros(32))
    rows.append(np.ldexp(np.arange(32) - 16.0, -133))        # subnormal bf16
    rows.append(np.ldexp(np.linspace(-1, 1, 32), -126))
    rows.append(np.full(32, 3.3e38) * np.where(np.arange(32) % 2, 1, -1))
    rows.append(np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * 4) * 2.0 ** 40)
    rows.append(np.concatenate([[1e-30], np.zeros(31)]))
    y = np.stack(rows)
    bits = synth.f64_to_bf16_bits(y)
    q, sf, yd = run_kind("identity", bits, 32, 0)
    parity.check(bits, 32, "identity", None, 0, np_(q), np_(sf), np_(yd))
    # the special rows pass through the identity exactly: no flags needed
    codes = parity.unpack(np_(q), 32)
    assert (codes[0] == 0).all() and (codes[1] == 8).all() and (np_(sf)[:2] == 0).all()
    # the Kronecker transform may grow values by up to sum_r |K_rc|; keep y
    # inside the fp32 range (larger y is outside the contract)
    y_k = y.copy()
    y_k[4] /= 2.0 ** 8
    bits_k = synth.f64_to_bf16_bits(y_k)
    Fg, Fo = lib_factors(1, 3)
    for kind in ("kron", "kron_umma", "kron_k2"):
        q, sf, yd = run_kind(kind, bits_k, 32, 0, Fg)
        parity.check(bits_k, 32, "kron", Fo, 0, np_(q), np_(sf), np_(yd))


def test_raw_factor_interface():
    """Arbitrary raw 2x2 entries (no determinant constraint) and both LU
    sign conventions."""
    m, d = 300, 640
    nb = d // 32
    A_bits = synth.activations(m, d, 9, "sana")
    F = synth.random_factors(nb, 12, scale=0.8)
    for kind in ("kron", "kron_umma", "kron_k2"):
        q, sf, y = run_kind(kind, A_bits, d, 1, F)
        parity.check(A_bits, d, "kron", F.astype(np.float64), 1, np_(q), np_(sf), np_(y))
    Fg, Fo = lib_factors(nb, 13, sign=-1)
    q, sf, y = run_kind("kron", A_bits, d, 0, Fg)
    parity.check(A_bits, d, "kron", Fo, 0, np_(q), np_(sf), np_(y))


def test_empty_input_is_noop():
    A = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    q, sf, _ = kq.kq_quantize_mxfp4(A, 64, layout=0)
    assert q.shape[0] == 0


# ------------------------------------------------------- dequant, expand --

def test_dequantize_exact():
    """P9: the dequantizer equals the oracle's value(code) * 2^e exactly, for
    both layouts (including the padded tiles)."""
    m, d = 333, 1152
    A_bits = synth.activations(m, d, 21, "flux")
    Fg, _ = lib_factors(d // 32, 21)
    for layout in (0, 1):
        q, sf, _ = run_kind("kron", A_bits, d, layout, Fg, y_debug=False)
        out = np_(kq.kq_dequantize(q, sf, m, d, layout=layout)).astype(np.float64)
        ref = O.dequantize(np_(q), np_(sf), layout, m, d)
        assert np.array_equal(out, ref)
        assert np.array_equal(np.signbit(out), np.signbit(ref))


def test_expand_blocks_fp32():
    """K1's dense blocks: the device product (fp64, then fp32) equals the
    oracle's eq. (12) expansion rounded to fp32, bit for bit."""
    nb = 70
    Fg, Fo = lib_factors(nb, 31)
    out = kq.kq_expand_blocks(dev(Fg), kq.KQ_K_FP32)
    K = np_(out).view(np.float32).reshape(nb, 32, 32)
    ref = O.expand_blocks(Fg.astype(np.float64)).astype(np.float32)
    assert np.array_equal(K.view(np.uint32), ref.view(np.uint32))


def bf16_bits_to_f64(b):
    return (np.asarray(b, np.uint32) << 16).view(np.float32).astype(np.float64)


def test_expand_blocks_bf16x3_records():
    """The tensor-core operand records (KQ_K_BF16X3), decoded from their
    documented layout, hold for every entry of the oracle's fp64 K_j
    (eq. 12) the three bf16 terms hi = RN(K), mid = RN(K - hi), lo = RN(K -
    hi - mid), bit for bit (the oracle's fp64 -> bf16 rounding)."""
    nb = 70
    Fg, Fo = lib_factors(nb, 32)
    rec = np_(kq.kq_expand_blocks(dev(Fg), kq.KQ_K_BF16X3))
    assert rec.size == nb * 6144
    body = rec.view(np.uint16).reshape(nb, 3072)
    t, r, c = np.meshgrid(np.arange(3), np.arange(32), np.arange(32), indexing="ij")
    h, k, n = r // 16, r % 16, 32 * t + c
    off = h * 3072 + (n // 8) * 256 + (k // 8) * 128 + (n % 8) * 16 + (k % 8) * 2
    got = body[:, off // 2]                                  # [nb][term][row][col]
    K = O.expand_blocks(Fg.astype(np.float64))
    rem = K.copy()
    for term in range(3):
        want = O.round_bf16(rem)
        assert np.array_equal(got[:, term], want), term
        rem = rem - bf16_bits_to_f64(want)
    assert np.all(np.abs(rem) <= 2.0 ** -24 * np.abs(K))


def test_blocked_layout_against_library_gemm():
    """P8: the 128x4 scale tiles, handed to a library's block-scaled GEMM,
    give the fp64 product of our own dequantized operands: the library's
    reading of the tiled scale layout agrees with ours.  Tried in order:
    cuBLASLt MXFP4 on the packed codes (also checks the nibble order),
    cuBLASLt MXFP8 on the codes widened to E4M3 bytes (every E2M1 value is
    exact in E4M3; the scales and their layout are used as written), and
    torch._scaled_mm.  Skipped if none offers an MX GEMM here."""
    import cublaslt_mxfp4 as lt
    m, d, o = 256, 1152, 384
    A_bits = synth.activations(m, d, 41, "pixart")
    W_bits = synth.weights(o, d, seed=42, std=1.0)
    Fg, _ = lib_factors(d // 32, 43)
    qa, sfa, _ = run_kind("kron", A_bits, d, 1, Fg, y_debug=False)
    qw, sfw, _ = run_kind("identity", W_bits, d, 1, None, y_debug=False)
    out, errors = None, []
    ws = torch.empty(32 << 20, dtype=torch.uint8, device="cuda")
    # E2M1 code -> E4M3 byte of the same value (sign bit 3 -> bit 7)
    e2m1 = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0] * 2) * \
        torch.tensor([1.0] * 8 + [-1.0] * 8)
    to_e4m3 = e2m1.to(torch.float8_e4m3fn).view(torch.uint8).cuda()

    def widen(q):
        q = q.long()
        return to_e4m3[torch.stack([q & 15, q >> 4], dim=-1).reshape(q.shape[0], -1)]

    wa, ww = widen(qa), widen(qw)
    for elem, pa, pw, name in ((lt.CUDA_R_4F_E2M1, qa, qw, "MXFP4"),
                               (lt.CUDA_R_8F_E4M3, wa, ww, "MXFP8")):
        for dtype, code in ((torch.float32, lt.CUDA_R_32F), (torch.bfloat16, lt.CUDA_R_16BF)):
            c = torch.zeros((m, o), dtype=dtype, device="cuda")
            why = lt.mx_gemm(pa.data_ptr(), sfa.data_ptr(), m, pw.data_ptr(), sfw.data_ptr(), o, d,
                             c.data_ptr(), code, ws.data_ptr(), ws.numel(),
                             torch.cuda.current_stream().cuda_stream, elem)
            if why is None:
                out = c
                break
            errors.append(f"cuBLASLt {name} {dtype}: {why}")
        if out is not None:
            print("library consumer: cuBLASLt", name, out.dtype)
            break
    if out is None and hasattr(torch, "float4_e2m1fn_x2") and hasattr(torch, "float8_e8m0fnu"):
        out = torch_scaled_mm_mxfp4(qa, sfa, qw, sfw, m, o, d, errors)
    if out is None:
        pytest.skip(f"no MXFP4 block-scaled GEMM here: {errors}")
    print("library MXFP4 GEMM:", out.dtype, "declined:", errors)
    torch.cuda.synchronize()
    Aq = np_(kq.kq_dequantize(qa, sfa, m, d, layout=1)).astype(np.float64)
    Wq = np_(kq.kq_dequantize(qw, sfw, o, d, layout=1)).astype(np.float64)
    ref = Aq @ Wq.T
    got = out.float().cpu().numpy().astype(np.float64)
    scale = np.abs(Aq) @ np.abs(Wq).T
    tol = 2 ** -13 if out.dtype == torch.float32 else 2 ** -7
    assert np.all(np.abs(got - ref) <= tol * scale + 1e-30), float(
        (np.abs(got - ref) / (scale + 1e-30)).max())
    assert np.linalg.norm(got - ref) <= (1e-5 if out.dtype == torch.float32 else 1e-2) * \
        np.linalg.norm(ref)


def torch_scaled_mm_mxfp4(qa, sfa, qw, sfw, m, o, d, errors):
    nbp = -(-(d // 32) // 4) * 4
    sa, sw = sfa.view(torch.float8_e8m0fnu), sfw.view(torch.float8_e8m0fnu)
    out = None
    for shape_a, shape_w in (((-(-m // 128) * 128, nbp), (-(-o // 128) * 128, nbp)),
                             ((-1,), (-1,))):
        for out_dtype in (torch.bfloat16, torch.float32):
            try:
                out = torch._scaled_mm(qa.view(torch.float4_e2m1fn_x2),
                                       qw.view(torch.float4_e2m1fn_x2).t(),
                                       sa.reshape(shape_a), sw.reshape(shape_w),
                                       out_dtype=out_dtype)
                break
            except (RuntimeError, TypeError, NotImplementedError, ValueError) as e:
                errors.append(str(e)[-300:])
        if out is not None:
            break
    return out


# -------------------------------------- 16-bit side output (low-rank branch) --

DUAL_SHAPES = [(256, 1152), (300, 2240), (7, 96), (129, 160), (1, 32)]


def run_dual(A_bits, d, layout, factors_gpu, y_debug=True, at=None, q=None, sf=None):
    records = kq.kq_expand_blocks(dev(factors_gpu), kq.KQ_K_BF16X3)
    return kq.kq_quantize_mxfp4_dual(to_bf16(A_bits), records, d, layout=layout, q=q, sf=sf,
                                     at=at, y_debug=y_debug)


@pytest.mark.parametrize("m,d", DUAL_SHAPES, ids=[f"{m}x{d}" for m, d in DUAL_SHAPES])
def test_dual_side_output_parity(m, d):
    """kq_quantize_mxfp4_dual: codes and scales under rules (i)-(iii) and
    identical to the single-output call; the bf16 side output under rules
    (iv)-(v); guard bytes around the side output (ldat > d) untouched."""
    nb = d // 32
    A_bits = synth.activations(m, d, 91 + m, "flux")
    pg, po = lib_factors(nb, 93 + d)
    ldat = d + 24
    for layout in (0, 1):
        at_store = torch.full((m + 2, ldat), -7.0, dtype=torch.bfloat16, device="cuda")
        at = at_store[1:m + 1, :]
        q, sf, at_out, y = run_dual(A_bits, d, layout, pg, at=at[:, :ldat])
        assert at_out.data_ptr() == at.data_ptr()
        res = parity.check(A_bits, d, "kron", po, layout, np_(q), np_(sf), np_(y))
        side = parity.check_side_output(A_bits, d, "kron", po,
                                        np_(at.contiguous().view(torch.int16)).view(np.uint16),
                                        np_(y))
        guard = np_(at_store.float())
        assert (guard[0] == -7.0).all() and (guard[m + 1] == -7.0).all()
        assert (guard[1:m + 1, d:] == -7.0).all(), "side-output row padding overwritten"
        nsf = kq.kq_sf_bytes(m, d, layout)       # the buffers may be longer (>= 16 bytes)
        q1, sf1, _ = run_kind("kron_umma", A_bits, d, layout, pg, y_debug=False)
        assert torch.equal(q, q1) and torch.equal(sf[:nsf], sf1[:nsf])
        # the production launch (no debug output) writes the same bytes
        q2, sf2, at2, _ = run_dual(A_bits, d, layout, pg, y_debug=False)
        assert torch.equal(q, q2) and torch.equal(sf[:nsf], sf2[:nsf])
        assert torch.equal(at[:, :d].contiguous().view(torch.int16), at2.view(torch.int16))
        print(m, d, layout, res, side)


def test_dual_side_output_flux_ffn_down():
    """FLUX FFN-down layer (4608 x 12288) at full size, sampled rows (first
    and last tiles included)."""
    m, d = 4608, 12288
    A_bits = synth.activations(m, d, synth.SEED_A + 3, "flux")
    pg, po = lib_factors(d // 32, synth.SEED_FACTORS + 3)
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([np.arange(130), np.arange(m - 130, m),
                                     rng.choice(m, 500, replace=False)]))
    q, sf, at, y = run_dual(A_bits, d, 1, pg)
    parity.check(A_bits, d, "kron", po, 1, np_(q), np_(sf), np_(y), rows)
    side = parity.check_side_output(A_bits, d, "kron", po, np_(at.view(torch.int16)).view(np.uint16),
                                    np_(y), rows)
    print(side)


# ------------------------------------------- full-row Walsh-Hadamard baseline --

FWHT_SHAPES = [(3, 128), (130, 256), (64, 1024), (129, 2048), (17, 4096), (5, 8192), (9, 16384)]


@pytest.mark.parametrize("m,d", FWHT_SHAPES, ids=[f"{m}x{d}" for m, d in FWHT_SHAPES])
def test_fwht_parity(m, d):
    """kq_fwht_quantize_mxfp4 against the oracle's fast transform: rules
    (i)-(iii), both scale layouts, ragged m, lda > d, guard bytes around q."""
    lda, ldq = d + 64, d // 2 + 32
    A_bits = synth.activations(m, d, 300 + m, "flux", lda=lda)
    for layout in (0, 1):
        sfb = kq.kq_sf_bytes(m, d, layout)
        q_store = torch.full((m + 2, ldq), 0xA5, dtype=torch.uint8, device="cuda")
        q = q_store[1:m + 1]
        sf = torch.full((max(sfb, 16),), 0xA5, dtype=torch.uint8, device="cuda")
        _, _, y = kq.kq_fwht_quantize_mxfp4(to_bf16(A_bits), d, layout=layout, q=q, sf=sf,
                                            y_debug=True)
        qs = np_(q_store)
        assert (qs[0] == 0xA5).all() and (qs[m + 1] == 0xA5).all()
        assert (qs[1:m + 1, d // 2:] == 0xA5).all()
        res = parity.check(np.ascontiguousarray(A_bits[:, :d]), d, "fwht", None, layout,
                           np_(q)[:, :d // 2], np_(sf)[:sfb], np_(y))
        q2, sf2, _ = kq.kq_fwht_quantize_mxfp4(to_bf16(A_bits), d, layout=layout)
        assert torch.equal(q[:, :d // 2], q2) and torch.equal(sf[:sfb], sf2[:sfb])
        print(m, d, layout, res)


def test_fwht_table3_shape_sampled():
    """The pages' Table 3 shape m = 4096, d = 16384 at full size (sampled rows)."""
    m, d = 4096, 16384
    A_bits = synth.activations(m, d, 333, "flux")
    q, sf, y = kq.kq_fwht_quantize_mxfp4(to_bf16(A_bits), d, layout=1, y_debug=True)
    rows = np.unique(np.concatenate([np.arange(4), np.arange(m - 4, m),
                                     np.random.default_rng(5).choice(m, 200, replace=False)]))
    parity.check(A_bits, d, "fwht", None, 1, np_(q), np_(sf), np_(y), rows)


def test_identity_factors_reduce_to_bare_quantizer():
    """Degenerate case of the method: with every factor the 2x2 identity,
    K_j = I and y = a exactly (the three-term bf16 split of 0 and 1 is exact,
    and so are the butterfly's products), so both KroQuant paths must write
    the bare quantizer's bytes, bit for bit, in both scale layouts."""
    m, d = 300, 2240
    A_bits = synth.activations(m, d, 404, "sana")
    eye = np.tile(np.eye(2, dtype=np.float32), (d // 32, 5, 1, 1))
    for layout in (0, 1):
        nsf = kq.kq_sf_bytes(m, d, layout)
        q0, sf0, _ = run_kind("identity", A_bits, d, layout, y_debug=False)
        for kind in ("kron", "kron_umma", "kron_k2"):
            q, sf, y = run_kind(kind, A_bits, d, layout, eye)
            assert torch.equal(q, q0) and torch.equal(sf[:nsf], sf0[:nsf]), kind
            assert np.array_equal(np_(y), synth.bf16_bits_to_f32(A_bits)), kind


# ------------------------------------------- consumer W4A4 product (eq. 11) --

def mx_operand(rows, k, seed, lo=112, hi=140):
    """Random packed codes and scales; the scales placed in the 128x4 tiled
    layout by the oracle, padding bytes 0xFF (E8M0 NaN: a kernel that used
    one would put NaN into the product).  Returns (q, sf_rowmajor, sf_tiled)."""
    q = synth.packed_codes(rows, k, seed)
    sf = synth.scale_bytes(rows, k // 32, seed + 1, lo, hi)
    return q, sf, O.sf_place(sf, 1, fill=255)


def gemm_tolerance(Aq, Wq, k):
    """fp32 accumulation: every product is exact; each 16-deep tensor-core
    step and each addition into the accumulator rounds once, relative to
    at most sum |a_k w_k|."""
    return (k / 16 + 16) * 2.0 ** -23 * (np.abs(Aq) @ np.abs(Wq).T)


def check_product(got, Aq, Wq, k):
    ref = Aq @ Wq.T
    tol = gemm_tolerance(Aq, Wq, k)
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(np.isfinite(got))
    assert np.all(err <= tol), float((err / (tol + 1e-300)).max())
    return float((err / (tol + 1e-300)).max())


GEMM_SHAPES = [(256, 256, 1152), (300, 200, 96), (129, 384, 160), (1, 1, 32), (131, 130, 3072),
               (128, 128, 64), (5, 700, 2240), (130, 136, 5600), (64, 64, 224), (257, 260, 1024)]


GEMM_VARIANTS = {"mxf4": kq.GEMM_MXF4, "mxf4_narrow": kq.GEMM_MXF4_NARROW,
                 "mxf4_wide": kq.GEMM_MXF4_WIDE, "dequant_bf16": kq.GEMM_DEQUANT_BF16}


@pytest.mark.parametrize("variant", list(GEMM_VARIANTS))
@pytest.mark.parametrize("m,n,k", GEMM_SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in GEMM_SHAPES])
def test_w4a4_gemm_random_codes(m, n, k, variant):
    """C = deq(qa) deq(qw)^T on random codes and scales against the fp64
    product of the oracle's dequantization; ragged m, n and k (an odd block
    count puts a padding block, scale byte 0xFF, inside the last K = 64
    instruction), C pitch wider than n with canaries in the gap."""
    qa, _, sfa = mx_operand(m, k, 7 * m + k)
    qw, _, sfw = mx_operand(n, k, 11 * n + k + 1)
    ldc = n + 4 + (-(n + 4)) % 4
    c = torch.full((m, ldc), 12345.0, dtype=torch.float32, device="cuda")
    kq.kq_w4a4_gemm(dev(qa), dev(sfa), dev(qw), dev(sfw), m, n, k, c=c,
                    variant=GEMM_VARIANTS[variant])
    got = np_(c)
    assert np.all(got[:, n:] == 12345.0)
    Aq = O.dequantize(qa, sfa, 1, m, k)
    Wq = O.dequantize(qw, sfw, 1, n, k)
    print("max error / bound:", check_product(got[:, :n], Aq, Wq, k))


def test_w4a4_gemm_scale_extremes():
    """Left scales 2^-127 .. 2^-125 (the dequantized left operand is partly
    subnormal) against right scales 2^123 .. 2^125: products of order one
    that only come out right if no operand is flushed to zero."""
    m, n, k = 130, 140, 256
    qa, _, sfa = mx_operand(m, k, 91, lo=0, hi=2)
    qw, _, sfw = mx_operand(n, k, 92, lo=250, hi=252)
    got = np_(kq.kq_w4a4_gemm(dev(qa), dev(sfa), dev(qw), dev(sfw), m, n, k))
    Aq = O.dequantize(qa, sfa, 1, m, k)
    Wq = O.dequantize(qw, sfw, 1, n, k)
    print("max error / bound:", check_product(got, Aq, Wq, k))


def test_w4a4_gemm_flux_ffn_down_sampled():
    """The FLUX.1 FFN down projection at full size (m = 4608 tokens, k = 12288,
    n = 3072 output channels); all columns of 192 sampled rows (first, last,
    random) against the oracle."""
    m, n, k = 4608, 3072, 12288
    qa, sfa_rm, sfa = mx_operand(m, k, 501)
    qw, _, sfw = mx_operand(n, k, 502)
    got = np_(kq.kq_w4a4_gemm(dev(qa), dev(sfa), dev(qw), dev(sfw), m, n, k))
    rows = np.unique(np.concatenate([np.arange(64), np.arange(m - 64, m),
                                     np.random.default_rng(503).choice(m, 64, replace=False)]))
    Aq = O.dequantize(qa[rows], O.sf_place(sfa_rm[rows], 1), 1, len(rows), k)
    Wq = O.dequantize(qw, sfw, 1, n, k)
    print("max error / bound:", check_product(got[rows], Aq, Wq, k))


@pytest.mark.parametrize("variant", ["mxf4_narrow", "mxf4_wide"])
def test_w4a4_gemm_many_tiles_ragged(variant):
    """Several tiles per CTA (2 to 4 on 152 SMs) with ragged m and n and an
    odd block count (k = 1120: a partial last stage with a padding block),
    so that the accumulators, stage ring and barrier phases run on across
    tile boundaries; all columns of 160 sampled rows against the oracle."""
    m, n, k = 4096 + 33, 1280 + 8, 1120
    qa, sfa_rm, sfa = mx_operand(m, k, 601)
    qw, _, sfw = mx_operand(n, k, 602)
    got = np_(kq.kq_w4a4_gemm(dev(qa), dev(sfa), dev(qw), dev(sfw), m, n, k,
                              variant=GEMM_VARIANTS[variant]))
    rows = np.unique(np.concatenate([np.arange(48), np.arange(m - 48, m),
                                     np.random.default_rng(603).choice(m, 64, replace=False)]))
    Aq = O.dequantize(qa[rows], O.sf_place(sfa_rm[rows], 1), 1, len(rows), k)
    Wq = O.dequantize(qw, sfw, 1, n, k)
    print("max error / bound:", check_product(got[rows], Aq, Wq, k))


BF16_GEMM_SHAPES = [(256, 384, 1152), (300, 129, 100), (1, 1, 8), (129, 257, 3072)]


@pytest.mark.parametrize("m,n,k", BF16_GEMM_SHAPES,
                         ids=[f"{m}x{n}x{k}" for m, n, k in BF16_GEMM_SHAPES])
def test_bf16_gemm(m, n, k):
    """C = A W^T for bf16 operands (row pitch wider than k, zero-padded by the
    caller's layout only up to the pitch) against the fp64 product."""
    lda = k + (-k) % 8 + 8
    A_bits = synth.activations(m, k, 600 + m, "pixart", lda=lda)
    W_bits = synth.activations(n, k, 700 + n, "gauss_outlier8", lda=lda)
    A_bits[:, k:] = 0x7FC0                     # NaN beyond k: must not be read
    W_bits[:, k:] = 0x7FC0
    got = np_(kq.kq_bf16_gemm(to_bf16(A_bits), to_bf16(W_bits), k=k))
    a = synth.bf16_bits_to_f32(A_bits[:, :k]).astype(np.float64)
    w = synth.bf16_bits_to_f32(W_bits[:, :k]).astype(np.float64)
    print("max error / bound:", check_product(got, a, w, k))


def test_gemm_empty_is_noop():
    c = torch.full((4, 8), 7.0, device="cuda")
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")
    kq.kq_w4a4_gemm(z, z, z, z, 0, 8, 64, c=c)
    kq.kq_w4a4_gemm(z, z, z, z, 4, 0, 64, c=c)
    assert torch.all(c == 7.0)
    out = kq.kq_layer_error(c[:0], c[:0])
    assert np.array_equal(np_(out), [0.0, 0.0])


def device_layer_error(A_bits, W_bits, d, Fg, layout_a_kind="kron_umma"):
    """eq. (2) entirely on the device: quantize A T (tensor-core path) and
    W T^{-T} (butterfly on the inverse-transposed factors), the W4A4 product,
    the bf16 reference product, the fp64 error sums."""
    m, o = A_bits.shape[0], W_bits.shape[0]
    qa, sfa, _ = run_kind(layout_a_kind, A_bits, d, 1, Fg, y_debug=False)
    qw, sfw, _ = run_kind("kron", W_bits, d, 1, kq.kq_invert_transpose_factors(Fg),
                          y_debug=False)
    cq = kq.kq_w4a4_gemm(qa, sfa, qw, sfw, m, o, d)
    cr = kq.kq_bf16_gemm(to_bf16(A_bits), to_bf16(W_bits))
    s = np_(kq.kq_layer_error(cq, cr))
    return math.sqrt(s[0]), math.sqrt(s[1])


def reference_norm_tolerance(A_bits, W_bits, d):
    """| ||C|| - ||A W^T|| | <= ||C - A W^T||_F, bounded element by element
    by the fp32 accumulation bound of the product."""
    a = synth.bf16_bits_to_f32(A_bits).astype(np.float64)
    w = synth.bf16_bits_to_f32(W_bits).astype(np.float64)
    return float(np.linalg.norm(gemm_tolerance(a, w, d)))


@pytest.mark.parametrize("factor_kind", ["random", "hadamard"])
def test_layer_error_on_device_config0(factor_kind):
    """Acceptance (iii) with every step on the GPU: ||E(T)||_F within 1e-3
    relative of the oracle's; ||A W^T||_F within the fp32 accumulation bound."""
    m, d, o = 256, 1152, 1152
    nb = d // 32
    A_bits = synth.activations(m, d, synth.SEED_A, "gauss_outlier8")
    W_bits = synth.weights(o, d)
    if factor_kind == "random":
        Fg, Fo = lib_factors(nb, synth.SEED_FACTORS)
    else:
        Fg = synth.hadamard_factors(nb)
        Fo = Fg.astype(np.float64)
    e_gpu, r_gpu = device_layer_error(A_bits, W_bits, d, Fg)
    e_ref, ref = O.layer_error(A_bits, W_bits, d, Fo, layout=1)
    assert abs(e_gpu - e_ref) <= 1e-3 * e_ref, (e_gpu, e_ref)
    assert abs(r_gpu - ref) <= reference_norm_tolerance(A_bits, W_bits, d), (r_gpu, ref)


@pytest.mark.parametrize("name,m,d,model,cfg", synth.CONFIG1 + synth.CONFIG2 + synth.CONFIG3,
                         ids=[c[0] for c in synth.CONFIG1 + synth.CONFIG2 + synth.CONFIG3])
def test_layer_error_on_device_configs(name, m, d, model, cfg):
    """The same on configs 1-3: the first 512 rows of A, a square weight of
    o = d output channels."""
    m, o = 512, d
    A_bits = synth.activations(m, d, synth.SEED_A + cfg, model)
    W_bits = synth.weights(o, d, seed=synth.SEED_W + cfg)
    Fg, Fo = lib_factors(d // 32, synth.SEED_FACTORS + cfg)
    e_gpu, r_gpu = device_layer_error(A_bits, W_bits, d, Fg)
    e_ref, ref = O.layer_error(A_bits, W_bits, d, Fo, layout=1)
    assert abs(e_gpu - e_ref) <= 1e-3 * e_ref, (e_gpu, e_ref)
    assert abs(r_gpu - ref) <= reference_norm_tolerance(A_bits, W_bits, d), (r_gpu, ref)


def test_w4a4_gemm_variants_agree_on_quantizer_output():
    """The block-scaled FP4 instruction and the bf16 dequantization route
    agree on the quantizer's own output to the fp32 accumulation bound
    (both form exact products)."""
    m, n, k = 384, 256, 3072
    A_bits = synth.activations(m, k, 801, "flux")
    W_bits = synth.weights(n, k, seed=802)
    Fg, _ = lib_factors(k // 32, 803)
    qa, sfa, _ = run_kind("kron_umma", A_bits, k, 1, Fg, y_debug=False)
    qw, sfw, _ = run_kind("kron", W_bits, k, 1, kq.kq_invert_transpose_factors(Fg), y_debug=False)
    c0 = np_(kq.kq_w4a4_gemm(qa, sfa, qw, sfw, m, n, k, variant=kq.GEMM_MXF4)).astype(np.float64)
    c1 = np_(kq.kq_w4a4_gemm(qa, sfa, qw, sfw, m, n, k, variant=kq.GEMM_DEQUANT_BF16))
    Aq = O.dequantize(np_(qa), np_(sfa), 1, m, k)
    Wq = O.dequantize(np_(qw), np_(sfw), 1, n, k)
    tol = 2 * gemm_tolerance(Aq, Wq, k)
    assert np.all(np.abs(c0 - c1) <= tol)


# ------------------------------------------------------- shared factors --

SHARED_SHAPES = [(256, 1152), (300, 2240), (7, 96), (129, 5600)]


@pytest.mark.parametrize("path", ["umma", "k2"])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("m,d", SHARED_SHAPES, ids=[f"{m}x{d}" for m, d in SHARED_SHAPES])
def test_shared_factors(m, d, layout, path):
    """One factor set for every block: parity with the oracle given the set
    repeated d/32 times (rules i-iii), and the same bytes as the per-block
    entry point given that repeated set (the expanded record, or the raw
    factors the K2 kernel builds it from)."""
    nb = d // 32
    A_bits = synth.activations(m, d, 1700 + m, "sana")
    lu = synth.lu_params(1, 1701)
    F1 = kq.kq_lu_to_factors(lu, +1)                          # [1, 5, 2, 2]
    Fo = np.broadcast_to(O.lu_to_factors(lu.astype(np.float64), +1).astype(np.float32)
                         .astype(np.float64), (nb, 5, 2, 2))
    A = to_bf16(A_bits)
    if path == "umma":
        rec = kq.kq_expand_blocks(dev(F1), kq.KQ_K_BF16X3)
        q, sf, y = kq.kq_quantize_mxfp4_shared(A, d, K_expanded=rec, layout=layout, y_debug=True)
        Frep = np.ascontiguousarray(np.broadcast_to(F1, (nb, 5, 2, 2)))
        q2, sf2, _ = kq.kq_quantize_mxfp4(A, d, K_expanded=kq.kq_expand_blocks(dev(Frep), kq.KQ_K_BF16X3),
                                          layout=layout, variant=kq.VARIANT_UMMA)
    else:
        q, sf, y = kq.kq_quantize_mxfp4_shared(A, d, factors=dev(F1[0]), layout=layout, y_debug=True)
        Frep = np.ascontiguousarray(np.broadcast_to(F1, (nb, 5, 2, 2)))
        q2, sf2, _ = kq.kq_quantize_mxfp4(A, d, factors=dev(Frep), layout=layout,
                                          variant=kq.VARIANT_K2)
    nbytes = kq.kq_sf_bytes(m, d, layout)
    assert np.array_equal(np_(q), np_(q2)) and np.array_equal(np_(sf)[:nbytes], np_(sf2)[:nbytes])
    parity.check(A_bits, d, "kron", np.ascontiguousarray(Fo), layout, np_(q), np_(sf), np_(y))


# ------------------------------------------------------------ fp16 input --

F16_SHAPES = [(256, 1152), (300, 2240), (7, 96), (4096, 4096)]


@pytest.mark.parametrize("kind", ["kron", "diag", "hadamard", "identity", "fwht"])
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("m,d", F16_SHAPES, ids=[f"{m}x{d}" for m, d in F16_SHAPES])
def test_f16_input_parity(m, d, layout, kind):
    """fp16 activations (PixArt-Sigma's format, and the pages' timing
    precision) through the CUDA-core quantizers, against the oracle reading
    the same fp16 patterns: rules (i)-(iii)."""
    if kind == "fwht" and (d & (d - 1) or d < 128):
        pytest.skip("the full-row transform needs a power-of-two d >= 128")
    A_bits = synth.activations(m, d, 1900 + m, "pixart", fmt="f16")
    A = dev(A_bits.view(np.int16)).view(torch.float16)
    gp, op = None, None
    if kind == "kron":
        gp, op = lib_factors(d // 32, 1901)
    elif kind == "diag":
        s = synth.smooth_scales(d)
        gp, op = s, s.astype(np.float64)
    q, sf, y = kq.kq_quantize_mxfp4_ex(A, kind, None if gp is None else dev(gp), d,
                                       in_format=kq.KQ_IN_F16, layout=layout, y_debug=True)
    rows = None if m * d <= 2_000_000 else np.arange(0, m, 7)
    parity.check(A_bits, d, kind, op, layout, np_(q), np_(sf), np_(y), rows, in_format="f16")


def test_ex_bf16_matches_entry_points():
    """kq_quantize_mxfp4_ex with bf16 input writes the bytes of the
    dedicated entry points (butterfly, diagonal, Hadamard, identity)."""
    m, d = 300, 2240
    A_bits = synth.activations(m, d, 1950, "sana")
    A = to_bf16(A_bits)
    F, _ = lib_factors(d // 32, 1951)
    s = synth.smooth_scales(d)
    pairs = [
        (kq.kq_quantize_mxfp4_ex(A, "kron", dev(F), d, layout=1),
         kq.kq_quantize_mxfp4(A, d, factors=dev(F), layout=1, variant=kq.VARIANT_BUTTERFLY)),
        (kq.kq_quantize_mxfp4_ex(A, "diag", dev(s), d, layout=1),
         kq.kq_smooth_quantize_mxfp4(A, dev(s), d, layout=1)),
        (kq.kq_quantize_mxfp4_ex(A, "hadamard", None, d, layout=1),
         kq.kq_hadamard_quantize_mxfp4(A, d, layout=1)),
        (kq.kq_quantize_mxfp4_ex(A, "identity", None, d, layout=1),
         kq.kq_quantize_mxfp4(A, d, layout=1)),
    ]
    for (q1, s1, _), (q2, s2, _) in pairs:
        assert torch.equal(q1, q2) and torch.equal(s1, s2)


@pytest.mark.parametrize("m,d", [(256, 1152), (1024, 1152), (1024, 3072), (4608, 3072)])
def test_default_dispatch(m, d):
    """kq_quantize_mxfp4 runs the records path whenever the expanded blocks
    are given (with or without the raw factors), and K2 when only the raw
    factors are: its bytes equal those of that variant called explicitly."""
    A_bits = synth.activations(m, d, 2100 + m, "flux")
    A = to_bf16(A_bits)
    F, _ = lib_factors(d // 32, 2101)
    Fd = dev(F)
    KX = kq.kq_expand_blocks(Fd, kq.KQ_K_BF16X3)
    want_r = kq.kq_quantize_mxfp4(A, d, K_expanded=KX, layout=1, variant=kq.VARIANT_UMMA)
    want_k2 = kq.kq_quantize_mxfp4(A, d, factors=Fd, layout=1, variant=kq.VARIANT_K2)
    for got, want in ((kq.kq_quantize_mxfp4(A, d, factors=Fd, K_expanded=KX, layout=1), want_r),
                      (kq.kq_quantize_mxfp4(A, d, K_expanded=KX, layout=1), want_r),
                      (kq.kq_quantize_mxfp4(A, d, factors=Fd, layout=1), want_k2)):
        assert torch.equal(got[0], want[0]) and torch.equal(got[1], want[1])


# ------------------------------------------ a pipeline wait that runs out --

STALL_LIMIT_NS = 20_000_000        # 20 ms: every normal wait ends in microseconds


def tile_blocks(t, ncol, nb, m):
    """(rows, blocks) of tile t of the tcgen05 kernel (128 rows x 2 blocks)."""
    rt, ct = divmod(t, ncol)
    rows = np.arange(rt * 128, min(rt * 128 + 128, m))
    blocks = np.array([j for j in (2 * ct, 2 * ct + 1) if j < nb])
    return rows, blocks


@pytest.mark.parametrize("layout", [0, 1])
def test_stalled_pipeline_marks_unfinished_blocks(layout):
    """The error path of the fixed-walk kernel, made to run by a wait that
    runs out (nothing faults): CTA 5's producer arms the ring stage of its
    4th tile but never issues that tile's loads, and every wait gives up
    after 20 ms.  The kernel must return; the blocks the CTA did not finish
    get the E8M0 NaN byte 0xFF and zero codes, every other byte equals a
    normal run.  With 6 ring stages and two MMA issuers taking alternate
    tiles, the CTA finishes its tiles 0-2, 4, 6 and 8 (the other issuer's
    tiles up to the one whose stage reuse waits on the skipped tile) and no
    other."""
    m, d = 4608, 3072                       # 36 x 48 tiles; CTA 5 owns 12 of them
    nb = d // 32
    A = to_bf16(synth.activations(m, d, 2500, "flux"))
    F, _ = lib_factors(nb, 2501)
    KX = kq.kq_expand_blocks(dev(F), kq.KQ_K_BF16X3)
    q0, s0, _ = kq.kq_quantize_mxfp4(A, d, K_expanded=KX, layout=layout)
    nsf = kq.kq_sf_bytes(m, d, layout)
    ncol, ntiles, grid, cta = 48, 36 * 48, 152, 5
    walk = list(range(cta, ntiles, grid))   # the CTA's tiles in order
    assert len(walk) == 12
    q1 = torch.full_like(q0, 0xA5)
    s1 = torch.full_like(s0, 0xA5)
    kq.kq_test_quantize_stall(A, KX, d, walk[3], STALL_LIMIT_NS, layout=layout, q=q1, sf=s1)
    torch.cuda.synchronize()
    want_q, want_s = np_(q0).copy(), np_(s0)[:nsf].copy()
    for pos in (3, 5, 7, 9, 10, 11):
        rows, blocks = tile_blocks(walk[pos], ncol, nb, m)
        for j in blocks:
            want_q[np.ix_(rows, np.arange(16 * j, 16 * j + 16))] = 0
            off = (rows * nb + j) if layout == 0 else \
                ((rows // 128) * ((nb + 3) // 4) + j // 4) * 512 + (rows % 32) * 16 + \
                ((rows % 128) // 32) * 4 + j % 4
            want_s[off] = 0xFF
    got_q, got_s = np_(q1), np_(s1)[:nsf]
    assert np.array_equal(got_s, want_s), int((got_s != want_s).sum())
    assert np.array_equal(got_q, want_q), int((got_q != want_q).sum())
    # the same hook with no tile skipped writes the normal bytes
    kq.kq_test_quantize_stall(A, KX, d, -1, STALL_LIMIT_NS, layout=layout, q=q1, sf=s1)
    torch.cuda.synchronize()
    assert torch.equal(q1, q0) and torch.equal(s1[:nsf], s0[:nsf])



def test_k2_matches_records_path_outside_flags():
    """K2 builds K_j from the factors in fp32 (products rounded four times,
    then split exactly into three bf16 terms); the records path expands it
    in fp64.  Both are checked against the oracle elsewhere; here their codes
    agree on every unflagged element of the FLUX FFN-down layer, and their
    y differ by no more than the sum of the two 2^-16 allowances."""
    m, d = 4608, 12288
    A_bits = synth.activations(m, d, synth.SEED_A + 3, "flux")
    Fg, Fo = lib_factors(d // 32, synth.SEED_FACTORS + 3)
    qk, sk, yk = run_kind("kron_k2", A_bits, d, 1, Fg)
    qr, sr, yr = run_kind("kron_umma", A_bits, d, 1, Fg)
    rows = np.arange(0, m, 5)
    ref = parity.reference(A_bits, d, "kron", Fo, rows)
    strict = ref["flags"] == 0
    ck, cr = parity.unpack(np_(qk)[rows], d), parity.unpack(np_(qr)[rows], d)
    assert np.array_equal(ck[strict], cr[strict])
    diff = np.abs(np_(yk)[rows].astype(np.float64) - np_(yr)[rows])
    assert np.all(diff <= np.ldexp(ref["bound"], -15))

"""Planted mistakes: each test builds a copy of the oracle with one
plausible mistake (the C arithmetic recompiled, or the Python layer-error
code re-executed as a separate module) and checks that the pins reject it.
This shows the pins are strong enough to catch that class of error in the
oracle itself.  The mistakes are planted only in temporary copies of the
oracle, on the CPU.
"""
import inspect
import types

import pytest

import test_oracle_pins as pins
from oracle import kq_oracle

# (name, original text, mutated text, pins that must fail)
MUTANTS = [
    ("ties_away_from_zero", "q = rint(a / step) * step;", "q = round(a / step) * step;",
     [pins.test_e2m1_rounding_golden, pins.test_worked_block]),
    ("reversed_bit_order", "int bit = 5 - k;", "int bit = k - 1;",
     [pins.test_orientation_and_bit_order, pins.test_expand_matches_nested_kron]),
    ("transposed_factor", "p *= G[(k - 1) * 4 + rb * 2 + cb];",
     "p *= G[(k - 1) * 4 + cb * 2 + rb];",
     [pins.test_orientation_and_bit_order, pins.test_expand_matches_nested_kron]),
    ("scale_offset_by_one", "int e = (ex - 1) - 2;", "int e = (ex - 1) - 1;",
     [pins.test_e8m0_edges, pins.test_worked_block]),
    ("sf_tile_rows_swapped", "return tile * 512 + (i % 32) * 16 + ((i % 128) / 32) * 4 + (kb % 4);",
     "return tile * 512 + (i % 32) * 4 + ((i % 128) / 32) * 16 + (kb % 4);",
     [pins.test_sf_blocked_offsets_golden]),
    ("nibbles_swapped", "(uint8_t)(codes[2 * k] | (codes[2 * k + 1] << 4))",
     "(uint8_t)(codes[2 * k + 1] | (codes[2 * k] << 4))",
     [pins.test_worked_block]),
    ("zero_sign_dropped", "uint8_t sign = signbit(v) ? 8 : 0;", "uint8_t sign = (v < 0) ? 8 : 0;",
     [pins.test_e2m1_rounding_golden, pins.test_worked_block]),
    ("dropped_last_term", "for (int r = 0; r < 32; ++r) {\n                    double t",
     "for (int r = 0; r < 31; ++r) {\n                    double t",
     [pins.test_orientation_and_bit_order, pins.bruteforce_small_case]),
    ("hadamard_sign", "? -s : s;", "? s : -s;", [pins.test_hadamard_closed_form]),
    ("lu_wrong_entry", "G[3] = c * b + u22;", "G[3] = c * a + u22;",
     [pins.test_lu_factor_determinants]),
    ("bf16_ties_away", "rint(a / spacing) * spacing", "round(a / spacing) * spacing",
     [pins.test_bf16_rounding_golden, pins.test_bf16_rounding_is_nearest_even]),
    ("bf16_subnormal_spacing", "if (e < -126) e = -126;", "if (e < -127) e = -127;",
     [pins.test_bf16_rounding_golden, pins.test_bf16_rounding_is_nearest_even]),
    ("fwht_butterfly_sign", "v[j + h] = x - z;", "v[j + h] = z - x;",
     [lambda o: pins.test_fwht_matches_library_hadamard(o, 64), pins.test_fwht_closed_forms]),
    ("f16_exponent_bias", "v = ldexp((double)(1024 + f), e - 25);",
     "v = ldexp((double)(1024 + f), e - 24);",
     [pins.test_f16_conversion_all_patterns, pins.test_f16_closed_forms]),
    ("f16_subnormal_scale", "v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);",
     [pins.test_f16_conversion_all_patterns, pins.test_f16_closed_forms]),
]


@pytest.mark.parametrize("name,orig,mut,must_fail", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, oracle_lib, name, orig, mut, must_fail):
    src = kq_oracle.source_text()
    assert src.count(orig) == 1, f"mutation anchor for {name} not found exactly once"
    path = kq_oracle.build_variant(src.replace(orig, mut), str(tmp_path / f"lib_{name}.so"))
    with kq_oracle.swapped_library(path):
        for pin in must_fail:
            with pytest.raises(AssertionError):
                pin(kq_oracle)


# Mistakes in the Python side of the oracle: eq. (2)'s layer error.
# (name, original text, mutated text, pins that must fail)
PY_MUTANTS = [
    ("activations_not_transformed",
     'qa = quantize_activations(A, d, "kron", factors, layout)',
     'qa = quantize_activations(A, d, "identity", None, layout)',
     [pins.test_layer_error_golden, pins.test_layer_error_exact_on_grid]),
    ("weights_inverse_not_transposed",
     "np.linalg.inv(K[j]).T for j", "np.linalg.inv(K[j]) for j",
     [pins.test_layer_error_golden, pins.test_layer_error_exact_on_grid]),
    ("weights_take_K",
     'yw, bw = transform(W, d, "dense", inverse_transpose_blocks(factors))',
     'yw, bw = transform(W, d, "kron", factors)',
     [pins.test_layer_error_golden, pins.test_layer_error_exact_on_grid]),
    ("weights_not_transformed",
     'yw, bw = transform(W, d, "dense", inverse_transpose_blocks(factors))',
     'yw, bw = transform(W, d, "identity")',
     [pins.test_layer_error_golden, pins.test_layer_error_exact_on_grid]),
    ("product_without_transpose", "E = Aq @ Wq.T - ref", "E = Aq @ Wq - ref",
     [pins.test_layer_error_exact_on_grid]),
    ("error_sign", "E = Aq @ Wq.T - ref", "E = Aq @ Wq.T + ref",
     [pins.test_layer_error_golden, pins.test_layer_error_exact_on_grid]),
    ("reference_from_quantized", "ref = a @ w.T", "ref = Aq @ Wq.T",
     [pins.test_layer_error_golden]),
    ("norms_swapped", "return float(np.linalg.norm(E)), float(np.linalg.norm(ref))",
     "return float(np.linalg.norm(ref)), float(np.linalg.norm(E))",
     [pins.test_layer_error_golden, pins.test_layer_error_exact_on_grid]),
]


def python_variant(src_text: str, name: str):
    """The oracle's Python module re-executed from modified source, as a
    separate module object (the shared C library is unchanged)."""
    mod = types.ModuleType(f"kq_oracle_{name}")
    mod.__file__ = kq_oracle.__file__
    exec(compile(src_text, kq_oracle.__file__, "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,orig,mut,must_fail", PY_MUTANTS, ids=[m[0] for m in PY_MUTANTS])
def test_pins_catch_planted_layer_error_mistake(oracle_lib, name, orig, mut, must_fail):
    src = inspect.getsource(kq_oracle)
    assert src.count(orig) == 1, f"mutation anchor for {name} not found exactly once"
    mutant = python_variant(src.replace(orig, mut), name)
    # the unmodified source, run the same way, passes the same pins
    for pin in must_fail:
        pin(python_variant(src, "copy"))
        with pytest.raises(AssertionError):
            pin(mutant)

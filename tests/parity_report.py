"""Markdown table of the flag counts the GPU parity tests record.

Run the GPU suite with KQ_PARITY_REPORT=<file> (tests/parity.py appends one
JSON line per comparison), then ``python tests/parity_report.py <file>``.
Per (config, layer, kernel) it prints the compared elements, the elements the
oracle flags as within 1e-3 of a rounding midpoint, the blocks whose amax is
within 1e-3 of a power of two, the zero-magnitude elements whose sign is
undecided, how many codes / scales differ inside those flags (none may differ
outside them: the tests fail otherwise) and the largest pre-quantization error
as a fraction of the 2^-16 tolerance.  When a comparison ran with both scale
layouts the counts agree; the row shows the larger differences.
"""
import json
import sys

KINDS = {"kron": "butterfly", "kron_umma": "tcgen05 (records)", "kron_k2": "tcgen05 (K2)",
         "diag": "diagonal scale", "hadamard": "block Hadamard", "identity": "bare Q4"}


def main(path):
    rows = {}
    for line in open(path):
        r = json.loads(line)
        key = (r["config"], r["layer"], r["m"], r["d"], r["kind"])
        prev = rows.get(key)
        if prev is None:
            rows[key] = r
        else:
            for k in ("flagged_code_diffs", "flagged_scale_diffs", "y_max_err_over_tol"):
                if k in r:
                    prev[k] = max(prev.get(k, 0), r[k])
    print("| config | layer | m x d | kernel | elements | midpoint flags | pow-2 blocks | "
          "zero-sign | code diffs in flags | scale diffs in flags | max y err / tol |")
    print("|" + "---|" * 11)
    for (cfg, layer, m, d, kind), r in rows.items():
        y = r.get("y_max_err_over_tol")
        print(f"| {cfg} | {layer} | {m}x{d} | {KINDS.get(kind, kind)} | {r['elements']} | "
              f"{r['flag_midpoint']} | {r['flag_pow2_blocks']} | {r['flag_zero_sign']} | "
              f"{r['flagged_code_diffs']} | {r['flagged_scale_diffs']} | "
              f"{'' if y is None else f'{y:.3f}'} |")


if __name__ == "__main__":
    main(sys.argv[1])

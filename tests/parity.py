"""Comparison rules between the CUDA quantizer and the CPU oracle.

For every (row, block) the rules are:
  (i)   pre-quantization values: |y_gpu - y_ref| <= 2^-16 * sum_r |a_r K_rc|
        (the error scale of the dot product; cancellation makes a plain
        element-relative bound meaningless);
  (ii)  E8M0 scales and E2M1 codes bit-exact, except where the oracle flags
        an element: within 1e-3 relative of a rounding midpoint (flag 1) or
        in a block whose amax is within 1e-3 relative of a power of two
        (flag 2, scale and all codes of the block); an element whose
        magnitude rounds to 0 with |y| inside the error scale (flag 4) must
        match in magnitude only (its sign is not decided);
  (iii) same-precision requantization: the oracle's quantizer applied to
        the kernel's own fp32 y reproduces the kernel's scales and codes
        exactly, with no exceptions.

For the 16-bit side output A T (bf16, round to nearest even) of the dual
quantizer:
  (iv)  its value lies between the oracle's rounding of y_ref - tol and of
        y_ref + tol (rounding is monotone, so this is exactly "the bf16 of some
        value within the rule-(i) tolerance of the exact y"; most elements
        admit one pattern only, and those that admit two are counted);
  (v)   with the kernel's own fp32 y at hand, the side output is the oracle's
        rounding of it, bit for bit.
"""
from __future__ import annotations

import json
import os

import numpy as np

from oracle import kq_oracle as O


def unpack(q: np.ndarray, d: int) -> np.ndarray:
    q = np.asarray(q, np.uint8)[:, : d // 2]
    return np.stack([q & 15, q >> 4], axis=-1).reshape(q.shape[0], d)


def gather_scales(sf: np.ndarray, rows: np.ndarray, nb: int, layout: int) -> np.ndarray:
    """Scales of the given (global) rows as [len(rows), nb]."""
    sf = np.asarray(sf, np.uint8).ravel()
    if layout == O.SF_ROWMAJOR:
        return sf[(rows[:, None] * nb + np.arange(nb)[None, :])]
    i = rows[:, None].astype(np.int64)
    kb = np.arange(nb)[None, :].astype(np.int64)
    ncb = (nb + 3) // 4
    off = ((i // 128) * ncb + kb // 4) * 512 + (i % 32) * 16 + ((i % 128) // 32) * 4 + (kb % 4)
    return sf[off]


CHUNK = 4096


def reference(A_bits: np.ndarray, d: int, kind: str, param, rows: np.ndarray | None = None,
              in_format: str = "bf16") -> dict:
    """The oracle's result on the given rows (all if None), for check(ref=...)
    when one input is compared with several outputs."""
    m = A_bits.shape[0]
    rows = np.arange(m) if rows is None else np.asarray(rows, np.int64)
    src = A_bits if len(rows) == m else np.ascontiguousarray(A_bits[rows])
    y_ref, bound = O.transform(np.ascontiguousarray(src), d, kind, param, in_format=in_format)
    q_ref, sf_ref, flags = O.quantize(y_ref, bound, O.SF_ROWMAJOR)
    return dict(rows=rows, y=y_ref, bound=bound, q=q_ref, sf=sf_ref, flags=flags)


def record(config: str, layer: str, m: int, d: int, kind: str, layout: int, res: dict):
    """Append one parity result as a JSON line to $KQ_PARITY_REPORT (if set):
    the per-config flag counts reported next to the benchmark."""
    path = os.environ.get("KQ_PARITY_REPORT")
    if not path:
        return
    with open(path, "a") as f:
        f.write(json.dumps({"config": config, "layer": layer, "m": m, "d": d, "kind": kind,
                            "layout": layout, **res}) + "\n")


def check(A_bits: np.ndarray, d: int, kind: str, param, layout: int, q_gpu: np.ndarray,
          sf_gpu: np.ndarray, y_gpu: np.ndarray | None, rows: np.ndarray | None = None,
          in_format: str = "bf16", ref: dict | None = None) -> dict:
    """Apply rules (i)-(iii) on the given rows (all rows if None).  Raises
    AssertionError on a violation; returns the flagged counts.  Without a
    precomputed ``ref``, large row sets are checked in chunks of CHUNK rows
    (the counts summed) to bound the host memory."""
    nb = d // 32
    if ref is None:
        all_rows = np.arange(A_bits.shape[0]) if rows is None else np.asarray(rows, np.int64)
        if len(all_rows) > CHUNK:
            out = {}
            for k in range(0, len(all_rows), CHUNK):
                part = check(A_bits, d, kind, param, layout, q_gpu, sf_gpu, y_gpu,
                             all_rows[k:k + CHUNK], in_format)
                for key, v in part.items():
                    out[key] = max(out.get(key, 0.0), v) if key == "y_max_err_over_tol" \
                        else out.get(key, 0) + v
            return out
        ref = reference(A_bits, d, kind, param, rows, in_format)
    rows = ref["rows"]
    y_ref, bound, q_ref, sf_ref, flags = ref["y"], ref["bound"], ref["q"], ref["sf"], ref["flags"]
    codes_ref = unpack(q_ref, d)
    codes_gpu = unpack(np.asarray(q_gpu)[rows], d)
    sf_g = gather_scales(sf_gpu, rows, nb, layout)
    sf_r = sf_ref.reshape(len(rows), nb)

    out = {"elements": int(len(rows) * d)}
    # (i)
    if y_gpu is not None:
        yg = np.asarray(y_gpu, np.float64)[rows]
        err = np.abs(yg - y_ref)
        tol = np.ldexp(bound, -16)
        bad = err > tol
        assert not bad.any(), (f"{int(bad.sum())} values outside 2^-16 rule; worst ratio "
                               f"{float((err / np.maximum(tol, 1e-300)).max()):.3g}")
        out["y_max_err_over_tol"] = float((err / np.maximum(tol, 1e-300)).max())
    # (ii)
    edge_block = (flags.reshape(len(rows), nb, 32) & O.FLAG_POW2_EDGE).any(axis=2)
    sbad = (sf_g != sf_r) & ~edge_block
    assert not sbad.any(), f"{int(sbad.sum())} scale mismatches outside flagged blocks"
    exempt = (flags & (O.FLAG_MIDPOINT | O.FLAG_POW2_EDGE)) != 0
    zero_sign = ((flags & O.FLAG_ZERO_SIGN) != 0) & ~exempt
    strict = ~exempt & ~zero_sign
    cbad = (codes_gpu != codes_ref) & strict
    assert not cbad.any(), f"{int(cbad.sum())} code mismatches outside flags"
    zbad = ((codes_gpu & 7) != (codes_ref & 7)) & zero_sign
    assert not zbad.any(), f"{int(zbad.sum())} zero-magnitude mismatches"
    out["flag_midpoint"] = int(((flags & O.FLAG_MIDPOINT) != 0).sum())
    out["flag_pow2_blocks"] = int(edge_block.sum())
    out["flag_zero_sign"] = int(zero_sign.sum())
    out["flagged_code_diffs"] = int(((codes_gpu != codes_ref) & ~strict).sum())
    out["flagged_scale_diffs"] = int(((sf_g != sf_r) & edge_block).sum())
    # (iii)
    if y_gpu is not None:
        q2, sf2, _ = O.quantize(np.asarray(y_gpu, np.float64)[rows], None, O.SF_ROWMAJOR)
        assert np.array_equal(sf2.reshape(len(rows), nb), sf_g), "requantized scales differ"
        assert np.array_equal(unpack(q2, d), codes_gpu), "requantized codes differ"
    return out


def check_side_output(A_bits: np.ndarray, d: int, kind: str, param, at_gpu: np.ndarray,
                      y_gpu: np.ndarray | None, rows: np.ndarray | None = None) -> dict:
    """Rules (iv)-(v) for the bf16 side output on the given rows (all if None)."""
    m = A_bits.shape[0]
    rows = np.arange(m) if rows is None else np.asarray(rows, np.int64)
    y_ref, bound = O.transform(np.ascontiguousarray(A_bits[rows]), d, kind, param)
    tol = np.ldexp(bound, -16)
    lo = O.round_bf16(y_ref - tol)
    hi = O.round_bf16(y_ref + tol)
    at = np.asarray(at_gpu)[rows][:, :d].astype(np.uint16)

    def val(b):
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)

    v, vlo, vhi = val(at), val(lo), val(hi)
    bad = (v < vlo) | (v > vhi) | np.isnan(v)
    assert not bad.any(), f"{int(bad.sum())} side-output values outside the rounding window"
    out = {"side_elements": int(at.size), "side_two_choices": int((lo != hi).sum())}
    if y_gpu is not None:
        want = O.round_bf16(np.asarray(y_gpu, np.float64)[rows])
        assert np.array_equal(want, at), (
            f"{int((want != at).sum())} side-output patterns differ from the rounding of y")
    return out

"""Helpers for GPU parity tests: move seeded inputs to the device and compare
kernel outputs with the oracle's fp64 results."""
from __future__ import annotations

import numpy as np

# Tolerances of the parity bar: bf16 output relative L2 and fp32 LSE absolute.
REL_L2_TOL = 3e-3
LSE_TOL = 1e-4
# Per output row (one query row of one head, a vector over the head dim): the
# relative L2 error of that row.  Rounding P to bf16 before P.V moves each
# key's weight by at most 2^-9 relative, and rounding O to bf16 each value by
# at most 2^-9 relative, so a row's error stays below about 2 * 2^-9 = 3.9e-3
# of its norm; the bound leaves a factor two over that.  Rows whose reference
# norm is below ROW_FLOOR of the root-mean-square row norm (near cancellation)
# are measured against that floor instead of their own norm.
ROW_REL_TOL = 8e-3
ROW_FLOOR = 0.1

# worst row of the last compare() call: (row index tuple, relative error)
last_worst_row = None


def dev(bits_or_array):
    import torch
    from attention_head_sinks_gb300 import workloads as W
    a = np.asarray(bits_or_array)
    if a.dtype == np.uint16:
        return W.to_torch(a).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def row_errors(o, ro):
    """Relative L2 error of every row (last axis) of ``o`` against ``ro``,
    with the denominator floored at ROW_FLOOR x the RMS row norm."""
    err = np.linalg.norm(o - ro, axis=-1)
    nrm = np.linalg.norm(ro, axis=-1)
    rms = float(np.sqrt(np.mean(nrm ** 2))) if nrm.size else 0.0
    den = np.maximum(nrm, ROW_FLOOR * rms)
    with np.errstate(divide="ignore", invalid="ignore"):
        rel = np.where(den > 0, err / np.where(den > 0, den, 1.0), err)
    return rel


def compare(out, lse, ref_out, ref_lse, rows=None, lse_layout="hq_t", row_tol=ROW_REL_TOL):
    """Relative L2 of ``out`` (bf16, any leading shape [R, ...]) and max
    |dLSE| against the oracle, optionally on a subset of rows (first axis of
    out, second axis of lse).  -inf LSE entries must match exactly, and every
    output row (a vector over the last axis) must be within ``row_tol``
    relative L2 of the oracle's; the worst row is printed and kept in
    ``last_worst_row``."""
    global last_worst_row
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        o, ro = o[rows], ref_out[rows]
        l, rl = l[:, rows], ref_lse[:, rows]
    else:
        ro, rl = ref_out, ref_lse
    den = np.linalg.norm(ro)
    rel = float(np.linalg.norm(o - ro) / den) if den > 0 else float(np.abs(o).max())
    fin = np.isfinite(rl)
    assert np.array_equal(np.isneginf(l), np.isneginf(rl)), "empty-row LSE mismatch"
    dl = float(np.abs(l[fin] - rl[fin]).max()) if fin.any() else 0.0
    # rows whose key set is empty must be exactly zero
    empty = ~fin
    if empty.any():
        if o.ndim == 3:
            zero_rows = o.transpose(1, 0, 2)[empty]
        else:
            zero_rows = o[empty.T]
        assert np.all(zero_rows == 0.0), "empty rows must be zero"
    if den > 0 and o.size:
        per_row = row_errors(o, ro)
        k = int(np.argmax(per_row))
        worst = (np.unravel_index(k, per_row.shape), float(per_row.flat[k]))
        last_worst_row = worst
        print("worst row %s: rel L2 %.3e (whole tensor %.3e)" % (worst[0], worst[1], rel))
        assert worst[1] <= row_tol, \
            "row %s: relative L2 %.3e > %.1e" % (worst[0], worst[1], row_tol)
    return rel, dl

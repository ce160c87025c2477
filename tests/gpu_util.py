"""Helpers for GPU parity tests: move seeded inputs to the device and compare
kernel outputs with the oracle's fp64 results."""
from __future__ import annotations

import numpy as np

# Tolerances of the parity bar: bf16 output relative L2 and fp32 LSE absolute.
REL_L2_TOL = 3e-3
LSE_TOL = 1e-4


def dev(bits_or_array):
    import torch
    from attention_head_sinks_gb300 import workloads as W
    a = np.asarray(bits_or_array)
    if a.dtype == np.uint16:
        return W.to_torch(a).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def compare(out, lse, ref_out, ref_lse, rows=None, lse_layout="hq_t"):
    """Relative L2 of ``out`` (bf16, any leading shape [R, ...]) and max
    |dLSE| against the oracle, optionally on a subset of rows (first axis of
    out, second axis of lse).  -inf LSE entries must match exactly."""
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
    return rel, dl

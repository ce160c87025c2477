"""Independent references used to pin the oracle (CPU only, fp64).

These build attention from library routines -- ``torch``'s
``scaled_dot_product_attention`` with explicit float masks, ``scipy``'s
``logsumexp`` -- not from the oracle's code, so that an error in the oracle
(a dropped term, a wrong sign or index, a transposed operand) shows up as a
mismatch.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def sdpa_with_bias(q, k, v, bias, scale, null_sink=None):
    """Attention by torch SDPA (fp64) with an additive float mask.

    q ``[R,Hq,D]``, k ``[N,Hq,Dk]``, v ``[N,Hq,Dv]`` float64 (kv already expanded
    to query heads), bias ``[Hq,R,N]`` (-inf = masked).  ``null_sink`` ``[Hq]``:
    append one extra key per head with zero key and zero value whose logit is
    the sink, i.e. ``exp(s)`` joins the denominator only.
    """
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]          # [1,H,R,D]
    kt = torch.from_numpy(k).permute(1, 0, 2)[None]
    vt = torch.from_numpy(v).permute(1, 0, 2)[None]
    bt = torch.from_numpy(bias)[None]                          # [1,H,R,N]
    if null_sink is not None:
        H, R = bias.shape[0], bias.shape[1]
        kt = torch.cat([kt, torch.zeros_like(kt[:, :, :1])], 2)
        vt = torch.cat([vt, torch.zeros_like(vt[:, :, :1])], 2)
        col = torch.from_numpy(np.asarray(null_sink, np.float64)).view(1, H, 1, 1)
        bt = torch.cat([bt, col.expand(1, H, R, 1)], 3)
    out = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=bt, scale=scale)
    return out[0].permute(1, 0, 2).numpy()


def expand_kv(x, hq):
    """``[N,Hkv,D]`` -> ``[N,Hq,D]``: query head h reads kv head h // (Hq/Hkv)."""
    hkv = x.shape[1]
    return np.repeat(x, hq // hkv, axis=1)


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))

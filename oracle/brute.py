"""Dense brute-force oracle in NumPy (fp64), for tiny inputs only.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Independent of the C
oracle: it builds the full ``[rows, keys]`` logit matrix for every head, a
boolean key-set mask that enumerates every (query, key) pair, adds the sink as
a bias matrix or an extra denominator term, and takes a masked softmax.

Definitions followed (page title, section):
* vLLM pull 49815 "[Bugfix][MiMo] Apply vision attention sinks in the window
  attention path" -- sink on the logit of each sequence's first key, LSE of the
  masked scaled logits;
* afierka-intel/vllm pull 76 "Apply DeepSeek-V4 attn_sink in the XPU
  sparse-MLA Triton kernel", Implementation -- sink in the denominator only,
  LSE over the selected keys;
* NeMo AutoModel "minimax_m3_vl.cp_sparse_attn" -- block selection + token
  causal + document mask, zero output for fully masked rows.
"""
from __future__ import annotations

import numpy as np

NONE, KEY0_BIAS, NULL_LOGIT = 0, 1, 2


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    u = bits.astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def masked_softmax_attention(logits, mask, values, null_sink=None):
    """Softmax over the masked entries of each row of ``logits``.

    logits ``[R,N]`` (already scaled and biased), mask ``[R,N]`` bool,
    values ``[N,Dv]``; ``null_sink`` (scalar or None) adds ``exp(s)`` to each
    row's denominator without touching the LSE.  Returns (out ``[R,Dv]``,
    lse ``[R]``); rows with no live entry give zeros and ``-inf``.
    """
    R = logits.shape[0]
    out = np.zeros((R, values.shape[1]))
    lse = np.full(R, -np.inf)
    for r in range(R):
        live = mask[r] & np.isfinite(logits[r])
        if not live.any():
            continue
        l = logits[r][live]
        m = l.max()
        z = np.exp(l - m).sum()
        lse[r] = m + np.log(z)
        den = z * np.exp(m)
        if null_sink is not None:
            den = den + np.exp(null_sink)
        out[r] = (np.exp(l)[:, None] * values[live]).sum(0) / den
    return out, lse


def window_mask(cu_seqlens, window_left, window_right):
    """``[T,T]`` bool: key j is in query i's window and in i's sequence."""
    cu = np.asarray(cu_seqlens, np.int64)
    T = int(cu[-1])
    seq = np.zeros(T, np.int64)
    for b in range(len(cu) - 1):
        seq[cu[b]:cu[b + 1]] = b
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    return (seq[:, None] == seq[None, :]) & (j >= i - window_left) & \
        (j <= i + window_right)


def window_fwd(q, k, v, cu_seqlens, window_left, window_right, sinks, mode,
               scale):
    qf, kf, vf = (bf16_bits_to_f64(x) for x in (q, k, v))
    T, hq, d = qf.shape
    hkv = kf.shape[1]
    cu = np.asarray(cu_seqlens, np.int64)
    mask = window_mask(cu, window_left, window_right)
    first_key = np.zeros(T, np.int64)
    for b in range(len(cu) - 1):
        first_key[cu[b]:cu[b + 1]] = cu[b]
    out = np.zeros((T, hq, d))
    lse = np.zeros((hq, T))
    for h in range(hq):
        g = h // (hq // hkv)
        logits = scale * (qf[:, h, :] @ kf[:, g, :].T)
        if mode == KEY0_BIAS:
            bias = np.zeros((T, T))
            bias[np.arange(T), first_key] = float(sinks[h])
            logits = logits + bias
        o, l = masked_softmax_attention(
            logits, mask, vf[:, g, :],
            float(sinks[h]) if mode == NULL_LOGIT else None)
        out[:, h, :] = o
        lse[h] = l
    return out, lse


def sparse_index_fwd(q, kv, indices, dv, sinks, mode, scale):
    """Dense form over all ``nkv`` keys with a membership mask.

    A key listed twice counts twice: the dense form expresses that as a
    per-pair multiplicity, folded in as ``log(multiplicity)`` on the logit.
    """
    qf = bf16_bits_to_f64(q)
    kvf = bf16_bits_to_f64(kv)
    nq, hq, dqk = qf.shape
    nkv = kvf.shape[0]
    mult = np.zeros((nq, nkv))
    for i in range(nq):
        for j in np.asarray(indices[i]):
            if 0 <= j < nkv:
                mult[i, j] += 1
    mask = mult > 0
    with np.errstate(divide="ignore"):
        logmult = np.where(mask, np.log(np.maximum(mult, 1)), 0.0)
    out = np.zeros((nq, hq, dv))
    lse = np.zeros((hq, nq))
    for h in range(hq):
        logits = scale * (qf[:, h, :] @ kvf.T) + logmult
        o, l = masked_softmax_attention(
            logits, mask, kvf[:, :dv],
            float(sinks[h]) if mode == NULL_LOGIT else None)
        out[:, h, :] = o
        lse[h] = l
    return out, lse


def block_mask(batch, seq_len, block_table, block_size, cu_docs):
    """``[T,T]`` bool over flattened tokens: selected block, causal, same doc,
    same batch row."""
    T = batch * seq_len
    cd = np.asarray(cu_docs, np.int64)
    doc = np.zeros(T, np.int64)
    for e in range(len(cd) - 1):
        doc[cd[e]:cd[e + 1]] = e
    row = np.arange(T) // seq_len
    pos = np.arange(T) % seq_len
    nblocks = -(-seq_len // block_size)
    sel = np.zeros((T, nblocks), bool)
    for i in range(T):
        for b in np.asarray(block_table[i]):
            if 0 <= b < nblocks:
                sel[i, b] = True
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    return (row[:, None] == row[None, :]) & (j <= i) & \
        (doc[:, None] == doc[None, :]) & sel[:, pos // block_size]


def block_sparse_fwd(q, k, v, batch, seq_len, block_table, block_size,
                     cu_docs, sinks, mode, scale):
    qf, kf, vf = (bf16_bits_to_f64(x) for x in (q, k, v))
    T, hq, d = qf.shape
    hkv = kf.shape[1]
    mask = block_mask(batch, seq_len, block_table, block_size, cu_docs)
    # KEY0_BIAS key of token i: the first token of its document, if that lies
    # in i's batch row
    cd = np.asarray(cu_docs, np.int64)
    first_key = np.full(T, -1, np.int64)
    for e in range(len(cd) - 1):
        first_key[cd[e]:cd[e + 1]] = cd[e]
    same_row = (first_key // seq_len) == (np.arange(T) // seq_len)
    out = np.zeros((T, hq, d))
    lse = np.zeros((hq, T))
    for h in range(hq):
        g = h // (hq // hkv)
        logits = scale * (qf[:, h, :] @ kf[:, g, :].T)
        if mode == KEY0_BIAS:
            rows = np.nonzero(same_row)[0]
            logits[rows, first_key[rows]] += float(sinks[h])
        o, l = masked_softmax_attention(
            logits, mask, vf[:, g, :],
            float(sinks[h]) if mode == NULL_LOGIT else None)
        out[:, h, :] = o
        lse[h] = l
    return out, lse

"""ctypes front end of the C oracle (``sa_oracle.c``), fp64 results.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Every function takes NumPy arrays: bf16 tensors as their ``uint16`` bit
patterns, ``cu_seqlens`` / indices / tables as ``int32``, sinks as ``float32``,
and returns ``(out, lse, key_count)`` as float64 / float64 / int32 arrays.
``rows=(begin, end)`` restricts the work to a slice of query rows (the other
rows of ``out`` and ``lse`` are NaN), which is how full-size workloads are
sampled.  ``bufs`` (a dict the caller keeps between calls) lends the output
arrays: a call finds those of an earlier call with the same shapes there
instead of allocating and filling full-size outputs each time (rows outside
``rows`` then hold what an earlier call left).  It changes no arithmetic.
"""
from __future__ import annotations

import ctypes
import functools

import numpy as np

from . import build_oracle

NONE, KEY0_BIAS, NULL_LOGIT = 0, 1, 2

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_F64 = ctypes.c_double


@functools.lru_cache(maxsize=1)
def _lib() -> ctypes.CDLL:
    lib = ctypes.CDLL(build_oracle.build())
    lib.oracle_window_fwd.argtypes = [
        _P, _P, _P, _P, _I32, _I64, _I32, _I32, _I32, _I32, _I32, _P, _I32,
        _F64, _P, _P, _P, _I64, _I64]
    lib.oracle_window_fwd.restype = ctypes.c_int
    lib.oracle_sparse_index_fwd.argtypes = [
        _P, _P, _I64, _I32, _I32, _P, _I32, _I32, _I32, _P, _I32, _F64, _P,
        _P, _P, _I64, _I64]
    lib.oracle_sparse_index_fwd.restype = ctypes.c_int
    lib.oracle_block_sparse_fwd.argtypes = [
        _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _I32, _I32, _P, _I32,
        _P, _I32, _F64, _P, _P, _P, _I64, _I64]
    lib.oracle_block_sparse_fwd.restype = ctypes.c_int
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


def num_threads() -> int:
    """OpenMP threads the oracle uses (the ``cores`` of a CPU timing)."""
    return int(_lib().oracle_num_threads())


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.dtype(dtype):
        raise TypeError("expected %s, got %s" % (np.dtype(dtype), a.dtype))
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _outputs(bufs, key, specs):
    """Output arrays for ``specs`` = ((shape, dtype, fill), ...): new ones, or
    with ``bufs`` the ones made under the same key and shapes before."""
    if bufs is None:
        return [np.full(sh, fill, dt) for sh, dt, fill in specs]
    k = (key,) + tuple((tuple(sh), np.dtype(dt).str) for sh, dt, _ in specs)
    if k not in bufs:
        bufs[k] = [np.full(sh, fill, dt) for sh, dt, fill in specs]
    return bufs[k]


def _sinks(sinks, hq):
    if sinks is None:
        return np.zeros(hq, np.float32)
    return _c(sinks, np.float32)


def window_fwd(q, k, v, cu_seqlens, window_left, window_right, sinks, mode,
               scale, rows=None, bufs=None):
    """Sliding-window attention over ``cu_seqlens``-packed sequences.

    q ``[T,Hq,D]``, k/v ``[T,Hkv,D]`` (uint16 bf16 bits); returns out
    ``[T,Hq,D]``, lse ``[Hq,T]`` and the key count per ``(token, head)``.
    """
    q, k, v = (_c(x, np.uint16) for x in (q, k, v))
    cu = _c(cu_seqlens, np.int32)
    T, hq, d = q.shape
    hkv = k.shape[1]
    s = _sinks(sinks, hq)
    b, e = (0, T) if rows is None else rows
    out, lse, cnt = _outputs(bufs, "window", (((T, hq, d), np.float64, np.nan),
                                              ((hq, T), np.float64, np.nan),
                                              ((T, hq), np.int32, -1)))
    rc = _lib().oracle_window_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(cu), len(cu) - 1, T, hq, hkv, d,
        int(window_left), int(window_right), _ptr(s), int(mode), float(scale),
        _ptr(out), _ptr(lse), _ptr(cnt), b, e)
    if rc != 0:
        raise ValueError("oracle_window_fwd rejected its arguments")
    return out, lse, cnt


def sparse_index_fwd(q, kv, indices, dv, sinks, mode, scale, rows=None, bufs=None):
    """Top-k index attention into one shared latent cache.

    q ``[Nq,Hq,dqk]``, kv ``[nkv,dqk]`` (uint16 bf16 bits), indices
    ``[Nq,topk]`` int32; V is the first ``dv`` columns of each kv row.
    Returns out ``[Nq,Hq,dv]``, lse ``[Hq,Nq]``, valid-key count ``[Nq]``.
    """
    q, kv = _c(q, np.uint16), _c(kv, np.uint16)
    idx = _c(indices, np.int32)
    nq, hq, dqk = q.shape
    topk = idx.shape[1]
    s = _sinks(sinks, hq)
    b, e = (0, nq) if rows is None else rows
    out, lse, cnt = _outputs(bufs, "index", (((nq, hq, dv), np.float64, np.nan),
                                             ((hq, nq), np.float64, np.nan),
                                             ((nq,), np.int32, -1)))
    rc = _lib().oracle_sparse_index_fwd(
        _ptr(q), _ptr(kv), kv.shape[0], dqk, int(dv), _ptr(idx), topk, nq, hq,
        _ptr(s), int(mode), float(scale), _ptr(out), _ptr(lse), _ptr(cnt), b, e)
    if rc != 0:
        raise ValueError("oracle_sparse_index_fwd rejected its arguments")
    return out, lse, cnt


def block_sparse_fwd(q, k, v, batch, seq_len, block_table, block_size,
                     cu_docs, sinks, mode, scale, rows=None, bufs=None):
    """Block-sparse causal attention with a document mask.

    q ``[B*S,Hq,D]``, k/v ``[B*S,Hkv,D]`` (uint16 bf16 bits), block_table
    ``[B*S,topk]`` int32, cu_docs ``[num_docs+1]`` int32.  Returns out
    ``[B*S,Hq,D]``, lse ``[Hq,B*S]``, key count per token ``[B*S]``.
    """
    q, k, v = (_c(x, np.uint16) for x in (q, k, v))
    tab = _c(block_table, np.int32)
    cd = _c(cu_docs, np.int32)
    T, hq, d = q.shape
    hkv = k.shape[1]
    s = _sinks(sinks, hq)
    b, e = (0, T) if rows is None else rows
    out, lse, cnt = _outputs(bufs, "block", (((T, hq, d), np.float64, np.nan),
                                             ((hq, T), np.float64, np.nan),
                                             ((T,), np.int32, -1)))
    rc = _lib().oracle_block_sparse_fwd(
        _ptr(q), _ptr(k), _ptr(v), int(batch), int(seq_len), hq, hkv, d,
        _ptr(tab), tab.shape[1], int(block_size), _ptr(cd), len(cd) - 1,
        _ptr(s), int(mode), float(scale), _ptr(out), _ptr(lse), _ptr(cnt), b, e)
    if rc != 0:
        raise ValueError("oracle_block_sparse_fwd rejected its arguments")
    return out, lse, cnt


def _widen(a):
    """bf16 bit patterns (uint16) to float64 exactly; other arrays as float64."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def merge_states(out_a, lse_a, out_b, lse_b, sinks, mode):
    """Attention over the union of two disjoint key sets of the same queries,
    from the two sink-free partial results (each the attention over its own
    set, with its LSE): the LSE-weighted merge, with a NULL_LOGIT sink folded
    once ([XPU sink] Implementation: the sink joins the denominator only, the
    LSE stays over real keys; [MiMo sinks] LSE paragraph: LSE of the masked
    scaled logits).  A partial with LSE = -inf has no keys; both empty gives
    out = 0, LSE = -inf.

    out_* ``[T,H,D]`` (bf16 bits as uint16, or float), lse_* ``[H,T]``.
    Returns out ``[T,H,D]`` and lse ``[H,T]`` as float64.
    """
    oa, ob = _widen(out_a), _widen(out_b)
    la = np.asarray(lse_a, np.float64).T[:, :, None]  # [T,H,1]
    lb = np.asarray(lse_b, np.float64).T[:, :, None]
    M = np.maximum(la, lb)
    empty = M == -np.inf
    Mr = np.where(empty, 0.0, M)
    wa = np.exp(la - Mr)
    wb = np.exp(lb - Mr)
    Z = wa + wb
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, Mr + np.log(np.where(empty, 1.0, Z)))
    den = Z
    if mode == NULL_LOGIT:
        s = np.asarray(sinks, np.float64)[None, :, None]
        den = Z + np.exp(s - Mr)
    out = np.where(empty, 0.0, (wa * oa + wb * ob) / np.where(empty, 1.0, den))
    return out, lse[:, :, 0].T.copy()


def e4m3_to_f64(codes):
    """Exact value of e4m3 codes (sign, 4-bit exponent with bias 7, 3-bit
    mantissa; exponent 0 is subnormal; 0x7F / 0xFF are NaN)."""
    c = np.asarray(codes, np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e, m = (c >> 3) & 0xF, c & 7
    v = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7))
    v = np.where((c & 0x7F) == 0x7F, np.nan, v)
    return s * v


def sparse_index_fwd_fp8(q, kv, kv_scale, indices, dv, sinks, mode, scale, rows=None,
                         bufs=None):
    """Top-k index attention into an e4m3 latent cache: latent row r is
    ``e4m3(kv[r]) * kv_scale[r]`` (fp64), K the whole row, V its first ``dv``
    columns; otherwise as ``sparse_index_fwd`` (afierka-intel/vllm pull 76,
    Implementation: the listed keys exactly, NULL_LOGIT in the denominator
    only, LSE over the listed keys).  q ``[Nq,Hq,dqk]`` as bf16 bits.
    Returns out ``[Nq,Hq,dv]``, lse ``[Hq,Nq]`` float64 and the valid-key count.
    """
    qf = _widen(q)
    nq, hq, dqk = qf.shape
    nkv = kv.shape[0]
    idx = np.asarray(indices, np.int64)
    b, e = (0, nq) if rows is None else rows
    out, lse, cnt = _outputs(bufs, "index_fp8", (((nq, hq, dv), np.float64, np.nan),
                                                 ((hq, nq), np.float64, np.nan),
                                                 ((nq,), np.int32, -1)))
    sk = np.asarray(sinks, np.float64) if sinks is not None else np.zeros(hq)
    for i in range(b, e):
        keys = idx[i][(idx[i] >= 0) & (idx[i] < nkv)]
        cnt[i] = len(keys)
        if len(keys) == 0:
            out[i] = 0.0
            lse[:, i] = -np.inf
            continue
        rows_f = e4m3_to_f64(kv[keys]) * np.asarray(kv_scale, np.float64)[keys][:, None]
        logits = float(scale) * (qf[i] @ rows_f.T)          # [hq, n]
        m = logits.max(axis=1, keepdims=True)
        w = np.exp(logits - m)
        z = w.sum(axis=1, keepdims=True)
        lse[:, i] = (m + np.log(z))[:, 0]
        den = z * np.exp(m)
        if mode == NULL_LOGIT:
            den = den + np.exp(sk)[:, None]
        out[i] = (np.exp(logits) @ rows_f[:, :dv]) / den
    return out, lse, cnt


def block_select(index_q, index_k, batch, seq_len, block_size, topk, rows=None, bufs=None):
    """Top-k key blocks per (index head, query token) from indexer scores
    ([M3 CP sparse] forward step 3 and ``_select_local_blocks``: the selection
    is built from index q / k over the causal sequence of the token's batch
    row, one selection per index head; documents are not consulted -- their
    mask is applied inside the attention).  Readings where the page is
    silent: the token score is the dot product q_idx[i, g] . k_idx[j]; a
    block's score is the max over its causal keys; the query's own (diagonal)
    block is always selected and the other ``topk - 1`` are the highest
    scoring earlier blocks, ties to the lower block id; a token with at most
    ``topk`` causal blocks selects them all.

    index_q ``[B*S, Hi, Di]`` and index_k ``[B*S, Di]`` (bf16 bits as uint16,
    or float).  Scores in fp64 from the exact inputs.  Returns the table
    ``[Hi, B*S, topk]`` int32 (ascending block ids, -1 padded) and the block
    scores ``[Hi, B*S, nblocks]`` float64 (-inf for blocks at or after the
    diagonal).  ``rows=(begin, end)`` restricts the work to those tokens (the
    rest of the table is -2, of the scores NaN).
    """
    qf = _widen(index_q)
    kf = _widen(index_k)
    T, hi, di = qf.shape
    nb = -(-seq_len // block_size)
    b0, e0 = (0, T) if rows is None else rows
    table, scores = _outputs(bufs, "select", (((hi, T, topk), np.int32, -2),
                                              ((hi, T, nb), np.float64, np.nan)))
    table[:, b0:e0] = -1
    for i in range(b0, e0):
        row0 = (i // seq_len) * seq_len
        pos = i - row0
        diag = pos // block_size
        keys = kf[row0:row0 + diag * block_size]          # keys of earlier blocks
        tok = qf[i] @ keys.T                              # [hi, diag * block_size]
        blk = tok.reshape(hi, diag, block_size).max(axis=2) if diag else \
            np.zeros((hi, 0))
        scores[:, i, :] = -np.inf
        scores[:, i, :diag] = blk
        for g in range(hi):
            if diag + 1 <= topk:
                sel = np.arange(diag + 1)
            else:
                # highest score first; among equal scores the lower id first
                order = np.lexsort((np.arange(diag), -blk[g]))[:topk - 1]
                sel = np.sort(np.append(order, diag))
            table[g, i, :len(sel)] = sel
    return table, scores


def block_sparse_fwd_index_heads(q, k, v, batch, seq_len, tables, block_size, cu_docs,
                                 sinks, mode, scale, rows=None, bufs=None):
    """Block-sparse attention with one selection per index head: attention
    head h uses ``tables[h // (Hq / Hi)]`` ([M3 CP sparse] ``_select_local_blocks``
    returns ``[batch, index_heads, sequence, key_blocks]``); each group of
    heads is ``block_sparse_fwd`` with its own table.  tables ``[Hi, B*S,
    topk]``; Hi must divide Hkv (a KV head's query heads share one index
    head).  Returns out ``[B*S,Hq,D]``, lse ``[Hq,B*S]``, key counts
    ``[Hi, B*S]``.
    """
    tables = np.asarray(tables, np.int32)
    hi = tables.shape[0]
    T, hq, d = np.asarray(q).shape
    hkv = np.asarray(k).shape[1]
    if hkv % hi:
        raise ValueError("the number of index heads must divide the KV heads")
    gq, gk = hq // hi, hkv // hi
    s = _sinks(sinks, hq)
    out, lse, cnt = _outputs(bufs, "block_heads", (((T, hq, d), np.float64, np.nan),
                                                   ((hq, T), np.float64, np.nan),
                                                   ((hi, T), np.int32, -1)))
    for g in range(hi):
        o, l, c = block_sparse_fwd(
            np.ascontiguousarray(np.asarray(q)[:, g * gq:(g + 1) * gq]),
            np.ascontiguousarray(np.asarray(k)[:, g * gk:(g + 1) * gk]),
            np.ascontiguousarray(np.asarray(v)[:, g * gk:(g + 1) * gk]),
            batch, seq_len, tables[g], block_size, cu_docs,
            s[g * gq:(g + 1) * gq], mode, scale, rows=rows, bufs=bufs)
        out[:, g * gq:(g + 1) * gq] = o
        lse[g * gq:(g + 1) * gq] = l
        cnt[g] = c
    return out, lse, cnt

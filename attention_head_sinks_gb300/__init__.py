"""Sink-aware varlen attention forward for GB300 (sm_103a).

Thin Python binding over the C ABI of ``libsa.so`` (``include/sa.h``): each
function checks and marshals torch tensors to raw device pointers and calls the
C entry point of the same name on the current CUDA stream.  All computation
runs in the library's CUDA kernels; there is no CPU or PyTorch fallback, and a
missing library raises.
"""
from __future__ import annotations

from ._lib import SINK_KEY0_BIAS, SINK_NONE, SINK_NULL_LOGIT, SAError, lib  # noqa: F401

__all__ = ["sa_varlen_window_fwd", "sa_sparse_index_fwd", "sa_sparse_index_fwd_fp8",
           "sa_block_sparse_fwd", "sa_block_sparse_fwd_index_heads", "sa_block_select",
           "sa_merge_attn_states",
           "sa_sparse_index_workspace_size", "sa_device_error", "sa_check_wait_expiry",
           "sa_version", "SAError",
           "SINK_NONE", "SINK_KEY0_BIAS", "SINK_NULL_LOGIT"]


def _torch():
    import torch
    return torch


def _dev_tensor(name, t, dtype, ndim=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if ndim is not None and t.dim() != ndim:
        raise ValueError("%s must have %d dims, got %d" % (name, ndim, t.dim()))
    return t


def _stream_handle(stream, device=None):
    """Raw cudaStream_t of ``stream`` (default: the current stream of
    ``device``)."""
    torch = _torch()
    if stream is not None:
        return stream.cuda_stream
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        idx = device.index if device is not None and device.index is not None \
            else torch.cuda.current_device()
        return raw(idx)
    return torch.cuda.current_stream().cuda_stream


def sa_varlen_window_fwd(q, k, v, cu_seqlens, window_left, window_right, sinks,
                         sink_mode, softmax_scale, out=None, lse=None,
                         stream=None):
    """Sliding-window attention with a per-head sink (C: ``sa_varlen_window_fwd``).

    q ``[T,Hq,D]``, k/v ``[T,Hkv,D]`` bf16; cu_seqlens int32 ``[B+1]``; sinks
    fp32 ``[Hq]`` (or None with ``SINK_NONE``).  Returns ``(out, lse)``:
    bf16 ``[T,Hq,D]`` and fp32 ``[Hq,T]`` (allocated when not given).
    """
    torch = _torch()
    _dev_tensor("q", q, torch.bfloat16, 3)
    _dev_tensor("k", k, torch.bfloat16, 3)
    _dev_tensor("v", v, torch.bfloat16, 3)
    _dev_tensor("cu_seqlens", cu_seqlens, torch.int32, 1)
    T, hq, d = q.shape
    hkv = k.shape[1]
    if k.shape != (T, hkv, d) or v.shape != (T, hkv, d):
        raise ValueError("k and v must be [T, Hkv, D] matching q")
    if sinks is not None:
        _dev_tensor("sinks", sinks, torch.float32, 1)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((hq, T), dtype=torch.float32, device=q.device)
    _dev_tensor("out", out, torch.bfloat16, 3)
    _dev_tensor("lse", lse, torch.float32, 2)
    from ._lib import check
    check(lib().sa_varlen_window_fwd(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), cu_seqlens.data_ptr(),
        cu_seqlens.numel() - 1, T, hq, hkv, d, int(window_left),
        int(window_right), None if sinks is None else sinks.data_ptr(),
        int(sink_mode), float(softmax_scale), out.data_ptr(), lse.data_ptr(),
        _stream_handle(stream, q.device)))
    return out, lse


def sa_sparse_index_workspace_size(num_queries, num_q_heads, dv, topk) -> int:
    """Workspace bytes ``sa_sparse_index_fwd`` needs (C: same name)."""
    return int(lib().sa_sparse_index_workspace_size(
        int(num_queries), int(num_q_heads), int(dv), int(topk)))


def sa_sparse_index_fwd(q, kv_latent, indices, dv, sinks, sink_mode,
                        softmax_scale, out=None, lse=None, workspace=None,
                        stream=None):
    """Top-k index attention into one shared latent cache (C:
    ``sa_sparse_index_fwd``).

    q ``[Nq,Hq,dqk]`` and kv_latent ``[nkv,dqk]`` bf16, indices int32
    ``[Nq,topk]`` (-1 padded), sinks fp32 ``[Hq]`` (or None with
    ``SINK_NONE``).  V is the first ``dv`` latent columns.  Returns
    ``(out, lse)``: bf16 ``[Nq,Hq,dv]`` and fp32 ``[Hq,Nq]``.  ``workspace``
    (a CUDA uint8 tensor) is allocated by torch when not given.
    """
    torch = _torch()
    _dev_tensor("q", q, torch.bfloat16, 3)
    _dev_tensor("kv_latent", kv_latent, torch.bfloat16, 2)
    _dev_tensor("indices", indices, torch.int32, 2)
    nq, hq, dqk = q.shape
    nkv = kv_latent.shape[0]
    topk = indices.shape[1]
    if kv_latent.shape[1] != dqk or indices.shape[0] != nq:
        raise ValueError("kv_latent must be [nkv, dqk] and indices [Nq, topk]")
    if sinks is not None:
        _dev_tensor("sinks", sinks, torch.float32, 1)
    if out is None:
        out = torch.empty((nq, hq, dv), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((hq, nq), dtype=torch.float32, device=q.device)
    need = sa_sparse_index_workspace_size(nq, hq, dv, topk)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _dev_tensor("out", out, torch.bfloat16, 3)
    _dev_tensor("lse", lse, torch.float32, 2)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _dev_tensor("workspace", workspace, torch.uint8, 1)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
    from ._lib import check
    check(lib().sa_sparse_index_fwd(
        q.data_ptr(), kv_latent.data_ptr(), nkv, dqk, int(dv),
        indices.data_ptr(), topk, nq, hq,
        None if sinks is None else sinks.data_ptr(), int(sink_mode),
        float(softmax_scale), out.data_ptr(), lse.data_ptr(), ws_ptr, ws_bytes,
        _stream_handle(stream, out.device)))
    return out, lse


def sa_sparse_index_fwd_fp8(q, kv_fp8, kv_scale, indices, dv, sinks, sink_mode,
                            softmax_scale, out=None, lse=None, workspace=None,
                            stream=None):
    """``sa_sparse_index_fwd`` over an e4m3 latent cache with one fp32 scale
    per row (C: ``sa_sparse_index_fwd_fp8``).

    kv_fp8 ``[nkv,dqk]`` e4m3 codes (uint8 or torch.float8_e4m3fn), kv_scale
    fp32 ``[nkv]``: row r is ``e4m3(kv_fp8[r]) * kv_scale[r]``.  Everything
    else as ``sa_sparse_index_fwd``.
    """
    torch = _torch()
    if isinstance(kv_fp8, torch.Tensor) and kv_fp8.dtype == torch.float8_e4m3fn:
        kv_fp8 = kv_fp8.view(torch.uint8)
    _dev_tensor("q", q, torch.bfloat16, 3)
    _dev_tensor("kv_fp8", kv_fp8, torch.uint8, 2)
    _dev_tensor("kv_scale", kv_scale, torch.float32, 1)
    _dev_tensor("indices", indices, torch.int32, 2)
    nq, hq, dqk = q.shape
    nkv = kv_fp8.shape[0]
    topk = indices.shape[1]
    if kv_fp8.shape[1] != dqk or indices.shape[0] != nq or kv_scale.shape[0] != nkv:
        raise ValueError("kv_fp8 must be [nkv, dqk], kv_scale [nkv] and indices [Nq, topk]")
    if sinks is not None:
        _dev_tensor("sinks", sinks, torch.float32, 1)
    if out is None:
        out = torch.empty((nq, hq, dv), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((hq, nq), dtype=torch.float32, device=q.device)
    need = sa_sparse_index_workspace_size(nq, hq, dv, topk)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _dev_tensor("out", out, torch.bfloat16, 3)
    _dev_tensor("lse", lse, torch.float32, 2)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        _dev_tensor("workspace", workspace, torch.uint8, 1)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
    from ._lib import check
    check(lib().sa_sparse_index_fwd_fp8(
        q.data_ptr(), kv_fp8.data_ptr(), kv_scale.data_ptr(), nkv, dqk, int(dv),
        indices.data_ptr(), topk, nq, hq,
        None if sinks is None else sinks.data_ptr(), int(sink_mode),
        float(softmax_scale), out.data_ptr(), lse.data_ptr(), ws_ptr, ws_bytes,
        _stream_handle(stream, out.device)))
    return out, lse


def sa_block_select(index_q, index_k, batch, seq_len, block_size, topk_blocks,
                    block_table=None, stream=None):
    """Top-k key blocks per (index head, token) from indexer scores (C:
    ``sa_block_select``).

    index_q ``[B*S,Hi,Di]`` and index_k ``[B*S,Di]`` bf16.  Returns the block
    table int32 ``[Hi,B*S,topk]`` (ascending, -1 padded).
    """
    torch = _torch()
    _dev_tensor("index_q", index_q, torch.bfloat16, 3)
    _dev_tensor("index_k", index_k, torch.bfloat16, 2)
    T, hi, di = index_q.shape
    if T != batch * seq_len or index_k.shape != (T, di):
        raise ValueError("index_q must be [batch*seq_len, Hi, Di] and index_k [batch*seq_len, Di]")
    if block_table is None:
        block_table = torch.empty((hi, T, int(topk_blocks)), dtype=torch.int32,
                                  device=index_q.device)
    _dev_tensor("block_table", block_table, torch.int32, 3)
    if block_table.shape != (hi, T, int(topk_blocks)):
        raise ValueError("block_table must be [Hi, batch*seq_len, topk_blocks]")
    from ._lib import check
    check(lib().sa_block_select(
        index_q.data_ptr(), index_k.data_ptr(), int(batch), int(seq_len), hi, di,
        int(block_size), int(topk_blocks), block_table.data_ptr(),
        _stream_handle(stream, block_table.device)))
    return block_table


def sa_block_sparse_fwd_index_heads(q, k, v, batch, seq_len, block_table, block_size,
                                    cu_docs, sinks, sink_mode, softmax_scale, out=None,
                                    lse=None, stream=None):
    """Block-sparse attention with one selection per index head (C:
    ``sa_block_sparse_fwd_index_heads``): block_table int32 ``[Hi,B*S,topk]``;
    query head h uses table ``h // (Hq / Hi)``.  Otherwise as
    ``sa_block_sparse_fwd``."""
    torch = _torch()
    _dev_tensor("q", q, torch.bfloat16, 3)
    _dev_tensor("k", k, torch.bfloat16, 3)
    _dev_tensor("v", v, torch.bfloat16, 3)
    _dev_tensor("block_table", block_table, torch.int32, 3)
    _dev_tensor("cu_docs", cu_docs, torch.int32, 1)
    T, hq, d = q.shape
    hkv = k.shape[1]
    if T != batch * seq_len or k.shape != (T, hkv, d) or v.shape != (T, hkv, d):
        raise ValueError("q must be [batch*seq_len, Hq, D] and k, v [batch*seq_len, Hkv, D]")
    if block_table.shape[1] != T:
        raise ValueError("block_table must be [Hi, batch*seq_len, topk]")
    if sinks is not None:
        _dev_tensor("sinks", sinks, torch.float32, 1)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((hq, T), dtype=torch.float32, device=q.device)
    _dev_tensor("out", out, torch.bfloat16, 3)
    _dev_tensor("lse", lse, torch.float32, 2)
    from ._lib import check
    check(lib().sa_block_sparse_fwd_index_heads(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), int(batch), int(seq_len), hq, hkv, d,
        block_table.data_ptr(), block_table.shape[0], block_table.shape[2],
        int(block_size), cu_docs.data_ptr(), cu_docs.numel() - 1,
        None if sinks is None else sinks.data_ptr(), int(sink_mode),
        float(softmax_scale), out.data_ptr(), lse.data_ptr(), _stream_handle(stream, out.device)))
    return out, lse


def sa_block_sparse_fwd(q, k, v, batch, seq_len, block_table, block_size,
                        cu_docs, sinks, sink_mode, softmax_scale, out=None,
                        lse=None, stream=None):
    """Block-sparse causal attention with packed documents (C:
    ``sa_block_sparse_fwd``).

    q ``[B*S,Hq,D]``, k/v ``[B*S,Hkv,D]`` bf16; block_table int32
    ``[B*S,topk]`` (-1 padded, block ids from the batch-row start); cu_docs
    int32 ``[num_docs+1]`` over the flattened tokens; sinks fp32 ``[Hq]`` (or
    None with ``SINK_NONE``).  Returns ``(out, lse)``: bf16 ``[B*S,Hq,D]`` and
    fp32 ``[Hq,B*S]``.
    """
    torch = _torch()
    _dev_tensor("q", q, torch.bfloat16, 3)
    _dev_tensor("k", k, torch.bfloat16, 3)
    _dev_tensor("v", v, torch.bfloat16, 3)
    _dev_tensor("block_table", block_table, torch.int32, 2)
    _dev_tensor("cu_docs", cu_docs, torch.int32, 1)
    T, hq, d = q.shape
    hkv = k.shape[1]
    if T != batch * seq_len or k.shape != (T, hkv, d) or v.shape != (T, hkv, d):
        raise ValueError("q must be [batch*seq_len, Hq, D] and k, v [batch*seq_len, Hkv, D]")
    if block_table.shape[0] != T:
        raise ValueError("block_table must have batch*seq_len rows")
    if sinks is not None:
        _dev_tensor("sinks", sinks, torch.float32, 1)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((hq, T), dtype=torch.float32, device=q.device)
    _dev_tensor("out", out, torch.bfloat16, 3)
    _dev_tensor("lse", lse, torch.float32, 2)
    from ._lib import check
    check(lib().sa_block_sparse_fwd(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), int(batch), int(seq_len), hq,
        hkv, d, block_table.data_ptr(), block_table.shape[1], int(block_size),
        cu_docs.data_ptr(), cu_docs.numel() - 1,
        None if sinks is None else sinks.data_ptr(), int(sink_mode),
        float(softmax_scale), out.data_ptr(), lse.data_ptr(), None, 0,
        _stream_handle(stream, out.device)))
    return out, lse


def sa_merge_attn_states(out_a, lse_a, out_b, lse_b, sinks, sink_mode, out=None,
                         lse=None, stream=None):
    """Merge two sink-free partial results over disjoint key sets of the same
    queries (C: ``sa_merge_attn_states``).

    out_a/out_b bf16 ``[T,H,D]``, lse_a/lse_b fp32 ``[H,T]``; sinks fp32
    ``[H]`` (or None with ``SINK_NONE``).  Returns ``(out, lse)`` (allocated
    when not given; ``out`` may be ``out_a`` or ``out_b``).
    """
    torch = _torch()
    _dev_tensor("out_a", out_a, torch.bfloat16, 3)
    _dev_tensor("out_b", out_b, torch.bfloat16, 3)
    _dev_tensor("lse_a", lse_a, torch.float32, 2)
    _dev_tensor("lse_b", lse_b, torch.float32, 2)
    T, h, d = out_a.shape
    if out_b.shape != (T, h, d) or lse_a.shape != (h, T) or lse_b.shape != (h, T):
        raise ValueError("partials must be out [T, H, D] and lse [H, T] of one shape")
    if sinks is not None:
        _dev_tensor("sinks", sinks, torch.float32, 1)
    if out is None:
        out = torch.empty_like(out_a)
    if lse is None:
        lse = torch.empty((h, T), dtype=torch.float32, device=out_a.device)
    _dev_tensor("out", out, torch.bfloat16, 3)
    _dev_tensor("lse", lse, torch.float32, 2)
    from ._lib import check
    check(lib().sa_merge_attn_states(
        out_a.data_ptr(), lse_a.data_ptr(), out_b.data_ptr(), lse_b.data_ptr(), T, h, d,
        None if sinks is None else sinks.data_ptr(), int(sink_mode), out.data_ptr(),
        lse.data_ptr(), _stream_handle(stream, out.device)))
    return out, lse


def sa_device_error() -> int:
    """Synchronise the device and return (and clear) its kernel error word."""
    import ctypes
    from ._lib import check
    code = ctypes.c_uint32(0)
    check(lib().sa_device_error(ctypes.byref(code)))
    return int(code.value)


def sa_check_wait_expiry(stream=None) -> None:
    """Enqueue one kernel whose bounded wait runs out (C:
    ``sa_check_wait_expiry``); ``sa_device_error()`` then returns 32."""
    from ._lib import check
    check(lib().sa_check_wait_expiry(_stream_handle(stream)))


def sa_version() -> int:
    return int(lib().sa_version())

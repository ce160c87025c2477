"""The allocation-free sparse-index entry point, called through the C ABI.

sa_sparse_index_fwd_noalloc is for callers that cannot allocate device memory
for a workspace (a plugin inside a runtime that owns the device memory pool,
a serving loop that must not allocate once running).  It keeps its split-KV
scratch in a fixed 64 MiB array inside the library, shared by every call and
never cleared.  Here, on consecutive calls whose inputs and layouts differ
(so each call finds the previous call's contents in the array), its results
must match the oracle within the parity tolerances and be bit-identical to
those of sa_sparse_index_fwd with a caller workspace; and it must reject sizes
whose scratch would exceed the array.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest

from attention_head_sinks_gb300 import workloads as W
from oracle import sa_oracle
from tests.gpu_util import LSE_TOL, REL_L2_TOL, compare, dev

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, kv, idx, dv, sinks, mode, scale, out, lse):
    import torch
    return lib.sa_sparse_index_fwd_noalloc(
        q.data_ptr(), kv.data_ptr(), kv.shape[0], q.shape[2], dv, idx.data_ptr(),
        idx.shape[1], q.shape[0], q.shape[1], sinks.data_ptr(), mode, scale,
        out.data_ptr(), lse.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _check_call(c):
    """One noalloc call: oracle parity and bit identity with the workspace
    entry point on the same inputs."""
    import torch
    import attention_head_sinks_gb300 as sa
    lib = sa.lib()
    nq, hq = c.q.shape[0], c.q.shape[1]
    topk = c.indices.shape[1]
    assert 0 < sa.sa_sparse_index_workspace_size(nq, hq, c.dv, topk) <= 64 << 20
    q, kv, idx, sk = dev(c.q), dev(c.kv), dev(c.indices), dev(c.sinks)
    out = torch.empty((nq, hq, c.dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((hq, nq), dtype=torch.float32, device="cuda")
    st = _noalloc(lib, q, kv, idx, c.dv, sk, c.mode, c.scale, out, lse)
    assert st == 0, lib.sa_last_error().decode()
    ws_out, ws_lse = sa.sa_sparse_index_fwd(q, kv, idx, c.dv, sk, c.mode, c.scale)
    torch.cuda.synchronize()
    ref_out, ref_lse, _ = sa_oracle.sparse_index_fwd(c.q, c.kv, c.indices, c.dv, c.sinks,
                                                     c.mode, c.scale)
    rel, dl = compare(out, lse, ref_out, ref_lse)
    assert rel <= REL_L2_TOL and dl <= LSE_TOL, (c.name, rel, dl)
    assert torch.equal(out, ws_out), c.name
    assert torch.equal(lse, ws_lse), c.name


def test_noalloc_matches_oracle_on_two_calls():
    import attention_head_sinks_gb300 as sa
    for seed in (4101, 4102):           # two calls in a row, different inputs
        c = W.index_case(12, 128, 576, 512, 8192, 2048, W.MLA_VALID_COUNTS[::-1]
                         if seed % 2 else W.MLA_VALID_COUNTS, (-2.20, 2.49),
                         W.SINK_NULL_LOGIT, seed, "noalloc_%d" % seed)
        _check_call(c)
    assert sa.sa_device_error() == 0


def test_noalloc_after_a_larger_layout():
    """A call that fills the array with a large layout (top-4096 lists, so
    queries with more than eight 256-key items take the plain-load merge),
    then one with fewer heads (another head stride), fewer queries and
    another list length, which finds the first call's contents in place."""
    import attention_head_sinks_gb300 as sa
    big = W.index_case(12, 128, 576, 512, 16384, 4096, (4096, 1, 3001, 2049, 300, 2048),
                       (-2.20, 2.49), W.SINK_NULL_LOGIT, 4103, "noalloc_top4096")
    _check_call(big)
    small = W.index_case(7, 40, 576, 512, 9000, 1000, (1000, 257, 3, 999, 512, 0, 700),
                         (-2.20, 2.49), W.SINK_NULL_LOGIT, 4104, "noalloc_40heads")
    _check_call(small)
    none = W.index_case(5, 40, 576, 512, 9000, 1000, (700, 1, 1000, 256, 513),
                        (-2.20, 2.49), W.SINK_NONE, 4105, "noalloc_nosink")
    _check_call(none)
    assert sa.sa_device_error() == 0


def test_noalloc_rejects_sizes_above_its_scratch():
    import torch
    import attention_head_sinks_gb300 as sa
    lib = sa.lib()
    # 64 queries x 128 heads x 8 items of partials need more than 64 MiB
    assert sa.sa_sparse_index_workspace_size(64, 128, 512, 2048) > 64 << 20
    q = torch.zeros((64, 128, 576), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((100, 576), dtype=torch.bfloat16, device="cuda")
    idx = torch.full((64, 2048), -1, dtype=torch.int32, device="cuda")
    sk = torch.zeros(128, dtype=torch.float32, device="cuda")
    out = torch.empty((64, 128, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((128, 64), dtype=torch.float32, device="cuda")
    st = _noalloc(lib, q, kv, idx, 512, sk, W.SINK_NULL_LOGIT, 0.04, out, lse)
    assert st == 2  # SA_ERR_UNSUPPORTED
    msg = lib.sa_last_error().decode()
    assert msg.startswith("sa_sparse_index_fwd_noalloc:") and "64 MiB" in msg

"""The allocation-free sparse-index entry point, called through the C ABI.

sa_sparse_index_fwd_noalloc is for callers that cannot allocate device memory
for a workspace (a plugin inside a runtime that owns the device memory pool,
a serving loop that must not allocate once running).  It keeps its split-KV
scratch in a fixed 64 MiB array inside the library.  Here it must give the
same results as sa_sparse_index_fwd with a caller workspace, within the
parity tolerances, on two calls in a row with different inputs (the second
call finds the first call's contents in the shared array), and it must reject
sizes whose scratch would exceed the array.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest

from attention_head_sinks_gb300 import workloads as W
from tests.gpu_util import LSE_TOL, REL_L2_TOL, dev

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, kv, idx, dv, sinks, mode, scale, out, lse):
    import torch
    return lib.sa_sparse_index_fwd_noalloc(
        q.data_ptr(), kv.data_ptr(), kv.shape[0], q.shape[2], dv, idx.data_ptr(),
        idx.shape[1], q.shape[0], q.shape[1], sinks.data_ptr(), mode, scale,
        out.data_ptr(), lse.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    import torch
    import attention_head_sinks_gb300 as sa
    lib = sa.lib()
    for seed in (4101, 4102):           # two calls in a row, different inputs
        c = W.index_case(12, 128, 576, 512, 8192, 2048, W.MLA_VALID_COUNTS[::-1]
                         if seed % 2 else W.MLA_VALID_COUNTS, (-2.20, 2.49),
                         W.SINK_NULL_LOGIT, seed, "noalloc")
        assert sa.sa_sparse_index_workspace_size(12, 128, 512, 2048) <= 64 << 20
        q, kv, idx, sk = dev(c.q), dev(c.kv), dev(c.indices), dev(c.sinks)
        out = torch.empty((12, 128, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((128, 12), dtype=torch.float32, device="cuda")
        st = _noalloc(lib, q, kv, idx, 512, sk, c.mode, c.scale, out, lse)
        assert st == 0, lib.sa_last_error().decode()
        ref_out, ref_lse = sa.sa_sparse_index_fwd(q, kv, idx, 512, sk, c.mode, c.scale)
        torch.cuda.synchronize()
        o = out.float().cpu().numpy().astype(np.float64)
        r = ref_out.float().cpu().numpy().astype(np.float64)
        rel = np.linalg.norm(o - r) / np.linalg.norm(r)
        l, rl = lse.cpu().numpy(), ref_lse.cpu().numpy()
        assert np.array_equal(np.isneginf(l), np.isneginf(rl))
        fin = np.isfinite(rl)
        assert rel <= REL_L2_TOL and np.abs(l[fin] - rl[fin]).max() <= LSE_TOL
    assert sa.sa_device_error() == 0


def test_noalloc_rejects_sizes_above_its_scratch():
    import torch
    import attention_head_sinks_gb300 as sa
    lib = sa.lib()
    # 64 queries x 128 heads x 8 slices of partials need 134 MB > 64 MiB
    assert sa.sa_sparse_index_workspace_size(64, 128, 512, 2048) > 64 << 20
    q = torch.zeros((64, 128, 576), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((100, 576), dtype=torch.bfloat16, device="cuda")
    idx = torch.full((64, 2048), -1, dtype=torch.int32, device="cuda")
    sk = torch.zeros(128, dtype=torch.float32, device="cuda")
    out = torch.empty((64, 128, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((128, 64), dtype=torch.float32, device="cuda")
    st = _noalloc(lib, q, kv, idx, 512, sk, W.SINK_NULL_LOGIT, 0.04, out, lse)
    assert st == 2  # SA_ERR_UNSUPPORTED
    assert "64 MiB" in lib.sa_last_error().decode()

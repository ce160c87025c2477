"""The benchmark's workload table, on the CPU: every workload builds, names
itself in its config, points at an existing kernel source, and reports the
algorithmic bytes and flops its roofline divides by (the default window
workload's and the decode batch's byte counts fixed to the values the
formulas give)."""
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("name", sorted(bench.RUNNERS))
def test_workload_builds_and_counts(name):
    r = bench.RUNNERS[name](name)
    cfg = r.config()
    assert cfg["workload"] == name
    assert r.bound in ("hbm", "tensor", "launch")
    assert os.path.exists(os.path.join(ROOT, r.source))
    nbytes, flops = r.counts()
    assert nbytes > 0 and flops > 0
    assert r.oracle_rows() > 0
    assert r.launches_per_call() >= 1


def test_default_window_bytes():
    # q and o once, k and v once per KV head (16 of them here), LSE: 4 x 4096
    # tokens, 16 heads, head dim 80
    r = bench.RUNNERS["vision_window_16384tok"]("vision_window_16384tok")
    T, H, D = 16384, 16, 80
    nbytes, _ = r.counts()
    assert nbytes == 2 * T * H * D * 2 + 2 * T * H * D * 2 + 4 * H * T


def test_decode_batch_bytes():
    # q and o once, each listed row once per query (1152 bytes), the index
    # rows, the LSE
    r = bench.RUNNERS["mla_sparse_decode"]("mla_sparse_decode")
    c = r.c
    nq, hq, dqk = c.q.shape
    topk = c.indices.shape[1]
    valid = int((c.indices >= 0).sum())
    assert (nq, hq, dqk, topk, valid) == (64, 128, 576, 2048, 27239)
    nbytes, _ = r.counts()
    assert nbytes == (nq * hq * dqk * 2 + nq * hq * 512 * 2 + valid * dqk * 2 +
                      nq * topk * 4 + hq * nq * 4)

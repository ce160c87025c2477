"""Parity of the sparse-index (MLA decode) CUDA path with the oracle.

Covers the full 64-query x 128-head decode workload with 1/4/16/128/512/2048
valid keys per query (afierka-intel/vllm pull 76, Why / Test plan), the
-inf no-op, empty rows, -1 padding anywhere in the row, out-of-range and
repeated indices, lists that end inside a slice, head counts below and above
one 128-row block, more than 256 queries, more than eight 256-key items per
query, the longest accepted list (topk 8192, 32 items), and workspace reuse across
calls.
"""
import numpy as np
import pytest

from attention_head_sinks_gb300 import workloads as W
from oracle import sa_oracle as O
from tests.gpu_util import LSE_TOL, REL_L2_TOL, compare, dev

pytestmark = pytest.mark.gpu

NONE, NULL = W.SINK_NONE, W.SINK_NULL_LOGIT


@pytest.fixture(autouse=True)
def _no_device_errors():
    import attention_head_sinks_gb300 as sa
    yield
    assert sa.sa_device_error() == 0


def gpu_run(c, mode, sinks=None, indices=None, workspace=None):
    import torch
    import attention_head_sinks_gb300 as sa
    s = c.sinks if sinks is None else sinks
    idx = c.indices if indices is None else indices
    out, lse = sa.sa_sparse_index_fwd(dev(c.q), dev(c.kv), dev(idx), c.dv, dev(s),
                                      mode, c.scale, workspace=workspace)
    torch.cuda.synchronize()
    return out, lse


def check(c, mode, sinks=None, indices=None, workspace=None):
    out, lse = gpu_run(c, mode, sinks, indices, workspace)
    ro, rl, _ = O.sparse_index_fwd(c.q, c.kv, c.indices if indices is None else indices,
                                   c.dv, c.sinks if sinks is None else sinks, mode,
                                   c.scale)
    rel, dl = compare(out, lse, ro, rl)
    assert rel <= REL_L2_TOL and dl <= LSE_TOL, (c.name, mode, rel, dl)
    return out, lse


@pytest.mark.parametrize("mode", [NULL, NONE])
def test_mla_sparse_decode_full(mode):
    check(W.mla_sparse_decode(mode), mode)


def test_mla_sparse_decode_per_valid_count():
    """Each valid-key class separately meets the bar (rows of one class)."""
    c = W.mla_sparse_decode(NULL, seed=1104)
    out, lse = gpu_run(c, NULL)
    ro, rl, n = O.sparse_index_fwd(c.q, c.kv, c.indices, c.dv, c.sinks, NULL, c.scale)
    for cnt in W.MLA_VALID_COUNTS:
        rows = np.nonzero(n == cnt)[0]
        rel, dl = compare(out, lse, ro, rl, rows=rows)
        assert rel <= REL_L2_TOL and dl <= LSE_TOL, (cnt, rel, dl)


def test_full_size_null_sink_is_applied_on_short_rows():
    """The full decode batch in the benchmark's launch configuration: for the
    short lists (1, 4 and 16 valid keys) the NULL_LOGIT output must differ
    from the no-sink output far beyond the tolerance, and the difference must
    be the oracle's, row by row (a row whose sink were dropped would show a
    difference of zero)."""
    from tests.gpu_util import ROW_REL_TOL, row_errors
    c = W.mla_sparse_decode(NULL)
    o2, l2 = gpu_run(c, NULL)
    o0, _ = gpu_run(c, NONE)
    r2, rl2, n = O.sparse_index_fwd(c.q, c.kv, c.indices, c.dv, c.sinks, NULL, c.scale)
    r0, _, _ = O.sparse_index_fwd(c.q, c.kv, c.indices, c.dv, c.sinks, NONE, c.scale)
    g2 = o2.float().cpu().numpy().astype(np.float64)
    g0 = o0.float().cpu().numpy().astype(np.float64)
    nr = np.linalg.norm(r2, axis=-1)
    scale = np.maximum(nr, 0.1 * np.sqrt(np.mean(nr ** 2)))
    err = np.linalg.norm((g2 - g0) - (r2 - r0), axis=-1) / scale
    assert err.max() <= 2 * ROW_REL_TOL, (np.unravel_index(err.argmax(), err.shape), err.max())
    for cnt in (1, 4, 16):
        rows = np.nonzero(n == cnt)[0]
        moved = np.linalg.norm((g2 - g0)[rows]) / np.linalg.norm(r2[rows])
        assert moved >= 30 * REL_L2_TOL, (cnt, moved)  # oracle: 1.14, 0.45, 0.15
        sig = (np.linalg.norm((r2 - r0)[rows], axis=-1) / scale[rows])
        assert (sig > 4 * ROW_REL_TOL).mean() >= 0.5
    assert row_errors(g2, r2).max() <= ROW_REL_TOL
    rel, dl = compare(o2, l2, r2, rl2)
    assert rel <= REL_L2_TOL and dl <= LSE_TOL


def test_neg_inf_sink_is_bitwise_no_sink():
    import torch
    c = W.mla_sparse_decode(NULL, seed=1204)
    ninf = np.full(c.num_q_heads, -np.inf, np.float32)
    o0, l0 = gpu_run(c, NONE)
    o2, l2 = gpu_run(c, NULL, sinks=ninf)
    assert torch.equal(o0.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l0, l2)


def ragged_indices(rng, nq, nkv, topk, counts):
    idx = np.full((nq, topk), -1, np.int32)
    for q in range(nq):
        c = counts[q % len(counts)]
        sel = rng.choice(nkv, size=c, replace=False).astype(np.int32)
        pos = np.sort(rng.choice(topk, size=c, replace=False))
        idx[q, pos] = sel                      # -1 padding anywhere in the row
    return idx


@pytest.mark.parametrize("hq", [128, 64, 192])
@pytest.mark.parametrize("mode", [NULL, NONE])
def test_ragged_lists(hq, mode):
    rng = np.random.default_rng(hq)
    counts = [0, 1, 3, 17, 255, 256, 257, 511, 600, 1000]
    c = W.index_case(10, hq, 576, 512, 5000, 1024, counts, (-2.2, 2.49), mode,
                     3000 + hq, "ragged_idx")
    idx = ragged_indices(rng, 10, 5000, 1024, counts)
    idx[3, 7] = 5000          # out of range: absent
    idx[4, 9] = -123          # negative: absent
    out, lse = check(c, mode, indices=idx)
    assert (out[0] == 0).all() and bool(lse[:, 0].isneginf().all())


def test_repeated_index_counts_twice():
    c = W.index_case(4, 128, 576, 512, 700, 300, (5, 40, 260, 299), (-2.2, 2.49),
                     NULL, 3100, "dup")
    idx = c.indices.copy()
    idx[1, 40] = idx[1, 0]
    idx[2, 270] = idx[2, 3]
    check(c, NULL, indices=idx)


@pytest.mark.parametrize("topk", [1, 16, 200, 256, 257, 513])
def test_list_lengths(topk):
    c = W.index_case(6, 128, 576, 512, 3000, topk, (topk, 1, topk // 2 + 1),
                     (-2.2, 2.49), NULL, 3200 + topk, "len")
    check(c, NULL)


def test_workspace_reuse_with_stale_contents():
    import torch
    import attention_head_sinks_gb300 as sa
    c = W.index_case(8, 128, 576, 512, 4000, 1024, (1000, 3, 700, 0), (-2.2, 2.49),
                     NULL, 3300, "reuse")
    ws = torch.empty(sa.sa_sparse_index_workspace_size(8, 128, 512, 1024),
                     dtype=torch.uint8, device="cuda")
    check(c, NULL, workspace=ws)
    # second call: the multi-slice rows become single-slice and vice versa
    idx2 = c.indices[::-1].copy()
    check(c, NULL, indices=idx2, workspace=ws)


def test_two_streams_own_workspaces():
    # two decode batches in flight at once on two streams, each with its own
    # workspace (the pattern of a pipelined caller): neither disturbs the other
    import torch
    import attention_head_sinks_gb300 as sa
    cs = [W.index_case(16, 128, 576, 512, 6000, 2048, cnt, (-2.2, 2.49), NULL, 3700 + i, "s%d" % i)
          for i, cnt in enumerate(((2048, 7, 600), (1, 1500, 256, 2048)))]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    ins = [(dev(c.q), dev(c.kv), dev(c.indices), dev(c.sinks)) for c in cs]
    wss = [torch.empty(sa.sa_sparse_index_workspace_size(16, 128, 512, 2048), dtype=torch.uint8,
                       device="cuda") for _ in cs]
    torch.cuda.synchronize()
    outs = []
    for rep in range(3):
        for k in range(2):
            with torch.cuda.stream(streams[k]):
                q, kv, idx, s = ins[k]
                o = sa.sa_sparse_index_fwd(q, kv, idx, 512, s, NULL, cs[k].scale, workspace=wss[k])
                if rep == 2:
                    outs.append(o)
    torch.cuda.synchronize()
    for c, (out, lse) in zip(cs, outs):
        ro, rl, _ = O.sparse_index_fwd(c.q, c.kv, c.indices, c.dv, c.sinks, NULL, c.scale)
        rel, dl = compare(out, lse, ro, rl)
        assert rel <= REL_L2_TOL and dl <= LSE_TOL, (c.name, rel, dl)


@pytest.mark.parametrize("nq", [600, 1100])
def test_many_queries(nq):
    # more than 256 queries: each CTA's item lookup scans several queries
    # per thread; full and short items of many queries interleave
    c = W.index_case(nq, 16, 576, 512, 4096, 520, (0, 520, 7, 256, 300, 1),
                     (-2.2, 2.49), NULL, 3400 + nq, "many_q")
    check(c, NULL)


@pytest.mark.parametrize("hq", [128, 192])
def test_all_lists_full(hq):
    # every query lists 2048 valid keys: 8 full items per query and 128-head
    # block, 512 or 1024 CTAs with work, several waves of them, and every
    # query goes through the combine
    c = W.index_case(64, hq, 576, 512, 65536, 2048, (2048,), (-2.2, 2.49), NULL, 3600 + hq,
                     "all_full")
    check(c, NULL)


@pytest.mark.parametrize("hq", [128, 40])
def test_more_than_eight_items(hq):
    # topk 3000: 2900 and 2100 valid keys give 12 and 9 items of 256 keys
    # (the merge path for more than eight items), 300 gives 2, 7 gives 1
    c = W.index_case(4, hq, 576, 512, 9000, 3000, (2900, 300, 2100, 7), (-2.2, 2.49),
                     NULL, 3500 + hq, "many_items")
    check(c, NULL)


@pytest.mark.parametrize("hq", [128, 40])
def test_maximum_topk(hq):
    # the longest list the entry point accepts (topk 8192): a full list is 32
    # items of 256 keys, merged eight items at a time; 8191 valid keys end one
    # key short of the last item; a single key needs no merge
    c = W.index_case(3, hq, 576, 512, 20000, 8192, (8192, 1, 8191), (-2.2, 2.49), NULL,
                     3700 + hq, "max_topk")
    check(c, NULL)

"""Parity of on-device block selection (``sa_block_select``) and of the
per-index-head block-sparse attention (``sa_block_sparse_fwd_index_heads``)
with the oracle.

Selection is an integer result decided by floating-point scores: the kernel
ranks fp32 block scores (tensor-core accumulation), the oracle fp64 ones.
Every row must therefore be a valid top-k under the oracle's scores within a
tolerance of a few fp32 ulps of the score scale (selected blocks no lower,
unselected blocks no higher, than the k-th score), carry its diagonal block
and the right count, ascending and -1 padded; rows with no near-tie must
match exactly, and nearly all rows do.  Where every score is exact in fp32
(the tie-heavy closed form) the tables must match exactly, ties included.
The attention with one table per index head is compared with the oracle on
random tables and on the tables the kernel selected.
"""
import numpy as np
import pytest

from attention_head_sinks_gb300 import workloads as W
from oracle import sa_oracle as O
from tests.gpu_util import LSE_TOL, REL_L2_TOL, compare, dev

pytestmark = pytest.mark.gpu

EPS = 1e-3  # |fp32 - fp64| block-score bound used for near-ties (scores ~ 1e1)


@pytest.fixture(autouse=True)
def _no_device_errors():
    import attention_head_sinks_gb300 as sa
    yield
    assert sa.sa_device_error() == 0


def gpu_select(c):
    import torch
    import attention_head_sinks_gb300 as sa
    tab = sa.sa_block_select(dev(c.index_q), dev(c.index_k), c.batch, c.seq_len,
                             c.block_size, c.topk)
    torch.cuda.synchronize()
    return tab.cpu().numpy()


def check_selection(c, got, rows=None):
    ref, sc = O.block_select(c.index_q, c.index_k, c.batch, c.seq_len, c.block_size, c.topk,
                             rows=rows)
    b, e = (0, c.batch * c.seq_len) if rows is None else rows
    mismatched = 0
    for g in range(c.num_index_heads):
        for i in range(b, e):
            row = got[g, i]
            diag = (i % c.seq_len) // c.block_size
            n = min(diag + 1, c.topk)
            assert (row[n:] == -1).all(), (g, i, row)
            sel = row[:n]
            assert (np.diff(sel) > 0).all() and sel[-1] == diag, (g, i, row)
            if np.array_equal(row, ref[g, i]):
                continue
            mismatched += 1
            # a near-tie: still a valid top-(k-1) of the earlier blocks
            s = sc[g, i, :diag]
            thr = np.sort(s)[::-1][c.topk - 2]
            chosen = [x for x in sel if x != diag]
            others = [x for x in range(diag) if x not in chosen]
            assert min(s[chosen]) >= thr - EPS, (g, i, row, ref[g, i])
            assert not others or max(s[others]) <= thr + EPS, (g, i, row, ref[g, i])
    return mismatched


@pytest.mark.parametrize("hi,topk", [(1, 4), (3, 16), (4, 1), (2, 9)])
def test_small_selection(hi, topk):
    c = W.select_case(2, 384, hi, 128, 64, topk, seed=40 + hi * 17 + topk)
    got = gpu_select(c)
    assert got.shape == (hi, 768, topk)
    mism = check_selection(c, got)
    assert mism <= 0.01 * hi * 768, mism


@pytest.mark.parametrize("batch,seq_len", [(1, 128), (3, 128), (1, 640)])
def test_short_rows_and_batches(batch, seq_len):
    # fewer tokens than one 256-key tile (the key box runs past the tensor),
    # rows that end inside a key tile, and a batch of one-tile rows
    c = W.select_case(batch, seq_len, 2, 128, 64, 3, seed=80 + batch + seq_len)
    got = gpu_select(c)
    assert check_selection(c, got) <= 0.01 * 2 * batch * seq_len


def test_dsa_block_select_sampled_rows():
    c = W.dsa_block_select()
    got = gpu_select(c)
    T = c.batch * c.seq_len
    total = 0
    for s in range(0, T, T // 8):          # 8 spans of 48 rows, both batch rows
        b = s + (T // 8) - 48
        total += check_selection(c, got, rows=(b, b + 48))
    assert total <= 0.01 * 8 * 48 * c.num_index_heads, total


def test_ties_match_exactly():
    # index q = e0 on every head; key j = f(block(j)) on one token of its
    # block and f - 1 on the rest: block score f(block), exact in fp32,
    # with many ties (broken toward the lower block id)
    bs, S, topk = 64, 1024, 6
    f = lambda blk: float((blk * 7) % 5)
    q = np.zeros((2 * S, 2, 128), np.float32)
    q[:, :, 0] = 1.0
    k = np.zeros((2 * S, 128), np.float32)
    for j in range(2 * S):
        blk = (j % S) // bs
        k[j, 0] = f(blk) if j % bs == (blk % bs) else f(blk) - 1.0
    c = W.SelectCase("ties", W.f32_to_bf16_bits(q), W.f32_to_bf16_bits(k), 2, S, bs, topk)
    got = gpu_select(c)
    ref, _ = O.block_select(c.index_q, c.index_k, 2, S, bs, topk)
    assert np.array_equal(got, ref)


def gpu_attend_ih(c, tables, mode, sinks=None):
    import torch
    import attention_head_sinks_gb300 as sa
    out, lse = sa.sa_block_sparse_fwd_index_heads(
        dev(c.q), dev(c.k), dev(c.v), c.batch, c.seq_len, dev(tables), c.block_size,
        dev(c.cu_docs), dev(c.sinks if sinks is None else sinks), mode, c.scale)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("hi", [1, 2, 4])
@pytest.mark.parametrize("mode", [W.SINK_NULL_LOGIT, W.SINK_KEY0_BIAS])
def test_index_head_attention_random_tables(hi, mode):
    c = W.block_case(2, 512, 16, 4, 128, 64, 5, 3, (-2.2, 2.49), mode, seed=50 + hi)
    rng = np.random.default_rng(60 + hi)
    tabs = np.stack([W.random_block_table(rng, 2, 512, 64, 5) for _ in range(hi)])
    out, lse = gpu_attend_ih(c, tabs, mode)
    ro, rl, _ = O.block_sparse_fwd_index_heads(c.q, c.k, c.v, 2, 512, tabs, 64, c.cu_docs,
                                               c.sinks, mode, c.scale)
    rel, dl = compare(out, lse, ro, rl)
    assert rel <= REL_L2_TOL and dl <= LSE_TOL, (hi, mode, rel, dl)


def test_index_head_attention_rejects_non_divisor():
    import torch
    import attention_head_sinks_gb300 as sa
    c = W.block_case(1, 256, 8, 4, 128, 64, 3, 1, (-2.2, 2.49), W.SINK_NONE, seed=70)
    tabs = np.stack([c.block_table] * 3)
    with pytest.raises(sa.SAError):
        gpu_attend_ih(c, tabs, W.SINK_NONE)
    torch.cuda.synchronize()


def test_select_then_attend_dsa_sampled_rows():
    """The DSA prefill batch with its selection made on the device: 4 index
    heads (one per KV head), top-16 of 64-token blocks, then the attention
    with those tables, against the oracle on the kernel's tables."""
    sc = W.dsa_block_select()
    ac = W.dsa_block_prefill(W.SINK_NULL_LOGIT)
    tabs = gpu_select(sc)
    out, lse = gpu_attend_ih(ac, tabs, W.SINK_NULL_LOGIT)
    T = ac.batch * ac.seq_len
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    for s in range(0, T, T // 8):
        b = s + (T // 8) - 32
        ro, rl, _ = O.block_sparse_fwd_index_heads(ac.q, ac.k, ac.v, ac.batch, ac.seq_len,
                                                   tabs, 64, ac.cu_docs, ac.sinks,
                                                   W.SINK_NULL_LOGIT, ac.scale,
                                                   rows=(b, b + 32))
        rel = np.linalg.norm(o[b:b + 32] - ro[b:b + 32]) / np.linalg.norm(ro[b:b + 32])
        fin = np.isfinite(rl[:, b:b + 32])
        dl = np.abs(l[:, b:b + 32][fin] - rl[:, b:b + 32][fin]).max()
        assert rel <= REL_L2_TOL and dl <= LSE_TOL, (b, rel, dl)

"""Parity of the block-sparse (DSA prefill) CUDA path with the oracle.

Covers the full 2 x 8192-token workload (32 query / 4 KV heads, head dim 128,
64-key blocks, top-16 blocks, 3 documents per batch row) on sampled rows in
all three sink modes (KEY0_BIAS: the document's first key), the padded-row
variant (empty key sets), the -inf and zero-bias no-ops, and small ragged
cases over every GQA ratio with repeated, out-of-range and future block ids
and document boundaries inside blocks.
"""
import numpy as np
import pytest

from attention_head_sinks_gb300 import workloads as W
from oracle import sa_oracle as O
from tests.gpu_util import LSE_TOL, REL_L2_TOL, compare, dev

pytestmark = pytest.mark.gpu

NONE, KEY0, NULL = W.SINK_NONE, W.SINK_KEY0_BIAS, W.SINK_NULL_LOGIT


@pytest.fixture(autouse=True)
def _no_device_errors():
    import attention_head_sinks_gb300 as sa
    yield
    assert sa.sa_device_error() == 0


def gpu_run(c, mode, sinks=None, table=None):
    import torch
    import attention_head_sinks_gb300 as sa
    s = c.sinks if sinks is None else sinks
    tab = c.block_table if table is None else table
    out, lse = sa.sa_block_sparse_fwd(dev(c.q), dev(c.k), dev(c.v), c.batch, c.seq_len,
                                      dev(tab), c.block_size, dev(c.cu_docs), dev(s),
                                      mode, c.scale)
    torch.cuda.synchronize()
    return out, lse


def oracle_run(c, mode, sinks=None, table=None, rows=None):
    o, l, _ = O.block_sparse_fwd(c.q, c.k, c.v, c.batch, c.seq_len,
                                 c.block_table if table is None else table,
                                 c.block_size, c.cu_docs,
                                 c.sinks if sinks is None else sinks, mode, c.scale,
                                 rows=rows)
    return o, l


def sample_rows(c, span=256):
    """Rows around batch-row starts and ends, document starts and a few
    interior stretches."""
    starts = set()
    for b in range(c.batch):
        starts.add(b * c.seq_len)
        starts.add((b + 1) * c.seq_len - span)
        starts.add(b * c.seq_len + c.seq_len // 2)
    for d in c.cu_docs[1:-1]:
        starts.add(max(0, int(d) - span // 2))
    rows = []
    for s in sorted(starts):
        rows.append((s, min(s + span, c.total_tokens)))
    return rows


def check_sampled(c, mode, sinks=None):
    out, lse = gpu_run(c, mode, sinks)
    idx = []
    ro = None
    for r in sample_rows(c):
        o, l = oracle_run(c, mode, sinks, rows=r)
        if ro is None:
            ro, rl = o, l
        else:
            ro[r[0]:r[1]] = o[r[0]:r[1]]
            rl[:, r[0]:r[1]] = l[:, r[0]:r[1]]
        idx.extend(range(*r))
    idx = np.unique(np.array(idx))
    rel, dl = compare(out, lse, ro, rl, rows=idx)
    assert rel <= REL_L2_TOL and dl <= LSE_TOL, (c.name, mode, rel, dl)
    return out, lse


@pytest.mark.parametrize("mode", [NULL, NONE, KEY0])
def test_dsa_block_prefill_full_size_sampled(mode):
    check_sampled(W.dsa_block_prefill(mode), mode)


def test_dsa_padded_rows_are_zero():
    c = W.dsa_block_prefill(NULL, pad_rows=64)
    out, lse = check_sampled(c, NULL)
    for b in range(c.batch):
        sl = slice((b + 1) * c.seq_len - 64, (b + 1) * c.seq_len)
        assert (out[sl] == 0).all() and bool(lse[:, sl].isneginf().all())


def test_dsa_neg_inf_sinks_are_bitwise_no_sink():
    import torch
    c = W.dsa_block_prefill(NULL, sinks_neg_inf=True)
    o0, l0 = gpu_run(c, NONE)
    o2, l2 = gpu_run(c, NULL)
    assert torch.equal(o0.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l0, l2)


SMALL = [
    # batch, seq_len, hq, hkv, topk, docs_per_row
    (2, 256, 8, 1, 4, 3),
    (3, 384, 16, 2, 3, 4),
    (1, 512, 16, 4, 5, 2),
    (2, 640, 32, 4, 16, 3),
    (1, 256, 16, 16, 2, 5),
    (2, 128, 16, 1, 2, 1),
    (1, 256, 8, 4, 4, 2),
]


@pytest.mark.parametrize("mode", [NULL, NONE, KEY0])
@pytest.mark.parametrize("ci", range(len(SMALL)))
def test_small_ragged(ci, mode):
    batch, S, hq, hkv, topk, docs = SMALL[ci]
    c = W.block_case(batch, S, hq, hkv, 128, 64, topk, docs, (-2.2, 2.49), mode,
                     5000 + ci, pad_rows=3, name="small%d" % ci)
    tab = c.block_table.copy()
    rng = np.random.default_rng(ci)
    T = c.total_tokens
    for i in rng.choice(T, size=T // 8, replace=False):
        k = rng.integers(0, topk)
        r = rng.integers(0, 4)
        if r == 0:
            tab[i, k] = tab[i, 0]                       # repeated id
        elif r == 1:
            tab[i, k] = S // 64 + int(rng.integers(0, 5))  # out of range
        elif r == 2:
            tab[i, k] = int(rng.integers(0, S // 64))   # any block, maybe future
        else:
            tab[i, k] = -1
    out, lse = gpu_run(c, mode, table=tab)
    ro, rl = oracle_run(c, mode, table=tab)
    rel, dl = compare(out, lse, ro, rl)
    assert rel <= REL_L2_TOL and dl <= LSE_TOL, (c.name, mode, rel, dl)


def test_all_rows_empty():
    c = W.block_case(1, 256, 16, 2, 128, 64, 4, 2, (-2.2, 2.49), NULL, 5100, name="empty")
    tab = np.full_like(c.block_table, -1)
    out, lse = gpu_run(c, NULL, table=tab)
    assert (out == 0).all() and bool(lse.isneginf().all())


def test_zero_key0_sink_is_bitwise_no_sink():
    import torch
    c = W.dsa_block_prefill(KEY0, seed=1405)
    o0, l0 = gpu_run(c, NONE)
    o1, l1 = gpu_run(c, KEY0, sinks=np.zeros_like(c.sinks))
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16))
    assert torch.equal(l0, l1)


def test_key0_extreme_sinks_and_dominant_first_key():
    # every document's first key carries the largest raw logit of its rows
    # (q = 4 e0, that key 8 e0, other keys random), with KEY0_BIAS sinks
    # -inf, -30, +4 and 0 over the four query heads of each KV head: the first
    # key removed (documents of one token become empty rows), far below the
    # rest, dominant, or unbiased
    c = W.block_case(2, 512, 16, 4, 128, 64, 5, 40, (-2.2, 2.49), KEY0, seed=4500,
                     name="k0_extremes")
    q = (c.q.astype(np.uint32) << 16).view(np.float32).copy()
    q[:] = 0.0
    q[:, :, 0] = 4.0
    k = (c.k.astype(np.uint32) << 16).view(np.float32).copy()
    firsts = np.unique(c.cu_docs[:-1])
    k[firsts, :, :] = 0.0
    k[firsts, :, 0] = 8.0
    c.q = W.f32_to_bf16_bits(q)
    c.k = W.f32_to_bf16_bits(k)
    sinks = np.tile(np.array([-np.inf, -30.0, 4.0, 0.0], np.float32), 4)
    out, lse = gpu_run(c, KEY0, sinks=sinks)
    ro, rl = oracle_run(c, KEY0, sinks=sinks)
    rel, dl = compare(out, lse, ro, rl)
    assert rel <= REL_L2_TOL and dl <= LSE_TOL, (rel, dl)


@pytest.mark.parametrize("docs_per_row", [200, 300])
@pytest.mark.parametrize("mode", [NULL, KEY0])
def test_many_documents(docs_per_row, mode):
    # hundreds of short documents: most key blocks are cut by a document
    # start, most tokens see only part of their selected blocks
    c = W.block_case(1, 4096, 16, 4, 128, 64, 8, docs_per_row, (-2.2, 2.49), mode,
                     seed=4000 + docs_per_row)
    out, lse = gpu_run(c, mode)
    ro, rl = oracle_run(c, mode)
    rel, dl = compare(out, lse, ro, rl)
    assert rel <= REL_L2_TOL and dl <= LSE_TOL, (docs_per_row, mode, rel, dl)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (16, 4), (16, 1)])
@pytest.mark.parametrize("mode", [NULL, KEY0])
def test_many_tiles_per_cta(hq, hkv, mode):
    # 2 x 4096 tokens: every CTA walks several tiles (G = 1, 2, 4, 16: 3.4 to
    # 6.7 tiles per CTA), so each tile's metadata, Q and O are handed over
    # from the previous tile's
    c = W.block_case(2, 4096, hq, hkv, 128, 64, 8, 3, (-2.2, 2.49), mode, seed=6000 + hq + hkv,
                     pad_rows=40)
    out, lse = gpu_run(c, mode)
    ro, rl = oracle_run(c, mode)
    rel, dl = compare(out, lse, ro, rl)
    assert rel <= REL_L2_TOL and dl <= LSE_TOL, (hq, hkv, mode, rel, dl)


def test_union_capacity_is_checked():
    import torch
    import attention_head_sinks_gb300 as sa
    # one token per KV group row tile of 128 tokens x topk 16 = 2048 possible
    # union blocks, and 1032 blocks per row: above the 1024-block capacity
    S = 66048
    q = torch.zeros((S, 1, 128), dtype=torch.bfloat16, device="cuda")
    tab = torch.full((S, 16), -1, dtype=torch.int32, device="cuda")
    cu = torch.tensor([0, S], dtype=torch.int32, device="cuda")
    with pytest.raises(sa.SAError) as e:
        sa.sa_block_sparse_fwd(q, q, q, 1, S, tab, 64, cu, None, NONE, 0.08)
    assert "union blocks" in str(e.value)

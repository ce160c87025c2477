"""Pins of the block-selection oracle (``block_select``) and of the
one-table-per-index-head attention oracle.

[M3 CP sparse] forward step 3 selects the top-k key blocks of each query from
index q / k over the causal sequence, one selection per index head
(``_select_local_blocks`` returns ``[batch, index_heads, sequence,
key_blocks]``); the page gives no score formula.  Readings pinned here: dot
product token scores, max over a block's keys, the diagonal block always
selected, ties to the lower block id.  Pins: a pure-Python brute force on
tiny inputs; a closed form where the index keys encode a known block ranking
(with ties); max pooling (order of keys inside a block does not matter, one
large key lifts its block); structural invariants; and the per-index-head
attention against the single-table oracle.
"""
import math

import numpy as np
import pytest

from attention_head_sinks_gb300 import workloads as W
from oracle import sa_oracle as O


def brute_select(qf, kf, batch, seq_len, bs, topk):
    """Pure-Python loops: score every (head, token, earlier block), then sort
    by (-score, id)."""
    T, hi, di = len(qf), len(qf[0]), len(qf[0][0])
    table = [[[-1] * topk for _ in range(T)] for _ in range(hi)]
    for i in range(T):
        row0 = (i // seq_len) * seq_len
        diag = (i - row0) // bs
        for g in range(hi):
            cand = []
            for c in range(diag):
                best = -math.inf
                for j in range(row0 + c * bs, row0 + (c + 1) * bs):
                    best = max(best, math.fsum(qf[i][g][d] * kf[j][d] for d in range(di)))
                cand.append((-best, c))
            cand.sort()
            if diag + 1 <= topk:
                sel = list(range(diag + 1))
            else:
                sel = sorted([c for _, c in cand[:topk - 1]] + [diag])
            table[g][i][:len(sel)] = sel
    return np.array(table, np.int32)


def test_matches_brute_force_on_tiny_inputs():
    c = W.select_case(2, 40, 2, 3, 4, 4, seed=11)
    qf, kf = O._widen(c.index_q), O._widen(c.index_k)
    tab, sc = O.block_select(c.index_q, c.index_k, c.batch, c.seq_len, c.block_size, c.topk)
    ref = brute_select(qf.tolist(), kf.tolist(), c.batch, c.seq_len, c.block_size, c.topk)
    assert np.array_equal(tab, ref)


def test_closed_form_ranking_with_ties():
    # index q = e0 for every head; index key j = f(block) in dim 0 on one
    # token of its block and f - 1 on the others: block score = f(block)
    bs, S, topk = 4, 64, 5
    f = lambda blk: float((blk * 7) % 5)          # many equal scores
    T = S
    q = np.zeros((T, 2, 4), np.float32)
    q[:, :, 0] = 1.0
    k = np.zeros((T, 4), np.float32)
    for j in range(T):
        blk = j // bs
        k[j, 0] = f(blk) if j % bs == (blk % bs) else f(blk) - 1.0
    qb, kb = W.f32_to_bf16_bits(q), W.f32_to_bf16_bits(k)
    tab, sc = O.block_select(qb, kb, 1, S, bs, topk)
    for i in range(T):
        diag = i // bs
        if diag + 1 <= topk:
            want = list(range(diag + 1))
        else:
            ranked = sorted(range(diag), key=lambda c: (-f(c), c))
            want = sorted(ranked[:topk - 1] + [diag])
        for g in range(2):
            got = [x for x in tab[g, i] if x >= 0]
            assert got == want, (i, got, want)
            assert np.array_equal(sc[g, i, :diag], [f(c) for c in range(diag)])


def test_max_pooling_and_invariants():
    c = W.select_case(1, 256, 3, 16, 16, 6, seed=12)
    tab, sc = O.block_select(c.index_q, c.index_k, 1, 256, 16, 6)
    for g in range(3):
        for i in range(256):
            diag = i // 16
            sel = [x for x in tab[g, i] if x >= 0]
            assert sel == sorted(sel) and diag in sel
            assert len(sel) == min(diag + 1, 6) and max(sel) == diag
            if diag + 1 > 6:
                # every unselected earlier block scores no higher than the
                # lowest selected one
                lo = min(sc[g, i, x] for x in sel if x != diag)
                others = [sc[g, i, x] for x in range(diag) if x not in sel]
                assert max(others) <= lo
    # permuting the keys inside every block leaves the selection unchanged
    rng = np.random.default_rng(3)
    perm = np.concatenate([b * 16 + rng.permutation(16) for b in range(16)])
    tab2, _ = O.block_select(c.index_q, c.index_k[perm], 1, 256, 16, 6)
    # tokens inside one block see different causal prefixes only through
    # earlier blocks, which are permuted within themselves
    assert np.array_equal(tab, tab2)
    # one large key lifts its block into every later token's selection:
    # index head 0 gets a positive first component, the key 60 e0
    qf = O._widen(c.index_q).astype(np.float32)
    qf[:, 0, 0] = 3.0
    kf = O._widen(c.index_k).astype(np.float32)
    kf[5 * 16 + 7] = 0.0
    kf[5 * 16 + 7, 0] = 60.0
    tab3, sc3 = O.block_select(W.f32_to_bf16_bits(qf), W.f32_to_bf16_bits(kf), 1, 256, 16, 6)
    assert all(5 in tab3[0, i] for i in range(6 * 16, 256))
    assert (sc3[0, 6 * 16:, 5] == 180.0).all()


def test_rows_restriction_matches_full():
    c = W.select_case(2, 128, 2, 8, 16, 3, seed=13)
    full, sf = O.block_select(c.index_q, c.index_k, 2, 128, 16, 3)
    part, sp = O.block_select(c.index_q, c.index_k, 2, 128, 16, 3, rows=(100, 180))
    assert np.array_equal(full[:, 100:180], part[:, 100:180])
    assert (part[:, :100] == -2).all() and (part[:, 180:] == -2).all()


@pytest.mark.parametrize("mode", [W.SINK_NULL_LOGIT, W.SINK_KEY0_BIAS])
def test_index_head_attention_reduces_to_single_table(mode):
    c = W.block_case(1, 256, 8, 4, 64, 64, 3, 2, (-2.2, 2.49), mode, seed=14)
    ref = O.block_sparse_fwd(c.q, c.k, c.v, 1, 256, c.block_table, 64, c.cu_docs, c.sinks,
                             mode, c.scale)
    for hi in (1, 2, 4):
        tabs = np.repeat(c.block_table[None], hi, axis=0)
        got = O.block_sparse_fwd_index_heads(c.q, c.k, c.v, 1, 256, tabs, 64, c.cu_docs,
                                             c.sinks, mode, c.scale)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
    # different tables per index head: head group g follows table g only
    rng = np.random.default_rng(5)
    t2 = np.stack([c.block_table, W.random_block_table(rng, 1, 256, 64, 3)])
    got = O.block_sparse_fwd_index_heads(c.q, c.k, c.v, 1, 256, t2, 64, c.cu_docs, c.sinks,
                                         mode, c.scale)
    other = O.block_sparse_fwd(c.q, c.k, c.v, 1, 256, t2[1], 64, c.cu_docs, c.sinks, mode,
                               c.scale)
    assert np.array_equal(got[0][:, :4], ref[0][:, :4])
    assert np.array_equal(got[0][:, 4:], other[0][:, 4:])
    assert np.array_equal(got[1][4:], other[1][4:])

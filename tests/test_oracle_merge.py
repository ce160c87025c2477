"""Pins of the merge oracle (``oracle.sa_oracle.merge_states``).

The merge is pinned by an identity, not by re-typing its formula: merging the
sink-free attention over two disjoint halves of an index list must give the
attention over the whole list (the LSE convention of vLLM pull 49815, LSE
paragraph), with the NULL_LOGIT sink folded once (afierka-intel/vllm pull 76,
Implementation).  Also: LSE against numpy's ``logaddexp``, empty partials,
symmetry and the -inf sink no-op.
"""
import numpy as np
import pytest

from attention_head_sinks_gb300 import workloads as W
from oracle import sa_oracle as O

NONE, NULL = W.SINK_NONE, W.SINK_NULL_LOGIT


def _split_case(seed, counts=(1, 2, 5, 40, 300), nq=10, hq=3, topk=320, nkv=2000):
    c = W.index_case(nq, hq, 24, 16, nkv, topk, counts, (-2.2, 2.49), NULL, seed, "msplit")
    idx = c.indices
    # disjoint halves of each row's slots: even slots to A, odd slots to B
    ia = np.full_like(idx, -1)
    ib = np.full_like(idx, -1)
    ia[:, 0::2] = idx[:, 0::2]
    ib[:, 1::2] = idx[:, 1::2]
    return c, ia, ib


@pytest.mark.parametrize("mode", [NONE, NULL])
def test_merge_of_disjoint_halves_is_the_whole_list(mode):
    c, ia, ib = _split_case(11)
    oa, la, _ = O.sparse_index_fwd(c.q, c.kv, ia, c.dv, c.sinks, NONE, c.scale)
    ob, lb, _ = O.sparse_index_fwd(c.q, c.kv, ib, c.dv, c.sinks, NONE, c.scale)
    om, lm = O.merge_states(oa, la, ob, lb, c.sinks, mode)
    of, lf, _ = O.sparse_index_fwd(c.q, c.kv, c.indices, c.dv, c.sinks, mode, c.scale)
    np.testing.assert_allclose(om, of, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lm, lf, rtol=1e-12, atol=1e-12)


def test_lse_is_logaddexp():
    m = W.merge_case(50, 4, 8, 12, empty_frac=0.0)
    _, lse = O.merge_states(m.out_a, m.lse_a, m.out_b, m.lse_b, m.sinks, NULL)
    ref = np.logaddexp(m.lse_a.astype(np.float64), m.lse_b.astype(np.float64))
    np.testing.assert_allclose(lse, ref, rtol=1e-13, atol=1e-13)


def test_empty_partials():
    m = W.merge_case(40, 3, 8, 13, empty_frac=0.3)
    oa = O._widen(m.out_a)
    out_n, lse_n = O.merge_states(m.out_a, m.lse_a, m.out_b, m.lse_b, None, NONE)
    out_s, lse_s = O.merge_states(m.out_a, m.lse_a, m.out_b, m.lse_b, m.sinks, NULL)
    a_only = np.isfinite(m.lse_a) & np.isneginf(m.lse_b)
    both = np.isneginf(m.lse_a) & np.isneginf(m.lse_b)
    assert a_only.any() and both.any()
    h, t = np.nonzero(a_only)
    # only A has keys: NONE returns A exactly; NULL_LOGIT scales it by
    # e^lse / (e^lse + e^s)
    np.testing.assert_array_equal(out_n[t, h], oa[t, h])
    la = m.lse_a[h, t].astype(np.float64)
    s = m.sinks[h].astype(np.float64)
    np.testing.assert_allclose(out_s[t, h], oa[t, h] * (1.0 / (1.0 + np.exp(s - la)))[:, None],
                               rtol=1e-13)
    np.testing.assert_array_equal(lse_n[h, t], la)
    np.testing.assert_array_equal(lse_s[h, t], la)
    h, t = np.nonzero(both)
    assert (out_s[t, h] == 0).all() and np.isneginf(lse_s[h, t]).all()


def test_symmetric_and_neg_inf_sink_is_no_sink():
    m = W.merge_case(30, 2, 16, 14)
    o1, l1 = O.merge_states(m.out_a, m.lse_a, m.out_b, m.lse_b, m.sinks, NULL)
    o2, l2 = O.merge_states(m.out_b, m.lse_b, m.out_a, m.lse_a, m.sinks, NULL)
    np.testing.assert_allclose(o1, o2, rtol=1e-15, atol=1e-15)
    np.testing.assert_array_equal(l1, l2)
    ninf = np.full_like(m.sinks, -np.inf)
    o3, l3 = O.merge_states(m.out_a, m.lse_a, m.out_b, m.lse_b, ninf, NULL)
    o4, l4 = O.merge_states(m.out_a, m.lse_a, m.out_b, m.lse_b, None, NONE)
    np.testing.assert_array_equal(o3, o4)
    np.testing.assert_array_equal(l3, l4)


def test_sink_changes_short_rows():
    # a sink of weight comparable to the keys must move the output well
    # beyond the GPU tolerance (the sink is really folded in)
    m = W.merge_case(20, 2, 8, 15, lse_range=(-1.0, 1.0), empty_frac=0.0,
                     sink_range=(0.5, 1.0))
    o_n, _ = O.merge_states(m.out_a, m.lse_a, m.out_b, m.lse_b, None, NONE)
    o_s, _ = O.merge_states(m.out_a, m.lse_a, m.out_b, m.lse_b, m.sinks, NULL)
    rel = np.linalg.norm(o_s - o_n) / np.linalg.norm(o_n)
    assert rel > 0.05

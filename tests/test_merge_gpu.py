"""Parity of sa_merge_attn_states (CUDA, through the C ABI) with the oracle.

Random partials with empty key sets (LSE = -inf, in one or both), head dims
8 ... 512, one and many heads, in-place output, the -inf sink no-op, and a
composed check: the sparse-index attention over two disjoint halves of each
index list, merged on the GPU, against the oracle over the whole list.
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


def gpu_merge(m, mode, sinks=None, in_place=False):
    import torch
    import attention_head_sinks_gb300 as sa
    oa, ob = dev(m.out_a), dev(m.out_b)
    s = m.sinks if sinks is None else sinks
    out, lse = sa.sa_merge_attn_states(oa, dev(m.lse_a), ob, dev(m.lse_b), dev(s), mode,
                                       out=oa if in_place else None)
    torch.cuda.synchronize()
    return out, lse


def check(m, mode, **kw):
    out, lse = gpu_merge(m, mode, **kw)
    ro, rl = O.merge_states(m.out_a, m.lse_a, m.out_b, m.lse_b, m.sinks, mode)
    rel, dl = compare(out, lse, ro, rl)
    assert rel <= REL_L2_TOL and dl <= LSE_TOL, (m.name, mode, rel, dl)
    both = np.isneginf(m.lse_a) & np.isneginf(m.lse_b)
    h, t = np.nonzero(both)
    o = out.float().cpu().numpy()
    assert (o[t, h] == 0).all() and bool(np.isneginf(lse.cpu().numpy()[h, t]).all())
    return out, lse


@pytest.mark.parametrize("mode", [NULL, NONE])
@pytest.mark.parametrize("shape", [(37, 3, 8), (4096, 16, 80), (64, 128, 512), (1, 1, 128),
                                   (300, 7, 120)])
def test_random_partials(shape, mode):
    T, H, D = shape
    check(W.merge_case(T, H, D, 4000 + T + H + D, empty_frac=0.1, mode=mode,
                       name="m%dx%dx%d" % shape), mode)


def test_in_place_output():
    check(W.merge_case(500, 8, 64, 4100, empty_frac=0.1), NULL, in_place=True)


def test_window_partials_full_size():
    m = W.merge_window_partials()
    check(m, NULL)


def test_neg_inf_sink_is_bitwise_no_sink():
    import torch
    m = W.merge_case(700, 16, 80, 4200, empty_frac=0.05)
    o0, l0 = gpu_merge(m, NONE)
    o2, l2 = gpu_merge(m, NULL, sinks=np.full_like(m.sinks, -np.inf))
    assert torch.equal(o0.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l0, l2)


def test_merged_halves_match_the_whole_list():
    import torch
    import attention_head_sinks_gb300 as sa
    c = W.mla_sparse_decode(NULL, seed=1304)
    idx = c.indices
    ia = np.full_like(idx, -1)
    ib = np.full_like(idx, -1)
    ia[:, 0::2] = idx[:, 0::2]
    ib[:, 1::2] = idx[:, 1::2]
    q, kv, s = dev(c.q), dev(c.kv), dev(c.sinks)
    oa, la = sa.sa_sparse_index_fwd(q, kv, dev(ia), c.dv, None, NONE, c.scale)
    ob, lb = sa.sa_sparse_index_fwd(q, kv, dev(ib), c.dv, None, NONE, c.scale)
    out, lse = sa.sa_merge_attn_states(oa, la, ob, lb, s, NULL)
    torch.cuda.synchronize()
    ro, rl, _ = O.sparse_index_fwd(c.q, c.kv, idx, c.dv, c.sinks, NULL, c.scale)
    rel, dl = compare(out, lse, ro, rl)
    assert rel <= REL_L2_TOL and dl <= LSE_TOL, (rel, dl)

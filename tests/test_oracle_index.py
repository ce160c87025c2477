"""Pins of the sparse-index (MLA) oracle.

Source: afierka-intel/vllm pull 76 "Apply DeepSeek-V4 attn_sink in the XPU
sparse-MLA Triton kernel" -- Why (sinks in [-2.20, 2.49]; error vs valid keys
per row), Implementation (sink folded into the denominator after the key
loop, LSE over the selected keys only, -inf is a bitwise no-op), Test plan
(1/4/16/128/512 valid keys; the no-sink result must differ for short rows).
"""
import numpy as np
import pytest

from attention_head_sinks_gb300 import workloads as W
from oracle import brute
from oracle import sa_oracle as O
from tests.oracle_pins_util import bits_to_f64, rel_l2, sdpa_with_bias

NONE, NULL = W.SINK_NONE, W.SINK_NULL_LOGIT


def tiny(seed=21, counts=(1, 3, 12, 7, 0, 5), nkv=50, topk=12):
    return W.index_case(6, 4, 24, 16, nkv, topk, counts, (-2.2, 2.49), NULL,
                        seed, "tiny_index")


def run(c, mode, sinks=None, indices=None, rows=None):
    return O.sparse_index_fwd(c.q, c.kv, c.indices if indices is None else indices,
                              c.dv, c.sinks if sinks is None else sinks, mode,
                              c.scale, rows=rows)


@pytest.mark.parametrize("mode", [NONE, NULL])
def test_brute_force_matches_set_enumeration(mode):
    c = tiny()
    idx = c.indices.copy()
    idx[1, 5] = idx[1, 0]           # a repeated index counts twice
    idx[2, 3] = 10**6               # out of range: skipped
    idx[3, 1] = -7                  # negative: skipped
    o, l, n = run(c, mode, indices=idx)
    ob, lb = brute.sparse_index_fwd(c.q, c.kv, idx, c.dv, c.sinks, mode, c.scale)
    assert np.allclose(o, ob, rtol=1e-12, atol=1e-12)
    assert np.allclose(l, lb, rtol=1e-12, atol=1e-12)
    valid = ((idx >= 0) & (idx < c.num_kv)).sum(1)
    assert np.array_equal(n, valid)


@pytest.mark.parametrize("mode", [NONE, NULL])
def test_all_keys_listed_is_dense_mla_attention(mode):
    """Listing every cache row = dense attention with K = the whole latent row
    and V = its first dv columns (torch SDPA, fp64)."""
    c = tiny(nkv=30, topk=30)
    idx = np.tile(np.arange(30, dtype=np.int32), (c.num_queries, 1))
    o, _, _ = run(c, mode, indices=idx)
    qf, kvf = bits_to_f64(c.q), bits_to_f64(c.kv)
    hq = c.num_q_heads
    kx = np.repeat(kvf[:, None, :], hq, 1)
    vx = np.repeat(kvf[:, None, :c.dv], hq, 1)
    bias = np.zeros((hq, c.num_queries, 30))
    ref = sdpa_with_bias(qf, kx, vx, bias, c.scale,
                         null_sink=c.sinks if mode == NULL else None)
    assert rel_l2(o, ref) < 1e-12


def test_single_valid_key_null_logit_closed_form():
    """One valid key with a null-logit sink: out = v e^l / (e^l + e^s), and
    the LSE is the single logit l."""
    c = tiny(counts=(1,))
    o, l, n = run(c, NULL)
    assert np.all(n == 1)
    qf, kvf = bits_to_f64(c.q), bits_to_f64(c.kv)
    for i in range(c.num_queries):
        j = c.indices[i, 0]
        for h in range(c.num_q_heads):
            lg = c.scale * float(qf[i, h] @ kvf[j])
            s = float(c.sinks[h])
            assert abs(l[h, i] - lg) < 1e-12
            w = np.exp(lg) / (np.exp(lg) + np.exp(s))
            assert np.allclose(o[i, h], w * kvf[j, :c.dv], rtol=1e-12, atol=1e-14)


def test_neg_inf_sink_is_bitwise_no_sink():
    c = tiny()
    ninf = np.full(c.num_q_heads, -np.inf, np.float32)
    o0, l0, _ = run(c, NONE)
    o2, l2, _ = run(c, NULL, sinks=ninf)
    assert np.array_equal(o0, o2) and np.array_equal(l0, l2)


def test_lse_over_selected_keys_only():
    c = tiny()
    _, l0, _ = run(c, NONE)
    _, l2, _ = run(c, NULL)
    assert np.array_equal(l0, l2)


def test_empty_row_is_zero_with_neg_inf_lse():
    c = tiny()
    idx = c.indices.copy()
    idx[2] = -1
    for mode in (NONE, NULL):
        o, l, n = run(c, mode, indices=idx)
        assert n[2] == 0
        assert np.all(o[2] == 0.0) and np.all(np.isneginf(l[:, 2]))


def test_order_and_padding_position_do_not_matter():
    c = tiny()
    rng = np.random.default_rng(5)
    idx = c.indices.copy()
    for i in range(c.num_queries):
        rng.shuffle(idx[i])          # -1 entries end up anywhere in the row
    o0, l0, _ = run(c, NULL)
    o1, l1, _ = run(c, NULL, indices=idx)
    assert np.allclose(o0, o1, rtol=1e-13, atol=1e-15)
    assert np.allclose(l0, l1, rtol=1e-13, atol=1e-13)


def test_sink_error_shrinks_with_valid_keys():
    """The sink-ignored vs sink-applied error falls as the row holds more
    valid keys (the Why table: tens of percent at 1-4 keys, under a percent
    at 512-2048)."""
    c = W.index_case(12, 16, 64, 48, 4096, 2048, W.MLA_VALID_COUNTS,
                     (-2.20, 2.49), NULL, 31, "trend")
    o0, _, n = run(c, NONE)
    o2, _, _ = run(c, NULL)
    err = {}
    for cnt in W.MLA_VALID_COUNTS:
        rows = np.nonzero(n == cnt)[0]
        err[cnt] = rel_l2(o0[rows], o2[rows])
    assert err[1] > 0.2 and err[2048] < 0.02
    assert err[1] > err[16] > err[512] and err[4] > err[128] > err[2048]


def test_mla_decode_generator_shape_and_causality():
    c = W.index_case(64, 2, 8, 8, 65536, 2048, W.MLA_VALID_COUNTS,
                     (-2.20, 2.49), NULL, 1004, "shape")
    idx = c.indices
    for q in range(64):
        cnt = W.MLA_VALID_COUNTS[q % 6]
        row = idx[q]
        assert np.all(row[cnt:] == -1)
        valid = row[:cnt]
        assert np.all(np.diff(valid) > 0)                 # sorted, distinct
        assert valid.min() >= 0 and valid.max() <= 65536 - 64 + q

"""Pins of the sliding-window oracle against what the pages and mathematics fix.

Sources: vLLM pull 49815 "[Bugfix][MiMo] Apply vision attention sinks in the
window attention path" (sink on each sequence's first key; closed-form
correction p0 = exp(logit0 - lse); only the first window_size + 1 queries
reach key 0; LSE of masked scaled logits, shape (nheads, total_q); s_aux is a
different operation) and afierka-intel/vllm pull 76, Implementation (null
logit in the denominator, LSE over real keys, -inf is a no-op).
"""
import numpy as np
import pytest
from scipy.special import logsumexp

from attention_head_sinks_gb300 import workloads as W
from oracle import brute
from oracle import sa_oracle as O
from tests.oracle_pins_util import bits_to_f64, expand_kv, rel_l2, sdpa_with_bias

NONE, KEY0, NULL = W.SINK_NONE, W.SINK_KEY0_BIAS, W.SINK_NULL_LOGIT


def small_cases():
    return [
        W.tiny_window(seed=11),
        # GQA, a length-1 sequence, a sequence shorter than the window
        W.window_case([1, 5, 40, 19], 4, 2, 16, 8, (-1.0, 3.0), KEY0, 12,
                      "gqa_small"),
        # asymmetric window
        W.window_case([23, 30], 2, 1, 8, 3, (-2.0, 2.0), KEY0, 13, "asym",
                      window_right=5),
        # window 0: each token sees only itself
        W.window_case([7, 9], 2, 2, 8, 0, (-1.0, 1.0), KEY0, 14, "w0"),
    ]


def run(c, mode, sinks=None, rows=None):
    s = c.sinks if sinks is None else sinks
    return O.window_fwd(c.q, c.k, c.v, c.cu_seqlens, c.window_left,
                        c.window_right, s, mode, c.scale, rows=rows)


def seq_of(cu, T):
    seq = np.zeros(T, np.int64)
    for b in range(len(cu) - 1):
        seq[cu[b]:cu[b + 1]] = b
    return seq


def window_bias(c, mode, sinks):
    """Additive mask [Hq,T,T] written from the key-set definition."""
    T, hq = c.total_tokens, c.num_q_heads
    cu = c.cu_seqlens.astype(np.int64)
    seq = seq_of(cu, T)
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    live = (seq[:, None] == seq[None, :]) & (j - i <= c.window_right) & \
        (i - j <= c.window_left)
    bias = np.where(live, 0.0, -np.inf)[None].repeat(hq, 0)
    if mode == KEY0:
        first = cu[seq]                                   # first key per row
        for h in range(hq):
            rows = np.nonzero(live[np.arange(T), first])[0]
            bias[h, rows, first[rows]] += float(sinks[h])
    return bias


@pytest.mark.parametrize("mode", [NONE, KEY0, NULL])
@pytest.mark.parametrize("ci", range(4))
def test_brute_force_matches_set_enumeration(ci, mode):
    c = small_cases()[ci]
    o, l, _ = run(c, mode)
    ob, lb = brute.window_fwd(c.q, c.k, c.v, c.cu_seqlens, c.window_left,
                              c.window_right, c.sinks, mode, c.scale)
    assert np.allclose(o, ob, rtol=1e-12, atol=1e-12)
    assert np.allclose(l, lb, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("mode", [NONE, KEY0, NULL])
@pytest.mark.parametrize("ci", range(4))
def test_matches_torch_sdpa_with_explicit_mask(ci, mode):
    """KEY0_BIAS = SDPA with s_h added to the first-key column; NULL_LOGIT =
    SDPA with one extra zero key whose logit is s_h; GQA via repeat."""
    c = small_cases()[ci]
    o, _, _ = run(c, mode)
    qf, kf, vf = bits_to_f64(c.q), bits_to_f64(c.k), bits_to_f64(c.v)
    hq = c.num_q_heads
    ref = sdpa_with_bias(qf, expand_kv(kf, hq), expand_kv(vf, hq),
                         window_bias(c, mode, c.sinks), c.scale,
                         null_sink=c.sinks if mode == NULL else None)
    assert rel_l2(o, ref) < 1e-12


@pytest.mark.parametrize("mode", [NONE, KEY0])
def test_lse_equals_logsumexp_of_masked_scaled_logits(mode):
    c = small_cases()[1]
    _, l, _ = run(c, mode)
    qf, kf = bits_to_f64(c.q), bits_to_f64(c.k)
    bias = window_bias(c, mode, c.sinks)
    kx = expand_kv(kf, c.num_q_heads)
    for h in range(c.num_q_heads):
        logits = c.scale * qf[:, h, :] @ kx[:, h, :].T + bias[h]
        assert np.allclose(l[h], logsumexp(logits, axis=1), rtol=0, atol=1e-12)


def test_null_logit_lse_stays_over_real_keys():
    c = small_cases()[0]
    _, l0, _ = run(c, NONE)
    _, l2, _ = run(c, NULL)
    assert np.array_equal(l0, l2)


def test_key0_closed_form_correction():
    """Apply p0 = exp(logit0 - lse), out' = (out + p0 (e^s - 1) v0) /
    (1 + p0 (e^s - 1)) to a no-sink run: equals the KEY0_BIAS oracle on the
    rows that reach key 0, and those rows' LSE moves by ln(1 + p0 (e^s - 1));
    every other row is bit-identical to the no-sink run."""
    for c in small_cases():
        o_none, l_none, _ = run(c, NONE)
        o_k0, l_k0, _ = run(c, KEY0)
        qf, kf, vf = bits_to_f64(c.q), bits_to_f64(c.k), bits_to_f64(c.v)
        T, hq = c.total_tokens, c.num_q_heads
        grp = hq // c.num_kv_heads
        cu = c.cu_seqlens.astype(np.int64)
        seq = seq_of(cu, T)
        for i in range(T):
            k0 = cu[seq[i]]
            for h in range(hq):
                g = h // grp
                if i - k0 <= c.window_left:
                    logit0 = c.scale * float(qf[i, h] @ kf[k0, g])
                    p0 = np.exp(logit0 - l_none[h, i])
                    es = np.expm1(float(c.sinks[h]))
                    corr = (o_none[i, h] + p0 * es * vf[k0, g]) / (1 + p0 * es)
                    assert np.allclose(o_k0[i, h], corr, rtol=1e-10, atol=1e-12)
                    assert abs(l_k0[h, i] - (l_none[h, i] + np.log1p(p0 * es))) < 1e-10
                else:
                    assert np.array_equal(o_k0[i, h], o_none[i, h])
                    assert l_k0[h, i] == l_none[h, i]


def test_null_logit_closed_form():
    """NULL_LOGIT rescales the no-sink output by e^LSE / (e^LSE + e^s)."""
    c = small_cases()[1]
    o_none, l_none, _ = run(c, NONE)
    o_null, _, _ = run(c, NULL)
    f = 1.0 / (1.0 + np.exp(c.sinks[:, None].astype(np.float64) - l_none))  # [Hq,T]
    assert np.allclose(o_null, o_none * f.T[:, :, None], rtol=1e-12, atol=1e-14)


def test_neg_inf_null_sink_is_bitwise_no_sink():
    c = small_cases()[0]
    ninf = np.full(c.num_q_heads, -np.inf, np.float32)
    o0, l0, _ = run(c, NONE)
    o2, l2, _ = run(c, NULL, sinks=ninf)
    assert np.array_equal(o0, o2) and np.array_equal(l0, l2)


def test_zero_key0_sink_is_bitwise_no_sink():
    c = small_cases()[1]
    zero = np.zeros(c.num_q_heads, np.float32)
    o0, l0, _ = run(c, NONE)
    o1, l1, _ = run(c, KEY0, sinks=zero)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def test_neg_inf_key0_sink_removes_key0():
    """A -inf bias drops key 0 from rows that reach it; a length-1 sequence
    then has an empty key set: zero output and LSE = -inf."""
    c = small_cases()[1]            # first sequence has length 1
    ninf = np.full(c.num_q_heads, -np.inf, np.float32)
    o, l, _ = run(c, KEY0, sinks=ninf)
    assert np.all(o[0] == 0.0) and np.all(np.isneginf(l[:, 0]))
    qf, kf, vf = bits_to_f64(c.q), bits_to_f64(c.k), bits_to_f64(c.v)
    bias = window_bias(c, NONE, None)
    cu = c.cu_seqlens.astype(np.int64)
    seq = seq_of(cu, c.total_tokens)
    for i in range(c.total_tokens):
        bias[:, i, cu[seq[i]]] = -np.inf
    rows = np.arange(1, c.total_tokens)         # skip the empty row
    hq = c.num_q_heads
    ref = sdpa_with_bias(qf[rows], expand_kv(kf, hq), expand_kv(vf, hq),
                         bias[:, rows], c.scale)
    assert rel_l2(o[rows], ref) < 1e-12


def test_key_count_is_window_clipped_to_sequence():
    c = small_cases()[2]
    _, _, n = run(c, NONE)
    cu = c.cu_seqlens.astype(np.int64)
    seq = seq_of(cu, c.total_tokens)
    for i in range(c.total_tokens):
        lo = max(cu[seq[i]], i - c.window_left)
        hi = min(cu[seq[i] + 1] - 1, i + c.window_right)
        assert np.all(n[i] == hi - lo + 1)


def test_sink_changes_short_rows_and_modes_differ():
    """Dropping the sink must change the output of rows with few keys far
    beyond bf16 noise, and KEY0_BIAS is a different operation from
    NULL_LOGIT (the 's_aux' alternative)."""
    c = W.gqa_window(seed=7)
    rows = (0, 256)
    o0, _, _ = run(c, NONE, rows=rows)
    o1, _, _ = run(c, KEY0, rows=rows)
    o2, _, _ = run(c, NULL, rows=rows)
    sl = slice(*rows)
    assert rel_l2(o1[sl], o0[sl]) > 3e-2
    assert rel_l2(o2[sl], o1[sl]) > 3e-2


def test_row_sampling_matches_full_run():
    c = small_cases()[0]
    o, l, _ = run(c, KEY0)
    os_, ls, _ = run(c, KEY0, rows=(30, 70))
    assert np.array_equal(o[30:70], os_[30:70])
    assert np.array_equal(l[:, 30:70], ls[:, 30:70])
    assert np.all(np.isnan(os_[:30])) and np.all(np.isnan(ls[:, 70:]))

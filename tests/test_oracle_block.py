"""Pins of the block-sparse oracle.

KEY0_BIAS on this path adds s_h to the logit of the first key of each
token's document (vLLM pull 49815, second paragraph, with documents as the
sequences), when that key is in the token's set.

Source: NeMo AutoModel "nemo_automodel.components.models.minimax_m3_vl.
cp_sparse_attn" -- MiniMaxM3CPSparseAttention step 4 (block selection +
token-level causal), _local_sparse_forward (packed document masks, zero output
for fully masked padding rows), cp_document_ids (doc_id = cumsum(positions ==
0) - 1); afierka-intel/vllm pull 76, Implementation (null-logit sink, LSE over
real keys, -inf no-op).
"""
import numpy as np
import pytest

from attention_head_sinks_gb300 import workloads as W
from oracle import brute
from oracle import sa_oracle as O
from tests.oracle_pins_util import bits_to_f64, expand_kv, rel_l2, sdpa_with_bias

NONE, KEY0, NULL = W.SINK_NONE, W.SINK_KEY0_BIAS, W.SINK_NULL_LOGIT


def tiny(seed=41, pad_rows=0, docs=2, topk=3):
    return W.block_case(2, 40, 4, 2, 8, 8, topk, docs, (-2.2, 2.49), NULL, seed,
                        pad_rows=pad_rows, name="tiny_block")


def run(c, mode, sinks=None, table=None, cu_docs=None, rows=None):
    return O.block_sparse_fwd(
        c.q, c.k, c.v, c.batch, c.seq_len,
        c.block_table if table is None else table, c.block_size,
        c.cu_docs if cu_docs is None else cu_docs,
        c.sinks if sinks is None else sinks, mode, c.scale, rows=rows)


@pytest.mark.parametrize("mode", [NONE, KEY0, NULL])
@pytest.mark.parametrize("pad", [0, 5])
def test_brute_force_matches_set_enumeration(mode, pad):
    c = tiny(pad_rows=pad)
    tab = c.block_table.copy()
    tab[30, 1] = tab[30, 0]          # repeated block id: one selection
    tab[31, 2] = 99                  # out of range: ignored
    o, l, _ = run(c, mode, table=tab)
    ob, lb = brute.block_sparse_fwd(c.q, c.k, c.v, c.batch, c.seq_len, tab,
                                    c.block_size, c.cu_docs, c.sinks, mode,
                                    c.scale)
    assert np.allclose(o, ob, rtol=1e-12, atol=1e-12)
    assert np.allclose(l, lb, rtol=1e-12, atol=1e-12)


def positions_from_cu_docs(cu_docs, T):
    pos = np.zeros(T, np.int64)
    for e in range(len(cu_docs) - 1):
        pos[cu_docs[e]:cu_docs[e + 1]] = np.arange(cu_docs[e + 1] - cu_docs[e])
    return pos


@pytest.mark.parametrize("mode", [NONE, NULL])
def test_all_blocks_is_document_causal_sdpa(mode):
    """Selecting every block leaves causal + document masking: torch SDPA with
    a mask built from doc ids = cumsum(positions == 0) - 1 per batch row."""
    c = tiny(topk=5)                 # 40 / 8 = 5 blocks: all selectable
    S, T = c.seq_len, c.total_tokens
    tab = np.tile(np.arange(5, dtype=np.int32), (T, 1))
    o, _, _ = run(c, mode, table=tab)
    pos = positions_from_cu_docs(c.cu_docs.astype(np.int64), T).reshape(c.batch, S)
    doc = (np.cumsum(pos == 0, axis=1) - 1).reshape(-1)
    row = np.arange(T) // S
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    live = (j <= i) & (row[:, None] == row[None, :]) & (doc[:, None] == doc[None, :])
    hq = c.num_q_heads
    bias = np.where(live, 0.0, -np.inf)[None].repeat(hq, 0)
    qf, kf, vf = bits_to_f64(c.q), bits_to_f64(c.k), bits_to_f64(c.v)
    ref = sdpa_with_bias(qf, expand_kv(kf, hq), expand_kv(vf, hq), bias, c.scale,
                         null_sink=c.sinks if mode == NULL else None)
    assert rel_l2(o, ref) < 1e-12


def test_single_document_all_blocks_is_causal_attention():
    import torch
    import torch.nn.functional as F
    c = tiny(docs=1, topk=5)
    T, S = c.total_tokens, c.seq_len
    tab = np.tile(np.arange(5, dtype=np.int32), (T, 1))
    o, _, n = run(c, NONE, table=tab)
    assert np.array_equal(n, np.tile(np.arange(1, S + 1), c.batch))
    qf, kf, vf = bits_to_f64(c.q), bits_to_f64(c.k), bits_to_f64(c.v)
    hq = c.num_q_heads
    for b in range(c.batch):
        sl = slice(b * S, (b + 1) * S)
        qt = torch.from_numpy(qf[sl]).permute(1, 0, 2)[None]
        kt = torch.from_numpy(expand_kv(kf[sl], hq)).permute(1, 0, 2)[None]
        vt = torch.from_numpy(expand_kv(vf[sl], hq)).permute(1, 0, 2)[None]
        ref = F.scaled_dot_product_attention(qt, kt, vt, is_causal=True,
                                             scale=c.scale)[0].permute(1, 0, 2)
        assert rel_l2(o[sl], ref.numpy()) < 1e-12


def test_padded_rows_are_zero_with_neg_inf_lse():
    c = tiny(pad_rows=5)
    for mode in (NONE, NULL):
        o, l, n = run(c, mode)
        for b in range(c.batch):
            rows = np.arange((b + 1) * c.seq_len - 5, (b + 1) * c.seq_len)
            assert np.all(n[rows] == 0)
            assert np.all(o[rows] == 0.0) and np.all(np.isneginf(l[:, rows]))


def test_neg_inf_sink_is_bitwise_no_sink():
    c = tiny(pad_rows=3)
    ninf = np.full(c.num_q_heads, -np.inf, np.float32)
    o0, l0, _ = run(c, NONE)
    o2, l2, _ = run(c, NULL, sinks=ninf)
    assert np.array_equal(o0, o2) and np.array_equal(l0, l2)


def test_null_logit_closed_form():
    c = tiny()
    o0, l0, _ = run(c, NONE)
    o2, l2, _ = run(c, NULL)
    assert np.array_equal(l0, l2)
    f = 1.0 / (1.0 + np.exp(c.sinks[:, None].astype(np.float64) - l0))
    ok = np.isfinite(l0)
    fo = np.where(ok, f, 0.0).T[:, :, None]
    assert np.allclose(o2, o0 * fo, rtol=1e-12, atol=1e-14)


def test_future_blocks_are_cut_by_causality():
    c = tiny(docs=1)
    T = c.total_tokens
    tab = np.full((T, 3), -1, np.int32)
    tab[:, 0] = 4                    # the last block, future for most rows
    _, _, n = run(c, NONE, table=tab)
    pos = np.arange(T) % c.seq_len
    expect = np.clip(pos - 32 + 1, 0, 8)
    assert np.array_equal(n, expect)


def test_dsa_generator_table_properties():
    rng = np.random.Generator(np.random.PCG64(3))
    tab = W.random_block_table(rng, 1, 2048, 64, 16)
    for p in range(2048):
        row = tab[p]
        diag = p // 64
        valid = row[row >= 0]
        assert np.all(np.diff(valid) > 0) and valid.max() == diag
        assert len(valid) == min(16, diag + 1)
    cu = W.document_cuts(rng, 2, 8192, 3)
    assert len(cu) == 7 and cu[0] == 0 and cu[3] == 8192 and cu[-1] == 16384
    assert np.all(np.diff(cu) > 0)


def test_key0_closed_form_correction():
    """The vLLM pull 49815 correction applied to a no-sink run, with the
    document's first token as key 0: p0 = exp(logit0 - lse), out' = (out +
    p0 (e^s - 1) v0) / (1 + p0 (e^s - 1)), lse' = lse + ln(1 + p0 (e^s - 1))
    on the rows whose set holds that key; the other rows are bit-identical."""
    c = tiny(docs=3, topk=4)
    o_none, l_none, _ = run(c, NONE)
    o_k0, l_k0, _ = run(c, KEY0)
    qf, kf, vf = bits_to_f64(c.q), bits_to_f64(c.k), bits_to_f64(c.v)
    T, hq = c.total_tokens, c.num_q_heads
    grp = hq // c.num_kv_heads
    cd = c.cu_docs.astype(np.int64)
    tab = c.block_table
    nb = c.seq_len // c.block_size
    reached = 0
    for i in range(T):
        e = int(np.searchsorted(cd, i, side="right") - 1)
        k0 = int(cd[e])
        row0 = (i // c.seq_len) * c.seq_len
        b0 = (k0 - row0) // c.block_size
        in_set = k0 >= row0 and any(0 <= b < nb and b == b0 for b in tab[i])
        for h in range(hq):
            g = h // grp
            if in_set:
                logit0 = c.scale * float(qf[i, h] @ kf[k0, g])
                p0 = np.exp(logit0 - l_none[h, i])
                es = np.expm1(float(c.sinks[h]))
                corr = (o_none[i, h] + p0 * es * vf[k0, g]) / (1 + p0 * es)
                assert np.allclose(o_k0[i, h], corr, rtol=1e-10, atol=1e-12)
                assert abs(l_k0[h, i] - (l_none[h, i] + np.log1p(p0 * es))) < 1e-10
                reached += 1
            else:
                assert np.array_equal(o_k0[i, h], o_none[i, h])
                assert l_k0[h, i] == l_none[h, i] or (np.isneginf(l_k0[h, i]) and
                                                      np.isneginf(l_none[h, i]))
    assert reached > 0


def test_key0_zero_sink_is_bitwise_no_sink():
    c = tiny(docs=3, topk=4)
    o0, l0, _ = run(c, NONE)
    o1, l1, _ = run(c, KEY0, sinks=np.zeros_like(c.sinks))
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)

"""Pins of the fp8 (e4m3) latent-cache oracle (``sparse_index_fwd_fp8``).

The pages name an fp8 decode path (afierka-intel/vllm pull 76, What / Why:
``xpu_sparse_decode_fp8``) but not its format; the reading taken is e4m3
codes with one fp32 scale per latent row.  Pins: the e4m3 decoder against
torch's ``float8_e4m3fn``; the generator's encoder round-trips every code;
with power-of-two row scales the dequantised rows are exact bf16 values, so
the fp8 oracle must equal the (independent, C) bf16 oracle on those rows; the
-inf sink no-op and the single-key closed form.
"""
import numpy as np
import pytest

from attention_head_sinks_gb300 import workloads as W
from oracle import sa_oracle as O

NONE, NULL = W.SINK_NONE, W.SINK_NULL_LOGIT


def test_e4m3_decoder_matches_torch():
    torch = pytest.importorskip("torch")
    c = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(c).view(torch.float8_e4m3fn).double().numpy()
    mine = O.e4m3_to_f64(c)
    assert np.array_equal(np.isnan(ref), np.isnan(mine))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], mine[ok])


def test_encoder_round_trips_every_code():
    c = np.array([x for x in range(256) if (x & 0x7F) != 0x7F], np.uint8)
    v = O.e4m3_to_f64(c)
    back = W.f32_to_e4m3_bits(v.astype(np.float32))
    # +0 and -0 both decode to 0; every other code comes back unchanged
    assert np.array_equal(O.e4m3_to_f64(back), v)
    assert np.array_equal(back[v != 0], c[v != 0])


@pytest.mark.parametrize("mode", [NONE, NULL])
def test_pow2_scales_equal_the_bf16_oracle(mode):
    c = W.index_fp8_case(6, 4, 64, 48, 700, 40, (1, 3, 17, 40), (-2.2, 2.49), mode, 21,
                         pow2_scales=True)
    rows = O.e4m3_to_f64(c.kv) * c.kv_scale.astype(np.float64)[:, None]
    bits = W.f32_to_bf16_bits(rows.astype(np.float32))
    # the dequantised rows are exactly representable in bf16
    assert np.array_equal(O._widen(bits), rows)
    o8, l8, n8 = O.sparse_index_fwd_fp8(c.q, c.kv, c.kv_scale, c.indices, c.dv, c.sinks,
                                         mode, c.scale)
    ob, lb, nb = O.sparse_index_fwd(c.q, bits, c.indices, c.dv, c.sinks, mode, c.scale)
    np.testing.assert_allclose(o8, ob, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(l8, lb, rtol=1e-12, atol=1e-12)
    assert np.array_equal(n8, nb)


def test_neg_inf_sink_is_no_sink_and_single_key_closed_form():
    c = W.index_fp8_case(4, 3, 32, 16, 300, 8, (1, 5), (-2.2, 2.49), NULL, 22)
    ninf = np.full_like(c.sinks, -np.inf)
    o0, l0, _ = O.sparse_index_fwd_fp8(c.q, c.kv, c.kv_scale, c.indices, c.dv, c.sinks,
                                        NONE, c.scale)
    o2, l2, _ = O.sparse_index_fwd_fp8(c.q, c.kv, c.kv_scale, c.indices, c.dv, ninf,
                                        NULL, c.scale)
    assert np.array_equal(o0, o2) and np.array_equal(l0, l2)
    o1, l1, _ = O.sparse_index_fwd_fp8(c.q, c.kv, c.kv_scale, c.indices, c.dv, c.sinks,
                                        NULL, c.scale)
    # query 0 has one valid key: out = v e^l / (e^l + e^s)
    j = int(c.indices[0][c.indices[0] >= 0][0])
    v = O.e4m3_to_f64(c.kv[j]) * float(c.kv_scale[j])
    f = 1.0 / (1.0 + np.exp(c.sinks.astype(np.float64) - l1[:, 0]))
    np.testing.assert_allclose(o1[0], f[:, None] * v[None, :c.dv], rtol=1e-12)

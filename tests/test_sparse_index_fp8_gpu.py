"""Parity of the fp8 (e4m3, one fp32 scale per latent row) sparse-index CUDA
path with the oracle.

The pages name an fp8 decode path (afierka-intel/vllm pull 76, What / Why:
``xpu_sparse_decode_fp8``) but not its format; the reading taken is e4m3
codes with one fp32 scale per row, the oracle dequantising exactly in fp64.
Covers the full 64-query x 128-head decode workload over an fp8 cache with
1/4/16/128/512/2048 valid keys per query, each valid-key class on its own,
the -inf no-op, bitwise agreement with the bf16 path on power-of-two scales
(the dequantised rows are then bf16 values and the scale commutes with every
rounding), ragged and repeated lists, head counts off one 128-row block,
more than eight 256-key items per query, the longest accepted list (topk
8192), and caches that hold every non-NaN
e4m3 code (subnormals, both zeros, +-448) under row scales over 16 octaves.
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


def gpu_run(c, mode, sinks=None, indices=None):
    import torch
    import attention_head_sinks_gb300 as sa
    s = c.sinks if sinks is None else sinks
    idx = c.indices if indices is None else indices
    out, lse = sa.sa_sparse_index_fwd_fp8(dev(c.q), dev(c.kv), dev(c.kv_scale), dev(idx),
                                          c.dv, dev(s), mode, c.scale)
    torch.cuda.synchronize()
    return out, lse


def check(c, mode, sinks=None, indices=None):
    out, lse = gpu_run(c, mode, sinks, indices)
    ro, rl, _ = O.sparse_index_fwd_fp8(c.q, c.kv, c.kv_scale,
                                       c.indices if indices is None else indices, c.dv,
                                       c.sinks if sinks is None else sinks, mode, c.scale)
    rel, dl = compare(out, lse, ro, rl)
    assert rel <= REL_L2_TOL and dl <= LSE_TOL, (c.name, mode, rel, dl)
    return out, lse


@pytest.mark.parametrize("mode", [NULL, NONE])
def test_mla_sparse_decode_fp8_full(mode):
    check(W.mla_sparse_decode_fp8(mode), mode)


def test_mla_sparse_decode_fp8_per_valid_count():
    c = W.mla_sparse_decode_fp8(NULL, seed=1105)
    out, lse = gpu_run(c, NULL)
    ro, rl, n = O.sparse_index_fwd_fp8(c.q, c.kv, c.kv_scale, c.indices, c.dv, c.sinks,
                                       NULL, c.scale)
    for cnt in W.MLA_VALID_COUNTS:
        rows = np.nonzero(n == cnt)[0]
        rel, dl = compare(out, lse, ro, rl, rows=rows)
        assert rel <= REL_L2_TOL and dl <= LSE_TOL, (cnt, rel, dl)


def test_neg_inf_sink_is_bitwise_no_sink():
    import torch
    c = W.mla_sparse_decode_fp8(NULL, seed=1205)
    ninf = np.full(c.num_q_heads, -np.inf, np.float32)
    o0, l0 = gpu_run(c, NONE)
    o2, l2 = gpu_run(c, NULL, sinks=ninf)
    assert torch.equal(o0.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l0, l2)


@pytest.mark.parametrize("mode", [NULL, NONE])
def test_pow2_scales_match_the_bf16_path_bitwise(mode):
    import torch
    import attention_head_sinks_gb300 as sa
    c = W.index_fp8_case(16, 128, 576, 512, 6000, 2048, W.MLA_VALID_COUNTS, (-2.2, 2.49),
                         mode, 1305, pow2_scales=True)
    rows = O.e4m3_to_f64(c.kv) * c.kv_scale.astype(np.float64)[:, None]
    bits = W.f32_to_bf16_bits(rows.astype(np.float32))
    o8, l8 = gpu_run(c, mode)
    ob, lb = sa.sa_sparse_index_fwd(dev(c.q), dev(bits), dev(c.indices), c.dv, dev(c.sinks),
                                    mode, c.scale)
    torch.cuda.synchronize()
    assert torch.equal(o8.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(l8, lb)


def ragged_indices(rng, nq, nkv, topk, counts):
    idx = np.full((nq, topk), -1, np.int32)
    for q in range(nq):
        c = counts[q % len(counts)]
        sel = rng.choice(nkv, size=c, replace=False).astype(np.int32)
        pos = np.sort(rng.choice(topk, size=c, replace=False))
        idx[q, pos] = sel
    return idx


@pytest.mark.parametrize("hq", [128, 64, 192])
def test_ragged_lists(hq):
    rng = np.random.default_rng(50 + hq)
    counts = [0, 1, 3, 17, 255, 256, 257, 511, 600, 1000]
    c = W.index_fp8_case(10, hq, 576, 512, 5000, 1024, counts, (-2.2, 2.49), NULL,
                         3600 + hq, "ragged_idx_fp8")
    idx = ragged_indices(rng, 10, 5000, 1024, counts)
    idx[3, 7] = 5000
    idx[4, 9] = -77
    out, lse = check(c, NULL, indices=idx)
    assert (out[0] == 0).all() and bool(lse[:, 0].isneginf().all())


def test_repeated_index_counts_twice():
    c = W.index_fp8_case(4, 128, 576, 512, 700, 300, (5, 40, 260, 299), (-2.2, 2.49),
                         NULL, 3700, "dup_fp8")
    idx = c.indices.copy()
    idx[1, 40] = idx[1, 0]
    idx[2, 270] = idx[2, 3]
    check(c, NULL, indices=idx)


@pytest.mark.parametrize("topk", [1, 16, 200, 257, 513])
def test_list_lengths(topk):
    c = W.index_fp8_case(6, 128, 576, 512, 3000, topk, (topk, 1, topk // 2 + 1),
                         (-2.2, 2.49), NULL, 3800 + topk, "len_fp8")
    check(c, NULL)


def test_all_lists_full():
    # 64 queries x 2048 valid keys: 512 full items, several waves of CTAs
    c = W.index_fp8_case(64, 128, 576, 512, 65536, 2048, (2048,), (-2.2, 2.49), NULL, 3950,
                         "all_full_fp8")
    check(c, NULL)


def test_more_than_eight_items():
    c = W.index_fp8_case(4, 40, 576, 512, 9000, 3000, (2900, 300, 2100, 7), (-2.2, 2.49),
                         NULL, 3900, "many_items_fp8")
    check(c, NULL)


def test_maximum_topk():
    # topk 8192, the longest accepted list: 32 items for the full list
    c = W.index_fp8_case(3, 128, 576, 512, 20000, 8192, (8192, 5, 8000), (-2.2, 2.49),
                         NULL, 3901, "max_topk_fp8")
    check(c, NULL)


@pytest.mark.parametrize("mode", [NULL, NONE])
def test_every_e4m3_code(mode):
    # latent rows cycle through all 254 non-NaN codes (subnormals, both
    # zeros, +-448) in shifted orders, with row scales from 2^-12 to 2^4 times
    # 1/448 (so values stay O(1)): every code reaches the MMAs and the scale
    # folding through the kernel's own conversion
    rng = np.random.default_rng(77)
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    nkv, dqk = 1024, 576
    kv = np.stack([np.roll(np.resize(codes, dqk), 7 * r) for r in range(nkv)]).astype(np.uint8)
    kv_scale = (2.0 ** rng.integers(-12, 5, size=nkv) / 448.0).astype(np.float32)
    base = W.index_fp8_case(8, 128, 576, 512, nkv, 300, (1, 5, 40, 256, 300, 17, 3, 128),
                            (-2.2, 2.49), mode, 4100)
    c = W.IndexFp8Case("all_codes", base.q, kv, kv_scale, base.indices, 512, base.sinks, mode,
                       base.scale)
    check(c, mode)

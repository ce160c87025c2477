"""Key-set exactness through the product path, for every key-set kind.

With q = 0 every logit is 0, so a row's softmax is uniform over its key set
K(i): the kernel's row sum is |K(i)| exactly (sums of ones in fp32), its LSE
is ln |K(i)| (the NULL_LOGIT sink stays out of the LSE, and a zero KEY0_BIAS
sink adds nothing), and its output is the mean of V over K(i), scaled by
|K| / (|K| + e^s) under NULL_LOGIT.  Two checks on every row and head:

* rint(exp(LSE)) equals the oracle's key count exactly (0 for an empty set,
  whose LSE is -inf);
* the output agrees with the oracle within one bf16 step (ulp) of the row's
  largest element: the bf16 paths round once (the output), within half a
  step; the fp8 path rounds P after the row scale is folded in, so it gets
  two steps.  A key taken or missed moves some element of the mean by about
  |v_j - v_j'| / |K|, several steps even for the 2048-key rows.

The oracle's counts are pinned on the CPU (brute-force masks, window
clipping, listed-index counting).
"""
import numpy as np
import pytest

from attention_head_sinks_gb300 import workloads as W
from oracle import sa_oracle as O
from tests.gpu_util import dev

pytestmark = pytest.mark.gpu

NONE, KEY0, NULL = W.SINK_NONE, W.SINK_KEY0_BIAS, W.SINK_NULL_LOGIT


@pytest.fixture(autouse=True)
def _no_device_errors():
    import attention_head_sinks_gb300 as sa
    yield
    assert sa.sa_device_error() == 0


def counts_from_lse(lse):
    """rint(exp(LSE)) per [head, row]; -inf gives 0."""
    l = lse.cpu().numpy().astype(np.float64)
    c = np.exp(l)
    n = np.rint(c)
    # the count must come out near an integer (a fractional weight would not)
    assert np.all(np.abs(c - n) <= 1e-4 * np.maximum(n, 1))
    return n.astype(np.int64)


def check_rows(out, ref, steps=1):
    """Per (row, head): max |out - ref| within ``steps`` bf16 ulps of the
    row's largest |ref| element (ulp(x) = 2^(floor(log2 x) - 7))."""
    o = out.float().cpu().numpy().astype(np.float64)
    r = ref
    err = np.abs(o - r).max(axis=-1)
    rmax = np.abs(r).max(axis=-1)
    ulp = np.where(rmax > 0, 2.0 ** (np.floor(np.log2(np.where(rmax > 0, rmax, 1.0))) - 7), 0.0)
    tol = steps * ulp + 1e-7
    bad = np.argwhere(err > tol)
    assert bad.size == 0, (bad[:5], err[tuple(bad[0])], tol[tuple(bad[0])])


def zero_q(c):
    return np.zeros_like(c.q)


def sinks_for(c, mode):
    return np.zeros_like(c.sinks) if mode == KEY0 else c.sinks


# ---------------------------------------------------------------------------
# sliding window
# ---------------------------------------------------------------------------
WINDOW = [
    ("tiny", lambda: W.tiny_window(NONE)),
    ("ragged", lambda: W.window_case([300, 1, 77, 129, 1000, 5], 4, 4, 80, 64, (-1, 3),
                                     NONE, 2400, "kc_ragged")),
    ("gqa_asym", lambda: W.window_case([1, 1, 2, 63, 64, 65, 500], 8, 2, 80, 64, (-1, 3),
                                       NONE, 2401, "kc_asym", window_right=5)),
    ("d128_spill", lambda: W.window_case([6000, 1, 6799], 24, 12, 128, 64, (-1, 3), NONE,
                                         2402, "kc_spill")),
    ("vision16k", lambda: W.vision_window(16384, NONE)),
    ("gqa16k", lambda: W.gqa_window(NONE)),
]


@pytest.mark.parametrize("mode", [NONE, KEY0, NULL])
@pytest.mark.parametrize("wi", range(len(WINDOW)))
def test_window_key_sets(wi, mode):
    import torch
    import attention_head_sinks_gb300 as sa
    c = WINDOW[wi][1]()
    q = zero_q(c)
    s = sinks_for(c, mode)
    out, lse = sa.sa_varlen_window_fwd(dev(q), dev(c.k), dev(c.v), dev(c.cu_seqlens),
                                       c.window_left, c.window_right, dev(s), mode, c.scale)
    torch.cuda.synchronize()
    ro, _, cnt = O.window_fwd(q, c.k, c.v, c.cu_seqlens, c.window_left, c.window_right, s,
                              mode, c.scale)
    assert np.array_equal(counts_from_lse(lse), cnt.T)
    check_rows(out, ro)


# ---------------------------------------------------------------------------
# top-k index lists into the latent cache (bf16 and fp8)
# ---------------------------------------------------------------------------
def ragged_index_case():
    rng = np.random.default_rng(2410)
    counts = [0, 1, 3, 17, 255, 256, 257, 511, 600, 1000]
    c = W.index_case(10, 128, 576, 512, 5000, 1024, counts, (-2.2, 2.49), NULL, 2411,
                     "kc_ragged_idx")
    idx = np.full((10, 1024), -1, np.int32)
    for qi, n in enumerate(counts):
        sel = rng.choice(5000, size=n, replace=False).astype(np.int32)
        idx[qi, np.sort(rng.choice(1024, size=n, replace=False))] = sel
    idx[3, 7] = 5000          # out of range: masked
    idx[4, 9] = -77           # negative: masked
    idx[5, np.nonzero(idx[5] < 0)[0][0]] = idx[5, np.nonzero(idx[5] >= 0)[0][0]]  # counts twice
    c.indices = idx
    return c


INDEX = [
    ("mla_decode", lambda: W.mla_sparse_decode(NULL)),
    ("ragged", ragged_index_case),
]


@pytest.mark.parametrize("mode", [NONE, NULL])
@pytest.mark.parametrize("ii", range(len(INDEX)))
def test_index_key_sets(ii, mode):
    import torch
    import attention_head_sinks_gb300 as sa
    c = INDEX[ii][1]()
    q = zero_q(c)
    out, lse = sa.sa_sparse_index_fwd(dev(q), dev(c.kv), dev(c.indices), c.dv, dev(c.sinks),
                                      mode, c.scale)
    torch.cuda.synchronize()
    ro, _, cnt = O.sparse_index_fwd(q, c.kv, c.indices, c.dv, c.sinks, mode, c.scale)
    got = counts_from_lse(lse)
    assert np.array_equal(got, np.broadcast_to(cnt[None, :], got.shape))
    check_rows(out, ro)


@pytest.mark.parametrize("mode", [NONE, NULL])
def test_index_fp8_key_sets(mode):
    import torch
    import attention_head_sinks_gb300 as sa
    c = W.mla_sparse_decode_fp8(NULL, seed=2420)
    q = zero_q(c)
    out, lse = sa.sa_sparse_index_fwd_fp8(dev(q), dev(c.kv), dev(c.kv_scale), dev(c.indices),
                                          c.dv, dev(c.sinks), mode, c.scale)
    torch.cuda.synchronize()
    ro, _, cnt = O.sparse_index_fwd_fp8(q, c.kv, c.kv_scale, c.indices, c.dv, c.sinks, mode,
                                        c.scale)
    got = counts_from_lse(lse)
    assert np.array_equal(got, np.broadcast_to(cnt[None, :], got.shape))
    check_rows(out, ro, steps=2)


# ---------------------------------------------------------------------------
# selected key blocks with causal and document masks
# ---------------------------------------------------------------------------
BLOCK = [
    ("dsa_padded", lambda: W.dsa_block_prefill(NULL, pad_rows=64)),
    ("small_docs", lambda: W.block_case(3, 384, 16, 2, 128, 64, 3, 4, (-2.2, 2.49), NULL,
                                        2430, name="kc_small")),
]


@pytest.mark.parametrize("mode", [NONE, KEY0, NULL])
@pytest.mark.parametrize("bi", range(len(BLOCK)))
def test_block_key_sets(bi, mode):
    import torch
    import attention_head_sinks_gb300 as sa
    c = BLOCK[bi][1]()
    q = zero_q(c)
    s = sinks_for(c, mode)
    out, lse = sa.sa_block_sparse_fwd(dev(q), dev(c.k), dev(c.v), c.batch, c.seq_len,
                                      dev(c.block_table), c.block_size, dev(c.cu_docs), dev(s),
                                      mode, c.scale)
    torch.cuda.synchronize()
    ro, _, cnt = O.block_sparse_fwd(q, c.k, c.v, c.batch, c.seq_len, c.block_table,
                                    c.block_size, c.cu_docs, s, mode, c.scale)
    got = counts_from_lse(lse)
    assert np.array_equal(got, np.broadcast_to(cnt[None, :], got.shape))
    check_rows(out, ro)


def test_block_index_head_key_sets():
    import torch
    import attention_head_sinks_gb300 as sa
    c = W.block_case(2, 512, 16, 4, 128, 64, 5, 3, (-2.2, 2.49), NULL, 2440,
                     name="kc_index_heads")
    rng = np.random.default_rng(2441)
    tabs = np.stack([W.random_block_table(rng, 2, 512, 64, 5) for _ in range(2)])
    q = zero_q(c)
    out, lse = sa.sa_block_sparse_fwd_index_heads(dev(q), dev(c.k), dev(c.v), 2, 512,
                                                  dev(tabs), 64, dev(c.cu_docs), dev(c.sinks),
                                                  NULL, c.scale)
    torch.cuda.synchronize()
    ro, _, cnt = O.block_sparse_fwd_index_heads(q, c.k, c.v, 2, 512, tabs, 64, c.cu_docs,
                                                c.sinks, NULL, c.scale)
    got = counts_from_lse(lse)
    per_head = np.repeat(cnt, 16 // 2, axis=0)   # head h uses table h // (Hq / Hi)
    assert np.array_equal(got, per_head)
    check_rows(out, ro)

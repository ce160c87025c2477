"""Seeded synthetic inputs for sink-aware varlen attention.

This module only draws inputs: random bf16 tensors, packed sequence lengths,
per-head sinks, top-k index lists and block-selection tables.  It holds none of
the attention arithmetic, so both the CUDA path and the CPU oracle can take
their inputs from it.  Everything is NumPy with an explicit PCG64 seed and
integer-exact bf16 rounding, so the same seed gives the same bits on every
host.

bf16 tensors are returned as ``uint16`` bit patterns; ``to_torch`` views them
as ``torch.bfloat16`` without a copy.

Workload shapes follow the pages:
* window attention of a vision tower: head dim 80, window 64, 16 heads,
  4096 / 16384 packed tokens, sinks in [-0.10, 0.59] (vLLM pull 49815,
  "[Bugfix][MiMo] Apply vision attention sinks in the window attention path",
  real-weights and Cost paragraphs);
* sparse MLA decode with sinks in [-2.20, 2.49] and 1 ... 2048 valid keys per
  row (afierka-intel/vllm pull 76, Why);
* DSA block-sparse prefill with document-packed rows (NeMo AutoModel
  "minimax_m3_vl.cp_sparse_attn", MiniMaxM3CPSparseAttention);
* two partial results (output, LSE) to merge, shaped like the window block.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

from ._lib import SINK_KEY0_BIAS, SINK_NONE, SINK_NULL_LOGIT  # noqa: F401


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(int(seed)))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even) with integer ops only."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    rounded = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_normal(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) samples rounded to bf16, as uint16 bit patterns."""
    return f32_to_bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


def to_torch(bits: np.ndarray):
    """View uint16 bf16 bits as a CPU ``torch.bfloat16`` tensor (no copy)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
        torch.bfloat16)


def uniform_sinks(rng, hq, lo, hi) -> np.ndarray:
    return rng.uniform(lo, hi, size=hq).astype(np.float32)


# --------------------------------------------------------------------------
# sliding window over cu_seqlens-packed sequences
# --------------------------------------------------------------------------
@dataclasses.dataclass
class WindowCase:
    name: str
    q: np.ndarray            # uint16 [T, Hq, D]
    k: np.ndarray            # uint16 [T, Hkv, D]
    v: np.ndarray            # uint16 [T, Hkv, D]
    cu_seqlens: np.ndarray   # int32 [B+1]
    window_left: int
    window_right: int
    sinks: np.ndarray        # float32 [Hq]
    mode: int
    scale: float             # an fp32 value

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def num_q_heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def num_kv_heads(self) -> int:
        return int(self.k.shape[1])

    @property
    def head_dim(self) -> int:
        return int(self.q.shape[2])


def window_case(lengths, hq, hkv, d, window, sink_range, mode, seed,
                name="window", window_right=None) -> WindowCase:
    rng = _rng(seed)
    lengths = [int(x) for x in lengths]
    cu = np.zeros(len(lengths) + 1, np.int32)
    cu[1:] = np.cumsum(lengths)
    T = int(cu[-1])
    q = bf16_normal(rng, (T, hq, d))
    k = bf16_normal(rng, (T, hkv, d))
    v = bf16_normal(rng, (T, hkv, d))
    sinks = uniform_sinks(rng, hq, *sink_range)
    wr = window if window_right is None else window_right
    return WindowCase(name, q, k, v, cu, int(window), int(wr), sinks, mode,
                      float(np.float32(1.0 / math.sqrt(d))))


def tiny_window(mode=SINK_KEY0_BIAS, seed=1001) -> WindowCase:
    """Two sequences of 37 and 91 tokens, 4 MHA heads, head dim 80, window 64,
    sinks U[-0.10, 0.59]."""
    return window_case([37, 91], 4, 4, 80, 64, (-0.10, 0.59), mode, seed,
                       "tiny_window_128tok")


def vision_window(tokens=16384, mode=SINK_KEY0_BIAS, seed=1002) -> WindowCase:
    """Vision-tower window block: 16 MHA heads, head dim 80, window 64, sinks
    U[-0.10, 0.59]; 4096 tokens as 1536 + 2560, or 16384 as 4 x 4096."""
    if tokens == 4096:
        lengths = [1536, 2560]
    elif tokens == 16384:
        lengths = [4096] * 4
    else:
        raise ValueError("vision_window: tokens must be 4096 or 16384")
    return window_case(lengths, 16, 16, 80, 64, (-0.10, 0.59), mode, seed,
                       "vision_window_%dtok" % tokens)


def gqa_lengths(rng, total=16384, nseq=8, lo=32, hi=4096, short=(32, 63)):
    """``nseq`` lengths summing to ``total``: one shorter than the window,
    the rest uniform in [lo, hi], the last one forced by the sum and
    redrawn until it lies in [lo, hi]; the order is shuffled."""
    first = int(rng.integers(short[0], short[1] + 1))
    while True:
        mid = rng.integers(lo, hi + 1, size=nseq - 2)
        last = total - first - int(mid.sum())
        if lo <= last <= hi:
            break
    lengths = np.array([first] + [int(x) for x in mid] + [last], np.int64)
    rng.shuffle(lengths)
    return [int(x) for x in lengths]


def gqa_window(mode=SINK_KEY0_BIAS, seed=1003) -> WindowCase:
    """16384 tokens in 8 seeded sequences (one shorter than the window),
    16 query / 4 KV heads, head dim 80, window 64, sinks U[-1.0, 3.0]."""
    lengths = gqa_lengths(_rng(seed + 500000))
    return window_case(lengths, 16, 4, 80, 64, (-1.0, 3.0), mode, seed,
                       "gqa_window_16384tok")


# --------------------------------------------------------------------------
# top-k index list into a shared latent KV cache (MLA decode)
# --------------------------------------------------------------------------
@dataclasses.dataclass
class IndexCase:
    name: str
    q: np.ndarray          # uint16 [Nq, Hq, dqk]
    kv: np.ndarray         # uint16 [nkv, dqk]
    indices: np.ndarray    # int32 [Nq, topk], -1 padded
    dv: int
    sinks: np.ndarray      # float32 [Hq]
    mode: int
    scale: float

    @property
    def num_queries(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_q_heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def dqk(self) -> int:
        return int(self.q.shape[2])

    @property
    def num_kv(self) -> int:
        return int(self.kv.shape[0])

    @property
    def topk(self) -> int:
        return int(self.indices.shape[1])


def causal_topk_indices(rng, nq, nkv, topk, counts):
    """Per decode query q (position nkv - nq + q): ``counts[q % len]`` key
    positions drawn without replacement from its causal prefix [0, pos],
    sorted ascending, padded with -1 to ``topk``."""
    idx = np.full((nq, topk), -1, np.int32)
    for qi in range(nq):
        pos = nkv - nq + qi
        c = min(int(counts[qi % len(counts)]), topk, pos + 1)
        sel = np.sort(rng.choice(pos + 1, size=c, replace=False))
        idx[qi, :c] = sel
    return idx


def index_case(nq, hq, dqk, dv, nkv, topk, counts, sink_range, mode, seed,
               name="sparse_index", indices=None) -> IndexCase:
    rng = _rng(seed)
    q = bf16_normal(rng, (nq, hq, dqk))
    kv = bf16_normal(rng, (nkv, dqk))
    sinks = uniform_sinks(rng, hq, *sink_range)
    if indices is None:
        indices = causal_topk_indices(rng, nq, nkv, topk, counts)
    return IndexCase(name, q, kv, np.ascontiguousarray(indices, np.int32), dv,
                     sinks, mode, float(np.float32(1.0 / math.sqrt(dqk))))


MLA_VALID_COUNTS = (1, 4, 16, 128, 512, 2048)


def mla_sparse_decode(mode=SINK_NULL_LOGIT, seed=1004, num_kv=65536) -> IndexCase:
    """64 decode queries x 128 heads, qk dim 576 (512 latent + 64 rope), v dim
    512, one shared latent cache of 65536 tokens, top-2048 causal indices with
    1/4/16/128/512/2048 valid entries cycled over queries, sinks
    U[-2.20, 2.49]."""
    return index_case(64, 128, 576, 512, num_kv, 2048, MLA_VALID_COUNTS,
                      (-2.20, 2.49), mode, seed, "mla_sparse_decode_64q")


# --------------------------------------------------------------------------
# block-sparse causal prefill with packed documents (DSA style)
# --------------------------------------------------------------------------
@dataclasses.dataclass
class BlockCase:
    name: str
    q: np.ndarray            # uint16 [B*S, Hq, D]
    k: np.ndarray            # uint16 [B*S, Hkv, D]
    v: np.ndarray            # uint16 [B*S, Hkv, D]
    batch: int
    seq_len: int
    block_table: np.ndarray  # int32 [B*S, topk], -1 padded
    block_size: int
    cu_docs: np.ndarray      # int32 [num_docs+1]
    sinks: np.ndarray        # float32 [Hq]
    mode: int
    scale: float

    @property
    def total_tokens(self) -> int:
        return self.batch * self.seq_len

    @property
    def num_q_heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def num_kv_heads(self) -> int:
        return int(self.k.shape[1])

    @property
    def head_dim(self) -> int:
        return int(self.q.shape[2])

    @property
    def topk_blocks(self) -> int:
        return int(self.block_table.shape[1])


def document_cuts(rng, batch, seq_len, docs_per_row):
    """cu_docs over the flattened [batch, seq_len] tokens: each row is cut at
    ``docs_per_row - 1`` distinct seeded positions in [1, seq_len - 1]."""
    starts = [0]
    for b in range(batch):
        ncut = min(docs_per_row - 1, max(seq_len - 1, 0))
        cuts = np.sort(rng.choice(np.arange(1, seq_len), size=ncut,
                                  replace=False)) if ncut > 0 else []
        starts += [b * seq_len + int(c) for c in cuts]
        starts.append((b + 1) * seq_len)
    return np.array(starts, np.int32)


def random_block_table(rng, batch, seq_len, block_size, topk):
    """Per token at row position p: its causal blocks 0 .. p // block_size;
    all of them when they number <= topk, else the diagonal block plus the
    top-(topk-1) earlier blocks by an i.i.d. U(0,1) fp32 score (ties to the
    lower id); ascending, -1 padded."""
    nblocks = -(-seq_len // block_size)
    T = batch * seq_len
    table = np.full((T, topk), -1, np.int32)
    pos = np.arange(T) % seq_len
    diag = pos // block_size
    scores = rng.random((T, nblocks), dtype=np.float32)
    blk = np.arange(nblocks)[None, :]
    # earlier (non-diagonal) causal blocks compete on score
    masked = np.where(blk < diag[:, None], scores, np.float32(-1.0))
    order = np.argsort(-masked, axis=1, kind="stable")[:, :max(topk - 1, 0)]
    for i in range(T):
        if diag[i] + 1 <= topk:
            table[i, :diag[i] + 1] = np.arange(diag[i] + 1)
        else:
            sel = np.sort(np.append(order[i], diag[i]))
            table[i, :] = sel
    return table


def block_case(batch, seq_len, hq, hkv, d, block_size, topk, docs_per_row,
               sink_range, mode, seed, pad_rows=0, name="block_sparse",
               sinks_neg_inf=False) -> BlockCase:
    rng = _rng(seed)
    T = batch * seq_len
    q = bf16_normal(rng, (T, hq, d))
    k = bf16_normal(rng, (T, hkv, d))
    v = bf16_normal(rng, (T, hkv, d))
    sinks = uniform_sinks(rng, hq, *sink_range)
    if sinks_neg_inf:
        sinks = np.full(hq, -np.inf, np.float32)
    cu_docs = document_cuts(rng, batch, seq_len, docs_per_row)
    table = random_block_table(rng, batch, seq_len, block_size, topk)
    if pad_rows:
        for b in range(batch):
            table[(b + 1) * seq_len - pad_rows:(b + 1) * seq_len] = -1
    return BlockCase(name, q, k, v, batch, seq_len, table, block_size, cu_docs,
                     sinks, mode, float(np.float32(1.0 / math.sqrt(d))))


def dsa_block_prefill(mode=SINK_NULL_LOGIT, seed=1005, pad_rows=0,
                      sinks_neg_inf=False) -> BlockCase:
    """Batch 2 x 8192 tokens, 3 documents per row, 32 query / 4 KV heads,
    head dim 128, key block 64, top-16 blocks per query row, sinks
    U[-2.2, 2.49] (or all -inf)."""
    tag = "dsa_block_prefill_2x8192" + ("_padrows" if pad_rows else "") + \
        ("_neginf" if sinks_neg_inf else "")
    return block_case(2, 8192, 32, 4, 128, 64, 16, 3, (-2.2, 2.49), mode,
                      seed, pad_rows=pad_rows, name=tag,
                      sinks_neg_inf=sinks_neg_inf)


# --------------------------------------------------------------------------
# indexer inputs for on-device block selection
# --------------------------------------------------------------------------
@dataclasses.dataclass
class SelectCase:
    name: str
    index_q: np.ndarray   # uint16 bf16 [B*S, Hi, Di]
    index_k: np.ndarray   # uint16 bf16 [B*S, Di]
    batch: int
    seq_len: int
    block_size: int
    topk: int

    @property
    def num_index_heads(self) -> int:
        return int(self.index_q.shape[1])

    @property
    def index_dim(self) -> int:
        return int(self.index_q.shape[2])


def select_case(batch, seq_len, hi, di, block_size, topk, seed,
                name="block_select") -> SelectCase:
    """Index queries [B*S, Hi, Di] and index keys [B*S, Di] ~ N(0,1) bf16."""
    rng = _rng(seed)
    T = batch * seq_len
    return SelectCase(name, bf16_normal(rng, (T, hi, di)), bf16_normal(rng, (T, di)),
                      batch, seq_len, block_size, topk)


def dsa_block_select(seed=1008) -> SelectCase:
    """Indexer inputs of the DSA prefill batch: 2 x 8192 tokens, 4 index
    heads of dim 128, key block 64, top-16 blocks per (index head, token)."""
    return select_case(2, 8192, 4, 128, 64, 16, seed, "dsa_block_select_2x8192")


# --------------------------------------------------------------------------
# two partial attention results to merge (cascade over two key sets)
# --------------------------------------------------------------------------
@dataclasses.dataclass
class MergeCase:
    name: str
    out_a: np.ndarray   # uint16 bf16 [T, H, D]
    lse_a: np.ndarray   # float32 [H, T]
    out_b: np.ndarray
    lse_b: np.ndarray
    sinks: np.ndarray   # float32 [H]
    mode: int


def merge_case(tokens, heads, dim, seed, lse_range=(-4.0, 6.0), empty_frac=0.05,
               sink_range=(-2.2, 2.49), mode=SINK_NULL_LOGIT, name="merge") -> MergeCase:
    """Two partials of ``tokens x heads`` rows of ``dim``: outputs N(0,1)
    bf16, LSEs U[lse_range] with ``empty_frac`` of each set to -inf (a key
    set with no keys; some rows get both), sinks U[sink_range]."""
    rng = _rng(seed)
    out_a = bf16_normal(rng, (tokens, heads, dim))
    out_b = bf16_normal(rng, (tokens, heads, dim))
    lse_a = rng.uniform(*lse_range, size=(heads, tokens)).astype(np.float32)
    lse_b = rng.uniform(*lse_range, size=(heads, tokens)).astype(np.float32)
    lse_a[rng.random((heads, tokens)) < empty_frac] = -np.inf
    lse_b[rng.random((heads, tokens)) < empty_frac] = -np.inf
    sinks = uniform_sinks(rng, heads, *sink_range)
    return MergeCase(name, out_a, lse_a, out_b, lse_b, sinks, mode)


def merge_window_partials(mode=SINK_NULL_LOGIT, seed=1006) -> MergeCase:
    """The two partials of a cascade over the vision window block's shape:
    16384 tokens x 16 heads x head dim 80."""
    return merge_case(16384, 16, 80, seed, empty_frac=0.0, mode=mode,
                      name="merge_window_16384tok")


# --------------------------------------------------------------------------
# fp8 (e4m3) latent cache for the MLA decode
# --------------------------------------------------------------------------
def _e4m3_table():
    """Positive e4m3 codes 0..126 (0x7F is NaN) and their values, ascending."""
    codes = np.arange(127, dtype=np.int64)
    e, m = codes >> 3, codes & 7
    vals = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7))
    return codes, vals


def f32_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Nearest e4m3 code (ties to the even code), saturating at +-448."""
    codes, vals = _e4m3_table()
    a = np.minimum(np.abs(np.asarray(x, np.float64)), 448.0)
    i = np.clip(np.searchsorted(vals, a), 1, len(vals) - 1)
    lo, hi = vals[i - 1], vals[i]
    up = (a - lo > hi - a) | ((a - lo == hi - a) & (codes[i] % 2 == 0))
    c = np.where(up, codes[i], codes[i - 1])
    return (c | np.where(np.signbit(np.asarray(x)), 0x80, 0)).astype(np.uint8)


@dataclasses.dataclass
class IndexFp8Case:
    name: str
    q: np.ndarray          # uint16 bf16 [Nq, Hq, dqk]
    kv: np.ndarray         # uint8 e4m3 codes [nkv, dqk]
    kv_scale: np.ndarray   # float32 [nkv]: row value = code value x scale
    indices: np.ndarray    # int32 [Nq, topk], -1 padded
    dv: int
    sinks: np.ndarray
    mode: int
    scale: float

    @property
    def num_queries(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_q_heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def num_kv(self) -> int:
        return int(self.kv.shape[0])

    @property
    def dqk(self) -> int:
        return int(self.q.shape[2])

    @property
    def topk(self) -> int:
        return int(self.indices.shape[1])


def index_fp8_case(nq, hq, dqk, dv, nkv, topk, counts, sink_range, mode, seed,
                   name="sparse_index_fp8", pow2_scales=False) -> IndexFp8Case:
    """Latent rows N(0,1) quantised per row to e4m3 with scale amax / 448
    (rounded to a power of two with ``pow2_scales``)."""
    rng = _rng(seed)
    q = bf16_normal(rng, (nq, hq, dqk))
    rows = rng.standard_normal(size=(nkv, dqk), dtype=np.float32)
    sinks = uniform_sinks(rng, hq, *sink_range)
    indices = causal_topk_indices(rng, nq, nkv, topk, counts)
    amax = np.abs(rows).max(axis=1).astype(np.float64)
    scale = amax / 448.0
    if pow2_scales:
        scale = 2.0 ** np.round(np.log2(scale))
    scale = scale.astype(np.float32)
    kv = f32_to_e4m3_bits(rows / scale[:, None].astype(np.float64))
    return IndexFp8Case(name, q, kv, scale, np.ascontiguousarray(indices, np.int32), dv,
                        sinks, mode, float(np.float32(1.0 / math.sqrt(dqk))))


def mla_sparse_decode_fp8(mode=SINK_NULL_LOGIT, seed=1007, num_kv=65536) -> IndexFp8Case:
    """The MLA decode batch over an e4m3 latent cache with one fp32 scale per
    row: 64 queries x 128 heads, qk dim 576, v dim 512, 65536 rows, top-2048
    with 1/4/16/128/512/2048 valid entries cycled, sinks U[-2.20, 2.49]."""
    return index_fp8_case(64, 128, 576, 512, num_kv, 2048, MLA_VALID_COUNTS,
                          (-2.20, 2.49), mode, seed, "mla_sparse_decode_fp8_64q")

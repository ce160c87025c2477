// window_common.cuh -- per-row pieces of the sliding-window forward shared by
// both window kernels: row metadata from cu_seqlens, the KEY0_BIAS sink added
// to S in tensor memory, the two-pass softmax over S (P written back as
// bf16), and the epilogue with the NULL_LOGIT fold.
//
// Operation: vLLM pull 49815 "[Bugfix][MiMo] Apply vision attention sinks in
// the window attention path" (KEY0_BIAS on each sequence's first key, which
// only the first window_size + 1 queries reach; LSE of the masked scaled
// logits); NULL_LOGIT per afierka-intel/vllm pull 76, Implementation.
#pragma once

#include <cuda_bf16.h>
#include <math.h>

#include "sa_internal.h"
#include "sa_ptx.cuh"

namespace sa {
namespace win {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Blackwell packed fp32 pair arithmetic (each lane rounded as the scalar
// instruction) and the three-input maximum.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f2_hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Largest b with cu[b] <= t (0 <= b < n), i.e. the sequence holding token t.
__device__ __forceinline__ int find_seq(const int32_t* cu, int n, int t) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct RowMeta {
  int clo, chi;  // live key columns [clo, chi] of the S tile
  int ck0;       // column of the sequence's first key when it gets the sink
  int t, h;      // token and query head of this row
  bool valid;    // t < total_tokens
  float sink2;   // sink in log2 units
};

// Row `row` of a tile of (128 / G) tokens from tok0 x the G query heads of KV
// head g; column 0 of S holds key token kstart.  Rows past the last token
// get a live range no column reaches.
template <int G, int MODE>
__device__ __forceinline__ RowMeta row_meta(const int32_t* cu, int num_seqs,
                                            int total_tokens, int row, int g,
                                            int tok0, int kstart, int wl, int wr,
                                            const float* sinks) {
  RowMeta r;
  r.t = tok0 + row / G;
  r.h = g * G + (row % G);
  r.valid = r.t < total_tokens;
  r.clo = 1 << 30;
  r.chi = 1 << 30;
  r.ck0 = -1;
  if (r.valid) {
    const int b = find_seq(cu, num_seqs, r.t);
    const int s0 = __ldg(cu + b);
    const int s1 = __ldg(cu + b + 1);
    const int lo = max(s0, r.t - wl);
    const int hi = min(s1 - 1, r.t + wr);
    r.clo = lo - kstart;
    r.chi = hi - kstart;
    if (MODE == SA_SINK_KEY0_BIAS && s0 >= lo) r.ck0 = s0 - kstart;
  }
  r.sink2 = (MODE != SA_SINK_NONE) ? __ldg(sinks + r.h) * kLog2e : 0.f;
  return r;
}

// Softmax pieces over the 32-column chunks of S at s_addr (this warp's TMEM
// lane base + column).  Only chunks some row of the warp can see are read;
// chunk c of P (bf16 pairs) is written at p_addr + 16 c, in place over S
// chunks that have already been read.  Tensor-memory loads are
// double-buffered: chunk c + 1 is requested before chunk c is processed.
// The softmax itself has no sink term: a KEY0_BIAS sink is already in S
// (key0_bias_in_tmem), a NULL_LOGIT one enters in finalize_row.

__device__ __forceinline__ void max_one(const float (&s)[32], int c, const RowMeta& r,
                                        uint32_t span, float (&mr)[4]) {
  const int c0 = 32 * c;
  const bool full = __all_sync(0xffffffffu, c0 >= r.clo && c0 + 31 <= r.chi);
  if (full) {
#pragma unroll
    for (int e = 0; e < 32; e += 2) mr[(e >> 1) & 3] = max3f(mr[(e >> 1) & 3], s[e], s[e + 1]);
  } else {
#pragma unroll
    for (int e = 0; e < 32; e += 2)
      mr[(e >> 1) & 3] =
          max3f(mr[(e >> 1) & 3], ((uint32_t)(c0 + e - r.clo) <= span) ? s[e] : -INFINITY,
                ((uint32_t)(c0 + e + 1 - r.clo) <= span) ? s[e + 1] : -INFINITY);
  }
}

// P = 2^(x - m_use) as bf16 for one chunk (in registers s, stored to
// p_addr + 16 c); adds the chunk's values to the partial pair sums lp.  The
// exponent is fma(s, c2, -m) in both branches (pairs by the packed fma, each
// lane rounded as the scalar one) and both accumulate in the same order.
__device__ __forceinline__ void exp_one(float (&s)[32], int c, const RowMeta& r, float c2,
                                        float m_use, uint32_t span, uint64_t (&lp)[4],
                                        uint32_t p_addr) {
  const int c0 = 32 * c;
  const bool full = __all_sync(0xffffffffu, c0 >= r.clo && c0 + 31 <= r.chi);
  const uint64_t c2c2 = f2_pack(c2, c2), nmnm = f2_pack(-m_use, -m_use);
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    const uint64_t t = f2_fma(f2_pack(s[e], s[e + 1]), c2c2, nmnm);
    s[e] = f2_lo(t);
    s[e + 1] = f2_hi(t);
  }
  if (full) {
#pragma unroll
    for (int e = 0; e < 32; ++e) s[e] = ex2_approx(s[e]);
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e)
      s[e] = ((uint32_t)(c0 + e - r.clo) <= span) ? ex2_approx(s[e]) : 0.f;
  }
  uint32_t pk[16];
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    lp[(e >> 1) & 3] = f2_add(lp[(e >> 1) & 3], f2_pack(s[e], s[e + 1]));
    pk[e >> 1] = pack_bf16x2(s[e], s[e + 1]);
  }
  tmem_st16(p_addr + 16 * c, pk);
}

// Max of the scaled (log2) logits of chunks [c_lo, c_hi]: the max of the raw
// logits times c2 (scaling by c2 > 0 is monotone, so max(s) * c2 ==
// max(s * c2) exactly).  Four partial maxima of three-input max operations
// keep the dependency chains short.  Returns -inf when no element is live.
template <bool DB = true>
__device__ __forceinline__ float max_chunks(uint32_t s_addr, int c_lo, int c_hi,
                                            const RowMeta& r, float c2) {
  float sa[32];
  [[maybe_unused]] float sb[DB ? 32 : 1];
  const uint32_t span = (uint32_t)(r.chi - r.clo);
  float mr[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  if constexpr (DB) {
    if (c_lo <= c_hi) {
      tmem_ld32(s_addr + 32 * c_lo, sa);
      tmem_wait_ld();
    }
    for (int c = c_lo; c <= c_hi; c += 2) {
      if (c + 1 <= c_hi) tmem_ld32(s_addr + 32 * (c + 1), sb);
      max_one(sa, c, r, span, mr);
      if (c + 1 > c_hi) break;
      tmem_wait_ld();
      if (c + 2 <= c_hi) tmem_ld32(s_addr + 32 * (c + 2), sa);
      max_one(sb, c + 1, r, span, mr);
      tmem_wait_ld();
    }
  } else {
    for (int c = c_lo; c <= c_hi; ++c) {
      tmem_ld32(s_addr + 32 * c, sa);
      tmem_wait_ld();
      max_one(sa, c, r, span, mr);
    }
  }
  const float mraw = fmaxf(fmaxf(mr[0], mr[1]), fmaxf(mr[2], mr[3]));
  return mraw * c2;
}

// P = 2^(x - m_use) as bf16 for chunks [c_lo, c_hi]; returns their row sum
// (eight partial sums, kept as four packed pairs).  Every branch forms the exponent as fma(s, c2, -m)
// (+ sink on key 0) so that a zero KEY0_BIAS sink reproduces the no-sink
// bits exactly.
template <bool DB = true>
__device__ __forceinline__ float exp_chunks(uint32_t s_addr, uint32_t p_addr, int c_lo,
                                            int c_hi, const RowMeta& r, float c2,
                                            float m_use) {
  float sa[32];
  [[maybe_unused]] float sb[DB ? 32 : 1];
  const uint32_t span = (uint32_t)(r.chi - r.clo);
  uint64_t lp[4] = {0, 0, 0, 0};
  if constexpr (DB) {
    if (c_lo <= c_hi) {
      tmem_ld32(s_addr + 32 * c_lo, sa);
      tmem_wait_ld();
    }
    for (int c = c_lo; c <= c_hi; c += 2) {
      if (c + 1 <= c_hi) tmem_ld32(s_addr + 32 * (c + 1), sb);
      exp_one(sa, c, r, c2, m_use, span, lp, p_addr);
      if (c + 1 > c_hi) break;
      tmem_wait_ld();
      if (c + 2 <= c_hi) tmem_ld32(s_addr + 32 * (c + 2), sa);
      exp_one(sb, c + 1, r, c2, m_use, span, lp, p_addr);
      tmem_wait_ld();
    }
  } else {
    for (int c = c_lo; c <= c_hi; ++c) {
      tmem_ld32(s_addr + 32 * c, sa);
      tmem_wait_ld();
      exp_one(sa, c, r, c2, m_use, span, lp, p_addr);
    }
  }
  const uint64_t s = f2_add(f2_add(lp[0], lp[1]), f2_add(lp[2], lp[3]));
  return f2_lo(s) + f2_hi(s);
}

// P = 0 for chunks [c_lo, c_hi].
__device__ __forceinline__ void zero_chunks(uint32_t p_addr, int c_lo, int c_hi) {
  uint32_t z[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) z[e] = 0u;
  for (int c = c_lo; c <= c_hi; ++c) tmem_st16(p_addr + 16 * c, z);
}

// Whole-row softmax over chunks [0, nchunks), the live ones being
// [ch_lo, ch_hi].  Returns the row max m (log2 units, -inf for an empty row)
// and the row sum l of 2^(x - m).
template <bool DB = true, bool DB_MAX = DB>
__device__ __forceinline__ void softmax_rows(uint32_t s_addr, uint32_t p_addr, int nchunks,
                                             int ch_lo, int ch_hi, const RowMeta& r,
                                             float c2, float& m_out, float& l_out) {
  const float m = max_chunks<DB_MAX>(s_addr, ch_lo, ch_hi, r, c2);
  // Rows with no finite logit use 0 as the reference so that -inf - m stays -inf.
  const float m_use = (m == -INFINITY) ? 0.f : m;
  l_out = exp_chunks<DB>(s_addr, p_addr, ch_lo, ch_hi, r, c2, m_use);
  zero_chunks(p_addr, 0, ch_lo - 1);
  zero_chunks(p_addr, ch_hi + 1, nchunks - 1);
  tmem_wait_st();
  m_out = m;
}

// KEY0_BIAS: the sink goes onto each row's first-key logit in S itself, in
// raw logit units (s + sink / (scale log2 e)), before the softmax, which is
// then the no-sink one.  Only warps whose rows see a first key do anything:
// one tensor-memory load and store of each distinct first-key column among
// the warp's rows (one per sequence start in reach), lanes without that
// column storing back what they read.
__device__ __forceinline__ void key0_bias_in_tmem(uint32_t s_addr, const RowMeta& r, float c2) {
  tmem_add_lane_column(s_addr, r.ck0, r.sink2 / c2);
}

// 1/den (with the NULL_LOGIT fold) and the natural-log LSE over real keys.
template <int MODE>
__device__ __forceinline__ void finalize_row(const RowMeta& r, float m, float l, float& inv,
                                             float& lse_v) {
  inv = 0.f;
  lse_v = -INFINITY;
  if (m != -INFINITY) {
    float den = l, alpha = 1.f;
    if (MODE == SA_SINK_NULL_LOGIT) {
      const float mp = fmaxf(m, r.sink2);
      alpha = ex2_approx(m - mp);
      den = l * alpha + ex2_approx(r.sink2 - mp);
    }
    inv = alpha / den;
    lse_v = (m + log2f(l)) * kLn2;
  }
}

// Normalise and store 16-column groups [g_lo, g_hi) of the O row, read from
// tensor memory at o_addr, at most BATCH groups per load batch.
template <int D, int BATCH = 4>
__device__ __forceinline__ void store_o_groups(uint32_t o_addr, int g_lo, int g_hi,
                                               const RowMeta& r, float inv,
                                               __nv_bfloat16* out, int num_q_heads) {
  __nv_bfloat16* orow = out + ((int64_t)r.t * num_q_heads + r.h) * D;
  for (int g0 = g_lo; g0 < g_hi; g0 += BATCH) {
    float oa[BATCH][16];
#pragma unroll
    for (int j = 0; j < BATCH; ++j)
      if (g0 + j < g_hi) tmem_ld16(o_addr + 16 * (g0 + j), oa[j]);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < BATCH; ++j) {
      if (g0 + j >= g_hi || !r.valid) continue;
      const float* o = oa[j];
      uint4 w0, w1;
      w0.x = pack_bf16x2(o[0] * inv, o[1] * inv);
      w0.y = pack_bf16x2(o[2] * inv, o[3] * inv);
      w0.z = pack_bf16x2(o[4] * inv, o[5] * inv);
      w0.w = pack_bf16x2(o[6] * inv, o[7] * inv);
      w1.x = pack_bf16x2(o[8] * inv, o[9] * inv);
      w1.y = pack_bf16x2(o[10] * inv, o[11] * inv);
      w1.z = pack_bf16x2(o[12] * inv, o[13] * inv);
      w1.w = pack_bf16x2(o[14] * inv, o[15] * inv);
      uint4* dst = reinterpret_cast<uint4*>(orow + 16 * (g0 + j));
      dst[0] = w0;
      dst[1] = w1;
    }
  }
}

// Sink fold, 1/den, bf16 O row and fp32 LSE for the whole row.
template <int D, int MODE>
__device__ __forceinline__ void epilogue_row(uint32_t o_addr, const RowMeta& r, float m,
                                             float l, __nv_bfloat16* out, float* lse,
                                             int num_q_heads, int total_tokens) {
  float inv, lse_v;
  finalize_row<MODE>(r, m, l, inv, lse_v);
  store_o_groups<D>(o_addr, 0, D / 16, r, inv, out, num_q_heads);
  if (r.valid) lse[(int64_t)r.h * total_tokens + r.t] = lse_v;
}

}  // namespace win
}  // namespace sa

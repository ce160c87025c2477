// sparse_index_fwd.cu -- attention of each decode query over its own top-k
// list of key indices into one shared latent (MLA) KV cache, with the
// NULL_LOGIT sink, plus the split-KV combine.
//
// Operation: afierka-intel/vllm pull 76 "Apply DeepSeek-V4 attn_sink in the
// XPU sparse-MLA Triton kernel", Implementation: the kernel attends exactly
// the selected keys; after the key loop m' = max(m, sink*log2e), the row sum
// and output are rescaled and 2^(sink*log2e - m') joins the sum, while the
// returned LSE stays over the selected keys; a -inf sink changes nothing.
// Layout: the latent row holds 576 values (512 latent + 64 rope); K is the
// whole row and V its first 512 values, shared by all query heads.
//
// Work split.  The index list of a query is cut into slices of 256 slots and
// V's 512 columns into two halves.  One CTA takes (slice, half, query, block of
// up to 128 heads):
//   S = Q K^T        M = 128 heads, N = valid keys of the slice (rounded to 16),
//                    K = 576 in nine 64-wide slabs;
//   O_half = P V     N = 256 V columns, K = the slice's keys.
// Tensor memory: S at columns [0, 256) (P in place, bf16, the A operand of the
// PV MMA), O_half at [256, 512).  Shared memory: the four 64-column slabs of
// the gathered rows that form this CTA's V half stay resident (they are also
// four of the nine K slabs); the other five K slabs and the nine Q slabs
// stream through a two-stage ring.  Rows are gathered by TMA tile::gather4
// into 128-byte-swizzled slabs, which are both the K-major B operand of S and
// the MN-major B operand of O.
// A query whose valid keys all sit in one slice is finished by that CTA
// (sink fold, bf16 O, LSE); otherwise each slice writes (O, m, l) partials
// and the combine kernel merges them and folds the sink once.
#include <cuda_bf16.h>
#include <math.h>

#include <atomic>

#include "sa_internal.h"
#include "sa_ptx.cuh"

namespace sa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kSlab = 64;                 // elements per 128-byte swizzled row
constexpr int kNumQkSlabs = kDqk / kSlab; // 9
constexpr int kHalfSlabs = 4;             // 256 V columns per CTA
constexpr int kSliceKeys = 256;
constexpr int kSlabBytesK = kSliceKeys * 128;  // one gathered K slab, 32 KB
constexpr int kSlabBytesQ = 128 * 128;         // one Q slab, 16 KB
constexpr int kStages = 2;
constexpr int kTmemCols = 512;
constexpr int kColS = 0;
constexpr int kColO = 256;
constexpr int kMaxSlices = 32;

struct IndexParams {
  const int32_t* indices;  // [nq, topk]
  int32_t topk;
  int32_t nslices;
  int64_t num_kv;
  int32_t num_q_heads;
  int32_t nq;
  const float* sinks;
  float scale_log2;
  __nv_bfloat16* out;  // [nq, hq, 512]
  float* lse;          // [hq, nq]
  float* part_o;       // [nq][nslices][hq][512]
  float* part_ml;      // [nq][nslices][hq][2]
  uint32_t* err;
};

struct __align__(8) IndexSmemCtl {
  uint64_t res_full[kHalfSlabs];
  uint64_t step_full[kStages];
  uint64_t step_empty[kStages];
  uint64_t s_full;
  uint64_t o_full;
  uint32_t tmem_base;
  int32_t n_slice;
  int32_t nonempty;
  int32_t warp_cnt[4][kMaxSlices];
  int32_t warp_ofs[2][4];
  int32_t kidx[kSliceKeys];
};

__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* map,
                                            uint64_t* bar, int x, int r0, int r1,
                                            int r2, int r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::"
      "complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
      : "memory");
}

// K slab id used at pipeline step j for V half `half`: the five slabs outside
// the half first (streamed), then the half's four (resident).
__device__ __forceinline__ int step_slab(int j, int half) {
  if (j < 5) {
    // streamed: half 0 -> 4,5,6,7,8 ; half 1 -> 0,1,2,3,8
    if (j == 4) return 8;
    return half == 0 ? 4 + j : j;
  }
  return half * kHalfSlabs + (j - 5);
}

template <int MODE>
__global__ void __launch_bounds__(128, 1)
sparse_index_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_kv,
                        const IndexParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ IndexSmemCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_res = smem;                                   // 4 x 32 KB
  uint8_t* s_kst = s_res + kHalfSlabs * kSlabBytesK;       // 2 x 32 KB
  uint8_t* s_qst = s_kst + kStages * kSlabBytesK;          // 2 x 16 KB

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = blockIdx.x;
  const int half = blockIdx.y & 1;
  const int hb = blockIdx.y >> 1;
  const int slice = blockIdx.z;
  const int32_t* idx_row = p.indices + (int64_t)q * p.topk;

  // ---- count valid entries per slice; compact this slice's indices --------
  for (int s = threadIdx.x; s < 4 * kMaxSlices; s += 128)
    (&ctl.warp_cnt[0][0])[s] = 0;
  __syncthreads();
  for (int k = 0; k * 128 < p.topk; k += 2) {
    // entries 128k + t and 128(k+1) + t both fall in slice k / 2
    int c = 0;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int e = (k + u) * 128 + threadIdx.x;
      if (e < p.topk) {
        const int32_t j = __ldg(idx_row + e);
        c += (j >= 0 && (int64_t)j < p.num_kv) ? 1 : 0;
      }
    }
    c = __reduce_add_sync(0xffffffffu, c);
    if (lane == 0) ctl.warp_cnt[warp][k >> 1] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int nonempty = 0, mine = 0;
    for (int s = 0; s < p.nslices; ++s) {
      const int c = ctl.warp_cnt[0][s] + ctl.warp_cnt[1][s] + ctl.warp_cnt[2][s] +
                    ctl.warp_cnt[3][s];
      nonempty += c > 0 ? 1 : 0;
      if (s == slice) mine = c;
    }
    ctl.nonempty = nonempty;
    ctl.n_slice = mine;
  }
  // compaction of slice entries (order preserved)
  int32_t my_idx[2];
  bool my_ok[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int e = slice * kSliceKeys + u * 128 + threadIdx.x;
    my_idx[u] = (e < p.topk) ? __ldg(idx_row + e) : -1;
    my_ok[u] = my_idx[u] >= 0 && (int64_t)my_idx[u] < p.num_kv;
    const uint32_t bal = __ballot_sync(0xffffffffu, my_ok[u]);
    if (lane == 0) ctl.warp_ofs[u][warp] = __popc(bal);
  }
  __syncthreads();
  {
    int base = 0;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint32_t bal = __ballot_sync(0xffffffffu, my_ok[u]);
      int before = base;
      for (int w = 0; w < warp; ++w) before += ctl.warp_ofs[u][w];
      if (my_ok[u]) ctl.kidx[before + __popc(bal & ((1u << lane) - 1u))] = my_idx[u];
      base += ctl.warp_ofs[u][0] + ctl.warp_ofs[u][1] + ctl.warp_ofs[u][2] +
              ctl.warp_ofs[u][3];
    }
  }
  __syncthreads();
  const int n = ctl.n_slice;
  const int nonempty = ctl.nonempty;
  const int row = threadIdx.x;
  const int h = hb * 128 + row;
  const bool row_valid = h < p.num_q_heads;
  const float sink2 = (MODE != SA_SINK_NONE && row_valid) ? __ldg(p.sinks + h) * kLog2e : 0.f;
  const bool direct = nonempty <= 1;  // this CTA produces the final output

  if (n == 0) {
    // every slice records its (m, l) so that a reused workspace never holds
    // stale entries for the combine to read
    if (p.part_ml && half == 0 && row_valid) {
      float* ml = p.part_ml + (((int64_t)q * p.nslices + slice) * p.num_q_heads + h) * 2;
      ml[0] = -INFINITY;
      ml[1] = 0.f;
    }
    if (nonempty == 0 && slice == 0 && row_valid) {
      // empty key set: zero output, LSE = -inf
      uint4* dst = reinterpret_cast<uint4*>(p.out + ((int64_t)q * p.num_q_heads + h) * kDv +
                                            half * 256);
      for (int i = 0; i < 32; ++i) dst[i] = make_uint4(0, 0, 0, 0);
      if (half == 0) p.lse[(int64_t)h * p.nq + q] = -INFINITY;
    }
    return;
  }
  const int npad = (n + 15) & ~15;  // MMA N and gathered rows

  if (threadIdx.x == 0) {
    for (int r = 0; r < kHalfSlabs; ++r) mbar_init(&ctl.res_full[r], 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl.step_full[s], 1);
      mbar_init(&ctl.step_empty[s], 1);
    }
    mbar_init(&ctl.s_full, 1);
    mbar_init(&ctl.o_full, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&ctl.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const int qrow0 = q * p.num_q_heads + hb * 128;  // first Q row of this block
  bool ok = true;

  if (threadIdx.x == 32) {
    // ---- producer ---------------------------------------------------------
    tma_prefetch_map(&tm_q);
    tma_prefetch_map(&tm_kv);
    const uint32_t slab_bytes = (uint32_t)npad * 128u;
    for (int r = 0; r < kHalfSlabs; ++r) {
      const int slab = half * kHalfSlabs + r;
      mbar_arrive_expect_tx(&ctl.res_full[r], slab_bytes);
      for (int g = 0; g < npad; g += 4) {
        const int r0 = g + 0 < n ? ctl.kidx[g + 0] : -1;
        const int r1 = g + 1 < n ? ctl.kidx[g + 1] : -1;
        const int r2 = g + 2 < n ? ctl.kidx[g + 2] : -1;
        const int r3 = g + 3 < n ? ctl.kidx[g + 3] : -1;
        tma_gather4(s_res + r * kSlabBytesK + g * 128, &tm_kv, &ctl.res_full[r],
                    slab * kSlab, r0, r1, r2, r3);
      }
    }
    for (int j = 0; j < kNumQkSlabs && ok; ++j) {
      const int st = j & 1;
      const int use = j >> 1;
      if (j >= kStages) ok = mbar_wait(&ctl.step_empty[st], (use - 1) & 1, p.err, kErrWaitFree);
      if (!ok) break;
      const int slab = step_slab(j, half);
      const bool streamed = j < 5;
      mbar_arrive_expect_tx(&ctl.step_full[st],
                            kSlabBytesQ + (streamed ? slab_bytes : 0u));
      tma_load_2d(s_qst + st * kSlabBytesQ, &tm_q, &ctl.step_full[st], slab * kSlab, qrow0);
      if (streamed) {
        for (int g = 0; g < npad; g += 4) {
          const int r0 = g + 0 < n ? ctl.kidx[g + 0] : -1;
          const int r1 = g + 1 < n ? ctl.kidx[g + 1] : -1;
          const int r2 = g + 2 < n ? ctl.kidx[g + 2] : -1;
          const int r3 = g + 3 < n ? ctl.kidx[g + 3] : -1;
          tma_gather4(s_kst + st * kSlabBytesK + g * 128, &tm_kv, &ctl.step_full[st],
                      slab * kSlab, r0, r1, r2, r3);
        }
      }
    }
  } else if (threadIdx.x == 0) {
    // ---- MMA issuer: S = Q K^T over nine slabs ----------------------------
    const uint32_t idesc = idesc_bf16(128, npad, false);
    for (int j = 0; j < kNumQkSlabs && ok; ++j) {
      const int st = j & 1;
      const int use = j >> 1;
      ok = mbar_wait(&ctl.step_full[st], use & 1, p.err, kErrWaitLoad);
      const bool streamed = j < 5;
      if (ok && !streamed) ok = mbar_wait(&ctl.res_full[j - 5], 0, p.err, kErrWaitLoad);
      if (!ok) break;
      tc_fence_after();
      const uint8_t* kb = streamed ? s_kst + st * kSlabBytesK : s_res + (j - 5) * kSlabBytesK;
      const uint8_t* qb = s_qst + st * kSlabBytesQ;
#pragma unroll
      for (int kk = 0; kk < kSlab / 16; ++kk) {
        const uint64_t a = smem_desc(smem_u32(qb) + kk * 32, 16, 1024, kLayoutSw128);
        const uint64_t b = smem_desc(smem_u32(kb) + kk * 32, 16, 1024, kLayoutSw128);
        mma_ss(tmem + kColS, a, b, idesc, (j > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit(&ctl.step_empty[st]);
    }
    if (ok) mma_commit(&ctl.s_full);
    else mbar_arrive(&ctl.s_full);
  }

  // ---- softmax over the slice's keys (thread = head row) -------------------
  const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
  ok = mbar_wait(&ctl.s_full, 0, p.err, kErrWaitMma) && ok;
  __syncwarp();
  tc_fence_after();
  const float c2 = p.scale_log2;
  const int nch = (npad + 31) >> 5;
  float m = -INFINITY;
  for (int c = 0; c < nch; ++c) {
    float s[32];
    tmem_ld32(lane_base + kColS + 32 * c, s);
    tmem_wait_ld();
    const int c0 = 32 * c;
#pragma unroll
    for (int e = 0; e < 32; ++e) m = fmaxf(m, (c0 + e < n) ? s[e] * c2 : -INFINITY);
  }
  float l = 0.f;
  for (int c = 0; c < nch; ++c) {
    float s[32];
    tmem_ld32(lane_base + kColS + 32 * c, s);
    tmem_wait_ld();
    const int c0 = 32 * c;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      s[e] = (c0 + e < n) ? ex2_approx(fmaf(s[e], c2, -m)) : 0.f;
      l += s[e];
    }
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(s[2 * e], s[2 * e + 1]);
    tmem_st16(lane_base + kColS + 16 * c, pk);
  }
  tmem_wait_st();
  tc_fence_before();
  __syncthreads();

  // ---- O_half = P V --------------------------------------------------------
  if (threadIdx.x == 0) {
    tc_fence_after();
    if (ok) {
      const uint32_t idesc = idesc_bf16(128, 256, true);
      for (int kk = 0; kk < npad / 16; ++kk) {
        const uint64_t b = smem_desc(smem_u32(s_res) + kk * 16 * 128, kSlabBytesK, 1024,
                                     kLayoutSw128);
        mma_ts(tmem + kColO, tmem + kColS + kk * 8, b, idesc, kk > 0 ? 1u : 0u);
      }
      mma_commit(&ctl.o_full);
    } else {
      mbar_arrive(&ctl.o_full);
    }
  }
  mbar_wait(&ctl.o_full, 0, p.err, kErrWaitMma);
  __syncwarp();
  tc_fence_after();

  // ---- epilogue --------------------------------------------------------------
  if (direct) {
    float den = l, alpha = 1.f;
    if (MODE == SA_SINK_NULL_LOGIT) {
      const float mp = fmaxf(m, sink2);
      alpha = ex2_approx(m - mp);
      den = l * alpha + ex2_approx(sink2 - mp);
    }
    const float inv = alpha / den;
    __nv_bfloat16* orow = p.out + ((int64_t)q * p.num_q_heads + h) * kDv + half * 256;
#pragma unroll 1
    for (int j = 0; j < 16; ++j) {
      float o[16];
      tmem_ld16(lane_base + kColO + 16 * j, o);
      tmem_wait_ld();
      if (row_valid) {
        uint4 w0, w1;
        w0.x = pack_bf16x2(o[0] * inv, o[1] * inv);
        w0.y = pack_bf16x2(o[2] * inv, o[3] * inv);
        w0.z = pack_bf16x2(o[4] * inv, o[5] * inv);
        w0.w = pack_bf16x2(o[6] * inv, o[7] * inv);
        w1.x = pack_bf16x2(o[8] * inv, o[9] * inv);
        w1.y = pack_bf16x2(o[10] * inv, o[11] * inv);
        w1.z = pack_bf16x2(o[12] * inv, o[13] * inv);
        w1.w = pack_bf16x2(o[14] * inv, o[15] * inv);
        uint4* dst = reinterpret_cast<uint4*>(orow + 16 * j);
        dst[0] = w0;
        dst[1] = w1;
      }
    }
    if (half == 0 && row_valid) p.lse[(int64_t)h * p.nq + q] = (m + log2f(l)) * kLn2;
    if (p.part_ml && half == 0 && row_valid) {
      float* ml = p.part_ml + (((int64_t)q * p.nslices + slice) * p.num_q_heads + h) * 2;
      ml[0] = m;
      ml[1] = l;
    }
  } else {
    float* prow = p.part_o + (((int64_t)q * p.nslices + slice) * p.num_q_heads + h) * kDv +
                  half * 256;
#pragma unroll 1
    for (int j = 0; j < 16; ++j) {
      float o[16];
      tmem_ld16(lane_base + kColO + 16 * j, o);
      tmem_wait_ld();
      if (row_valid) {
        float4* dst = reinterpret_cast<float4*>(prow + 16 * j);
        dst[0] = make_float4(o[0], o[1], o[2], o[3]);
        dst[1] = make_float4(o[4], o[5], o[6], o[7]);
        dst[2] = make_float4(o[8], o[9], o[10], o[11]);
        dst[3] = make_float4(o[12], o[13], o[14], o[15]);
      }
    }
    if (half == 0 && row_valid) {
      float* ml = p.part_ml + (((int64_t)q * p.nslices + slice) * p.num_q_heads + h) * 2;
      ml[0] = m;
      ml[1] = l;
    }
  }

  // ---- teardown ----------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 32 && !ok) {
    // bounded drain of any gather still in flight
    for (int r = 0; r < kHalfSlabs; ++r) mbar_wait(&ctl.res_full[r], 0, p.err, kErrWaitDrain);
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Merge the (O, m, l) partials of queries whose keys span several slices;
// one CTA per (head, query), 128 threads x 4 V columns.
template <int MODE>
__global__ void __launch_bounds__(128)
sparse_index_combine_kernel(const IndexParams p) {
  const int q = blockIdx.x;
  const int h = blockIdx.y;
  const float* ml = p.part_ml + ((int64_t)q * p.nslices * p.num_q_heads + h) * 2;
  const int64_t ml_stride = (int64_t)p.num_q_heads * 2;
  int nonempty = 0;
  float M = -INFINITY;
  for (int s = 0; s < p.nslices; ++s) {
    const float l = ml[s * ml_stride + 1];
    if (l > 0.f) {
      ++nonempty;
      M = fmaxf(M, ml[s * ml_stride]);
    }
  }
  if (nonempty < 2) return;  // finished by the slice kernel
  float L = 0.f;
  for (int s = 0; s < p.nslices; ++s) {
    const float l = ml[s * ml_stride + 1];
    if (l > 0.f) L += l * ex2_approx(ml[s * ml_stride] - M);
  }
  float den = L, alpha = 1.f;
  if (MODE == SA_SINK_NULL_LOGIT) {
    const float sink2 = __ldg(p.sinks + h) * kLog2e;
    const float mp = fmaxf(M, sink2);
    alpha = ex2_approx(M - mp);
    den = L * alpha + ex2_approx(sink2 - mp);
  }
  const float inv = alpha / den;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const int d = threadIdx.x * 4;
  for (int s = 0; s < p.nslices; ++s) {
    const float l = ml[s * ml_stride + 1];
    if (!(l > 0.f)) continue;
    const float w = ex2_approx(ml[s * ml_stride] - M);
    const float4 o = *reinterpret_cast<const float4*>(
        p.part_o + (((int64_t)q * p.nslices + s) * p.num_q_heads + h) * kDv + d);
    acc.x = fmaf(w, o.x, acc.x);
    acc.y = fmaf(w, o.y, acc.y);
    acc.z = fmaf(w, o.z, acc.z);
    acc.w = fmaf(w, o.w, acc.w);
  }
  uint2 packed;
  packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(p.out + ((int64_t)q * p.num_q_heads + h) * kDv + d) = packed;
  if (threadIdx.x == 0) p.lse[(int64_t)h * p.nq + q] = (M + log2f(L)) * kLn2;
}

template <int MODE>
sa_status launch_typed(const IndexArgs& a, int nslices) {
  CUtensorMap tq, tkv;
  const uint64_t dq[2] = {(uint64_t)kDqk, (uint64_t)a.num_queries * a.num_q_heads};
  const uint64_t sq[1] = {(uint64_t)kDqk * 2};
  const uint32_t bq[2] = {kSlab, 128};
  const uint64_t dk[2] = {(uint64_t)kDqk, (uint64_t)a.num_kv};
  const uint32_t bk[2] = {kSlab, 1};
  if (!encode_tiled(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, dq, sq, bq,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled(&tkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.kv, dk, sq, bk,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B))
    return SA_ERR_INVALID_ARG;
  IndexParams p;
  p.indices = a.indices;
  p.topk = a.topk;
  p.nslices = nslices;
  p.num_kv = a.num_kv;
  p.num_q_heads = a.num_q_heads;
  p.nq = a.num_queries;
  p.sinks = a.sinks;
  p.scale_log2 = a.softmax_scale * kLog2e;
  p.out = reinterpret_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  float* ws = reinterpret_cast<float*>(a.workspace);
  p.part_o = ws;
  p.part_ml = ws ? ws + (size_t)a.num_queries * nslices * a.num_q_heads * kDv : nullptr;
  p.err = device_error_word();

  const size_t smem = 1024 + (size_t)(kHalfSlabs + kStages) * kSlabBytesK +
                      (size_t)kStages * kSlabBytesQ;
  auto kern = sparse_index_fwd_kernel<MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess)
    return fail(SA_ERR_CUDA, "sa_sparse_index_fwd: %s", cudaGetErrorString(e));
  const int nhb = (a.num_q_heads + 127) / 128;
  dim3 grid((unsigned)a.num_queries, (unsigned)(2 * nhb), (unsigned)nslices);
  kern<<<grid, 128, smem, a.stream>>>(tq, tkv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(SA_ERR_CUDA, "sa_sparse_index_fwd launch: %s", cudaGetErrorString(e));
  if (nslices > 1) {
    dim3 g2((unsigned)a.num_queries, (unsigned)a.num_q_heads);
    sparse_index_combine_kernel<MODE><<<g2, 128, 0, a.stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess)
      return fail(SA_ERR_CUDA, "sa_sparse_index_fwd combine launch: %s", cudaGetErrorString(e));
  }
  return SA_OK;
}

}  // namespace

size_t sparse_index_workspace_bytes(int32_t num_queries, int32_t num_q_heads, int32_t topk) {
  const int nslices = topk <= kSliceKeys ? 1 : (topk + kSliceKeys - 1) / kSliceKeys;
  if (nslices <= 1) return 0;
  return (size_t)num_queries * nslices * num_q_heads * (kDv + 2) * sizeof(float);
}

int sparse_index_max_topk() { return kMaxSlices * kSliceKeys; }

sa_status launch_sparse_index_fwd(const IndexArgs& a) {
  if (a.dqk != kDqk || a.dv != kDv)
    return fail(SA_ERR_UNSUPPORTED,
                "sa_sparse_index_fwd: dqk %d / dv %d (supported: 576 / 512)", a.dqk, a.dv);
  const int nslices = a.topk <= kSliceKeys ? 1 : (a.topk + kSliceKeys - 1) / kSliceKeys;
  if (a.sink_mode == SA_SINK_NULL_LOGIT) return launch_typed<SA_SINK_NULL_LOGIT>(a, nslices);
  return launch_typed<SA_SINK_NONE>(a, nslices);
}

}  // namespace sa

// ---------------------------------------------------------------------------
// Allocation-free entry point.
//
// Some callers cannot obtain device memory for a workspace: code embedded in a
// host runtime that owns the whole device memory pool and hands its plugins no
// allocator, or a serving loop that forbids any allocation once it is running.
// sa_sparse_index_fwd_noalloc serves them by keeping the split-KV partials in
// the fixed array below instead of a caller workspace.  The array is reserved
// on every GPU that loads this library and stays reserved until the process
// exits.  Every call shares it and it keeps the last call's contents; nothing
// in it has to start at zero, because each call writes every (m, l) entry and
// every partial row it later reads.  Two calls whose work overlaps on the GPU
// (different streams, or different host threads) race on the array.
namespace sa {
namespace {
constexpr size_t kNoAllocScratchBytes = (size_t)64 << 20;  // 64 MiB
constexpr int kNoAllocMaxDevices = 64;
std::atomic<void*> g_noalloc_scratch_ptr[kNoAllocMaxDevices];
}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

}  // namespace sa

extern "C" sa_status sa_sparse_index_fwd_noalloc(
    const void* q, const void* kv_latent, int64_t num_kv, int32_t dqk, int32_t dv,
    const int32_t* indices, int32_t topk, int32_t num_queries, int32_t num_q_heads,
    const float* sinks, int32_t sink_mode, float softmax_scale, void* out, float* lse,
    void* stream) {
  const char* fn = "sa_sparse_index_fwd_noalloc";
  const size_t need = sa_sparse_index_workspace_size(num_queries, num_q_heads, dv, topk);
  if (need > sa::kNoAllocScratchBytes)
    return sa::fail(SA_ERR_UNSUPPORTED,
                    "%s: these sizes need %zu bytes of scratch, above the fixed %zu bytes "
                    "(64 MiB) of this entry point; use sa_sparse_index_fwd with a workspace",
                    fn, need, sa::kNoAllocScratchBytes);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= sa::kNoAllocMaxDevices)
    return sa::fail(SA_ERR_CUDA, "%s: no usable CUDA device", fn);
  void* ptr = sa::g_noalloc_scratch_ptr[dev].load(std::memory_order_acquire);
  if (!ptr) {
    // One-time set-up on this device (the device is current): the host-side
    // name of the array is not a device address, so ask the runtime for it.
    e = cudaGetSymbolAddress(&ptr, sa::g_noalloc_scratch);
    if (e != cudaSuccess || !ptr)
      return sa::fail(SA_ERR_CUDA, "%s: cudaGetSymbolAddress failed: %s", fn,
                      cudaGetErrorString(e));
    sa::g_noalloc_scratch_ptr[dev].store(ptr, std::memory_order_release);
  }
  return sa_sparse_index_fwd(q, kv_latent, num_kv, dqk, dv, indices, topk, num_queries,
                             num_q_heads, sinks, sink_mode, softmax_scale, out, lse, ptr,
                             sa::kNoAllocScratchBytes, stream);
}

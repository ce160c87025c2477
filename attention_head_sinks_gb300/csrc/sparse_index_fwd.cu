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
// Work split.  The index list of a query is cut into slices of 256 slots; one
// CTA takes (query, slice, block of up to 128 heads):
//   S = Q K^T        M = 128 heads, N = valid keys of the slice (rounded to 16),
//                    K = 576 in nine 64-wide slabs;
//   O_half = P V     twice, N = 256 V columns each, K = the slice's keys.
// Tensor memory: S at columns [0, 256) (P in place, bf16, the A operand of the
// PV MMAs), O_half at [256, 512), reused by the second half.  Shared memory:
// slabs 0..3 of the gathered rows (V columns 0..255, also K slabs) stay
// resident; K slabs 4..8 and the nine Q slabs stream through two-stage rings;
// after the first P V, slabs 4..7 are gathered again (from L2) over the
// resident buffer for the second.  Warps 0..3 own the 128 head rows (softmax,
// epilogue; thread 0 issues the MMAs, thread 32 loads Q by TMA); warps 4..7
// gather the key rows with 16-byte cp.async copies straight into
// 128-byte-swizzled slabs -- the K-major B operand of S and the MN-major B
// operand of O.
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
  uint64_t res_full;         // resident slabs 0..3 gathered
  uint64_t res2_full;        // slabs 4..7 gathered over them for the second V half
  uint64_t kst_full[kStages];
  uint64_t kst_empty[kStages];
  uint64_t q_full[kStages];
  uint64_t q_empty[kStages];
  uint64_t s_full;
  uint64_t o_full;           // phase 0: first V half, phase 1: second
  uint32_t tmem_base;
  int32_t warp_cnt[4][kMaxSlices];
  int32_t warp_ofs[2][4];
  int32_t kidx[kSliceKeys];
};

// K slab used at S step j: slabs 4..8 stream through the ring first, then
// the resident slabs 0..3 (which are also V columns 0..255).
__device__ __forceinline__ int step_slab(int j) { return j < 5 ? 4 + j : j - 5; }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void bar_rows() {  // the four row warps only
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// Gather 64 columns (slab `slab`) of the slice's npad key rows into a
// 128-byte-swizzled [npad][64] bf16 slab at dst; rows past n are zero.
// Thread gt of 128 copies 16-byte chunks gt, gt + 128, ... (8 per row).
__device__ __forceinline__ void gather_slab(uint32_t dst, const uint16_t* kv,
                                            const int32_t* kidx, int n, int npad, int slab,
                                            int gt) {
  for (int ch = gt; ch < npad * 8; ch += 128) {
    const int r = ch >> 3, c = ch & 7;
    const bool live = r < n;
    const uint16_t* src = kv + (live ? (int64_t)kidx[r] * kDqk + slab * kSlab + c * 8 : 0);
    cp_async16(dst + r * 128 + ((c ^ (r & 7)) << 4), src, live ? 16u : 0u);
  }
}

template <int MODE>
__global__ void __launch_bounds__(256, 1)
sparse_index_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const uint16_t* kv,
                        const IndexParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ IndexSmemCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_res = smem;                                   // 4 x 32 KB
  uint8_t* s_kst = s_res + kHalfSlabs * kSlabBytesK;       // 2 x 32 KB
  uint8_t* s_qst = s_kst + kStages * kSlabBytesK;          // 2 x 16 KB

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int q = blockIdx.x;
  const int hb = blockIdx.y;
  const int slice = blockIdx.z;
  const int32_t* idx_row = p.indices + (int64_t)q * p.topk;

  // ---- compact this slice's valid indices (warps 0..3) ---------------------
  int32_t my_idx[2] = {-1, -1};
  bool my_ok[2] = {false, false};
  if (tid < 128) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int e = slice * kSliceKeys + u * 128 + tid;
      my_idx[u] = (e < p.topk) ? __ldg(idx_row + e) : -1;
      my_ok[u] = my_idx[u] >= 0 && (int64_t)my_idx[u] < p.num_kv;
      const uint32_t bal = __ballot_sync(0xffffffffu, my_ok[u]);
      if (lane == 0) ctl.warp_ofs[u][warp] = __popc(bal);
    }
  }
  __syncthreads();
  int n = 0;
#pragma unroll
  for (int u = 0; u < 2; ++u)
    n += ctl.warp_ofs[u][0] + ctl.warp_ofs[u][1] + ctl.warp_ofs[u][2] + ctl.warp_ofs[u][3];
  if (n == 0 && slice != 0) {
    // Empty slice: record (m, l) = (-inf, 0) so that a reused workspace never
    // holds stale entries for the combine to read, and leave.
    if (tid < 128 && p.part_ml) {
      const int h = hb * 128 + tid;
      if (h < p.num_q_heads) {
        float* ml = p.part_ml + (((int64_t)q * p.nslices + slice) * p.num_q_heads + h) * 2;
        ml[0] = -INFINITY;
        ml[1] = 0.f;
      }
    }
    return;
  }
  if (tid < 128) {
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
    // non-empty slices of the whole row (decides final output vs partial)
    for (int s2 = tid; s2 < 4 * kMaxSlices; s2 += 128) (&ctl.warp_cnt[0][0])[s2] = 0;
  }
  __syncthreads();
  if (tid < 128) {
    for (int k = 0; k * 128 < p.topk; k += 2) {
      // entries 128k + t and 128(k+1) + t both fall in slice k / 2
      int c = 0;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int e = (k + u) * 128 + tid;
        if (e < p.topk) {
          const int32_t jj = __ldg(idx_row + e);
          c += (jj >= 0 && (int64_t)jj < p.num_kv) ? 1 : 0;
        }
      }
      c = __reduce_add_sync(0xffffffffu, c);
      if (lane == 0) ctl.warp_cnt[warp][k >> 1] = c;
    }
  }
  __syncthreads();
  int nonempty = 0;
  for (int s2 = 0; s2 < p.nslices; ++s2)
    nonempty += (ctl.warp_cnt[0][s2] + ctl.warp_cnt[1][s2] + ctl.warp_cnt[2][s2] +
                 ctl.warp_cnt[3][s2]) > 0 ? 1 : 0;
  const bool direct = nonempty <= 1;  // this CTA produces the final output

  if (n == 0) {
    // slice 0 of a row: an empty key set gets zero output and LSE = -inf
    if (tid < 128) {
      const int h = hb * 128 + tid;
      if (h < p.num_q_heads) {
        if (p.part_ml) {
          float* ml = p.part_ml + (((int64_t)q * p.nslices + slice) * p.num_q_heads + h) * 2;
          ml[0] = -INFINITY;
          ml[1] = 0.f;
        }
        if (nonempty == 0) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + ((int64_t)q * p.num_q_heads + h) * kDv);
          for (int i = 0; i < kDv / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
          p.lse[(int64_t)h * p.nq + q] = -INFINITY;
        }
      }
    }
    return;
  }
  const int npad = (n + 15) & ~15;  // MMA N and gathered rows

  if (tid == 0) {
    mbar_init(&ctl.res_full, 128);
    mbar_init(&ctl.res2_full, 128);
    for (int s2 = 0; s2 < kStages; ++s2) {
      mbar_init(&ctl.kst_full[s2], 128);
      mbar_init(&ctl.kst_empty[s2], 1);
      mbar_init(&ctl.q_full[s2], 1);
      mbar_init(&ctl.q_empty[s2], 1);
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

  if (warp >= 4) {
    // ---- gatherers (warps 4..7) --------------------------------------------
    const int gt = tid - 128;
    bool ok = true;
    // resident slabs 0..3 first (one cp.async group)
    for (int r = 0; r < kHalfSlabs; ++r)
      gather_slab(smem_u32(s_res + r * kSlabBytesK), kv, ctl.kidx, n, npad, r, gt);
    cp_async_commit();
    // streamed slabs 4..8 through the two-stage ring
    for (int j = 0; j < 5; ++j) {
      const int st = j & 1;
      if (j >= kStages && ok)
        ok = mbar_wait(&ctl.kst_empty[st], ((j >> 1) - 1) & 1, p.err, kErrWaitFree);
      if (ok) gather_slab(smem_u32(s_kst + st * kSlabBytesK), kv, ctl.kidx, n, npad, 4 + j, gt);
      cp_async_commit();
      // every group but the newest has landed: publish it
      cp_async_wait<1>();
      fence_proxy_async();
      if (j == 0) mbar_arrive(&ctl.res_full);
      else mbar_arrive(&ctl.kst_full[(j - 1) & 1]);
    }
    cp_async_wait<0>();
    fence_proxy_async();
    mbar_arrive(&ctl.kst_full[4 & 1]);
    // second V half: once P V of the first half is done, slabs 4..7 replace
    // slabs 0..3 in the resident buffer
    if (ok) ok = mbar_wait(&ctl.o_full, 0, p.err, kErrWaitMma);
    if (ok)
      for (int r = 0; r < kHalfSlabs; ++r)
        gather_slab(smem_u32(s_res + r * kSlabBytesK), kv, ctl.kidx, n, npad, 4 + r, gt);
    cp_async_commit();
    cp_async_wait<0>();
    fence_proxy_async();
    mbar_arrive(&ctl.res2_full);
  } else {
    // ---- warps 0..3: MMA issue (thread 0), softmax and epilogue (rows) -----
    const int row = tid;
    const int h = hb * 128 + row;
    const bool row_valid = h < p.num_q_heads;
    const float sink2 = (MODE != SA_SINK_NONE && row_valid) ? __ldg(p.sinks + h) * kLog2e : 0.f;
    bool ok = true;
    if (tid == 0) {
      const uint32_t idesc = idesc_bf16(128, npad, false);
      for (int j = 0; j < kNumQkSlabs && ok; ++j) {
        const int st = j & 1;
        ok = mbar_wait(&ctl.q_full[st], (j >> 1) & 1, p.err, kErrWaitLoad);
        if (ok && j < 5) ok = mbar_wait(&ctl.kst_full[st], (j >> 1) & 1, p.err, kErrWaitLoad);
        if (ok && j == 5) ok = mbar_wait(&ctl.res_full, 0, p.err, kErrWaitLoad);
        if (!ok) break;
        tc_fence_after();
        const uint8_t* kb = j < 5 ? s_kst + st * kSlabBytesK : s_res + (j - 5) * kSlabBytesK;
        const uint8_t* qb = s_qst + st * kSlabBytesQ;
#pragma unroll
        for (int kk = 0; kk < kSlab / 16; ++kk) {
          const uint64_t a = smem_desc(smem_u32(qb) + kk * 32, 16, 1024, kLayoutSw128);
          const uint64_t b = smem_desc(smem_u32(kb) + kk * 32, 16, 1024, kLayoutSw128);
          mma_ss(tmem + kColS, a, b, idesc, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&ctl.q_empty[st]);
        if (j < 5) mma_commit(&ctl.kst_empty[st]);
      }
      if (ok) mma_commit(&ctl.s_full);
      else mbar_arrive(&ctl.s_full);
    } else if (tid == 32) {
      // Q slab of each S step by TMA through its two-stage ring
      tma_prefetch_map(&tm_q);
      int issued = 0;
      for (int j = 0; j < kNumQkSlabs; ++j) {
        const int st = j & 1;
        if (j >= kStages && !mbar_wait(&ctl.q_empty[st], ((j >> 1) - 1) & 1, p.err, kErrWaitFree))
          break;
        mbar_arrive_expect_tx(&ctl.q_full[st], kSlabBytesQ);
        tma_load_2d(s_qst + st * kSlabBytesQ, &tm_q, &ctl.q_full[st], step_slab(j) * kSlab,
                    qrow0);
        ++issued;
      }
      // bounded drain of the last copies (immediate once the MMAs consumed them)
      for (int j = max(0, issued - kStages); j < issued; ++j)
        mbar_wait(&ctl.q_full[j & 1], (j >> 1) & 1, p.err, kErrWaitDrain);
    }

    // ---- softmax over the slice's keys (thread = head row) -----------------
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    ok = mbar_wait(&ctl.s_full, 0, p.err, kErrWaitMma) && ok;
    __syncwarp();
    tc_fence_after();
    const float c2 = p.scale_log2;
    const int nch = (npad + 31) >> 5;
    float mr[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) mr[e] = -INFINITY;
    for (int c = 0; c < nch; ++c) {
      float sv[32];
      tmem_ld32(lane_base + kColS + 32 * c, sv);
      tmem_wait_ld();
      const int c0 = 32 * c;
#pragma unroll
      for (int e = 0; e < 32; ++e) mr[e & 7] = fmaxf(mr[e & 7], (c0 + e < n) ? sv[e] : -INFINITY);
    }
    // max(s) * c2 == max(s * c2) exactly (c2 > 0, rounding is monotone)
    const float m = fmaxf(fmaxf(fmaxf(mr[0], mr[1]), fmaxf(mr[2], mr[3])),
                          fmaxf(fmaxf(mr[4], mr[5]), fmaxf(mr[6], mr[7]))) * c2;
    float lp[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) lp[e] = 0.f;
    for (int c = 0; c < nch; ++c) {
      float sv[32];
      tmem_ld32(lane_base + kColS + 32 * c, sv);
      tmem_wait_ld();
      const int c0 = 32 * c;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        sv[e] = (c0 + e < n) ? ex2_approx(fmaf(sv[e], c2, -m)) : 0.f;
        lp[e & 7] += sv[e];
      }
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(sv[2 * e], sv[2 * e + 1]);
      tmem_st16(lane_base + kColS + 16 * c, pk);
    }
    const float l = ((lp[0] + lp[1]) + (lp[2] + lp[3])) + ((lp[4] + lp[5]) + (lp[6] + lp[7]));
    tmem_wait_st();
    float inv;
    {
      float den = l, alpha = 1.f;
      if (MODE == SA_SINK_NULL_LOGIT) {
        const float mp = fmaxf(m, sink2);
        alpha = ex2_approx(m - mp);
        den = l * alpha + ex2_approx(sink2 - mp);
      }
      inv = alpha / den;
    }

    // ---- the two V halves: O_half = P V_half, then store -------------------
    for (int half = 0; half < 2; ++half) {
      tc_fence_before();
      bar_rows();
      if (tid == 0) {
        tc_fence_after();
        bool go = ok;
        if (go && half == 1) go = mbar_wait(&ctl.res2_full, 0, p.err, kErrWaitLoad);
        if (go) {
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
      ok = mbar_wait(&ctl.o_full, half, p.err, kErrWaitMma) && ok;
      __syncwarp();
      tc_fence_after();
      if (direct) {
        __nv_bfloat16* orow = p.out + ((int64_t)q * p.num_q_heads + h) * kDv + half * 256;
#pragma unroll 1
        for (int jj = 0; jj < 16; ++jj) {
          float o[16];
          tmem_ld16(lane_base + kColO + 16 * jj, o);
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
            uint4* dst = reinterpret_cast<uint4*>(orow + 16 * jj);
            dst[0] = w0;
            dst[1] = w1;
          }
        }
      } else {
        float* prow = p.part_o + (((int64_t)q * p.nslices + slice) * p.num_q_heads + h) * kDv +
                      half * 256;
#pragma unroll 1
        for (int jj = 0; jj < 16; ++jj) {
          float o[16];
          tmem_ld16(lane_base + kColO + 16 * jj, o);
          tmem_wait_ld();
          if (row_valid) {
            float4* dst = reinterpret_cast<float4*>(prow + 16 * jj);
            dst[0] = make_float4(o[0], o[1], o[2], o[3]);
            dst[1] = make_float4(o[4], o[5], o[6], o[7]);
            dst[2] = make_float4(o[8], o[9], o[10], o[11]);
            dst[3] = make_float4(o[12], o[13], o[14], o[15]);
          }
        }
      }
    }
    if (row_valid) {
      if (direct) p.lse[(int64_t)h * p.nq + q] = (m + log2f(l)) * kLn2;
      if (p.part_ml) {
        float* ml = p.part_ml + (((int64_t)q * p.nslices + slice) * p.num_q_heads + h) * 2;
        ml[0] = m;
        ml[1] = l;
      }
    }
  }

  // ---- teardown ----------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Merge the (O, m, l) partials of queries whose keys span several slices and
// fold the sink once.  One CTA per (query, 4 heads): thread t takes head
// t / 64 and V columns 8 (t mod 64) .. + 8, reading every slice's partial row
// with independent 16-byte loads.
template <int MODE>
__global__ void __launch_bounds__(256)
sparse_index_combine_kernel(const IndexParams p) {
  const int q = blockIdx.x;
  const int h = blockIdx.y * 4 + (threadIdx.x >> 6);
  if (h >= p.num_q_heads) return;
  const int d = (threadIdx.x & 63) * 8;
  const float* ml = p.part_ml + ((int64_t)q * p.nslices * p.num_q_heads + h) * 2;
  const int64_t ml_stride = (int64_t)p.num_q_heads * 2;
  const float* base = p.part_o + ((int64_t)q * p.nslices * p.num_q_heads + h) * kDv + d;
  const int64_t o_stride = (int64_t)p.num_q_heads * kDv;
  // (m, l) of every slice first, all loads independent
  float2 v[kMaxSlices];
#pragma unroll
  for (int s = 0; s < kMaxSlices; ++s)
    v[s] = s < p.nslices ? *reinterpret_cast<const float2*>(ml + s * ml_stride)
                         : make_float2(-INFINITY, 0.f);
  int nonempty = 0;
  float M = -INFINITY;
#pragma unroll
  for (int s = 0; s < kMaxSlices; ++s) {
    nonempty += v[s].y > 0.f ? 1 : 0;
    M = v[s].y > 0.f ? fmaxf(M, v[s].x) : M;
  }
  if (nonempty < 2) return;  // finished by the slice kernel
  float L = 0.f;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  // partial rows in groups of eight slices, loads issued before use
  for (int s0 = 0; s0 < p.nslices; s0 += 8) {
    float4 o0[8], o1[8];
    float w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int s = s0 + k;
      float2 vs = make_float2(-INFINITY, 0.f);
#pragma unroll
      for (int t = 0; t < kMaxSlices; ++t) vs = (t == s) ? v[t] : vs;
      const bool live = s < p.nslices && vs.y > 0.f;
      w[k] = live ? ex2_approx(vs.x - M) : 0.f;
      L += live ? vs.y * w[k] : 0.f;
      o0[k] = live ? *reinterpret_cast<const float4*>(base + s * o_stride) : make_float4(0.f, 0.f, 0.f, 0.f);
      o1[k] = live ? *reinterpret_cast<const float4*>(base + s * o_stride + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      acc[0] = fmaf(w[k], o0[k].x, acc[0]);
      acc[1] = fmaf(w[k], o0[k].y, acc[1]);
      acc[2] = fmaf(w[k], o0[k].z, acc[2]);
      acc[3] = fmaf(w[k], o0[k].w, acc[3]);
      acc[4] = fmaf(w[k], o1[k].x, acc[4]);
      acc[5] = fmaf(w[k], o1[k].y, acc[5]);
      acc[6] = fmaf(w[k], o1[k].z, acc[6]);
      acc[7] = fmaf(w[k], o1[k].w, acc[7]);
    }
  }
  float den = L, alpha = 1.f;
  if (MODE == SA_SINK_NULL_LOGIT) {
    const float sink2 = __ldg(p.sinks + h) * kLog2e;
    const float mp = fmaxf(M, sink2);
    alpha = ex2_approx(M - mp);
    den = L * alpha + ex2_approx(sink2 - mp);
  }
  const float inv = alpha / den;
  uint4 packed;
  packed.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  packed.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
  packed.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
  packed.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
  *reinterpret_cast<uint4*>(p.out + ((int64_t)q * p.num_q_heads + h) * kDv + d) = packed;
  if ((threadIdx.x & 63) == 0) p.lse[(int64_t)h * p.nq + q] = (M + log2f(L)) * kLn2;
}

template <int MODE>
sa_status launch_typed(const IndexArgs& a, int nslices) {
  CUtensorMap tq;
  const uint64_t dq[2] = {(uint64_t)kDqk, (uint64_t)a.num_queries * a.num_q_heads};
  const uint64_t sq[1] = {(uint64_t)kDqk * 2};
  const uint32_t bq[2] = {kSlab, 128};
  if (!encode_tiled(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, dq, sq, bq,
                    CU_TENSOR_MAP_SWIZZLE_128B))
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
  dim3 grid((unsigned)a.num_queries, (unsigned)nhb, (unsigned)nslices);
  kern<<<grid, 256, smem, a.stream>>>(tq, reinterpret_cast<const uint16_t*>(a.kv), p);
  e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(SA_ERR_CUDA, "sa_sparse_index_fwd launch: %s", cudaGetErrorString(e));
  if (nslices > 1) {
    dim3 g2((unsigned)a.num_queries, (unsigned)((a.num_q_heads + 3) / 4));
    sparse_index_combine_kernel<MODE><<<g2, 256, 0, a.stream>>>(p);
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

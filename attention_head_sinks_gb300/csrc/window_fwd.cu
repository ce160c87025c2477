// window_fwd.cu -- sliding-window attention with per-head sinks over
// cu_seqlens-packed sequences, one tcgen05 tile per CTA.
//
// Operation: vLLM pull 49815 "[Bugfix][MiMo] Apply vision attention sinks in
// the window attention path" -- the KEY0_BIAS sink is added to the logit of
// each sequence's first key, which only the first window_size + 1 queries of
// the sequence reach; the LSE is that of the masked scaled logits, laid out
// (nheads, total_q).  NULL_LOGIT follows afierka-intel/vllm pull 76,
// Implementation: after the key loop m' = max(m, s), the row sum and output
// are rescaled by 2^(m - m') and 2^(s - m') joins the sum; the LSE keeps the
// real keys only.
//
// Tile: M = 128 query rows = (128 / G) consecutive tokens x the G query heads
// that share one KV head (G = Hq / Hkv), packed row = token * G + head.  Keys:
// the NK >= TQ + wl + wr consecutive tokens starting at tok0 - wl, read once
// per tile.  Tiles ignore sequence boundaries: each row masks keys outside
// its own sequence, so no per-sequence launch or host-side metadata exists.
//
// Shared memory: Q, K, V as head_dim/16 slabs of [rows][16] bf16, each 32-byte
// row swizzled by the 32B pattern (TMA SWIZZLE_32B), which is also the
// tcgen05 canonical layout: K-major for Q (A) and K (B) of S = Q K^T, and
// MN-major for V (B) of O = P V.
// Tensor memory (256 columns): S fp32 [128 x NK] at column 0; P bf16 written
// in place over S's first NK/2 columns (A operand of the P V MMA, read from
// tensor memory); O fp32 [128 x D] at column 128.
#include <cuda_bf16.h>
#include <math.h>
#include <stdio.h>

#include "sa_internal.h"
#include "sa_ptx.cuh"
#include "window_common.cuh"

namespace sa {
namespace {

using win::kLog2e;
constexpr int kTmemCols = 256;
constexpr int kColS = 0;
constexpr int kColP = 0;
constexpr int kColO = 128;
constexpr int kMaxNK = 256;

struct WindowParams {
  const int32_t* cu_seqlens;
  int32_t num_seqs;
  int32_t total_tokens;
  int32_t num_q_heads;
  int32_t wl;
  int32_t wr;
  int32_t nk;  // key columns per tile, multiple of 32, <= 256
  const float* sinks;
  float scale_log2;  // softmax_scale * log2(e)
  __nv_bfloat16* out;
  float* lse;
  uint32_t* err;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int D, int G, int MODE>
__global__ void __launch_bounds__(128, 1)
window_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v,
                  const WindowParams p) {
  constexpr int TQ = 128 / G;
  constexpr int NSLAB = D / 16;
  static_assert(TQ * G == 128, "tile rows");
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_load, bar_s, bar_o;
  __shared__ uint32_t tmem_base_sh;

  uint8_t* smem = align1024(smem_raw);
  const int nk = p.nk;
  uint8_t* sQ = smem;                       // NSLAB x [128][16]
  uint8_t* sK = sQ + 128 * 32 * NSLAB;      // NSLAB x [nk][16]
  uint8_t* sV = sK + nk * 32 * NSLAB;       // NSLAB x [nk][16]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = blockIdx.y;
  const int tok0 = blockIdx.x * TQ;
  const int kstart = tok0 - p.wl;

  if (threadIdx.x == 0) {
    mbar_init(&bar_load, 1);
    mbar_init(&bar_s, 1);
    mbar_init(&bar_o, 1);
    fence_mbar_init();
    tma_prefetch_map(&tm_q);
    tma_prefetch_map(&tm_k);
    tma_prefetch_map(&tm_v);
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  // ---- producer + S = Q K^T (one thread) --------------------------------
  bool load_ok = true;
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bar_load, (uint32_t)((128 + 2 * nk) * 32 * NSLAB));
#pragma unroll
    for (int s = 0; s < NSLAB; ++s) {
      tma_load_3d(sQ + s * 128 * 32, &tm_q, &bar_load, 16 * s, g * G, tok0);
      tma_load_3d(sK + s * nk * 32, &tm_k, &bar_load, 16 * s, g, kstart);
      tma_load_3d(sV + s * nk * 32, &tm_v, &bar_load, 16 * s, g, kstart);
    }
    load_ok = mbar_wait(&bar_load, 0, p.err, kErrWaitLoad);
    if (load_ok) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(128, nk, false);
#pragma unroll
      for (int s = 0; s < NSLAB; ++s) {
        const uint64_t a = smem_desc(smem_u32(sQ + s * 128 * 32), 16, 256, kLayoutSw32);
        const uint64_t b = smem_desc(smem_u32(sK + s * nk * 32), 16, 256, kLayoutSw32);
        mma_ss(tmem + kColS, a, b, idesc, s > 0 ? 1u : 0u);
      }
      mma_commit(&bar_s);
    } else {
      mbar_arrive(&bar_s);  // release the other warps; results are garbage
    }
  }

  // ---- per-row metadata -------------------------------------------------
  const int row = warp * 32 + lane;  // TMEM lane == M row
  const win::RowMeta r = win::row_meta<G, MODE>(p.cu_seqlens, p.num_seqs, p.total_tokens,
                                                 row, g, tok0, kstart, p.wl, p.wr, p.sinks);
  // Columns any row of this warp can see (before sequence clipping).
  const int wc_lo = (warp * 32) / G;
  const int wc_hi = min((warp * 32 + 31) / G + p.wl + p.wr, nk - 1);
  const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);

  bool s_ok = mbar_wait(&bar_s, 0, p.err, kErrWaitMma);
  __syncwarp();
  tc_fence_after();

  // ---- softmax: P = 2^(x - m) as bf16 into TMEM, row max and sum ----------
  float m, l;
  if constexpr (MODE == SA_SINK_KEY0_BIAS)
    win::key0_bias_in_tmem(lane_base + kColS, r, p.scale_log2);
  win::softmax_rows(lane_base + kColS, lane_base + kColP, nk / 32, wc_lo >> 5, wc_hi >> 5, r,
                    p.scale_log2, m, l);
  tc_fence_before();
  __syncthreads();

  // ---- O = P V (one thread) ----------------------------------------------
  if (threadIdx.x == 0) {
    tc_fence_after();
    if (load_ok) {
      const uint32_t idesc = idesc_bf16(128, D, true);
      for (int kk = 0; kk < nk / 16; ++kk) {
        const uint64_t b = smem_desc(smem_u32(sV + kk * 16 * 32),
                                     (uint32_t)(nk * 32), 256, kLayoutSw32);
        mma_ts(tmem + kColO, tmem + kColP + kk * 8, b, idesc, kk > 0 ? 1u : 0u);
      }
      mma_commit(&bar_o);
    } else {
      mbar_arrive(&bar_o);
    }
  }
  const bool o_ok = mbar_wait(&bar_o, 0, p.err, kErrWaitMma);
  __syncwarp();
  tc_fence_after();

  // ---- epilogue: sink fold, normalise, store O (bf16) and LSE (fp32) ------
  win::epilogue_row<D, MODE>(lane_base + kColO, r, m, l, p.out, p.lse, p.num_q_heads,
                             p.total_tokens);

  // ---- teardown ------------------------------------------------------------
  if (threadIdx.x == 0 && !load_ok) {
    // The copies may still be in flight: give them one more bounded wait.
    mbar_wait(&bar_load, 0, p.err, kErrWaitDrain);
  }
  (void)s_ok;
  (void)o_ok;
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int G, int MODE>
sa_status launch_typed(const WindowArgs& a, int nk) {
  constexpr int TQ = 128 / G;
  CUtensorMap tq, tk, tv;
  const uint64_t dq[3] = {(uint64_t)D, (uint64_t)a.num_q_heads, (uint64_t)a.total_tokens};
  const uint64_t sq[2] = {(uint64_t)D * 2, (uint64_t)a.num_q_heads * D * 2};
  const uint32_t bq[3] = {16, (uint32_t)G, (uint32_t)TQ};
  const uint64_t dk[3] = {(uint64_t)D, (uint64_t)a.num_kv_heads, (uint64_t)a.total_tokens};
  const uint64_t sk[2] = {(uint64_t)D * 2, (uint64_t)a.num_kv_heads * D * 2};
  const uint32_t bk[3] = {16, 1, (uint32_t)nk};
  if (!encode_tiled(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.q, dq, sq, bq,
                    CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_NONE) ||
      !encode_tiled(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.k, dk, sk, bk,
                    CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_NONE) ||
      !encode_tiled(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.v, dk, sk, bk,
                    CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_NONE))
    return SA_ERR_INVALID_ARG;

  WindowParams p;
  p.cu_seqlens = a.cu_seqlens;
  p.num_seqs = a.num_seqs;
  p.total_tokens = (int32_t)a.total_tokens;
  p.num_q_heads = a.num_q_heads;
  p.wl = a.window_left;
  p.wr = a.window_right;
  p.nk = nk;
  p.sinks = a.sinks;
  p.scale_log2 = a.softmax_scale * kLog2e;
  p.out = reinterpret_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.err = device_error_word();

  // At most two CTAs per SM so that two 256-column TMEM allocations fit.
  size_t smem = 1024 + (size_t)(128 + 2 * nk) * D * 2;
  if (smem < 80 * 1024) smem = 80 * 1024;
  auto kern = window_fwd_kernel<D, G, MODE>;
  if (!set_dynamic_smem_once((const void*)kern, (int)smem))
    return fail(SA_ERR_CUDA, "sa_varlen_window_fwd: %s", cudaGetErrorString(cudaGetLastError()));
  cudaError_t e;
  dim3 grid((unsigned)((a.total_tokens + TQ - 1) / TQ), (unsigned)a.num_kv_heads);
  kern<<<grid, 128, smem, a.stream>>>(tq, tk, tv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(SA_ERR_CUDA, "sa_varlen_window_fwd launch: %s", cudaGetErrorString(e));
  return SA_OK;
}

template <int D, int G>
sa_status by_mode(const WindowArgs& a, int nk) {
  switch (a.sink_mode) {
    case SA_SINK_NONE: return launch_typed<D, G, SA_SINK_NONE>(a, nk);
    case SA_SINK_KEY0_BIAS: return launch_typed<D, G, SA_SINK_KEY0_BIAS>(a, nk);
    default: return launch_typed<D, G, SA_SINK_NULL_LOGIT>(a, nk);
  }
}

template <int D>
sa_status by_group(const WindowArgs& a, int G, int nk) {
  switch (G) {
    case 1: return by_mode<D, 1>(a, nk);
    case 2: return by_mode<D, 2>(a, nk);
    case 4: return by_mode<D, 4>(a, nk);
    case 8: return by_mode<D, 8>(a, nk);
    default: return by_mode<D, 16>(a, nk);
  }
}

}  // namespace

sa_status launch_window_fwd(const WindowArgs& a) {
  const int G = a.num_q_heads / a.num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16)
    return fail(SA_ERR_UNSUPPORTED,
                "sa_varlen_window_fwd: num_q_heads / num_kv_heads = %d (supported: 1, 2, 4, 8, 16)", G);
  if (a.head_dim == 64 || a.head_dim == 80 || a.head_dim == 128) {
    sa_status st = SA_OK;
    if (launch_window_ring(a, &st)) return st;
  }
  const int TQ = 128 / G;
  const int span = TQ + a.window_left + a.window_right;
  const int nk = (span + 31) / 32 * 32;
  if (nk > kMaxNK)
    return fail(SA_ERR_UNSUPPORTED,
                "sa_varlen_window_fwd: %d tokens per tile + window %d + %d exceeds 256 keys",
                TQ, a.window_left, a.window_right);
  switch (a.head_dim) {
    case 64: return by_group<64>(a, G, nk);
    case 80: return by_group<80>(a, G, nk);
    case 128: return by_group<128>(a, G, nk);
    default:
      return fail(SA_ERR_UNSUPPORTED,
                  "sa_varlen_window_fwd: head_dim %d (supported: 64, 80, 128)", a.head_dim);
  }
}

}  // namespace sa

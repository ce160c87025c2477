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
// Three kernels, back to back on the stream (the second and third start
// early under programmatic dependent launch and wait for their input):
//  1. plan: one CTA per query compacts the valid entries of its index row
//     (order kept) into the workspace and stores their count c.  A query with
//     c = 0 gets its zero output and LSE = -inf here.
//  2. attend: the compacted list of a query is cut into items of up to 256
//     keys; CTA b takes item b of the order "all full 256-key items (query
//     order), then the shorter last items (query order)", so the long items
//     start first and the CTAs past the last item leave at once.  One CTA
//     per (item, block of 128 heads):
//       S = Q K^T      M = 128 heads, N = item keys (rounded to 16), K = 576
//                      in nine 64-wide slabs;
//       O_half = P V   twice, N = 256 V columns each, K = the item's keys.
//  3. combine: queries with more than one item merge the (O, m, l) partials
//     and fold the sink once.
// A query with a single item is finished by its attend CTA (sink fold, bf16
// O, LSE).
//
// Attend CTA.  Tensor memory: S at columns [0, 256) (P in place, bf16, the A
// operand of P V), O_half at [256, 512).  Shared memory: six 32 KB slots
// R0 R1 R2 R3 K0 K1 of gathered 64-column slabs, 128-byte swizzled (the
// K-major B operand of S, the MN-major B operand of P V), and two 16 KB Q
// slab buffers fed by TMA.  Slabs 0..3 (V columns 0..255) sit in R0..R3;
// slabs 8, 4, 5, 7, 6 stream through K0/K1, so that after S the ring holds
// K0 = slab 6, K1 = slab 7.  After the first P V, slabs 4 and 5 are gathered
// again (from L2) into R2, R3 and the second P V reads R2 R3 K0 K1 = slabs
// 4..7.  Warps 4..7 gather rows with 16-byte cp.async copies; thread 0
// issues the MMAs, thread 32 the Q loads; all eight warps then share the
// softmax and the epilogues (warps w and w + 4 split the columns of the same
// 32 TMEM lanes).
// Split-KV partials are stored heads-fastest ([query][item][column][head],
// the head stride rounded up to 32), so each warp store of the epilogue
// writes 128 contiguous, aligned bytes.
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>
#include <mutex>
#include <utility>

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
constexpr int kItemKeys = 256;
constexpr int kSlotBytes = kItemKeys * 128;  // one gathered slab, 32 KB
constexpr int kNumSlots = 6;                 // R0..R3, K0, K1
constexpr int kSlabBytesQ = 128 * 128;       // one Q slab, 16 KB
constexpr int kTmemCols = 512;
constexpr int kColS = 0;
constexpr int kColO = 256;
constexpr int kMaxSlices = 32;  // topk <= 32 * 256
constexpr int kThreads = 256;

// S step j: slab of Q/K and the slot it sits in (0..3 = R0..R3, 4 = K0,
// 5 = K1).  The ring slabs come first so that the ring refills overlap the
// resident steps.
__device__ __forceinline__ int step_slab(int j) {
  constexpr int kSlab_[9] = {8, 4, 0, 1, 5, 2, 7, 3, 6};
  return kSlab_[j];
}
__device__ __forceinline__ int step_slot(int j) {
  constexpr int kSlot_[9] = {4, 5, 0, 1, 4, 2, 5, 3, 4};
  return kSlot_[j];
}

struct PlanParams {
  const int32_t* indices;  // [nq, topk]
  int32_t topk;
  int64_t num_kv;
  int32_t nq;
  int32_t num_q_heads;
  int32_t* cidx;    // [nq, topk]: valid entries first, in order
  int32_t* qcount;  // [nq]
  __nv_bfloat16* out;
  float* lse;
};

struct IndexParams {
  const float* kv_scale;  // fp8 cache: fp32 scale per latent row (else null)
  const int32_t* cidx;    // compacted index rows [nq, topk]
  const int32_t* qcount;  // valid keys per query
  int32_t topk;
  int32_t nslices;        // items per query at most (= ceil(topk / 256))
  int32_t num_q_heads;
  int32_t nhb;            // blocks of 128 heads
  int32_t nq;
  const float* sinks;
  float scale_log2;
  __nv_bfloat16* out;     // [nq, hq, 512]
  float* lse;             // [hq, nq]
  float* part_o;          // [nq][nslices][512][head_stride]
  float* part_ml;         // [nq][nslices][2][head_stride]  (m, then l)
  int32_t head_stride;    // num_q_heads rounded up to 32
  int32_t combine_min_items;  // the warp-unit combine takes queries with at least this many items
  uint32_t* err;
};

struct __align__(8) IndexSmemCtl {
  uint64_t res_full[4];      // R0..R3 gathered
  uint64_t res2_full;        // slabs 4, 5 gathered over R2, R3
  uint64_t kst_full[2];
  uint64_t kst_empty[2];
  uint64_t q_full[2];
  uint64_t q_empty[2];
  uint64_t s_full;
  uint64_t o_full;           // phase 0: first V half, phase 1: second
  uint32_t tmem_base;
  int32_t item_q, item_s, item_n, item_nitems;
  int32_t scan_f[8], scan_p[8];
  int32_t kidx[kItemKeys];  // the item's key rows
};

// Softmax exchange between the two threads of a row; it lives in the Q slab
// buffers, which are idle once S is complete.
struct IndexRed {
  float m[2][128];
  float l[2][128];
};
// fp8 cache: the item's 256 row scales s_r, then s_r * scale * log2(e),
// follow the reductions
constexpr int kScaleOffset = (int)sizeof(IndexRed);
static_assert(kScaleOffset % 16 == 0 && kScaleOffset + 2 * kItemKeys * 4 <= kSlabBytesQ, "");

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
// Blackwell packed fp32 pair arithmetic (each lane correctly rounded, as the
// scalar instruction) and the three-input maximum.
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
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
__device__ __forceinline__ void bar_gather() {  // the four gatherer warps only
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Block-wide exclusive prefix sum of x over the 256 threads; *total gets the
// sum.  `scratch` holds 8 ints.  Contains two __syncthreads.
__device__ __forceinline__ int block_exclusive_sum(int x, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = x;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, d);
    if (lane >= d) inc += y;
  }
  if (lane == 31) scratch[warp] = inc;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const int t = scratch[w];
    before += (w < warp) ? t : 0;
    all += t;
  }
  __syncthreads();
  *total = all;
  return before + inc - x;
}

// ---------------------------------------------------------------------------
// 1. plan
__global__ void __launch_bounds__(kThreads)
sparse_index_plan_kernel(const PlanParams p) {
  griddep_launch_dependents();
  __shared__ int32_t s_cnt[kMaxSlices * 8];
  __shared__ int32_t s_pre[kMaxSlices * 8];
  __shared__ int32_t s_scan[8];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = blockIdx.x;
  const int32_t* row = p.indices + (int64_t)q * p.topk;
  // the whole row first: every load independent
  int32_t v[kMaxSlices];
#pragma unroll
  for (int c = 0; c < kMaxSlices; ++c) {
    const int e = c * kThreads + tid;
    v[c] = e < p.topk ? __ldg(row + e) : -1;
  }
#pragma unroll
  for (int c = 0; c < kMaxSlices; ++c) {
    const bool ok = v[c] >= 0 && (int64_t)v[c] < p.num_kv;
    const uint32_t bal = __ballot_sync(0xffffffffu, ok);
    if (lane == 0) s_cnt[c * 8 + warp] = __popc(bal);
  }
  __syncthreads();
  // entry tid of s_cnt is (chunk tid / 8, warp tid % 8): row order
  int total = 0;
  s_pre[tid] = block_exclusive_sum(s_cnt[tid], s_scan, &total);
  __syncthreads();
  const uint32_t lt = (1u << lane) - 1u;
  int32_t* crow = p.cidx + (int64_t)q * p.topk;
#pragma unroll
  for (int c = 0; c < kMaxSlices; ++c) {
    const bool ok = v[c] >= 0 && (int64_t)v[c] < p.num_kv;
    const uint32_t bal = __ballot_sync(0xffffffffu, ok);
    if (ok) crow[s_pre[c * 8 + warp] + __popc(bal & lt)] = v[c];
  }
  if (tid == 0 && p.qcount) p.qcount[q] = total;
  if (total == 0) {
    // empty key set: zero output, LSE = -inf
    uint4* dst = reinterpret_cast<uint4*>(p.out + (int64_t)q * p.num_q_heads * kDv);
    for (int i = tid; i < p.num_q_heads * (kDv / 8); i += kThreads) dst[i] = make_uint4(0, 0, 0, 0);
    for (int h = tid; h < p.num_q_heads; h += kThreads) p.lse[(int64_t)h * p.nq + q] = -INFINITY;
  }
}

// ---------------------------------------------------------------------------
// 2. attend

// Item `item` of the global order (see the file header) -> ctl.item_*; q = -1
// past the last item.  All 256 threads take part.  Thread t owns queries
// [t K, t K + K), K = ceil(nq / 256).
__device__ void find_item(const IndexParams& p, int item, IndexSmemCtl& ctl) {
  const int tid = threadIdx.x;
  const int K = (p.nq + kThreads - 1) / kThreads;
  const int q0 = tid * K;
  int cache[4];
  int nfull = 0, npart = 0;
  for (int i = 0; i < K; ++i) {
    const int qq = q0 + i;
    const int c = qq < p.nq ? __ldcg(p.qcount + qq) : 0;
    if (i < 4) cache[i & 3] = c;
    nfull += c / kItemKeys;
    npart += (c % kItemKeys) != 0 ? 1 : 0;
  }
  if (tid == 0) ctl.item_q = -1;
  int tot_f = 0, tot_p = 0;
  const int pre_f = block_exclusive_sum(nfull, ctl.scan_f, &tot_f);
  const int pre_p = block_exclusive_sum(npart, ctl.scan_p, &tot_p);
  const bool heavy = item < tot_f;
  const int target = heavy ? item : item - tot_f;
  const int pre = heavy ? pre_f : pre_p;
  const int mine = heavy ? nfull : npart;
  if ((heavy || target < tot_p) && pre <= target && target < pre + mine) {
    int acc = pre;
    for (int i = 0; i < K; ++i) {
      const int qq = q0 + i;
      const int c = i < 4 ? cache[i & 3] : __ldcg(p.qcount + qq);
      const int f = c / kItemKeys, r = c % kItemKeys;
      const int here = heavy ? f : (r != 0 ? 1 : 0);
      if (target < acc + here) {
        ctl.item_q = qq;
        ctl.item_s = heavy ? target - acc : f;
        ctl.item_n = heavy ? kItemKeys : r;
        ctl.item_nitems = f + (r != 0 ? 1 : 0);
        break;
      }
      acc += here;
    }
  }
  __syncthreads();
}

// fp8 cache: e4m3 bytes (b_lo, b_hi) of word w, picked by `sel`, as a bf16
// pair.  prmt puts each byte over its sign byte; shifted left by 4 and masked,
// that is the bf16 encoding of value * 2^-120 (sign, 4 exponent bits, 3
// mantissa bits; e4m3 subnormals and zero land on bf16 subnormals and zero),
// and the bf16 multiply by 2^120 gives the value exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t w, uint32_t sel) {
  uint32_t x;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(x) : "r"(w), "r"(sel));
  x = (x << 4) & 0x87f087f0u;
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(0x7B807B80u));  // 2^120
  return r;
}

// fp8 cache, stage 1: the 64 e4m3 columns of slab `slab` of rows r0 + 32 k
// (< npad) go, 16 bytes per (row, chunk c4), into the upper half of the 32 KB
// slot at dst (row r at dst + 16 KB + 64 r); rows past n are zero-filled.
__device__ __noinline__ void stage_slab_fp8(uint32_t dst, const uint8_t* kv8,
                                               const int32_t* kidx, int npad, int n, int r0,
                                               int c4, int slab) {
#pragma unroll
  for (int k = 0; k < kItemKeys / 32; ++k) {
    const int r = r0 + 32 * k;
    if (r < npad) {
      const bool live = r < n;
      const uint8_t* src = kv8 + (live ? (int64_t)kidx[r] * kDqk + slab * kSlab + c4 * 16 : 0);
      cp_async16(dst + kItemKeys * 64 + r * 64 + c4 * 16, src, live ? 16u : 0u);
    }
  }
}

// fp8 cache, stage 2 (after the staged copies landed): read this thread's
// staged chunks, wait for every gatherer (bf16 rows 128.. overwrite the
// staging half), then write the values as bf16 chunks 2 c4 and 2 c4 + 1 of
// each row of the slot's 128-byte-swizzled [npad][64] layout.  The row scales
// are not applied here: the softmax multiplies them into the logits and P.
// Not inlined (nor the stage above): one copy of the code serves the eleven
// call sites, each run once per CTA, so it stays in the instruction cache.
__device__ __noinline__ void convert_slab_fp8(uint32_t dst, int npad, int r0, int c4) {
  uint4 raw[kItemKeys / 32];
#pragma unroll
  for (int k = 0; k < kItemKeys / 32; ++k) {
    const int r = r0 + 32 * k;
    if (r < npad) {
      const uint32_t a = dst + kItemKeys * 64 + r * 64 + c4 * 16;
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(raw[k].x), "=r"(raw[k].y), "=r"(raw[k].z), "=r"(raw[k].w)
                   : "r"(a));
    }
  }
  bar_gather();
#pragma unroll
  for (int k = 0; k < kItemKeys / 32; ++k) {
    const int r = r0 + 32 * k;
    if (r < npad) {
      const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        o[2 * i] = e4m3x2_to_bf16x2(w[i], 0x9180u);      // bytes 0, 1
        o[2 * i + 1] = e4m3x2_to_bf16x2(w[i], 0xB3A2u);  // bytes 2, 3
      }
      const uint32_t row = dst + r * 128;
      const uint32_t a0 = row + (((2 * c4) ^ (r & 7)) << 4);
      const uint32_t a1 = row + (((2 * c4 + 1) ^ (r & 7)) << 4);
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a0), "r"(o[0]), "r"(o[1]),
                   "r"(o[2]), "r"(o[3])
                   : "memory");
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a1), "r"(o[4]), "r"(o[5]),
                   "r"(o[6]), "r"(o[7])
                   : "memory");
    }
  }
}

// Gather 16-byte chunk c of slab `slab` of rows r0, r0 + 16, ... (< npad) into
// the 128-byte-swizzled [npad][64] slot at dst; rows past n are zero-filled.
__device__ __forceinline__ void gather_slab(uint32_t dst, const uint16_t* kv,
                                            const int32_t* kidx, int iters, int n, int r0,
                                            int c, int slab) {
#pragma unroll 4
  for (int k = 0; k < iters; ++k) {
    const int r = r0 + 16 * k;
    const bool live = r < n;
    const uint16_t* src = kv + (live ? (int64_t)kidx[r] * kDqk + slab * kSlab + c * 8 : 0);
    cp_async16(dst + r * 128 + ((c ^ (r & 7)) << 4), src, live ? 16u : 0u);
  }
}

template <int MODE, bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
sparse_index_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const void* kv_raw,
                        const IndexParams p) {
  // bf16 cache: rows of 576 bf16; fp8 cache: rows of 576 e4m3 bytes
  const uint16_t* kv = reinterpret_cast<const uint16_t*>(kv_raw);
  const uint8_t* kv8 = reinterpret_cast<const uint8_t*>(kv_raw);
  extern __shared__ uint8_t smem_raw[];
  __shared__ IndexSmemCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_slot = smem;                             // 6 x 32 KB
  uint8_t* s_qst = s_slot + kNumSlots * kSlotBytes;   // 2 x 16 KB
  auto slot_u32 = [&](int s) { return smem_u32(s_slot + s * kSlotBytes); };
  IndexRed& red = *reinterpret_cast<IndexRed*>(s_qst);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  griddep_launch_dependents();

  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(&ctl.res_full[i], 128);
    mbar_init(&ctl.res2_full, 128);
    for (int s2 = 0; s2 < 2; ++s2) {
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
  griddep_wait();  // the plan kernel's counts and lists are complete
  find_item(p, (int)(blockIdx.x / p.nhb), ctl);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const int q = ctl.item_q;

  if (q >= 0) {
    const int hb = blockIdx.x % p.nhb;
    const int slice = ctl.item_s;
    const int n = ctl.item_n;
    const bool direct = ctl.item_nitems == 1;  // this CTA writes the final output
    const int npad = (n + 15) & ~15;           // MMA N and gathered rows
    const int part = tid >> 7;                 // column half of the softmax / epilogue
    const int row = tid & 127;                 // head row = TMEM lane
    const int h = hb * 128 + row;
    const bool row_valid = h < p.num_q_heads;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    bool ok = true;

    // gatherers (warps 4..7): thread gt copies 16-byte chunk gc of rows
    // gr0 + 16 k of every slab
    const int gt = tid - 128;
    const int gr0 = (gt >> 3) & 15, gc = gt & 7;
    const int fr0 = gt >> 2, fc4 = gt & 3;  // fp8 cache: rows fr0 + 32 k, 16-byte chunk fc4
    const int iters = npad >> 4;
    float ks0 = 0.f, ks1 = 0.f;
    if (warp >= 4) {
      const int32_t* crow = p.cidx + (int64_t)q * p.topk + slice * kItemKeys;
      const int32_t i0 = gt < n ? __ldcg(crow + gt) : 0;
      const int32_t i1 = gt + 128 < n ? __ldcg(crow + gt + 128) : 0;
      ctl.kidx[gt] = i0;
      ctl.kidx[gt + 128] = i1;
      if (FP8) {  // stored once S is complete (they go where Q was staged)
        ks0 = gt < n ? __ldg(p.kv_scale + i0) : 0.f;
        ks1 = gt + 128 < n ? __ldg(p.kv_scale + i1) : 0.f;
      }
      bar_gather();
    }

    if (warp >= 4) {
      auto gather = [&](int slot, int slab) {
        if (ok) {
          if (FP8) stage_slab_fp8(slot_u32(slot), kv8, ctl.kidx, npad, n, fr0, fc4, slab);
          else gather_slab(slot_u32(slot), kv, ctl.kidx, iters, n, gr0, gc, slab);
        }
        cp_async_commit();
      };
      // the slot's copies have landed: (fp8: convert it, then) hand it over
      auto publish_slot = [&](uint64_t* bar, int slot) {
        if (FP8) convert_slab_fp8(slot_u32(slot), npad, fr0, fc4);
        fence_proxy_async();
        mbar_arrive(bar);
      };
      gather(4, 8);  // G0 -> K0
      gather(5, 4);  // G1 -> K1
      gather(0, 0);  // G2
      gather(1, 1);  // G3
      gather(2, 2);  // G4
      gather(3, 3);  // G5
      // the ring refills (slabs 5, 6, 7) wait for free slots: start their
      // DRAM reads now so that the copies find them in L2
      for (int r = gt; r < n; r += 128) {
        const int64_t row = (int64_t)ctl.kidx[r] * kDqk;
        if (FP8) {  // bytes [320, 512): every 128-byte line holds one of these
          prefetch_l2(kv8 + row + 5 * kSlab);
          prefetch_l2(kv8 + row + 7 * kSlab);
          prefetch_l2(kv8 + row + 8 * kSlab - 1);
        } else {
          prefetch_l2(kv + row + 5 * kSlab);
          prefetch_l2(kv + row + 6 * kSlab);
          prefetch_l2(kv + row + 7 * kSlab);
        }
      }
      cp_async_wait<5>();
      publish_slot(&ctl.kst_full[0], 4);
      cp_async_wait<4>();
      publish_slot(&ctl.kst_full[1], 5);
      cp_async_wait<3>();
      publish_slot(&ctl.res_full[0], 0);
      if (ok) ok = mbar_wait(&ctl.kst_empty[0], 0, p.err, kErrWaitFree);  // step 0 done
      gather(4, 5);  // G6
      cp_async_wait<3>();
      publish_slot(&ctl.res_full[1], 1);
      if (ok) ok = mbar_wait(&ctl.kst_empty[1], 0, p.err, kErrWaitFree);  // step 1 done
      gather(5, 7);  // G7
      cp_async_wait<3>();
      publish_slot(&ctl.res_full[2], 2);
      cp_async_wait<2>();
      publish_slot(&ctl.res_full[3], 3);
      cp_async_wait<1>();
      publish_slot(&ctl.kst_full[0], 4);  // slab 5
      if (ok) ok = mbar_wait(&ctl.kst_empty[0], 1, p.err, kErrWaitFree);  // step 4 done
      gather(4, 6);  // G8
      cp_async_wait<1>();
      publish_slot(&ctl.kst_full[1], 5);  // slab 7
      cp_async_wait<0>();
      publish_slot(&ctl.kst_full[0], 4);  // slab 6
    } else if (tid == 0) {
      // ---- S = Q K^T, nine slab steps -------------------------------------
      const uint32_t idesc = idesc_bf16(128, npad, false);
      for (int j = 0; j < kNumQkSlabs && ok; ++j) {
        const int st = j & 1;
        const int slot = step_slot(j);
        ok = mbar_wait(&ctl.q_full[st], (j >> 1) & 1, p.err, kErrWaitLoad);
        if (ok) {
          if (slot < 4) {
            ok = mbar_wait(&ctl.res_full[slot], 0, p.err, kErrWaitLoad);
          } else {
            // K0 fills are consumed at steps 0, 4, 8; K1 fills at 1, 6
            const uint32_t par = slot == 4 ? (j == 4 ? 1u : 0u) : (j == 6 ? 1u : 0u);
            ok = mbar_wait(&ctl.kst_full[slot - 4], par, p.err, kErrWaitLoad);
          }
        }
        if (!ok) break;
        tc_fence_after();
        const uint32_t kb = slot_u32(slot);
        const uint32_t qb = smem_u32(s_qst + st * kSlabBytesQ);
#pragma unroll
        for (int kk = 0; kk < kSlab / 16; ++kk) {
          const uint64_t a = smem_desc(qb + kk * 32, 16, 1024, kLayoutSw128);
          const uint64_t b = smem_desc(kb + kk * 32, 16, 1024, kLayoutSw128);
          mma_ss(tmem + kColS, a, b, idesc, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&ctl.q_empty[st]);
        if (j == 0 || j == 4) mma_commit(&ctl.kst_empty[0]);
        if (j == 1) mma_commit(&ctl.kst_empty[1]);
      }
      if (ok) mma_commit(&ctl.s_full);
      else mbar_arrive(&ctl.s_full);
    } else if (tid == 32) {
      // ---- Q slab of each S step by TMA through a two-stage ring ----------
      tma_prefetch_map(&tm_q);
      const int qrow0 = q * p.num_q_heads + hb * 128;
      int issued = 0;
      for (int j = 0; j < kNumQkSlabs; ++j) {
        const int st = j & 1;
        if (j >= 2 && !mbar_wait(&ctl.q_empty[st], ((j >> 1) - 1) & 1, p.err, kErrWaitFree))
          break;
        mbar_arrive_expect_tx(&ctl.q_full[st], kSlabBytesQ);
        tma_load_2d(s_qst + st * kSlabBytesQ, &tm_q, &ctl.q_full[st], step_slab(j) * kSlab, qrow0);
        ++issued;
      }
      // bounded drain of the last copies (immediate once the MMAs consumed them)
      for (int j = max(0, issued - 2); j < issued; ++j)
        mbar_wait(&ctl.q_full[j & 1], (j >> 1) & 1, p.err, kErrWaitDrain);
    }

    // ---- softmax: thread (row, part) takes key columns [128 part, +128) ----
    const float sink2 = (MODE != SA_SINK_NONE && row_valid) ? __ldg(p.sinks + h) * kLog2e : 0.f;
    ok = mbar_wait(&ctl.s_full, 0, p.err, kErrWaitMma) && ok;
    // fp8 cache: the row scales, after the reductions in the Q staging area
    // (free once S is complete)
    float* s_ks = reinterpret_cast<float*>(s_qst + kScaleOffset);
    float* s_kc = s_ks + kItemKeys;
    if (FP8) {
      if (warp >= 4) {
        // keys past n: scale 0 (P = 0) and logit factor 1 (their -inf mask
        // must not meet a zero factor)
        s_ks[gt] = ks0;
        s_ks[gt + 128] = ks1;
        s_kc[gt] = gt < n ? ks0 * p.scale_log2 : 1.f;
        s_kc[gt + 128] = gt + 128 < n ? ks1 * p.scale_log2 : 1.f;
      }
      __syncthreads();
    }
    __syncwarp();
    tc_fence_after();
    const float c2 = p.scale_log2;
    // fp8 cache: S holds q . e_r for the unscaled row e_r; the log2-domain
    // logit is (q . e_r) * kc_r with kc_r = s_r * scale * log2(e).
    auto load32 = [&](const float* src, float* dst) {
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 t = *reinterpret_cast<const float4*>(src + e);
        dst[e] = t.x;
        dst[e + 1] = t.y;
        dst[e + 2] = t.z;
        dst[e + 3] = t.w;
      }
    };
    const int k0 = part * 128;
    const int nch = (min(max(npad - k0, 0), 128) + 31) >> 5;
    {
      // pass 1: row max over this thread's keys (keys past n masked)
      float mr[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
      for (int ch = 0; ch < nch; ++ch) {
        float v[32];
        tmem_ld32(lane_base + kColS + k0 + 32 * ch, v);
        tmem_wait_ld();
        const int c0 = k0 + 32 * ch;
        if (FP8) {
          float kc[32];
          load32(s_kc + c0, kc);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const uint64_t t = f2_fma(f2_pack(v[e], v[e + 1]), f2_pack(kc[e], kc[e + 1]),
                                      f2_pack(-0.f, -0.f));
            v[e] = f2_lo(t);
            v[e + 1] = f2_hi(t);
          }
        }
        if (c0 + 32 > n) {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = (c0 + e < n) ? v[e] : -INFINITY;
        }
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          mr[0] = max3f(mr[0], v[e + 0], v[e + 1]);
          mr[1] = max3f(mr[1], v[e + 2], v[e + 3]);
          mr[2] = max3f(mr[2], v[e + 4], v[e + 5]);
          mr[3] = max3f(mr[3], v[e + 6], v[e + 7]);
        }
      }
      red.m[part][row] = fmaxf(fmaxf(mr[0], mr[1]), fmaxf(mr[2], mr[3]));
    }
    __syncthreads();
    // max(s) * c2 == max(s * c2) exactly (c2 > 0, rounding is monotone); the
    // fp8 maxima are already in the log2 domain
    const float m = fmaxf(red.m[0][row], red.m[1][row]) * (FP8 ? 1.f : c2);
    {
      // pass 2: P = 2^(s c2 - m) (bf16, written over S: key columns [k0, k0 +
      // 128) go to TMEM columns [k0, k0 + 64), inside this thread's half) and
      // the row sum
      const uint64_t c2c2 = f2_pack(c2, c2), nmnm = f2_pack(-m, -m);
      uint64_t lp[4] = {0, 0, 0, 0};
#pragma unroll 1
      for (int ch = 0; ch < nch; ++ch) {
        float v[32];
        tmem_ld32(lane_base + kColS + k0 + 32 * ch, v);
        tmem_wait_ld();
        const int c0 = k0 + 32 * ch;
        float ks[32], kc[32];
        if (FP8) {
          load32(s_kc + c0, kc);
          load32(s_ks + c0, ks);
        }
        if (c0 + 32 > n) {  // 2^(-inf) = 0 for keys past n
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = (c0 + e < n) ? v[e] : -INFINITY;
        }
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const uint64_t t = f2_fma(f2_pack(v[e], v[e + 1]),
                                    FP8 ? f2_pack(kc[e], kc[e + 1]) : c2c2, nmnm);
          const float x0 = ex2_approx(f2_lo(t)), x1 = ex2_approx(f2_hi(t));
          lp[(e >> 1) & 3] = f2_add(lp[(e >> 1) & 3], f2_pack(x0, x1));
          // fp8 cache: P V takes the unscaled rows, so P carries s_r
          if (FP8) {
            const uint64_t w = f2_fma(f2_pack(x0, x1), f2_pack(ks[e], ks[e + 1]),
                                      f2_pack(-0.f, -0.f));
            pk[e >> 1] = pack_bf16x2(f2_lo(w), f2_hi(w));
          } else {
            pk[e >> 1] = pack_bf16x2(x0, x1);
          }
        }
        tmem_st16(lane_base + kColS + k0 + 16 * ch, pk);
      }
      const uint64_t s01 = f2_add(lp[0], lp[1]), s23 = f2_add(lp[2], lp[3]);
      const uint64_t s = f2_add(s01, s23);
      red.l[part][row] = f2_lo(s) + f2_hi(s);
    }
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();
    const float l = red.l[0][row] + red.l[1][row];
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

    // ---- O_half = P V_half (thread 0), then the epilogue of that half ------
    auto issue_pv = [&](int first_slot) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(128, 256, true);
      const uint32_t vb = slot_u32(first_slot);
      for (int kk = 0; kk < npad / 16; ++kk) {
        // P of keys [16 kk, 16 kk + 16): TMEM column 8 kk (keys < 128) or
        // 128 + 8 (kk - 8)
        const uint32_t pa = tmem + kColS + (kk < 8 ? kk * 8 : 128 + (kk - 8) * 8);
        const uint64_t b = smem_desc(vb + kk * 16 * 128, kSlotBytes, 1024, kLayoutSw128);
        mma_ts(tmem + kColO, pa, b, idesc, kk > 0 ? 1u : 0u);
      }
      mma_commit(&ctl.o_full);
    };
    if (tid == 0) {
      if (ok) issue_pv(0);
      else mbar_arrive(&ctl.o_full);
    }
    const int64_t hq = p.num_q_heads;
    auto epilogue = [&](int half) {
      const int col0 = half * 256 + part * 128;  // V column of this thread's first value
      __nv_bfloat16* orow = p.out + ((int64_t)q * hq + h) * kDv + col0;
      const int64_t hs = p.head_stride;
      float* pcol = p.part_o + (((int64_t)q * p.nslices + slice) * kDv + col0) * hs + h;
#pragma unroll 1
      for (int jj = 0; jj < 4; ++jj) {
        float o[32];
        tmem_ld32(lane_base + kColO + part * 128 + 32 * jj, o);
        tmem_wait_ld();
        if (row_valid && direct) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint4 w;
            w.x = pack_bf16x2(o[8 * g + 0] * inv, o[8 * g + 1] * inv);
            w.y = pack_bf16x2(o[8 * g + 2] * inv, o[8 * g + 3] * inv);
            w.z = pack_bf16x2(o[8 * g + 4] * inv, o[8 * g + 5] * inv);
            w.w = pack_bf16x2(o[8 * g + 6] * inv, o[8 * g + 7] * inv);
            *reinterpret_cast<uint4*>(orow + 32 * jj + 8 * g) = w;
          }
        } else if (row_valid) {
#pragma unroll
          for (int e = 0; e < 32; ++e) pcol[(int64_t)(32 * jj + e) * hs] = o[e];
        }
      }
    };
    ok = mbar_wait(&ctl.o_full, 0, p.err, kErrWaitMma) && ok;
    __syncwarp();
    tc_fence_after();
    if (warp >= 4) {
      // slabs 4, 5 over R2, R3 (the first P V has read them), landing while
      // the first half is stored
      if (ok) {
        if (FP8) {
          stage_slab_fp8(slot_u32(2), kv8, ctl.kidx, npad, n, fr0, fc4, 4);
          stage_slab_fp8(slot_u32(3), kv8, ctl.kidx, npad, n, fr0, fc4, 5);
        } else {
          gather_slab(slot_u32(2), kv, ctl.kidx, iters, n, gr0, gc, 4);
          gather_slab(slot_u32(3), kv, ctl.kidx, iters, n, gr0, gc, 5);
        }
      }
      cp_async_commit();
      epilogue(0);
      cp_async_wait<0>();
      if (FP8) {
        convert_slab_fp8(slot_u32(2), npad, fr0, fc4);
        convert_slab_fp8(slot_u32(3), npad, fr0, fc4);
      }
      fence_proxy_async();
      mbar_arrive(&ctl.res2_full);
    } else {
      epilogue(0);
    }
    tc_fence_before();
    __syncthreads();  // every TMEM read of the first half is done
    if (tid == 0) {
      tc_fence_after();
      if (ok && mbar_wait(&ctl.res2_full, 0, p.err, kErrWaitLoad)) issue_pv(2);
      else mbar_arrive(&ctl.o_full);
    }
    ok = mbar_wait(&ctl.o_full, 1, p.err, kErrWaitMma) && ok;
    __syncwarp();
    tc_fence_after();
    epilogue(1);
    if (row_valid && part == 0) {
      if (direct) {
        p.lse[(int64_t)h * p.nq + q] = (m + log2f(l)) * kLn2;
      } else {
        float* ml = p.part_ml + ((int64_t)q * p.nslices + slice) * 2 * p.head_stride + h;
        ml[0] = m;
        ml[p.head_stride] = l;
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

// ---------------------------------------------------------------------------
// 3a. combine of queries with 2..8 items, TMA-fed.  Units of (query, 16 V
// columns, 128 heads) are dealt round-robin to one CTA per SM; a CTA keeps
// three units in flight.  Thread 0 loads a unit with two TMA copies on its
// mbarrier: the [8 items][16 columns][128 heads] fp32 O box of a 3-D view of
// the partials and the [8 items x (m, l)][128 heads] box of a 2-D view of
// the (m, l) rows (items past the query's last are loaded and ignored), so a
// CTA has ~200 KB of reads outstanding without holding any of it in
// registers and without paying one copy instruction per item.  Thread t then
// merges head t mod 128, columns 8 (t / 128) .. + 8 from shared memory (the
// formula of the warp-unit combine below).
constexpr int kFcCols = 16;
constexpr int kFcMaxItems = 8;
constexpr int kFcStages = 3;
constexpr int kFcList = 1024;  // queries listed per round

struct __align__(128) FcStage {
  float o[kFcMaxItems][kFcCols][128];  // row stride: the tile's head count
  float ml[kFcMaxItems][2][128];
};

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
sparse_index_combine_tma_kernel(const __grid_constant__ CUtensorMap tm_part,
                                const __grid_constant__ CUtensorMap tm_part1,
                                const __grid_constant__ CUtensorMap tm_ml, const IndexParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[kFcStages];
  __shared__ int32_t s_q[kFcList];
  __shared__ int32_t s_ns[kFcList];
  __shared__ int32_t s_scan[8];
  __shared__ int32_t s_ok;
  FcStage* stage = reinterpret_cast<FcStage*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int i = 0; i < kFcStages; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
    s_ok = 1;
    tma_prefetch_map(&tm_part);
    tma_prefetch_map(&tm_part1);
    tma_prefetch_map(&tm_ml);
  }
  __syncthreads();
  griddep_wait();  // the attend kernel's partials are complete
  const int64_t hs = p.head_stride;
  const int bi = hs < 128 ? (int)hs : 128;  // heads per tile row
  const int units_per_q = (kDv / kFcCols) * p.nhb;
  const int64_t G = gridDim.x;
  const int h = tid & 127, half = tid >> 7;
  uint32_t phase = 0;
  int64_t unit_base = 0;
  for (int qb = 0; qb < p.nq; qb += kFcList) {
    int nact = 0;
    for (int r = 0; r < kFcList; r += kThreads) {
      const int qq = qb + r + tid;
      const int c = qq < p.nq ? __ldcg(p.qcount + qq) : 0;
      const int ns = (c + kItemKeys - 1) / kItemKeys;
      const int act = ns >= 2 && ns <= kFcMaxItems ? 1 : 0;
      int tot = 0;
      const int pos = block_exclusive_sum(act, s_scan, &tot);
      if (act) {
        s_q[nact + pos] = qq;
        s_ns[nact + pos] = ns;
      }
      nact += tot;
    }
    __syncthreads();
    const int64_t nunits = (int64_t)nact * units_per_q;
    int64_t first = ((int64_t)blockIdx.x - unit_base) % G;
    if (first < 0) first += G;
    const int64_t mine = first < nunits ? (nunits - first + G - 1) / G : 0;
    auto unit_of = [&](int64_t k, int& q, int& ns, int& colblk, int& hb) {
      const int64_t u = first + k * G;
      const int a = (int)(u / units_per_q);
      const int r = (int)(u % units_per_q);
      q = s_q[a];
      ns = s_ns[a];
      colblk = r % (kDv / kFcCols);
      hb = r / (kDv / kFcCols);
    };
    auto issue = [&](int64_t k, int st) {
      int q, ns, colblk, hb;
      unit_of(k, q, ns, colblk, hb);
      // full boxes (out-of-range parts zero-filled) count in the transaction;
      // up to four items one box each, more in one eight-item box
      const int nbox = ns <= 4 ? ns : kFcMaxItems;
      mbar_arrive_expect_tx(&full[st], (uint32_t)((nbox * kFcCols + 2 * kFcMaxItems) * bi * 4));
      if (ns <= 4) {
        for (int s = 0; s < ns; ++s)
          tma_load_3d(&stage[st].o[0][0][0] + s * kFcCols * bi, &tm_part1, &full[st], hb * 128,
                      colblk * kFcCols, q * p.nslices + s);
      } else {
        tma_load_3d(&stage[st].o[0][0][0], &tm_part, &full[st], hb * 128, colblk * kFcCols,
                    q * p.nslices);
      }
      tma_load_2d(&stage[st].ml[0][0][0], &tm_ml, &full[st], hb * 128, q * p.nslices * 2);
    };
    if (tid == 0)
      for (int64_t k = 0; k < mine && k < kFcStages; ++k) issue(k, (int)k);
    for (int64_t k = 0; k < mine; ++k) {
      if (!s_ok) break;  // a load never arrived (error recorded): stop
      const int st = (int)(k % kFcStages);
      int q, ns, colblk, hb;
      unit_of(k, q, ns, colblk, hb);
      if (!mbar_wait(&full[st], (phase >> st) & 1u, p.err, kErrWaitLoad)) s_ok = 0;
      phase ^= 1u << st;
      const FcStage& S = stage[st];
      const int head = hb * 128 + h;
      if (head < p.num_q_heads) {
        // every item has at least one key, so every l > 0
        // box rows: item s has m at row 2 s and l at row 2 s + 1
        const float* mlt = &S.ml[0][0][0];
        float M = -INFINITY;
#pragma unroll
        for (int s = 0; s < kFcMaxItems; ++s)
          if (s < ns) M = fmaxf(M, mlt[(2 * s) * bi + h]);
        float L = 0.f, w[kFcMaxItems];
#pragma unroll
        for (int s = 0; s < kFcMaxItems; ++s) {
          w[s] = s < ns ? ex2_approx(mlt[(2 * s) * bi + h] - M) : 0.f;
          L = fmaf(s < ns ? mlt[(2 * s + 1) * bi + h] : 0.f, w[s], L);
        }
        float den = L, alpha = 1.f;
        if (MODE == SA_SINK_NULL_LOGIT) {
          const float sink2 = __ldg(p.sinks + head) * kLog2e;
          const float mp = fmaxf(M, sink2);
          alpha = ex2_approx(M - mp);
          den = L * alpha + ex2_approx(sink2 - mp);
        }
        const float inv = alpha / den;
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        const float* ot = &S.o[0][0][0];
#pragma unroll
        for (int s = 0; s < kFcMaxItems; ++s) {
          if (s < ns) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              acc[e] = fmaf(w[s], ot[(s * kFcCols + half * 8 + e) * bi + h], acc[e]);
          }
        }
        uint4 pk;
        pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        pk.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        pk.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
        pk.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
        *reinterpret_cast<uint4*>(p.out + ((int64_t)q * p.num_q_heads + head) * kDv +
                                  colblk * kFcCols + half * 8) = pk;
        if (colblk == 0 && half == 0) p.lse[(int64_t)head * p.nq + q] = (M + log2f(L)) * kLn2;
      }
      __syncthreads();  // stage st is consumed
      if (tid == 0 && s_ok && k + kFcStages < mine) issue(k + kFcStages, st);
    }
    unit_base += nunits;
    __syncthreads();  // the lists are rewritten by the next round
  }
}

// ---------------------------------------------------------------------------
// 3b. combine: merge the (O, m, l) partials of queries with more than one item
// and fold the sink once:
//   O = sum_s 2^(m_s - M) O_s * alpha / (L alpha + 2^(s_h log2e - M')),
//   M = max m_s, L = sum_s l_s 2^(m_s - M), M' = max(M, s_h log2e),
//   alpha = 2^(M - M'), LSE = (M + log2 L) ln 2 over the listed keys only.
// The work is cut into warp units of (query, 8 V columns, 32 heads), walked
// round-robin by every warp of a grid of a few CTAs per SM.  Each CTA lists
// the multi-item queries itself (256 queries at a time, in shared memory), so
// no warp is spent on a query that needs no merge.  In a unit, lane i loads
// the (m, l) of head i and lane (g, c) -- g = lane mod 8, c = lane / 8 -- the
// O of heads 4 g .. + 4, columns 2 c, 2 c + 1 as float4s (eight lanes read 128
// contiguous bytes), all in one batch; the weights meet the O values through
// a warp-private table in shared memory, and the bf16 result goes through a
// warp-private buffer so that each lane stores one 16-byte row segment.
constexpr int kCombineCols = 8;
constexpr int kCombineGroup = 8;
constexpr int kCombineWarps = kThreads / 32;

struct CombineSmem {
  float w[kCombineWarps][kMaxSlices][32];  // 2^(m_s - M) per item and head
  float inv[kCombineWarps][32];            // alpha / denominator per head
  __nv_bfloat16 o[kCombineWarps][32][kCombineCols];
  int32_t q[kThreads];
  int32_t ns[kThreads];
  int32_t scan[8];
};

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
sparse_index_combine_kernel(const IndexParams p) {
  __shared__ __align__(16) CombineSmem sm;
  griddep_wait();  // the attend kernel's partials are complete
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t hs = p.head_stride;
  const int64_t nwarps = (int64_t)gridDim.x * kCombineWarps;
  const int64_t gw = (int64_t)blockIdx.x * kCombineWarps + warp;
  const int ncolblk = kDv / kCombineCols;
  const int units_per_q = ncolblk * (p.head_stride / 32);
  const int g = lane & 7, cpair = lane >> 3;
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  int64_t unit_base = 0;  // units of the earlier query chunks
  for (int qb = 0; qb < p.nq; qb += kThreads) {
    const int qq = qb + tid;
    const int c = qq < p.nq ? __ldcg(p.qcount + qq) : 0;
    const int ns_q = (c + kItemKeys - 1) / kItemKeys;
    const int act = ns_q >= 2 && ns_q >= p.combine_min_items ? 1 : 0;
    int nact = 0;
    const int pos = block_exclusive_sum(act, sm.scan, &nact);
    if (act) {
      sm.q[pos] = qq;
      sm.ns[pos] = ns_q;
    }
    __syncthreads();
    const int64_t nunits = (int64_t)nact * units_per_q;
    // this warp's units: global unit index = gw (mod nwarps)
    int64_t u = (gw - unit_base) % nwarps;
    if (u < 0) u += nwarps;
    for (; u < nunits; u += nwarps) {
      const int a = (int)(u / units_per_q);
      const int r = (int)(u % units_per_q);
      const int q = sm.q[a], ns = sm.ns[a];
      const int colblk = r % ncolblk, hg = r / ncolblk;
      const int hm = hg * 32 + lane;    // head of this lane's (m, l)
      const bool hm_ok = hm < p.num_q_heads;
      const int h0 = hg * 32 + 4 * g;   // first of this lane's four O heads (< head_stride)
      const int d = colblk * kCombineCols + 2 * cpair;
      const float* ml = p.part_ml + (int64_t)q * p.nslices * 2 * hs + hm;
      const float* po = p.part_o + ((int64_t)q * p.nslices * kDv + d) * hs + h0;
      // first group: (m, l) and O together
      float mv[kCombineGroup], lv[kCombineGroup];
      float4 o0[kCombineGroup], o1[kCombineGroup];
#pragma unroll
      for (int k = 0; k < kCombineGroup; ++k) {
        const bool live = k < ns;
        mv[k] = live && hm_ok ? __ldcg(ml + k * 2 * hs) : -INFINITY;
        lv[k] = live && hm_ok ? __ldcg(ml + k * 2 * hs + hs) : 0.f;
        o0[k] = live ? __ldcg(reinterpret_cast<const float4*>(po + (int64_t)k * kDv * hs)) : z4;
        o1[k] = live ? __ldcg(reinterpret_cast<const float4*>(po + (int64_t)k * kDv * hs + hs)) : z4;
      }
      // every item has at least one key, so every l > 0
      float M = -INFINITY;
#pragma unroll
      for (int k = 0; k < kCombineGroup; ++k) M = fmaxf(M, mv[k]);
      for (int s = kCombineGroup; s < ns; ++s)
        M = fmaxf(M, hm_ok ? __ldcg(ml + s * 2 * hs) : -INFINITY);
      float L = 0.f;
#pragma unroll
      for (int k = 0; k < kCombineGroup; ++k) {
        const float w = ex2_approx(mv[k] - M);  // 0 for absent items
        L = fmaf(lv[k], w, L);
        sm.w[warp][k][lane] = w;
      }
      for (int s = kCombineGroup; s < ns; ++s) {
        const float w = hm_ok ? ex2_approx(__ldcg(ml + s * 2 * hs) - M) : 0.f;
        L = fmaf(hm_ok ? __ldcg(ml + s * 2 * hs + hs) : 0.f, w, L);
        sm.w[warp][s][lane] = w;
      }
      float den = L, alpha = 1.f;
      if (MODE == SA_SINK_NULL_LOGIT) {
        const float sink2 = hm_ok ? __ldg(p.sinks + hm) * kLog2e : 0.f;
        const float mp = fmaxf(M, sink2);
        alpha = ex2_approx(M - mp);
        den = L * alpha + ex2_approx(sink2 - mp);
      }
      sm.inv[warp][lane] = hm_ok ? alpha / den : 0.f;
      if (colblk == 0 && hm_ok) p.lse[(int64_t)hm * p.nq + q] = (M + log2f(L)) * kLn2;
      __syncwarp();
      float4 a0 = z4, a1 = z4;
      for (int s0 = 0; s0 < ns; s0 += kCombineGroup) {
        if (s0 > 0) {
#pragma unroll
          for (int k = 0; k < kCombineGroup; ++k) {
            const bool live = s0 + k < ns;
            const float* src = po + (int64_t)(s0 + k) * kDv * hs;
            o0[k] = live ? __ldcg(reinterpret_cast<const float4*>(src)) : z4;
            o1[k] = live ? __ldcg(reinterpret_cast<const float4*>(src + hs)) : z4;
          }
        }
#pragma unroll
        for (int k = 0; k < kCombineGroup; ++k) {
          if (s0 + k < ns) {
            const float4 w = *reinterpret_cast<const float4*>(&sm.w[warp][s0 + k][4 * g]);
            a0.x = fmaf(w.x, o0[k].x, a0.x);
            a0.y = fmaf(w.y, o0[k].y, a0.y);
            a0.z = fmaf(w.z, o0[k].z, a0.z);
            a0.w = fmaf(w.w, o0[k].w, a0.w);
            a1.x = fmaf(w.x, o1[k].x, a1.x);
            a1.y = fmaf(w.y, o1[k].y, a1.y);
            a1.z = fmaf(w.z, o1[k].z, a1.z);
            a1.w = fmaf(w.w, o1[k].w, a1.w);
          }
        }
      }
      const float4 iv = *reinterpret_cast<const float4*>(&sm.inv[warp][4 * g]);
      *reinterpret_cast<uint32_t*>(&sm.o[warp][4 * g + 0][2 * cpair]) = pack_bf16x2(a0.x * iv.x, a1.x * iv.x);
      *reinterpret_cast<uint32_t*>(&sm.o[warp][4 * g + 1][2 * cpair]) = pack_bf16x2(a0.y * iv.y, a1.y * iv.y);
      *reinterpret_cast<uint32_t*>(&sm.o[warp][4 * g + 2][2 * cpair]) = pack_bf16x2(a0.z * iv.z, a1.z * iv.z);
      *reinterpret_cast<uint32_t*>(&sm.o[warp][4 * g + 3][2 * cpair]) = pack_bf16x2(a0.w * iv.w, a1.w * iv.w);
      __syncwarp();
      if (hm_ok)
        *reinterpret_cast<uint4*>(p.out + ((int64_t)q * p.num_q_heads + hm) * kDv +
                                  colblk * kCombineCols) =
            *reinterpret_cast<const uint4*>(&sm.o[warp][lane][0]);
      __syncwarp();  // sm.w / sm.o of this warp are rewritten by its next unit
    }
    unit_base += nunits;
    __syncthreads();  // sm.q is rewritten by the next chunk
  }
}

struct WorkspaceLayout {
  size_t cidx, qcount, ml, o, total;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
int head_stride(int hq) { return (hq + 31) & ~31; }

WorkspaceLayout workspace_layout(int32_t nq, int32_t hq, int32_t topk) {
  WorkspaceLayout w;
  const int nslices = (topk + kItemKeys - 1) / kItemKeys;
  w.cidx = 0;
  w.qcount = align256((size_t)nq * topk * sizeof(int32_t));
  w.ml = w.qcount + align256((size_t)nq * sizeof(int32_t));
  w.o = w.total = w.ml;
  if (nslices > 1) {
    const size_t hs = (size_t)head_stride(hq);
    w.o = w.ml + align256((size_t)nq * nslices * 2 * hs * sizeof(float));
    w.total = w.o + (size_t)nq * nslices * kDv * hs * sizeof(float);
  }
  return w;
}

template <int MODE, bool FP8>
sa_status launch_typed(const IndexArgs& a) {
  const char* fn = a.fn;
  const int nslices = (a.topk + kItemKeys - 1) / kItemKeys;
  uint8_t* ws = reinterpret_cast<uint8_t*>(a.workspace);
  const WorkspaceLayout wl = workspace_layout(a.num_queries, a.num_q_heads, a.topk);

  PlanParams pp;
  pp.indices = a.indices;
  pp.topk = a.topk;
  pp.num_kv = a.num_kv;
  pp.nq = a.num_queries;
  pp.num_q_heads = a.num_q_heads;
  pp.cidx = a.topk > 0 ? reinterpret_cast<int32_t*>(ws + wl.cidx) : nullptr;
  pp.qcount = a.topk > 0 ? reinterpret_cast<int32_t*>(ws + wl.qcount) : nullptr;
  pp.out = reinterpret_cast<__nv_bfloat16*>(a.out);
  pp.lse = a.lse;
  sparse_index_plan_kernel<<<(unsigned)a.num_queries, kThreads, 0, a.stream>>>(pp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(SA_ERR_CUDA, "%s plan launch: %s", fn, cudaGetErrorString(e));
  if (a.topk == 0) return SA_OK;  // every key set is empty

  CUtensorMap tq;
  const uint64_t dq[2] = {(uint64_t)kDqk, (uint64_t)a.num_queries * a.num_q_heads};
  const uint64_t sq[1] = {(uint64_t)kDqk * 2};
  const uint32_t bq[2] = {kSlab, 128};
  if (!encode_tiled(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, dq, sq, bq,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return SA_ERR_INVALID_ARG;
  IndexParams p;
  p.kv_scale = a.kv_scale;
  p.cidx = pp.cidx;
  p.qcount = pp.qcount;
  p.topk = a.topk;
  p.nslices = nslices;
  p.num_q_heads = a.num_q_heads;
  p.nhb = (a.num_q_heads + 127) / 128;
  p.nq = a.num_queries;
  p.sinks = a.sinks;
  p.scale_log2 = a.softmax_scale * kLog2e;
  p.out = reinterpret_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.part_ml = nslices > 1 ? reinterpret_cast<float*>(ws + wl.ml) : nullptr;
  p.part_o = nslices > 1 ? reinterpret_cast<float*>(ws + wl.o) : nullptr;
  p.head_stride = head_stride(a.num_q_heads);
  p.combine_min_items = 2;
  p.err = device_error_word();

  const size_t smem = 1024 + (size_t)kNumSlots * kSlotBytes + 2 * (size_t)kSlabBytesQ;
  auto kern = sparse_index_fwd_kernel<MODE, FP8>;
  if (!set_dynamic_smem_once((const void*)kern, (int)smem))
    return fail(SA_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(cudaGetLastError()));
  // at most one item per (query, 256 index slots)
  const unsigned items = (unsigned)((int64_t)a.num_queries * nslices * p.nhb);
  e = launch_dependent(kern, dim3(items), dim3(kThreads), smem, a.stream, tq, a.kv, p);
  if (e != cudaSuccess) return fail(SA_ERR_CUDA, "%s launch: %s", fn, cudaGetErrorString(e));
  if (nslices > 1) {
    // queries with 2..8 items: TMA-fed combine over the partials viewed as
    // [query x item][512 columns][head_stride] and the (m, l) rows as
    // [query x item x 2][head_stride], fp32
    const int64_t items = (int64_t)a.num_queries * nslices;
    if (items * 2 >= ((int64_t)1 << 31))
      return fail(SA_ERR_UNSUPPORTED, "%s: %lld partial items", fn, (long long)items);
    const uint32_t bh = (uint32_t)std::min(128, p.head_stride);
    CUtensorMap tp, tp1, tml;
    const uint64_t dp[3] = {(uint64_t)p.head_stride, (uint64_t)kDv, (uint64_t)items};
    const uint64_t sp[2] = {(uint64_t)p.head_stride * 4, (uint64_t)p.head_stride * 4 * kDv};
    const uint32_t bp[3] = {bh, (uint32_t)kFcCols, (uint32_t)kFcMaxItems};
    const uint32_t bp1[3] = {bh, (uint32_t)kFcCols, 1u};
    if (!encode_tiled(&tp, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.part_o, dp, sp, bp,
                      CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tiled(&tp1, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.part_o, dp, sp, bp1,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
      return SA_ERR_INVALID_ARG;
    const uint64_t dm[2] = {(uint64_t)p.head_stride, (uint64_t)items * 2};
    const uint64_t sm_[1] = {(uint64_t)p.head_stride * 4};
    const uint32_t bm[2] = {bh, (uint32_t)(2 * kFcMaxItems)};
    if (!encode_tiled(&tml, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p.part_ml, dm, sm_, bm,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
      return SA_ERR_INVALID_ARG;
    const int64_t max_units = (int64_t)(a.num_queries / 2) * (kDv / kFcCols) * p.nhb;
    const unsigned g1 = (unsigned)std::max<int64_t>(1, std::min<int64_t>(max_units, num_sms()));
    const size_t smem_c = 128 + kFcStages * sizeof(FcStage);
    auto kc = sparse_index_combine_tma_kernel<MODE>;
    if (!set_dynamic_smem_once((const void*)kc, (int)smem_c))
      return fail(SA_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(cudaGetLastError()));
    e = launch_dependent(kc, dim3(g1), dim3(kThreads), smem_c, a.stream, tp, tp1, tml, p);
    if (e != cudaSuccess)
      return fail(SA_ERR_CUDA, "%s combine launch: %s", fn, cudaGetErrorString(e));
    if (nslices > kFcMaxItems) {
      // queries with more than 8 items: warp-unit combine
      p.combine_min_items = kFcMaxItems + 1;
      const int64_t wunits = (int64_t)(a.num_queries / (kFcMaxItems + 1)) * (kDv / kCombineCols) *
                             (p.head_stride / 32);
      const int64_t per_cta = kThreads / 32;
      const unsigned g2 = (unsigned)std::max<int64_t>(
          1, std::min<int64_t>((wunits + per_cta - 1) / per_cta, num_sms()));
      e = launch_dependent(sparse_index_combine_kernel<MODE>, dim3(g2), dim3(kThreads), 0,
                           a.stream, p);
      if (e != cudaSuccess)
        return fail(SA_ERR_CUDA, "%s combine launch: %s", fn, cudaGetErrorString(e));
    }
  }
  return SA_OK;
}

}  // namespace

size_t sparse_index_workspace_bytes(int32_t num_queries, int32_t num_q_heads, int32_t topk) {
  if (num_queries <= 0 || topk <= 0) return 0;
  return workspace_layout(num_queries, num_q_heads, topk).total;
}

int sparse_index_max_topk() { return kMaxSlices * kItemKeys; }

sa_status launch_sparse_index_fwd(const IndexArgs& a) {
  if (a.dqk != kDqk || a.dv != kDv)
    return fail(SA_ERR_UNSUPPORTED, "%s: dqk %d / dv %d (supported: 576 / 512)", a.fn, a.dqk,
                a.dv);
  if (a.fp8) {
    if (a.sink_mode == SA_SINK_NULL_LOGIT) return launch_typed<SA_SINK_NULL_LOGIT, true>(a);
    return launch_typed<SA_SINK_NONE, true>(a);
  }
  if (a.sink_mode == SA_SINK_NULL_LOGIT) return launch_typed<SA_SINK_NULL_LOGIT, false>(a);
  return launch_typed<SA_SINK_NONE, false>(a);
}

}  // namespace sa

// ---------------------------------------------------------------------------
// Allocation-free entry point.
//
// Some callers cannot obtain device memory for a workspace: code embedded in a
// host runtime that owns the whole device memory pool and hands its plugins no
// allocator, or a serving loop that forbids any allocation once it is running.
// sa_sparse_index_fwd_noalloc serves them by keeping the split-KV scratch in
// the fixed array below instead of a caller workspace.  The array is reserved
// on every GPU that loads this library and stays reserved until the process
// exits.  Every call shares it and it keeps the last call's contents; each
// call writes every entry it later reads, so nothing in it has to start at
// zero.  Two calls whose work overlaps on the GPU (different streams, or
// different host threads) race on the array.
namespace sa {
namespace {
constexpr size_t kNoAllocScratchBytes = (size_t)64 << 20;  // 64 MiB
constexpr int kNoAllocMaxDevices = 64;

// The array's device address per device, with the id of the context it was
// looked up in: a context destroyed and re-created (cudaDeviceReset) may
// place the array elsewhere, and gets a new id, so the address is looked up
// again in it.
struct NoAllocSlot {
  uint64_t ctx;
  void* ptr;
};
std::mutex g_noalloc_mu;
NoAllocSlot g_noalloc_slot[kNoAllocMaxDevices];
}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
// Set-up, once per device and context, with that device current: the
// host-side name of the array is not a device address, so the runtime is
// asked for it.
sa_status noalloc_scratch_address(const char* fn, void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices)
    return fail(SA_ERR_CUDA, "%s: no usable CUDA device", fn);
  const uint64_t ctx = current_context_id();
  std::lock_guard<std::mutex> guard(g_noalloc_mu);
  NoAllocSlot& slot = g_noalloc_slot[dev];
  if (slot.ptr && ctx != 0 && slot.ctx == ctx) {
    *out = slot.ptr;
    return SA_OK;
  }
  void* ptr = nullptr;
  e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (e != cudaSuccess || !ptr)
    return fail(SA_ERR_CUDA, "%s: cudaGetSymbolAddress of the scratch array failed: %s", fn,
                cudaGetErrorString(e));
  slot.ctx = current_context_id();
  slot.ptr = ptr;
  *out = ptr;
  return SA_OK;
}
}  // namespace
}  // namespace sa

extern "C" sa_status sa_sparse_index_fwd_noalloc(
    const void* q, const void* kv_latent, int64_t num_kv, int32_t dqk, int32_t dv,
    const int32_t* indices, int32_t topk, int32_t num_queries, int32_t num_q_heads,
    const float* sinks, int32_t sink_mode, float softmax_scale, void* out, float* lse,
    void* stream) {
  static const sa::FixedScratch fixed = {sa::kNoAllocScratchBytes, sa::noalloc_scratch_address};
  return sa::sparse_index_entry("sa_sparse_index_fwd_noalloc", q, kv_latent, nullptr, false,
                                num_kv, dqk, dv, indices, topk, num_queries, num_q_heads, sinks,
                                sink_mode, softmax_scale, out, lse, nullptr, 0, stream, &fixed);
}

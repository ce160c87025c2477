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
// Two kernels, back to back on the stream (the second starts early under
// programmatic dependent launch and waits for the first):
//  1. plan: one CTA per query compacts the valid entries of its index row
//     (order kept) into the workspace, stores their count c and clears the
//     query's completion counter.  A query with c = 0 gets its zero output and
//     LSE = -inf here.
//  2. attend, persistent (one CTA per SM at most): the compacted list of a
//     query is cut into items of up to 256 keys, ordered "all full 256-key
//     items (query order), then the shorter last items (query order)", and
//     CTA b takes items b, b + grid, ... (so the long items start first and
//     no CTA is launched without work).  Per (item, block of 128 heads):
//       S = Q K^T      M = 128 heads, N = item keys (rounded to 16), K = 576
//                      in nine 64-wide slabs;
//       O = P V        in three parts of 256, 128 and 128 V columns (tensor
//                      memory holds S and one 128 x 512 fp32 O only in
//                      part), K = the item's keys.
//     A query with a single item is finished there (sink fold, bf16 O, LSE).
//     Otherwise the item's (O, m, l) partial goes to the workspace and the
//     query's completion counter is raised.  Once a CTA has no items left it
//     merges: units of (query with several items, block of 128 heads, 16 V
//     columns) are split into one contiguous range per CTA; a unit waits
//     (bounded) for its query's counter, then merges the partials by their LSE weights
//     and folds the sink once.  Every CTA of the grid is resident (one per
//     SM), and a CTA merges only after finishing its own items, so every
//     wait ends.
// Split-KV partials are stored heads-fastest ([query][item][column][head],
// the head stride rounded up to 32), so each warp store of the epilogue
// writes 128 contiguous, aligned bytes.
#include <cuda_bf16.h>
#include <math.h>
#include <string.h>

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
constexpr int kMergeCols = 32;  // V columns per merge unit
constexpr int kMergeSegs = kMergeCols / 16;  // 8-column segments per merge thread
static_assert(kMergeCols % 16 == 0 && kMergeCols <= 32, "a merge unit lies inside one scale chunk");
constexpr int kMergeGroup = 8;  // items whose partials are loaded at once
constexpr int kMergeStages = 3; // merge units in flight per CTA (TMA-fed)
constexpr int kPartChunk = 32;  // V columns sharing one fp16 scale in a partial

// One merge unit's partials in shared memory (row stride: the tile's head
// count): the [8 items][16 column pairs][128 heads] O box (fp16 pairs) and the
// [8 items][128 heads] scale exponents of the unit's 32-column chunk.
struct __align__(128) MergeStage {
  uint32_t o[kMergeGroup][kMergeCols / 2][128];
  int8_t e[kMergeGroup][128];
};
// The [8 items x (m, l)][128 heads] fp32 box of a (query, head block): loaded
// once per CTA for the run of its units that share it, into one of two
// buffers.
struct __align__(128) MergeMl {
  float ml[kMergeGroup][2][128];
};
constexpr int kUnitsPerHb = kDv / kMergeCols;  // merge units per (query, head block)
// Two ml buffers are enough: a CTA's units are one contiguous range, so a
// (query, head block) that is neither its first nor its last one has all
// kUnitsPerHb of its units in the range, more than the units in flight.
static_assert(kMergeStages < kUnitsPerHb, "ml buffer reuse needs runs longer than the stages");
constexpr size_t kMergeSmem =
    kMergeStages * sizeof(MergeStage) + 2 * sizeof(MergeMl) + kThreads * sizeof(int32_t);
static_assert(kMergeSmem <= kNumSlots * kSlotBytes + 2 * kSlabBytesQ,
              "merge stages, ml buffers and item counts reuse the attend buffers");

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
  int32_t* done;    // [nq]: items (x head blocks) finished, cleared here
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
  uint32_t* part_o;       // [nq][nslices][256 column pairs][head_stride] fp16 pairs
  int8_t* part_e;         // [nq][nslices][16 chunks][head_stride]: O = fp16 x 2^e
  float* part_ml;         // [nq][nslices][2][head_stride]  (m, then l)
  int32_t head_stride;    // num_q_heads rounded up to 32
  int32_t* done;          // [nq]: items x head blocks finished (merge readiness)
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
  uint64_t oa_full;          // O of V columns 0..255 (slabs 0..3)
  uint64_t ob1_full;         // O of V columns 384..511 (slabs 6, 7)
  uint64_t ob2_full;         // O of V columns 256..383 (slabs 4, 5, gathered again)
  uint32_t tmem_base;
  int32_t item_q, item_s, item_n, item_nitems;
  int32_t merge_ok;
  int32_t merge_range[2];    // this CTA's merge units [first, end) of a chunk
  uint64_t merge_full[kMergeStages];
  uint64_t merge_free[kMergeStages];  // every warp has read the stage
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
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ void unpack_half2(uint32_t v, float& lo, float& hi) {
  asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\t"
      "cvt.f32.f16 %1, b;\n\t}\n"
      : "=f"(lo), "=f"(hi)
      : "r"(v));
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
__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Pull one tensor box into L2 (no shared-memory destination, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map),
               "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
// Named barrier of the gatherer warps (the last N / 32 warps of the CTA).
template <int N = 128>
__device__ __forceinline__ void bar_gather() {
  asm volatile("bar.sync 1, %0;" ::"n"(N) : "memory");
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
  griddep_wait();  // the previous call's kernels may still read the workspace
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
  if (tid == 0 && p.qcount) {
    p.qcount[q] = total;
    p.done[q] = 0;
  }
  if (total == 0) {
    // empty key set: zero output, LSE = -inf
    uint4* dst = reinterpret_cast<uint4*>(p.out + (int64_t)q * p.num_q_heads * kDv);
    for (int i = tid; i < p.num_q_heads * (kDv / 8); i += kThreads) dst[i] = make_uint4(0, 0, 0, 0);
    for (int h = tid; h < p.num_q_heads; h += kThreads) p.lse[(int64_t)h * p.nq + q] = -INFINITY;
  }
}

// ---------------------------------------------------------------------------
// 2. attend

// The global item order (see the file header).  scan_items() takes the
// prefix sums once (all 256 threads; thread t owns queries [t K, t K + K),
// K = ceil(nq / 256)); lookup_item() then resolves item `item` into
// ctl.item_* (q = -1 past the last item).  Both contain __syncthreads.
struct ItemScan {
  int pre_f, pre_p, nfull, npart, tot_f, tot_p;
  int cnt0, cnt1;  // counts of this thread's first two queries (lookup reuses them)
};

__device__ ItemScan scan_items(const IndexParams& p, IndexSmemCtl& ctl) {
  const int tid = threadIdx.x;
  const int K = (p.nq + kThreads - 1) / kThreads;
  ItemScan sc;
  sc.nfull = 0;
  sc.npart = 0;
  sc.cnt0 = 0;
  sc.cnt1 = 0;
  for (int i = 0; i < K; ++i) {
    const int qq = tid * K + i;
    const int c = qq < p.nq ? __ldcg(p.qcount + qq) : 0;
    if (i == 0) sc.cnt0 = c;
    if (i == 1) sc.cnt1 = c;
    sc.nfull += c / kItemKeys;
    sc.npart += (c % kItemKeys) != 0 ? 1 : 0;
  }
  sc.pre_f = block_exclusive_sum(sc.nfull, ctl.scan_f, &sc.tot_f);
  sc.pre_p = block_exclusive_sum(sc.npart, ctl.scan_p, &sc.tot_p);
  return sc;
}

__device__ void lookup_item(const IndexParams& p, const ItemScan& sc, int item,
                            IndexSmemCtl& ctl) {
  const int tid = threadIdx.x;
  const int K = (p.nq + kThreads - 1) / kThreads;
  if (tid == 0) ctl.item_q = -1;
  __syncthreads();
  const bool heavy = item < sc.tot_f;
  const int target = heavy ? item : item - sc.tot_f;
  const int pre = heavy ? sc.pre_f : sc.pre_p;
  const int mine = heavy ? sc.nfull : sc.npart;
  if ((heavy || target < sc.tot_p) && pre <= target && target < pre + mine) {
    int acc = pre;
    for (int i = 0; i < K; ++i) {
      const int qq = tid * K + i;
      const int c = i == 0 ? sc.cnt0 : i == 1 ? sc.cnt1 : __ldcg(p.qcount + qq);
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

// Gather 16-byte chunk c of slab `slab` of rows r0, r0 + step, ... (< npad)
// into the 128-byte-swizzled [npad][64] slot at dst; rows past n are
// zero-filled.
__device__ __forceinline__ void gather_slab(uint32_t dst, const uint16_t* kv,
                                            const int32_t* kidx, int npad, int step, int n,
                                            int r0, int c, int slab) {
#pragma unroll 4
  for (int r = r0; r < npad; r += step) {
    const bool live = r < n;
    const uint16_t* src = kv + (live ? (int64_t)kidx[r] * kDqk + slab * kSlab + c * 8 : 0);
    cp_async16(dst + r * 128 + ((c ^ (r & 7)) << 4), src, live ? 16u : 0u);
  }
}

template <int MODE, bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
sparse_index_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_part,
                        const __grid_constant__ CUtensorMap tm_part1,
                        const __grid_constant__ CUtensorMap tm_ml,
                        const __grid_constant__ CUtensorMap tm_e, const void* kv_raw,
                        const IndexParams p) {
  // Warps that gather latent rows during S: six for the bf16 cache (every
  // warp but the two that hold the MMA and Q-load threads; more warps issue
  // 16-byte copies faster), four for the fp8 cache (its staging and
  // conversion are laid out for 128 threads).
  constexpr int kGatherWarps = FP8 ? 4 : 6;
  constexpr int kGatherThreads = 32 * kGatherWarps;
  static_assert(kGatherThreads % 8 == 0 && kGatherThreads <= kThreads - 64, "");
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
  if (warp == 0) {
    tmem_alloc(&ctl.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  griddep_wait();  // the plan kernel's counts and lists are complete
  const ItemScan isc = scan_items(p, ctl);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  // work w = (item w / nhb, head block w % nhb); CTA b takes w = b, b + grid, ...
  const int nwork = (isc.tot_f + isc.tot_p) * p.nhb;

  for (int w = (int)blockIdx.x; w < nwork; w += (int)gridDim.x) {
  lookup_item(p, isc, w / p.nhb, ctl);
  if (tid == 0) {
    // every barrier starts each item at phase 0 (the previous item's
    // arrivals have all landed: its last waits saw them)
    for (int i = 0; i < 4; ++i) mbar_init(&ctl.res_full[i], kGatherThreads);
    mbar_init(&ctl.res2_full, kGatherThreads);
    for (int s2 = 0; s2 < 2; ++s2) {
      mbar_init(&ctl.kst_full[s2], kGatherThreads);
      mbar_init(&ctl.kst_empty[s2], 1);
      mbar_init(&ctl.q_full[s2], 1);
      mbar_init(&ctl.q_empty[s2], 1);
    }
    mbar_init(&ctl.s_full, 1);
    mbar_init(&ctl.oa_full, 1);
    mbar_init(&ctl.ob1_full, 1);
    mbar_init(&ctl.ob2_full, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int q = ctl.item_q;

  if (q >= 0) {
    const int hb = w % p.nhb;
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

    // gatherers (the last kGatherWarps warps; warps 0 and 1 carry the MMA
    // and Q-load threads): thread gt copies 16-byte chunk gc of rows
    // gr0 + kGatherThreads / 8 k of every slab
    const bool gatherer = warp >= kThreads / 32 - kGatherWarps;
    const int gt = tid - (kThreads - kGatherThreads);
    const int gstep = kGatherThreads / 8;
    const int gr0 = gt >> 3, gc = gt & 7;
    const int fr0 = gt >> 2, fc4 = gt & 3;  // fp8 cache: rows fr0 + 32 k, 16-byte chunk fc4
    float ks0 = 0.f, ks1 = 0.f;
    if (gatherer) {
      const int32_t* crow = p.cidx + (int64_t)q * p.topk + slice * kItemKeys;
      if (FP8) {
        const int32_t i0 = gt < n ? __ldcg(crow + gt) : 0;
        const int32_t i1 = gt + 128 < n ? __ldcg(crow + gt + 128) : 0;
        ctl.kidx[gt] = i0;
        ctl.kidx[gt + 128] = i1;
        // stored once S is complete (they go where Q was staged)
        ks0 = gt < n ? __ldg(p.kv_scale + i0) : 0.f;
        ks1 = gt + 128 < n ? __ldg(p.kv_scale + i1) : 0.f;
      } else {
        for (int r = gt; r < kItemKeys; r += kGatherThreads) ctl.kidx[r] = r < n ? __ldcg(crow + r) : 0;
      }
      bar_gather<kGatherThreads>();
    }

    if (gatherer) {
      auto gather = [&](int slot, int slab) {
        if (ok) {
          if (FP8) stage_slab_fp8(slot_u32(slot), kv8, ctl.kidx, npad, n, fr0, fc4, slab);
          else gather_slab(slot_u32(slot), kv, ctl.kidx, npad, gstep, n, gr0, gc, slab);
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
      for (int r = gt; r < n; r += kGatherThreads) {
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
      // the ring below holds two Q slabs, each refilled only once the MMAs
      // of two steps ago have read it; pull the later slabs into L2 now so
      // that those refills do not wait out DRAM behind the row gathers
      for (int j = 2; j < kNumQkSlabs; ++j) tma_prefetch_l2_2d(&tm_q, step_slab(j) * kSlab, qrow0);
      int issued = 0;
      for (int j = 0; j < kNumQkSlabs; ++j) {
        const int st = j & 1;
        if (j >= 2 && !mbar_wait(&ctl.q_empty[st], ((j >> 1) - 1) & 1, p.err, kErrWaitFree))
          break;
        mbar_arrive_expect_tx(&ctl.q_full[st], kSlabBytesQ);
        tma_load_2d(s_qst + st * kSlabBytesQ, &tm_q, &ctl.q_full[st], step_slab(j) * kSlab, qrow0);
        ++issued;
      }
      // bounded drain of the last copies (immediate once the MMAs consumed
      // them), and of the MMAs' releases of them: no arrival may follow the
      // next item's barrier initialisation
      for (int j = max(0, issued - 2); j < issued; ++j) {
        mbar_wait(&ctl.q_full[j & 1], (j >> 1) & 1, p.err, kErrWaitDrain);
        mbar_wait(&ctl.q_empty[j & 1], (j >> 1) & 1, p.err, kErrWaitDrain);
      }
    }

    // ---- softmax: thread (row, part) takes key columns [128 part, +128) ----
    const float sink2 = (MODE != SA_SINK_NONE && row_valid) ? __ldg(p.sinks + h) * kLog2e : 0.f;
    ok = mbar_wait(&ctl.s_full, 0, p.err, kErrWaitMma) && ok;
    // fp8 cache: the row scales, after the reductions in the Q staging area
    // (free once S is complete)
    float* s_ks = reinterpret_cast<float*>(s_qst + kScaleOffset);
    float* s_kc = s_ks + kItemKeys;
    if (FP8) {
      if (gatherer) {
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
    // only the two warps of the same rows (w and w + 4) exchange the max
    asm volatile("bar.sync %0, 64;" ::"r"(2 + (warp & 3)) : "memory");
    // max(s) * c2 == max(s * c2) exactly (c2 > 0, rounding is monotone); the
    // fp8 maxima are already in the log2 domain
    const float m = fmaxf(red.m[0][row], red.m[1][row]) * (FP8 ? 1.f : c2);
    {
      // pass 2: P = 2^(s c2 - m) (bf16, written over S inside this thread's
      // half) and the row sum.  Key chunk ch of 32 keys goes to TMEM columns
      // pcol0 + 16 ch: part 0 fills [0, 64) in ascending chunk order, part 1
      // fills [192, 256) in descending order, so every store lands on
      // columns this thread has already read, and [64, 192) is left free
      // as one 128-column block for an O part
      const uint64_t c2c2 = f2_pack(c2, c2), nmnm = f2_pack(-m, -m);
      const int pcol0 = part == 0 ? 0 : 192;
      uint64_t lp[4] = {0, 0, 0, 0};
#pragma unroll 1
      for (int i = 0; i < nch; ++i) {
        const int ch = part == 0 ? i : nch - 1 - i;
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
        tmem_st16(lane_base + kColS + pcol0 + 16 * ch, pk);
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

    // ---- O = P V in three parts (thread 0 issues), each with its epilogue ----
    // After S the resident slabs are 0..3 (R0..R3) and 6, 7 (K0, K1):
    //   A:  V columns 0..255   <- R0..R3, N = 256, into TMEM [256, 512);
    //   B1: V columns 384..511 <- K0, K1, N = 128, into the S columns the
    //       softmax left free, [64, 192) (P sits in [0, 64) and [192, 256));
    //   B2: V columns 256..383 <- slabs 4, 5 gathered again over R2, R3 once
    //       A has read them, N = 128, into TMEM [256, 384) once the
    //       epilogue of A has read it.
    // A and B1 go to the tensor pipe together; the regather overlaps the
    // epilogue of A, and B2 the epilogue of B1.
    auto issue_pv = [&](int first_slot, uint32_t col, int ncols) {
      const uint32_t idesc = idesc_bf16(128, ncols, true);
      const uint32_t vb = slot_u32(first_slot);
      for (int kk = 0; kk < npad / 16; ++kk) {
        // P of keys [16 kk, 16 kk + 16): TMEM column 8 kk (keys < 128) or
        // 192 + 8 (kk - 8)
        const uint32_t pa = tmem + kColS + (kk < 8 ? kk * 8 : 192 + (kk - 8) * 8);
        const uint64_t b = smem_desc(vb + kk * 16 * 128, kSlotBytes, 1024, kLayoutSw128);
        mma_ts(tmem + col, pa, b, idesc, kk > 0 ? 1u : 0u);
      }
    };
    if (tid == 0) {
      if (ok) {
        tc_fence_after();
        issue_pv(0, kColO, 256);
        mma_commit(&ctl.oa_full);
        issue_pv(4, kColS + 64, 128);
        mma_commit(&ctl.ob1_full);
      } else {
        mbar_arrive(&ctl.oa_full);
        mbar_arrive(&ctl.ob1_full);
      }
    }
    const int64_t hq = p.num_q_heads;
    // this thread's row, nch chunks of 32 values: TMEM columns tcol + 32 j,
    // V columns vcol + 32 j
    auto epilogue = [&](int tcol, int vcol, int nch) {
      __nv_bfloat16* orow = p.out + ((int64_t)q * hq + h) * kDv + vcol;
      const int64_t hs = p.head_stride;
      const int64_t pitem = (int64_t)q * p.nslices + slice;
      uint32_t* pcol = p.part_o + (pitem * (kDv / 2) + vcol / 2) * hs + h;
      int8_t* ecol = p.part_e + (pitem * (kDv / kPartChunk) + vcol / kPartChunk) * hs + h;
#pragma unroll 1
      for (int jj = 0; jj < nch; ++jj) {
        float o[32];
        tmem_ld32(lane_base + tcol + 32 * jj, o);
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
          // fp16 with a power-of-two scale per 32-column chunk: the chunk's
          // largest magnitude lands in [2^14, 2^15), every value keeps fp16's
          // 11-bit relative precision, nothing overflows
          float amax = 0.f;
#pragma unroll
          for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(o[e]));
          int ex = amax > 0.f ? (int)((__float_as_uint(amax) >> 23) & 0xffu) - 127 - 14 : 0;
          ex = max(ex, -126);
          const float sc = __uint_as_float((uint32_t)(127 - ex) << 23);  // 2^-ex
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pcol[(int64_t)(16 * jj + e) * hs] = pack_half2(o[2 * e] * sc, o[2 * e + 1] * sc);
          ecol[(int64_t)jj * hs] = (int8_t)ex;
        }
      }
    };
    ok = mbar_wait(&ctl.oa_full, 0, p.err, kErrWaitMma) && ok;
    __syncwarp();
    tc_fence_after();
    if (gatherer) {
      // slabs 4, 5 over R2, R3 (A has read them), landing while A is stored
      if (ok) {
        if (FP8) {
          stage_slab_fp8(slot_u32(2), kv8, ctl.kidx, npad, n, fr0, fc4, 4);
          stage_slab_fp8(slot_u32(3), kv8, ctl.kidx, npad, n, fr0, fc4, 5);
        } else {
          gather_slab(slot_u32(2), kv, ctl.kidx, npad, gstep, n, gr0, gc, 4);
          gather_slab(slot_u32(3), kv, ctl.kidx, npad, gstep, n, gr0, gc, 5);
        }
      }
      cp_async_commit();
      epilogue(kColO + part * 128, part * 128, 4);
      cp_async_wait<0>();
      if (FP8) {
        convert_slab_fp8(slot_u32(2), npad, fr0, fc4);
        convert_slab_fp8(slot_u32(3), npad, fr0, fc4);
      }
      fence_proxy_async();
      mbar_arrive(&ctl.res2_full);
    } else {
      epilogue(kColO + part * 128, part * 128, 4);
    }
    tc_fence_before();
    __syncthreads();  // every TMEM read of A is done
    if (tid == 0) {
      tc_fence_after();
      if (ok && mbar_wait(&ctl.res2_full, 0, p.err, kErrWaitLoad)) {
        issue_pv(2, kColO, 128);
        mma_commit(&ctl.ob2_full);
      } else {
        mbar_arrive(&ctl.ob2_full);
      }
    }
    ok = mbar_wait(&ctl.ob1_full, 0, p.err, kErrWaitMma) && ok;
    __syncwarp();
    tc_fence_after();
    epilogue(kColS + 64 + part * 64, 384 + part * 64, 2);
    ok = mbar_wait(&ctl.ob2_full, 0, p.err, kErrWaitMma) && ok;
    __syncwarp();
    tc_fence_after();
    epilogue(kColO + part * 64, 256 + part * 64, 2);
    if (row_valid && part == 0) {
      if (direct) {
        p.lse[(int64_t)h * p.nq + q] = (m + log2f(l)) * kLn2;
      } else {
        float* ml = p.part_ml + ((int64_t)q * p.nslices + slice) * 2 * p.head_stride + h;
        ml[0] = m;
        ml[p.head_stride] = l;
      }
    }
    if (!direct) {
      // this item's partial is written: count it for the query's merge
      __syncthreads();
      if (tid == 0) {
        __threadfence();
        atomicAdd(p.done + q, 1);
      }
    }
  }
  // the next item rewrites tensor memory and the barriers
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  }  // items

  // ---- split-KV merge -------------------------------------------------------------
  // Units of (query with several items, block of 128 heads, 32 V columns:
  // one scale chunk), 256 queries at a time, split into one contiguous range
  // of about equal unit count per CTA, so a CTA's units mostly share a query:
  // it waits for one counter and loads one (m, l) box per run, not one per
  // unit.  A unit waits (bounded) until
  // every item of its query is counted.  Thread t merges head t mod 128 of
  // the unit's head block, half t / 128 of the unit's V columns:
  //   O = sum_s 2^(m_s - M) O_s * alpha / (L alpha + 2^(s_h log2e - M')),
  //   M = max m_s, L = sum_s l_s 2^(m_s - M), M' = max(M, s_h log2e),
  //   alpha = 2^(M - M'), LSE = (M + log2 L) ln 2 over the listed keys only.
  // Queries of at most eight items: lane 0 of warp st loads the units of
  // stage st (one issuing thread per stage) by TMA into one of kMergeStages
  // shared-memory stages (the attend buffers, free now): each unit's O and
  // scale boxes, and the (m, l) box once per run of units of one (query,
  // head block), so several units' reads are in flight without register
  // cost.  More items: plain loads, eight items at a time.
  {
    const int h_in = tid & 127, half = tid >> 7;
    const int64_t hs = p.head_stride;
    const int bi = hs < 128 ? (int)hs : 128;  // heads per TMA box row
    const int64_t per_q = (int64_t)p.nhb * kUnitsPerHb;
    const int64_t G = gridDim.x;
    MergeStage* stage = reinterpret_cast<MergeStage*>(s_slot);
    MergeMl* s_ml = reinterpret_cast<MergeMl*>(s_slot + kMergeStages * sizeof(MergeStage));
    // item counts of the chunk's merged queries (ctl.kidx holds the queries)
    int32_t* s_mns = reinterpret_cast<int32_t*>(s_ml + 2);
    int last_ready = -1;  // the last query this thread found complete
    // the stage this thread fills (lane 0 of warps 0 .. kMergeStages - 1), or -1
    const int lane0_of_stage = (tid & 31) == 0 && tid / 32 < kMergeStages ? tid / 32 : -1;
    // the stages overlay buffers this CTA wrote through the generic proxy
    // (the softmax exchange); order those writes before the copies' writes
    fence_proxy_async();
    if (tid == 0) {
      for (int i = 0; i < kMergeStages; ++i) {
        mbar_init(&ctl.merge_full[i], 1);
        mbar_init(&ctl.merge_free[i], kThreads / 32);
      }
      fence_mbar_init();
      tma_prefetch_map(&tm_part);
      tma_prefetch_map(&tm_part1);
      tma_prefetch_map(&tm_ml);
      tma_prefetch_map(&tm_e);
      ctl.merge_ok = 1;
    }
    __syncthreads();
    // thread 0: wait (bounded) until query q's items are all counted
    auto wait_ready = [&](int q, int ns) -> bool {
      const int want = ns * p.nhb;
      if (ld_acquire(p.done + q) >= want) return true;
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire(p.done + q) < want) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          atomicOr(p.err, kErrWaitLoad);
          return false;
        }
        __nanosleep(64);
      }
      return true;
    };
    // the merged row segment of head h, columns c0 .. c0 + 8, and its LSE
    auto finish = [&](int q, int h, int c0, float M, float L, const float (&acc)[8]) {
      float den = L, alpha = 1.f;
      if (MODE == SA_SINK_NULL_LOGIT) {
        const float sink2 = __ldg(p.sinks + h) * kLog2e;
        const float mp = fmaxf(M, sink2);
        alpha = ex2_approx(M - mp);
        den = L * alpha + ex2_approx(sink2 - mp);
      }
      const float inv = alpha / den;
      uint4 pk;
      pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
      pk.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
      pk.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
      pk.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
      *reinterpret_cast<uint4*>(p.out + ((int64_t)q * p.num_q_heads + h) * kDv + c0) = pk;
      if (c0 == 0) p.lse[(int64_t)h * p.nq + q] = (M + log2f(L)) * kLn2;
    };
    uint32_t phase = 0;
    // pass 0: queries of 2..8 items (TMA-fed); pass 1: more than 8 (plain loads)
    for (int pass = 0; pass < 2; ++pass) {
      for (int qc = 0; qc < p.nq; qc += kThreads) {
        const int qq = qc + tid;
        const int nsq = qq < p.nq ? (__ldcg(p.qcount + qq) + kItemKeys - 1) / kItemKeys : 0;
        const int act = (pass == 0 ? (nsq >= 2 && nsq <= kMergeGroup) : nsq > kMergeGroup) ? 1 : 0;
        int nact = 0;
        const int pos = block_exclusive_sum(act, ctl.scan_f, &nact);
        if (act) {
          ctl.kidx[pos] = qq;
          s_mns[pos] = nsq;
        }
        // a unit of this query weighs the items its copies load; CTA b takes
        // the units whose weight starts in [W b / G, W (b + 1) / G)
        const int wq = act ? 1 : 0;
        int wtot = 0;
        const int wpre = block_exclusive_sum(wq, ctl.scan_p, &wtot);
        const int64_t nunits = (int64_t)nact * per_q;
        const int64_t W = per_q * wtot;
        const int64_t xb = W * blockIdx.x / G, xe = W * (blockIdx.x + 1) / G;
        if (act) {
          const int64_t lo = per_q * wpre, hi = lo + per_q * wq;
          if (xb >= lo && xb < hi) ctl.merge_range[0] = (int)(pos * per_q + (xb - lo + wq - 1) / wq);
          if (xe >= lo && xe < hi) ctl.merge_range[1] = (int)(pos * per_q + (xe - lo + wq - 1) / wq);
        }
        if (tid == 0) {
          if (xb >= W) ctl.merge_range[0] = (int)nunits;
          if (xe >= W) ctl.merge_range[1] = (int)nunits;
        }
        __syncthreads();
        const int64_t first = ctl.merge_range[0];
        const int64_t mine = ctl.merge_range[1] - first;
        auto unit_of = [&](int64_t k, int& q, int& ns, int& hb, int& cb) {
          const int64_t u = first + k;
          q = ctl.kidx[(int)(u / per_q)];
          ns = s_mns[(int)(u / per_q)];
          const int r = (int)(u % per_q);
          hb = r / kUnitsPerHb;
          cb = r % kUnitsPerHb;
        };
        if (pass == 0) {
          // thread 0: unit k's two copies into stage st, once its query is ready
          auto issue = [&](int64_t k, int st) {
            int q, ns, hb, cb;
            unit_of(k, q, ns, hb, cb);
            if (q != last_ready) {
              if (!wait_ready(q, ns)) ctl.merge_ok = 0;
              // the partials were written through the generic proxy by
              // other SMs; this orders them before every later copy
              asm volatile("fence.proxy.async.global;" ::: "memory");
              last_ready = q;
            }
            // the (m, l) box once per run of units of one (query, head
            // block), into the buffer of the run's parity in the range
            const int64_t u = first + k;
            const bool load_ml = k == 0 || u % kUnitsPerHb == 0;
            const int iss_ml = (int)((u / kUnitsPerHb - first / kUnitsPerHb) & 1);
            // full boxes (out-of-range parts zero-filled) count in the
            // transaction; up to four items one box each, more in one box
            const int nbox = ns <= 4 ? ns : kMergeGroup;
            mbar_arrive_expect_tx(&ctl.merge_full[st],
                                  (uint32_t)((nbox * (kMergeCols / 2) + (load_ml ? 2 * kMergeGroup : 0)) *
                                                 bi * 4 +
                                             kMergeGroup * bi));
            if (ns <= 4) {
              for (int s2 = 0; s2 < ns; ++s2)
                tma_load_3d(&stage[st].o[0][0][0] + s2 * (kMergeCols / 2) * bi, &tm_part1,
                            &ctl.merge_full[st], hb * 128, cb * (kMergeCols / 2),
                            q * p.nslices + s2);
            } else {
              tma_load_3d(&stage[st].o[0][0][0], &tm_part, &ctl.merge_full[st], hb * 128,
                          cb * (kMergeCols / 2), q * p.nslices);
            }
            if (load_ml)
              tma_load_2d(&s_ml[iss_ml].ml[0][0][0], &tm_ml, &ctl.merge_full[st], hb * 128,
                          q * p.nslices * 2);
            tma_load_3d(&stage[st].e[0][0], &tm_e, &ctl.merge_full[st], hb * 128,
                        (cb * kMergeCols) / kPartChunk, q * p.nslices);
          };
          // stage st is filled by lane 0 of warp st: one issuing thread per
          // stage, each with its own copies in flight
          if (lane0_of_stage >= 0 && lane0_of_stage < mine) issue(lane0_of_stage, lane0_of_stage);
          for (int64_t k = 0; k < mine; ++k) {
            const int st = (int)(k % kMergeStages);
            int q, ns, hb, cb;
            unit_of(k, q, ns, hb, cb);
            const uint32_t use_par = (phase >> st) & 1u;  // this use of stage st
            if (!mbar_wait(&ctl.merge_full[st], use_par, p.err, kErrWaitLoad))
              ctl.merge_ok = 0;
            phase ^= 1u << st;
            const int con_ml = (int)(((first + k) / kUnitsPerHb - first / kUnitsPerHb) & 1);
            const int h = hb * 128 + h_in;
            if (ctl.merge_ok && h < p.num_q_heads) {
              // box rows: item s has m at row 2 s and l at row 2 s + 1
              const float* mlt = &s_ml[con_ml].ml[0][0][0];
              const uint32_t* ot = &stage[st].o[0][0][0];
              const int8_t* et = &stage[st].e[0][0];
              float M = -INFINITY;
#pragma unroll
              for (int s2 = 0; s2 < kMergeGroup; ++s2)
                if (s2 < ns) M = fmaxf(M, mlt[(2 * s2) * bi + h_in]);
              float L = 0.f, acc[kMergeSegs][8];
#pragma unroll
              for (int g = 0; g < kMergeSegs; ++g)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;
#pragma unroll
              for (int s2 = 0; s2 < kMergeGroup; ++s2) {
                if (s2 < ns) {
                  const float dm = mlt[(2 * s2) * bi + h_in] - M;
                  L = fmaf(mlt[(2 * s2 + 1) * bi + h_in], ex2_approx(dm), L);
                  // the item's weight times its chunk scale 2^e
                  const float wk = ex2_approx(dm + (float)et[s2 * bi + h_in]);
#pragma unroll
                  for (int i = 0; i < 4 * kMergeSegs; ++i) {
                    float lo, hi;
                    unpack_half2(ot[(s2 * (kMergeCols / 2) + half * 4 * kMergeSegs + i) * bi + h_in],
                                 lo, hi);
                    acc[i >> 2][2 * (i & 3)] = fmaf(wk, lo, acc[i >> 2][2 * (i & 3)]);
                    acc[i >> 2][2 * (i & 3) + 1] = fmaf(wk, hi, acc[i >> 2][2 * (i & 3) + 1]);
                  }
                }
              }
#pragma unroll
              for (int g = 0; g < kMergeSegs; ++g)
                finish(q, h, cb * kMergeCols + (half * kMergeSegs + g) * 8, M, L, acc[g]);
            }
            // stage st is consumed by this warp; its filler waits for every warp
            // (the warps need not wait for each other)
            __syncwarp();
            if ((tid & 31) == 0) mbar_arrive(&ctl.merge_free[st]);
            if (lane0_of_stage == st && k + kMergeStages < mine) {
              if (!mbar_wait(&ctl.merge_free[st], use_par, p.err, kErrWaitFree))
                ctl.merge_ok = 0;
              issue(k + kMergeStages, st);
            }
          }
        } else {
          for (int64_t k = 0; k < mine; ++k) {
            int q, ns, hb, cb;
            unit_of(k, q, ns, hb, cb);
            if (tid == 0 && q != last_ready) {
              if (!wait_ready(q, ns)) ctl.merge_ok = 0;
              last_ready = q;
            }
            __syncthreads();
            const int h = hb * 128 + h_in;
            if (ctl.merge_ok && h < p.num_q_heads) {
              const float* ml = p.part_ml + (int64_t)q * p.nslices * 2 * hs + h;
              const int8_t* pe =
                  p.part_e + ((int64_t)q * p.nslices * (kDv / kPartChunk) + (cb * kMergeCols) / kPartChunk) * hs + h;
              // every item has at least one key, so every l > 0
              float M = -INFINITY, L = 0.f;
              for (int s2 = 0; s2 < ns; ++s2) M = fmaxf(M, __ldcg(ml + s2 * 2 * hs));
              for (int s2 = 0; s2 < ns; ++s2)
                L = fmaf(__ldcg(ml + s2 * 2 * hs + hs), ex2_approx(__ldcg(ml + s2 * 2 * hs) - M), L);
#pragma unroll 1
              for (int g = 0; g < kMergeSegs; ++g) {
              const uint32_t* po = p.part_o + ((int64_t)q * p.nslices * (kDv / 2) +
                                               cb * (kMergeCols / 2) + (half * kMergeSegs + g) * 4) * hs + h;
              float acc[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[e] = 0.f;
              for (int s0 = 0; s0 < ns; s0 += kMergeGroup) {
                float wv[kMergeGroup];
                uint32_t ov[kMergeGroup][4];
#pragma unroll
                for (int k2 = 0; k2 < kMergeGroup; ++k2) {
                  const bool live = s0 + k2 < ns;
                  const int64_t si = s0 + k2;
                  const float mk = live ? __ldcg(ml + si * 2 * hs) : -INFINITY;
                  const float ek = live ? (float)__ldcg(pe + si * (kDv / kPartChunk) * hs) : 0.f;
                  wv[k2] = ex2_approx(mk - M + ek);  // 0 for absent items
#pragma unroll
                  for (int i = 0; i < 4; ++i)
                    ov[k2][i] = live ? __ldcg(po + (si * (kDv / 2) + i) * hs) : 0u;
                }
#pragma unroll
                for (int k2 = 0; k2 < kMergeGroup; ++k2)
#pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    float lo, hi;
                    unpack_half2(ov[k2][i], lo, hi);
                    acc[2 * i] = fmaf(wv[k2], lo, acc[2 * i]);
                    acc[2 * i + 1] = fmaf(wv[k2], hi, acc[2 * i + 1]);
                  }
              }
              finish(q, h, cb * kMergeCols + (half * kMergeSegs + g) * 8, M, L, acc);
              }
            }
            __syncthreads();  // ctl.merge_ok may be rewritten by the next unit
          }
        }
        __syncthreads();  // ctl.kidx and s_mns are rewritten by the next chunk
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

struct WorkspaceLayout {
  size_t cidx, qcount, done, ml, e, o, total;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
int head_stride(int hq) { return (hq + 31) & ~31; }

WorkspaceLayout workspace_layout(int32_t nq, int32_t hq, int32_t topk) {
  WorkspaceLayout w;
  const int nslices = (topk + kItemKeys - 1) / kItemKeys;
  w.cidx = 0;
  w.qcount = align256((size_t)nq * topk * sizeof(int32_t));
  w.done = w.qcount + align256((size_t)nq * sizeof(int32_t));
  w.ml = w.done + align256((size_t)nq * sizeof(int32_t));
  w.e = w.o = w.total = w.ml;
  if (nslices > 1) {
    const size_t hs = (size_t)head_stride(hq);
    w.e = w.ml + align256((size_t)nq * nslices * 2 * hs * sizeof(float));
    w.o = w.e + align256((size_t)nq * nslices * (kDv / kPartChunk) * hs);
    w.total = w.o + (size_t)nq * nslices * (kDv / 2) * hs * sizeof(uint32_t);
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
  pp.done = a.topk > 0 ? reinterpret_cast<int32_t*>(ws + wl.done) : nullptr;
  pp.out = reinterpret_cast<__nv_bfloat16*>(a.out);
  pp.lse = a.lse;
  cudaError_t e = launch_dependent(sparse_index_plan_kernel, dim3((unsigned)a.num_queries),
                                   dim3(kThreads), 0, a.stream, pp);
  if (e == cudaSuccess) e = cudaGetLastError();
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
  p.part_o = nslices > 1 ? reinterpret_cast<uint32_t*>(ws + wl.o) : nullptr;
  p.part_e = nslices > 1 ? reinterpret_cast<int8_t*>(ws + wl.e) : nullptr;
  p.head_stride = head_stride(a.num_q_heads);
  p.done = pp.done;
  p.err = device_error_word();

  // the partials viewed as [query x item][512 columns][head_stride] (O) and
  // [query x item x 2][head_stride] (m, l), fp32, for the TMA-fed merge
  CUtensorMap tp, tp1, tml, te;
  memset(&tp, 0, sizeof tp);
  memset(&tp1, 0, sizeof tp1);
  memset(&tml, 0, sizeof tml);
  memset(&te, 0, sizeof te);
  if (nslices > 1) {
    const int64_t pitems = (int64_t)a.num_queries * nslices;
    if (pitems * 2 >= ((int64_t)1 << 31))
      return fail(SA_ERR_UNSUPPORTED, "%s: %lld partial items", fn, (long long)pitems);
    const uint32_t bh = (uint32_t)std::min(128, p.head_stride);
    const uint64_t dp[3] = {(uint64_t)p.head_stride, (uint64_t)(kDv / 2), (uint64_t)pitems};
    const uint64_t sp[2] = {(uint64_t)p.head_stride * 4, (uint64_t)p.head_stride * 4 * (kDv / 2)};
    const uint32_t bp[3] = {bh, (uint32_t)(kMergeCols / 2), (uint32_t)kMergeGroup};
    const uint32_t bp1[3] = {bh, (uint32_t)(kMergeCols / 2), 1u};
    const uint64_t de[3] = {(uint64_t)p.head_stride, (uint64_t)(kDv / kPartChunk), (uint64_t)pitems};
    const uint64_t se[2] = {(uint64_t)p.head_stride, (uint64_t)p.head_stride * (kDv / kPartChunk)};
    const uint32_t be[3] = {bh, 1u, (uint32_t)kMergeGroup};
    const uint64_t dm[2] = {(uint64_t)p.head_stride, (uint64_t)pitems * 2};
    const uint64_t sm_[1] = {(uint64_t)p.head_stride * 4};
    const uint32_t bm[2] = {bh, (uint32_t)(2 * kMergeGroup)};
    if (!encode_tiled(&tp, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, p.part_o, dp, sp, bp,
                      CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tiled(&tp1, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, p.part_o, dp, sp, bp1,
                      CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tiled(&te, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, p.part_e, de, se, be,
                      CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tiled(&tml, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p.part_ml, dm, sm_, bm,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
      return SA_ERR_INVALID_ARG;
  }
  const size_t smem = 1024 + (size_t)kNumSlots * kSlotBytes + 2 * (size_t)kSlabBytesQ;
  auto kern = sparse_index_fwd_kernel<MODE, FP8>;
  if (!set_dynamic_smem_once((const void*)kern, (int)smem))
    return fail(SA_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(cudaGetLastError()));
  // persistent: at most one CTA per SM (the shared memory allows one, and the
  // merge waits rely on every CTA being resident), none beyond the most work
  // there can be (one item per query and 256 index slots, per head block)
  const int64_t max_work = (int64_t)a.num_queries * nslices * p.nhb;
  if (max_work >= ((int64_t)1 << 31))
    return fail(SA_ERR_UNSUPPORTED, "%s: %lld work items", fn, (long long)max_work);
  const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(max_work, num_sms()));
  e = launch_dependent(kern, dim3(grid), dim3(kThreads), smem, a.stream, tq, tp, tp1, tml, te,
                       a.kv, p);
  if (e != cudaSuccess) return fail(SA_ERR_CUDA, "%s launch: %s", fn, cudaGetErrorString(e));
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

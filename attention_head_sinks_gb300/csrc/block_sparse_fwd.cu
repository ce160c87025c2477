// block_sparse_fwd.cu -- block-sparse causal attention with packed documents
// and a per-head NULL_LOGIT sink (DSA-style prefill).
//
// Operation: NeMo AutoModel "nemo_automodel.components.models.minimax_m3_vl.
// cp_sparse_attn", MiniMaxM3CPSparseAttention step 4 -- each query attends
// the key blocks selected for it, with token-level causality; the packed
// document mask and the zero output of fully masked rows come from
// _local_sparse_forward.  Key set of token i (row position p, document start
// d): { j in i's batch row : block(j) selected by i, d <= j <= p }.  The sink
// follows afierka-intel/vllm pull 76, Implementation (folded after the key
// loop, LSE over real keys only).  KEY0_BIAS adds s_h to the logit of the first
// key of the token's document (vLLM pull 49815, second paragraph, with
// documents as the sequences), when that key is in the token's set.
//
// With several index heads (one selection each, [M3 CP sparse]
// _select_local_blocks), a KV head's query heads share one: KV head g reads
// the table of index head g / (Hkv / Hi).
// Tile: M = 128 rows = (128 / G) consecutive tokens x the G query heads of
// one KV head (row = token * G + head).  Keys: the union, over the tile's
// tokens, of their selected blocks that intersect [document start, token] --
// built in shared memory as a bitmap over the batch row's blocks, compacted
// to an ascending list, with a per-block bitmask of the tokens that chose it.
// The loop walks that list two 64-key blocks per step:
//   S_j = Q K_j^T (N = 128) into one of two TMEM buffers,
//   softmax over S_j with per-element selection / causal / document masks
//   (a KEY0_BIAS sink is first added to the document's first-key logit in
//   S_j itself, so the softmax has no sink term),
//   P_j (bf16) written over S_j, O += P_j V_j with P_j read from TMEM.
// Persistent: one CTA per SM walks tiles blockIdx.x + n * gridDim.x.
// Warp roles: warp 2 allocates TMEM, then builds each tile's metadata (token
// positions, union list, token masks) a tile ahead into one of two buffers;
// thread 0 streams K, thread 96 streams Q and V (separate two-stage rings);
// thread 32 issues the MMAs; warps 4..11 run the softmax and the epilogue:
// warps w and w + 4 read TMEM lanes 32 (w mod 4) ... and split each step's
// two blocks (and the O columns) between them; each reads its 64 scores once
// per step.  mbarriers hand over every buffer (metadata, Q, K, V, S, P, O);
// step parities run on per-CTA step counters.
// The running max is rescaled lazily: O and l are rescaled only when a row's
// max grows by more than 2^8, so P stays below 256.
#include <cuda_bf16.h>

#include <algorithm>
#include <math.h>

#include "sa_internal.h"
#include "sa_ptx.cuh"

namespace sa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kD = 128;
constexpr int kBlk = 64;
constexpr int kStepKeys = 128;                 // two blocks per step
constexpr int kKStages = 2;                    // K ring
constexpr int kVStages = 2;                    // V ring
constexpr int kQSlab = 128 * 128;              // 128 rows x 64 dims, 16 KB
constexpr int kKVSlab = kStepKeys * 128;       // 128 keys x 64 dims, 16 KB
constexpr int kStepBytes = 2 * kKVSlab;        // K (or V) of one step: 2 slabs
constexpr int kMaxUnion = 1024;                // union blocks per tile (per metadata buffer)
constexpr int kMaxBitmapWords = 512;           // 16384 blocks per batch row
constexpr int kTmemCols = 512;
constexpr int kSBufs = 3;                      // S / P buffers in tensor memory
constexpr int kColO = kSBufs * 128;            // O after them
constexpr float kRescaleThreshold = 8.0f;
constexpr int kThreads = 384;  // warps 0..3: roles; 4..7 and 8..11: softmax parts 0 and 1

struct BlockParams {
  const int32_t* table;  // [Hi, T, topk]
  int64_t table_head_stride;  // T * topk
  int32_t kv_per_index_head;  // Hkv / Hi
  int32_t topk;
  int32_t seq_len;
  int32_t nblocks;
  int32_t total_tokens;
  const int32_t* cu_docs;
  int32_t num_docs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  const float* sinks;
  float scale_log2;
  __nv_bfloat16* out;  // [T, Hq, 128]
  float* lse;          // [Hq, T]
  uint32_t* err;
};

struct __align__(8) BlockSmemCtl {
  uint64_t q_full, q_empty;
  uint64_t k_full[kKStages];
  uint64_t k_empty[kKStages];
  uint64_t v_full[kVStages];
  uint64_t v_empty[kVStages];
  uint64_t s_full[kSBufs];
  uint64_t p_full[kSBufs];
  uint64_t o_done[2];       // [step parity]: one phase per such step, O += P V done
  uint64_t o_free;          // one phase per tile: its epilogue has read O
  uint64_t meta_full[2];    // tile metadata buffer [tile parity] written
  uint64_t meta_empty[2];   // ... and read by every role
  uint32_t tmem_base;
  int32_t abort_flag;       // a role's bounded wait ran out: every role stops
  int32_t sm_stop[2];       // the softmax warps' stop decision, by checkpoint parity
  int32_t nunion[2];
  float red_m[kSBufs][2][128];  // [step mod kSBufs][part][row]: row max exchange
  float red_l[2][2][128];   // [tile parity][part][row]: row sums at the end
  // per tile parity: row-local position (-1 past the last token), row-local
  // start of the token's document, KEY0_BIAS key (-1 if before the row)
  int32_t tok_pos[2][128];
  int32_t tok_lo[2][128];
  int32_t tok_k0[2][128];
  uint32_t bitmap[kMaxBitmapWords];  // scratch of the metadata warp
  int32_t prefix[kMaxBitmapWords];
};

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
__device__ __forceinline__ void bar_softmax() {  // the eight softmax warps
  asm volatile("bar.sync 1, 256;" ::: "memory");
}
// The two softmax warps that share a TMEM lane quadrant (warps w and w + 4,
// the two blocks of a step for the same 32 rows): named barrier 2 + w mod 4.
__device__ __forceinline__ void bar_softmax_pair(int warp) {
  asm volatile("bar.sync %0, 64;" ::"r"(2 + (warp & 3)) : "memory");
}

__device__ __forceinline__ int upper_doc(const int32_t* cu, int n, int t) {
  int lo = 0, hi = n - 1;  // largest e with cu[e] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return __ldg(cu + lo);
}

// Dynamic shared memory: Q, the K and V rings, and two metadata buffers
// (union list and its token masks).  (Measured: a third K stage, or a second
// Q buffer with the next tile's first S issued early, made the persistent
// kernel slower; the shared memory they take comes out of the L1 cache.)
__host__ __device__ constexpr size_t block_smem_bytes(int G) {
  return 1024 + 2 * (size_t)kQSlab + (size_t)kKStages * kStepBytes +
         (size_t)kVStages * kStepBytes +
         2 * ((size_t)kMaxUnion * 4 +
              (size_t)kMaxUnion * ((128 / G) > 32 ? (128 / G) / 32 : 1) * 4);
}

template <int G, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
block_sparse_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const BlockParams p) {
  constexpr int TQ = 128 / G;
  constexpr int TW = TQ > 32 ? TQ / 32 : 1;  // token-mask words per block
  constexpr int KST = kKStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ BlockSmemCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                                  // 2 x 16 KB
  uint8_t* sK = sQ + 2 * kQSlab;                       // KST x 32 KB
  uint8_t* sV = sK + KST * kStepBytes;                 // 2 x 32 KB
  int32_t* ulist2 = reinterpret_cast<int32_t*>(sV + kVStages * kStepBytes);   // [2][kMaxUnion]
  uint32_t* tokmask2 = reinterpret_cast<uint32_t*>(ulist2 + 2 * kMaxUnion);  // [2][kMaxUnion*TW]

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  // tiles of this CTA: blockIdx.x + n * gridDim.x over (KV head, token tile)
  const int ntx = p.total_tokens / TQ;
  const int ntiles = ntx * p.num_kv_heads;
  const int nmine = (ntiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  auto tile_of = [&](int n, int& g, int& tok0) {
    const int tt = (int)blockIdx.x + n * (int)gridDim.x;
    g = tt / ntx;
    tok0 = (tt - g * ntx) * TQ;
  };
  const int nwords = (p.nblocks + 31) >> 5;

  if (tid == 0) {
    mbar_init(&ctl.q_full, 1);
    mbar_init(&ctl.q_empty, 1);
    for (int s = 0; s < KST; ++s) {
      mbar_init(&ctl.k_full[s], 1);
      mbar_init(&ctl.k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&ctl.v_full[s], 1);
      mbar_init(&ctl.v_empty[s], 1);
    }
    for (int b = 0; b < kSBufs; ++b) {
      mbar_init(&ctl.s_full[b], 1);
      mbar_init(&ctl.p_full[b], 8);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl.meta_full[b], 1);
      mbar_init(&ctl.meta_empty[b], 11);  // 8 softmax warps, K, V, MMA
    }
    mbar_init(&ctl.o_done[0], 1);
    mbar_init(&ctl.o_done[1], 1);
    mbar_init(&ctl.o_free, 8);
    ctl.abort_flag = 0;
    ctl.sm_stop[0] = ctl.sm_stop[1] = 0;
    fence_mbar_init();
    tma_prefetch_map(&tm_q);
    tma_prefetch_map(&tm_k);
    tma_prefetch_map(&tm_v);
  }
  if (warp == 2) {
    tmem_alloc(&ctl.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  volatile int32_t* abort_flag = &ctl.abort_flag;
  // A bounded wait that ran out stops every role: each checks the flag
  // before its next wait, so a failure costs at most one more time-out per
  // role instead of one per remaining step.
  auto wait_or_abort = [&](uint64_t* bar, uint32_t parity, uint32_t site) -> bool {
    if (*abort_flag) return false;
    if (mbar_wait(bar, parity, p.err, site)) return true;
    *abort_flag = 1;
    return false;
  };

  if (warp == 2) {
    // ---- metadata of each tile (one warp), a tile ahead of the others --------
    for (int n = 0; n < nmine; ++n) {
      const int tb = n & 1;
      if (n >= 2 && !wait_or_abort(&ctl.meta_empty[tb], ((n >> 1) - 1) & 1, kErrWaitFree)) break;
      int g, tok0;
      tile_of(n, g, tok0);
      const int row_start = (tok0 / p.seq_len) * p.seq_len;
      int32_t* tpos = ctl.tok_pos[tb];
      int32_t* tlo = ctl.tok_lo[tb];
      for (int i = lane; i < TQ; i += 32) {
        const int t = tok0 + i;
        if (t < p.total_tokens) {
          const int doc = upper_doc(p.cu_docs, p.num_docs, t);
          tpos[i] = t - row_start;
          tlo[i] = max(doc - row_start, 0);
          ctl.tok_k0[tb][i] = doc >= row_start ? doc - row_start : -1;
        } else {
          tpos[i] = -1;
          tlo[i] = 0;
          ctl.tok_k0[tb][i] = -1;
        }
      }
      for (int w = lane; w < nwords; w += 32) ctl.bitmap[w] = 0u;
      __syncwarp();
      // the selection of this KV head's index head, rows of the tile's tokens
      const int32_t* table = p.table + (int64_t)(g / p.kv_per_index_head) * p.table_head_stride +
                             (int64_t)tok0 * p.topk;
      const int npairs = TQ * p.topk;
      // pair w = (token i, entry): its block b is live when it intersects
      // [document start, position]
      auto live_block = [&](int w, int& i, int& b) -> bool {
        i = w / p.topk;
        b = __ldg(table + w);
        const int pos = tpos[i];
        return pos >= 0 && b >= 0 && b < p.nblocks && b * kBlk <= pos &&
               b * kBlk + kBlk - 1 >= tlo[i];
      };
      for (int w = lane; w < npairs; w += 32) {
        int i, b;
        if (live_block(w, i, b)) atomicOr(&ctl.bitmap[b >> 5], 1u << (b & 31));
      }
      __syncwarp();
      {
        // exclusive prefix of popcounts over the bitmap words
        const int per = (nwords + 31) >> 5;
        int local = 0;
        for (int k = 0; k < per; ++k) {
          const int w = lane * per + k;
          if (w < nwords) local += __popc(ctl.bitmap[w]);
        }
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        int run = incl - local;
        for (int k = 0; k < per; ++k) {
          const int w = lane * per + k;
          if (w < nwords) {
            ctl.prefix[w] = run;
            run += __popc(ctl.bitmap[w]);
          }
        }
        if (lane == 31) ctl.nunion[tb] = incl;
      }
      __syncwarp();
      const int U = ctl.nunion[tb];
      int32_t* ulist = ulist2 + tb * kMaxUnion;
      uint32_t* tokmask = tokmask2 + tb * kMaxUnion * TW;
      for (int w = lane; w < nwords; w += 32) {
        uint32_t bits = ctl.bitmap[w];
        int o = ctl.prefix[w];
        while (bits) {
          const int b = __ffs(bits) - 1;
          bits &= bits - 1;
          ulist[o++] = w * 32 + b;
        }
      }
      for (int w = lane; w < U * TW; w += 32) tokmask[w] = 0u;
      __syncwarp();
      for (int w = lane; w < npairs; w += 32) {
        int i, b;
        if (live_block(w, i, b)) {
          const uint32_t word = ctl.bitmap[b >> 5];
          const int u = ctl.prefix[b >> 5] + __popc(word & ((1u << (b & 31)) - 1u));
          atomicOr(&tokmask[u * TW + (i >> 5)], 1u << (i & 31));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.meta_full[tb]);
    }
  } else if (tid == 0) {
    // ---- K producer: runs KST steps ahead of S, across tile boundaries -------
    int gk = 0, issued = 0;
    for (int n = 0; n < nmine; ++n) {
      const int tb = n & 1;
      if (!wait_or_abort(&ctl.meta_full[tb], (n >> 1) & 1, kErrWaitLoad)) break;
      int g, tok0;
      tile_of(n, g, tok0);
      const int row_start = (tok0 / p.seq_len) * p.seq_len;
      const int U = ctl.nunion[tb];
      const int32_t* ulist = ulist2 + tb * kMaxUnion;
      bool pok = true;
      for (int j = 0; 2 * j < U; ++j, ++gk) {
        const int st = gk % KST;
        if (gk >= KST && !(pok = wait_or_abort(&ctl.k_empty[st], ((gk / KST) - 1) & 1, kErrWaitFree)))
          break;
        const int nb = min(2, U - 2 * j);
        uint8_t* stage = sK + st * kStepBytes;
        mbar_arrive_expect_tx(&ctl.k_full[st], (uint32_t)nb * 2u * (kBlk * 128));
        for (int bi = 0; bi < nb; ++bi) {
          const int kpos = row_start + ulist[2 * j + bi] * kBlk;
          for (int s = 0; s < 2; ++s)
            tma_load_3d(stage + s * kKVSlab + bi * (kBlk * 128), &tm_k, &ctl.k_full[st], 64 * s,
                        g, kpos);
        }
        issued = gk + 1;
      }
      mbar_arrive(&ctl.meta_empty[tb]);
      if (!pok) break;
    }
    if (*abort_flag) {
      // bounded drain of the copies still in flight
      for (int q = max(0, issued - KST); q < issued; ++q)
        mbar_wait(&ctl.k_full[q % KST], (q / KST) & 1, p.err, kErrWaitDrain);
    }
  } else if (tid == 96) {
    // ---- Q and V producer: Q of a tile once the previous tile's last S has
    // read Q, then V two steps ahead of P V ----------------------------------
    int gv = 0, issued = 0, nq = 0;
    for (int n = 0; n < nmine; ++n) {
      const int tb = n & 1;
      if (!wait_or_abort(&ctl.meta_full[tb], (n >> 1) & 1, kErrWaitLoad)) break;
      int g, tok0;
      tile_of(n, g, tok0);
      const int row_start = (tok0 / p.seq_len) * p.seq_len;
      const int U = ctl.nunion[tb];
      const int32_t* ulist = ulist2 + tb * kMaxUnion;
      if (n >= 1 && !wait_or_abort(&ctl.q_empty, (n - 1) & 1, kErrWaitFree)) {
        mbar_arrive(&ctl.meta_empty[tb]);
        break;
      }
      mbar_arrive_expect_tx(&ctl.q_full, 2 * kQSlab);
      for (int s2 = 0; s2 < 2; ++s2)
        tma_load_3d(sQ + s2 * kQSlab, &tm_q, &ctl.q_full, 64 * s2, g * G, tok0);
      nq = n + 1;
      bool pok = true;
      for (int j = 0; 2 * j < U; ++j, ++gv) {
        const int st = gv % kVStages;
        if (gv >= kVStages &&
            !(pok = wait_or_abort(&ctl.v_empty[st], ((gv / kVStages) - 1) & 1, kErrWaitFree)))
          break;
        const int nb = min(2, U - 2 * j);
        uint8_t* stage = sV + st * kStepBytes;
        mbar_arrive_expect_tx(&ctl.v_full[st], (uint32_t)nb * 2u * (kBlk * 128));
        for (int bi = 0; bi < nb; ++bi) {
          const int kpos = row_start + ulist[2 * j + bi] * kBlk;
          for (int s = 0; s < 2; ++s)
            tma_load_3d(stage + s * kKVSlab + bi * (kBlk * 128), &tm_v, &ctl.v_full[st], 64 * s,
                        g, kpos);
        }
        issued = gv + 1;
      }
      mbar_arrive(&ctl.meta_empty[tb]);
      if (!pok) break;
    }
    if (*abort_flag) {
      for (int q = max(0, issued - kVStages); q < issued; ++q)
        mbar_wait(&ctl.v_full[q % kVStages], (q / kVStages) & 1, p.err, kErrWaitDrain);
      if (nq > 0) mbar_wait(&ctl.q_full, (nq - 1) & 1, p.err, kErrWaitDrain);
    }
  } else if (tid == 32) {
    // ---- MMA issuer ----------------------------------------------------------
    int gs = 0;  // steps of earlier tiles: S / P buffers and o_done phases
    for (int n = 0; n < nmine; ++n) {
      const int tb = n & 1;
      if (!wait_or_abort(&ctl.meta_full[tb], (n >> 1) & 1, kErrWaitLoad)) break;
      const int U = ctl.nunion[tb];
      const int nsteps = (U + 1) >> 1;
      bool ok = wait_or_abort(&ctl.q_full, n & 1, kErrWaitLoad);
      if (ok && nsteps == 0) mbar_arrive(&ctl.q_empty);  // Q unused: release it
      auto issue_s = [&](int j) -> bool {
        const int gj = gs + j;
        const int st = gj % kSBufs;  // S buffer
        const int ks = gj % KST;
        if (!wait_or_abort(&ctl.k_full[ks], (gj / KST) & 1, kErrWaitLoad)) return false;
        tc_fence_after();
        const int nb = min(2, U - 2 * j);
        const uint32_t idesc = idesc_bf16(128, nb * kBlk, false);
        const uint8_t* kst = sK + ks * kStepBytes;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t a = smem_desc(smem_u32(sQ + s * kQSlab) + kk * 32, 16, 1024, kLayoutSw128);
            const uint64_t b = smem_desc(smem_u32(kst + s * kKVSlab) + kk * 32, 16, 1024, kLayoutSw128);
            mma_ss(tmem + (uint32_t)(st * 128), a, b, idesc, (s | kk) ? 1u : 0u);
          }
        }
        mma_commit(&ctl.k_empty[ks]);
        if (j == nsteps - 1) mma_commit(&ctl.q_empty);  // the tile's last read of Q
        mma_commit(&ctl.s_full[st]);
        return true;
      };
      // S runs kSBufs - 1 steps ahead of P V: S(j + 2) goes to the pipe
      // before P V(j), so the softmax of step j has two S's worth of tensor
      // time to finish in before the pipe would wait for it
      for (int j = 0; j < kSBufs - 1 && j < nsteps && ok; ++j) ok = issue_s(j);
      for (int j = 0; j < nsteps && ok; ++j) {
        if (j + kSBufs - 1 < nsteps) {
          ok = issue_s(j + kSBufs - 1);
          if (!ok) break;
        }
        const int gj = gs + j;
        const int st = gj % kSBufs;
        ok = wait_or_abort(&ctl.p_full[st], (gj / kSBufs) & 1, kErrWaitMma);
        if (!ok) break;
        // the first P V of a tile overwrites O: the previous epilogue must have read it
        if (j == 0 && n > 0) {
          ok = wait_or_abort(&ctl.o_free, (n - 1) & 1, kErrWaitFree);
          if (!ok) break;
        }
        const int vs = gj % kVStages;
        ok = wait_or_abort(&ctl.v_full[vs], (gj / kVStages) & 1, kErrWaitLoad);
        if (!ok) break;
        tc_fence_after();
        const int nb = min(2, U - 2 * j);
        const uint32_t idesc = idesc_bf16(128, kD, true);
        const uint8_t* vst = sV + vs * kStepBytes;
        for (int kk = 0; kk < nb * kBlk / 16; ++kk) {
          const uint64_t b = smem_desc(smem_u32(vst) + kk * 16 * 128, kKVSlab, 1024, kLayoutSw128);
          // P of block kk / 4 sits in the first half of that block's S columns
          mma_ts(tmem + kColO, tmem + (uint32_t)(st * 128 + 64 * (kk >> 2) + 8 * (kk & 3)), b,
                 idesc, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&ctl.v_empty[vs]);
        mma_commit(&ctl.o_done[gj & 1]);
      }
      mbar_arrive(&ctl.meta_empty[tb]);
      if (!ok) break;
      gs += nsteps;
    }
  } else if (warp >= 4) {
    // ---- softmax + epilogue -------------------------------------------------
    // Thread (row, part): row = TMEM lane, part = which of the step's two
    // 64-key blocks it owns (S columns [64 part, 64 part + 64)); warps w and
    // w + 4 share the 32 lanes of quadrant w mod 4.  The row max meets in
    // shared memory once per step; each part keeps its own row sum.
    const int part = (warp - 4) >> 2;
    const int row = (warp & 3) * 32 + lane;
    const int tok = row / G;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const float c2 = p.scale_log2;
    int gs = 0, cp = 0;
    // The eight warps share named barrier 1, which has no time limit, so they
    // stop together or not at all: a failure is posted before a barrier and
    // every thread reads the decision right after it (the slot alternates, so
    // a later post cannot race a late reader).
    // P V of global step k is complete.  Steps alternate between two
    // barriers, so a barrier is never more than one phase past the step
    // waited for: the next step on it needs this thread's P first.
    auto wait_pv = [&](int k) -> bool {
      return wait_or_abort(&ctl.o_done[k & 1], (uint32_t)(k >> 1) & 1u, kErrWaitMma);
    };
    auto checkpoint = [&](bool fail) -> bool {
      if (fail) ctl.sm_stop[cp & 1] = 1;
      if (warp == 4 && lane == 0 && *abort_flag) ctl.sm_stop[cp & 1] = 1;
      bar_softmax();
      const bool stop = ctl.sm_stop[cp & 1] != 0;
      ++cp;
      return stop;
    };
    for (int n = 0; n < nmine; ++n) {
      const int tb = n & 1;
      const bool meta_ok = wait_or_abort(&ctl.meta_full[tb], (n >> 1) & 1, kErrWaitLoad);
      if (checkpoint(!meta_ok)) break;
      bool ok = true;
      int g, tok0;
      tile_of(n, g, tok0);
      const int h = g * G + (row % G);
      const int t = tok0 + tok;
      const int pos = ctl.tok_pos[tb][tok];
      const int dlo = ctl.tok_lo[tb][tok];
      const int k0 = ctl.tok_k0[tb][tok];
      const int U = ctl.nunion[tb];
      const int nsteps = (U + 1) >> 1;
      const int32_t* ulist = ulist2 + tb * kMaxUnion;
      const uint32_t* tokmask = tokmask2 + tb * kMaxUnion * TW;
      const float k0_sink2 = (MODE == SA_SINK_KEY0_BIAS) ? __ldg(p.sinks + h) * kLog2e : 0.f;
      float m_use = -INFINITY, l = 0.f;

      for (int j = 0; j < nsteps; ++j) {
        const int gj = gs + j;
        const int st = gj % kSBufs;
        ok = wait_or_abort(&ctl.s_full[st], (gj / kSBufs) & 1, kErrWaitMma) && ok;
        __syncwarp();
        tc_fence_after();
        // live columns of this thread's block: [clo, chi] within the block
        const int u = 2 * j + part;
        int clo = 1 << 30, chi = 1 << 30;
        int k0c = -1;  // KEY0_BIAS: column of the document's first key in this block
        if (u < U && pos >= 0 && ((tokmask[u * TW + (tok >> 5)] >> (tok & 31)) & 1u)) {
          const int bs = ulist[u] * kBlk;
          clo = max(dlo, bs) - bs;
          chi = min(pos, bs + kBlk - 1) - bs;
          if (MODE == SA_SINK_KEY0_BIAS) {
            if (k0 >= bs && k0 < bs + kBlk) k0c = k0 - bs;  // then k0c == clo: live
          }
        }
        const uint32_t span = (uint32_t)(chi - clo);
        const bool warp_live = __any_sync(0xffffffffu, clo != (1 << 30));
        const uint32_t sbase = lane_base + (uint32_t)(st * 128 + 64 * part);
        float s[2][32];
        float mx = -INFINITY;
        if (warp_live) {
          // KEY0_BIAS: the sink goes onto the first key's logit in S itself
          // (raw units), so the softmax below is the no-sink one; only warps
          // with a document's first key in this block do anything
          if (MODE == SA_SINK_KEY0_BIAS && __any_sync(0xffffffffu, k0c >= 0))
            tmem_add_lane_column(sbase, k0c, k0_sink2 / c2);
          tmem_ld32(sbase, s[0]);
          tmem_ld32(sbase + 32, s[1]);
          tmem_wait_ld();
          float mr[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              s[c][e] = ((uint32_t)(32 * c + e - clo) <= span) ? s[c][e] : -INFINITY;
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int e = 0; e < 32; e += 2)
              mr[(e >> 1) & 3] = max3f(mr[(e >> 1) & 3], s[c][e], s[c][e + 1]);
          // max(s) * c2 == max(s * c2) exactly
          mx = fmaxf(fmaxf(mr[0], mr[1]), fmaxf(mr[2], mr[3])) * c2;
        }
        ctl.red_m[st][part][row] = mx;
        // only the two warps of these rows meet: the row max of the step
        bar_softmax_pair(warp);
        mx = fmaxf(ctl.red_m[st][0][row], ctl.red_m[st][1][row]);
        // lazy rescale of O and l when this row's max grew by more than 2^8
        const bool need = mx > m_use + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = need ? mx : m_use;
          const float alpha = need ? ex2_approx(m_use - m_new) : 1.f;
          if (j > 0) {
            // S(j) went to the pipe before P V(j - 2): both earlier steps
            // may still be running
            if (j > 1) ok = wait_pv(gj - 2) && ok;
            ok = wait_pv(gj - 1) && ok;
            __syncwarp();
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
              float o[32];
              const uint32_t oa = lane_base + kColO + 64 * part + 32 * c;
              tmem_ld32(oa, o);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] *= alpha;
              tmem_st32(oa, o);
            }
            tmem_wait_st();
            l *= alpha;
          }
          m_use = m_new;
        }
        if (warp_live) {
          // P = 2^(x - m) (bf16) into the first 32 columns of this block's S
          // region, behind this thread's own reads; masked columns give 0
          const float m_ref = (m_use == -INFINITY) ? 0.f : m_use;
          const uint64_t c2c2 = f2_pack(c2, c2), nmnm = f2_pack(-m_ref, -m_ref);
          uint64_t lp[4] = {0, 0, 0, 0};
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const uint64_t x = f2_fma(f2_pack(s[c][e], s[c][e + 1]), c2c2, nmnm);
              const float p0 = ex2_approx(f2_lo(x)), p1 = ex2_approx(f2_hi(x));
              lp[(e >> 1) & 3] = f2_add(lp[(e >> 1) & 3], f2_pack(p0, p1));
              pk[e >> 1] = pack_bf16x2(p0, p1);
            }
            tmem_st16(sbase + 16 * c, pk);
          }
          const uint64_t ls = f2_add(f2_add(lp[0], lp[1]), f2_add(lp[2], lp[3]));
          l += f2_lo(ls) + f2_hi(ls);
        } else if (u < U) {
          // block present for the tile but not for these rows: P = 0
          uint32_t z[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) z[e] = 0u;
          tmem_st16(sbase, z);
          tmem_st16(sbase + 16, z);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.p_full[st]);
      }
      if (nsteps > 0) {
        // O is final once the last P V is done.  S(last), whose completion is
        // all this thread has seen, went to the pipe before the P V of the
        // last kSBufs steps.  P V(last - 2) is not waited for by itself: its
        // barrier also carries P V(last), and a parity wait for it that began
        // after P V(last) had completed would wait for a phase that never
        // comes.  One thread issues every P V and each commit arrives only
        // after that thread's earlier MMAs, so once P V(last - 1) is seen,
        // P V(last - 2) has arrived and the wait for P V(last) is exact.
        for (int k = max(0, nsteps - 2); k < nsteps; ++k) ok = wait_pv(gs + k) && ok;
        __syncwarp();
        tc_fence_after();
      }
      ctl.red_l[tb][part][row] = l;
      const bool stop = checkpoint(!ok);  // (also the barrier of the row-sum exchange)
      const float lt = ctl.red_l[tb][0][row] + ctl.red_l[tb][1][row];
      // epilogue: this thread stores O columns [64 part, 64 part + 64)
      float inv = 0.f, lse = -INFINITY;
      if (m_use != -INFINITY) {
        float den = lt, alpha = 1.f;
        if (MODE == SA_SINK_NULL_LOGIT) {
          const float sink2 = __ldg(p.sinks + h) * kLog2e;
          const float mp = fmaxf(m_use, sink2);
          alpha = ex2_approx(m_use - mp);
          den = lt * alpha + ex2_approx(sink2 - mp);
        }
        inv = alpha / den;
        lse = (m_use + log2f(lt)) * kLn2;
      }
      const bool row_valid = pos >= 0;
      __nv_bfloat16* orow = p.out + ((int64_t)t * p.num_q_heads + h) * kD + 64 * part;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        float o[32];
        if (nsteps > 0) {
          tmem_ld32(lane_base + kColO + 64 * part + 32 * c, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0.f;
        }
        if (row_valid) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack_bf16x2(o[8 * q4 + 0] * inv, o[8 * q4 + 1] * inv);
            w.y = pack_bf16x2(o[8 * q4 + 2] * inv, o[8 * q4 + 3] * inv);
            w.z = pack_bf16x2(o[8 * q4 + 4] * inv, o[8 * q4 + 5] * inv);
            w.w = pack_bf16x2(o[8 * q4 + 6] * inv, o[8 * q4 + 7] * inv);
            *reinterpret_cast<uint4*>(orow + 32 * c + 8 * q4) = w;
          }
        }
      }
      // O has been read: the next tile's first P V may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.o_free);
      if (row_valid && part == 0) p.lse[(int64_t)h * p.total_tokens + t] = lse;
      if (lane == 0) mbar_arrive(&ctl.meta_empty[tb]);
      if (stop) {
        *abort_flag = 1;
        break;
      }
      gs += nsteps;
    }
  }

  // ---- teardown ----------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int G, int MODE>
sa_status launch_typed(const BlockArgs& a) {
  constexpr int TQ = 128 / G;
  static_assert(block_smem_bytes(G) + sizeof(BlockSmemCtl) <= 227 * 1024, "shared memory");
  const int64_t T = (int64_t)a.batch * a.seq_len;
  CUtensorMap tq, tk, tv;
  const uint64_t dq[3] = {(uint64_t)kD, (uint64_t)a.num_q_heads, (uint64_t)T};
  const uint64_t sq[2] = {(uint64_t)kD * 2, (uint64_t)a.num_q_heads * kD * 2};
  const uint32_t bq[3] = {64, (uint32_t)G, (uint32_t)TQ};
  const uint64_t dk[3] = {(uint64_t)kD, (uint64_t)a.num_kv_heads, (uint64_t)T};
  const uint64_t sk[2] = {(uint64_t)kD * 2, (uint64_t)a.num_kv_heads * kD * 2};
  const uint32_t bk[3] = {64, 1, (uint32_t)kBlk};
  if (!encode_tiled(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.q, dq, sq, bq,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.k, dk, sk, bk,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.v, dk, sk, bk,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return SA_ERR_INVALID_ARG;
  BlockParams p;
  p.table = a.block_table;
  p.table_head_stride = T * a.topk_blocks;
  p.kv_per_index_head = a.num_kv_heads / a.num_index_heads;
  p.topk = a.topk_blocks;
  p.seq_len = a.seq_len;
  p.nblocks = a.seq_len / kBlk;
  p.total_tokens = (int32_t)T;
  p.cu_docs = a.cu_docs;
  p.num_docs = a.num_docs;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.sinks = a.sinks;
  p.scale_log2 = a.softmax_scale * kLog2e;
  p.out = reinterpret_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.err = device_error_word();
  const size_t smem = block_smem_bytes(G);
  auto kern = block_sparse_fwd_kernel<G, MODE>;
  if (!set_dynamic_smem_once((const void*)kern, (int)smem))
    return fail(SA_ERR_CUDA, "sa_block_sparse_fwd: %s", cudaGetErrorString(cudaGetLastError()));
  cudaError_t e;
  // persistent: one CTA per SM (the shared memory allows one), each walking
  // tiles blockIdx.x, blockIdx.x + grid, ...
  const int64_t ntiles = (T / TQ) * a.num_kv_heads;
  const unsigned grid = (unsigned)std::min<int64_t>(ntiles, num_sms());
  kern<<<grid, kThreads, smem, a.stream>>>(tq, tk, tv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(SA_ERR_CUDA, "sa_block_sparse_fwd launch: %s", cudaGetErrorString(e));
  return SA_OK;
}

template <int G>
sa_status by_mode(const BlockArgs& a) {
  if (a.sink_mode == SA_SINK_NULL_LOGIT) return launch_typed<G, SA_SINK_NULL_LOGIT>(a);
  if (a.sink_mode == SA_SINK_KEY0_BIAS) return launch_typed<G, SA_SINK_KEY0_BIAS>(a);
  return launch_typed<G, SA_SINK_NONE>(a);
}

}  // namespace

sa_status launch_block_sparse_fwd(const BlockArgs& a) {
  const int G = a.num_q_heads / a.num_kv_heads;
  const char* fn = "sa_block_sparse_fwd";
  if (a.head_dim != kD)
    return fail(SA_ERR_UNSUPPORTED, "%s: head_dim %d (supported: 128)", fn, a.head_dim);
  if (a.block_size != kBlk)
    return fail(SA_ERR_UNSUPPORTED, "%s: block_size %d (supported: 64)", fn, a.block_size);
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16)
    return fail(SA_ERR_UNSUPPORTED,
                "%s: num_q_heads / num_kv_heads = %d (supported: 1, 2, 4, 8, 16)", fn, G);
  if (a.seq_len % 128 != 0)
    return fail(SA_ERR_UNSUPPORTED, "%s: seq_len %d is not a multiple of 128", fn, a.seq_len);
  if (a.seq_len / kBlk > kMaxBitmapWords * 32)
    return fail(SA_ERR_UNSUPPORTED, "%s: seq_len %d above %d", fn, a.seq_len,
                kMaxBitmapWords * 32 * kBlk);
  // blocks in a tile's union: at most its selections and at most the row's blocks
  if (std::min<int64_t>((int64_t)(128 / G) * a.topk_blocks, a.seq_len / kBlk) > kMaxUnion)
    return fail(SA_ERR_UNSUPPORTED,
                "%s: %d tokens per tile x topk_blocks %d (and %d blocks per row) above %d "
                "union blocks per tile",
                fn, 128 / G, a.topk_blocks, a.seq_len / kBlk, kMaxUnion);
  switch (G) {
    case 1: return by_mode<1>(a);
    case 2: return by_mode<2>(a);
    case 4: return by_mode<4>(a);
    case 8: return by_mode<8>(a);
    default: return by_mode<16>(a);
  }
}

}  // namespace sa

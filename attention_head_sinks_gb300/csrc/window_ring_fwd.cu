// window_ring_fwd.cu -- persistent sliding-window attention with per-head
// sinks: a sliding ring of K/V blocks in shared memory, warp-specialised
// tcgen05 pipeline, two softmax warpgroups on double-buffered tensor memory.
//
// Operation: vLLM pull 49815 "[Bugfix][MiMo] Apply vision attention sinks in
// the window attention path" (sink on each sequence's first key; LSE of the
// masked scaled logits, (nheads, total_q)); NULL_LOGIT per afierka-intel/vllm
// pull 76, Implementation.  Same tile and per-row math as window_fwd.cu
// (window_common.cuh); what differs is the schedule.
//
// Work: items (KV head g, tile j) with tile = (128 / G) tokens x G query heads
// (M = 128).  Each CTA takes a contiguous range of items, so consecutive items
// of one head share all but their newest keys.  Keys are handled in blocks of
// KB = min(128 / G, 64) tokens aligned to multiples of KB; a tile needs NBT
// consecutive blocks and the next tile of the same head TQ / KB new ones.  The
// producer loads only those new blocks into a ring of NR slots, so K and V are
// read from memory about once.
//
// Warps: 0 = TMA producer of Q and of the even ring blocks, 1 = MMA issuer,
// 2 = TMEM owner, 3 = TMA producer of the odd ring blocks (one thread's TMA
// copies complete one after another, about one transaction per 0.3 us, so
// the ring refills go through two issuing threads), 4..7 and 8..11 =
// softmax warpgroups 0 and 1, which take alternate items.  Tensor memory: two
// 256-column buffers (one per warpgroup), each holding S [128 x NBT*KB] at
// column 0, P (bf16) in place over it, and O [128 x D] at column 128.
// The MMA warp issues S of the next item before P V of the current one when
// both belong to the same head run, so the tensor pipe works on item i+1 while
// a warpgroup runs the softmax of item i.
#include <cuda_bf16.h>

#include <algorithm>
#include <math.h>

#include "sa_internal.h"
#include "sa_ptx.cuh"
#include "window_common.cuh"

namespace sa {
namespace {

constexpr int kNQ = 2;            // Q stages
constexpr int kRingBudget = 220 * 1024;
constexpr int kBufCols = 256;     // TMEM columns per buffer
constexpr int kColO = 128;        // O within a buffer

// Shared-memory layout.  A TMA copy spends about the same time on every row
// segment it moves, whatever its width (measured: 32-byte rows cap a copy
// stream near 20 GB/s per SM, 128-byte rows reach 37), so the rows are cut as
// wide as the MMA operand layouts allow:
//   Q and K (K-major): D / 64 chunks of 64 dimensions in 128-byte swizzled
//   rows, then (D mod 64) / 16 slabs of 16 in 32-byte swizzled rows;
//   V (the MN-major B operand of P V): atoms of 64 dimensions (128-byte
//   swizzle) when D is a multiple of 64, else of 32 (64-byte swizzle) with the
//   last atom zero-filled past D by the copy; P V then runs with N = VN >= D
//   and the columns past D are ignored.
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(map),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}

template <int D, int G>
struct RingShape {
  static constexpr int TQ = 128 / G;
  static constexpr int KB = TQ < 64 ? TQ : 64;
  static constexpr int NEWB = TQ / KB;
  static constexpr int NC = D / 64;                 // 64-dim chunks of Q and K
  static constexpr int NT = (D % 64) / 16;          // 16-dim tail slabs of Q and K
  static constexpr bool V128 = (D % 64) == 0;
  static constexpr int VW = V128 ? 64 : 32;         // dims per V atom
  static constexpr int VA = (D + VW - 1) / VW;      // V atoms
  static constexpr int VN = VA * VW;                // N of P V
  static constexpr int QC = 128 * 128;              // bytes of one Q chunk
  static constexpr int QT = 128 * 32;               // bytes of one Q tail slab
  static constexpr int QBYTES = NC * QC + NT * QT;  // one Q stage
  static constexpr int SLOT = KB * (NC * 128 + NT * 32 + VA * VW * 2);  // K + V of one block
  static constexpr int NR_FIT = (kRingBudget - kNQ * QBYTES) / SLOT;
  static constexpr int NR = NR_FIT > 16 ? 16 : NR_FIT;
  // K and V are stored array by array over the whole ring: in each array
  // slot k holds keys [k KB, (k + 1) KB), so consecutive slots are
  // consecutive rows and one MMA can span several blocks
  static constexpr int KC_BYTES = NR * KB * 128;    // one K chunk array
  static constexpr int KT_BYTES = NR * KB * 32;     // one K tail array
  static constexpr int VA_BYTES = NR * KB * VW * 2; // one V atom array
  static constexpr size_t SMEM = 1024 + (size_t)kNQ * QBYTES + (size_t)NR * SLOT;
  static_assert(VN <= 256 - kColO, "O fits its buffer");
};

struct RingParams {
  const int32_t* cu_seqlens;
  int32_t num_seqs;
  int32_t total_tokens;
  int32_t num_q_heads;
  int32_t wl, wr;
  int32_t nt;       // tiles per head
  int32_t items;    // nt * num_kv_heads
  int32_t num_kv_heads;
  int32_t chunks;   // token chunks per head (main CTAs: chunks * num_kv_heads)
  int32_t chunk_size;      // tiles per main CTA, or 0: nt split evenly over chunks
  int32_t spill_per_head;  // last tiles of every head left to the spill CTAs
  int32_t nbt;      // key blocks per tile
  int32_t bf_off;   // first block of tile j = j * NEWB + bf_off
  const float* sinks;
  float scale_log2;
  __nv_bfloat16* out;
  float* lse;
  uint32_t* err;
};

template <int NR>
struct __align__(8) RingCtl {
  uint64_t q_full[kNQ], q_empty[kNQ];
  uint64_t kv_full[NR], kv_empty[NR];
  uint64_t s_full[2], p_full[2], o_full[2], t_free[2];
  uint32_t tmem_base;
};

// Per-item bookkeeping shared by the producer and the MMA warp: the item's
// head and tile, its first block, and the ring sequence number of that block
// (blocks of one head run are loaded with consecutive sequence numbers).
struct ItemWalk {
  int prev_g = -1, prev_j = -2;
  int run_first_b = 0, run_seq0 = 0, total_seq = 0;
};

struct ItemInfo {
  int g, j, bf, seq_bf;
  bool same_run;  // continues the previous item's head run
};

template <int NEWB>
__device__ __forceinline__ ItemInfo walk_item(ItemWalk& w, int u, const RingParams& p) {
  ItemInfo it;
  it.g = u / p.nt;
  it.j = u - it.g * p.nt;
  it.bf = it.j * NEWB + p.bf_off;
  it.same_run = (it.g == w.prev_g && it.j == w.prev_j + 1);
  if (it.same_run) {
    w.total_seq += NEWB;
  } else {
    w.run_first_b = it.bf;
    w.run_seq0 = w.total_seq;
    w.total_seq += p.nbt;
  }
  it.seq_bf = w.run_seq0 + (it.bf - w.run_first_b);
  w.prev_g = it.g;
  w.prev_j = it.j;
  return it;
}

// The items of one CTA.  Main CTAs (the first chunks * num_kv_heads) take a
// contiguous run of one head's tiles, heads fastest.  When the SM count is not
// a multiple of the head count, the CTAs past them (spill CTAs) share the last
// spill_per_head tiles of every head, listed head by head, so that no main CTA
// needs a tile more than the average: a spill CTA's list is a few short head
// runs, each restarting the ring.
struct CtaItems {
  int u0, n;
  bool spill;
};

__device__ __forceinline__ CtaItems cta_items(const RingParams& p) {
  const int b = blockIdx.x;
  const int nmain = p.chunks * p.num_kv_heads;
  CtaItems c;
  if (b < nmain) {
    // heads fastest: CTAs that run at the same time cover every head of the
    // same token range, so the DRAM pages holding the rows of neighbouring
    // heads are read while they are open (a version with contiguous item
    // ranges over all SMs ran 10 % slower)
    const int cg = b % p.num_kv_heads;
    const int cr = b / p.num_kv_heads;
    int j0, j1;
    if (p.chunk_size > 0) {
      j0 = cr * p.chunk_size;
      j1 = j0 + p.chunk_size;
    } else {
      j0 = (int)(((int64_t)cr * p.nt) / p.chunks);
      j1 = (int)(((int64_t)(cr + 1) * p.nt) / p.chunks);
    }
    c.u0 = cg * p.nt + j0;
    c.n = j1 - j0;
    c.spill = false;
  } else {
    const int e = b - nmain, ne = (int)gridDim.x - nmain;
    const int64_t tot = (int64_t)p.num_kv_heads * p.spill_per_head;
    c.u0 = (int)((int64_t)e * tot / ne);
    c.n = (int)((int64_t)(e + 1) * tot / ne) - c.u0;
    c.spill = true;
  }
  return c;
}

// Global item u = head * nt + tile of the CTA's it-th item.
__device__ __forceinline__ int cta_item_u(const CtaItems& c, int it, const RingParams& p) {
  if (!c.spill) return c.u0 + it;
  const int l = c.u0 + it;
  const int g = l / p.spill_per_head;
  return g * p.nt + (p.nt - p.spill_per_head) + (l - g * p.spill_per_head);
}

template <int D, int G, int MODE>
__global__ void __launch_bounds__(384, 1)
window_ring_kernel(const __grid_constant__ CUtensorMap tm_qc,
                   const __grid_constant__ CUtensorMap tm_qt,
                   const __grid_constant__ CUtensorMap tm_kc,
                   const __grid_constant__ CUtensorMap tm_kt,
                   const __grid_constant__ CUtensorMap tm_v, const RingParams p) {
  using S = RingShape<D, G>;
  constexpr int NR = S::NR;
  extern __shared__ uint8_t smem_raw[];
  __shared__ RingCtl<NR> ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                         // kNQ x ([NC][128][64] [NT][128][16])
  uint8_t* sK = sQ + kNQ * S::QBYTES;         // [NC][NR KB][64] [NT][NR KB][16]
  uint8_t* sV = sK + S::NC * S::KC_BYTES + S::NT * S::KT_BYTES;  // [VA][NR KB][VW]

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  griddep_launch_dependents();
  const CtaItems ci = cta_items(p);
  const int n = ci.n;

  if (tid == 0) {
    for (int i = 0; i < kNQ; ++i) {
      mbar_init(&ctl.q_full[i], 1);
      mbar_init(&ctl.q_empty[i], 1);
    }
    for (int i = 0; i < NR; ++i) {
      mbar_init(&ctl.kv_full[i], 1);
      mbar_init(&ctl.kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl.s_full[i], 1);
      mbar_init(&ctl.p_full[i], 4);
      mbar_init(&ctl.o_full[i], 1);
      mbar_init(&ctl.t_free[i], 4);
    }
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(&ctl.tmem_base, 2 * kBufCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  if (G == 1 && (tid == 0 || tid == 96) && n > 0) {
    // The first item's Q and K/V boxes into L2 while the previous kernel
    // finishes (a prefetch only warms L2, which that kernel's writes keep
    // coherent, so it may run before the dependency wait); blocks before the
    // first token are skipped.  MHA tiles only: with G = 4 the first item's
    // five 32-key blocks took 27 prefetch instructions and the call got slower
    // (38.4 -> 39.7 us for the 16384-token GQA block; MHA 41.7 -> 41.2).
    ItemWalk w0;
    const ItemInfo f = walk_item<S::NEWB>(w0, cta_item_u(ci, 0, p), p);
    if (tid == 0) {
#pragma unroll
      for (int c = 0; c < S::NC; ++c) tma_prefetch_l2_3d(&tm_qc, 64 * c, f.g * G, f.j * S::TQ);
#pragma unroll
      for (int t = 0; t < S::NT; ++t)
        tma_prefetch_l2_3d(&tm_qt, 64 * S::NC + 16 * t, f.g * G, f.j * S::TQ);
    }
    for (int kb = tid == 0 ? 0 : 1; kb < p.nbt; kb += 2) {
      const int b = f.bf + kb;
      if (b < 0 || b * S::KB >= p.total_tokens) continue;
#pragma unroll
      for (int c = 0; c < S::NC; ++c) tma_prefetch_l2_3d(&tm_kc, 64 * c, f.g, b * S::KB);
#pragma unroll
      for (int t = 0; t < S::NT; ++t)
        tma_prefetch_l2_3d(&tm_kt, 64 * S::NC + 16 * t, f.g, b * S::KB);
#pragma unroll
      for (int a = 0; a < S::VA; ++a) tma_prefetch_l2_3d(&tm_v, S::VW * a, f.g, b * S::KB);
    }
  }
  griddep_wait();  // set-up above overlaps the previous kernel; memory from here

  if (tid == 0 || tid == 96) {
    // ---- TMA producers: thread 0 loads Q and the even ring blocks, thread
    // 96 the odd ones (each thread's copies complete one after another);
    // both walk every item and keep the same sequence numbers
    const int par = tid == 0 ? 0 : 1;
    const bool do_q = tid == 0;
    tma_prefetch_map(&tm_qc);
    if (S::NT) tma_prefetch_map(&tm_qt);
    tma_prefetch_map(&tm_kc);
    if (S::NT) tma_prefetch_map(&tm_kt);
    tma_prefetch_map(&tm_v);
    ItemWalk w;
    int seq = 0, last_bl = 0, nq = 0;
    bool ok = true;
    for (int it = 0; it < n && ok; ++it) {
      const ItemInfo info = walk_item<S::NEWB>(w, cta_item_u(ci, it, p), p);
      const int qs = it % kNQ;
      if (do_q) {
        if (it >= kNQ) ok = mbar_wait(&ctl.q_empty[qs], ((it / kNQ) - 1) & 1, p.err, kErrWaitFree);
        if (!ok) break;
        mbar_arrive_expect_tx(&ctl.q_full[qs], S::QBYTES);
        uint8_t* qst = sQ + qs * S::QBYTES;
#pragma unroll
        for (int c = 0; c < S::NC; ++c)
          tma_load_3d(qst + c * S::QC, &tm_qc, &ctl.q_full[qs], 64 * c, info.g * G, info.j * S::TQ);
#pragma unroll
        for (int t = 0; t < S::NT; ++t)
          tma_load_3d(qst + S::NC * S::QC + t * S::QT, &tm_qt, &ctl.q_full[qs], 64 * S::NC + 16 * t,
                      info.g * G, info.j * S::TQ);
        ++nq;
      }
      const int bl = info.bf + p.nbt - 1;
      for (int b = info.same_run ? last_bl + 1 : info.bf; b <= bl; ++b, ++seq) {
        if ((seq & 1) != par) continue;
        const int slot = seq % NR;
        if (seq >= NR) ok = mbar_wait(&ctl.kv_empty[slot], ((seq / NR) - 1) & 1, p.err, kErrWaitFree);
        if (!ok) break;
        mbar_arrive_expect_tx(&ctl.kv_full[slot], S::SLOT);
#pragma unroll
        for (int c = 0; c < S::NC; ++c)
          tma_load_3d(sK + c * S::KC_BYTES + slot * S::KB * 128, &tm_kc, &ctl.kv_full[slot],
                      64 * c, info.g, b * S::KB);
#pragma unroll
        for (int t = 0; t < S::NT; ++t)
          tma_load_3d(sK + S::NC * S::KC_BYTES + t * S::KT_BYTES + slot * S::KB * 32, &tm_kt,
                      &ctl.kv_full[slot], 64 * S::NC + 16 * t, info.g, b * S::KB);
#pragma unroll
        for (int a = 0; a < S::VA; ++a)
          tma_load_3d(sV + a * S::VA_BYTES + slot * S::KB * S::VW * 2, &tm_v, &ctl.kv_full[slot],
                      S::VW * a, info.g, b * S::KB);
      }
      last_bl = bl;
    }
    // Bounded drain: every copy issued must have landed before the CTA exits
    // (immediate when the MMA warp consumed them all).
    for (int sq = max(0, seq - NR); sq < seq; ++sq)
      if ((sq & 1) == par) mbar_wait(&ctl.kv_full[sq % NR], (sq / NR) & 1, p.err, kErrWaitDrain);
    for (int it = max(0, nq - kNQ); it < nq; ++it)
      mbar_wait(&ctl.q_full[it % kNQ], (it / kNQ) & 1, p.err, kErrWaitDrain);
  } else if (tid == 32 && n > 0) {
    // ---- MMA issuer --------------------------------------------------------
    ItemWalk w;
    bool ok = true;
    const uint32_t idesc_o = idesc_bf16(128, S::VN, true);
    auto issue_s = [&](int it, const ItemInfo& info) -> bool {
      const int b = it & 1;
      if (it >= 2 && !mbar_wait(&ctl.t_free[b], ((it >> 1) - 1) & 1, p.err, kErrWaitFree))
        return false;
      const int qs = it % kNQ;
      if (!mbar_wait(&ctl.q_full[qs], (it / kNQ) & 1, p.err, kErrWaitLoad)) return false;
      const uint8_t* qb = sQ + qs * S::QBYTES;
      for (int kb = 0; kb < p.nbt; ++kb) {
        const int sq = info.seq_bf + kb;
        if (!mbar_wait(&ctl.kv_full[sq % NR], (sq / NR) & 1, p.err, kErrWaitLoad)) return false;
      }
      tc_fence_after();
      // The tile's blocks sit in consecutive slots, wrapping at most once:
      // one MMA per slab for each contiguous run (N = run keys <= 256).
      const int k0 = info.seq_bf % NR;
      const int n1 = min(p.nbt, NR - k0);
      for (int run = 0; run < 2; ++run) {
        const int nb = run == 0 ? n1 : p.nbt - n1;
        if (nb == 0) break;
        const int slot0 = run == 0 ? k0 : 0;
        const uint32_t col = (uint32_t)(b * kBufCols + (run == 0 ? 0 : n1 * S::KB));
        const uint32_t idesc_s = idesc_bf16(128, nb * S::KB, false);
        // 16 dimensions per MMA: four within each 128-byte swizzled chunk,
        // then one per 32-byte swizzled tail slab
#pragma unroll
        for (int c = 0; c < S::NC; ++c) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const uint64_t a = smem_desc(smem_u32(qb + c * S::QC) + q4 * 32, 16, 1024, kLayoutSw128);
            const uint64_t bd = smem_desc(
                smem_u32(sK + c * S::KC_BYTES + slot0 * S::KB * 128) + q4 * 32, 16, 1024,
                kLayoutSw128);
            mma_ss(tmem + col, a, bd, idesc_s, (c | q4) ? 1u : 0u);
          }
        }
#pragma unroll
        for (int t = 0; t < S::NT; ++t) {
          const uint64_t a = smem_desc(smem_u32(qb + S::NC * S::QC + t * S::QT), 16, 256, kLayoutSw32);
          const uint64_t bd = smem_desc(
              smem_u32(sK + S::NC * S::KC_BYTES + t * S::KT_BYTES + slot0 * S::KB * 32), 16, 256,
              kLayoutSw32);
          mma_ss(tmem + col, a, bd, idesc_s, (S::NC > 0 || t > 0) ? 1u : 0u);
        }
      }
      mma_commit(&ctl.q_empty[qs]);
      mma_commit(&ctl.s_full[b]);
      return true;
    };
    ItemInfo cur = walk_item<S::NEWB>(w, cta_item_u(ci, 0, p), p);
    ok = issue_s(0, cur);
    for (int it = 0; it < n && ok; ++it) {
      const bool have_next = it + 1 < n;
      ItemInfo nxt = cur;
      if (have_next) nxt = walk_item<S::NEWB>(w, cta_item_u(ci, it + 1, p), p);
      const bool ahead = have_next && nxt.same_run;
      if (ahead && !(ok = issue_s(it + 1, nxt))) break;
      const int b = it & 1;
      ok = mbar_wait(&ctl.p_full[b], (it >> 1) & 1, p.err, kErrWaitMma);
      if (!ok) break;
      tc_fence_after();
      // P V block by block, oldest first; a block the next item does not use
      // is released as soon as its own MMAs complete, so its slot's refill
      // starts while the rest of P V runs.  O is signalled last, so that
      // every earlier arrival has landed once O is seen complete.
      const int nrel = ahead ? S::NEWB : p.nbt;
      for (int kb = 0; kb < p.nbt; ++kb) {
        const int sq = cur.seq_bf + kb;
        // V rows of this block: VW * 2 bytes each, atoms VA_BYTES apart
        const uint8_t* vbase = sV + (sq % NR) * S::KB * S::VW * 2;
#pragma unroll
        for (int ks = 0; ks < S::KB / 16; ++ks) {
          const uint64_t bd = smem_desc(smem_u32(vbase + ks * 16 * S::VW * 2), S::VA_BYTES,
                                        8 * S::VW * 2, S::V128 ? kLayoutSw128 : kLayoutSw64);
          mma_ts(tmem + (uint32_t)(b * kBufCols + kColO),
                 tmem + (uint32_t)(b * kBufCols + (kb * S::KB + ks * 16) / 2), bd, idesc_o,
                 (kb | ks) ? 1u : 0u);
        }
        if (kb < nrel) mma_commit(&ctl.kv_empty[sq % NR]);
      }
      mma_commit(&ctl.o_full[b]);
      if (have_next && !ahead && !(ok = issue_s(it + 1, nxt))) break;
      cur = nxt;
    }
  } else if (warp >= 4) {
    // ---- softmax warpgroups --------------------------------------------------
    const int wg = (warp - 4) >> 2;
    const int wq = warp & 3;  // TMEM lane quadrant
    const int row = wq * 32 + lane;
    const uint32_t lane_base = tmem + (uint32_t)(wg * kBufCols) + ((uint32_t)(wq * 32) << 16);
    const int nk = p.nbt * S::KB;
    const int nchunks = (nk + 31) >> 5;
    for (int it = wg; it < n; it += 2) {
      const int k = it >> 1;
      const int u = cta_item_u(ci, it, p);
      const int g = u / p.nt;
      const int j = u - g * p.nt;
      const int tok0 = j * S::TQ;
      const int kstart = (j * S::NEWB + p.bf_off) * S::KB;
      const win::RowMeta r = win::row_meta<G, MODE>(p.cu_seqlens, p.num_seqs, p.total_tokens,
                                                     row, g, tok0, kstart, p.wl, p.wr, p.sinks);
      const int off = tok0 - p.wl - kstart;
      const int wc_lo = off + (wq * 32) / G;
      const int wc_hi = min(off + (wq * 32 + 31) / G + p.wl + p.wr, nk - 1);
      bool ok = mbar_wait(&ctl.s_full[wg], k & 1, p.err, kErrWaitMma);
      __syncwarp();
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      float m, l;
      if constexpr (MODE == SA_SINK_KEY0_BIAS) win::key0_bias_in_tmem(lane_base, r, p.scale_log2);
      win::softmax_rows<false>(lane_base, lane_base, nchunks, wc_lo >> 5, wc_hi >> 5, r,
                               p.scale_log2, m, l);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.p_full[wg]);
      ok = mbar_wait(&ctl.o_full[wg], k & 1, p.err, kErrWaitMma);
      __syncwarp();
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      float inv, lse_v;
      win::finalize_row<MODE>(r, m, l, inv, lse_v);
      if constexpr (D <= 80) {
        // Free the buffer as soon as O is in registers; normalise and store after.
        float oa[D / 16][16];
#pragma unroll
        for (int jj = 0; jj < D / 16; ++jj) tmem_ld16(lane_base + kColO + 16 * jj, oa[jj]);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.t_free[wg]);
        if (r.valid) {
          __nv_bfloat16* orow = p.out + ((int64_t)r.t * p.num_q_heads + r.h) * D;
#pragma unroll
          for (int jj = 0; jj < D / 16; ++jj) {
            const float* o = oa[jj];
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
        win::store_o_groups<D>(lane_base + kColO, 0, D / 16, r, inv, p.out, p.num_q_heads);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.t_free[wg]);
      }
      if (r.valid) p.lse[(int64_t)r.h * p.total_tokens + r.t] = lse_v;
    }
  }

  // ---- teardown ----------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kBufCols);
  }
}

template <int D, int G, int MODE>
sa_status launch_ring_typed(const WindowArgs& a, int nbt, int bf_off) {
  using S = RingShape<D, G>;
  // Q and K: 64-dim chunks (128-byte swizzle) and 16-dim tail slabs (32-byte
  // swizzle); V: atoms of VW dims (the last zero-filled past D)
  CUtensorMap tqc, tqt, tkc, tkt, tv;
  const uint64_t dq[3] = {(uint64_t)D, (uint64_t)a.num_q_heads, (uint64_t)a.total_tokens};
  const uint64_t sq[2] = {(uint64_t)D * 2, (uint64_t)a.num_q_heads * D * 2};
  const uint32_t bqc[3] = {64, (uint32_t)G, (uint32_t)S::TQ};
  const uint32_t bqt[3] = {16, (uint32_t)G, (uint32_t)S::TQ};
  const uint64_t dk[3] = {(uint64_t)D, (uint64_t)a.num_kv_heads, (uint64_t)a.total_tokens};
  const uint64_t sk[2] = {(uint64_t)D * 2, (uint64_t)a.num_kv_heads * D * 2};
  const uint32_t bkc[3] = {64, 1, (uint32_t)S::KB};
  const uint32_t bkt[3] = {16, 1, (uint32_t)S::KB};
  const uint32_t bv[3] = {(uint32_t)S::VW, 1, (uint32_t)S::KB};
  if (!encode_tiled(&tqc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.q, dq, sq, bqc,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE) ||
      !encode_tiled(&tkc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.k, dk, sk, bkc,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE) ||
      !encode_tiled(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.v, dk, sk, bv,
                    S::V128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE))
    return SA_ERR_INVALID_ARG;
  if (S::NT > 0) {
    if (!encode_tiled(&tqt, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.q, dq, sq, bqt,
                      CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_NONE) ||
        !encode_tiled(&tkt, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.k, dk, sk, bkt,
                      CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_NONE))
      return SA_ERR_INVALID_ARG;
  } else {
    tqt = tqc;  // never read: no tail slabs
    tkt = tkc;
  }
  RingParams p;
  p.cu_seqlens = a.cu_seqlens;
  p.num_seqs = a.num_seqs;
  p.total_tokens = (int32_t)a.total_tokens;
  p.num_q_heads = a.num_q_heads;
  p.wl = a.window_left;
  p.wr = a.window_right;
  p.nt = (int32_t)((a.total_tokens + S::TQ - 1) / S::TQ);
  p.items = p.nt * a.num_kv_heads;
  p.nbt = nbt;
  p.bf_off = bf_off;
  p.sinks = a.sinks;
  p.scale_log2 = a.softmax_scale * win::kLog2e;
  p.out = reinterpret_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.err = device_error_word();
  auto kern = window_ring_kernel<D, G, MODE>;
  if (!set_dynamic_smem_once((const void*)kern, (int)S::SMEM))
    return fail(SA_ERR_CUDA, "sa_varlen_window_fwd: %s", cudaGetErrorString(cudaGetLastError()));
  cudaError_t e;
  p.num_kv_heads = a.num_kv_heads;
  const int sms = num_sms();
  p.chunks = sms / a.num_kv_heads;
  if (p.chunks < 1) p.chunks = 1;
  if (p.chunks > p.nt) p.chunks = p.nt;
  p.chunk_size = 0;
  p.spill_per_head = 0;
  int grid = p.chunks * a.num_kv_heads;
  // Tiles per CTA at best: ceil(items / SMs).  If the main CTAs at that size
  // leave tiles over and SMs are free, those SMs take the leftover tiles
  // (at most as many each, since chunks * num_kv_heads + spare = SMs).
  const int64_t cmax = (p.items + (int64_t)sms - 1) / sms;
  const int spare = sms - grid;
  if (spare > 0 && (int64_t)p.chunks * cmax < p.nt) {
    p.chunk_size = (int32_t)cmax;
    p.spill_per_head = p.nt - p.chunks * (int32_t)cmax;
    grid += (int)std::min<int64_t>(spare, (int64_t)p.spill_per_head * a.num_kv_heads);
  }
  e = launch_dependent(kern, dim3(grid), dim3(384), S::SMEM, a.stream, tqc, tqt, tkc, tkt, tv, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(SA_ERR_CUDA, "sa_varlen_window_fwd launch: %s", cudaGetErrorString(e));
  return SA_OK;
}

template <int D, int G>
sa_status ring_by_mode(const WindowArgs& a, int nbt, int bf_off) {
  switch (a.sink_mode) {
    case SA_SINK_NONE: return launch_ring_typed<D, G, SA_SINK_NONE>(a, nbt, bf_off);
    case SA_SINK_KEY0_BIAS: return launch_ring_typed<D, G, SA_SINK_KEY0_BIAS>(a, nbt, bf_off);
    default: return launch_ring_typed<D, G, SA_SINK_NULL_LOGIT>(a, nbt, bf_off);
  }
}

// Blocks per tile and first-block offset for this window, and whether the
// ring of this (D, G) holds one tile plus the next tile's new blocks.
template <int D, int G>
bool ring_plan(const WindowArgs& a, int* nbt, int* bf_off) {
  using S = RingShape<D, G>;
  const int first = -((a.window_left + S::KB - 1) / S::KB);        // floor(-wl / KB)
  const int last = (S::TQ - 1 + a.window_right) / S::KB;           // floor((TQ-1+wr) / KB)
  *nbt = last - first + 1;
  *bf_off = first;
  return S::NR >= 1 && *nbt * S::KB <= kBufCols && *nbt + S::NEWB <= S::NR &&
         S::SMEM <= 227 * 1024;
}

template <int D, int G>
bool ring_try(const WindowArgs& a, sa_status* st) {
  int nbt, bf_off;
  if (!ring_plan<D, G>(a, &nbt, &bf_off)) return false;
  *st = ring_by_mode<D, G>(a, nbt, bf_off);
  return true;
}

template <int D>
bool ring_by_group(const WindowArgs& a, int G, sa_status* st) {
  switch (G) {
    case 1: return ring_try<D, 1>(a, st);
    case 2: return ring_try<D, 2>(a, st);
    case 4: return ring_try<D, 4>(a, st);
    case 8: return ring_try<D, 8>(a, st);
    default: return false;
  }
}

}  // namespace

bool launch_window_ring(const WindowArgs& a, sa_status* st) {
  const int G = a.num_q_heads / a.num_kv_heads;
  switch (a.head_dim) {
    case 64: return ring_by_group<64>(a, G, st);
    case 80: return ring_by_group<80>(a, G, st);
    case 128: return ring_by_group<128>(a, G, st);
    default: return false;
  }
}

}  // namespace sa

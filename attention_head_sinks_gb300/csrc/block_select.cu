// block_select.cu -- on-device top-k key-block selection from indexer scores,
// one selection per index head (the step before the block-sparse attention).
//
// Operation: NeMo AutoModel "nemo_automodel.components.models.minimax_m3_vl.
// cp_sparse_attn", MiniMaxM3CPSparseAttention forward step 3 (the top-k key
// blocks of each query from index q / k over the causal sequence) and
// _select_local_blocks (one boolean selection per index head,
// [batch, index_heads, sequence, key_blocks]); documents are not consulted
// here -- _local_sparse_forward composes their mask inside the attention.
// The page leaves the score open; the readings taken: token score
// q_idx[i, g] . k_idx[j] (fp32 accumulation of the bf16 inputs), a block's
// score is the max over its keys, the query's own (diagonal) block is always
// selected and the other topk - 1 are the highest-scoring earlier blocks,
// ties to the lower block id; a token with at most topk causal blocks takes
// them all.  Output: block table [Hi, B*S, topk] int32, ascending, -1 padded
// (offsets in int64, after the lesson of _block_sel_flat_offset).
//
// Tile: one CTA per (128 query tokens of one batch row, pair of index heads).
// The blocks a token ranks (those before its diagonal block) lie wholly
// before it, so no per-key causal mask is needed.  The CTA walks the batch
// row's keys in 256-key tiles up to its last needed block:
//   S_h = Qidx_h Kidx^T (M = 128 tokens, N = 256 keys, K = index dim) for
//   both heads of the pair, into TMEM columns [256 h, 256 h + 256);
//   warps 0..3 (thread = token = TMEM lane) reduce each needed 64-key block
//   to its max and insert it into a register list of the best topk - 1
//   blocks, kept sorted by score (blocks arrive in ascending id order and a
//   candidate must be strictly higher to pass an entry, so ties keep the
//   lower id).
// The index keys are shared by all index heads; taking two heads per CTA
// halves the key traffic from L2, which otherwise limits the MMAs.
// Warp roles: warp 4 (lane 0) TMA producer, warp 5 (lane 0) MMA issuer and
// TMEM owner.
#include <climits>
#include <math.h>

#include "sa_internal.h"
#include "sa_ptx.cuh"

namespace sa {
namespace {

constexpr int kBlk = 64;
constexpr int kDi = 128;                      // index head dim
constexpr int kSlabs = kDi / 64;              // 128-byte swizzled K slabs
constexpr int kTileKeys = 256;
constexpr int kTileRows = 128;
constexpr int kHeadsPerCta = 2;
constexpr int kStages = 2;
constexpr int kList = 15;                     // topk - 1 <= 15
constexpr int kQSlabBytes = kTileRows * 128;  // 128 tokens x 64 dims
constexpr int kKSlabBytes = kTileKeys * 128;  // 256 keys x 64 dims
constexpr int kStageBytes = kSlabs * kKSlabBytes;
constexpr int kThreads = 192;
constexpr int kTmemCols = kHeadsPerCta * kTileKeys;

struct SelectParams {
  int32_t* table;  // [Hi, T, topk]
  int64_t total_tokens;
  int32_t seq_len;
  int32_t batch;
  int32_t num_index_heads;
  int32_t topk;
  int32_t ntiles_q;  // seq_len / 128
  int32_t npairs;    // ceil(Hi / 2)
  uint32_t* err;
};

struct SelectCtl {
  uint64_t q_full;
  uint64_t k_full[kStages];
  uint64_t k_empty[kStages];
  uint64_t s_full[kHeadsPerCta];
  uint64_t s_free[kHeadsPerCta];
  uint32_t tmem_base;
};

// Insert (v, c) into the list sorted by descending score: the candidate
// passes only entries it strictly beats.
__device__ __forceinline__ void list_insert(float (&s)[kList], int (&id)[kList], float v,
                                            int c) {
  if (!(v > s[kList - 1])) return;
#pragma unroll
  for (int i = 0; i < kList; ++i) {
    const bool gt = v > s[i];
    const float ts = s[i];
    const int ti = id[i];
    s[i] = gt ? v : ts;
    id[i] = gt ? c : ti;
    v = gt ? ts : v;
    c = gt ? ti : c;
  }
}

// Max of 64 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ float block_max(uint32_t taddr) {
  float a[32], b[32];
  tmem_ld32(taddr, a);
  tmem_ld32(taddr + 32, b);
  tmem_wait_ld();
  float m0 = a[0], m1 = b[0];
#pragma unroll
  for (int e = 1; e < 31; e += 2) {
    m0 = fmaxf(m0, fmaxf(a[e], a[e + 1]));
    m1 = fmaxf(m1, fmaxf(b[e], b[e + 1]));
  }
  return fmaxf(fmaxf(m0, a[31]), fmaxf(m1, b[31]));
}

// The token's table row: list ids (the best topk - 1 earlier blocks; fewer
// when it has fewer) plus the diagonal block, ascending, -1 padded.
__device__ __forceinline__ void write_row(int32_t* dst, const int (&id)[kList], int diag,
                                          int topk) {
  int v[kList + 1];
#pragma unroll
  for (int i = 0; i < kList; ++i) v[i] = (i < topk - 1 && id[i] >= 0) ? id[i] : INT_MAX;
  v[kList] = diag;
  // odd-even transposition sort, ascending (INT_MAX = empty goes last)
#pragma unroll
  for (int r = 0; r < kList + 1; ++r) {
#pragma unroll
    for (int i = r & 1; i + 1 < kList + 1; i += 2) {
      const int lo = min(v[i], v[i + 1]), hi = max(v[i], v[i + 1]);
      v[i] = lo;
      v[i + 1] = hi;
    }
  }
#pragma unroll
  for (int i = 0; i < kList + 1; ++i)
    if (i < topk) dst[i] = v[i] == INT_MAX ? -1 : v[i];
}

__global__ void __launch_bounds__(kThreads, 1)
block_select_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k, const SelectParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ SelectCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                                        // [heads][slabs][128][64]
  uint8_t* sK = smem + kHeadsPerCta * kSlabs * kQSlabBytes;  // [stages][slabs][256][64]

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  // heavy tiles (late in the row: more keys) first
  const int per_qt = p.batch * p.npairs;
  const int qt = p.ntiles_q - 1 - (int)(blockIdx.x / per_qt);
  const int rem = (int)(blockIdx.x % per_qt);
  const int b = rem / p.npairs;
  const int pair = rem % p.npairs;
  const int nh = min(kHeadsPerCta, p.num_index_heads - kHeadsPerCta * pair);
  const int row0 = b * p.seq_len;                   // first token of the batch row
  const int tok0 = qt * kTileRows;                  // first query position of the tile
  // needed blocks: c < diag of the tile's last token = 2 qt + 1
  const int ntiles_k = (tok0 + kTileRows / 2 + kTileKeys - 1) / kTileKeys;

  if (tid == 0) {
    mbar_init(&ctl.q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl.k_full[s], 1);
      mbar_init(&ctl.k_empty[s], 1);
    }
    for (int h = 0; h < kHeadsPerCta; ++h) {
      mbar_init(&ctl.s_full[h], 1);
      mbar_init(&ctl.s_free[h], 128);
    }
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&ctl.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;

  if (warp == 4) {
    if ((tid & 31) == 0) {
      // ---- TMA producer ----------------------------------------------------
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      mbar_arrive_expect_tx(&ctl.q_full, (uint32_t)(nh * kSlabs * kQSlabBytes));
      for (int h = 0; h < nh; ++h)
        for (int s = 0; s < kSlabs; ++s)
          tma_load_3d(sQ + (h * kSlabs + s) * kQSlabBytes, &tm_q, &ctl.q_full, 64 * s,
                      kHeadsPerCta * pair + h, row0 + tok0);
      int issued = 0;
      for (int t = 0; t < ntiles_k; ++t) {
        const int st = t % kStages;
        if (t >= kStages &&
            !mbar_wait(&ctl.k_empty[st], ((t / kStages) - 1) & 1, p.err, kErrWaitFree))
          break;
        mbar_arrive_expect_tx(&ctl.k_full[st], (uint32_t)kStageBytes);
        for (int s = 0; s < kSlabs; ++s)
          tma_load_2d(sK + st * kStageBytes + s * kKSlabBytes, &tm_k, &ctl.k_full[st], 64 * s,
                      row0 + t * kTileKeys);
        ++issued;
      }
      // bounded drain of copies the MMAs may not have consumed
      for (int t = max(0, issued - kStages); t < issued; ++t)
        mbar_wait(&ctl.k_full[t % kStages], (t / kStages) & 1, p.err, kErrWaitDrain);
      mbar_wait(&ctl.q_full, 0, p.err, kErrWaitDrain);
    }
  } else if (warp == 5) {
    if ((tid & 31) == 0) {
      // ---- MMA issuer -------------------------------------------------------
      const uint32_t idesc = idesc_bf16(128, kTileKeys, false);
      bool ok = mbar_wait(&ctl.q_full, 0, p.err, kErrWaitLoad);
      for (int t = 0; t < ntiles_k && ok; ++t) {
        const int st = t % kStages;
        ok = mbar_wait(&ctl.k_full[st], (t / kStages) & 1, p.err, kErrWaitLoad);
        if (!ok) break;
        for (int h = 0; h < nh && ok; ++h) {
          if (t > 0) ok = mbar_wait(&ctl.s_free[h], (t - 1) & 1, p.err, kErrWaitFree);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kDi / 16; ++kk) {
            const uint32_t qa = smem_u32(sQ + (h * kSlabs + kk / 4) * kQSlabBytes) + (kk % 4) * 32;
            const uint32_t ka =
                smem_u32(sK + st * kStageBytes + (kk / 4) * kKSlabBytes) + (kk % 4) * 32;
            mma_ss(tmem + (uint32_t)(h * kTileKeys), smem_desc(qa, 16, 1024, kLayoutSw128),
                   smem_desc(ka, 16, 1024, kLayoutSw128), idesc, kk > 0 ? 1u : 0u);
          }
          mma_commit(&ctl.s_full[h]);
        }
        mma_commit(&ctl.k_empty[st]);
      }
    }
  } else {
    // ---- epilogue: thread = query token (TMEM lane) ------------------------
    const int r = tid;                       // 0..127
    const int diag = 2 * qt + (r >> 6);      // the token's own block
    const uint32_t lane = tmem + ((uint32_t)(warp * 32) << 16);
    float sc[kHeadsPerCta][kList];
    int id[kHeadsPerCta][kList];
#pragma unroll
    for (int h = 0; h < kHeadsPerCta; ++h)
#pragma unroll
      for (int i = 0; i < kList; ++i) {
        sc[h][i] = -INFINITY;
        id[h][i] = -1;
      }
    bool ok = true;
    for (int t = 0; t < ntiles_k; ++t) {
#pragma unroll
      for (int h = 0; h < kHeadsPerCta; ++h) {
        if (h >= nh) break;
        ok = mbar_wait(&ctl.s_full[h], t & 1, p.err, kErrWaitMma) && ok;
        __syncwarp();
        tc_fence_after();
        float bm[4];
        const int nblk = min(4, diag - 4 * t);  // this warp's needed blocks (warp-uniform)
#pragma unroll
        for (int bb = 0; bb < 4; ++bb)
          bm[bb] = bb < nblk ? block_max(lane + (uint32_t)(h * kTileKeys + bb * kBlk)) : 0.f;
        tc_fence_before();
        mbar_arrive(&ctl.s_free[h]);
#pragma unroll
        for (int bb = 0; bb < 4; ++bb)
          if (bb < nblk) list_insert(sc[h], id[h], bm[bb], 4 * t + bb);
      }
    }
    const int64_t tok = (int64_t)row0 + tok0 + r;
#pragma unroll
    for (int h = 0; h < kHeadsPerCta; ++h) {
      if (h >= nh) break;
      const int g = kHeadsPerCta * pair + h;
      write_row(p.table + ((int64_t)g * p.total_tokens + tok) * p.topk, id[h], diag, p.topk);
    }
  }

  // ---- teardown ------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

sa_status launch_block_select(const SelectArgs& a) {
  const char* fn = "sa_block_select";
  if (a.index_dim != kDi)
    return fail(SA_ERR_UNSUPPORTED, "%s: index_dim %d (supported: 128)", fn, a.index_dim);
  if (a.block_size != kBlk)
    return fail(SA_ERR_UNSUPPORTED, "%s: block_size %d (supported: 64)", fn, a.block_size);
  if (a.seq_len % kTileRows != 0)
    return fail(SA_ERR_UNSUPPORTED, "%s: seq_len %d is not a multiple of 128", fn, a.seq_len);
  if (a.topk_blocks > kList + 1)
    return fail(SA_ERR_UNSUPPORTED, "%s: topk_blocks %d above %d", fn, a.topk_blocks, kList + 1);
  const int64_t T = (int64_t)a.batch * a.seq_len;
  CUtensorMap tq, tk;
  const uint64_t dq[3] = {(uint64_t)kDi, (uint64_t)a.num_index_heads, (uint64_t)T};
  const uint64_t sq[2] = {(uint64_t)kDi * 2, (uint64_t)a.num_index_heads * kDi * 2};
  const uint32_t bq[3] = {64, 1, (uint32_t)kTileRows};
  const uint64_t dk[2] = {(uint64_t)kDi, (uint64_t)T};
  const uint64_t sk[1] = {(uint64_t)kDi * 2};
  const uint32_t bk[2] = {64, (uint32_t)kTileKeys};
  if (!encode_tiled(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.index_q, dq, sq, bq,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.index_k, dk, sk, bk,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return SA_ERR_INVALID_ARG;
  SelectParams p;
  p.table = a.block_table;
  p.total_tokens = T;
  p.seq_len = a.seq_len;
  p.batch = a.batch;
  p.num_index_heads = a.num_index_heads;
  p.topk = a.topk_blocks;
  p.ntiles_q = a.seq_len / kTileRows;
  p.npairs = (a.num_index_heads + kHeadsPerCta - 1) / kHeadsPerCta;
  p.err = device_error_word();
  const size_t smem = 1024 + (size_t)kHeadsPerCta * kSlabs * kQSlabBytes +
                      (size_t)kStages * kStageBytes;
  if (!set_dynamic_smem_once((const void*)block_select_kernel, (int)smem))
    return fail(SA_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(cudaGetLastError()));
  cudaError_t e;
  const int64_t ctas = (int64_t)p.ntiles_q * a.batch * p.npairs;
  if (ctas >= ((int64_t)1 << 31))
    return fail(SA_ERR_UNSUPPORTED, "%s: %lld tiles", fn, (long long)ctas);
  block_select_kernel<<<(unsigned)ctas, kThreads, smem, a.stream>>>(tq, tk, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(SA_ERR_CUDA, "%s launch: %s", fn, cudaGetErrorString(e));
  return SA_OK;
}

}  // namespace sa

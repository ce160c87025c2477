// merge_states.cu -- LSE-weighted merge of two sink-free partial attention
// results over disjoint key sets of the same queries, with the NULL_LOGIT
// sink folded once.
//
// Operation: the LSE convention of vLLM pull 49815 (LSE paragraph: LSE of
// the masked scaled logits, [nheads, total_q]) makes partial results over
// disjoint key sets mergeable: with M = max(lse_a, lse_b),
//   w_x = e^(lse_x - M),  Z = w_a + w_b,  LSE = M + ln Z,
//   out = (w_a out_a + w_b out_b) / den,  den = Z (+ e^(s_h - M) for
//   NULL_LOGIT, folded after the key loop as afierka-intel/vllm pull 76,
//   Implementation does; the LSE stays over real keys).
// Both partials empty (LSE = -inf): out = 0, LSE = -inf.
//
// HBM-bound: each thread takes one 16-byte group (8 bf16) of one output row
// per grid-stride step, with streaming loads of both partial rows and a
// streaming store; the two LSEs of a row are read through the read-only
// cache by the row's D / 8 threads.  Work unit: one (token, head) row =
// 3 * 2 D bytes of rows + 12 bytes of LSE.
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>

#include "sa_internal.h"
#include "sa_ptx.cuh"

namespace sa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kThreads = 256;

struct MergeParams {
  const uint4* out_a;
  const float* lse_a;
  const uint4* out_b;
  const float* lse_b;
  uint4* out;
  float* lse;
  const float* sinks;
  int64_t num_tokens;
  int32_t num_heads;
  int32_t groups_per_row;  // head_dim / 8
};

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

template <int MODE>
__global__ void __launch_bounds__(kThreads)
merge_states_kernel(const MergeParams p) {
  griddep_wait();  // the partials come from the previous kernels of the stream
  const int64_t rows = p.num_tokens * p.num_heads;
  const int64_t ngroups = rows * p.groups_per_row;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t gi = (int64_t)blockIdx.x * kThreads + threadIdx.x; gi < ngroups; gi += stride) {
    const int64_t row = gi / p.groups_per_row;
    const int c8 = (int)(gi - row * p.groups_per_row);
    const int64_t t = row / p.num_heads;
    const int h = (int)(row - t * p.num_heads);
    const int64_t li = (int64_t)h * p.num_tokens + t;
    const uint4 a = __ldcs(p.out_a + gi);
    const uint4 b = __ldcs(p.out_b + gi);
    const float la = __ldg(p.lse_a + li), lb = __ldg(p.lse_b + li);
    // log2 domain
    const float m = fmaxf(la, lb) * kLog2e;
    uint4 o = make_uint4(0, 0, 0, 0);
    float lse_v = -INFINITY;
    if (m != -INFINITY) {
      const float wa = ex2_approx(fmaf(la, kLog2e, -m));
      const float wb = ex2_approx(fmaf(lb, kLog2e, -m));
      const float z = wa + wb;
      float den = z;
      if (MODE == SA_SINK_NULL_LOGIT) den = z + ex2_approx(fmaf(__ldg(p.sinks + h), kLog2e, -m));
      const float inv = 1.f / den;
      const float ca = wa * inv, cb = wb * inv;
      o.x = pack_bf16x2(fmaf(ca, bf_lo(a.x), cb * bf_lo(b.x)), fmaf(ca, bf_hi(a.x), cb * bf_hi(b.x)));
      o.y = pack_bf16x2(fmaf(ca, bf_lo(a.y), cb * bf_lo(b.y)), fmaf(ca, bf_hi(a.y), cb * bf_hi(b.y)));
      o.z = pack_bf16x2(fmaf(ca, bf_lo(a.z), cb * bf_lo(b.z)), fmaf(ca, bf_hi(a.z), cb * bf_hi(b.z)));
      o.w = pack_bf16x2(fmaf(ca, bf_lo(a.w), cb * bf_lo(b.w)), fmaf(ca, bf_hi(a.w), cb * bf_hi(b.w)));
      lse_v = (m + log2f(z)) * kLn2;
    }
    __stcs(p.out + gi, o);
    if (c8 == 0) p.lse[li] = lse_v;
  }
}

}  // namespace

sa_status launch_merge_states(const MergeArgs& a) {
  MergeParams p;
  p.out_a = reinterpret_cast<const uint4*>(a.out_a);
  p.lse_a = a.lse_a;
  p.out_b = reinterpret_cast<const uint4*>(a.out_b);
  p.lse_b = a.lse_b;
  p.out = reinterpret_cast<uint4*>(a.out);
  p.lse = a.lse;
  p.sinks = a.sinks;
  p.num_tokens = a.num_tokens;
  p.num_heads = a.num_heads;
  p.groups_per_row = a.head_dim / 8;
  const int64_t ngroups = a.num_tokens * a.num_heads * p.groups_per_row;
  // a few resident CTAs per SM, each thread looping over groups
  const int64_t want = (ngroups + kThreads - 1) / kThreads;
  const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, 8LL * num_sms()));
  cudaError_t e;
  if (a.sink_mode == SA_SINK_NULL_LOGIT)
    e = launch_dependent(merge_states_kernel<SA_SINK_NULL_LOGIT>, dim3(grid), dim3(kThreads), 0,
                         a.stream, p);
  else
    e = launch_dependent(merge_states_kernel<SA_SINK_NONE>, dim3(grid), dim3(kThreads), 0,
                         a.stream, p);
  if (e != cudaSuccess)
    return fail(SA_ERR_CUDA, "sa_merge_attn_states launch: %s", cudaGetErrorString(e));
  return SA_OK;
}

}  // namespace sa

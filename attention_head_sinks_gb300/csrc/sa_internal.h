// sa_internal.h -- declarations shared by the C ABI (sa_api.cu) and the
// kernel translation units.  Host-side only types; no framework types.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sa.h"

namespace sa {

// Records a formatted message for sa_last_error() and returns `st`.
sa_status fail(sa_status st, const char* fmt, ...);

// Encodes a tiled TMA descriptor through the driver entry point (no libcuda
// link dependency).  Returns false with a message on failure.
// `promotion` is the L2 fetch granularity for the map's misses: rows that are
// narrower than it and strided apart (one head of a token) want NONE, or the
// L2 pulls bytes of neighbouring heads that may be evicted before use.
bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank,
                  const void* base, const uint64_t* dims,
                  const uint64_t* strides_bytes, const uint32_t* box,
                  CUtensorMapSwizzle swizzle,
                  CUtensorMapL2promotion promotion = CU_TENSOR_MAP_L2_PROMOTION_L2_256B);

// Raise a kernel's dynamic shared memory limit to `bytes` on the current
// device, calling the runtime only the first time per (kernel, device, size).
// False (with the runtime's error pending) when the runtime refuses.
bool set_dynamic_smem_once(const void* func, int bytes);

// Address of this device's error word (a __device__ variable).
uint32_t* device_error_word();

// Launch with programmatic stream serialisation: the kernel may begin while
// the previous kernel of the stream finishes, and must call griddep_wait()
// before its first global memory access that the previous kernel could
// affect (every kernel here waits before any global access at all).
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

struct WindowArgs {
  const void* q;
  const void* k;
  const void* v;
  const int32_t* cu_seqlens;
  int32_t num_seqs;
  int64_t total_tokens;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t window_left;
  int32_t window_right;
  const float* sinks;
  int32_t sink_mode;
  float softmax_scale;
  void* out;
  float* lse;
  cudaStream_t stream;
};

sa_status launch_window_fwd(const WindowArgs& a);

// Persistent ring kernel for the window path.  Returns false (launching
// nothing) when the shape does not fit it; otherwise launches and stores the
// launch status in *st.
bool launch_window_ring(const WindowArgs& a, sa_status* st);

// Number of SMs of the current device (cached per device).
int num_sms();

struct IndexArgs {
  const void* q;
  const void* kv;          // bf16 rows, or e4m3 rows when fp8
  const float* kv_scale;   // fp8: fp32 scale per row (else null)
  bool fp8;
  const char* fn;          // entry-point name for error messages
  int64_t num_kv;
  int32_t dqk;
  int32_t dv;
  const int32_t* indices;
  int32_t topk;
  int32_t num_queries;
  int32_t num_q_heads;
  const float* sinks;
  int32_t sink_mode;
  float softmax_scale;
  void* out;
  float* lse;
  void* workspace;
  size_t workspace_bytes;
  cudaStream_t stream;
};

// Id of the current CUDA context (unique for the life of the process; a
// context destroyed and re-created gets a new one), or 0 if none is current.
uint64_t current_context_id();

// A fixed device array used in place of a caller workspace: its size, and a
// function that returns its device address on the current device (or a
// status with a message naming `fn`).
struct FixedScratch {
  size_t bytes;
  sa_status (*address)(const char* fn, void** ptr);
};

// Checks and dispatch shared by the sparse-index entry points; with `fixed`
// set, its array serves as the workspace once every argument check passed.
sa_status sparse_index_entry(const char* fn, const void* q, const void* kv_latent,
                             const float* kv_scale, bool fp8, int64_t num_kv, int32_t dqk,
                             int32_t dv, const int32_t* indices, int32_t topk,
                             int32_t num_queries, int32_t num_q_heads, const float* sinks,
                             int32_t sink_mode, float softmax_scale, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, void* stream,
                             const FixedScratch* fixed);

size_t sparse_index_workspace_bytes(int32_t num_queries, int32_t num_q_heads, int32_t topk);
int sparse_index_max_topk();
sa_status launch_sparse_index_fwd(const IndexArgs& a);

struct BlockArgs {
  const void* q;
  const void* k;
  const void* v;
  int32_t batch;
  int32_t seq_len;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  const int32_t* block_table;  // [num_index_heads, T, topk]
  int32_t num_index_heads;     // divides num_kv_heads
  int32_t topk_blocks;
  int32_t block_size;
  const int32_t* cu_docs;
  int32_t num_docs;
  const float* sinks;
  int32_t sink_mode;
  float softmax_scale;
  void* out;
  float* lse;
  cudaStream_t stream;
};

sa_status launch_block_sparse_fwd(const BlockArgs& a);

struct SelectArgs {
  const void* index_q;  // bf16 [T, Hi, Di]
  const void* index_k;  // bf16 [T, Di]
  int32_t batch;
  int32_t seq_len;
  int32_t num_index_heads;
  int32_t index_dim;
  int32_t block_size;
  int32_t topk_blocks;
  int32_t* block_table;  // [Hi, T, topk] (written)
  cudaStream_t stream;
};

sa_status launch_block_select(const SelectArgs& a);

struct MergeArgs {
  const void* out_a;
  const float* lse_a;
  const void* out_b;
  const float* lse_b;
  int64_t num_tokens;
  int32_t num_heads;
  int32_t head_dim;
  const float* sinks;
  int32_t sink_mode;
  void* out;
  float* lse;
  cudaStream_t stream;
};

sa_status launch_merge_states(const MergeArgs& a);

}  // namespace sa

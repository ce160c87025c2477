// sa_api.cu -- the C ABI declared in include/sa.h: host-side argument checks,
// TMA descriptor encoding, the per-device error word, and dispatch to the
// kernel launchers.  Everything here only enqueues work on the caller's stream.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "sa_internal.h"
#include "sa_ptx.cuh"

namespace sa {

// Per-device word the kernels OR error codes into when a bounded wait expires.
__device__ uint32_t g_device_error;

namespace {
thread_local char t_last_error[512] = "";

bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t,
                                   void*, const cuuint64_t*, const cuuint64_t*,
                                   const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

constexpr int kMaxDevices = 64;
// Device address of the error word per device, with the id of the context it
// was looked up in.
struct ErrSlot {
  uint64_t ctx;
  uint32_t* ptr;
};
std::mutex g_err_mu;
ErrSlot g_err_slot[kMaxDevices];
}  // namespace

uint64_t current_context_id() {
  static std::once_flag once;
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&c) != CUDA_SUCCESS || !c ||
      get_id(c, &id) != CUDA_SUCCESS)
    return 0;
  return (uint64_t)id;
}

sa_status fail(sa_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_error, sizeof t_last_error, fmt, ap);
  va_end(ap);
  return st;
}

namespace {
// Encoded maps of recent calls, per host thread.  An encoding is a pure
// function of its arguments (no device state), so a call with the same
// arguments -- the same buffers, shapes and boxes, as in a serving or
// training loop -- reuses it instead of encoding again.
struct MapKey {
  const void* base;
  uint64_t dims[5], strides[4];
  uint32_t box[5];
  int32_t dtype, rank, swizzle, promotion;
  bool operator==(const MapKey& o) const { return memcmp(this, &o, sizeof *this) == 0; }
};
struct MapEntry {
  bool used;
  MapKey key;
  CUtensorMap map;
};
constexpr int kMapCacheSlots = 64;
thread_local MapEntry t_map_cache[kMapCacheSlots];

uint32_t map_slot(const MapKey& k) {
  const unsigned char* b = reinterpret_cast<const unsigned char*>(&k);
  uint32_t h = 2166136261u;  // FNV-1a
  for (size_t i = 0; i < sizeof k; ++i) h = (h ^ b[i]) * 16777619u;
  return h % kMapCacheSlots;
}
}  // namespace

bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank,
                  const void* base, const uint64_t* dims,
                  const uint64_t* strides_bytes, const uint32_t* box,
                  CUtensorMapSwizzle swizzle, CUtensorMapL2promotion promotion) {
  MapKey key;
  memset(&key, 0, sizeof key);  // padding bytes take part in the comparison
  key.base = base;
  for (int i = 0; i < rank && i < 5; ++i) {
    key.dims[i] = dims[i];
    key.box[i] = box[i];
    if (i + 1 < rank) key.strides[i] = strides_bytes[i];
  }
  key.dtype = (int32_t)dtype;
  key.rank = rank;
  key.swizzle = (int32_t)swizzle;
  key.promotion = (int32_t)promotion;
  MapEntry& slot = t_map_cache[map_slot(key)];
  if (slot.used && slot.key == key) {
    *map = slot.map;
    return true;
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    fail(SA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable (no CUDA driver?)");
    return false;
  }
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map, dtype, (cuuint32_t)rank, const_cast<void*>(base),
                  reinterpret_cast<const cuuint64_t*>(dims),
                  reinterpret_cast<const cuuint64_t*>(strides_bytes),
                  reinterpret_cast<const cuuint32_t*>(box), estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  promotion, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    fail(SA_ERR_INVALID_ARG, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return false;
  }
  slot.used = true;
  slot.key = key;
  slot.map = *map;
  return true;
}

bool set_dynamic_smem_once(const void* func, int bytes) {
  // (kernel, device) pairs whose attribute is already at least `bytes`
  struct Done {
    const void* func;
    int dev;
    int bytes;
  };
  static std::mutex mu;
  static Done done[256];
  static int ndone = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < ndone; ++i)
    if (done[i].func == func && done[i].dev == dev && done[i].bytes >= bytes) return true;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return false;
  for (int i = 0; i < ndone; ++i)
    if (done[i].func == func && done[i].dev == dev) {
      done[i].bytes = bytes;
      return true;
    }
  if (ndone < 256) done[ndone++] = Done{func, dev, bytes};
  return true;
}

uint32_t* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return nullptr;
  const uint64_t ctx = current_context_id();  // 0 before the runtime made one
  std::lock_guard<std::mutex> guard(g_err_mu);
  ErrSlot& slot = g_err_slot[dev];
  if (slot.ptr && ctx != 0 && slot.ctx == ctx) return slot.ptr;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_device_error) != cudaSuccess) return nullptr;
  slot.ctx = current_context_id();
  slot.ptr = static_cast<uint32_t*>(addr);
  return slot.ptr;
}

int num_sms() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1)
    v = 1;
  cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

}  // namespace sa

using sa::fail;

extern "C" {

const char* sa_last_error(void) { return sa::t_last_error; }

uint32_t sa_version(void) { return (0u << 16) | 1u; }

namespace sa {
namespace {
// One bounded wait on an mbarrier that nothing ever arrives on: it runs out
// after kWaitLimitNs, records kErrWaitCheck and the kernel returns normally.
__global__ void wait_expiry_kernel(uint32_t* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_wait(&bar, 0, err, kErrWaitCheck);
  }
}
}  // namespace
}  // namespace sa

sa_status sa_check_wait_expiry(void* stream) {
  uint32_t* err = sa::device_error_word();
  if (!err) return fail(SA_ERR_CUDA, "sa_check_wait_expiry: no usable CUDA device");
  sa::wait_expiry_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(SA_ERR_CUDA, "sa_check_wait_expiry launch: %s", cudaGetErrorString(e));
  return SA_OK;
}

sa_status sa_device_error(uint32_t* code) {
  if (!code) return fail(SA_ERR_INVALID_ARG, "sa_device_error: code is NULL");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess)
    return fail(SA_ERR_CUDA, "sa_device_error: %s", cudaGetErrorString(e));
  uint32_t v = 0, zero = 0;
  e = cudaMemcpyFromSymbol(&v, sa::g_device_error, sizeof v);
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(sa::g_device_error, &zero, sizeof zero);
  if (e != cudaSuccess)
    return fail(SA_ERR_CUDA, "sa_device_error: %s", cudaGetErrorString(e));
  *code = v;
  return SA_OK;
}

sa_status sa_varlen_window_fwd(const void* q, const void* k, const void* v,
                               const int32_t* cu_seqlens, int32_t num_seqs,
                               int64_t total_tokens, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim,
                               int32_t window_left, int32_t window_right,
                               const float* sinks, int32_t sink_mode,
                               float softmax_scale, void* out, float* lse,
                               void* stream) {
  const char* fn = "sa_varlen_window_fwd";
  if (!q || !k || !v || !cu_seqlens || !out || !lse)
    return fail(SA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
  if (sink_mode < SA_SINK_NONE || sink_mode > SA_SINK_NULL_LOGIT)
    return fail(SA_ERR_INVALID_ARG, "%s: unknown sink_mode %d", fn, sink_mode);
  if (sink_mode != SA_SINK_NONE && !sinks)
    return fail(SA_ERR_INVALID_ARG, "%s: sinks is NULL with sink_mode %d", fn, sink_mode);
  if (num_seqs < 1)
    return fail(SA_ERR_INVALID_ARG, "%s: num_seqs %d < 1", fn, num_seqs);
  if (total_tokens < 0 || total_tokens > (int64_t)0x7FFFF000)
    return fail(SA_ERR_INVALID_ARG, "%s: total_tokens %lld out of range [0, 2^31 - 4096]",
                fn, (long long)total_tokens);
  if (num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads != 0)
    return fail(SA_ERR_INVALID_ARG,
                "%s: num_q_heads %d must be a positive multiple of num_kv_heads %d",
                fn, num_q_heads, num_kv_heads);
  if (head_dim < 1)
    return fail(SA_ERR_INVALID_ARG, "%s: head_dim %d < 1", fn, head_dim);
  if (window_left < 0 || window_right < 0)
    return fail(SA_ERR_INVALID_ARG, "%s: negative window (%d, %d)", fn, window_left,
                window_right);
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale))
    return fail(SA_ERR_INVALID_ARG, "%s: softmax_scale must be finite and > 0", fn);
  if (!sa::aligned(q, 16) || !sa::aligned(k, 16) || !sa::aligned(v, 16) ||
      !sa::aligned(out, 16) || !sa::aligned(lse, 4) || !sa::aligned(cu_seqlens, 4) ||
      (sinks && !sa::aligned(sinks, 4)))
    return fail(SA_ERR_INVALID_ARG, "%s: misaligned pointer (bf16 tensors need 16 bytes)", fn);
  if (total_tokens == 0) return SA_OK;
  if (!sa::device_error_word())
    return fail(SA_ERR_CUDA, "%s: no usable CUDA device", fn);

  sa::WindowArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.cu_seqlens = cu_seqlens;
  a.num_seqs = num_seqs;
  a.total_tokens = total_tokens;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.window_left = window_left;
  a.window_right = window_right;
  a.sinks = sinks;
  a.sink_mode = sink_mode;
  a.softmax_scale = softmax_scale;
  a.out = out;
  a.lse = lse;
  a.stream = static_cast<cudaStream_t>(stream);
  return sa::launch_window_fwd(a);
}

namespace {
// Shared checks and dispatch of the single-table and per-index-head entries.
sa_status block_sparse_entry(const char* fn, const void* q, const void* k, const void* v,
                             int32_t batch, int32_t seq_len, int32_t num_q_heads,
                             int32_t num_kv_heads, int32_t head_dim,
                             const int32_t* block_table, int32_t num_index_heads,
                             int32_t topk_blocks, int32_t block_size, const int32_t* cu_docs,
                             int32_t num_docs, const float* sinks, int32_t sink_mode,
                             float softmax_scale, void* out, float* lse, void* stream) {
  if (!q || !k || !v || !cu_docs || !out || !lse || (topk_blocks > 0 && !block_table))
    return fail(SA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
  if (sink_mode < SA_SINK_NONE || sink_mode > SA_SINK_NULL_LOGIT)
    return fail(SA_ERR_INVALID_ARG, "%s: unknown sink_mode %d", fn, sink_mode);
  if (sink_mode != SA_SINK_NONE && !sinks)
    return fail(SA_ERR_INVALID_ARG, "%s: sinks is NULL with sink_mode %d", fn, sink_mode);
  if (batch < 0 || seq_len < 0 || topk_blocks < 0 || block_size < 1 || num_docs < 1 ||
      head_dim < 1)
    return fail(SA_ERR_INVALID_ARG,
                "%s: bad sizes (batch %d, seq_len %d, topk_blocks %d, block_size %d, "
                "num_docs %d, head_dim %d)",
                fn, batch, seq_len, topk_blocks, block_size, num_docs, head_dim);
  if (num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads != 0)
    return fail(SA_ERR_INVALID_ARG,
                "%s: num_q_heads %d must be a positive multiple of num_kv_heads %d", fn,
                num_q_heads, num_kv_heads);
  if (num_index_heads < 1 || num_kv_heads % num_index_heads != 0)
    return fail(SA_ERR_INVALID_ARG,
                "%s: num_index_heads %d must divide num_kv_heads %d", fn, num_index_heads,
                num_kv_heads);
  if ((int64_t)batch * seq_len >= ((int64_t)1 << 31))
    return fail(SA_ERR_INVALID_ARG, "%s: batch * seq_len >= 2^31", fn);
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale))
    return fail(SA_ERR_INVALID_ARG, "%s: softmax_scale must be finite and > 0", fn);
  if (!sa::aligned(q, 16) || !sa::aligned(k, 16) || !sa::aligned(v, 16) ||
      !sa::aligned(out, 16) || !sa::aligned(lse, 4) || !sa::aligned(cu_docs, 4) ||
      (block_table && !sa::aligned(block_table, 4)) || (sinks && !sa::aligned(sinks, 4)))
    return fail(SA_ERR_INVALID_ARG, "%s: misaligned pointer (bf16 tensors need 16 bytes)", fn);
  if ((int64_t)batch * seq_len == 0) return SA_OK;
  if (!sa::device_error_word())
    return fail(SA_ERR_CUDA, "%s: no usable CUDA device", fn);
  sa::BlockArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.batch = batch;
  a.seq_len = seq_len;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_table = block_table;
  a.num_index_heads = num_index_heads;
  a.topk_blocks = topk_blocks;
  a.block_size = block_size;
  a.cu_docs = cu_docs;
  a.num_docs = num_docs;
  a.sinks = sinks;
  a.sink_mode = sink_mode;
  a.softmax_scale = softmax_scale;
  a.out = out;
  a.lse = lse;
  a.stream = static_cast<cudaStream_t>(stream);
  return sa::launch_block_sparse_fwd(a);
}
}  // namespace

sa_status sa_block_sparse_fwd(const void* q, const void* k, const void* v, int32_t batch,
                              int32_t seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_dim, const int32_t* block_table,
                              int32_t topk_blocks, int32_t block_size,
                              const int32_t* cu_docs, int32_t num_docs, const float* sinks,
                              int32_t sink_mode, float softmax_scale, void* out, float* lse,
                              void* workspace, size_t workspace_bytes, void* stream) {
  (void)workspace;
  (void)workspace_bytes;
  return block_sparse_entry("sa_block_sparse_fwd", q, k, v, batch, seq_len, num_q_heads,
                            num_kv_heads, head_dim, block_table, 1, topk_blocks, block_size,
                            cu_docs, num_docs, sinks, sink_mode, softmax_scale, out, lse,
                            stream);
}

sa_status sa_block_sparse_fwd_index_heads(
    const void* q, const void* k, const void* v, int32_t batch, int32_t seq_len,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, const int32_t* block_table,
    int32_t num_index_heads, int32_t topk_blocks, int32_t block_size, const int32_t* cu_docs,
    int32_t num_docs, const float* sinks, int32_t sink_mode, float softmax_scale, void* out,
    float* lse, void* stream) {
  return block_sparse_entry("sa_block_sparse_fwd_index_heads", q, k, v, batch, seq_len,
                            num_q_heads, num_kv_heads, head_dim, block_table, num_index_heads,
                            topk_blocks, block_size, cu_docs, num_docs, sinks, sink_mode,
                            softmax_scale, out, lse, stream);
}

sa_status sa_block_select(const void* index_q, const void* index_k, int32_t batch,
                          int32_t seq_len, int32_t num_index_heads, int32_t index_dim,
                          int32_t block_size, int32_t topk_blocks, int32_t* block_table,
                          void* stream) {
  const char* fn = "sa_block_select";
  if (!index_q || !index_k || !block_table)
    return fail(SA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
  if (batch < 0 || seq_len < 0 || num_index_heads < 1 || index_dim < 1 || block_size < 1 ||
      topk_blocks < 1)
    return fail(SA_ERR_INVALID_ARG,
                "%s: bad sizes (batch %d, seq_len %d, num_index_heads %d, index_dim %d, "
                "block_size %d, topk_blocks %d)",
                fn, batch, seq_len, num_index_heads, index_dim, block_size, topk_blocks);
  if ((int64_t)batch * seq_len >= ((int64_t)1 << 31))
    return fail(SA_ERR_INVALID_ARG, "%s: batch * seq_len >= 2^31", fn);
  if (!sa::aligned(index_q, 16) || !sa::aligned(index_k, 16) || !sa::aligned(block_table, 4))
    return fail(SA_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
  if ((int64_t)batch * seq_len == 0) return SA_OK;
  if (!sa::device_error_word())
    return fail(SA_ERR_CUDA, "%s: no usable CUDA device", fn);
  sa::SelectArgs a;
  a.index_q = index_q;
  a.index_k = index_k;
  a.batch = batch;
  a.seq_len = seq_len;
  a.num_index_heads = num_index_heads;
  a.index_dim = index_dim;
  a.block_size = block_size;
  a.topk_blocks = topk_blocks;
  a.block_table = block_table;
  a.stream = static_cast<cudaStream_t>(stream);
  return sa::launch_block_select(a);
}

size_t sa_sparse_index_workspace_size(int32_t num_queries, int32_t num_q_heads,
                                      int32_t dv, int32_t topk) {
  if (num_queries <= 0 || num_q_heads <= 0 || dv != 512 || topk <= 0) return 0;
  return sa::sparse_index_workspace_bytes(num_queries, num_q_heads, topk);
}

}  // extern "C"

namespace sa {
// Shared checks and dispatch of the bf16 and fp8 latent-cache entry points
// and of the allocation-free one (fixed != null: its scratch replaces the
// workspace once every argument check has passed).
sa_status sparse_index_entry(const char* fn, const void* q, const void* kv_latent,
                             const float* kv_scale, bool fp8, int64_t num_kv, int32_t dqk,
                             int32_t dv, const int32_t* indices, int32_t topk,
                             int32_t num_queries, int32_t num_q_heads, const float* sinks,
                             int32_t sink_mode, float softmax_scale, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, void* stream,
                             const FixedScratch* fixed) {
  if (!q || !kv_latent || !indices || !out || !lse || (fp8 && !kv_scale))
    return fail(SA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
  if (sink_mode < SA_SINK_NONE || sink_mode > SA_SINK_NULL_LOGIT)
    return fail(SA_ERR_INVALID_ARG, "%s: unknown sink_mode %d", fn, sink_mode);
  if (sink_mode != SA_SINK_NONE && !sinks)
    return fail(SA_ERR_INVALID_ARG, "%s: sinks is NULL with sink_mode %d", fn, sink_mode);
  if (num_queries < 0 || num_q_heads < 1 || topk < 0 || num_kv < 1 || dqk < 1 || dv < 1 ||
      dv > dqk)
    return fail(SA_ERR_INVALID_ARG,
                "%s: bad sizes (num_queries %d, num_q_heads %d, topk %d, num_kv %lld, dqk %d, dv %d)",
                fn, num_queries, num_q_heads, topk, (long long)num_kv, dqk, dv);
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale))
    return fail(SA_ERR_INVALID_ARG, "%s: softmax_scale must be finite and > 0", fn);
  if (!sa::aligned(q, 16) || !sa::aligned(kv_latent, 16) || !sa::aligned(out, 16) ||
      !sa::aligned(lse, 4) || !sa::aligned(indices, 4) || (sinks && !sa::aligned(sinks, 4)) ||
      (workspace && !sa::aligned(workspace, 16)) || (kv_scale && !sa::aligned(kv_scale, 4)))
    return fail(SA_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
  if (sink_mode == SA_SINK_KEY0_BIAS)
    return fail(SA_ERR_UNSUPPORTED, "%s: KEY0_BIAS needs a sequence start; an index list has none",
                fn);
  if (num_kv >= ((int64_t)1 << 31))
    return fail(SA_ERR_UNSUPPORTED, "%s: num_kv %lld >= 2^31", fn, (long long)num_kv);
  if (topk > sa::sparse_index_max_topk())
    return fail(SA_ERR_UNSUPPORTED, "%s: topk %d > %d", fn, topk, sa::sparse_index_max_topk());
  if (dqk != 576 || dv != 512)
    return fail(SA_ERR_UNSUPPORTED, "%s: dqk %d / dv %d (supported: 576 / 512)", fn, dqk, dv);
  if (num_queries > 0) {
    const size_t need = sa::sparse_index_workspace_bytes(num_queries, num_q_heads, topk);
    if (fixed) {
      if (need > fixed->bytes)
        return fail(SA_ERR_UNSUPPORTED,
                    "%s: these sizes need %zu bytes of scratch, above the fixed %zu bytes "
                    "(%zu MiB) of this entry point; use sa_sparse_index_fwd with a workspace",
                    fn, need, fixed->bytes, fixed->bytes >> 20);
      if (need > 0) {
        const sa_status st = fixed->address(fn, &workspace);
        if (st != SA_OK) return st;
        workspace_bytes = fixed->bytes;
      }
    } else if (need > 0 && (!workspace || workspace_bytes < need)) {
      return fail(SA_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", fn, need,
                  workspace ? workspace_bytes : (size_t)0);
    }
  }
  if (num_queries == 0) return SA_OK;
  if (!sa::device_error_word())
    return fail(SA_ERR_CUDA, "%s: no usable CUDA device", fn);
  sa::IndexArgs a;
  a.q = q;
  a.kv = kv_latent;
  a.kv_scale = fp8 ? kv_scale : nullptr;
  a.fp8 = fp8;
  a.fn = fn;
  a.num_kv = num_kv;
  a.dqk = dqk;
  a.dv = dv;
  a.indices = indices;
  a.topk = topk;
  a.num_queries = num_queries;
  a.num_q_heads = num_q_heads;
  a.sinks = sinks;
  a.sink_mode = sink_mode;
  a.softmax_scale = softmax_scale;
  a.out = out;
  a.lse = lse;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.stream = static_cast<cudaStream_t>(stream);
  return sa::launch_sparse_index_fwd(a);
}
}  // namespace sa

extern "C" {

sa_status sa_sparse_index_fwd(const void* q, const void* kv_latent, int64_t num_kv,
                              int32_t dqk, int32_t dv, const int32_t* indices,
                              int32_t topk, int32_t num_queries, int32_t num_q_heads,
                              const float* sinks, int32_t sink_mode, float softmax_scale,
                              void* out, float* lse, void* workspace,
                              size_t workspace_bytes, void* stream) {
  return sa::sparse_index_entry("sa_sparse_index_fwd", q, kv_latent, nullptr, false, num_kv,
                                dqk, dv, indices, topk, num_queries, num_q_heads, sinks,
                                sink_mode, softmax_scale, out, lse, workspace, workspace_bytes,
                                stream, nullptr);
}

sa_status sa_sparse_index_fwd_fp8(const void* q, const void* kv_fp8, const float* kv_scale,
                                  int64_t num_kv, int32_t dqk, int32_t dv,
                                  const int32_t* indices, int32_t topk, int32_t num_queries,
                                  int32_t num_q_heads, const float* sinks, int32_t sink_mode,
                                  float softmax_scale, void* out, float* lse, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  return sa::sparse_index_entry("sa_sparse_index_fwd_fp8", q, kv_fp8, kv_scale, true, num_kv,
                                dqk, dv, indices, topk, num_queries, num_q_heads, sinks,
                                sink_mode, softmax_scale, out, lse, workspace, workspace_bytes,
                                stream, nullptr);
}

sa_status sa_merge_attn_states(const void* out_a, const float* lse_a, const void* out_b,
                               const float* lse_b, int64_t num_tokens, int32_t num_heads,
                               int32_t head_dim, const float* sinks, int32_t sink_mode,
                               void* out, float* lse, void* stream) {
  const char* fn = "sa_merge_attn_states";
  if (!out_a || !lse_a || !out_b || !lse_b || !out || !lse)
    return fail(SA_ERR_INVALID_ARG, "%s: a required pointer is NULL", fn);
  if (sink_mode < SA_SINK_NONE || sink_mode > SA_SINK_NULL_LOGIT)
    return fail(SA_ERR_INVALID_ARG, "%s: unknown sink_mode %d", fn, sink_mode);
  if (sink_mode == SA_SINK_NULL_LOGIT && !sinks)
    return fail(SA_ERR_INVALID_ARG, "%s: sinks is NULL with sink_mode %d", fn, sink_mode);
  if (num_tokens < 0 || num_heads < 1 || head_dim < 1)
    return fail(SA_ERR_INVALID_ARG, "%s: bad sizes (num_tokens %lld, num_heads %d, head_dim %d)",
                fn, (long long)num_tokens, num_heads, head_dim);
  if (!sa::aligned(out_a, 16) || !sa::aligned(out_b, 16) || !sa::aligned(out, 16) ||
      !sa::aligned(lse_a, 4) || !sa::aligned(lse_b, 4) || !sa::aligned(lse, 4) ||
      (sinks && !sa::aligned(sinks, 4)))
    return fail(SA_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
  if (sink_mode == SA_SINK_KEY0_BIAS)
    return fail(SA_ERR_UNSUPPORTED,
                "%s: KEY0_BIAS lives in the partial holding key 0; merge with SA_SINK_NONE", fn);
  if (head_dim % 8 != 0 || head_dim > 1024)
    return fail(SA_ERR_UNSUPPORTED, "%s: head_dim %d (supported: multiples of 8 up to 1024)", fn,
                head_dim);
  {
    // the merged LSE must not overlap an input LSE (a row's threads read the
    // inputs while one of them writes the result)
    const uintptr_t n = (uintptr_t)num_heads * (uintptr_t)num_tokens * sizeof(float);
    const uintptr_t o = reinterpret_cast<uintptr_t>(lse);
    for (const float* in : {lse_a, lse_b}) {
      const uintptr_t i = reinterpret_cast<uintptr_t>(in);
      if (n > 0 && o < i + n && i < o + n)
        return fail(SA_ERR_INVALID_ARG, "%s: lse overlaps an input lse", fn);
    }
  }
  if (num_tokens == 0) return SA_OK;
  if (!sa::device_error_word()) return fail(SA_ERR_CUDA, "%s: no usable CUDA device", fn);
  sa::MergeArgs a;
  a.out_a = out_a;
  a.lse_a = lse_a;
  a.out_b = out_b;
  a.lse_b = lse_b;
  a.num_tokens = num_tokens;
  a.num_heads = num_heads;
  a.head_dim = head_dim;
  a.sinks = sinks;
  a.sink_mode = sink_mode;
  a.out = out;
  a.lse = lse;
  a.stream = static_cast<cudaStream_t>(stream);
  return sa::launch_merge_states(a);
}

}  // extern "C"

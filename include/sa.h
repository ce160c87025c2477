/*
 * sa.h -- C ABI of the sink-aware varlen attention forward for GB300 (sm_103a).
 *
 * One shared library (libsa.so), plain pointers and sizes, no framework types.
 *
 * Operation (all entry points).  For each query row i and query head h with
 * key set K(i) and KV head g = h / (num_q_heads / num_kv_heads):
 *
 *   l_j  = softmax_scale * <q[i,h,:], k[j,g,:]>                 j in K(i)
 *   KEY0_BIAS : l_j += sinks[h] for the first key of i's sequence
 *   LSE  = ln sum_j exp(l_j)                 (over K(i) only, natural log)
 *   out  = sum_j exp(l_j) v[j,g,:] / den,
 *          den = sum_j exp(l_j)               (NONE, KEY0_BIAS)
 *          den = sum_j exp(l_j) + exp(sinks[h])   (NULL_LOGIT)
 *   K(i) empty  ->  out = 0, LSE = -inf.
 *
 * Sources (page title, section):
 *   vLLM pull 49815 "[Bugfix][MiMo] Apply vision attention sinks in the window
 *     attention path": the sink is added to the logit of each sequence's first
 *     key; only the first window_size + 1 queries of a sequence reach that
 *     key; the LSE is that of the masked scaled logits, laid out
 *     (nheads, total_q); the null logit ("s_aux") is a different operation.
 *   afierka-intel/vllm pull 76 "Apply DeepSeek-V4 attn_sink in the XPU
 *     sparse-MLA Triton kernel", Implementation: the null-logit sink joins the
 *     denominator after the key loop, the LSE stays over the selected keys,
 *     and a -inf sink is a bitwise no-op.
 *   NeMo AutoModel "nemo_automodel.components.models.minimax_m3_vl.
 *     cp_sparse_attn": top-k key-block selection with token-level causal and
 *     packed-document masks (MiniMaxM3CPSparseAttention, _local_sparse_forward),
 *     zero output for fully masked rows, 64-bit flat offsets
 *     (_block_sel_flat_offset).
 *
 * Conventions shared by every entry point:
 *   - Tensors are caller-owned DEVICE memory, dense row-major (C order),
 *     16-byte aligned.  bf16 tensors are passed as `const void*` / `void*`.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *     enqueue work: no host synchronisation, no device-to-host reads, no
 *     allocation.  Results are valid once the stream reaches the call.
 *   - sinks: fp32 [num_q_heads], finite or -inf; may be NULL when
 *     sink_mode == SA_SINK_NONE (it is then not read).
 *   - softmax_scale: finite and > 0.
 *   - Arguments checkable on the host are checked before anything is
 *     enqueued; a rejected call returns a non-OK status, enqueues nothing and
 *     leaves a message for sa_last_error().  Errors of device-resident
 *     content (unsorted cu_seqlens, ...) are not detected; indices and block
 *     ids outside their range are treated as absent keys.
 *   - Kernels never hang: each wait on the GPU is bounded; a wait that runs
 *     out sets a bit in the device error word (sa_device_error).
 */
#ifndef SA_H_
#define SA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SA_API __attribute__((visibility("default")))
#else
#define SA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SA_SINK_NONE = 0,       /* plain softmax over K(i)                         */
  SA_SINK_KEY0_BIAS = 1,  /* sinks[h] added to the first key's logit         */
  SA_SINK_NULL_LOGIT = 2  /* exp(sinks[h]) added to the denominator only     */
} sa_sink_mode;

typedef enum {
  SA_OK = 0,
  SA_ERR_INVALID_ARG = 1, /* a null pointer, a bad size, a bad alignment     */
  SA_ERR_UNSUPPORTED = 2, /* valid request outside what the kernels cover    */
  SA_ERR_CUDA = 3,        /* the CUDA runtime refused a launch / attribute   */
  SA_ERR_WORKSPACE = 4    /* workspace missing or smaller than required      */
} sa_status;

/*
 * Sliding-window attention over cu_seqlens-packed sequences (vLLM pull 49815,
 * window attention path).  Key set of token i in sequence b:
 *   { j : cu_seqlens[b] <= j < cu_seqlens[b+1],  i - window_left <= j <= i + window_right }.
 * KEY0_BIAS biases key cu_seqlens[b] (when it lies in the window).  NULL_LOGIT
 * and NONE are also accepted.
 *
 *   q          bf16 [total_tokens, num_q_heads, head_dim]
 *   k, v       bf16 [total_tokens, num_kv_heads, head_dim]
 *   cu_seqlens int32 [num_seqs + 1], cu_seqlens[0] = 0, non-decreasing,
 *              cu_seqlens[num_seqs] = total_tokens (device memory)
 *   out        bf16 [total_tokens, num_q_heads, head_dim]   (written)
 *   lse        fp32 [num_q_heads, total_tokens]              (written)
 * Supported: head_dim in {64, 80, 128}; num_q_heads / num_kv_heads in
 * {1, 2, 4, 8, 16}; (128 / that ratio) + window_left + window_right <= 256;
 * total_tokens < 2^31.  Other valid requests return SA_ERR_UNSUPPORTED.
 */
SA_API sa_status sa_varlen_window_fwd(const void* q, const void* k, const void* v,
                               const int32_t* cu_seqlens, int32_t num_seqs,
                               int64_t total_tokens, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim,
                               int32_t window_left, int32_t window_right,
                               const float* sinks, int32_t sink_mode,
                               float softmax_scale, void* out, float* lse,
                               void* stream);

/*
 * Top-k index attention into one shared latent KV cache (MLA decode) -- the
 * sparse-MLA kernel of afierka-intel/vllm pull 76 "Apply DeepSeek-V4 attn_sink
 * in the XPU sparse-MLA Triton kernel".  Query q attends exactly the keys
 * listed in indices[q, :]; entries outside [0, num_kv) (the -1 padding, at any
 * position) are absent; a repeated index counts twice.  K is the whole latent
 * row, V its first dv columns, shared by all query heads.  NONE and NULL_LOGIT
 * (LSE over the listed keys only) are supported; KEY0_BIAS has no first key
 * here and returns SA_ERR_UNSUPPORTED.
 *
 *   q          bf16 [num_queries, num_q_heads, dqk]
 *   kv_latent  bf16 [num_kv, dqk]
 *   indices    int32 [num_queries, topk]
 *   out        bf16 [num_queries, num_q_heads, dv]            (written)
 *   lse        fp32 [num_q_heads, num_queries]                 (written)
 *   workspace  device scratch of at least
 *              sa_sparse_index_workspace_size(num_queries, num_q_heads, dv, topk)
 *              bytes (may be NULL when that size is 0: no queries or topk = 0),
 *              16-byte aligned; its contents need no initialisation and are
 *              overwritten.  It holds the compacted index rows, the valid
 *              count of each query and, when topk > 256, the split-KV partials
 *              (O, m, l per query, 256-key item and head).
 * Supported: dqk = 576, dv = 512, topk <= 8192, num_kv < 2^31.
 */
SA_API sa_status sa_sparse_index_fwd(const void* q, const void* kv_latent,
                                     int64_t num_kv, int32_t dqk, int32_t dv,
                                     const int32_t* indices, int32_t topk,
                                     int32_t num_queries, int32_t num_q_heads,
                                     const float* sinks, int32_t sink_mode,
                                     float softmax_scale, void* out, float* lse,
                                     void* workspace, size_t workspace_bytes,
                                     void* stream);

/*
 * sa_sparse_index_fwd over an fp8 latent cache -- the decode call site of
 * afierka-intel/vllm pull 76 ("What": the V4 decode path, whose cache is
 * fp8).  The page does not fix the cache format; this call takes e4m3 codes
 * (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 is
 * subnormal; codes 0x7F / 0xFF are NaN) with one fp32 scale per latent row:
 * row r's value in column c is e4m3(kv_fp8[r, c]) * kv_scale[r].  K is the
 * whole row, V its first dv columns, exactly as in sa_sparse_index_fwd; key
 * sets, sink modes, results, workspace (same size function) and errors are
 * those of sa_sparse_index_fwd.  The rows enter the MMAs unscaled and exact
 * (every e4m3 value is a bf16 value); the scale multiplies each logit and
 * each probability in fp32.
 *
 *   kv_fp8     e4m3 bytes [num_kv, dqk], 16-byte aligned
 *   kv_scale   fp32 [num_kv] (device memory, finite and > 0 for listed rows)
 */
SA_API sa_status sa_sparse_index_fwd_fp8(const void* q, const void* kv_fp8,
                                         const float* kv_scale, int64_t num_kv,
                                         int32_t dqk, int32_t dv,
                                         const int32_t* indices, int32_t topk,
                                         int32_t num_queries, int32_t num_q_heads,
                                         const float* sinks, int32_t sink_mode,
                                         float softmax_scale, void* out, float* lse,
                                         void* workspace, size_t workspace_bytes,
                                         void* stream);

/* Workspace bytes sa_sparse_index_fwd (and _fp8) needs for these sizes (0 if none). */
SA_API size_t sa_sparse_index_workspace_size(int32_t num_queries,
                                             int32_t num_q_heads, int32_t dv,
                                             int32_t topk);

/*
 * Block-sparse causal attention with packed documents (DSA-style prefill) --
 * the sparse attention of NeMo AutoModel "nemo_automodel.components.models.
 * minimax_m3_vl.cp_sparse_attn" (MiniMaxM3CPSparseAttention step 4: selected
 * key blocks + token-level causal; _local_sparse_forward: packed document
 * masks, zero output for fully masked rows).  Tokens are batch rows of
 * seq_len packed back to back.  Key set of token i at row position p whose
 * document starts at row position d:
 *   { j in i's batch row : (j's row position) / block_size listed in
 *     block_table[i, :],  d <= j's row position <= p }.
 * Block ids count blocks from the start of the batch row; ids outside
 * [0, seq_len / block_size) (the -1 padding) are absent; a repeated id is one
 * selection.  One selection per token is shared by all heads.  A row with an
 * empty key set gives zero output and LSE = -inf.  NONE, NULL_LOGIT and
 * KEY0_BIAS are supported; KEY0_BIAS adds s_h to the logit of the first token
 * of the token's document (vLLM pull 49815, second paragraph, with documents
 * as the sequences) when that key is in the token's set.
 *
 *   q            bf16 [batch * seq_len, num_q_heads, head_dim]
 *   k, v         bf16 [batch * seq_len, num_kv_heads, head_dim]
 *   block_table  int32 [batch * seq_len, topk_blocks]
 *   cu_docs      int32 [num_docs + 1]: document starts over the flattened
 *                tokens, cu_docs[0] = 0, non-decreasing, last = batch*seq_len
 *   out          bf16 [batch * seq_len, num_q_heads, head_dim]   (written)
 *   lse          fp32 [num_q_heads, batch * seq_len]              (written)
 *   workspace    reserved: the current kernel needs none (NULL / 0 accepted)
 * Supported: head_dim = 128, block_size = 64, num_q_heads / num_kv_heads in
 * {1, 2, 4, 8, 16}, seq_len a multiple of 128 and <= 1048576,
 * (128 / that ratio) * topk_blocks <= 2048, batch * seq_len < 2^31.
 */
SA_API sa_status sa_block_sparse_fwd(const void* q, const void* k, const void* v,
                                     int32_t batch, int32_t seq_len,
                                     int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t head_dim, const int32_t* block_table,
                                     int32_t topk_blocks, int32_t block_size,
                                     const int32_t* cu_docs, int32_t num_docs,
                                     const float* sinks, int32_t sink_mode,
                                     float softmax_scale, void* out, float* lse,
                                     void* workspace, size_t workspace_bytes,
                                     void* stream);

/*
 * sa_block_sparse_fwd with one block selection per index head ([M3 CP
 * sparse] _select_local_blocks: [batch, index_heads, sequence, key_blocks]).
 * block_table is int32 [num_index_heads, batch * seq_len, topk_blocks] (the
 * layout sa_block_select writes); query head h uses index head
 * h / (num_q_heads / num_index_heads).  num_index_heads must divide
 * num_kv_heads (the query heads of one KV head share one selection),
 * otherwise SA_ERR_INVALID_ARG.  Everything else -- key sets, sink modes,
 * layouts, supported sizes and errors -- as sa_block_sparse_fwd, which is
 * this call with num_index_heads = 1.
 */
SA_API sa_status sa_block_sparse_fwd_index_heads(
    const void* q, const void* k, const void* v, int32_t batch, int32_t seq_len,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    const int32_t* block_table, int32_t num_index_heads, int32_t topk_blocks,
    int32_t block_size, const int32_t* cu_docs, int32_t num_docs, const float* sinks,
    int32_t sink_mode, float softmax_scale, void* out, float* lse, void* stream);

/*
 * Top-k key-block selection from indexer scores, one selection per index
 * head -- [M3 CP sparse] MiniMaxM3CPSparseAttention forward step 3 (top-k
 * key blocks of each query from index q / k over the causal sequence of its
 * batch row) and _select_local_blocks (one selection per index head;
 * documents are not consulted -- their mask is applied in the attention).
 * The page gives no score formula; this call takes: token score
 * index_q[i, g] . index_k[j] (fp32 accumulation of the bf16 inputs); a
 * block's score is the max over its keys; token i at row position p always
 * selects its own block p / block_size, plus the topk_blocks - 1
 * highest-scoring earlier blocks of its batch row (ties to the lower id); a
 * token with at most topk_blocks causal blocks selects them all.  Scores
 * that differ only in the last fp32 bits may rank either way.
 *
 *   index_q      bf16 [batch * seq_len, num_index_heads, index_dim]
 *   index_k      bf16 [batch * seq_len, index_dim]  (one index key per token)
 *   block_table  int32 [num_index_heads, batch * seq_len, topk_blocks]
 *                (written: ascending block ids from the batch-row start,
 *                -1 padded) -- the input of sa_block_sparse_fwd_index_heads
 * Supported: index_dim = 128, block_size = 64, seq_len a multiple of 128,
 * 1 <= topk_blocks <= 16, batch * seq_len < 2^31.  No workspace.
 */
SA_API sa_status sa_block_select(const void* index_q, const void* index_k, int32_t batch,
                                 int32_t seq_len, int32_t num_index_heads,
                                 int32_t index_dim, int32_t block_size,
                                 int32_t topk_blocks, int32_t* block_table, void* stream);

/*
 * Merge of two partial attention results over disjoint key sets of the same
 * queries (a cascade / split of one key set over calls) into the attention
 * over their union.  Each partial is the sink-free attention over its own
 * keys (computed with SA_SINK_NONE) with its LSE; the merge weighs them by
 * their LSEs -- the LSE convention of vLLM pull 49815, LSE paragraph -- and,
 * with SA_SINK_NULL_LOGIT, folds the sink once as afierka-intel/vllm pull 76,
 * Implementation does after its key loop (the sink joins the denominator
 * only; the merged LSE stays over real keys; a -inf sink changes nothing).
 * A partial with LSE = -inf holds no keys; if both do, out = 0, LSE = -inf.
 * KEY0_BIAS is a bias on a real key, already inside the partial that holds
 * that key: merge those partials with SA_SINK_NONE (KEY0_BIAS returns
 * SA_ERR_UNSUPPORTED).
 *
 *   out_a, out_b  bf16 [num_tokens, num_heads, head_dim]
 *   lse_a, lse_b  fp32 [num_heads, num_tokens]
 *   out           bf16 [num_tokens, num_heads, head_dim]  (written; may be
 *                 out_a or out_b itself)
 *   lse           fp32 [num_heads, num_tokens]            (written; must not
 *                 overlap lse_a or lse_b)
 * Supported: head_dim a multiple of 8 and <= 1024; 16-byte aligned out
 * pointers.  No workspace.
 */
SA_API sa_status sa_merge_attn_states(const void* out_a, const float* lse_a,
                                      const void* out_b, const float* lse_b,
                                      int64_t num_tokens, int32_t num_heads,
                                      int32_t head_dim, const float* sinks,
                                      int32_t sink_mode, void* out, float* lse,
                                      void* stream);

/*
 * Allocation-free variant of sa_sparse_index_fwd.  The pages have no
 * counterpart: it exists for callers that cannot allocate device memory for a
 * workspace -- for example code running inside a host runtime that owns the
 * whole device memory pool and gives its plugins no allocator, or a serving
 * loop that must not allocate once it runs.  Arguments, layouts, results and
 * errors are those of sa_sparse_index_fwd, without the workspace.
 *
 * The split-KV scratch is a fixed 64 MiB array inside the library, reserved on
 * every GPU that loads the library until the process exits.  Every argument
 * is checked first, as sa_sparse_index_fwd checks it (same statuses, messages
 * naming this entry point); then sizes whose sa_sparse_index_workspace_size()
 * exceeds 64 MiB are rejected with SA_ERR_UNSUPPORTED and a message; use
 * sa_sparse_index_fwd for them.  The call itself allocates nothing.  The first
 * call on each device looks up the array's device address once (make that
 * first call before any stream capture); the address is kept with the id of
 * the CUDA context it belongs to, and looked up again when the device's
 * context has been destroyed and re-created (cudaDeviceReset).  All calls
 * share the array: calls whose work overlaps on the GPU (other streams or
 * host threads) race and must be serialised by the caller.
 */
SA_API sa_status sa_sparse_index_fwd_noalloc(const void* q, const void* kv_latent,
                                             int64_t num_kv, int32_t dqk, int32_t dv,
                                             const int32_t* indices, int32_t topk,
                                             int32_t num_queries, int32_t num_q_heads,
                                             const float* sinks, int32_t sink_mode,
                                             float softmax_scale, void* out, float* lse,
                                             void* stream);

/* Message of the last non-OK status returned on this host thread ("" if none). */
SA_API const char* sa_last_error(void);

/*
 * Device error word of the current device: bits set by kernels whose bounded
 * waits ran out (1 load, 2 MMA, 4 buffer release, 8 drain, 16 config,
 * 32 the wait of sa_check_wait_expiry).  Synchronises the device, reads the
 * word into *code and clears it.
 */
SA_API sa_status sa_device_error(uint32_t* code);

/*
 * Exercises the failure path of the bounded waits without faulting anything:
 * enqueues one kernel whose thread waits on an mbarrier that nothing ever
 * arrives on.  The wait runs out after about one second, the kernel sets
 * bit 32 of the device error word and returns normally; the context stays
 * usable.  A caller checks the mechanism with this call followed by
 * sa_device_error (expect 32).
 */
SA_API sa_status sa_check_wait_expiry(void* stream);

/* Library version as (major << 16) | minor. */
SA_API uint32_t sa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SA_H_ */

/*
 * sa_oracle.c -- CPU oracle for sink-aware varlen attention (forward).
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load or run this file.  It
 * shares no code, header or constant with the CUDA library and never calls it.
 *
 * Precision: every quantity is double (fp64).  Inputs arrive as the exact
 * bf16 bit patterns the GPU receives, widened exactly to double; sinks and the
 * softmax scale arrive as the fp32 values the GPU receives, widened to double.
 *
 * Sources (cited by page title and section):
 *  [P1] vLLM pull 49815, "[Bugfix][MiMo] Apply vision attention sinks in the
 *       window attention path": the sink is added to the logit of each
 *       sequence's first key (second paragraph); only the first
 *       window_size + 1 queries of a sequence reach key 0 (paragraph after the
 *       closed form); the returned LSE is the log-sum-exp of the masked,
 *       scaled logits with shape (nheads, total_q) (LSE-convention paragraph);
 *       a null logit in the denominator ("s_aux") is a different operation
 *       (first of the "Two alternatives").
 *  [P2] afierka-intel/vllm pull 76, "Apply DeepSeek-V4 attn_sink in the XPU
 *       sparse-MLA Triton kernel", section "Implementation": the sink enters
 *       only the denominator, the LSE stays over the selected keys, and a
 *       -inf sink changes nothing.
 *  [P3] NeMo AutoModel API page
 *       "nemo_automodel.components.models.minimax_m3_vl.cp_sparse_attn":
 *       block selection + token-level causal (MiniMaxM3CPSparseAttention,
 *       step 4), packed document mask and zero output for fully masked rows
 *       (_local_sparse_forward), 64-bit flat offsets (_block_sel_flat_offset).
 *
 * The definition implemented, per query row i and query head h with key set
 * K(i) and kv head g = h / (Hq / Hkv):
 *     l_j   = scale * <q[i,h,:], k[j,g,:]>                       j in K(i)
 *     KEY0_BIAS:  l_j += s_h   for j = first key of i's sequence (window) or
 *                 document (block), if j in K(i)
 *     M     = max_j l_j,   Z = sum_j exp(l_j - M),   LSE = M + ln Z
 *     den   = Z e^M                    (NONE, KEY0_BIAS)
 *           = Z e^M + e^{s_h}          (NULL_LOGIT; LSE unchanged)
 *     out   = sum_j e^{l_j} v[j,g,:] / den
 *     K(i) empty  ->  out = 0, LSE = -inf.
 * Everything is evaluated directly from this definition, key by key.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_NONE = 0, OR_KEY0_BIAS = 1, OR_NULL_LOGIT = 2 };

/* Exact widening of a bf16 bit pattern to double. */
static double bf16_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/*
 * One query row of one head over an explicit list of keys.
 *   qrow   : dqk query values (already widened).
 *   keys   : nkeys key positions; key j's vector starts at K + keys[j]*kstride,
 *            its value vector at V + keys[j]*vstride (first dv entries).
 *   bias_key: position that receives the KEY0_BIAS sink, or -1.
 *   mode / sink: sink convention and s_h.
 * Writes out[0..dv) and *lse.  logit is scratch of length >= nkeys.
 */
static void attend_row(const double* qrow, int dqk, int dv,
                       const uint16_t* K, int64_t kstride,
                       const uint16_t* V, int64_t vstride,
                       const int64_t* keys, int64_t nkeys, int64_t bias_key,
                       int mode, double sink, double scale,
                       double* out, double* lse, double* logit) {
  int64_t j;
  int d;
  for (d = 0; d < dv; ++d) out[d] = 0.0;
  if (nkeys == 0) {
    *lse = -INFINITY;
    return;
  }
  /* logits l_j = scale * <q, k_j> (+ s_h on the first key, KEY0_BIAS) */
  double M = -INFINITY;
  for (j = 0; j < nkeys; ++j) {
    const uint16_t* kr = K + keys[j] * kstride;
    double acc = 0.0;
    for (d = 0; d < dqk; ++d) acc += qrow[d] * bf16_to_double(kr[d]);
    double l = scale * acc;
    if (mode == OR_KEY0_BIAS && keys[j] == bias_key) l += sink;
    logit[j] = l;
    if (l > M) M = l;
  }
  if (M == -INFINITY) {
    /* every logit is -inf (a -inf KEY0 bias on the only key): empty set */
    *lse = -INFINITY;
    return;
  }
  double Z = 0.0;
  for (j = 0; j < nkeys; ++j) Z += exp(logit[j] - M);
  *lse = M + log(Z);
  /* den = Z e^M (+ e^s); evaluated as e^{M'} (Z e^{M-M'} + e^{s-M'}). */
  double Mp = M;
  double den_scaled = Z; /* den / e^{Mp} */
  if (mode == OR_NULL_LOGIT && sink > M) Mp = sink;
  if (mode == OR_NULL_LOGIT) den_scaled = Z * exp(M - Mp) + exp(sink - Mp);
  for (j = 0; j < nkeys; ++j) {
    double w = exp(logit[j] - Mp) / den_scaled;
    const uint16_t* vr = V + keys[j] * vstride;
    for (d = 0; d < dv; ++d) out[d] += w * bf16_to_double(vr[d]);
  }
}

/* ------------------------------------------------------------------------ */
/* Sliding window over cu_seqlens-packed sequences ([P1]).                   */
/* Key set: keys j of i's own sequence with i - wl <= j <= i + wr.           */
/* KEY0_BIAS key: the sequence's first token cu_seqlens[b].                  */
/* q [T,Hq,D], k/v [T,Hkv,D]; out [T,Hq,D]; lse [Hq,T]; key_count [T,Hq].    */
/* Rows i in [row_begin, row_end) are computed; others are left untouched.   */
/* Returns 0, or -1 on bad arguments.                                        */
/* ------------------------------------------------------------------------ */
int oracle_window_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                      const int32_t* cu_seqlens, int32_t num_seqs,
                      int64_t total_tokens, int32_t hq, int32_t hkv, int32_t d,
                      int32_t wl, int32_t wr, const float* sinks,
                      int32_t mode, double scale, double* out, double* lse,
                      int32_t* key_count, int64_t row_begin, int64_t row_end) {
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0 || d <= 0 || wl < 0 || wr < 0)
    return -1;
  if (num_seqs < 0 || cu_seqlens[0] != 0 || cu_seqlens[num_seqs] != total_tokens)
    return -1;
  if (row_begin < 0) row_begin = 0;
  if (row_end > total_tokens) row_end = total_tokens;
  const int64_t group = hq / hkv;
  const int64_t nrows = (row_end > row_begin) ? (row_end - row_begin) : 0;
  const int64_t nwork = nrows * hq;
  int64_t w;
#pragma omp parallel
  {
    double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
    int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)(wl + wr + 1));
    double* logit = (double*)malloc(sizeof(double) * (size_t)(wl + wr + 1));
#pragma omp for schedule(dynamic, 64)
    for (w = 0; w < nwork; ++w) {
      const int64_t i = row_begin + w / hq;
      const int h = (int)(w % hq);
      const int g = (int)(h / group);
      /* sequence b with cu_seqlens[b] <= i < cu_seqlens[b+1] */
      int b = 0;
      while (b + 1 < num_seqs && cu_seqlens[b + 1] <= i) ++b;
      const int64_t s0 = cu_seqlens[b], s1 = cu_seqlens[b + 1];
      int64_t lo = i - wl, hi = i + wr;
      if (lo < s0) lo = s0;
      if (hi > s1 - 1) hi = s1 - 1;
      int64_t n = 0, j;
      for (j = lo; j <= hi; ++j) keys[n++] = j;
      int dd;
      for (dd = 0; dd < d; ++dd)
        qrow[dd] = bf16_to_double(q[(i * hq + h) * (int64_t)d + dd]);
      const double s = (mode == OR_NONE) ? 0.0 : (double)sinks[h];
      double l;
      attend_row(qrow, d, d, k + (int64_t)g * d, (int64_t)hkv * d,
                 v + (int64_t)g * d, (int64_t)hkv * d, keys, n,
                 (mode == OR_KEY0_BIAS) ? s0 : -1, mode, s, scale,
                 out + (i * hq + h) * (int64_t)d, &l, logit);
      lse[(int64_t)h * total_tokens + i] = l;
      if (key_count) key_count[i * hq + h] = (int32_t)n;
    }
    free(qrow);
    free(keys);
    free(logit);
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Top-k index list into one shared latent KV cache (MLA style, [P2]).      */
/* q [Nq,Hq,dqk]; kv [nkv,dqk], V = first dv columns of each kv row;        */
/* idx [Nq,topk]; entries outside [0,nkv) (the -1 padding) are skipped.     */
/* Listed keys are attended as listed (a repeated index counts twice).      */
/* out [Nq,Hq,dv]; lse [Hq,Nq]; key_count [Nq] (valid entries per query).   */
/* ------------------------------------------------------------------------ */
int oracle_sparse_index_fwd(const uint16_t* q, const uint16_t* kv, int64_t nkv,
                            int32_t dqk, int32_t dv, const int32_t* idx,
                            int32_t topk, int32_t nq, int32_t hq,
                            const float* sinks, int32_t mode, double scale,
                            double* out, double* lse, int32_t* key_count,
                            int64_t row_begin, int64_t row_end) {
  if (dqk <= 0 || dv <= 0 || dv > dqk || topk < 0 || nq < 0 || hq <= 0)
    return -1;
  if (mode == OR_KEY0_BIAS) return -1; /* no sequence start in an index list */
  if (row_begin < 0) row_begin = 0;
  if (row_end > nq) row_end = nq;
  const int64_t nrows = (row_end > row_begin) ? (row_end - row_begin) : 0;
  const int64_t nwork = nrows * hq;
  int64_t w;
#pragma omp parallel
  {
    double* qrow = (double*)malloc(sizeof(double) * (size_t)dqk);
    int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)(topk + 1));
    double* logit = (double*)malloc(sizeof(double) * (size_t)(topk + 1));
#pragma omp for schedule(dynamic, 16)
    for (w = 0; w < nwork; ++w) {
      const int64_t i = row_begin + w / hq;
      const int h = (int)(w % hq);
      int64_t n = 0;
      int t;
      for (t = 0; t < topk; ++t) {
        const int64_t j = idx[i * topk + t];
        if (j >= 0 && j < nkv) keys[n++] = j;
      }
      int dd;
      for (dd = 0; dd < dqk; ++dd)
        qrow[dd] = bf16_to_double(q[(i * hq + h) * (int64_t)dqk + dd]);
      const double s = (mode == OR_NONE) ? 0.0 : (double)sinks[h];
      double l;
      attend_row(qrow, dqk, dv, kv, dqk, kv, dqk, keys, n, -1, mode, s, scale,
                 out + (i * hq + h) * (int64_t)dv, &l, logit);
      lse[(int64_t)h * nq + i] = l;
      if (key_count && h == 0) key_count[i] = (int32_t)n;
    }
    free(qrow);
    free(keys);
    free(logit);
  }
  return 0;
}

static int cmp_i32(const void* a, const void* b) {
  const int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

/* ------------------------------------------------------------------------ */
/* Block-sparse causal attention with document mask ([P3]).                */
/* Tokens are [batch, seq_len] flattened; q [B*S,Hq,D], k/v [B*S,Hkv,D].    */
/* table [B*S, topk_blocks]: key-block ids counted from the start of the    */
/* query's batch row; ids outside [0, ceil(S/block)) are ignored, repeats   */
/* are one selection (membership).  cu_docs [num_docs+1] marks document     */
/* starts over the flattened tokens.  Key set of token i (row position p):  */
/*   { j in i's batch row : (j's row position)/block in table(i),           */
/*     j <= i, doc(j) == doc(i) }.                                          */
/* KEY0_BIAS key: the first token of i's document (the [P1] bias on each    */
/* sequence's first key, with documents as the sequences), if in the row.   */
/* out [B*S,Hq,D]; lse [Hq,B*S]; key_count [B*S] (keys per token).          */
/* ------------------------------------------------------------------------ */
int oracle_block_sparse_fwd(const uint16_t* q, const uint16_t* k,
                            const uint16_t* v, int32_t batch, int32_t seq_len,
                            int32_t hq, int32_t hkv, int32_t d,
                            const int32_t* table, int32_t topk_blocks,
                            int32_t block_size, const int32_t* cu_docs,
                            int32_t num_docs, const float* sinks, int32_t mode,
                            double scale, double* out, double* lse,
                            int32_t* key_count, int64_t row_begin,
                            int64_t row_end) {
  const int64_t T = (int64_t)batch * seq_len;
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0 || d <= 0 || block_size <= 0 ||
      topk_blocks < 0 || batch < 0 || seq_len < 0)
    return -1;
  if (num_docs < 1 || cu_docs[0] != 0 || cu_docs[num_docs] != T) return -1;
  if (row_begin < 0) row_begin = 0;
  if (row_end > T) row_end = T;
  const int64_t group = hq / hkv;
  const int32_t nblocks = (seq_len + block_size - 1) / block_size;
  const int64_t nrows = (row_end > row_begin) ? (row_end - row_begin) : 0;
  int64_t r;
#pragma omp parallel
  {
    double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
    int64_t* keys =
        (int64_t*)malloc(sizeof(int64_t) * (size_t)(seq_len > 0 ? seq_len : 1));
    double* logit =
        (double*)malloc(sizeof(double) * (size_t)(seq_len > 0 ? seq_len : 1));
    int32_t* sel =
        (int32_t*)malloc(sizeof(int32_t) * (size_t)(topk_blocks > 0 ? topk_blocks : 1));
#pragma omp for schedule(dynamic, 8)
    for (r = 0; r < nrows; ++r) {
      const int64_t i = row_begin + r;
      const int64_t row0 = (i / seq_len) * seq_len; /* batch-row start */
      /* document of i: cu_docs[e] <= i < cu_docs[e+1] */
      int e = 0;
      while (e + 1 < num_docs && cu_docs[e + 1] <= i) ++e;
      const int64_t doc0 = cu_docs[e];
      /* KEY0_BIAS key: the first token of i's document, when it lies in
         i's batch row (a key of another row is never in the set) */
      const int64_t bias_key = doc0 >= row0 ? doc0 : -1;
      /* selected blocks of i as a sorted set */
      int nsel = 0, t;
      for (t = 0; t < topk_blocks; ++t) {
        const int32_t b = table[i * topk_blocks + t];
        if (b >= 0 && b < nblocks) sel[nsel++] = b;
      }
      qsort(sel, (size_t)nsel, sizeof(int32_t), cmp_i32);
      int64_t n = 0;
      int u;
      for (u = 0; u < nsel; ++u) {
        if (u > 0 && sel[u] == sel[u - 1]) continue; /* membership */
        int64_t j0 = row0 + (int64_t)sel[u] * block_size;
        int64_t j1 = j0 + block_size;
        if (j1 > row0 + seq_len) j1 = row0 + seq_len;
        int64_t j;
        for (j = j0; j < j1; ++j)
          if (j <= i && j >= doc0) keys[n++] = j; /* causal + same document */
      }
      int h;
      for (h = 0; h < hq; ++h) {
        const int g = (int)(h / group);
        int dd;
        for (dd = 0; dd < d; ++dd)
          qrow[dd] = bf16_to_double(q[(i * hq + h) * (int64_t)d + dd]);
        const double s = (mode == OR_NONE) ? 0.0 : (double)sinks[h];
        double l;
        attend_row(qrow, d, d, k + (int64_t)g * d, (int64_t)hkv * d,
                   v + (int64_t)g * d, (int64_t)hkv * d, keys, n, bias_key, mode, s,
                   scale, out + (i * hq + h) * (int64_t)d, &l, logit);
        lse[(int64_t)h * T + i] = l;
      }
      if (key_count) key_count[i] = (int32_t)n;
    }
    free(qrow);
    free(keys);
    free(logit);
    free(sel);
  }
  return 0;
}

/* Threads the OpenMP runtime will use for the loops above. */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

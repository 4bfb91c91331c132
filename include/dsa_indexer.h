/*
 * dsa_indexer.h -- C ABI of the GB300 (sm_103a) decode-step DSA indexer.
 *
 * For each request b of a decode batch the indexer
 *   1. reads the request's C4-compressed 64-dim index keys (one key per 4
 *      tokens, 64 keys per 256-token page) through its row of the page table;
 *   2. scores every live position t < n_b = ceil(seq_len_b / 4):
 *          score[b, t] = sum_{h < 32} w[b, h] * max(0, q[b, h, :] . k[t, :]);
 *   3. writes -inf into the rest of a full-width row of max_context / 4
 *      positions;
 *   4. selects the min(k, n_b) live positions with the largest scores.
 *
 * Where each step is defined:
 *   - the operator chain (gather through the page table, bmm of q against
 *     the keys, clamp_min at 0, multiply by the head weights, sum over heads,
 *     -inf past the live length) and the 32-head, 64-dim shapes:
 *     "The Indexer O(max_context) Breakthrough", section "The Indexer
 *     O(max_context) Breakthrough" (per-op table and tensor shapes), and
 *     "The Final Piece: Documenting a ~17x Throughput Breakthrough", section
 *     "The Context: Why This Message Was Written";
 *   - row width = page_table width x (page_size / 4):
 *     "The Moment of Breakthrough: Validating the Indexer Fix That Unlocked
 *     17x Throughput on Blackwell", section "The Context: A Long Hunt for the
 *     Hidden Wall";
 *   - a fixed grid whose pages past the live length take a cheap -inf path,
 *     with a full-size output row for the downstream top-k and for CUDA-graph
 *     capture: "The O(Actual) Indexer: Validating 128K Context at 500 tok/s on
 *     Blackwell", section "The Bottleneck That Was";
 *   - the top-k over the logits row that feeds sparse attention: same page,
 *     sections "The Benchmark Results" and "The Reasoning Process".
 * The pages print no formula, no tie rule and no output order.  Readings used
 * here: relu acts on each head's dot product before the weighted head sum;
 * equal scores are ranked by lower position; top-k indices are listed in
 * ascending position, then padded with -1.
 *
 * Conventions shared by every entry point:
 *   - Device pointers unless stated otherwise; all buffers are owned by the
 *     caller.  The library allocates, frees and synchronises nothing inside a
 *     compute call, so every compute call may be captured in a CUDA graph.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls are asynchronous on it.
 *   - The launch configuration depends only on (batch, max_context, k) and the
 *     device, never on the contents of seq_lens or page_table, so a captured
 *     graph stays valid when those contents change between replays.
 *   - Arguments are checked on the host before any launch; a failed check
 *     returns a status and launches nothing.  No C++ exception crosses the ABI.
 *   - Fixed shape: 32 heads, head dim 64, 64 C4 entries (256 tokens) per page.
 *   - Layouts (C-contiguous):
 *       q          bf16  [batch, 32, 64]                 16-byte aligned
 *       w          fp32  [batch, 32]                     16-byte aligned
 *       key_pool   bf16  [num_pages, 64, 64]  (page, entry, dim), 16-byte aligned
 *       page_table int32 [batch, max_context / 256]       physical page ids
 *       seq_lens   int32 [batch]                          tokens per request
 *       scores     fp32  [batch, max_context / 4]         16-byte aligned
 *       topk_idx   int32 [batch, k]
 *   - Page-table entries at or past slot ceil(n_b / 64) are never read.
 *   - Device data out of contract is never dereferenced: a seq_len above
 *     max_context is treated as max_context and a negative one as 0; a live
 *     page id outside [0, num_pages) is not read and its positions score -inf.
 *     Each case sets a bit in the workspace error word (DSA_DEVERR_*).
 *   - Workspace: a caller-owned device buffer, 256-byte aligned, of at least
 *     dsa_indexer_workspace_size() bytes (every entry point accepts that
 *     size), zeroed once before first use (dsa_indexer_workspace_init or any
 *     memset to 0).  Its first 256 bytes hold the sticky device error word;
 *     the rest of them is reserved and stays zero.  Calls that share a
 *     workspace must be ordered on one stream.
 */
#ifndef DSA_INDEXER_H
#define DSA_INDEXER_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DSA_API __attribute__((visibility("default")))
#else
#define DSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size or shape */
    DSA_ERR_UNSUPPORTED = 2, /* shape outside what the kernels handle (e.g. batch too large) */
    DSA_ERR_WORKSPACE = 3,   /* workspace missing, misaligned or too small */
    DSA_ERR_CUDA = 4         /* a CUDA runtime/driver call failed; see dsa_indexer_last_cuda_error */
} dsa_status_t;

/* Bits of the device error word (sticky until read with clear = 1). */
#define DSA_DEVERR_SEQ_LEN_CLAMPED 0x1u /* a seq_len was < 0 or > max_context */
#define DSA_DEVERR_BAD_PAGE        0x2u /* a live page id was outside [0, num_pages) */
#define DSA_DEVERR_WAIT_TIMEOUT    0x4u /* an in-kernel pipeline wait gave up (about 1 s) */

#define DSA_HEADS 32
#define DSA_HEAD_DIM 64
#define DSA_PAGE_TOKENS 256
#define DSA_PAGE_ENTRIES 64
#define DSA_MAX_BATCH 1024

/*
 * Bytes of workspace any entry point needs for this shape: 256 bytes of
 * header plus, for dsa_indexer_fused without a scores row, batch x
 * max_context / 4 fp32 live-score slots (only live positions are touched).
 * Returns 0 for an invalid shape.
 */
DSA_API size_t dsa_indexer_workspace_size(int32_t batch, int64_t max_context, int32_t k);

/* Zero the workspace header (error word) on `stream`.  Capture-safe. */
DSA_API dsa_status_t dsa_indexer_workspace_init(void *workspace, size_t workspace_bytes, void *stream);

/*
 * Steps 1-3: scores [batch, max_context / 4], every position written (live
 * scores, -inf elsewhere).  Cost: live key bytes, plus one streaming -inf store
 * per dead position (the full-width row).
 */
DSA_API dsa_status_t dsa_indexer_scores(const void *q, const float *w, const void *key_pool,
                                int64_t num_pages, const int32_t *page_table,
                                const int32_t *seq_lens, int32_t batch, int64_t max_context,
                                float *scores, void *workspace, size_t workspace_bytes,
                                void *stream);

/*
 * Step 4 on a scores row: topk_idx [batch, k] = the min(k, n_b) positions
 * t < n_b with the largest scores[b, t] (fp32 order, -0 == +0; equal scores:
 * lower t first), in ascending t, then -1.  A NaN score ranks by its bits:
 * above +inf with the sign bit clear, below -inf with it set, NaNs of one sign
 * ordered as their bits read as an integer (larger first when positive,
 * smaller first when negative).  Reads only scores[b, t] for t < n_b, and
 * none when n_b <= k.  1 <= k <= max_context / 4.
 */
DSA_API dsa_status_t dsa_indexer_topk(const float *scores, const int32_t *seq_lens, int32_t batch,
                              int64_t max_context, int32_t k, int32_t *topk_idx,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * Steps 1-4.  With scores_opt != NULL the full-width row is written exactly as
 * by dsa_indexer_scores and topk_idx equals dsa_indexer_topk on it.  With
 * scores_opt == NULL nothing of size max_context is written: live scores go to
 * the workspace and the cost is O(live positions) plus O(batch x k).
 * The two kernels run back to back on `stream`; the top-k kernel is the one
 * dsa_indexer_topk launches.
 */
DSA_API dsa_status_t dsa_indexer_fused(const void *q, const float *w, const void *key_pool,
                               int64_t num_pages, const int32_t *page_table,
                               const int32_t *seq_lens, int32_t batch, int64_t max_context,
                               int32_t k, int32_t *topk_idx, float *scores_opt,
                               void *workspace, size_t workspace_bytes, void *stream);

/*
 * dsa_indexer_fused without a scores row and without a workspace argument,
 * for callers that cannot allocate device memory on the path that runs the
 * indexer (a serving engine that owns all of HBM and hands kernels only
 * their tensors, custom-op hosts that provide no scratch, code that must not
 * call cudaMalloc because it can synchronise the device).  The source pages
 * have no counterpart to this entry point; it exists for those callers.
 *
 * Scratch: a library-owned device array of 256 B + 16 MiB, held by every GPU
 * that loads the library until the process exits.  batch x max_context / 4
 * fp32 live-score slots must fit in the 16 MiB (e.g. 64 requests at 256K
 * tokens, 128 at 128K), otherwise the call returns
 * DSA_ERR_UNSUPPORTED and launches nothing.  Arguments are checked exactly as
 * by dsa_indexer_fused, before the scratch is touched.  The first call on a
 * device looks up the array's device address (once per device) and must come
 * before any stream capture on that device.  All calls share the array: calls
 * that overlap on the GPU (unordered streams) race on it.  The array's device
 * error word is sticky like a workspace's; read it with
 * dsa_indexer_noalloc_get_error.  Same inputs and output as dsa_indexer_fused.
 */
DSA_API dsa_status_t dsa_indexer_fused_noalloc(const void *q, const float *w, const void *key_pool,
                                       int64_t num_pages, const int32_t *page_table,
                                       const int32_t *seq_lens, int32_t batch, int64_t max_context,
                                       int32_t k, int32_t *topk_idx, void *stream);

/*
 * dsa_indexer_get_error on the current device's scratch array of
 * dsa_indexer_fused_noalloc (DSA_DEVERR_* bits of every noalloc call since the
 * last clear).  Synchronises `stream`; allocates nothing.  No counterpart on
 * the source pages either.
 */
DSA_API dsa_status_t dsa_indexer_noalloc_get_error(uint32_t *code, int clear, void *stream);

/*
 * fp8 key cache.  The deployment on the pages keeps its KV cache in fp8
 * ("The Indexer O(max_context) Breakthrough", section "The Indexer
 * O(max_context) Breakthrough"); the pages do not give the index-key format.
 * This library's format: each C4 key is 64 OCP e4m3 codes (bias 7, no
 * infinities, 0x7F/0xFF NaN) and one fp32 scale, k[t, d] = scale[t] x
 * e4m3(code[t, d]).  Layouts (C-contiguous):
 *     key_codes   uint8 [num_pages, 64, 64]  (page, entry, dim), 16-byte aligned
 *     key_scales  fp32  [num_pages, 64]      (page, entry),      16-byte aligned
 * Scales of live keys must be positive and finite: the kernel computes
 * scale[t] x sum_h w[b, h] x max(0, q[b, h, :] . e4m3(code[t, :])), which
 * equals step 2 on k = scale x e4m3(code) exactly when scale > 0.  Codes and
 * scales of entries past the live length, or of pages no live slot names,
 * are never used (NaN there does not leak).  Everything else (q, w,
 * page_table, seq_lens, outputs, workspace, error bits, capture safety) is
 * as for the bf16 entry points above.  A key costs 68 bytes instead of 128.
 */
DSA_API dsa_status_t dsa_indexer_scores_fp8(const void *q, const float *w, const void *key_codes,
                                    const float *key_scales, int64_t num_pages,
                                    const int32_t *page_table, const int32_t *seq_lens,
                                    int32_t batch, int64_t max_context, float *scores,
                                    void *workspace, size_t workspace_bytes, void *stream);

/* dsa_indexer_fused on the fp8 key cache (same outputs, same workspace rule). */
DSA_API dsa_status_t dsa_indexer_fused_fp8(const void *q, const float *w, const void *key_codes,
                                   const float *key_scales, int64_t num_pages,
                                   const int32_t *page_table, const int32_t *seq_lens,
                                   int32_t batch, int64_t max_context, int32_t k,
                                   int32_t *topk_idx, float *scores_opt, void *workspace,
                                   size_t workspace_bytes, void *stream);

/*
 * Multi-token decoding (the MTP / EAGLE draft tokens the deployment tried to
 * enable: "The Indexer O(max_context) Breakthrough", section "MTP/EAGLE
 * Integration (Phase 2)"): next_n query tokens per request score the same
 * paged keys.  The pages give
 * no per-token rule; reading used here: the request's seq_len counts all
 * next_n tokens, and token j (0-based) sees its causal prefix of
 * L_j = seq_len - (next_n - 1 - j) tokens, i.e. n_bj = ceil(max(L_j, 0) / 4)
 * keys.  Token j of request b is row b x next_n + j of every output.
 * Layouts (C-contiguous): q bf16 [batch, next_n, 32, 64], w fp32
 * [batch, next_n, 32], scores fp32 [batch, next_n, max_context / 4],
 * topk_idx int32 [batch, next_n, k]; key_pool, page_table, seq_lens as above.
 * The keys are read once for all next_n tokens.  1 <= next_n <= 4.  next_n = 1
 * gives exactly the results of the single-token entry points.
 */
#define DSA_MAX_NEXT_N 4

/* Workspace bytes for the multi-token entry points (0 for an invalid shape):
 * 256 bytes of header plus, for dsa_indexer_fused_mtp without a scores row,
 * batch x next_n x max_context / 4 fp32 live-score slots. */
DSA_API size_t dsa_indexer_workspace_size_mtp(int32_t batch, int32_t next_n, int64_t max_context, int32_t k);

/* dsa_indexer_scores for next_n tokens per request. */
DSA_API dsa_status_t dsa_indexer_scores_mtp(const void *q, const float *w, const void *key_pool,
                                    int64_t num_pages, const int32_t *page_table,
                                    const int32_t *seq_lens, int32_t batch, int32_t next_n,
                                    int64_t max_context, float *scores, void *workspace,
                                    size_t workspace_bytes, void *stream);

/* dsa_indexer_topk over the batch x next_n rows, each with its own causal length. */
DSA_API dsa_status_t dsa_indexer_topk_mtp(const float *scores, const int32_t *seq_lens, int32_t batch,
                                  int32_t next_n, int64_t max_context, int32_t k,
                                  int32_t *topk_idx, void *workspace, size_t workspace_bytes,
                                  void *stream);

/* dsa_indexer_fused for next_n tokens per request (same rules for scores_opt and workspace). */
DSA_API dsa_status_t dsa_indexer_fused_mtp(const void *q, const float *w, const void *key_pool,
                                   int64_t num_pages, const int32_t *page_table,
                                   const int32_t *seq_lens, int32_t batch, int32_t next_n,
                                   int64_t max_context, int32_t k, int32_t *topk_idx,
                                   float *scores_opt, void *workspace, size_t workspace_bytes,
                                   void *stream);

/*
 * The indexer's query / head-weight projection from the bf16 hidden state
 * (row f4).  The pages replace forced-fp32 GEMMs on the indexer path by bf16
 * tensor-core GEMMs fed the bf16 hidden state directly ("The Indexer
 * O(max_context) Breakthrough", section "Phase 3: The FP32-to-bf16 GEMM
 * Flip"); they give no weight shapes, so the model width is a parameter:
 *     q[b, h, e] = sum_d x[b, d] * w_q[h * 64 + e, d]   -> bf16 (round to nearest even)
 *     w[b, h]    = sum_d x[b, d] * w_w[h, d]            -> fp32
 * with fp32 accumulation.  Layouts (C-contiguous, 16-byte aligned):
 *     x      bf16 [batch, d_model]     (1 <= batch <= DSA_PROJ_MAX_TOKENS)
 *     w_q    bf16 [32 * 64, d_model]   (d_model a multiple of 64, <= 65536)
 *     w_w    bf16 [32, d_model]
 *     q_out  bf16 [batch, 32, 64]      (the q layout of the indexer entry points)
 *     w_out  fp32 [batch, 32]
 * Workspace: dsa_indexer_qw_proj_workspace_size(batch, d_model) bytes (the
 * 256-byte header with the error word; the partial sums stay on chip).  The
 * reduction over d is split across the CTAs of a thread-block cluster and
 * summed in a fixed order: results are deterministic.  Returns
 * DSA_ERR_INVALID_ARG for a null or misaligned pointer or a shape outside the
 * limits above (the workspace size query then returns 0).
 */
#define DSA_PROJ_MAX_TOKENS 256

DSA_API size_t dsa_indexer_qw_proj_workspace_size(int32_t batch, int64_t d_model);

DSA_API dsa_status_t dsa_indexer_qw_proj(const void *x, const void *w_q, const void *w_w, int32_t batch,
                                 int64_t d_model, void *q_out, float *w_out, void *workspace,
                                 size_t workspace_bytes, void *stream);

/* ---- Sparse multi-head latent attention decode over the top-k entries ----
 *
 * The attention step the indexer feeds ("The Indexer O(max_context)
 * Breakthrough", sections "Phase 1: The MMA Sparse-MLA Decode Kernel" and
 * "Phase 2: Split-K Parallelization"): for each request b and head h,
 *     s_t     = sm_scale * q[b, h, :] . kv_t[:]          (576 dims)
 *     o[b, h] = sum_t softmax_t(s) * kv_t[0:512]
 *     lse[b,h]= log sum_t exp(s_t)
 * over the entries t of topk_idx[b, :] that are used: 0 <= t < ceil(seq_len/4)
 * (-1 padding and positions past the live length are skipped; a position given
 * twice counts twice).  Entry t is kv_cache[page_table[b, t / 64], t % 64, :];
 * the cache is paged exactly like the index keys (64 C4 entries per page).
 * A request with no used entry gets o = 0 and lse = -inf.
 *
 *   q          [batch, 64, 576] bf16, device, 16-byte aligned
 *   kv_cache   [num_pages, 64, 576] bf16, device, 16-byte aligned
 *   page_table [batch, max_context / 256] int32; seq_lens [batch] int32 (tokens)
 *   topk_idx   [batch, k] int32 C4 positions (the indexer's top-k rows), 1 <= k <= 2048
 *   out        [batch, 64, 512] fp32; lse [batch, 64] fp32 (natural log), 16-byte aligned
 *   workspace  >= dsa_sparse_mla_workspace_size(batch, k) bytes, 256-byte aligned,
 *              header zeroed once (dsa_indexer_workspace_init); holds the error word
 *              and the per-split partial outputs (sized for the current device).
 * Asynchronous on `stream`; allocates nothing.  A live page id outside
 * [0, num_pages) sets DSA_DEVERR_BAD_PAGE and that page is not read (another
 * of the request's rows stands in for the entry); results are unspecified
 * while the error word is non-zero.  num_pages above 2^25 - 1 (cache rows
 * past 32-bit coordinates) returns DSA_ERR_UNSUPPORTED. */
#define DSA_MLA_HEADS 64
#define DSA_MLA_DIM 576
#define DSA_MLA_DV 512
#define DSA_MLA_MAX_TOPK 2048

DSA_API size_t dsa_sparse_mla_workspace_size(int32_t batch, int32_t k);

DSA_API dsa_status_t dsa_sparse_mla_decode(const void *q, const void *kv_cache, int64_t num_pages,
                                           const int32_t *page_table, const int32_t *seq_lens, int32_t batch,
                                           int64_t max_context, const int32_t *topk_idx, int32_t k, float sm_scale,
                                           float *out, float *lse, void *workspace, size_t workspace_bytes,
                                           void *stream);


/*
 * Read the sticky device error word into *code (host pointer).  Synchronises
 * `stream` (not capture-safe).  clear != 0 zeroes the word afterwards.
 */
DSA_API dsa_status_t dsa_indexer_get_error(void *workspace, uint32_t *code, int clear, void *stream);

/* Static string for a status code. */
DSA_API const char *dsa_status_string(dsa_status_t status);

/* Text of the last CUDA error this thread saw inside the library ("" if none). */
DSA_API const char *dsa_indexer_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* DSA_INDEXER_H */

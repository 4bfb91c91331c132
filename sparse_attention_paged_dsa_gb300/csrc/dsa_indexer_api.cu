// dsa_indexer_api.cu -- the C ABI (include/dsa_indexer.h): argument checks,
// TMA descriptor set-up, and kernel launches on the caller's stream.
// Nothing here allocates, frees or synchronises during a compute call.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>

#include "../../include/dsa_indexer.h"
#include "api_checks.h"
#include "indexer_kernels.h"

namespace {

using dsa::kHeadDim;
using dsa::kHeads;
using dsa::kPageEntries;

constexpr int64_t kMaxContext = int64_t(1) << 24;  // 16M tokens per request row
constexpr int64_t kMaxPages = (int64_t(1) << 31) - 1;

thread_local char g_last_cuda_error[256] = "";

dsa_status_t cuda_fail(cudaError_t e, const char* where) {
    std::snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "%s: %s (%d)", where, cudaGetErrorString(e),
                  int(e));
    return DSA_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// Key pool [num_pages, 64, 64] bf16 as a 3-D tensor (dim, entry, page); one
// box = one whole page, stored with the 128-byte swizzle the MMA reads.
dsa_status_t make_keys_map(CUtensorMap* map, const void* key_pool, int64_t num_pages) {
    auto enc = encode_tiled();
    if (!enc) return cuda_fail(cudaErrorNotSupported, "cuTensorMapEncodeTiled lookup");
    const cuuint64_t dims[3] = {cuuint64_t(kHeadDim), cuuint64_t(kPageEntries), cuuint64_t(num_pages)};
    const cuuint64_t strides[2] = {cuuint64_t(kHeadDim * 2), cuuint64_t(kPageEntries * kHeadDim * 2)};
    const cuuint32_t box[3] = {cuuint32_t(kHeadDim), cuuint32_t(kPageEntries), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(key_pool), dims, strides,
                           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        std::snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "cuTensorMapEncodeTiled(keys): CUresult %d",
                      int(r));
        return DSA_ERR_CUDA;
    }
    return DSA_OK;
}

// fp8 key cache: codes [num_pages, 64, 64] uint8 as a 3-D tensor (dim, entry,
// page), one box = one page of codes stored with the 64-byte swizzle the
// 8-bit MMA reads.  (The scales are copied by the kernel with cp.async.)
dsa_status_t make_codes_map(CUtensorMap* codes_map, const void* key_codes, int64_t num_pages) {
    auto enc = encode_tiled();
    if (!enc) return cuda_fail(cudaErrorNotSupported, "cuTensorMapEncodeTiled lookup");
    const cuuint64_t cdims[3] = {cuuint64_t(kHeadDim), cuuint64_t(kPageEntries), cuuint64_t(num_pages)};
    const cuuint64_t cstrides[2] = {cuuint64_t(kHeadDim), cuuint64_t(kPageEntries * kHeadDim)};
    const cuuint32_t cbox[3] = {cuuint32_t(kHeadDim), cuuint32_t(kPageEntries), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(codes_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(key_codes), cdims, cstrides,
                     cbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        std::snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "cuTensorMapEncodeTiled(codes): CUresult %d",
                      int(r));
        return DSA_ERR_CUDA;
    }
    return DSA_OK;
}

// Query [batch * tokens * 32, 64] bf16; one box = the tokens x 32 heads of one request.
dsa_status_t make_q_map(CUtensorMap* map, const void* q, int32_t batch, int32_t tokens = 1) {
    auto enc = encode_tiled();
    if (!enc) return cuda_fail(cudaErrorNotSupported, "cuTensorMapEncodeTiled lookup");
    const cuuint64_t dims[2] = {cuuint64_t(kHeadDim), cuuint64_t(batch) * cuuint64_t(tokens) * kHeads};
    const cuuint64_t strides[1] = {cuuint64_t(kHeadDim * 2)};
    const cuuint32_t box[2] = {cuuint32_t(kHeadDim), cuuint32_t(kHeads * tokens)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        std::snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "cuTensorMapEncodeTiled(q): CUresult %d",
                      int(r));
        return DSA_ERR_CUDA;
    }
    return DSA_OK;
}

// Plain (unswizzled) maps for the fp8 kernel's query splitter: q [batch * 32,
// 64] bf16 with one request's 32 heads per box, and w [batch, 32] fp32 with
// one request's weights per box.
dsa_status_t make_plain_q_w_maps(CUtensorMap* q_map, CUtensorMap* w_map, const void* q, const float* w,
                                 int32_t batch) {
    auto enc = encode_tiled();
    if (!enc) return cuda_fail(cudaErrorNotSupported, "cuTensorMapEncodeTiled lookup");
    const cuuint64_t qdims[2] = {cuuint64_t(kHeadDim), cuuint64_t(batch) * kHeads};
    const cuuint64_t qstrides[1] = {cuuint64_t(kHeadDim * 2)};
    const cuuint32_t qbox[2] = {cuuint32_t(kHeadDim), cuuint32_t(kHeads)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(q_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), qdims, qstrides, qbox, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        std::snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "cuTensorMapEncodeTiled(q plain): CUresult %d",
                      int(r));
        return DSA_ERR_CUDA;
    }
    const cuuint64_t wdims[2] = {cuuint64_t(kHeads), cuuint64_t(batch)};
    const cuuint64_t wstrides[1] = {cuuint64_t(kHeads * sizeof(float))};
    const cuuint32_t wbox[2] = {cuuint32_t(kHeads), 1};
    r = enc(w_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(w), wdims, wstrides, wbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        std::snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "cuTensorMapEncodeTiled(w): CUresult %d", int(r));
        return DSA_ERR_CUDA;
    }
    return DSA_OK;
}

// bf16 2-D tensor [rows, cols] (cols contiguous) with a 128-byte-swizzled box of box_rows x 64.
dsa_status_t make_rows_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, uint32_t box_rows,
                           const char* what) {
    auto enc = encode_tiled();
    if (!enc) return cuda_fail(cudaErrorNotSupported, "cuTensorMapEncodeTiled lookup");
    const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        std::snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "cuTensorMapEncodeTiled(%s): CUresult %d", what,
                      int(r));
        return DSA_ERR_CUDA;
    }
    return DSA_OK;
}

constexpr int kProjMaxSplit = 8;  // CTAs per cluster (portable size)
constexpr int kProjQTiles = (DSA_HEADS * DSA_HEAD_DIM) / 128;
constexpr int64_t kProjMaxModel = 65536;

dsa_status_t check_shape(int32_t batch, int64_t max_context) {
    if (batch < 1 || max_context < 1 || max_context % DSA_PAGE_TOKENS != 0) return DSA_ERR_INVALID_ARG;
    if (batch > DSA_MAX_BATCH || max_context > kMaxContext) return DSA_ERR_UNSUPPORTED;
    return DSA_OK;
}

dsa_status_t check_workspace(const void* ws, size_t bytes, size_t need) {
    if (ws == nullptr || !aligned(ws, 256) || bytes < need) return DSA_ERR_WORKSPACE;
    return DSA_OK;
}

dsa_status_t check_score_inputs(const void* q, const float* w, const void* key_pool, int64_t num_pages,
                                const int32_t* page_table, const int32_t* seq_lens) {
    if (!q || !w || !key_pool || !page_table || !seq_lens) return DSA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(w, 16) || !aligned(key_pool, 16) || !aligned(page_table, 4) ||
        !aligned(seq_lens, 4))
        return DSA_ERR_INVALID_ARG;
    if (num_pages < 1 || num_pages > kMaxPages) return DSA_ERR_INVALID_ARG;
    return DSA_OK;
}

dsa::ScoresParams score_params(const float* w, int64_t num_pages, const int32_t* page_table,
                               const int32_t* seq_lens, int32_t batch, int64_t max_context, float* out,
                               int fill_dead, void* workspace, int32_t tokens = 1) {
    dsa::ScoresParams p{};
    p.page_table = page_table;
    p.seq_lens = seq_lens;
    p.w = w;
    p.out = out;
    p.err = static_cast<uint32_t*>(workspace);
    p.num_pages = num_pages;
    p.max_context = max_context;
    p.row_width = max_context / 4;
    p.table_width = int32_t(max_context / DSA_PAGE_TOKENS);
    p.batch = batch;
    p.fill_dead = fill_dead;
    p.tokens = tokens;
    return p;
}

dsa_status_t run_scores(const void* q, const float* w, const void* key_pool, int64_t num_pages,
                        const int32_t* page_table, const int32_t* seq_lens, int32_t batch, int64_t max_context,
                        float* out, int fill_dead, void* workspace, cudaStream_t stream, int32_t tokens = 1) {
    CUtensorMap keys_map, q_map;
    dsa_status_t st = make_keys_map(&keys_map, key_pool, num_pages);
    if (st != DSA_OK) return st;
    st = make_q_map(&q_map, q, batch, tokens);
    if (st != DSA_OK) return st;
    const dsa::ScoresParams p =
        score_params(w, num_pages, page_table, seq_lens, batch, max_context, out, fill_dead, workspace, tokens);
    const cudaError_t e = dsa::launch_scores(keys_map, q_map, p, stream);
    return e == cudaSuccess ? DSA_OK : cuda_fail(e, "scores kernel launch");
}

dsa_status_t run_scores_fp8(const void* q, const float* w, const void* key_codes, const float* key_scales,
                            int64_t num_pages, const int32_t* page_table, const int32_t* seq_lens, int32_t batch,
                            int64_t max_context, float* out, int fill_dead, void* workspace, cudaStream_t stream) {
    CUtensorMap codes_map, q_map, w_map;
    dsa_status_t st = make_codes_map(&codes_map, key_codes, num_pages);
    if (st != DSA_OK) return st;
    st = make_plain_q_w_maps(&q_map, &w_map, q, w, batch);
    if (st != DSA_OK) return st;
    dsa::ScoresParams p =
        score_params(w, num_pages, page_table, seq_lens, batch, max_context, out, fill_dead, workspace);
    p.key_scales = key_scales;
    const cudaError_t e = dsa::launch_scores_fp8(codes_map, q_map, w_map, p, stream);
    return e == cudaSuccess ? DSA_OK : cuda_fail(e, "fp8 scores kernel launch");
}

dsa_status_t run_topk(const float* scores, const int32_t* seq_lens, int32_t batch, int64_t max_context, int32_t k,
                      int32_t* topk_idx, void* workspace, cudaStream_t stream, int32_t tokens = 1) {
    dsa::TopkParams p{};
    p.scores = scores;
    p.seq_lens = seq_lens;
    p.out = topk_idx;
    p.err = static_cast<uint32_t*>(workspace);
    p.max_context = max_context;
    p.row_width = max_context / 4;
    p.batch = batch;
    p.k = k;
    p.tokens = tokens;
    const cudaError_t e = dsa::launch_topk(p, stream);
    return e == cudaSuccess ? DSA_OK : cuda_fail(e, "top-k kernel launch");
}

// Workspace of a fused call over `nrows` score rows: the header, plus the
// live-score slots when no scores row is given.
size_t fused_workspace_bytes(int64_t nrows, int64_t max_context, bool with_slots) {
    return dsa::kWorkspaceHeaderBytes + (with_slots ? size_t(nrows) * size_t(max_context / 4) * sizeof(float) : 0);
}

float* fused_rows(void* workspace, float* scores_opt) {
    return scores_opt ? scores_opt
                      : reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + dsa::kWorkspaceHeaderBytes);
}

// Splits of a request's top-k row across CTAs (one CTA per SM): enough to fill
// the current device once, at most one per 64-entry block and kMlaMaxSplits.
int mla_splits(int32_t batch, int32_t k) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                   cudaSuccess)
        sms = 148;
    const int blocks = (k + 63) / 64;
    int s = sms / batch;
    if (s > blocks) s = blocks;
    if (s > dsa::kMlaMaxSplits) s = dsa::kMlaMaxSplits;
    return s < 1 ? 1 : s;
}
size_t mla_partial_floats(int32_t batch, int splits) {
    return splits > 1 ? size_t(batch) * size_t(splits) * dsa::kMlaHeads * (dsa::kMlaDv + 1) : 0;
}

}  // namespace

namespace dsa {

dsa_status_t check_fused_args(const void* q, const float* w, const void* key_pool, int64_t num_pages,
                              const int32_t* page_table, const int32_t* seq_lens, int32_t batch,
                              int64_t max_context, int32_t k, const int32_t* topk_idx, const float* scores_opt) {
    dsa_status_t st = check_shape(batch, max_context);
    if (st != DSA_OK) return st;
    st = check_score_inputs(q, w, key_pool, num_pages, page_table, seq_lens);
    if (st != DSA_OK) return st;
    if (!topk_idx || !aligned(topk_idx, 4)) return DSA_ERR_INVALID_ARG;
    if (scores_opt && !aligned(scores_opt, 16)) return DSA_ERR_INVALID_ARG;
    if (k < 1 || int64_t(k) > max_context / 4) return DSA_ERR_INVALID_ARG;
    return DSA_OK;
}

}  // namespace dsa

extern "C" {

size_t dsa_indexer_workspace_size(int32_t batch, int64_t max_context, int32_t k) {
    (void)k;
    if (check_shape(batch, max_context) != DSA_OK) return 0;
    return fused_workspace_bytes(batch, max_context, true);
}

dsa_status_t dsa_indexer_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
    if (check_workspace(workspace, workspace_bytes, dsa::kWorkspaceHeaderBytes) != DSA_OK) return DSA_ERR_WORKSPACE;
    const cudaError_t e =
        cudaMemsetAsync(workspace, 0, dsa::kWorkspaceHeaderBytes, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DSA_OK : cuda_fail(e, "workspace init");
}

dsa_status_t dsa_indexer_scores(const void* q, const float* w, const void* key_pool, int64_t num_pages,
                                const int32_t* page_table, const int32_t* seq_lens, int32_t batch,
                                int64_t max_context, float* scores, void* workspace, size_t workspace_bytes,
                                void* stream) {
    dsa_status_t st = check_shape(batch, max_context);
    if (st != DSA_OK) return st;
    st = check_score_inputs(q, w, key_pool, num_pages, page_table, seq_lens);
    if (st != DSA_OK) return st;
    if (!scores || !aligned(scores, 16)) return DSA_ERR_INVALID_ARG;
    st = check_workspace(workspace, workspace_bytes, dsa::kWorkspaceHeaderBytes);
    if (st != DSA_OK) return st;
    return run_scores(q, w, key_pool, num_pages, page_table, seq_lens, batch, max_context, scores, 1, workspace,
                      static_cast<cudaStream_t>(stream));
}

dsa_status_t dsa_indexer_topk(const float* scores, const int32_t* seq_lens, int32_t batch, int64_t max_context,
                              int32_t k, int32_t* topk_idx, void* workspace, size_t workspace_bytes,
                              void* stream) {
    dsa_status_t st = check_shape(batch, max_context);
    if (st != DSA_OK) return st;
    if (!scores || !seq_lens || !topk_idx || !aligned(scores, 16) || !aligned(seq_lens, 4) || !aligned(topk_idx, 4))
        return DSA_ERR_INVALID_ARG;
    if (k < 1 || int64_t(k) > max_context / 4) return DSA_ERR_INVALID_ARG;
    st = check_workspace(workspace, workspace_bytes, dsa::kWorkspaceHeaderBytes);
    if (st != DSA_OK) return st;
    return run_topk(scores, seq_lens, batch, max_context, k, topk_idx, workspace, static_cast<cudaStream_t>(stream));
}

dsa_status_t dsa_indexer_fused(const void* q, const float* w, const void* key_pool, int64_t num_pages,
                               const int32_t* page_table, const int32_t* seq_lens, int32_t batch,
                               int64_t max_context, int32_t k, int32_t* topk_idx, float* scores_opt,
                               void* workspace, size_t workspace_bytes, void* stream) {
    dsa_status_t st = dsa::check_fused_args(q, w, key_pool, num_pages, page_table, seq_lens, batch, max_context, k,
                                            topk_idx, scores_opt);
    if (st != DSA_OK) return st;
    st = check_workspace(workspace, workspace_bytes, fused_workspace_bytes(batch, max_context, !scores_opt));
    if (st != DSA_OK) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    float* rows = fused_rows(workspace, scores_opt);
    st = run_scores(q, w, key_pool, num_pages, page_table, seq_lens, batch, max_context, rows, scores_opt ? 1 : 0,
                    workspace, s);
    if (st != DSA_OK) return st;
    return run_topk(rows, seq_lens, batch, max_context, k, topk_idx, workspace, s);
}

dsa_status_t dsa_indexer_scores_fp8(const void* q, const float* w, const void* key_codes, const float* key_scales,
                                    int64_t num_pages, const int32_t* page_table, const int32_t* seq_lens,
                                    int32_t batch, int64_t max_context, float* scores, void* workspace,
                                    size_t workspace_bytes, void* stream) {
    dsa_status_t st = check_shape(batch, max_context);
    if (st != DSA_OK) return st;
    st = check_score_inputs(q, w, key_codes, num_pages, page_table, seq_lens);
    if (st != DSA_OK) return st;
    if (!key_scales || !aligned(key_scales, 16)) return DSA_ERR_INVALID_ARG;
    if (!scores || !aligned(scores, 16)) return DSA_ERR_INVALID_ARG;
    st = check_workspace(workspace, workspace_bytes, dsa::kWorkspaceHeaderBytes);
    if (st != DSA_OK) return st;
    return run_scores_fp8(q, w, key_codes, key_scales, num_pages, page_table, seq_lens, batch, max_context, scores, 1,
                          workspace, static_cast<cudaStream_t>(stream));
}

dsa_status_t dsa_indexer_fused_fp8(const void* q, const float* w, const void* key_codes, const float* key_scales,
                                   int64_t num_pages, const int32_t* page_table, const int32_t* seq_lens,
                                   int32_t batch, int64_t max_context, int32_t k, int32_t* topk_idx,
                                   float* scores_opt, void* workspace, size_t workspace_bytes, void* stream) {
    dsa_status_t st = check_shape(batch, max_context);
    if (st != DSA_OK) return st;
    st = check_score_inputs(q, w, key_codes, num_pages, page_table, seq_lens);
    if (st != DSA_OK) return st;
    if (!key_scales || !aligned(key_scales, 16)) return DSA_ERR_INVALID_ARG;
    if (!topk_idx || !aligned(topk_idx, 4)) return DSA_ERR_INVALID_ARG;
    if (scores_opt && !aligned(scores_opt, 16)) return DSA_ERR_INVALID_ARG;
    if (k < 1 || int64_t(k) > max_context / 4) return DSA_ERR_INVALID_ARG;
    st = check_workspace(workspace, workspace_bytes, fused_workspace_bytes(batch, max_context, !scores_opt));
    if (st != DSA_OK) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    float* rows = fused_rows(workspace, scores_opt);
    st = run_scores_fp8(q, w, key_codes, key_scales, num_pages, page_table, seq_lens, batch, max_context, rows,
                        scores_opt ? 1 : 0, workspace, s);
    if (st != DSA_OK) return st;
    return run_topk(rows, seq_lens, batch, max_context, k, topk_idx, workspace, s);
}

size_t dsa_indexer_workspace_size_mtp(int32_t batch, int32_t next_n, int64_t max_context, int32_t k) {
    (void)k;
    if (check_shape(batch, max_context) != DSA_OK || next_n < 1 || next_n > DSA_MAX_NEXT_N) return 0;
    return fused_workspace_bytes(int64_t(batch) * next_n, max_context, true);
}

dsa_status_t dsa_indexer_scores_mtp(const void* q, const float* w, const void* key_pool, int64_t num_pages,
                                    const int32_t* page_table, const int32_t* seq_lens, int32_t batch,
                                    int32_t next_n, int64_t max_context, float* scores, void* workspace,
                                    size_t workspace_bytes, void* stream) {
    dsa_status_t st = check_shape(batch, max_context);
    if (st != DSA_OK) return st;
    if (next_n < 1 || next_n > DSA_MAX_NEXT_N) return DSA_ERR_INVALID_ARG;
    st = check_score_inputs(q, w, key_pool, num_pages, page_table, seq_lens);
    if (st != DSA_OK) return st;
    if (!scores || !aligned(scores, 16)) return DSA_ERR_INVALID_ARG;
    st = check_workspace(workspace, workspace_bytes, dsa::kWorkspaceHeaderBytes);
    if (st != DSA_OK) return st;
    return run_scores(q, w, key_pool, num_pages, page_table, seq_lens, batch, max_context, scores, 1, workspace,
                      static_cast<cudaStream_t>(stream), next_n);
}

dsa_status_t dsa_indexer_topk_mtp(const float* scores, const int32_t* seq_lens, int32_t batch, int32_t next_n,
                                  int64_t max_context, int32_t k, int32_t* topk_idx, void* workspace,
                                  size_t workspace_bytes, void* stream) {
    dsa_status_t st = check_shape(batch, max_context);
    if (st != DSA_OK) return st;
    if (next_n < 1 || next_n > DSA_MAX_NEXT_N) return DSA_ERR_INVALID_ARG;
    if (!scores || !seq_lens || !topk_idx || !aligned(scores, 16) || !aligned(seq_lens, 4) || !aligned(topk_idx, 4))
        return DSA_ERR_INVALID_ARG;
    if (k < 1 || int64_t(k) > max_context / 4) return DSA_ERR_INVALID_ARG;
    st = check_workspace(workspace, workspace_bytes, dsa::kWorkspaceHeaderBytes);
    if (st != DSA_OK) return st;
    return run_topk(scores, seq_lens, batch, max_context, k, topk_idx, workspace, static_cast<cudaStream_t>(stream),
                    next_n);
}

dsa_status_t dsa_indexer_fused_mtp(const void* q, const float* w, const void* key_pool, int64_t num_pages,
                                   const int32_t* page_table, const int32_t* seq_lens, int32_t batch,
                                   int32_t next_n, int64_t max_context, int32_t k, int32_t* topk_idx,
                                   float* scores_opt, void* workspace, size_t workspace_bytes, void* stream) {
    dsa_status_t st = check_shape(batch, max_context);
    if (st != DSA_OK) return st;
    if (next_n < 1 || next_n > DSA_MAX_NEXT_N) return DSA_ERR_INVALID_ARG;
    st = check_score_inputs(q, w, key_pool, num_pages, page_table, seq_lens);
    if (st != DSA_OK) return st;
    if (!topk_idx || !aligned(topk_idx, 4)) return DSA_ERR_INVALID_ARG;
    if (scores_opt && !aligned(scores_opt, 16)) return DSA_ERR_INVALID_ARG;
    if (k < 1 || int64_t(k) > max_context / 4) return DSA_ERR_INVALID_ARG;
    st = check_workspace(workspace, workspace_bytes,
                         fused_workspace_bytes(int64_t(batch) * next_n, max_context, !scores_opt));
    if (st != DSA_OK) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    float* rows = fused_rows(workspace, scores_opt);
    st = run_scores(q, w, key_pool, num_pages, page_table, seq_lens, batch, max_context, rows, scores_opt ? 1 : 0,
                    workspace, s, next_n);
    if (st != DSA_OK) return st;
    return run_topk(rows, seq_lens, batch, max_context, k, topk_idx, workspace, s, next_n);
}

size_t dsa_indexer_qw_proj_workspace_size(int32_t batch, int64_t d_model) {
    if (batch < 1 || batch > DSA_PROJ_MAX_TOKENS || d_model < 64 || d_model % 64 != 0 || d_model > kProjMaxModel)
        return 0;
    return dsa::kWorkspaceHeaderBytes;  // the error word only: partial sums stay on chip
}

dsa_status_t dsa_indexer_qw_proj(const void* x, const void* w_q, const void* w_w, int32_t batch, int64_t d_model,
                                 void* q_out, float* w_out, void* workspace, size_t workspace_bytes,
                                 void* stream) {
    const size_t need = dsa_indexer_qw_proj_workspace_size(batch, d_model);
    if (need == 0) return DSA_ERR_INVALID_ARG;
    if (!x || !w_q || !w_w || !q_out || !w_out) return DSA_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w_q, 16) || !aligned(w_w, 16) || !aligned(q_out, 4) || !aligned(w_out, 4))
        return DSA_ERR_INVALID_ARG;
    dsa_status_t st = check_workspace(workspace, workspace_bytes, need);
    if (st != DSA_OK) return st;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    const int atoms = int(d_model / 64);
    int k_split = sms / (kProjQTiles + 1);  // about one weight-streaming CTA per SM
    k_split = k_split < 1 ? 1 : (k_split > kProjMaxSplit ? kProjMaxSplit : k_split);
    k_split = k_split > atoms ? atoms : k_split;
    const int bp = dsa::proj_batch_pad(batch);
    CUtensorMap wq_map, ww_map, x_map;
    st = make_rows_map(&wq_map, w_q, kProjQTiles * 128, d_model, 128, "w_q");
    if (st != DSA_OK) return st;
    st = make_rows_map(&ww_map, w_w, DSA_HEADS, d_model, 128, "w_w");
    if (st != DSA_OK) return st;
    st = make_rows_map(&x_map, x, batch, d_model, uint32_t(bp), "x");
    if (st != DSA_OK) return st;
    dsa::ProjParams p{};
    p.q_out = static_cast<__nv_bfloat16_raw*>(q_out);
    p.w_out = w_out;
    p.err = static_cast<uint32_t*>(workspace);
    p.batch = batch;
    p.batch_pad = bp;
    p.d_model = int32_t(d_model);
    p.q_tiles = kProjQTiles;
    p.k_split = k_split;
    e = dsa::launch_proj(wq_map, ww_map, x_map, p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DSA_OK : cuda_fail(e, "projection kernel launch");
}

dsa_status_t dsa_indexer_get_error(void* workspace, uint32_t* code, int clear, void* stream) {
    if (!workspace || !code || !aligned(workspace, 256)) return DSA_ERR_INVALID_ARG;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && clear) e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "read error word");
    *code = v;
    return DSA_OK;
}

const char* dsa_status_string(dsa_status_t status) {
    switch (status) {
        case DSA_OK: return "ok";
        case DSA_ERR_INVALID_ARG: return "invalid argument";
        case DSA_ERR_UNSUPPORTED: return "unsupported shape";
        case DSA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case DSA_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

const char* dsa_indexer_last_cuda_error(void) { return g_last_cuda_error; }

size_t dsa_sparse_mla_workspace_size(int32_t batch, int32_t k) {
    if (batch < 1 || batch > DSA_MAX_BATCH || k < 1 || k > DSA_MLA_MAX_TOPK) return 0;
    return dsa::kWorkspaceHeaderBytes + mla_partial_floats(batch, mla_splits(batch, k)) * sizeof(float);
}
dsa_status_t dsa_sparse_mla_decode(const void* q, const void* kv_cache, int64_t num_pages,
                                   const int32_t* page_table, const int32_t* seq_lens, int32_t batch,
                                   int64_t max_context, const int32_t* topk_idx, int32_t k, float sm_scale,
                                   float* out, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
    dsa_status_t st = check_shape(batch, max_context);
    if (st != DSA_OK) return st;
    if (!q || !kv_cache || !page_table || !seq_lens || !topk_idx || !out || !lse) return DSA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(page_table, 4) || !aligned(seq_lens, 4) ||
        !aligned(topk_idx, 4) || !aligned(out, 16) || !aligned(lse, 16))
        return DSA_ERR_INVALID_ARG;
    if (num_pages < 1 || num_pages > kMaxPages) return DSA_ERR_INVALID_ARG;
    if (k < 1 || k > DSA_MLA_MAX_TOPK || !std::isfinite(sm_scale))
        return DSA_ERR_INVALID_ARG;
    const int splits = mla_splits(batch, k);
    st = check_workspace(workspace, workspace_bytes,
                         dsa::kWorkspaceHeaderBytes + mla_partial_floats(batch, splits) * sizeof(float));
    if (st != DSA_OK) return st;
    // The row gathers address cache rows with 32-bit coordinates.
    if (num_pages > (int64_t(1) << 31) / dsa::kPageEntries - 1) return DSA_ERR_UNSUPPORTED;
    CUtensorMap q_map, kv_map;
    st = make_rows_map(&q_map, q, int64_t(batch) * DSA_MLA_HEADS, DSA_MLA_DIM, 64, "mla q");
    if (st != DSA_OK) return st;
    st = make_rows_map(&kv_map, kv_cache, num_pages * dsa::kPageEntries, DSA_MLA_DIM, 1, "mla kv");
    if (st != DSA_OK) return st;
    dsa::MlaParams p{};
    p.kv = static_cast<const uint8_t*>(kv_cache);
    p.page_table = page_table;
    p.seq_lens = seq_lens;
    p.topk = topk_idx;
    p.out = out;
    p.lse = lse;
    float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + dsa::kWorkspaceHeaderBytes);
    p.o_part = splits > 1 ? part : nullptr;
    p.lse_part = splits > 1 ? part + size_t(batch) * splits * dsa::kMlaHeads * dsa::kMlaDv : nullptr;
    p.err = static_cast<uint32_t*>(workspace);
    p.num_pages = num_pages;
    p.max_context = max_context;
    p.table_width = int32_t(max_context / DSA_PAGE_TOKENS);
    p.batch = batch;
    p.k = k;
    p.splits = splits;
    p.sm_scale_log2 = sm_scale * 1.4426950408889634f;
    const cudaError_t e = dsa::launch_mla(q_map, kv_map, p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DSA_OK : cuda_fail(e, "sparse MLA decode launch");
}
}  // extern "C"

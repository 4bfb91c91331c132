// indexer_kernels.h -- host-side launch interface of the indexer kernels
// (internal to the library; the public ABI is include/dsa_indexer.h).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <mutex>

namespace dsa {

constexpr int kMaxDevices = 64;

// A kernel's dynamic shared-memory limit, set once per device.  Safe when
// several host threads make their first calls at the same time (call_once
// per device); every later call returns the first call's result.  One
// static instance per kernel, used on the launching thread's current device.
struct SmemLimitOnce {
    std::once_flag flag[kMaxDevices];
    cudaError_t result[kMaxDevices] = {};

    template <typename Kernel>
    cudaError_t apply(int dev, Kernel* kernel, int bytes) {
        if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
        std::call_once(flag[dev], [&] {
            result[dev] = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        });
        return result[dev];
    }
};

// Fixed problem geometry.
constexpr int kHeads = 32;
constexpr int kHeadDim = 64;
constexpr int kPageEntries = 64;                          // C4 keys per page
constexpr int kPageBytes = kPageEntries * kHeadDim * 2;   // 8 KiB of bf16
constexpr int kPageCodeBytes = kPageEntries * kHeadDim;   // 4 KiB of e4m3 codes (fp8 cache)
constexpr int kPageScaleBytes = kPageEntries * 4;         // 256 B of fp32 key scales (fp8 cache)
constexpr int kQRowBytes = kHeads * kHeadDim * 2;         // 4 KiB of bf16
constexpr int kUnitPositions = 2 * kPageEntries;          // one work unit = 2 pages = 128 keys
constexpr int kMaxBatch = 1024;
constexpr size_t kWorkspaceHeaderBytes = 256;

// Device error bits (same values as DSA_DEVERR_* in the public header).
constexpr uint32_t kErrSeqLenClamped = 0x1u;
constexpr uint32_t kErrBadPage = 0x2u;
constexpr uint32_t kErrWaitTimeout = 0x4u;

struct ScoresParams {
    const int32_t* page_table;  // [batch, table_width]
    const int32_t* seq_lens;    // [batch]
    const float* w;             // [batch, 32]
    float* out;                 // [batch, row_width]
    uint32_t* err;              // device error word
    int64_t num_pages;
    int64_t max_context;        // tokens
    int64_t row_width;          // max_context / 4
    int32_t table_width;        // max_context / 256
    int32_t batch;
    int32_t fill_dead;          // 1: write -inf from the live extent to the row end
    int32_t tokens;             // query tokens per request (q [batch, tokens, 32, 64], rows batch x tokens)
    const float* key_scales;    // [num_pages, 64] per-key scales of the fp8 cache (fp8 kernel only)
};

struct TopkParams {
    const float* scores;  // [batch x tokens, row_width]
    const int32_t* seq_lens;  // [batch]
    int32_t* out;         // [batch x tokens, k]
    uint32_t* err;
    int64_t max_context;
    int64_t row_width;
    int32_t batch;
    int32_t k;
    int32_t tokens;       // query tokens per request: row r is token r % tokens of request r / tokens
};

// Scores kernel: persistent, one CTA per SM, TMA page gather + tcgen05 QK.
cudaError_t launch_scores(const CUtensorMap& keys_map, const CUtensorMap& q_map, const ScoresParams& p,
                          cudaStream_t stream);

// Scores kernel on the fp8 key cache (e4m3 codes + per-key fp32 scale in
// p.key_scales): the codes feed tcgen05.mma kind::f8f6f4 directly, against
// each query split into two e4m3 terms in the kernel.  qraw_map: bf16
// queries, unswizzled; w_map: head weights.
cudaError_t launch_scores_fp8(const CUtensorMap& codes_map, const CUtensorMap& qraw_map, const CUtensorMap& w_map,
                              const ScoresParams& p, cudaStream_t stream);

// Top-k kernel: one CTA per request row, radix select over live positions.
cudaError_t launch_topk(const TopkParams& p, cudaStream_t stream);

// Query / head-weight projection (split-K weight stream over a thread-block
// cluster, deterministic reduction through distributed shared memory).
struct ProjParams {
    __nv_bfloat16_raw* q_out; // [batch, 32, 64] bf16
    float* w_out;             // [batch, 32]
    uint32_t* err;            // device error word
    int32_t batch;
    int32_t batch_pad;        // tokens padded to the MMA's N: 32, 64, 128 or 256
    int32_t d_model;          // multiple of 64
    int32_t q_tiles;          // 2048 / 128
    int32_t k_split;          // CTAs along d (one cluster), 1..8, <= d_model / 64
};
int proj_batch_pad(int batch);
cudaError_t launch_proj(const CUtensorMap& wq_map, const CUtensorMap& ww_map, const CUtensorMap& x_map,
                        const ProjParams& p, cudaStream_t stream);

// Sparse multi-head latent attention decode over the top-k entries: 64 heads,
// 576-wide bf16 cache entries paged like the index keys, value = first 512 dims.
constexpr int kMlaHeads = 64;
constexpr int kMlaDim = 576;
constexpr int kMlaDv = 512;
constexpr int kMlaMaxTopk = 2048;
constexpr int kMlaMaxSplits = 32;
struct MlaParams {
    const uint8_t* kv;         // [num_pages, 64, 576] bf16
    const int32_t* page_table; // [batch, table_width]
    const int32_t* seq_lens;   // [batch] tokens
    const int32_t* topk;       // [batch, k] C4 positions, -1 = unused
    float* out;                // [batch, 64, 512]
    float* lse;                // [batch, 64]
    float* o_part;             // [batch, splits, 64, 512] (splits > 1)
    float* lse_part;           // [batch, splits, 64]
    uint32_t* err;             // device error word
    int64_t num_pages;
    int64_t max_context;
    int32_t table_width;
    int32_t batch;
    int32_t k;
    int32_t splits;            // CTAs per request, 1..32
    float sm_scale_log2;       // sm_scale * log2(e)
};
size_t mla_smem_bytes();
// Decode kernel (grid splits x batch) and, for splits > 1, the log-sum-exp merge.
// q_map: q [batch * 64, 576] bf16, 128-byte-swizzled boxes of 64 x 64.
// kv_map: the cache as [num_pages * 64, 576] bf16 rows, 128-byte-swizzled boxes of
// one row x 64 (the row gathers' map).
cudaError_t launch_mla(const CUtensorMap& q_map, const CUtensorMap& kv_map, const MlaParams& p, cudaStream_t stream);

}  // namespace dsa

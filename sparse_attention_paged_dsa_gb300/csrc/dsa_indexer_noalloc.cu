// dsa_indexer_noalloc.cu -- dsa_indexer_fused_noalloc: the fused indexer
// (scores + top-k, no full-width row) for callers that cannot hand the
// library a workspace, and dsa_indexer_noalloc_get_error, which reads its
// device error word.
//
// Who needs this.  Some hosts of this library cannot call cudaMalloc or any
// allocator on the path that runs the indexer: a serving engine that has
// carved all of HBM into its own KV-cache and activation pools and passes
// kernels only the tensors they read and write; plugin and custom-op
// interfaces that give a kernel its inputs and outputs but no scratch
// buffer; and code that must not call cudaMalloc there because it can
// synchronise the device and stall the other decode streams.  For them the
// scratch the fused path needs (the error word and the live-score slots) is
// a fixed device array owned by this library.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds kScratchBytes of it until the process exits.  In host code
// its name is only a host-side stand-in, so its device address is taken with
// cudaGetSymbolAddress once per device, with that device current, on the
// first call made on that device.  That first call should therefore come
// before any stream capture.  Every call shares the one array per device:
// calls whose work overlaps on the GPU (different streams, no ordering)
// race on it.  The live-score slots need no clearing (each slot read is
// written first in the same call).  The error word is sticky, as in a
// caller's workspace: dsa_indexer_noalloc_get_error reads (and may clear) it.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/dsa_indexer.h"
#include "api_checks.h"
#include "indexer_kernels.h"

namespace {

// 256-byte header + 16 MiB of live-score slots: batch x max_context / 4 fp32
// values must fit, e.g. 64 requests at 256K tokens or 128 at 128K.
constexpr size_t kScratchBytes = dsa::kWorkspaceHeaderBytes + (size_t(16) << 20);

__device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[dsa::kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up once).
dsa_status_t scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= dsa::kMaxDevices) return DSA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return DSA_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return DSA_OK;
}

}  // namespace

extern "C" DSA_API dsa_status_t dsa_indexer_fused_noalloc(const void* q, const float* w, const void* key_pool,
                                                          int64_t num_pages, const int32_t* page_table,
                                                          const int32_t* seq_lens, int32_t batch,
                                                          int64_t max_context, int32_t k, int32_t* topk_idx,
                                                          void* stream) {
    // The same checks as dsa_indexer_fused, before anything touches the scratch.
    dsa_status_t st = dsa::check_fused_args(q, w, key_pool, num_pages, page_table, seq_lens, batch, max_context, k,
                                            topk_idx, nullptr);
    if (st != DSA_OK) return st;
    if (dsa_indexer_workspace_size(batch, max_context, k) > kScratchBytes) return DSA_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != DSA_OK) return st;
    return dsa_indexer_fused(q, w, key_pool, num_pages, page_table, seq_lens, batch, max_context, k, topk_idx,
                             nullptr, scratch, kScratchBytes, stream);
}

extern "C" DSA_API dsa_status_t dsa_indexer_noalloc_get_error(uint32_t* code, int clear, void* stream) {
    if (!code) return DSA_ERR_INVALID_ARG;
    void* scratch = nullptr;
    const dsa_status_t st = scratch_address(&scratch);
    if (st != DSA_OK) return st;
    return dsa_indexer_get_error(scratch, code, clear, stream);
}

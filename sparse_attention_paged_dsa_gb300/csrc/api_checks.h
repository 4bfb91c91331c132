// api_checks.h -- host-side argument checks shared by entry points of the
// C ABI (internal to the library).
#pragma once

#include <cstdint>

#include "../../include/dsa_indexer.h"

namespace dsa {

// Every check dsa_indexer_fused makes before it looks at its workspace: shape
// (DSA_ERR_INVALID_ARG, or DSA_ERR_UNSUPPORTED past the size limits), inputs
// (null, misaligned, pool size), output, optional scores row and k.
dsa_status_t check_fused_args(const void* q, const float* w, const void* key_pool, int64_t num_pages,
                              const int32_t* page_table, const int32_t* seq_lens, int32_t batch,
                              int64_t max_context, int32_t k, const int32_t* topk_idx, const float* scores_opt);

}  // namespace dsa

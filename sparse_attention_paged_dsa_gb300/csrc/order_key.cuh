// order_key.cuh -- the order-preserving 32-bit key of an fp32 score, shared by
// the top-k kernels and by the scores epilogues that histogram their scores.
#pragma once

#include <cstdint>

namespace dsa {

// a > b as fp32 values iff order_key(a) > order_key(b).  -0 is first mapped to
// +0: the two are equal in fp32 order, so they must tie (and a tie goes to
// the lower position).
__device__ __forceinline__ uint32_t order_key(float x) {
    uint32_t u = __float_as_uint(x);
    u = u == 0x80000000u ? 0u : u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Bin of a key in the first-level histogram: its top 11 bits.
__device__ __forceinline__ uint32_t order_bin(uint32_t key) { return key >> 21; }

}  // namespace dsa

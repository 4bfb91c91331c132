// topk_kernel.cu -- per-request top-k over the live part of a scores row.
//
// The pages feed a top-k over the full-width logits row to sparse attention
// and name that top-k, being O(max_context), as the remaining cost of the
// indexer ("The O(Actual) Indexer: Validating 128K Context at 500 tok/s on
// Blackwell", sections "The Benchmark Results" and "The Reasoning Process").
// This kernel only ever looks at positions t < n_b, so its cost is
// O(live positions), and it does nothing but write indices when n_b <= k.
//
// Selection (exact, deterministic): scores are mapped to order-preserving
// 32-bit keys; three histogram passes (11 + 11 + 10 bits) find the key T of
// the k-th largest score and how many of the keys equal to T are taken; a
// final ordered pass keeps every key > T and the first ones equal to T in
// position order (equal scores: lower position wins), writing positions in
// ascending order.  One 1024-thread CTA per request; rows of up to 49152 live
// positions are held in shared memory between passes, longer rows are
// re-read from global memory (L2) on each pass.
#include <cuda_runtime.h>

#include <cstdint>

#include "indexer_kernels.h"

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kCacheCap = 49152;  // keys held in shared memory (192 KiB)

__device__ __forceinline__ uint32_t order_key(float x) {
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct TopkSmem {
    uint32_t hist[2048];
    uint32_t warp_tot[kWarps];
    uint32_t warp_gt[kWarps];
    uint32_t warp_eq[kWarps];
    uint32_t result[2];
};

// Find the bin holding the kk-th largest key: result[0] = bin,
// result[1] = how many keys of that bin are still to be taken.  Ends with a
// barrier, so result[] is visible to all threads on return.
template <int kBins>
__device__ __forceinline__ void select_bin(TopkSmem& sm, uint32_t kk) {
    constexpr int per = kBins / kThreads;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t h[per];
    uint32_t v = 0;
#pragma unroll
    for (int i = 0; i < per; ++i) {
        h[i] = sm.hist[tid * per + i];
        v += h[i];
    }
    uint32_t incl = v;  // sum over this and higher lanes (higher bins)
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += x;
    }
    if (lane == 0) sm.warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const uint32_t t = sm.warp_tot[lane];
        uint32_t s = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t x = __shfl_down_sync(0xffffffffu, s, o);
            if (lane + o < 32) s += x;
        }
        sm.warp_tot[lane] = s - t;  // keys in higher warps' bins
    }
    __syncthreads();
    uint32_t above = sm.warp_tot[warp] + incl - v;  // keys in bins above this thread's bins
#pragma unroll
    for (int i = per - 1; i >= 0; --i) {
        if (above < kk && above + h[i] >= kk) {
            sm.result[0] = uint32_t(tid * per + i);
            sm.result[1] = kk - above;
        }
        above += h[i];
    }
    __syncthreads();
}

template <bool kCached>
__device__ __forceinline__ uint32_t key_at(const uint32_t* cache, const float* row, int t) {
    if constexpr (kCached)
        return cache[t];
    else
        return order_key(__ldcg(row + t));
}

template <bool kCached>
__device__ void select_row(TopkSmem& sm, uint32_t* cache, const float* row, int n, int k, int32_t* out) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // Pass 1: top 11 bits of every live key (and fill the cache).
    for (int i = tid; i < 2048; i += kThreads) sm.hist[i] = 0;
    __syncthreads();
    for (int t = tid; t < n; t += kThreads) {
        const uint32_t key = order_key(__ldcg(row + t));
        if constexpr (kCached) cache[t] = key;
        atomicAdd(&sm.hist[key >> 21], 1u);
    }
    __syncthreads();
    select_bin<2048>(sm, uint32_t(k));
    const uint32_t bin1 = sm.result[0];
    uint32_t kk = sm.result[1];

    // Pass 2: next 11 bits among keys of bin1.
    for (int i = tid; i < 2048; i += kThreads) sm.hist[i] = 0;
    __syncthreads();
    for (int t = tid; t < n; t += kThreads) {
        const uint32_t key = key_at<kCached>(cache, row, t);
        if ((key >> 21) == bin1) atomicAdd(&sm.hist[(key >> 10) & 0x7FFu], 1u);
    }
    __syncthreads();
    select_bin<2048>(sm, kk);
    const uint32_t prefix22 = (bin1 << 11) | sm.result[0];
    kk = sm.result[1];

    // Pass 3: last 10 bits among keys sharing the top 22 bits.
    for (int i = tid; i < 1024; i += kThreads) sm.hist[i] = 0;
    __syncthreads();
    for (int t = tid; t < n; t += kThreads) {
        const uint32_t key = key_at<kCached>(cache, row, t);
        if ((key >> 10) == prefix22) atomicAdd(&sm.hist[key & 0x3FFu], 1u);
    }
    __syncthreads();
    select_bin<1024>(sm, kk);
    const uint32_t T = (prefix22 << 10) | sm.result[0];
    const uint32_t take_eq = sm.result[1];  // keys equal to T that are kept (lowest positions)

    // Ordered compaction: warp w owns a contiguous segment of positions.
    const int seg = (((n + kWarps - 1) / kWarps) + 31) & ~31;
    const int beg = warp * seg;
    const int end = min(beg + seg, n);
    uint32_t gt = 0, eq = 0;
    for (int t0 = beg; t0 < end; t0 += 32) {
        const int t = t0 + lane;
        const bool valid = t < end;
        const uint32_t key = valid ? key_at<kCached>(cache, row, t) : 0u;
        gt += __popc(__ballot_sync(0xffffffffu, valid && key > T));
        eq += __popc(__ballot_sync(0xffffffffu, valid && key == T));
    }
    if (lane == 0) {
        sm.warp_gt[warp] = gt;
        sm.warp_eq[warp] = eq;
    }
    __syncthreads();
    if (warp == 0) {
        const uint32_t g = sm.warp_gt[lane], e = sm.warp_eq[lane];
        uint32_t gi = g, ei = e;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t x = __shfl_up_sync(0xffffffffu, gi, o);
            const uint32_t y = __shfl_up_sync(0xffffffffu, ei, o);
            if (lane >= o) {
                gi += x;
                ei += y;
            }
        }
        sm.warp_gt[lane] = gi - g;
        sm.warp_eq[lane] = ei - e;
    }
    __syncthreads();
    uint32_t gt_before = sm.warp_gt[warp], eq_before = sm.warp_eq[warp];
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int t0 = beg; t0 < end; t0 += 32) {
        const int t = t0 + lane;
        const bool valid = t < end;
        const uint32_t key = valid ? key_at<kCached>(cache, row, t) : 0u;
        const bool is_gt = valid && key > T;
        const bool is_eq = valid && key == T;
        const uint32_t bgt = __ballot_sync(0xffffffffu, is_gt);
        const uint32_t beq = __ballot_sync(0xffffffffu, is_eq);
        const uint32_t eq_rank = eq_before + __popc(beq & lt_mask);
        if (is_gt || (is_eq && eq_rank < take_eq)) {
            const uint32_t pos = gt_before + __popc(bgt & lt_mask) + min(eq_rank, take_eq);
            out[pos] = t;
        }
        gt_before += __popc(bgt);
        eq_before += __popc(beq);
    }
}

__global__ void __launch_bounds__(kThreads, 1) topk_kernel(const TopkParams p, int cache_cap) {
    extern __shared__ uint32_t cache[];
    __shared__ TopkSmem sm;
    const int b = blockIdx.x;
    int64_t s = p.seq_lens[b];
    s = s < 0 ? 0 : (s > p.max_context ? p.max_context : s);
    const int n = int((s + 3) >> 2);
    const int k = p.k;
    int32_t* out = p.out + int64_t(b) * k;
    if (n <= k) {
        for (int i = threadIdx.x; i < k; i += kThreads) out[i] = i < n ? i : -1;
        return;
    }
    const float* row = p.scores + int64_t(b) * p.row_width;
    if (n <= cache_cap)
        select_row<true>(sm, cache, row, n, k, out);
    else
        select_row<false>(sm, cache, row, n, k, out);
}

}  // namespace

cudaError_t launch_topk(const TopkParams& p, cudaStream_t stream) {
    const int64_t cap64 = p.row_width < kCacheCap ? p.row_width : kCacheCap;
    const int cache_cap = p.row_width > p.k ? int(cap64) : 0;
    const size_t smem = size_t(cache_cap) * sizeof(uint32_t);
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(kCacheCap * sizeof(uint32_t)));
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    topk_kernel<<<p.batch, kThreads, smem, stream>>>(p, cache_cap);
    return cudaGetLastError();
}

}  // namespace dsa

// topk_kernel.cu -- per-request top-k over the live part of a scores row.
//
// The pages feed a top-k over the full-width logits row to sparse attention
// and name that top-k, being O(max_context), as the remaining cost of the
// indexer ("The O(Actual) Indexer: Validating 128K Context at 500 tok/s on
// Blackwell", sections "The Benchmark Results" and "The Reasoning Process").
// This kernel only ever looks at positions t < n_b, so its cost is
// O(live positions), and it does nothing but write indices when n_b <= k.
//
// Selection is exact and deterministic: scores are mapped to order-preserving
// 32-bit keys; radix histograms (11 + 11 + 10 bits) find the key T of the
// k-th largest score and how many keys equal to T are taken (the lowest
// positions); every key > T and those keys == T are written in ascending
// position.  One 1024-thread CTA per request.
//   * n_b <= 32768, first choice (sampled path): the row is copied into shared
//     memory by the bulk-copy engine; meanwhile a histogram of a sixteenth of
//     the keys (four in every 64), read straight from global memory, gives a threshold that keeps a little
//     more than k keys; once the row has landed those are appended with
//     their positions to a short list, the radix passes run on that list
//     only, and the selected positions are marked in bitmaps whose prefix
//     counts place each one in ascending order.
//   * n_b <= 32768 when the sample misjudges (fewer than k or too many keys
//     pass): each thread holds 32 consecutive keys (transposed through padded
//     shared memory); the radix passes run over all keys in registers and
//     one block scan orders the output.
//   * longer rows: keys stay in shared memory (up to 49152) or are re-read
//     from global memory (L2) on each pass, and the output is an ordered
//     compaction over per-warp segments.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "indexer_kernels.h"
#include "order_key.cuh"
#include "sm103_ptx.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kCacheCap = 49152;                    // keys held in shared memory (192 KiB)
constexpr int kKeysPerThread = 32;                  // register path: keys per thread
constexpr int kRegCap = kThreads * kKeysPerThread;  // 32768
constexpr int kLoadsPerThread = kRegCap / 4 / kThreads;  // float4 loads per thread on the register path
constexpr int kCandCap = 8192;                      // sampled path: candidate list capacity

struct TopkSmem {
    uint64_t row_bar;                            // sampled path: the row's bulk copy
    int abort;                                   // never set (bounded waits read it)
    uint32_t ncand;                              // sampled path: candidates appended
    uint32_t hist[2048];
    uint32_t warp_tot[kWarps];
    uint32_t warp_gt[kWarps];
    uint32_t warp_eq[kWarps];
    uint32_t result[2];
    alignas(16) uint32_t hist23[4096];           // sampled path: the sample (12-bit bins), then radix
                                                 // passes 1 and 2 in its two halves
    uint32_t bits_gt[kRegCap / 32];              // sampled path: positions with key > T
    uint32_t bits_eq[kRegCap / 32];              // sampled path: positions with key == T
};

static_assert(offsetof(TopkSmem, hist23) % 16 == 0, "the sample histogram is cleared with 16-byte stores");

// Shared-memory words the sampled path needs for a row of n keys: the row,
// rounded up to whole groups of four, then the candidate list (keys, positions).
__host__ __device__ constexpr int sampled_row_words(int n) { return (n + 3) & ~3; }

// Find the bin holding the kk-th largest key: result[0] = bin,
// result[1] = how many keys of that bin are still to be taken.  Ends with a
// barrier, so result[] is visible to all threads on return.  Every warp scans
// the 32 warp totals itself (two barriers, no single-warp step between them).
template <int kBins>
__device__ __forceinline__ void select_bin_from(TopkSmem& sm, const uint32_t* hist, uint32_t kk) {
    constexpr int per = kBins / kThreads;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t h[per];
    uint32_t v = 0;
#pragma unroll
    for (int i = 0; i < per; ++i) {
        h[i] = hist[tid * per + i];
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
    const uint32_t t = sm.warp_tot[lane];  // lane l: warp l's total
    uint32_t sfx = t;                      // over warps l .. 31
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_down_sync(0xffffffffu, sfx, o);
        if (lane + o < 32) sfx += x;
    }
    const uint32_t higher = __shfl_sync(0xffffffffu, sfx - t, warp);  // keys in higher warps' bins
    uint32_t above = higher + incl - v;  // keys in bins above this thread's bins
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

template <int kBins>
__device__ __forceinline__ void select_bin(TopkSmem& sm, uint32_t kk) {
    select_bin_from<kBins>(sm, sm.hist, kk);
}

__device__ __forceinline__ void clear_hist(TopkSmem& sm) {
    for (int i = threadIdx.x; i < 2048; i += kThreads) sm.hist[i] = 0;
}

// Exclusive prefix over the block, in thread order, of two per-thread counts.
// One barrier: every warp scans the 32 warp totals itself.  The totals are not
// written again by any caller afterwards, so no barrier is needed at the end.
__device__ __forceinline__ void block_scan2(TopkSmem& sm, uint32_t a, uint32_t b, uint32_t& a_before,
                                            uint32_t& b_before) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t ai = a, bi = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(0xffffffffu, ai, o);
        const uint32_t y = __shfl_up_sync(0xffffffffu, bi, o);
        if (lane >= o) {
            ai += x;
            bi += y;
        }
    }
    if (lane == 31) {
        sm.warp_gt[warp] = ai;
        sm.warp_eq[warp] = bi;
    }
    __syncthreads();
    const uint32_t g = sm.warp_gt[lane], e = sm.warp_eq[lane];  // lane l: warp l's totals
    uint32_t gs = g, es = e;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(0xffffffffu, gs, o);
        const uint32_t y = __shfl_up_sync(0xffffffffu, es, o);
        if (lane >= o) {
            gs += x;
            es += y;
        }
    }
    a_before = __shfl_sync(0xffffffffu, gs - g, warp) + ai - a;
    b_before = __shfl_sync(0xffffffffu, es - e, warp) + bi - b;
}

// --------------------------------------------------------------- short rows
// k < n <= kSmallRow: every thread ranks its key against the whole row (equal
// scores: lower position first); the k keys with rank < k are listed in
// position order by one block scan.  A few hundred comparisons per thread and
// two barriers, instead of the histogram passes.
constexpr int kSmallRow = 256;

__device__ __forceinline__ void select_row_small(TopkSmem& sm, uint32_t* keys, const float* __restrict__ row, int n,
                                                 int k, int32_t* __restrict__ out) {
    const int tid = threadIdx.x;
    if (tid < n) keys[tid] = order_key(__ldcg(row + tid));
    __syncthreads();
    uint32_t sel = 0;
    if (tid < n) {
        const uint32_t me = keys[tid];
        int rank = 0;
        for (int j = 0; j < n; ++j) {
            const uint32_t o = keys[j];
            rank += (o > me || (o == me && j < tid)) ? 1 : 0;
        }
        sel = rank < k ? 1u : 0u;
    }
    uint32_t before, unused;
    block_scan2(sm, sel, 0u, before, unused);
    if (sel) out[before] = tid;
}

// ------------------------------------------------------------ register path
// Shared-memory slot of position p: one pad word after every 32 keys, so that
// thread i reading its key j hits bank (i + j) % 32.
__device__ __forceinline__ int pad_slot(int p) { return p + (p >> 5); }

// Not inlined: the fallback of the sampled path, kept out of its register budget.
__device__ __noinline__ void select_row_regs(TopkSmem& sm, uint32_t* stage, const float* __restrict__ row, int n,
                                             int k, int32_t* __restrict__ out) {
    const int tid = threadIdx.x;
    clear_hist(sm);

    // All of this thread's 16-byte loads first (lane-consecutive: coalesced), then keys to shared memory.
    const int n4 = n >> 2;
    const float4* row4 = reinterpret_cast<const float4*>(row);
    float4 v[kLoadsPerThread];
#pragma unroll
    for (int j = 0; j < kLoadsPerThread; ++j) {
        const int i = tid + j * kThreads;
        v[j] = i < n4 ? __ldcg(row4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const int tail = (4 * n4 + tid < n) ? 4 * n4 + tid : -1;  // at most 3 trailing scores
    const float vt = tail >= 0 ? __ldcg(row + tail) : 0.f;
#pragma unroll
    for (int j = 0; j < kLoadsPerThread; ++j) {
        const int i = tid + j * kThreads;
        if (i < n4) {
            const int p = 4 * i;
            stage[pad_slot(p + 0)] = order_key(v[j].x);
            stage[pad_slot(p + 1)] = order_key(v[j].y);
            stage[pad_slot(p + 2)] = order_key(v[j].z);
            stage[pad_slot(p + 3)] = order_key(v[j].w);
        }
    }
    if (tail >= 0) stage[pad_slot(tail)] = order_key(vt);
    __syncthreads();

    const int base = tid * kKeysPerThread;  // this thread's positions [base, base + 32)
    const int valid = max(0, min(kKeysPerThread, n - base));
    uint32_t key[kKeysPerThread];
#pragma unroll
    for (int j = 0; j < kKeysPerThread; ++j) key[j] = j < valid ? stage[pad_slot(base + j)] : 0u;

#pragma unroll
    for (int j = 0; j < kKeysPerThread; ++j)
        if (j < valid) atomicAdd(&sm.hist[key[j] >> 21], 1u);
    __syncthreads();
    select_bin<2048>(sm, uint32_t(k));
    const uint32_t bin1 = sm.result[0];
    uint32_t kk = sm.result[1];

    clear_hist(sm);
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kKeysPerThread; ++j)
        if (j < valid && (key[j] >> 21) == bin1) atomicAdd(&sm.hist[(key[j] >> 10) & 0x7FFu], 1u);
    __syncthreads();
    select_bin<2048>(sm, kk);
    const uint32_t prefix22 = (bin1 << 11) | sm.result[0];
    kk = sm.result[1];

    clear_hist(sm);
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kKeysPerThread; ++j)
        if (j < valid && (key[j] >> 10) == prefix22) atomicAdd(&sm.hist[key[j] & 0x3FFu], 1u);
    __syncthreads();
    select_bin<1024>(sm, kk);
    const uint32_t T = (prefix22 << 10) | sm.result[0];
    const uint32_t take_eq = sm.result[1];

    uint32_t gt = 0, eq = 0;
#pragma unroll
    for (int j = 0; j < kKeysPerThread; ++j) {
        gt += (j < valid && key[j] > T) ? 1u : 0u;
        eq += (j < valid && key[j] == T) ? 1u : 0u;
    }
    uint32_t gt_run, eq_run;  // keys > T and == T at lower positions
    block_scan2(sm, gt, eq, gt_run, eq_run);
#pragma unroll
    for (int j = 0; j < kKeysPerThread; ++j) {
        if (j < valid) {
            if (key[j] > T) {
                out[gt_run + min(eq_run, take_eq)] = base + j;
                ++gt_run;
            } else if (key[j] == T) {
                if (eq_run < take_eq) out[gt_run + eq_run] = base + j;
                ++eq_run;
            }
        }
    }
    __syncthreads();
}

// ------------------------------------------------------------ sampled path
// Rows of up to 32768 live positions.  One thread copies the row's whole
// groups of four into shared memory with bulk copies (the last partial group
// by plain loads); thread t then reads groups t + 1024 j, positions
// 4 (t + 1024 j) + c.  While the copy is in flight thread t reads the four
// samples at positions 64 t .. 64 t + 3 from global memory; the floor of the
// bin of their 12-bit histogram that holds rank r (the expected
// rank of the k-th largest among the samples plus three standard deviations
// and four) is a threshold tau that all but rarely keeps at least k keys.
// (One bit finer than the radix passes' first digit: a sixteenth of the row
// then keeps about as few extra keys as a quarter of it at 11 bits.)  Where r
// reaches the whole sample it cannot bound the k-th key from below, and tau
// stays 0: every key is a candidate (such rows hold under 2700 keys, within
// the list).  Keys >= tau are appended, with their positions and in no
// particular order, to a list after the row; the exact 3-pass radix select
// runs on that list; the selected positions are
// set in two bitmaps (key > T, key == T), and one block scan of the bitmap
// words' bit counts gives every selected position its output slot, in
// ascending position with the lowest positions of key T taken first.
// Returns 1 when the row is done, 0 (nothing written) when fewer than k or
// more keys than the list holds pass tau -- the caller then runs the exact
// full-row path -- and -1 when the row's copy did not land within the wait
// limit (error bit set, the row padded with -1).
// (With an L2 eviction policy: the scores kernels store the row evict-last so that it waits in L2
// for this read; reading it evict-first hands those lines back.)
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void bulk_load(void* sdst, const void* gsrc, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(sdst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ int select_row_sampled(TopkSmem& sm, uint32_t* buf, int buf_words,
                                                  const float* __restrict__ row, int n, int k,
                                                  int32_t* __restrict__ out, uint32_t* err) {
    const int tid = threadIdx.x, lane = tid & 31;
    const int row_words = sampled_row_words(n);
    const int cap = min(kCandCap, (buf_words - row_words) / 2);
    if (cap < k) return 0;
    const int n4 = n >> 2;        // whole groups
    const int ng = row_words >> 2;  // groups, the last one possibly partial
    float* rs = reinterpret_cast<float*>(buf);
    uint32_t* cand_key = buf + row_words;
    uint32_t* cand_pos = cand_key + cap;

    if (tid == 0) {  // the copy goes first; this thread is the barrier's only user until the block barrier
        mbar_init(&sm.row_bar, 1);
        fence_mbar_init();
        constexpr uint32_t kChunk = 32768;
        const uint32_t bytes = uint32_t(n4) * 16u;
        const uint64_t pol = l2_policy_evict_first();
        mbar_arrive_expect_tx(&sm.row_bar, bytes);
        for (uint32_t off = 0; off < bytes; off += kChunk)
            bulk_load(reinterpret_cast<uint8_t*>(rs) + off, reinterpret_cast<const uint8_t*>(row) + off,
                      min(kChunk, bytes - off), &sm.row_bar, pol);
        sm.abort = 0;
        sm.ncand = 0;
        sm.result[0] = 0;  // tau = 0 unless the sample sets it
    }
    // Samples: the four scores at positions 64 g .. 64 g + 3 of every group g (thread g), one
    // 16-byte load each, so that the sample takes a quarter of the load slots that one score in
    // sixteen read one by one would, beside the copy.  In bounds: 64 g < n and the row width
    // is a multiple of 64.
    constexpr int kGroupStride = 64;
    static_assert(kRegCap <= kGroupStride * kThreads, "one sample group per thread covers the longest sampled row");
    static_assert(4 * kThreads == 4096, "each thread clears four bins of the sample histogram");
    const int n_groups = (n + kGroupStride - 1) / kGroupStride;
    const int ns = (n / kGroupStride) * 4 + min(n % kGroupStride, 4);  // live samples
    const int mine = tid < n_groups ? min(n - kGroupStride * tid, 4) : 0;
    const float4 sv = tid < n_groups ? __ldcg(reinterpret_cast<const float4*>(row + kGroupStride * tid))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
    if (tid < 4 && 4 * n4 + tid < row_words)  // the partial group: live scores, then zeros
        rs[4 * n4 + tid] = 4 * n4 + tid < n ? __ldcg(row + 4 * n4 + tid) : 0.f;
    reinterpret_cast<uint4*>(sm.hist23)[tid] = make_uint4(0u, 0u, 0u, 0u);
    for (int i = tid; i < 2048; i += kThreads) sm.hist[i] = 0;
    sm.bits_gt[tid] = 0;
    sm.bits_eq[tid] = 0;
    __syncthreads();
    const float expect = float(k) * float(ns) / float(n);
    const int r = int(expect + 3.f * sqrtf(expect)) + 4;
    if (r < ns) {
        if (mine > 0) atomicAdd(&sm.hist23[order_key(sv.x) >> 20], 1u);
        if (mine > 1) atomicAdd(&sm.hist23[order_key(sv.y) >> 20], 1u);
        if (mine > 2) atomicAdd(&sm.hist23[order_key(sv.z) >> 20], 1u);
        if (mine > 3) atomicAdd(&sm.hist23[order_key(sv.w) >> 20], 1u);
        __syncthreads();
        select_bin_from<4096>(sm, sm.hist23, uint32_t(r));
    }
    const uint32_t tau = sm.result[0] << 20;
    const bool landed = mbar_wait(&sm.row_bar, 0, &sm.abort);
    if (__syncthreads_or(!landed)) {
        if (tid == 0) atomicOr(err, kErrWaitTimeout);
        for (int i = tid; i < k; i += kThreads) out[i] = -1;
        if (!landed) mbar_wait(&sm.row_bar, 0, &sm.abort);  // once more (bounded) for the copy in flight
        return -1;
    }
    const float4* rs4 = reinterpret_cast<const float4*>(rs);

    // Candidates: bit 4 j + c of `flags` marks position 4 (tid + 1024 j) + c.  The test
    // key(v) >= tau is made in fp32 as v >= f_tau, which is the same for every non-NaN v
    // (-0 == +0 on both sides); the unordered compare also admits every NaN and, when tau
    // lies past +inf, +inf itself.  Extra candidates are harmless as long as the k-th
    // largest key of the list is >= tau, which is checked after the radix passes.
    const float f_tau = tau < 0x00800000u   ? __int_as_float(0xff800000)  // every non-NaN key >= tau
                        : tau > 0xFF800000u ? __int_as_float(0x7f800000)
                        : (tau & 0x80000000u) ? __uint_as_float(tau & 0x7FFFFFFFu)
                                              : __uint_as_float(~tau);
    uint32_t flags = 0;
#pragma unroll
    for (int j = 0; j < kLoadsPerThread; ++j) {
        const int g = tid + j * kThreads;
        const int live = n - 4 * g;  // > 3: the whole group
        const float4 v = g < ng ? rs4[g] : make_float4(0.f, 0.f, 0.f, 0.f);
        const uint32_t f = (live > 0 && !(v.x < f_tau) ? 1u : 0u) | (live > 1 && !(v.y < f_tau) ? 2u : 0u) |
                           (live > 2 && !(v.z < f_tau) ? 4u : 0u) | (live > 3 && !(v.w < f_tau) ? 8u : 0u);
        flags |= f << (4 * j);
    }
    // The sample histogram has been read (select_bin_from ended with a barrier): zero it for
    // radix passes 1 and 2 (the barrier after the append orders this before them).
    reinterpret_cast<uint4*>(sm.hist23)[tid] = make_uint4(0u, 0u, 0u, 0u);
    const uint32_t cnt = __popc(flags);
    uint32_t incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
    }
    uint32_t base = 0;
    if (lane == 31) base = atomicAdd(&sm.ncand, incl);
    uint32_t slot = __shfl_sync(0xffffffffu, base, 31) + incl - cnt;
    while (flags) {
        const int i = __ffs(flags) - 1;
        flags &= flags - 1u;
        const int pos = 4 * (tid + kThreads * (i >> 2)) + (i & 3);
        if (slot < uint32_t(cap)) {
            cand_key[slot] = order_key(rs[pos]);
            cand_pos[slot] = uint32_t(pos);
        }
        ++slot;
    }
    __syncthreads();
    const int C = int(sm.ncand);
    if (C < k || C > cap) return 0;

    // Exact selection on the list: passes 1 and 2 count into the halves of hist23, pass 3 into
    // hist (all zero by now).
    uint32_t* hist2 = sm.hist23;
    uint32_t* hist3 = sm.hist23 + 2048;
    for (int i = tid; i < C; i += kThreads) atomicAdd(&hist2[cand_key[i] >> 21], 1u);
    __syncthreads();
    select_bin_from<2048>(sm, hist2, uint32_t(k));
    const uint32_t bin1 = sm.result[0];
    uint32_t kk = sm.result[1];
    for (int i = tid; i < C; i += kThreads) {
        const uint32_t ck = cand_key[i];
        if ((ck >> 21) == bin1) atomicAdd(&hist3[(ck >> 10) & 0x7FFu], 1u);
    }
    __syncthreads();
    select_bin_from<2048>(sm, hist3, kk);
    const uint32_t prefix22 = (bin1 << 11) | sm.result[0];
    kk = sm.result[1];
    for (int i = tid; i < C; i += kThreads) {
        const uint32_t ck = cand_key[i];
        if ((ck >> 10) == prefix22) atomicAdd(&sm.hist[ck & 0x3FFu], 1u);
    }
    __syncthreads();
    select_bin<1024>(sm, kk);
    const uint32_t T = (prefix22 << 10) | sm.result[0];
    const uint32_t take_eq = sm.result[1];
    if (T < tau) return 0;  // the list's extra candidates (NaN, +inf) reached rank k

    // Mark the selected positions, then write them in ascending order: thread t owns
    // bitmap word t (positions 32 t .. 32 t + 31).
    for (int i = tid; i < C; i += kThreads) {
        const uint32_t ck = cand_key[i], pos = cand_pos[i];
        if (ck > T)
            atomicOr(&sm.bits_gt[pos >> 5], 1u << (pos & 31u));
        else if (ck == T)
            atomicOr(&sm.bits_eq[pos >> 5], 1u << (pos & 31u));
    }
    __syncthreads();
    const uint32_t g = sm.bits_gt[tid], e = sm.bits_eq[tid];
    uint32_t g_before, e_before;
    block_scan2(sm, __popc(g), __popc(e), g_before, e_before);
    uint32_t m = g;
    for (uint32_t ee = e, c = e_before; ee != 0u && c < take_eq; ++c) {  // the lowest equal keys still wanted
        m |= ee & (0u - ee);
        ee &= ee - 1u;
    }
    uint32_t at = g_before + min(e_before, take_eq);
    while (m) {
        const int bit = __ffs(m) - 1;
        m &= m - 1u;
        out[at++] = 32 * tid + bit;
    }
    return 1;
}

// ------------------------------------------------------- long-row path
template <bool kCached>
__device__ __forceinline__ uint32_t key_at(const uint32_t* cache, const float* row, int t) {
    if constexpr (kCached)
        return cache[t];
    else
        return order_key(__ldcg(row + t));
}

template <bool kCached>
__device__ __forceinline__ void select_row(TopkSmem& sm, uint32_t* cache, const float* __restrict__ row, int n,
                                           int k, int32_t* __restrict__ out) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // Pass 1: top 11 bits of every live key (and fill the cache); 8 loads in flight per thread.
    clear_hist(sm);
    __syncthreads();
    for (int t0 = 0; t0 < n; t0 += 8 * kThreads) {
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int t = t0 + j * kThreads + tid;
            v[j] = t < n ? __ldcg(row + t) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int t = t0 + j * kThreads + tid;
            if (t < n) {
                const uint32_t key = order_key(v[j]);
                if constexpr (kCached) cache[t] = key;
                atomicAdd(&sm.hist[key >> 21], 1u);
            }
        }
    }
    __syncthreads();
    select_bin<2048>(sm, uint32_t(k));
    const uint32_t bin1 = sm.result[0];
    uint32_t kk = sm.result[1];

    // Pass 2: next 11 bits among keys of bin1.
    clear_hist(sm);
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
    clear_hist(sm);
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
    extern __shared__ __align__(16) uint32_t cache[];
    __shared__ TopkSmem sm;
    // Launched as a programmatic dependent of the scores kernel: wait for its
    // results before reading global memory.  Before the wait, L2 prefetches of
    // the row, its length and its output (no data is consumed, and L2 is where
    // the scores kernel's writes land) let the SM translate those addresses
    // while the scores kernel finishes.
    if (threadIdx.x == 0) prefetch_l2(p.seq_lens + blockIdx.x / p.tokens);
    if (threadIdx.x == 32) prefetch_l2(p.scores + int64_t(blockIdx.x) * p.row_width);
    if (threadIdx.x == 64) prefetch_l2(p.out + int64_t(blockIdx.x) * p.k);
    pdl_wait_prior_grid();
    pdl_allow_next_grid();
    const int b = blockIdx.x;  // row: request b / tokens, query token b % tokens
    int64_t s = p.seq_lens[b / p.tokens];
    s = s < 0 ? 0 : (s > p.max_context ? p.max_context : s);
    s -= p.tokens - 1 - b % p.tokens;  // token j sees the first L - (tokens - 1 - j) tokens
    s = s < 0 ? 0 : s;
    const int n = int((s + 3) >> 2);
    const int k = p.k;
    int32_t* out = p.out + int64_t(b) * k;
    if (n <= k) {
        for (int i = threadIdx.x; i < k; i += kThreads) out[i] = i < n ? i : -1;
        return;
    }
    const float* row = p.scores + int64_t(b) * p.row_width;
    if (n <= kSmallRow) {
        select_row_small(sm, cache, row, n, k, out);
        return;
    }
    if (n <= kRegCap && pad_slot(n) <= cache_cap) {
        const int done = select_row_sampled(sm, cache, cache_cap, row, n, k, out, p.err);
        if (done == 0) {
            __syncthreads();
            select_row_regs(sm, cache, row, n, k, out);
        }
    }
    else if (n <= cache_cap)
        select_row<true>(sm, cache, row, n, k, out);
    else
        select_row<false>(sm, cache, row, n, k, out);
}

}  // namespace

cudaError_t launch_topk(const TopkParams& p, cudaStream_t stream) {
    // Shared keys: the larger of the row padded by one word per 32 (register path) and the
    // row plus a candidate list (sampled path), capped at kCacheCap.
    const int64_t padded = p.row_width + p.row_width / 32 + 1;
    const int64_t cand = p.row_width < kCandCap ? p.row_width : kCandCap;
    const int64_t sampled = ((p.row_width + 3) & ~int64_t(3)) + 2 * cand;
    const int64_t want = padded > sampled ? padded : sampled;
    const int cache_cap = p.row_width > p.k ? int(want < kCacheCap ? want : kCacheCap) : 0;
    const size_t smem = size_t(cache_cap) * sizeof(uint32_t);
    static SmemLimitOnce smem_limit;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = smem_limit.apply(dev, topk_kernel, int(kCacheCap * sizeof(uint32_t)));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(p.batch) * unsigned(p.tokens));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, topk_kernel, p, cache_cap);
}

}  // namespace dsa

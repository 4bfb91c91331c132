// scores_kernel.cu -- paged indexer scores on sm_103a.
//
// Computes, for each request b and live C4 position t < n_b = ceil(seq_len/4),
//     score[b, t] = sum_h w[b, h] * max(0, q[b, h, :] . k[t, :])
// with k[t] = key_pool[page_table[b, t / 64], t % 64, :], and -inf at the
// positions of the row that hold no live key.  The operator chain (gather
// through the page table, bmm, clamp_min, mul by head weights, sum over
// heads, -inf mask) is the one named in "The Indexer O(max_context)
// Breakthrough", section "The Indexer O(max_context) Breakthrough"; the fixed,
// capture-safe grid with a cheap -inf path for pages past the live length is
// from "The O(Actual) Indexer: Validating 128K Context at 500 tok/s on
// Blackwell", section "The Bottleneck That Was".
//
// Design (GB300-first, not the pages' one-program-per-page Triton kernel):
//   * Persistent grid of one CTA per SM.  The grid size depends only on the
//     device, so graph capture is safe; the work is split by live work units,
//     so the cost is O(live positions), not O(max_context).
//   * Work unit = 2 consecutive pages of one request = 128 keys = 16 KiB.
//     Each CTA takes a contiguous range of the batch's live units.
//   * Warp 0 (one lane) gathers pages with TMA tiled loads (128-byte swizzle)
//     into an 8-stage shared-memory ring, plus the request's 4 KiB query
//     tile; page ids for 32 units at a time are fetched by the whole warp so
//     that the page-table latency is paid once per 32 units.
//   * Warp 1 (one lane) issues tcgen05.mma kind::f16, M=128 keys x N=32 heads
//     x K=64 dims (4 instructions of K=16), fp32 accumulators in TMEM, 4
//     accumulator stages of 32 columns.
//   * Warps 2-5 read the accumulators with tcgen05.ld (thread = key row,
//     registers = 32 heads), apply relu, the head weights and the head sum in
//     registers, mask, and store 128 contiguous fp32 scores per unit.  Before
//     the unit loop they also stream -inf over the dead part of every row
//     (split evenly over all CTAs) when a full-width row is requested.
//   * Every wait is bounded (about 1 s); a timeout sets an error bit, stops
//     all roles, drains in-flight copies and MMAs and frees TMEM.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "indexer_kernels.h"
#include "sm103_ptx.cuh"

namespace dsa {
namespace {

constexpr int kStages = 8;
constexpr int kAccStages = 4;
constexpr int kAccCols = 32;                         // fp32 columns per accumulator (N = 32 heads)
constexpr uint32_t kTmemCols = kAccStages * kAccCols;  // 128 (power of two >= 32)
constexpr int kThreads = 192;                        // 6 warps
constexpr int kATileBytes = 2 * kPageBytes;          // 16 KiB: 128 keys x 128 B
constexpr int kStageBytes = kATileBytes + kQRowBytes;  // 20 KiB, multiple of 1024
constexpr uint32_t kIdesc = idesc_bf16_f32(128, kAccCols);

struct __align__(8) SmemCtl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tfull[kAccStages];
    uint64_t tempty[kAccStages];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int32_t n_live[kMaxBatch];
    int32_t unit_start[kMaxBatch + 1];
};

constexpr size_t kSmemBytes = 1024 /* alignment slack */ + size_t(kStages) * kStageBytes + sizeof(SmemCtl);
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kStageBytes % 1024 == 0, "stage tiles must stay 1024-byte aligned");

// Largest b in [0, batch) with unit_start[b] <= u (rows without units share
// their start with the next row, so this lands on the row that owns u).
__device__ __forceinline__ int row_of_unit(const int32_t* unit_start, int batch, int u) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (unit_start[mid] <= u)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

__global__ void __launch_bounds__(kThreads, 1)
    scores_kernel(const __grid_constant__ CUtensorMap keys_map, const __grid_constant__ CUtensorMap q_map,
                  const ScoresParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    SmemCtl& ctl = *reinterpret_cast<SmemCtl*>(tiles + size_t(kStages) * kStageBytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int batch = p.batch;

    // ---- set-up: barriers, TMEM, per-row live counts and unit prefix.
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl.full[s], 1);
            mbar_init(&ctl.empty[s], 1);
        }
        for (int a = 0; a < kAccStages; ++a) {
            mbar_init(&ctl.tfull[a], 1);
            mbar_init(&ctl.tempty[a], 4 * 32);
        }
        mbar_init(&ctl.drain, 1);
        ctl.abort = 0;
        fence_mbar_init();
        tma_prefetch_map(&keys_map);
        tma_prefetch_map(&q_map);
    }
    if (warp == 1) {
        tmem_alloc(&ctl.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 2) {
        // 32 lanes scan the batch: lane l owns rows [l*per, (l+1)*per).
        const int per = (batch + 31) / 32;
        const int b0 = min(lane * per, batch), b1 = min(b0 + per, batch);
        int units = 0;
        bool clamped = false;
        for (int b = b0; b < b1; ++b) {
            int64_t s = p.seq_lens[b];
            if (s < 0 || s > p.max_context) clamped = true;
            s = s < 0 ? 0 : (s > p.max_context ? p.max_context : s);
            const int n = static_cast<int>((s + 3) >> 2);
            ctl.n_live[b] = n;
            units += (n + kUnitPositions - 1) / kUnitPositions;
        }
        int incl = units;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - units;
        for (int b = b0; b < b1; ++b) {
            ctl.unit_start[b] = run;
            run += (ctl.n_live[b] + kUnitPositions - 1) / kUnitPositions;
        }
        if (lane == 31) ctl.unit_start[batch] = incl;
        if (clamped && blockIdx.x == 0) atomicOr(p.err, kErrSeqLenClamped);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    const int total_units = ctl.unit_start[batch];
    const int grid = gridDim.x;
    const int u_begin = static_cast<int>((int64_t(total_units) * blockIdx.x) / grid);
    const int u_end = static_cast<int>((int64_t(total_units) * (blockIdx.x + 1)) / grid);
    const uint32_t tmem_base = ctl.tmem_base;
    const int64_t M = p.row_width;
    const int W = p.table_width;

    if (warp == 0) {
        // ================= producer: page ids, then TMA gathers =================
        const uint64_t pol_keys = l2_policy_evict_first();
        const uint64_t pol_q = l2_policy_evict_last();
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        bool stop = false;
        for (int u0 = u_begin; u0 < u_end && !stop; u0 += 32) {
            const int cnt = min(32, u_end - u0);
            int b = 0, pg0 = -1, pg1 = -2;
            if (lane < cnt) {
                const int u = u0 + lane;
                b = row_of_unit(ctl.unit_start, batch, u);
                const int pair = u - ctl.unit_start[b];
                const int live_pages = (ctl.n_live[b] + kPageEntries - 1) / kPageEntries;
                const int32_t* row = p.page_table + int64_t(b) * W;
                pg0 = __ldg(row + 2 * pair);
                pg1 = (2 * pair + 1 < live_pages) ? __ldg(row + 2 * pair + 1) : -2;  // -2: no live page
            }
            for (int i = 0; i < cnt; ++i) {
                const int bi = __shfl_sync(0xffffffffu, b, i);
                const int g0 = __shfl_sync(0xffffffffu, pg0, i);
                const int g1 = __shfl_sync(0xffffffffu, pg1, i);
                int failed = 0;
                if (lane == 0) {
                    if (!mbar_wait(&ctl.empty[stage], phase ^ 1u, &ctl.abort)) {
                        failed = 1;
                    } else {
                        const bool ok0 = g0 >= 0 && g0 < p.num_pages;
                        const bool ok1 = g1 >= 0 && g1 < p.num_pages;
                        if (!ok0 || (g1 != -2 && !ok1)) atomicOr(p.err, kErrBadPage);
                        const uint32_t bytes = kQRowBytes + (ok0 ? kPageBytes : 0) + (ok1 ? kPageBytes : 0);
                        uint8_t* a = tiles + size_t(stage) * kStageBytes;
                        mbar_arrive_expect_tx(&ctl.full[stage], bytes);
                        if (ok0) tma_load_3d(a, &keys_map, &ctl.full[stage], 0, 0, g0, pol_keys);
                        if (ok1) tma_load_3d(a + kPageBytes, &keys_map, &ctl.full[stage], 0, 0, g1, pol_keys);
                        tma_load_2d(a + kATileBytes, &q_map, &ctl.full[stage], 0, bi * kHeads, pol_q);
                        ++issued;
                    }
                }
                if (__shfl_sync(0xffffffffu, failed, 0)) {
                    stop = true;
                    break;
                }
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (lane == 0 && stop) {
            atomicOr(p.err, kErrWaitTimeout);
            ctl.abort = 1;
        }
        // Let every copy this CTA issued land before the CTA may exit.
        if (lane == 0 && ctl.abort) {
            const int outstanding = issued < kStages ? issued : kStages;
            int s = stage;
            uint32_t ph = phase;
            for (int i = 0; i < outstanding; ++i) {
                if (s == 0) {
                    s = kStages - 1;
                    ph ^= 1u;
                } else {
                    --s;
                }
                const uint32_t a = smem_u32(&ctl.full[s]);
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(a, ph) && global_timer_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
    } else if (warp == 1) {
        // ================= MMA issuer (one lane) =================
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool stop = false;
            for (int u = u_begin; u < u_end; ++u) {
                if (!mbar_wait(&ctl.full[stage], phase, &ctl.abort) ||
                    !mbar_wait(&ctl.tempty[acc], acc_phase ^ 1u, &ctl.abort)) {
                    stop = true;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t a_addr = smem_u32(tiles + size_t(stage) * kStageBytes);
                const uint64_t a_desc = smem_desc_kmajor_sw128(a_addr);
                const uint64_t b_desc = smem_desc_kmajor_sw128(a_addr + kATileBytes);
                const uint32_t d_tmem = tmem_base + uint32_t(acc * kAccCols);
#pragma unroll
                for (int kk = 0; kk < kHeadDim / 16; ++kk)  // K = 16 per MMA: +32 bytes = +2 in the address field
                    umma_bf16_ss(d_tmem, a_desc + 2u * kk, b_desc + 2u * kk, kIdesc, kk > 0 ? 1u : 0u);
                umma_commit(&ctl.empty[stage]);
                umma_commit(&ctl.tfull[acc]);
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (++acc == kAccStages) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (stop) {
                atomicOr(p.err, kErrWaitTimeout);
                ctl.abort = 1;
            }
            // Every MMA issued so far completes before TMEM is released.
            umma_commit(&ctl.drain);
            const uint32_t a = smem_u32(&ctl.drain);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(a, 0) && global_timer_ns() - t0 < kWaitLimitNs) {
            }
        }
        __syncwarp();
    } else {
        // ================= epilogue: warps 2..5 =================
        const int et = threadIdx.x - 64;   // 0..127
        const int quad = warp & 3;         // TMEM lanes [32*quad, 32*quad + 32)
        const float neg_inf = __int_as_float(0xff800000);

        if (p.fill_dead) {
            const float4 ninf4 = make_float4(neg_inf, neg_inf, neg_inf, neg_inf);
            const int64_t stride = int64_t(grid) * 128;
            for (int b = 0; b < batch; ++b) {
                const int64_t units = ctl.unit_start[b + 1] - ctl.unit_start[b];
                const int64_t extent = units * kUnitPositions < M ? units * kUnitPositions : M;
                float4* row = reinterpret_cast<float4*>(p.out + int64_t(b) * M);
                for (int64_t i = extent / 4 + int64_t(blockIdx.x) * 128 + et; i < M / 4; i += stride)
                    __stcs(row + i, ninf4);
            }
        }

        int acc = 0;
        uint32_t acc_phase = 0;
        int cur_b = -1;
        float wv[kHeads];
#pragma unroll
        for (int h = 0; h < kHeads; ++h) wv[h] = 0.f;
        bool stop = false;
        for (int u0 = u_begin; u0 < u_end && !stop; u0 += 32) {
            const int cnt = min(32, u_end - u0);
            int b = 0, pair = 0, pg = -2, n = 0;
            if (lane < cnt) {
                const int u = u0 + lane;
                b = row_of_unit(ctl.unit_start, batch, u);
                pair = u - ctl.unit_start[b];
                n = ctl.n_live[b];
                const int j = 2 * pair + (quad >> 1);  // page holding this warp's 32 keys
                const int live_pages = (n + kPageEntries - 1) / kPageEntries;
                pg = j < live_pages ? __ldg(p.page_table + int64_t(b) * W + j) : -2;
            }
            for (int i = 0; i < cnt; ++i) {
                const int bi = __shfl_sync(0xffffffffu, b, i);
                const int pi = __shfl_sync(0xffffffffu, pair, i);
                const int gi = __shfl_sync(0xffffffffu, pg, i);
                const int ni = __shfl_sync(0xffffffffu, n, i);
                if (bi != cur_b) {
                    const float4* wr = reinterpret_cast<const float4*>(p.w + int64_t(bi) * kHeads);
#pragma unroll
                    for (int h4 = 0; h4 < kHeads / 4; ++h4) {
                        const float4 v = __ldg(wr + h4);
                        wv[4 * h4 + 0] = v.x;
                        wv[4 * h4 + 1] = v.y;
                        wv[4 * h4 + 2] = v.z;
                        wv[4 * h4 + 3] = v.w;
                    }
                    cur_b = bi;
                }
                const bool ok = mbar_wait(&ctl.tfull[acc], acc_phase, &ctl.abort);
                if (!__all_sync(0xffffffffu, ok)) {
                    stop = true;
                    break;
                }
                tc_fence_after_sync();
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(acc * kAccCols), r);
                tmem_ld_wait(r);
                tc_fence_before_sync();
                mbar_arrive(&ctl.tempty[acc]);

                float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
                for (int h = 0; h < kHeads; h += 4) {
                    s0 = fmaf(wv[h + 0], fmaxf(__uint_as_float(r[h + 0]), 0.f), s0);
                    s1 = fmaf(wv[h + 1], fmaxf(__uint_as_float(r[h + 1]), 0.f), s1);
                    s2 = fmaf(wv[h + 2], fmaxf(__uint_as_float(r[h + 2]), 0.f), s2);
                    s3 = fmaf(wv[h + 3], fmaxf(__uint_as_float(r[h + 3]), 0.f), s3);
                }
                const float s = (s0 + s1) + (s2 + s3);
                const int64_t t = int64_t(pi) * kUnitPositions + quad * 32 + lane;
                const bool valid = t < ni && gi >= 0 && gi < p.num_pages;
                if (t < M) p.out[int64_t(bi) * M + t] = valid ? s : neg_inf;
                if (++acc == kAccStages) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
        }
        if (stop && lane == 0) {
            atomicOr(p.err, kErrWaitTimeout);
            ctl.abort = 1;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_scores(const CUtensorMap& keys_map, const CUtensorMap& q_map, const ScoresParams& p,
                          cudaStream_t stream) {
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes));
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    scores_kernel<<<sms, kThreads, kSmemBytes, stream>>>(keys_map, q_map, p);
    return cudaGetLastError();
}

}  // namespace dsa

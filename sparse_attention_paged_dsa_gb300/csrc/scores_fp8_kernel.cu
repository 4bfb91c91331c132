// scores_fp8_kernel.cu -- paged indexer scores on an fp8 key cache, sm_103a.
//
// Same scores as scores_kernel.cu,
//     score[b, t] = sum_h w[b, h] * max(0, q[b, h, :] . k[t, :]),  -inf past n_b,
// with each C4 key stored as 64 OCP e4m3 codes and one positive fp32 scale,
// k[t, d] = scale[t] * e4m3(code[t, d]).  The deployment on the pages keeps
// an fp8 KV cache ("The Indexer O(max_context) Breakthrough", section "The
// Indexer O(max_context) Breakthrough"); the scale format is not given there
// and is this library's choice.  A key costs 68 bytes instead of 128.
//
// The key codes go from HBM to shared memory by TMA and from there straight
// into tcgen05.mma kind::f8f6f4 (no conversion pass over the keys).  The MMA
// wants both operands in 8-bit formats, so each bf16 query head is written as
// a sum of two e4m3 terms under a per-head power-of-two scale S_h:
//     q_h / S_h = hi_h + lo_h,   hi_h = e4m3(q_h / S_h),   lo_h = e4m3(q_h / S_h - hi_h),
// with S_h = 2^(e_h - 7), e_h the binary exponent of max_d |q_h,d| (so the
// largest element of the head lies in [128, 256)).  A bf16 value carries 8
// significant bits; hi keeps the top 4 (rounded) and the remainder is at most
// 8 of the value's last bits, which e4m3 holds exactly down to its smallest
// quantum 2^-9.  So every element within a factor 2^9 of its head's largest
// one is represented exactly, and smaller ones keep an absolute error of at
// most 2^-10 in units of S_h, below 2^-17 of the head's largest element.
// The hi rows and the lo rows of the split query are stacked into one
// N = 64 operand (hi heads 0..31, then lo heads 0..31), so two MMAs of K = 32
// per unit accumulate  hi_acc[h] = sum_d code_t,d * hi_h,d  and lo_acc[h]
// into two fp32 columns per head, and with acc[h] = hi_acc[h] + lo_acc[h]
//     q_h . k_t = S_h * scale_t * acc[h].
// (Each tcgen05.mma costs about as much of a unit's time as its data: four
// MMAs of N = 32 per unit, hi and lo in turn into one column, ran 1 us
// slower on the dense 128K workload.)
// S_h and scale_t are positive, so relu commutes with them: the epilogue
// forms w_h * S_h * relu(acc[h]), sums over heads and multiplies by scale_t
// once.
//
// Pipeline (per CTA, three CTAs per SM, persistent grid sized by the device):
//   * warps 0 and 3 (producers): the unit schedule and page ids
//     (scores_common.cuh); warp 0 takes the CTA's even units, warp 3 the odd
//     ones (one TMA-issuing thread keeps too few 4 KiB boxes in flight to
//     cover HBM latency).  Per unit, lane 0 issues two TMA code boxes (64-byte
//     swizzle) into the stage ring and all 32 lanes copy the 2 x 256 B of
//     scales into a scale ring with 16-byte cp.async that arrive on the
//     stage's full barrier (a TMA instruction costs about as much issue time
//     as a whole page, so the small scale rows do not go through TMA).  Per
//     request change the owner of the first unit stages the bf16 query and
//     its head weights (TMA) for the splitters.
//   * warps 8 and 9: per request change, split the query into the hi and lo
//     e4m3 tiles the MMA reads (64-byte swizzle) and w_h * S_h, in a small
//     ring that the epilogue frees when it leaves the request.  The split is
//     on the path to each request's first MMA, so two warps share it, each
//     thread taking half of one head.
//   * warp 2: the -inf fill of the rows' dead parts (full-width rows), with
//     the same flat per-CTA share as the bf16 kernel's set-up warp.
//   * warp 1: tcgen05.mma kind::f8f6f4, M=128 keys x N=64 (hi, lo) x K=32,
//     two per unit (the two K-slices), into one of 2 TMEM accumulators of 64
//     columns (three CTAs' accumulators fill 384 of the SM's 512 columns).
//   * warps 4-7: tcgen05.ld, relu, weighted head sum, key scale, live mask,
//     128-byte stores.
//   * Every wait is bounded (about 1 s); a timeout sets an error bit, stops
//     all roles, drains in-flight copies and MMAs and frees TMEM.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "indexer_kernels.h"
#include "scores_common.cuh"
#include "sm103_ptx.cuh"

namespace dsa {
namespace {

using namespace scores;

// Three CTAs per SM, two TMA-issuing producer warps each: one issuing thread
// keeps too few 4 KiB boxes in flight to cover HBM latency (a TMA instruction
// takes about 120 cycles to issue), so each SM runs six issuers.  The kernel
// is a template on its number S of 8 KiB key-code stages (two pages each,
// shared by the producer warps); five are used (four and six measured the
// same).
constexpr int kQRaw = 2;         // staged bf16 query rows
constexpr int kQSlots = 2;       // split e4m3 query tiles
constexpr int kAccStages = 2;
constexpr int kRing = 16;        // metadata and scale ring, >= S + kAccStages + 1 (a power of two)
constexpr int kCtasPerSm = 3;
constexpr int kAccCols = 64;     // N = 64: the 32 heads' hi terms, then their lo terms
constexpr uint32_t kTmemCols = kAccStages * kAccCols;  // 128
constexpr int kSplitWarps = 2;                  // warps 8, 9
constexpr int kConvThreads = 32 * kSplitWarps;
constexpr int kEpiThreads = 128;
constexpr int kThreads = 128 + kEpiThreads + kConvThreads;  // producers 0 and 3, MMA 1, fill 2, epilogue 4..7, splitters 8, 9
constexpr int kStageBytes = 2 * kPageCodeBytes;            // 8 KiB: 128 keys x 64 B
constexpr int kQHalfBytes = kHeads * kHeadDim;             // 2 KiB: 32 heads x 64 B (hi or lo)
constexpr int kQ8Bytes = 2 * kQHalfBytes;                  // hi tile, then lo tile
constexpr int kUnitScaleBytes = 2 * kPageScaleBytes;       // 512 B
constexpr int kWRowBytes = kHeads * 4;                     // 128 B
constexpr uint32_t kFullArrivals = 1 + 32;                 // producer lane 0 + its 32 lanes' scale copies
constexpr uint32_t kIdesc = idesc_e4m3_f32(128, kAccCols);
static_assert(kTmemCols * kCtasPerSm <= 512, "TMEM columns per SM");

template <int S>
struct __align__(16) SmemCtl {
    uint64_t full[S];
    uint64_t empty[S];
    uint64_t qraw_full[kQRaw];
    uint64_t qraw_empty[kQRaw];
    uint64_t q8_full[kQSlots];
    uint64_t q8_empty[kQSlots];
    uint64_t tfull[kAccStages];
    uint64_t tempty[kAccStages];
    uint64_t tmeta[kAccStages];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int32_t meta[kRing];
    int32_t qrow[kQRaw];                      // request of each staged query (-1: no more)
    int32_t split_flag[kSplitWarps];          // each splitter warp's view of the current raw query
    __align__(8) uint32_t split_amax[kHeads][kSplitWarps];  // partial max |q| bits per head and warp
    __align__(16) float wq[kQSlots][kHeads];  // w_h * S_h of each split query
};

// Shared memory: the tile region (1024-byte aligned base: stages | q8 slots |
// raw queries | scales | raw weights), the control block, the row table.
template <int S>
struct Fp8Layout {
    static_assert(kRing >= S + kAccStages + 1, "metadata ring too small");
    static constexpr size_t kOffQ8 = size_t(S) * kStageBytes;
    static constexpr size_t kOffQRaw = kOffQ8 + size_t(kQSlots) * kQ8Bytes;
    static constexpr size_t kOffScales = kOffQRaw + size_t(kQRaw) * kQRowBytes;
    static constexpr size_t kOffWRaw = kOffScales + size_t(kRing) * kUnitScaleBytes;
    static constexpr size_t kTileBytes = kOffWRaw + size_t(kQRaw) * kWRowBytes;
    static_assert(kTileBytes % 16 == 0, "control block alignment");
    static constexpr size_t kFixedBytes = 1024 /* alignment slack */ + kTileBytes + sizeof(SmemCtl<S>);
    static constexpr size_t bytes(int batch) { return kFixedBytes + row_table_bytes(batch); }
    static constexpr bool fits(int batch) { return bytes(batch) * kCtasPerSm <= 226 * 1024; }
};
constexpr int kFp8Stages = 5;
static_assert(Fp8Layout<kFp8Stages>::fits(kMaxBatch), "shared memory budget per SM");

// 16-byte global -> shared copy through L2 only (cp.async), and the arrival on
// `bar` that fires once all of this thread's earlier cp.async copies landed
// (counted in the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Named barrier 1 over the splitter warps.
__device__ __forceinline__ void split_bar_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConvThreads) : "memory"); }

// Two floats to two e4m3 codes (round to nearest even, saturating); `lo_val` in the low byte.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo_val, float hi_val) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi_val), "f"(lo_val));
    return r;
}

// Two e4m3 codes (low byte first) to two floats, exactly.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t codes) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(static_cast<unsigned short>(codes & 0xFFFFu)));
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// Split 8 consecutive query values (already divided by S_h) into 8 hi and 8 lo codes.
__device__ __forceinline__ void split8(const float* x, uint2& hi, uint2& lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        h[i] = f32x2_to_e4m3x2(x[2 * i], x[2 * i + 1]);
        const float2 hv = e4m3x2_to_f32x2(h[i]);
        l[i] = f32x2_to_e4m3x2(x[2 * i] - hv.x, x[2 * i + 1] - hv.y);
    }
    hi = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
    lo = make_uint2(l[0] | (l[1] << 16), l[2] | (l[3] << 16));
}

template <int S>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    scores_fp8_kernel(const __grid_constant__ CUtensorMap codes_map, const __grid_constant__ CUtensorMap qraw_map,
                      const __grid_constant__ CUtensorMap w_map, const ScoresParams p) {
    constexpr int kStages = S;
    constexpr size_t kOffQ8 = Fp8Layout<S>::kOffQ8, kOffQRaw = Fp8Layout<S>::kOffQRaw;
    constexpr size_t kOffScales = Fp8Layout<S>::kOffScales, kOffWRaw = Fp8Layout<S>::kOffWRaw;
    constexpr size_t kTileBytes = Fp8Layout<S>::kTileBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* q8 = tiles + kOffQ8;
    uint8_t* qraw = tiles + kOffQRaw;
    const float* scale_ring = reinterpret_cast<const float*>(tiles + kOffScales);
    const float* wraw = reinterpret_cast<const float*>(tiles + kOffWRaw);
    SmemCtl<S>& ctl = *reinterpret_cast<SmemCtl<S>*>(tiles + kTileBytes);
    const RowTable rows = row_table_at(tiles + kTileBytes + sizeof(SmemCtl<S>), p.batch);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int batch = p.batch;

    // ---- set-up that touches no global memory (overlaps the previous kernel).
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl.full[s], kFullArrivals);
            mbar_init(&ctl.empty[s], 1);
        }
        for (int s = 0; s < kQRaw; ++s) {
            mbar_init(&ctl.qraw_full[s], 1);
            mbar_init(&ctl.qraw_empty[s], kConvThreads);
        }
        for (int s = 0; s < kQSlots; ++s) {
            mbar_init(&ctl.q8_full[s], kConvThreads);
            mbar_init(&ctl.q8_empty[s], kEpiThreads / 32);
        }
        for (int a = 0; a < kAccStages; ++a) {
            mbar_init(&ctl.tfull[a], 1);
            mbar_init(&ctl.tempty[a], kEpiThreads);
            mbar_init(&ctl.tmeta[a], 1);
        }
        mbar_init(&ctl.drain, 1);
        ctl.abort = 0;
        fence_mbar_init();
        tma_prefetch_map(&codes_map);
        tma_prefetch_map(&qraw_map);
        tma_prefetch_map(&w_map);
    }
    if (warp == 1) {
        tmem_alloc(&ctl.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    pdl_wait_prior_grid();
    pdl_allow_next_grid();
    if (warp == 1) build_row_table(rows, p, lane);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    const int total_units = rows.unit_start[batch];
    const uint32_t tmem_base = ctl.tmem_base;
    const int64_t M = p.row_width;

    if (warp == 0 || warp == 3) {
        // ================= producers: warp 0 issues the CTA's even units, warp 3 the odd ones =================
        // Both walk the same unit sequence (page ids fetched one batch ahead).  Per own unit:
        // lane 0 posts the metadata and issues the two code boxes; all 32 lanes copy the
        // unit's scales (cp.async, arriving on the stage's full barrier).  A row change is
        // numbered in sequence order; warp 0 stages every row's query and head weights for the
        // splitters, in that order, so that its waits on a raw-query slot are one phase apart.
        const int me = warp == 0 ? 0 : 1;
        const uint64_t pol_keys = l2_policy_evict_first();
        const uint64_t pol_q = l2_policy_evict_last();
        int seq = 0, nrows = 0, prev_b = -1, last_mine = -1;
        int q_mine[kQRaw];  // the last row-change numbers whose query this warp staged
#pragma unroll
        for (int j = 0; j < kQRaw; ++j) q_mine[j] = -1;
        bool stop = false;

        UnitSchedule sched(total_units);
        int cur_u0, cur_cnt;
        sched.next(cur_u0, cur_cnt);
        UnitPrep cur = prepare_units(rows, p, cur_u0, cur_cnt, lane);
        while (cur_cnt > 0 && !stop) {
            int nxt_u0, nxt_cnt;
            sched.next(nxt_u0, nxt_cnt);
            const UnitPrep nxt = prepare_units(rows, p, nxt_u0, nxt_cnt, lane);  // loads in flight
            for (int i = 0; i < cur_cnt; ++i, ++seq) {
                const int bi = __shfl_sync(0xffffffffu, cur.b, i);
                const bool new_row = bi != prev_b;
                if (new_row) {
                    ++nrows;
                    prev_b = bi;
                }
                int failed = 0;
                if (new_row && me == 0) {  // stage the request's query and head weights for the splitters
                    if (lane == 0) {
                        const int k = nrows - 1, qs = k % kQRaw;
                        if (!mbar_wait(&ctl.qraw_empty[qs], ((k / kQRaw) & 1) ^ 1u, &ctl.abort)) {
                            failed = 1;
                        } else {
                            ctl.qrow[qs] = bi;
                            mbar_arrive_expect_tx(&ctl.qraw_full[qs], kQRowBytes + kWRowBytes);
                            tma_load_2d(qraw + size_t(qs) * kQRowBytes, &qraw_map, &ctl.qraw_full[qs], 0,
                                        bi * kHeads, pol_q);
                            tma_load_2d(tiles + kOffWRaw + size_t(qs) * kWRowBytes, &w_map, &ctl.qraw_full[qs], 0,
                                        bi, pol_q);
#pragma unroll
                            for (int j = 0; j + 1 < kQRaw; ++j) q_mine[j] = q_mine[j + 1];
                            q_mine[kQRaw - 1] = k;
                        }
                    }
                    if (__shfl_sync(0xffffffffu, failed, 0)) {
                        stop = true;
                        break;
                    }
                }
                if ((seq & 1) != me) continue;  // the other producer's unit
                const int pi = __shfl_sync(0xffffffffu, cur.pair, i);
                const int g0 = __shfl_sync(0xffffffffu, cur.pg0, i);
                const int g1 = __shfl_sync(0xffffffffu, cur.pg1, i);
                const bool ok0 = g0 >= 0 && g0 < p.num_pages;
                const bool ok1 = g1 >= 0 && g1 < p.num_pages;
                const int stage = seq % kStages;
                if (lane == 0) {
                    if (!mbar_wait(&ctl.empty[stage], (uint32_t(seq / kStages) & 1u) ^ 1u, &ctl.abort))
                        failed = 1;
                    if (!failed) {
                        if (!ok0 || (g1 != -2 && !ok1)) atomicOr(p.err, kErrBadPage);
                        ctl.meta[seq % kRing] = pack_meta(bi, pi, ok0, ok1);
                        const uint32_t bytes = (ok0 ? kPageCodeBytes : 0) + (ok1 ? kPageCodeBytes : 0);
                        uint8_t* a = tiles + size_t(stage) * kStageBytes;
                        if (bytes != 0) {
                            mbar_arrive_expect_tx(&ctl.full[stage], bytes);
                            if (ok0) tma_load_3d(a, &codes_map, &ctl.full[stage], 0, 0, g0, pol_keys);
                            if (ok1) tma_load_3d(a + kPageCodeBytes, &codes_map, &ctl.full[stage], 0, 0, g1, pol_keys);
                        } else {
                            mbar_arrive(&ctl.full[stage]);  // nothing to load
                        }
                        last_mine = seq;
                    }
                }
                if (__shfl_sync(0xffffffffu, failed, 0)) {
                    stop = true;
                    break;
                }
                {  // lane l copies 16 B of scales: page l / 16, entries 4 (l % 16) .. + 3
                    const int g = lane < 16 ? g0 : g1;
                    const bool ok = lane < 16 ? ok0 : ok1;
                    if (ok)
                        cp_async_16(tiles + kOffScales + size_t(seq % kRing) * kUnitScaleBytes + lane * 16,
                                    p.key_scales + int64_t(g) * kPageEntries + (lane & 15) * 4);
                    cp_async_arrive_noinc(&ctl.full[stage]);
                }
            }
            cur_u0 = nxt_u0;
            cur_cnt = nxt_cnt;
            cur = nxt;
        }
        // End-of-work markers: the splitters' (row-change number nrows) from warp 0, which
        // stages every query; the MMA issuer's and epilogue's (unit number seq) from the warp
        // that owns that place.
        if (!stop && me == 0) {
            int failed = 0;
            if (lane == 0) {
                const int qs = nrows % kQRaw;
                if (!mbar_wait(&ctl.qraw_empty[qs], ((nrows / kQRaw) & 1) ^ 1u, &ctl.abort)) {
                    failed = 1;
                } else {
                    ctl.qrow[qs] = -1;
                    mbar_arrive(&ctl.qraw_full[qs]);
                }
            }
            if (__shfl_sync(0xffffffffu, failed, 0)) stop = true;
        }
        if (!stop && (seq & 1) == me) {
            const int stage = seq % kStages;
            int failed = 0;
            if (lane == 0) {
                if (!mbar_wait(&ctl.empty[stage], (uint32_t(seq / kStages) & 1u) ^ 1u, &ctl.abort)) {
                    failed = 1;
                } else {
                    ctl.meta[seq % kRing] = kEndOfWork;
                    mbar_arrive(&ctl.full[stage]);
                }
            }
            if (__shfl_sync(0xffffffffu, failed, 0)) stop = true;
            else cp_async_arrive_noinc(&ctl.full[stage]);
        }
        if (lane == 0 && stop) {
            atomicOr(p.err, kErrWaitTimeout);
            ctl.abort = 1;
        }
        if (lane == 0 && ctl.abort) {  // let every copy this warp issued land before the CTA may exit
            for (int s2 = last_mine; s2 >= 0 && s2 > last_mine - kStages; s2 -= 2)  // this warp's stages
                wait_landed(&ctl.full[s2 % kStages], uint32_t(s2 / kStages) & 1u);
#pragma unroll
            for (int j = 0; j < kQRaw; ++j)
                if (q_mine[j] >= 0) wait_landed(&ctl.qraw_full[q_mine[j] % kQRaw], uint32_t(q_mine[j] / kQRaw) & 1u);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");  // no scale copy outlives the CTA
    } else if (warp == 1) {
        // ================= MMA issuer (one lane) =================
        if (lane == 0) {
            int stage = 0, acc = 0, seq = 0, q_row = -1, q_used = -1;
            uint32_t phase = 0, acc_phase = 0;
            bool stop = false;
            while (true) {
                if (!mbar_wait(&ctl.full[stage], phase, &ctl.abort) ||
                    !mbar_wait(&ctl.tempty[acc], acc_phase ^ 1u, &ctl.abort)) {
                    stop = true;
                    break;
                }
                const int m = ctl.meta[seq % kRing];
                if (m != kEndOfWork) {
                    const int b = meta_row(m);
                    if (b != q_row) {
                        ++q_used;
                        q_row = b;
                        if (!mbar_wait(&ctl.q8_full[q_used % kQSlots], (q_used / kQSlots) & 1, &ctl.abort)) {
                            stop = true;
                            break;
                        }
                    }
                    tc_fence_after_sync();
                    const uint64_t a_desc = smem_desc_kmajor_sw64(smem_u32(tiles + size_t(stage) * kStageBytes));
                    const uint8_t* qt = q8 + size_t(q_used % kQSlots) * kQ8Bytes;
                    const uint64_t b_hi = smem_desc_kmajor_sw64(smem_u32(qt));
                    const uint32_t d_tmem = tmem_base + uint32_t(acc * kAccCols);
                    // K = 32 codes per MMA: +32 bytes = +2 in the address field.  The lo tile
                    // follows the hi tile (rows 32..63 of one N = 64 operand: with 64-byte rows the
                    // swizzle pattern repeats every 8 rows, so the two 32-row tiles are one tile).
#pragma unroll
                    for (int kk = 0; kk < kHeadDim / 32; ++kk)
                        umma_f8_ss(d_tmem, a_desc + 2u * kk, b_hi + 2u * kk, kIdesc, kk > 0 ? 1u : 0u);
                    umma_commit(&ctl.empty[stage]);
                    umma_commit(&ctl.tfull[acc]);
                }
                mbar_arrive(&ctl.tmeta[acc]);
                ++seq;
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (++acc == kAccStages) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
                if (m == kEndOfWork) break;
            }
            if (stop) {
                atomicOr(p.err, kErrWaitTimeout);
                ctl.abort = 1;
            }
            umma_commit(&ctl.drain);
            wait_landed(&ctl.drain, 0);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ================= the -inf fill of the rows' dead parts (full-width rows) =================
        if (p.fill_dead) fill_dead_tails_warp(rows, p, lane);
    } else if (warp >= 8) {
        // ================= query splitters: bf16 q -> hi/lo e4m3 tile and w_h * S_h =================
        // Two warps split each request's query: thread (sw, h) takes two of head h's four
        // 16-element chunks, c and c ^ 2 with c = (sw + h) mod 2 + 2 ((h >> 1) mod 2), and loads
        // the first or second 16-byte half of a chunk first by (h >> 2) mod 2, so that every
        // shared-memory access of a warp spreads over all eight 16-byte bank groups (one lane
        // per head reading whole rows hit one group 32 times).  The two partial maxima of a head
        // meet in shared memory.  Every splitter thread reaches both named barriers of every
        // round, so a wait that fails in one warp stops both together.
        const int sw = warp - 8;
        const int h = lane;
        const int c = ((sw + h) & 1) + 2 * ((h >> 1) & 1);
        const int v0 = (h >> 2) & 1;  // the chunk half loaded first
        bool stop = false;
        for (int j = 0;; ++j) {
            const int rs = j % kQRaw, qs = j % kQSlots;
            bool ok = mbar_wait(&ctl.qraw_full[rs], (j / kQRaw) & 1, &ctl.abort);
            const bool end = ok && ctl.qrow[rs] < 0;
            if (ok && !end) ok = mbar_wait(&ctl.q8_empty[qs], ((j / kQSlots) & 1) ^ 1u, &ctl.abort);
            if (lane == 0) ctl.split_flag[sw] = ok ? (end ? 2 : 1) : 0;
            split_bar_sync();
            const int fmin = min(ctl.split_flag[0], ctl.split_flag[1]);
            if (fmin == 0) {
                stop = true;
                break;
            }
            if (fmin == 2) break;  // the end marker
            // Thread (sw, h): chunks c and c ^ 2 of head h, c = (sw + h) mod 2 + 2 ((h >> 1) mod 2).
            const uint8_t* hrow = qraw + size_t(rs) * kQRowBytes + h * 128;
            uint4 u[2][2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const uint4* src = reinterpret_cast<const uint4*>(hrow + (c ^ (2 * k)) * 32);
                const uint4 ua = src[v0], ub = src[v0 ^ 1];
                u[k][0] = v0 ? ub : ua;
                u[k][1] = v0 ? ua : ub;
            }
            uint32_t amax_bits = 0;  // max |q| over the two chunks, on the bf16 magnitude bits
#pragma unroll
            for (int k = 0; k < 2; ++k)
#pragma unroll
                for (int v = 0; v < 2; ++v) {
                    const uint32_t wds[4] = {u[k][v].x, u[k][v].y, u[k][v].z, u[k][v].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        amax_bits = max(amax_bits, max(wds[i] & 0x7FFFu, (wds[i] >> 16) & 0x7FFFu));
                }
            ctl.split_amax[h][sw] = amax_bits;
            split_bar_sync();
            {
                const uint2 m2 = *reinterpret_cast<const uint2*>(ctl.split_amax[h]);
                amax_bits = max(m2.x, m2.y);
            }
            // S_h = 2^(e - 7) with e the exponent of the head's largest magnitude (clamped so
            // that S_h and 1 / S_h are normal floats); all-zero heads take e = 0.
            int e = amax_bits != 0 ? int(amax_bits >> 7) - 127 : 0;
            e = max(e, -119);
            const float inv_s = __uint_as_float(uint32_t(127 + 7 - e) << 23);
            const float s_h = __uint_as_float(uint32_t(127 + e - 7) << 23);
            uint8_t* tile = q8 + size_t(qs) * kQ8Bytes;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int ck = c ^ (2 * k);
                float x[16];
                const uint32_t wds[8] = {u[k][0].x, u[k][0].y, u[k][0].z, u[k][0].w,
                                         u[k][1].x, u[k][1].y, u[k][1].z, u[k][1].w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    x[2 * i] = __uint_as_float(wds[i] << 16) * inv_s;
                    x[2 * i + 1] = __uint_as_float(wds[i] & 0xFFFF0000u) * inv_s;
                }
                uint2 hi0, lo0, hi1, lo1;
                split8(x, hi0, lo0);
                split8(x + 8, hi1, lo1);
                const int swz = (ck ^ ((h >> 1) & 3)) << 4;  // 64-byte swizzle: 16-byte chunk ck of row h
                *reinterpret_cast<uint4*>(tile + h * 64 + swz) = make_uint4(hi0.x, hi0.y, hi1.x, hi1.y);
                *reinterpret_cast<uint4*>(tile + kQHalfBytes + h * 64 + swz) = make_uint4(lo0.x, lo0.y, lo1.x, lo1.y);
            }
            if (sw == 0) ctl.wq[qs][h] = wraw[rs * kHeads + h] * s_h;
            mbar_arrive(&ctl.qraw_empty[rs]);
            fence_proxy_async_smem();
            mbar_arrive(&ctl.q8_full[qs]);
        }
        if (stop && lane == 0) {
            atomicOr(p.err, kErrWaitTimeout);
            ctl.abort = 1;
        }
    } else if (warp >= 4 && warp < 8) {
        // ================= epilogue: warps 4..7 =================
        const int quad = warp & 3;         // TMEM lanes [32*quad, 32*quad + 32)
        const float neg_inf = __int_as_float(0xff800000);
        // The scores stay in L2 for the top-k that reads them next (the keys stream through
        // it evict-first); without the hint about two thirds of a dense 128K step's 8 MB of
        // scores were written back to HBM before the top-k read them.
        const uint64_t pol_row = l2_policy_evict_last();

        int cur_b = -1, n = 0, q_used = -1;
        const float* wv = ctl.wq[0];  // w_h * S_h of the current request (shared memory)
        bool stop = false;
        for (int i = 0;; ++i) {
            const int acc = i % kAccStages;
            const uint32_t acc_phase = uint32_t(i / kAccStages) & 1u;
            if (!__all_sync(0xffffffffu, mbar_wait(&ctl.tmeta[acc], acc_phase, &ctl.abort))) {
                stop = true;
                break;
            }
            const int m = ctl.meta[i % kRing];
            if (m == kEndOfWork) break;
            const int b = meta_row(m);
            const int pair = meta_pair(m);
            const bool page_ok = (m >> (quad >> 1)) & 1;
            const float key_scale = scale_ring[(i % kRing) * (kUnitScaleBytes / 4) + quad * 32 + lane];
            if (b != cur_b) {
                if (q_used >= 0 && lane == 0) mbar_arrive(&ctl.q8_empty[q_used % kQSlots]);  // done with that query
                ++q_used;
                wv = ctl.wq[q_used % kQSlots];
                n = rows.n_live[b];
                cur_b = b;
            }
            if (!__all_sync(0xffffffffu, mbar_wait(&ctl.tfull[acc], acc_phase, &ctl.abort))) {
                stop = true;
                break;
            }
            tc_fence_after_sync();
            const uint32_t taddr = tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(acc * kAccCols);
            float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
            {
                const float4* w4 = reinterpret_cast<const float4*>(wv);
#pragma unroll
                for (int half = 0; half < 2; ++half) {  // heads 16 half .. 16 half + 15
                    uint32_t hi[16], lo[16];
                    tmem_ld_32x32b_x16(taddr + uint32_t(16 * half), hi);
                    tmem_ld_32x32b_x16(taddr + uint32_t(kHeads + 16 * half), lo);
                    tmem_ld_wait16(hi);
                    tmem_ld_wait16(lo);
                    if (half == 1) {
                        tc_fence_before_sync();
                        mbar_arrive(&ctl.tempty[acc]);
                    }
#pragma unroll
                    for (int h4 = 0; h4 < 4; ++h4) {
                        const float4 wq = w4[4 * half + h4];
                        const float a0 = __uint_as_float(hi[4 * h4 + 0]) + __uint_as_float(lo[4 * h4 + 0]);
                        const float a1 = __uint_as_float(hi[4 * h4 + 1]) + __uint_as_float(lo[4 * h4 + 1]);
                        const float a2 = __uint_as_float(hi[4 * h4 + 2]) + __uint_as_float(lo[4 * h4 + 2]);
                        const float a3 = __uint_as_float(hi[4 * h4 + 3]) + __uint_as_float(lo[4 * h4 + 3]);
                        fma2(s0, s1, wq.x, wq.y, fmaxf(a0, 0.f), fmaxf(a1, 0.f));
                        fma2(s2, s3, wq.z, wq.w, fmaxf(a2, 0.f), fmaxf(a3, 0.f));
                    }
                }
            }
            const float s = key_scale * ((s0 + s1) + (s2 + s3));
            const int64_t t = int64_t(pair) * kUnitPositions + quad * 32 + lane;
            if (t < M) st_global_hint(p.out + int64_t(b) * M + t, (t < n && page_ok) ? s : neg_inf, pol_row);
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

template <int S>
cudaError_t launch_scores_fp8_s(const CUtensorMap& codes_map, const CUtensorMap& qraw_map, const CUtensorMap& w_map,
                                const ScoresParams& p, cudaStream_t stream) {
    static SmemLimitOnce smem_limit;  // the dynamic shared-memory limit, enough for any batch
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = smem_limit.apply(dev, scores_fp8_kernel<S>, int(Fp8Layout<S>::bytes(kMaxBatch)));
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(sms * kCtasPerSm));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Fp8Layout<S>::bytes(p.batch);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, scores_fp8_kernel<S>, codes_map, qraw_map, w_map, p);
}

}  // namespace

cudaError_t launch_scores_fp8(const CUtensorMap& codes_map, const CUtensorMap& qraw_map, const CUtensorMap& w_map,
                              const ScoresParams& p, cudaStream_t stream) {
    return launch_scores_fp8_s<kFp8Stages>(codes_map, qraw_map, w_map, p, stream);
}

}  // namespace dsa

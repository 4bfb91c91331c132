// scores_fp8_kernel.cu -- paged indexer scores on an fp8 key cache, sm_103a.
//
// Same scores as scores_kernel.cu,
//     score[b, t] = sum_h w[b, h] * max(0, q[b, h, :] . k[t, :]),  -inf past n_b,
// with each C4 key stored as 64 OCP e4m3 codes and one positive fp32 scale,
// k[t, d] = scale[t] * e4m3(code[t, d]).  The deployment on the pages keeps
// an fp8 KV cache ("The Indexer O(max_context) Breakthrough", section "The
// Indexer O(max_context) Breakthrough"); the scale format is not given there
// and is this library's choice.  Because the scale is positive,
// relu(scale * x) = scale * relu(x), so it is applied once per key after the
// head sum.  A key costs 68 bytes instead of 128.
//
// Pipeline (per CTA, two CTAs per SM, persistent grid sized by the device):
//   * warp 0: the unit schedule and page ids of scores_common.cuh; per unit
//     two 4 KiB TMA code boxes and two 256 B scale boxes into a raw ring;
//     query tiles into a 2-slot ring; unit metadata into a ring.
//   * warps 2-5 (converters): widen the 128 x 64 codes to bf16 (exact: every
//     e4m3 value is a bf16 value) straight into the 128-byte-swizzled K-major
//     tile the MMA reads, copy the 128 scales to a scale ring, release the
//     raw stage, fence the async proxy and publish the tile.
//   * warp 1: tcgen05.mma kind::f16 M=128 x N=32 x K=64 into one of 4 TMEM
//     accumulators, as in the bf16 kernel.
//   * warps 6-9: tcgen05.ld, relu, head weights and head sum in registers,
//     times the key's scale, live mask, 128-byte stores; the -inf fill of the
//     dead tail of every row when a full row is requested.
//   * Every wait is bounded (about 1 s); a timeout sets an error bit, stops
//     all roles, drains in-flight copies and MMAs and frees TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "indexer_kernels.h"
#include "scores_common.cuh"
#include "sm103_ptx.cuh"

namespace dsa {
namespace {

using namespace scores;

constexpr int kRawStages = 3;
constexpr int kATiles = 3;
constexpr int kQSlots = 2;
constexpr int kAccStages = 4;
constexpr int kMetaRing = 16;  // >= kRawStages + kATiles + kAccStages + 1
constexpr int kCtasPerSm = 2;
constexpr int kAccCols = 32;
constexpr uint32_t kTmemCols = kAccStages * kAccCols;  // 128
constexpr int kConvThreads = 128;
constexpr int kEpiThreads = 128;
constexpr int kThreads = 64 + kConvThreads + kEpiThreads;  // 320
constexpr int kATileBytes = 2 * kPageBytes;                 // 16 KiB of bf16: 128 keys x 128 B
constexpr int kRawBytes = 9216;                             // 2 x 4 KiB codes + 2 x 256 B scales, 1 KiB aligned
constexpr int kRawScaleOffset = 2 * kPageCodeBytes;
constexpr uint32_t kIdesc = idesc_bf16_f32(128, kAccCols);
static_assert(kMetaRing >= kRawStages + kATiles + kAccStages + 1, "metadata ring too small");
static_assert(kRawScaleOffset + 2 * kPageScaleBytes <= kRawBytes, "raw stage layout");

struct __align__(8) SmemCtl {
    uint64_t rfull[kRawStages];
    uint64_t rempty[kRawStages];
    uint64_t afull[kATiles];
    uint64_t aempty[kATiles];
    uint64_t qfull[kQSlots];
    uint64_t qempty[kQSlots];
    uint64_t tfull[kAccStages];
    uint64_t tempty[kAccStages];
    uint64_t tmeta[kAccStages];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int32_t meta[kMetaRing];
    float scale[kMetaRing][128];  // the unit's 128 key scales, by unit sequence number
    RowTable rows;
};

constexpr size_t kTileBytes = size_t(kATiles) * kATileBytes + size_t(kQSlots) * kQRowBytes +
                              size_t(kRawStages) * kRawBytes;
constexpr size_t kSmemBytes = 1024 /* alignment slack */ + kTileBytes + sizeof(SmemCtl);
static_assert(kSmemBytes * kCtasPerSm <= 228 * 1024, "shared memory budget per SM");

// Four e4m3 codes (lowest byte first) to four bf16 values, exactly.
__device__ __forceinline__ uint2 e4m3x4_to_bf16x4(uint32_t codes) {
    uint32_t h01, h23;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"(static_cast<unsigned short>(codes & 0xFFFFu)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"(static_cast<unsigned short>(codes >> 16)));
    const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
    const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
    const __nv_bfloat162 b01 = __float22bfloat162_rn(f01);
    const __nv_bfloat162 b23 = __float22bfloat162_rn(f23);
    return make_uint2(*reinterpret_cast<const uint32_t*>(&b01), *reinterpret_cast<const uint32_t*>(&b23));
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    scores_fp8_kernel(const __grid_constant__ CUtensorMap codes_map, const __grid_constant__ CUtensorMap scales_map,
                      const __grid_constant__ CUtensorMap q_map, const ScoresParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* atiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* qtiles = atiles + size_t(kATiles) * kATileBytes;
    uint8_t* raw = qtiles + size_t(kQSlots) * kQRowBytes;
    SmemCtl& ctl = *reinterpret_cast<SmemCtl*>(atiles + kTileBytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int batch = p.batch;

    // ---- set-up that touches no global memory (overlaps the previous kernel).
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRawStages; ++s) {
            mbar_init(&ctl.rfull[s], 1);
            mbar_init(&ctl.rempty[s], kConvThreads);
        }
        for (int s = 0; s < kATiles; ++s) {
            mbar_init(&ctl.afull[s], kConvThreads);
            mbar_init(&ctl.aempty[s], 1);
        }
        for (int s = 0; s < kQSlots; ++s) {
            mbar_init(&ctl.qfull[s], 1);
            mbar_init(&ctl.qempty[s], 1);
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
        tma_prefetch_map(&scales_map);
        tma_prefetch_map(&q_map);
    }
    if (warp == 1) {
        tmem_alloc(&ctl.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    pdl_wait_prior_grid();
    pdl_allow_next_grid();
    if (warp == 2) build_row_table(ctl.rows, p, lane);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    const int total_units = ctl.rows.unit_start[batch];
    const uint32_t tmem_base = ctl.tmem_base;
    const int64_t M = p.row_width;

    if (warp == 0) {
        // ================= producer: schedule, page ids, TMA of codes and scales =================
        const uint64_t pol_keys = l2_policy_evict_first();
        const uint64_t pol_q = l2_policy_evict_last();
        int stage = 0, issued = 0, q_issued = 0, q_row = -1, seq = 0;
        uint32_t phase = 0;
        bool stop = false;
        UnitSchedule sched(p, total_units, lane);
        int cur_u0, cur_cnt;
        sched.next(cur_u0, cur_cnt, lane);
        UnitPrep cur = prepare_units(ctl.rows, p, cur_u0, cur_cnt, lane);
        while (cur_cnt > 0 && !stop) {
            int nxt_u0, nxt_cnt;
            sched.next(nxt_u0, nxt_cnt, lane);
            const UnitPrep nxt = prepare_units(ctl.rows, p, nxt_u0, nxt_cnt, lane);  // loads in flight
            for (int i = 0; i < cur_cnt; ++i) {
                const int bi = __shfl_sync(0xffffffffu, cur.b, i);
                const int pi = __shfl_sync(0xffffffffu, cur.pair, i);
                const int g0 = __shfl_sync(0xffffffffu, cur.pg0, i);
                const int g1 = __shfl_sync(0xffffffffu, cur.pg1, i);
                int failed = 0;
                if (lane == 0) {
                    if (bi != q_row) {
                        const int qs = q_issued % kQSlots;
                        if (!mbar_wait(&ctl.qempty[qs], ((q_issued / kQSlots) & 1) ^ 1u, &ctl.abort)) {
                            failed = 1;
                        } else {
                            mbar_arrive_expect_tx(&ctl.qfull[qs], kQRowBytes);
                            tma_load_2d(qtiles + size_t(qs) * kQRowBytes, &q_map, &ctl.qfull[qs], 0, bi * kHeads,
                                        pol_q);
                            ++q_issued;
                            q_row = bi;
                        }
                    }
                    if (!failed && !mbar_wait(&ctl.rempty[stage], phase ^ 1u, &ctl.abort)) failed = 1;
                    if (!failed) {
                        const bool ok0 = g0 >= 0 && g0 < p.num_pages;
                        const bool ok1 = g1 >= 0 && g1 < p.num_pages;
                        if (!ok0 || (g1 != -2 && !ok1)) atomicOr(p.err, kErrBadPage);
                        ctl.meta[seq % kMetaRing] = pack_meta(bi, pi, ok0, ok1);
                        const uint32_t bytes = (ok0 ? kPageCodeBytes + kPageScaleBytes : 0) +
                                               (ok1 ? kPageCodeBytes + kPageScaleBytes : 0);
                        uint8_t* r = raw + size_t(stage) * kRawBytes;
                        if (bytes != 0) {
                            mbar_arrive_expect_tx(&ctl.rfull[stage], bytes);
                            if (ok0) {
                                tma_load_3d(r, &codes_map, &ctl.rfull[stage], 0, 0, g0, pol_keys);
                                tma_load_2d(r + kRawScaleOffset, &scales_map, &ctl.rfull[stage], 0, g0, pol_keys);
                            }
                            if (ok1) {
                                tma_load_3d(r + kPageCodeBytes, &codes_map, &ctl.rfull[stage], 0, 0, g1, pol_keys);
                                tma_load_2d(r + kRawScaleOffset + kPageScaleBytes, &scales_map, &ctl.rfull[stage], 0,
                                            g1, pol_keys);
                            }
                        } else {
                            mbar_arrive(&ctl.rfull[stage]);  // nothing to load
                        }
                        ++issued;
                    }
                }
                if (__shfl_sync(0xffffffffu, failed, 0)) {
                    stop = true;
                    break;
                }
                ++seq;
                if (++stage == kRawStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            cur_u0 = nxt_u0;
            cur_cnt = nxt_cnt;
            cur = nxt;
        }
        if (!stop) {  // end-of-work marker
            int failed = 0;
            if (lane == 0) {
                if (!mbar_wait(&ctl.rempty[stage], phase ^ 1u, &ctl.abort)) {
                    failed = 1;
                } else {
                    ctl.meta[seq % kMetaRing] = kEndOfWork;
                    mbar_arrive(&ctl.rfull[stage]);
                }
            }
            if (__shfl_sync(0xffffffffu, failed, 0)) stop = true;
            if (++stage == kRawStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (lane == 0 && stop) {
            atomicOr(p.err, kErrWaitTimeout);
            ctl.abort = 1;
        }
        if (lane == 0 && ctl.abort) {  // let every copy this CTA issued land before it may exit
            int s = stage;
            uint32_t ph = phase;
            for (int i = 0; i < min(issued, kRawStages); ++i) {
                if (s == 0) {
                    s = kRawStages - 1;
                    ph ^= 1u;
                } else {
                    --s;
                }
                wait_landed(&ctl.rfull[s], ph);
            }
            for (int j = max(0, q_issued - kQSlots); j < q_issued; ++j)
                wait_landed(&ctl.qfull[j % kQSlots], (j / kQSlots) & 1);
        }
    } else if (warp == 1) {
        // ================= MMA issuer (one lane) =================
        if (lane == 0) {
            int as = 0, acc = 0, seq = 0, q_row = -1, q_used = -1;
            uint32_t aphase = 0, acc_phase = 0;
            bool stop = false;
            while (true) {
                if (!mbar_wait(&ctl.afull[as], aphase, &ctl.abort) ||
                    !mbar_wait(&ctl.tempty[acc], acc_phase ^ 1u, &ctl.abort)) {
                    stop = true;
                    break;
                }
                const int m = ctl.meta[seq % kMetaRing];
                if (m != kEndOfWork) {
                    const int b = meta_row(m);
                    if (b != q_row) {
                        if (q_used >= 0) umma_commit(&ctl.qempty[q_used % kQSlots]);
                        ++q_used;
                        q_row = b;
                        if (!mbar_wait(&ctl.qfull[q_used % kQSlots], (q_used / kQSlots) & 1, &ctl.abort)) {
                            stop = true;
                            break;
                        }
                    }
                    tc_fence_after_sync();
                    const uint64_t a_desc = smem_desc_kmajor_sw128(smem_u32(atiles + size_t(as) * kATileBytes));
                    const uint64_t b_desc =
                        smem_desc_kmajor_sw128(smem_u32(qtiles + size_t(q_used % kQSlots) * kQRowBytes));
                    const uint32_t d_tmem = tmem_base + uint32_t(acc * kAccCols);
#pragma unroll
                    for (int kk = 0; kk < kHeadDim / 16; ++kk)
                        umma_bf16_ss(d_tmem, a_desc + 2u * kk, b_desc + 2u * kk, kIdesc, kk > 0 ? 1u : 0u);
                    umma_commit(&ctl.aempty[as]);
                    umma_commit(&ctl.tfull[acc]);
                }
                mbar_arrive(&ctl.tmeta[acc]);
                ++seq;
                if (++as == kATiles) {
                    as = 0;
                    aphase ^= 1u;
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
    } else if (warp < 6) {
        // ================= converters: e4m3 codes -> bf16 swizzled tile, scales =================
        const int ct = threadIdx.x - 64;  // 0..127
        const int cw = warp - 2;          // rows [32 cw, 32 cw + 32)
        const int half = lane >> 4;       // which of the two rows of an iteration
        const int col4 = lane & 15;       // codes [4 col4, 4 col4 + 4) of the row
        int rs = 0, as = 0, seq = 0;
        uint32_t rphase = 0, aphase = 0;
        bool stop = false;
        while (true) {
            if (!mbar_wait(&ctl.rfull[rs], rphase, &ctl.abort) ||
                !mbar_wait(&ctl.aempty[as], aphase ^ 1u, &ctl.abort)) {
                stop = true;
                break;
            }
            const int m = ctl.meta[seq % kMetaRing];
            if (m != kEndOfWork) {
                const uint8_t* r = raw + size_t(rs) * kRawBytes;
                uint8_t* tile = atiles + size_t(as) * kATileBytes;
#pragma unroll 4
                for (int it = 0; it < 16; ++it) {
                    const int row = 32 * cw + 2 * it + half;  // key row of the unit: page row >> 6, entry row & 63
                    const uint32_t codes =
                        *reinterpret_cast<const uint32_t*>(r + (row >> 6) * kPageCodeBytes + (row & 63) * kHeadDim +
                                                           4 * col4);
                    const uint2 v = e4m3x4_to_bf16x4(codes);
                    *reinterpret_cast<uint2*>(tile + row * 128 + (((col4 >> 1) ^ (row & 7)) << 4) + ((col4 & 1) << 3)) =
                        v;
                }
                ctl.scale[seq % kMetaRing][ct] =
                    *reinterpret_cast<const float*>(r + kRawScaleOffset + (ct >> 6) * kPageScaleBytes + (ct & 63) * 4);
            }
            mbar_arrive(&ctl.rempty[rs]);
            fence_proxy_async_smem();
            mbar_arrive(&ctl.afull[as]);
            ++seq;
            if (++rs == kRawStages) {
                rs = 0;
                rphase ^= 1u;
            }
            if (++as == kATiles) {
                as = 0;
                aphase ^= 1u;
            }
            if (m == kEndOfWork) break;
        }
        if (stop && lane == 0) {
            atomicOr(p.err, kErrWaitTimeout);
            ctl.abort = 1;
        }
    } else {
        // ================= epilogue: warps 6..9 =================
        const int et = threadIdx.x - 192;  // 0..127
        const int quad = warp & 3;         // TMEM lanes [32*quad, 32*quad + 32)
        const float neg_inf = __int_as_float(0xff800000);
        if (p.fill_dead) fill_dead_tails(ctl.rows, p, et, kEpiThreads);

        int cur_b = -1, n = 0;
        float wv[kHeads];
#pragma unroll
        for (int h = 0; h < kHeads; ++h) wv[h] = 0.f;
        bool stop = false;
        for (int i = 0;; ++i) {
            const int acc = i % kAccStages;
            const uint32_t acc_phase = uint32_t(i / kAccStages) & 1u;
            if (!__all_sync(0xffffffffu, mbar_wait(&ctl.tmeta[acc], acc_phase, &ctl.abort))) {
                stop = true;
                break;
            }
            const int m = ctl.meta[i % kMetaRing];
            if (m == kEndOfWork) break;
            const int b = meta_row(m);
            const int pair = meta_pair(m);
            const bool page_ok = (m >> (quad >> 1)) & 1;
            const float key_scale = ctl.scale[i % kMetaRing][quad * 32 + lane];
            if (b != cur_b) {
                const float4* wr = reinterpret_cast<const float4*>(p.w + int64_t(b) * kHeads);
#pragma unroll
                for (int h4 = 0; h4 < kHeads / 4; ++h4) {
                    const float4 v = __ldg(wr + h4);
                    wv[4 * h4 + 0] = v.x;
                    wv[4 * h4 + 1] = v.y;
                    wv[4 * h4 + 2] = v.z;
                    wv[4 * h4 + 3] = v.w;
                }
                n = ctl.rows.n_live[b];
                cur_b = b;
            }
            if (!__all_sync(0xffffffffu, mbar_wait(&ctl.tfull[acc], acc_phase, &ctl.abort))) {
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
            const float s = key_scale * ((s0 + s1) + (s2 + s3));
            const int64_t t = int64_t(pair) * kUnitPositions + quad * 32 + lane;
            if (t < M) p.out[int64_t(b) * M + t] = (t < n && page_ok) ? s : neg_inf;
        }
        if (stop && lane == 0) {
            atomicOr(p.err, kErrWaitTimeout);
            ctl.abort = 1;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0) release_schedule(p);
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_scores_fp8(const CUtensorMap& codes_map, const CUtensorMap& scales_map, const CUtensorMap& q_map,
                              const ScoresParams& p, cudaStream_t stream) {
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(scores_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes));
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(sms * kCtasPerSm));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, scores_fp8_kernel, codes_map, scales_map, q_map, p);
}

}  // namespace dsa

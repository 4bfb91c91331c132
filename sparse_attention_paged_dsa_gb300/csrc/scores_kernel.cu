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
//   * Persistent grid of kCtasPerSm CTAs per SM; its size depends only on the
//     device, so graph capture is safe and a 1M-token max_context launches the
//     same grid as an 8K one.
//   * Work unit = 2 consecutive pages of one request = 128 keys = 16 KiB.
//     Each CTA takes an equal contiguous range of floor(U / grid) of the
//     batch's U live units (few request changes per CTA), plus at most one of
//     the fewer than `grid` units left over; the schedule is fixed by U, the
//     grid and the CTA index.  Cost is O(live units), not O(max_context).
//   * Q query tokens per request (Q = 1 for the plain decode step; 2..4 for
//     multi-token decoding, row f3): the request's Q x 32 query heads form
//     the N = 32 Q side of one MMA per unit, so the key bytes are read once
//     for all Q tokens; token j of a request with seq_len L scores the
//     ceil((L - (Q - 1 - j)) / 4) keys of its own causal prefix and writes
//     row b Q + j.
//   * Two producer warps (one lane each issues) gather pages with TMA tiled
//     loads (128-byte swizzle) into a kStages ring of 16 KiB stages: warp 0
//     the CTA's even units, warp 2 the odd ones.  One issuing thread keeps
//     too few page boxes in flight to cover HBM latency; two per CTA do.
//     Page ids are fetched one batch ahead.  The request's 4 KiB query tile
//     is loaded once per request change into a small ring of its own.  Each
//     unit's request, page pair and page validity go to a small metadata
//     ring.
//   * Warp 1 (one lane) issues tcgen05.mma kind::f16, M=128 keys x N=32 Q
//     heads x K=64 dims (4 instructions of K=16) into one of kAccStages TMEM
//     accumulators of 32 Q fp32 columns, then publishes the accumulator and
//     the unit's metadata.
//   * kEpiGroups groups of 4 warps (group g takes every kEpiGroups-th unit)
//     read the accumulators with tcgen05.ld (thread = key row, registers =
//     32 heads), apply relu, the head weights and the head sum in registers,
//     mask, and store 128 contiguous fp32 scores per unit.
//   * Warp 3 builds the per-request table of live counts and unit offsets;
//     when a full-width row is requested it then streams -inf over the dead
//     part of every row (an equal share per CTA), beside the pipeline.
//   * Programmatic dependent launch: barrier and TMEM set-up overlap the tail
//     of the previous kernel; global memory is touched only after
//     griddepcontrol.wait.
//   * Every wait is bounded (about 1 s); a timeout sets an error bit, stops
//     all roles, drains in-flight copies and MMAs and frees TMEM.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "indexer_kernels.h"
#include "scores_common.cuh"
#include "sm103_ptx.cuh"


namespace dsa {
namespace {

using namespace scores;

// Per query-token count Q and stage count S.  Q = 1: three CTAs per SM, two
// TMA-issuing producer warps each: one issuing thread keeps too few page
// boxes in flight to cover HBM latency (a TMA instruction takes about 120
// cycles to issue), so each SM runs six issuers, with three stages each (four
// measured the same: at this depth the ring is not the limit).  Q = 2: also
// three CTAs per SM (three stages, two 64-column accumulators each, so that
// three CTAs' TMEM fits).  Q >= 3: the 32 Q-column accumulators need the TMEM
// of two CTAs per SM (four stages).
template <int Q, int S>
struct Cfg {
    static constexpr int kCtasPerSm = Q <= 2 ? 3 : 2;  // Q >= 3: the accumulators need the TMEM of 2
    static constexpr int kStages = S;                         // 16 KiB stages per CTA, shared by the producers
    static constexpr int kEpiGroups = Q >= 3 ? 2 : 1;         // epilogue groups of 4 warps (Q >= 3: Q passes per unit)
    static constexpr int kQSlots = 2;
    static constexpr int kAccStages = Q == 1 ? 4 : 2;
    static constexpr int kMetaRing = 16;                      // >= kStages + kAccStages + 1
    static constexpr int kAccCols = 32 * Q;                   // fp32 columns per accumulator (N = 32 Q heads)
    static constexpr uint32_t kTmemCols =                     // power of two >= 32
        kAccStages * kAccCols <= 128 ? 128u : 256u;
    static constexpr int kEpiThreads = 128 * kEpiGroups;
    static constexpr int kThreads = 128 + kEpiThreads;       // producers 0 and 2, MMA 1, set-up 3, epilogue 4..
    static constexpr int kStageBytes = 2 * kPageBytes;        // 16 KiB: 128 keys x 128 B
    static constexpr int kQTileBytes = Q * kQRowBytes;        // Q tokens x 32 heads x 64 dims of bf16
    static constexpr uint32_t kIdesc = idesc_bf16_f32(128, kAccCols);
    static_assert(kAccStages % kEpiGroups == 0, "each epilogue group owns whole accumulator stages");
    static_assert(kMetaRing >= kStages + kAccStages + 1, "metadata ring too small");
    static_assert(kAccStages * kAccCols <= int(kTmemCols), "accumulators fit the allocation");
    static_assert(int(kTmemCols) * kCtasPerSm <= 512, "TMEM columns per SM");
};

template <int Q, int S>
struct __align__(16) SmemCtl {
    uint64_t full[Cfg<Q, S>::kStages];
    uint64_t empty[Cfg<Q, S>::kStages];
    uint64_t qfull[Cfg<Q, S>::kQSlots];
    uint64_t qempty[Cfg<Q, S>::kQSlots];
    uint64_t tfull[Cfg<Q, S>::kAccStages];
    uint64_t tempty[Cfg<Q, S>::kAccStages];
    uint64_t tmeta[Cfg<Q, S>::kAccStages];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int32_t meta[Cfg<Q, S>::kMetaRing];
    __align__(16) float wtok[4 * Cfg<Q, S>::kEpiGroups][Q > 1 ? Q : 1][kHeads];  // Q > 1: each epilogue warp's copy of the head weights
};

// Shared memory: 1024-byte aligned tiles (stages, query slots), the control
// block, then the batch-sized row table.
template <int Q, int S>
struct Layout {
    static constexpr size_t kTileBytes =
        size_t(Cfg<Q, S>::kStages) * Cfg<Q, S>::kStageBytes + size_t(Cfg<Q, S>::kQSlots) * Cfg<Q, S>::kQTileBytes;
    static constexpr size_t kFixedBytes = 1024 /* alignment slack */ + kTileBytes + sizeof(SmemCtl<Q, S>);
    static constexpr size_t bytes(int batch) { return kFixedBytes + row_table_bytes(batch); }
    // Whether kCtasPerSm CTAs fit one SM's shared memory for this batch.
    static constexpr bool fits(int batch) { return bytes(batch) * Cfg<Q, S>::kCtasPerSm <= 226 * 1024; }
};
static_assert(Layout<1, 3>::fits(kMaxBatch) && Layout<2, 3>::fits(kMaxBatch) && Layout<3, 4>::fits(kMaxBatch) &&
                  Layout<4, 4>::fits(kMaxBatch),
              "shared memory budget per SM");

template <int Q, int S>
__global__ void __launch_bounds__(Cfg<Q, S>::kThreads, Cfg<Q, S>::kCtasPerSm)
    scores_kernel(const __grid_constant__ CUtensorMap keys_map, const __grid_constant__ CUtensorMap q_map,
                  const ScoresParams p) {
    using C = Cfg<Q, S>;
    constexpr int kStages = C::kStages, kEpiGroups = C::kEpiGroups, kQSlots = C::kQSlots;
    constexpr int kAccStages = C::kAccStages, kMetaRing = C::kMetaRing, kAccCols = C::kAccCols;
    constexpr int kStageBytes = C::kStageBytes, kQTileBytes = C::kQTileBytes;
    constexpr uint32_t kTmemCols = C::kTmemCols, kIdesc = C::kIdesc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* qtiles = tiles + size_t(kStages) * kStageBytes;
    SmemCtl<Q, S>& ctl = *reinterpret_cast<SmemCtl<Q, S>*>(tiles + Layout<Q, S>::kTileBytes);
    const RowTable rows = row_table_at(tiles + Layout<Q, S>::kTileBytes + sizeof(SmemCtl<Q, S>), p.batch);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int batch = p.batch;

    // ---- set-up that touches no global memory (overlaps the previous kernel).
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl.full[s], 1);
            mbar_init(&ctl.empty[s], 1);
        }
        for (int s = 0; s < kQSlots; ++s) {
            mbar_init(&ctl.qfull[s], 1);
            mbar_init(&ctl.qempty[s], 1);
        }
        for (int a = 0; a < kAccStages; ++a) {
            mbar_init(&ctl.tfull[a], 1);
            mbar_init(&ctl.tempty[a], 128);
            mbar_init(&ctl.tmeta[a], 1);
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
    pdl_wait_prior_grid();
    pdl_allow_next_grid();

    // ---- per-row live counts and unit prefix.
    if (warp == 3) build_row_table(rows, p, lane);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    const int total_units = rows.unit_start[batch];
    const uint32_t tmem_base = ctl.tmem_base;
    const int64_t M = p.row_width;

    if (warp == 3) {
        // ================= set-up warp, then the -inf fill of the rows' dead parts (full-width rows) =================
        if (p.fill_dead) fill_dead_tails_warp(rows, p, lane, Q);
    } else if (warp == 0 || warp == 2) {
        // ================= producers: warp 0 issues the CTA's even units, warp 2 the odd ones =================
        // Both walk the same unit sequence (page ids fetched one batch ahead); a row change is
        // numbered in sequence order and warp 0 loads every row's query tile, in that order, so
        // that its waits on a query slot are one phase apart (a slot's next load waits for the
        // release of the load before it, which it issued itself).
        const int me = warp >> 1;
        const uint64_t pol_keys = l2_policy_evict_first();
        const uint64_t pol_q = l2_policy_evict_last();
        int seq = 0, nrows = 0, prev_b = -1, last_mine = -1;
        int q_mine[kQSlots];  // the last row-change numbers whose query this warp loaded
#pragma unroll
        for (int j = 0; j < kQSlots; ++j) q_mine[j] = -1;
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
                if (new_row && me == 0) {  // this request's query tile goes to the row's q slot
                    if (lane == 0) {
                        const int k = nrows - 1, qs = k % kQSlots;
                        if (!mbar_wait(&ctl.qempty[qs], ((k / kQSlots) & 1) ^ 1u, &ctl.abort)) {
                            failed = 1;
                        } else {
                            mbar_arrive_expect_tx(&ctl.qfull[qs], kQTileBytes);
                            tma_load_2d(qtiles + size_t(qs) * kQTileBytes, &q_map, &ctl.qfull[qs], 0,
                                        bi * Q * kHeads, pol_q);
#pragma unroll
                            for (int j = 0; j + 1 < kQSlots; ++j) q_mine[j] = q_mine[j + 1];
                            q_mine[kQSlots - 1] = k;
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
                if (lane == 0) {
                    const int stage = seq % kStages;
                    const uint32_t phase = uint32_t(seq / kStages) & 1u;
                    if (!mbar_wait(&ctl.empty[stage], phase ^ 1u, &ctl.abort)) failed = 1;
                    if (!failed) {
                        const bool ok0 = g0 >= 0 && g0 < p.num_pages;
                        const bool ok1 = g1 >= 0 && g1 < p.num_pages;
                        if (!ok0 || (g1 != -2 && !ok1)) atomicOr(p.err, kErrBadPage);
                        ctl.meta[seq % kMetaRing] = pack_meta(bi, pi, ok0, ok1);
                        const uint32_t bytes = (ok0 ? kPageBytes : 0) + (ok1 ? kPageBytes : 0);
                        uint8_t* a = tiles + size_t(stage) * kStageBytes;
                        if (bytes != 0) {
                            mbar_arrive_expect_tx(&ctl.full[stage], bytes);
                            if (ok0) tma_load_3d(a, &keys_map, &ctl.full[stage], 0, 0, g0, pol_keys);
                            if (ok1) tma_load_3d(a + kPageBytes, &keys_map, &ctl.full[stage], 0, 0, g1, pol_keys);
                        } else {
                            mbar_arrive(&ctl.full[stage]);  // nothing to load: the stage is full at once
                        }
                        last_mine = seq;
                    }
                }
                if (__shfl_sync(0xffffffffu, failed, 0)) {
                    stop = true;
                    break;
                }
            }
            cur_u0 = nxt_u0;
            cur_cnt = nxt_cnt;
            cur = nxt;
        }
        // One end-of-work marker per epilogue group, each posted by the warp that owns its place.
        for (int e = 0; e < kEpiGroups && !stop; ++e) {
            const int s_end = seq + e;
            if ((s_end & 1) != me) continue;
            int failed = 0;
            if (lane == 0) {
                const int stage = s_end % kStages;
                if (!mbar_wait(&ctl.empty[stage], (uint32_t(s_end / kStages) & 1u) ^ 1u, &ctl.abort)) {
                    failed = 1;
                } else {
                    ctl.meta[s_end % kMetaRing] = kEndOfWork;
                    mbar_arrive(&ctl.full[stage]);
                }
            }
            if (__shfl_sync(0xffffffffu, failed, 0)) stop = true;
        }
        if (lane == 0 && stop) {
            atomicOr(p.err, kErrWaitTimeout);
            ctl.abort = 1;
        }
        // Let every copy this warp issued land before the CTA may exit.
        if (lane == 0 && ctl.abort) {
            for (int s2 = last_mine; s2 >= 0 && s2 > last_mine - kStages; s2 -= 2)  // this warp's stages
                wait_landed(&ctl.full[s2 % kStages], uint32_t(s2 / kStages) & 1u);
#pragma unroll
            for (int j = 0; j < kQSlots; ++j)
                if (q_mine[j] >= 0) wait_landed(&ctl.qfull[q_mine[j] % kQSlots], uint32_t(q_mine[j] / kQSlots) & 1u);
        }
    } else if (warp == 1) {
        // ================= MMA issuer (one lane) =================
        if (lane == 0) {
            int stage = 0, acc = 0, seq = 0, ends = 0;
            uint32_t phase = 0, acc_phase = 0;
            int q_row = -1, q_used = -1;
            bool stop = false;
            while (true) {
                bool ok = mbar_wait(&ctl.full[stage], phase, &ctl.abort);
                ok = ok && mbar_wait(&ctl.tempty[acc], acc_phase ^ 1u, &ctl.abort);
                if (!ok) {
                    stop = true;
                    break;
                }
                const int m = ctl.meta[seq % kMetaRing];
                if (m != kEndOfWork) {
                    const int b = meta_row(m);
                    if (b != q_row) {
                        if (q_used >= 0) umma_commit(&ctl.qempty[q_used % kQSlots]);  // after the last MMA on it
                        ++q_used;
                        q_row = b;
                        if (!mbar_wait(&ctl.qfull[q_used % kQSlots], (q_used / kQSlots) & 1, &ctl.abort)) {
                            stop = true;
                            break;
                        }
                    }
                    tc_fence_after_sync();
                    const uint64_t a_desc = smem_desc_kmajor_sw128(smem_u32(tiles + size_t(stage) * kStageBytes));
                    const uint64_t b_desc =
                        smem_desc_kmajor_sw128(smem_u32(qtiles + size_t(q_used % kQSlots) * kQTileBytes));
                    const uint32_t d_tmem = tmem_base + uint32_t(acc * kAccCols);
#pragma unroll
                    for (int kk = 0; kk < kHeadDim / 16; ++kk)  // K = 16 per MMA: +32 bytes = +2 in the address field
                        umma_bf16_ss(d_tmem, a_desc + 2u * kk, b_desc + 2u * kk, kIdesc, kk > 0 ? 1u : 0u);
                    umma_commit(&ctl.empty[stage]);
                    umma_commit(&ctl.tfull[acc]);
                }
                mbar_arrive(&ctl.tmeta[acc]);  // the unit's metadata (or the end marker) is readable
                ++seq;
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (++acc == kAccStages) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
                if (m == kEndOfWork && ++ends == kEpiGroups) break;
            }
            if (stop) {
                atomicOr(p.err, kErrWaitTimeout);
                ctl.abort = 1;
            }
            // Every MMA issued so far completes before TMEM is released.
            umma_commit(&ctl.drain);
            wait_landed(&ctl.drain, 0);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ================= epilogue: kEpiGroups groups of 4 warps =================
        const int group = (warp - 4) >> 2;  // takes the group-th, (group + kEpiGroups)-th, ... units
        const int quad = warp & 3;          // TMEM lanes [32*quad, 32*quad + 32)
        const float neg_inf = __int_as_float(0xff800000);
        // The scores stay in L2 for the top-k that reads them next (the keys stream through
        // it evict-first); without the hint about two thirds of a dense 128K step's 8 MB of
        // scores were written back to HBM before the top-k read them.
        const uint64_t pol_row = l2_policy_evict_last();


        int cur_b = -1, n = 0;
        int n_tok[Q];  // live keys of each token of the current request
        float wv[Q == 1 ? kHeads : 1];
#pragma unroll
        for (int h = 0; h < (Q == 1 ? kHeads : 1); ++h) wv[h] = 0.f;
#pragma unroll
        for (int j = 0; j < Q; ++j) n_tok[j] = 0;
        bool stop = false;
        for (int i = group;; i += kEpiGroups) {
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
            const bool page_ok = (m >> (quad >> 1)) & 1;  // quadrants 0-1: first page, 2-3: second
            if (b != cur_b) {
                if constexpr (Q == 1) {
                    const float4* wr = reinterpret_cast<const float4*>(p.w + int64_t(b) * kHeads);
#pragma unroll
                    for (int h4 = 0; h4 < kHeads / 4; ++h4) {
                        const float4 v = __ldg(wr + h4);
                        wv[4 * h4 + 0] = v.x;
                        wv[4 * h4 + 1] = v.y;
                        wv[4 * h4 + 2] = v.z;
                        wv[4 * h4 + 3] = v.w;
                    }
                    n_tok[0] = rows.n_live[b];
                } else {  // this warp's copy of the Q x 32 head weights; per-token causal lengths
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < Q; ++j) ctl.wtok[warp - 4][j][lane] = __ldg(p.w + (int64_t(b) * Q + j) * kHeads + lane);
                    __syncwarp();
                    int64_t L = p.seq_lens[b];
                    L = L < 0 ? 0 : (L > p.max_context ? p.max_context : L);
#pragma unroll
                    for (int j = 0; j < Q; ++j) {
                        const int64_t Lj = L - (Q - 1 - j);
                        n_tok[j] = Lj > 0 ? int((Lj + 3) >> 2) : 0;
                    }
                }
                n = rows.n_live[b];
                cur_b = b;
            }
            const bool okf = mbar_wait(&ctl.tfull[acc], acc_phase, &ctl.abort);
            if (!__all_sync(0xffffffffu, okf)) {
                stop = true;
                break;
            }
            tc_fence_after_sync();
            const int64_t t = int64_t(pair) * kUnitPositions + quad * 32 + lane;
            const uint32_t taddr = tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(acc * kAccCols);
            if constexpr (Q == 1) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(taddr, r);
                tmem_ld_wait(r);
                tc_fence_before_sync();
                mbar_arrive(&ctl.tempty[acc]);

                float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;  // heads h = 0, 1, 2, 3 mod 4
#pragma unroll
                for (int h = 0; h < kHeads; h += 4) {
                    fma2(s0, s1, wv[h + 0], wv[h + 1], fmaxf(__uint_as_float(r[h + 0]), 0.f),
                         fmaxf(__uint_as_float(r[h + 1]), 0.f));
                    fma2(s2, s3, wv[h + 2], wv[h + 3], fmaxf(__uint_as_float(r[h + 2]), 0.f),
                         fmaxf(__uint_as_float(r[h + 3]), 0.f));
                }
                const float s = (s0 + s1) + (s2 + s3);
                if (t < M) st_global_hint(p.out + int64_t(b) * M + t, (t < n && page_ok) ? s : neg_inf, pol_row);
            } else {
                // Token j's logits are accumulator columns [32 j, 32 j + 32), read in halves of 16:
                // the load of the next half is in flight while the current one is summed.
                uint32_t ra[16], rb[16];
                tmem_ld_32x32b_x16(taddr, ra);
                tmem_ld_wait16(ra);
                float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;  // heads h = 0, 1, 2, 3 mod 4
#pragma unroll
                for (int hh = 0; hh < 2 * Q; ++hh) {
                    const int j = hh >> 1;
                    if (hh + 1 < 2 * Q) {
                        tmem_ld_32x32b_x16(taddr + uint32_t(16 * (hh + 1)), rb);
                    } else {  // every load from this accumulator has completed
                        tc_fence_before_sync();
                        mbar_arrive(&ctl.tempty[acc]);
                    }
                    const float4* wr = reinterpret_cast<const float4*>(ctl.wtok[warp - 4][j]) + 4 * (hh & 1);
#pragma unroll
                    for (int h4 = 0; h4 < 4; ++h4) {
                        const float4 wq = wr[h4];
                        fma2(s0, s1, wq.x, wq.y, fmaxf(__uint_as_float(ra[4 * h4 + 0]), 0.f),
                             fmaxf(__uint_as_float(ra[4 * h4 + 1]), 0.f));
                        fma2(s2, s3, wq.z, wq.w, fmaxf(__uint_as_float(ra[4 * h4 + 2]), 0.f),
                             fmaxf(__uint_as_float(ra[4 * h4 + 3]), 0.f));
                    }
                    if (hh & 1) {  // token j complete
                        const float s = (s0 + s1) + (s2 + s3);
                        if (t < M)
                            st_global_hint(p.out + (int64_t(b) * Q + j) * M + t,
                                           (t < n_tok[j] && page_ok) ? s : neg_inf, pol_row);
                        s0 = s1 = s2 = s3 = 0.f;
                    }
                    if (hh + 1 < 2 * Q) {
                        tmem_ld_wait16(rb);
#pragma unroll
                        for (int c = 0; c < 16; ++c) ra[c] = rb[c];
                    }
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

template <int Q, int S>
cudaError_t launch_scores_q(const CUtensorMap& keys_map, const CUtensorMap& q_map, const ScoresParams& p,
                            cudaStream_t stream) {
    static SmemLimitOnce smem_limit;  // the dynamic shared-memory limit, enough for any batch
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = smem_limit.apply(dev, scores_kernel<Q, S>, int(Layout<Q, S>::bytes(kMaxBatch)));
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(sms * Cfg<Q, S>::kCtasPerSm));
    cfg.blockDim = dim3(Cfg<Q, S>::kThreads);
    cfg.dynamicSmemBytes = Layout<Q, S>::bytes(p.batch);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, scores_kernel<Q, S>, keys_map, q_map, p);
}

}  // namespace

cudaError_t launch_scores(const CUtensorMap& keys_map, const CUtensorMap& q_map, const ScoresParams& p,
                          cudaStream_t stream) {
    switch (p.tokens) {
        case 1: return launch_scores_q<1, 3>(keys_map, q_map, p, stream);
        case 2: return launch_scores_q<2, 3>(keys_map, q_map, p, stream);
        case 3: return launch_scores_q<3, 4>(keys_map, q_map, p, stream);
        case 4: return launch_scores_q<4, 4>(keys_map, q_map, p, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace dsa

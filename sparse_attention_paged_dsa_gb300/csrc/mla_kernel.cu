// mla_kernel.cu -- sparse multi-head latent attention decode over the indexer's
// top-k entries, sm_103a.
//
//     s[h, t] = sm_scale * q[b, h] . kv_t            (576-wide entries)
//     o[b, h] = sum_t softmax_t(s[h, :]) kv_t[:512],  lse[b, h] = log sum_t exp(s[h, t])
//
// over the used entries t of request b's top-k row, each entry gathered through
// the page table ("The Indexer O(max_context) Breakthrough", sections "Phase 1:
// The MMA Sparse-MLA Decode Kernel" -- one gathered tile serves every head --
// and "Phase 2: Split-K Parallelization" -- the top-k list split across CTAs
// and merged by log-sum-exp).
//
// One CTA per (split, request), one CTA per SM (all of shared memory and
// TMEM).  The request's non-empty 64-entry blocks of the top-k row are divided
// into `splits` contiguous ranges; a CTA streams its blocks:
//   * warps 0, 2, 3: gather every block's 64 entries by TMA row gathers
//     (tile::gather4: four cache rows of 64 dims per instruction, from a
//     tensor map over the cache viewed as [pages x 64 rows, 576]) into nine
//     128-byte-swizzled slabs of 64 rows x 64 dims (a ring of 8 slab pairs for
//     the 512 value dims, 2 slabs for the rotary 64); each warp gathers a
//     third of every slab's 4-row groups, one group per lane.  Unused entries
//     repeat the row of the block's first used entry (their weights are 0).
//     Warp 0 also loads q once by TMA.
//   * warp 1: tcgen05.mma kind::f16 --
//       MMA1  S[head, entry] = Q . K^T, M = 64 heads, N = 64 entries, K = 576
//             (36 instructions; TMEM rows 16 q + i in lanes 32 q + i, i < 16);
//       MMA2  O^T[dim, head] += V^T . P^T, M = 128 dims x 4, N = 64 heads,
//             K = 64 entries, V read in place as an MN-major operand; the four
//             accumulators' instructions interleaved.
//   * warps 4-7: softmax.  Lanes 0-15 of each hold one head's 64 scores in
//     registers: block max, 2^x, row sum, P row (bf16) to shared memory.  The
//     running max is raised only when a block exceeds it by more than 2^8; then
//     all four warps rescale O^T in TMEM (tcgen05.ld / st) before MMA2.  At the
//     end they normalise O^T into the drained value ring and store o (or the
//     split's partial) with bulk copies, and write lse.
// MMA1(n+1) is issued after MMA2(n), so one S accumulator and one P buffer
// suffice and each completion barrier orders everything before it.  Every wait
// is bounded (about 1 s); a timeout sets an error bit, the roles drain, and
// TMEM is freed.
//
// What bounds it: a gathered row is 9 separate 128-byte segments; a 2-block
// ring (all the shared memory beside q) holds one block in flight while the
// previous one is computed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "indexer_kernels.h"
#include "sm103_ptx.cuh"

namespace dsa {
namespace {

constexpr int kBlk = 64;                       // entries per block
constexpr int kSlabBytes = kBlk * 128;         // 64 rows x 64 bf16 dims, 8 KiB
constexpr int kPairBytes = 2 * kSlabBytes;     // value dims [128 j, 128 j + 128)
constexpr int kVRing = 8;                      // slab pairs (two blocks' values)
constexpr int kRRing = 2;                      // rotary slabs
constexpr int kQSlabs = kMlaDim / 64;          // 9
constexpr int kOffQ = 0;
constexpr int kOffP = kOffQ + kQSlabs * kSlabBytes;  // P [64 heads x 64 entries] bf16 (also the
                                                     // ignored rows 64..127 of q's last slab)
constexpr int kOffV = kOffP + kSlabBytes;
constexpr int kOffR = kOffV + kVRing * kPairBytes;
constexpr int kOffCtl = kOffR + kRRing * kSlabBytes;
constexpr int kThreadsM = 256;
constexpr int kProducers = 3;    // warps 0, 2, 3: each gathers row groups k = p, p + 3, ... of every slab
constexpr int kRowGroups = 16;   // 4 rows x 128 bytes per gather
constexpr uint32_t kTmemColsM = 512;
constexpr uint32_t kColS = 0;    // S: 64 columns
constexpr uint32_t kColO = 128;  // O^T: 4 x 64 columns
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.69314718055994531f;

struct __align__(8) MlaCtl {
    uint64_t v_full[kVRing], v_empty[kVRing];
    uint64_t r_full[kRRing], r_empty[kRRing];
    uint64_t q_full, s_full, p_full, o_done;
    uint32_t tmem_base;
    uint32_t blk_mask;
    int abort;
    int nblk;
    int blocks[kMlaMaxTopk / kBlk];
    float alpha[kMlaHeads];
    float inv_l[kMlaHeads];
};
constexpr int kSmemM = 1024 + kOffCtl + int(sizeof(MlaCtl));
static_assert(kSmemM <= 232448, "fits one CTA per SM");
static_assert(kVRing * kPairBytes == kMlaHeads * kMlaDv * 4, "o fits the value ring");

__device__ __forceinline__ uint64_t desc_mn_sw128(uint32_t addr, uint32_t mn_stride) {
    // MN-major, 128-byte swizzle: atoms of 8 K-rows x 64 MN elements (1024 B); atoms
    // repeat along MN every mn_stride bytes (leading offset), along K every 1024 B.
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((mn_stride >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 2^x by the hardware's approximate base-2 exponential (flushes subnormal results to zero).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Bulk copy of `bytes` (multiple of 16) from shared to global memory, tracked by this
// thread's bulk-async group.
__device__ __forceinline__ void bulk_store(void* gdst, uint32_t ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc), "r"(bytes)
                 : "memory");
}

// TMA row gather: rows y0..y3 of a 2-D tensor map (box = one row of 64 bf16), columns
// [x, x + 64), into 4 x 128 bytes at `dst` (swizzled by the map, like a 4-row tile).
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, uint64_t* bar, int32_t x,
                                            int32_t y0, int32_t y1, int32_t y2, int32_t y3, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(smem_u32(bar)),
        "l"(policy)
        : "memory");
}

// Bounded wait for a phase of `bar` (only while draining after an abort).
__device__ __forceinline__ void wait_landed_m(uint64_t* bar, uint32_t parity) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(a, parity) && global_timer_ns() - t0 < kWaitLimitNs) {
    }
}

// Named barrier over the 128 softmax threads returning the OR of `v`.
__device__ __forceinline__ bool softmax_bar_or(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, 1, 128, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void softmax_bar_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Entry e of request b is used when it lies in the row and points inside the live length.
__device__ __forceinline__ int entry_pos(const MlaParams& p, int b, int e, int n_live) {
    if (e >= p.k) return -1;
    const int t = __ldg(p.topk + int64_t(b) * p.k + e);
    return (t >= 0 && t < n_live) ? t : -1;
}

__global__ void __launch_bounds__(kThreadsM, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap kv_map,
                      const MlaParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    MlaCtl& ctl = *reinterpret_cast<MlaCtl*>(tiles + kOffCtl);
    const uint32_t s_base = smem_u32(tiles);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int split = blockIdx.x;
    const int b = blockIdx.y;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kVRing; ++i) {
            mbar_init(&ctl.v_full[i], kProducers);  // one expect-tx arrival per producer warp
            mbar_init(&ctl.v_empty[i], 1);
        }
        for (int i = 0; i < kRRing; ++i) {
            mbar_init(&ctl.r_full[i], kProducers);
            mbar_init(&ctl.r_empty[i], 1);
        }
        mbar_init(&ctl.q_full, 1);
        mbar_init(&ctl.s_full, 1);
        mbar_init(&ctl.p_full, 128);
        mbar_init(&ctl.o_done, 1);
        ctl.abort = 0;
        ctl.blk_mask = 0;
        fence_mbar_init();
        tma_prefetch_map(&q_map);
        tma_prefetch_map(&kv_map);
    }
    if (warp == 1) {
        tmem_alloc(&ctl.tmem_base, kTmemColsM);
        tmem_relinquish();
    }
    pdl_wait_prior_grid();  // the top-k row may come from the previous kernel
    pdl_allow_next_grid();

    // Live length (C4 entries) of the request.
    int seq = __ldg(p.seq_lens + b);
    if (seq < 0 || int64_t(seq) > p.max_context) {
        if (threadIdx.x == 0 && split == 0) atomicOr(p.err, kErrSeqLenClamped);
        seq = seq < 0 ? 0 : int(p.max_context);
    }
    const int n_live = (seq + 3) >> 2;

    // Which 64-entry blocks of the row hold a used entry.
    __syncthreads();
    const int nb_row = (p.k + kBlk - 1) / kBlk;
    for (int blk = warp; blk < nb_row; blk += kThreadsM / 32) {
        const bool u0 = entry_pos(p, b, blk * kBlk + lane, n_live) >= 0;
        const bool u1 = entry_pos(p, b, blk * kBlk + 32 + lane, n_live) >= 0;
        if (__any_sync(0xffffffffu, u0 || u1) && lane == 0) atomicOr(&ctl.blk_mask, 1u << blk);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0) {  // this split's contiguous share of the non-empty blocks, in row order
        const uint32_t mask = ctl.blk_mask;
        const int total = __popc(mask);
        const int lo = int((int64_t(total) * split) / p.splits);
        const int hi = int((int64_t(total) * (split + 1)) / p.splits);
        int rank = 0, n = 0;
        for (int blk = 0; blk < nb_row; ++blk) {
            if (!((mask >> blk) & 1u)) continue;
            if (rank >= lo && rank < hi) ctl.blocks[n++] = blk;
            ++rank;
        }
        ctl.nblk = n;
    }
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = ctl.tmem_base;
    const int nblk = ctl.nblk;
    float* o_dst = p.splits == 1 ? p.out + int64_t(b) * kMlaHeads * kMlaDv
                                 : p.o_part + (int64_t(b) * p.splits + split) * kMlaHeads * kMlaDv;
    float* lse_dst = p.splits == 1 ? p.lse + int64_t(b) * kMlaHeads
                                   : p.lse_part + (int64_t(b) * p.splits + split) * kMlaHeads;

    if (warp == 0 || warp == 2 || warp == 3) {
        // ================= producers: gather the blocks' entries =================
        const int pw = warp == 0 ? 0 : warp - 1;
        bool stop = false;
        if (warp == 0 && lane == 0 && nblk > 0) {
            mbar_arrive_expect_tx(&ctl.q_full, uint32_t(kQSlabs * kSlabBytes));
            const uint64_t pol = l2_policy_evict_first();
            for (int s = 0; s < kQSlabs; ++s)
                tma_load_2d(tiles + kOffQ + s * kSlabBytes, &q_map, &ctl.q_full, s * 64, b * kMlaHeads, pol);
        }
        const uint64_t pol_kv = l2_policy_evict_first();
        // Lane i < ngw gathers row group k = pw + 3 i (rows 4k .. 4k + 3) of every slab.
        const int ngw = (kRowGroups - pw + kProducers - 1) / kProducers;
        const int k = pw + kProducers * lane;
        int last_v = -1, last_r = -1;  // the last value / rotary fills this warp took part in
#pragma unroll 1
        for (int n = 0; n < nblk && !stop; ++n) {
            const int blk = ctl.blocks[n];
            // cache rows of entries lane and lane + 32 (-1: unused or on a bad page)
            int row[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int t = entry_pos(p, b, blk * kBlk + h * 32 + lane, n_live);
                row[h] = -1;
                if (t >= 0) {
                    const int page = __ldg(p.page_table + int64_t(b) * p.table_width + (t >> 6));
                    if (page >= 0 && int64_t(page) < p.num_pages)
                        row[h] = page * kPageEntries + (t & 63);
                    else
                        atomicOr(p.err, kErrBadPage);
                }
            }
            // Rows of unused entries repeat the block's first used row (row 0 if none is readable):
            // every gathered row is one the request uses, and its softmax weight there is 0.
            const uint32_t u0 = __ballot_sync(0xffffffffu, row[0] >= 0);
            const uint32_t u1 = __ballot_sync(0xffffffffu, row[1] >= 0);
            const int f0 = __shfl_sync(0xffffffffu, row[0], u0 ? __ffs(u0) - 1 : 0);
            const int f1 = __shfl_sync(0xffffffffu, row[1], u1 ? __ffs(u1) - 1 : 0);
            const int first = u0 ? f0 : (u1 ? f1 : 0);
            row[0] = row[0] >= 0 ? row[0] : first;
            row[1] = row[1] >= 0 ? row[1] : first;
            int y[4];  // rows of this lane's group (entries 4k .. 4k + 3)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int e = 4 * k + c;
                const int a0 = __shfl_sync(0xffffffffu, row[0], e & 31);
                const int a1 = __shfl_sync(0xffffffffu, row[1], e & 31);
                y[c] = e < 32 ? a0 : a1;
            }
#pragma unroll 1
            for (int j = 0; j <= 4; ++j) {  // value pairs 0..3, then the rotary slab
                uint64_t* full;
                uint32_t dst_base;
                int nslabs, slab0;
                if (j < 4) {
                    const int pos = 4 * n + j, slot = pos & (kVRing - 1), use = pos / kVRing;
                    const bool ok = lane != 0 || mbar_wait(&ctl.v_empty[slot], uint32_t(use & 1) ^ 1u, &ctl.abort);
                    if (!__all_sync(0xffffffffu, ok)) {  // the lanes stop together
                        stop = true;
                        break;
                    }
                    full = &ctl.v_full[slot];
                    dst_base = s_base + kOffV + slot * kPairBytes;
                    nslabs = 2;
                    slab0 = 2 * j;
                    last_v = pos;
                } else {
                    const int slot = n & (kRRing - 1), use = n / kRRing;
                    const bool ok = lane != 0 || mbar_wait(&ctl.r_empty[slot], uint32_t(use & 1) ^ 1u, &ctl.abort);
                    if (!__all_sync(0xffffffffu, ok)) {
                        stop = true;
                        break;
                    }
                    full = &ctl.r_full[slot];
                    dst_base = s_base + kOffR + slot * kSlabBytes;
                    nslabs = 1;
                    slab0 = 8;
                    last_r = n;
                }
                if (lane == 0) mbar_arrive_expect_tx(full, uint32_t(ngw * nslabs * 4 * 128));
                __syncwarp();
                if (lane < ngw) {
                    for (int hs = 0; hs < nslabs; ++hs)
                        tma_gather4(dst_base + hs * kSlabBytes + k * 512, &kv_map, full, (slab0 + hs) * 64, y[0], y[1],
                                    y[2], y[3], pol_kv);
                }
            }
        }
        if (stop && lane == 0) {
            atomicOr(p.err, kErrWaitTimeout);
            ctl.abort = 1;
        }
        if (lane == 0 && ctl.abort) {  // no gather this warp issued outlives the CTA (bounded waits)
            for (int pos = last_v; pos >= 0 && pos > last_v - kVRing; --pos)
                wait_landed_m(&ctl.v_full[pos & (kVRing - 1)], uint32_t(pos / kVRing) & 1u);
            for (int n = last_r; n >= 0 && n > last_r - kRRing; --n)
                wait_landed_m(&ctl.r_full[n & (kRRing - 1)], uint32_t(n / kRRing) & 1u);
        }
        if (warp == 0 && lane == 0 && nblk > 0) {  // nor the q load
            const uint32_t addr = smem_u32(&ctl.q_full);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(addr, 0) && global_timer_ns() - t0 < kWaitLimitNs) {
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            constexpr uint32_t kIdesc1 = idesc_bf16_f32(64, 64);  // S: 64 heads x 64 entries
            constexpr uint32_t kIdesc2 = idesc_bf16_f32(128, 64) | (1u << 15);  // A (V^T) MN-major
            const uint32_t q_addr = s_base + kOffQ;
            const uint32_t p_addr = s_base + kOffP;
            bool stop = nblk > 0 && !mbar_wait(&ctl.q_full, 0, &ctl.abort);
#pragma unroll 1
            for (int n = 0; n < nblk && !stop; ++n) {
                int vslot[4];
#pragma unroll 1
                for (int j = 0; j < 4; ++j) {  // MMA1 over the value dims, slab pair by slab pair
                    const int pos = 4 * n + j, slot = pos & (kVRing - 1), use = pos / kVRing;
                    vslot[j] = slot;
                    if (!mbar_wait(&ctl.v_full[slot], uint32_t(use & 1), &ctl.abort)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after_sync();
#pragma unroll
                    for (int hs = 0; hs < 2; ++hs) {
                        const int s = 2 * j + hs;
                        const uint32_t kslab = s_base + kOffV + slot * kPairBytes + hs * kSlabBytes;
                        const uint64_t a = smem_desc_kmajor_sw128(q_addr + s * kSlabBytes);
                        const uint64_t bd = smem_desc_kmajor_sw128(kslab);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_bf16_ss(tmem_base + kColS, a + 2u * kk, bd + 2u * kk, kIdesc1,
                                         (s | kk) != 0 ? 1u : 0u);
                    }
                }
                if (stop) break;
                {  // rotary dims
                    const int slot = n & (kRRing - 1), use = n / kRRing;
                    if (!mbar_wait(&ctl.r_full[slot], uint32_t(use & 1), &ctl.abort)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint64_t a = smem_desc_kmajor_sw128(q_addr + 8 * kSlabBytes);
                    const uint64_t bd = smem_desc_kmajor_sw128(s_base + kOffR + slot * kSlabBytes);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16_ss(tmem_base + kColS, a + 2u * kk, bd + 2u * kk, kIdesc1, 1u);
                    umma_commit(&ctl.r_empty[slot]);
                }
                umma_commit(&ctl.s_full);
                if (!mbar_wait(&ctl.p_full, uint32_t(n & 1), &ctl.abort)) {
                    stop = true;
                    break;
                }
                tc_fence_after_sync();
                const uint64_t bp = smem_desc_kmajor_sw128(p_addr);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {  // MMA2: dims [128 j, 128 j + 128), the four interleaved
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        umma_bf16_ss(tmem_base + kColO + 64u * j,
                                     desc_mn_sw128(s_base + kOffV + vslot[j] * kPairBytes + kk * 2048, kSlabBytes),
                                     bp + 2u * kk, kIdesc2, (n > 0 || kk > 0) ? 1u : 0u);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) umma_commit(&ctl.v_empty[vslot[j]]);
            }
            if (stop) {
                atomicOr(p.err, kErrWaitTimeout);
                ctl.abort = 1;
            }
            umma_commit(&ctl.o_done);  // every MMA issued has completed when this arrives
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ================= softmax and output: warps 4..7 =================
        const int quad = warp & 3;
        // MMA1 (M = 64) leaves head 16 q + i in TMEM lane 32 q + i, i < 16: lanes 0..15 of each
        // softmax warp own one head each
        const bool head_thr = lane < 16;
        const int h = quad * 16 + (lane & 15);
        const uint32_t lane_addr = tmem_base + (uint32_t(quad * 32) << 16);
        const float c2 = p.sm_scale_log2;
        float m_used = -INFINITY, l_sum = 0.f;
        bool failed = false;
        uint8_t* prow = tiles + kOffP + h * 128;
#pragma unroll 1
        for (int n = 0; n < nblk; ++n) {
            const int blk = ctl.blocks[n];
            const uint32_t u_lo = __ballot_sync(0xffffffffu, entry_pos(p, b, blk * kBlk + lane, n_live) >= 0);
            const uint32_t u_hi = __ballot_sync(0xffffffffu, entry_pos(p, b, blk * kBlk + 32 + lane, n_live) >= 0);
            const bool ok = mbar_wait(&ctl.s_full, uint32_t(n & 1), &ctl.abort);
            if (softmax_bar_or(!ok)) {
                failed = true;
                break;
            }
            tc_fence_after_sync();
            float x[kBlk];
            float m_blk = -INFINITY;
            {   // whole warp: tcgen05.ld is warp-collective; lanes 16..31 read unused lanes
                uint32_t r[32];
                tmem_ld_32x32b_x32(lane_addr + kColS, r);
                tmem_ld_wait(r);
#pragma unroll
                for (int i = 0; i < 32; ++i) x[i] = ((u_lo >> i) & 1u) ? __uint_as_float(r[i]) * c2 : -INFINITY;
                tmem_ld_32x32b_x32(lane_addr + kColS + 32, r);
                tmem_ld_wait(r);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    x[32 + i] = ((u_hi >> i) & 1u) ? __uint_as_float(r[i]) * c2 : -INFINITY;
            }
            if (head_thr) {
#pragma unroll
                for (int i = 0; i < kBlk; ++i) m_blk = fmaxf(m_blk, x[i]);
                if (n == 0) m_used = m_blk;
            }
            const bool need = head_thr && n > 0 && m_blk > m_used + kRescaleLog2;
            if (softmax_bar_or(need)) {  // raise the running max: rescale l and O^T (rare)
                if (head_thr) {
                    float alpha = 1.f;
                    if (need) {
                        alpha = exp2f(m_used - m_blk);
                        m_used = m_blk;
                        l_sum *= alpha;
                    }
                    ctl.alpha[h] = alpha;
                }
                softmax_bar_sync();
#pragma unroll 1
                for (int j = 0; j < 8; ++j) {
                    uint32_t r[32];
                    const uint32_t col = kColO + 32u * j;  // heads [32 (j & 1), +32) of dims block j / 2
                    tmem_ld_32x32b_x32(lane_addr + col, r);
                    tmem_ld_wait(r);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        r[i] = __float_as_uint(__uint_as_float(r[i]) * ctl.alpha[(j & 1) * 32 + i]);
                    tmem_st_x32(lane_addr + col, r);
                }
                tmem_st_wait();
            }
            if (head_thr) {  // P row h (bf16) for MMA2, K-major 128-byte swizzle
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    uint32_t packed[4];
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2) {
                        const float p0 = ex2_approx(x[8 * ch + 2 * q2] - m_used);
                        const float p1 = ex2_approx(x[8 * ch + 2 * q2 + 1] - m_used);
                        const __nv_bfloat162 v = __floats2bfloat162_rn(p0, p1);
                        const float2 back = __bfloat1622float2(v);
                        l_sum += back.x + back.y;
                        packed[q2] = *reinterpret_cast<const uint32_t*>(&v);
                    }
                    *reinterpret_cast<uint4*>(prow + ((ch ^ (h & 7)) << 4)) =
                        make_uint4(packed[0], packed[1], packed[2], packed[3]);
                }
                fence_proxy_async_smem();
            }
            tc_fence_before_sync();
            mbar_arrive(&ctl.p_full);
        }
        if (nblk > 0 && !failed) {
            const bool ok = mbar_wait(&ctl.o_done, 0, &ctl.abort);
            failed = softmax_bar_or(!ok);
        }
        if (failed && threadIdx.x == 128) {
            atomicOr(p.err, kErrWaitTimeout);
            ctl.abort = 1;
        }
        if (nblk == 0) {  // no used entry in this split: o = 0, lse = -inf
            for (int i = threadIdx.x - 128; i < kMlaHeads * kMlaDv; i += 128) o_dst[i] = 0.f;
            if (threadIdx.x - 128 < kMlaHeads) lse_dst[threadIdx.x - 128] = -INFINITY;
        } else if (!failed) {
            tc_fence_after_sync();
            if (head_thr) {
                ctl.inv_l[h] = 1.f / l_sum;
                lse_dst[h] = (m_used + log2f(l_sum)) * kLn2;
            }
            softmax_bar_sync();
            // o [64 heads, 512 dims] fp32 staged in the drained value ring, then bulk stores
            float* o_s = reinterpret_cast<float*>(tiles + kOffV);
#pragma unroll 1
            for (int j = 0; j < 8; ++j) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(lane_addr + kColO + 32u * j, r);
                tmem_ld_wait(r);
                const int d = (j >> 1) * 128 + quad * 32 + lane;
                const int h0 = (j & 1) * 32;
#pragma unroll
                for (int i = 0; i < 32; ++i) o_s[(h0 + i) * kMlaDv + d] = __uint_as_float(r[i]) * ctl.inv_l[h0 + i];
            }
            fence_proxy_async_smem();
            softmax_bar_sync();
            if (threadIdx.x == 128) {
                for (int c = 0; c < 4; ++c)
                    bulk_store(o_dst + c * (kMlaHeads * kMlaDv / 4), s_base + kOffV + c * (kMlaHeads * kMlaDv),
                               uint32_t(kMlaHeads * kMlaDv));
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        const uint32_t addr = smem_u32(&ctl.o_done);
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(addr, 0) && global_timer_ns() - t0 < kWaitLimitNs) {
        }
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kTmemColsM);
    }
}

// o[b, h] = sum_j exp(lse_j - lse) o_j over the splits, lse = log sum_j exp(lse_j).
// Grid (8 head groups, batch), 256 threads, two dims per thread and head.
__global__ void __launch_bounds__(256) mla_merge_kernel(const MlaParams p) {
    __shared__ float wgt[8][kMlaMaxSplits];
    pdl_wait_prior_grid();
    const int b = blockIdx.y;
    const int h0 = blockIdx.x * 8;
    const int S = p.splits;
    if (threadIdx.x < 8) {
        const int h = h0 + threadIdx.x;
        const float* lp = p.lse_part + int64_t(b) * S * kMlaHeads + h;
        float mx = -INFINITY;
        for (int j = 0; j < S; ++j) mx = fmaxf(mx, lp[int64_t(j) * kMlaHeads]);
        float sum = 0.f;
        for (int j = 0; j < S; ++j) {
            const float e = mx == -INFINITY ? 0.f : expf(lp[int64_t(j) * kMlaHeads] - mx);
            wgt[threadIdx.x][j] = e;
            sum += e;
        }
        const float inv = sum > 0.f ? 1.f / sum : 0.f;
        for (int j = 0; j < S; ++j) wgt[threadIdx.x][j] *= inv;
        p.lse[int64_t(b) * kMlaHeads + h] = mx == -INFINITY ? -INFINITY : mx + logf(sum);
    }
    __syncthreads();
    pdl_allow_next_grid();
    const int d = threadIdx.x * 2;
    for (int hh = 0; hh < 8; ++hh) {
        const int h = h0 + hh;
        float2 acc = make_float2(0.f, 0.f);
        for (int j = 0; j < S; ++j) {
            const float w = wgt[hh][j];
            const float2 v = *reinterpret_cast<const float2*>(
                p.o_part + ((int64_t(b) * S + j) * kMlaHeads + h) * kMlaDv + d);
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
        }
        *reinterpret_cast<float2*>(p.out + (int64_t(b) * kMlaHeads + h) * kMlaDv + d) = acc;
    }
}

}  // namespace

size_t mla_smem_bytes() { return size_t(kSmemM); }

cudaError_t launch_mla(const CUtensorMap& q_map, const CUtensorMap& kv_map, const MlaParams& p, cudaStream_t stream) {
    static SmemLimitOnce smem_limit;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = smem_limit.apply(dev, mla_decode_kernel, kSmemM);
    if (e != cudaSuccess) return e;
    if (p.splits < 1 || p.splits > kMlaMaxSplits) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(p.splits), unsigned(p.batch));
    cfg.blockDim = dim3(kThreadsM);
    cfg.dynamicSmemBytes = size_t(kSmemM);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, mla_decode_kernel, q_map, kv_map, p);
    if (e != cudaSuccess || p.splits == 1) return e;
    cfg.gridDim = dim3(kMlaHeads / 8, unsigned(p.batch));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, mla_merge_kernel, p);
}

}  // namespace dsa

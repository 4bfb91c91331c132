// proj_kernel.cu -- the indexer's query / head-weight projection, sm_103a.
//
//     q[b, o] = sum_d x[b, d] * Wq[o, d]   (o = 32 heads x 64 dims), stored bf16 [B, 32, 64]
//     w[b, h] = sum_d x[b, d] * Ww[h, d]   (32 heads),              stored fp32 [B, 32]
//
// on the bf16 hidden state with fp32 accumulation: the pages replace forced-fp32
// SIMT GEMMs on the indexer path by bf16 tensor-core GEMMs fed the bf16 hidden
// state directly ("The Indexer O(max_context) Breakthrough", section "Phase 3:
// The FP32-to-bf16 GEMM Flip").  The weight shapes are not on the pages; the
// model width d is a parameter.
//
// A decode batch is a few tokens, so the GEMM is a stream over the weights:
// each weight byte is read once, and the whole GPU must stream.  The output
// features are the MMA's M side (tiles of 128 rows of [Wq; Ww], the last tile
// holding Ww's 32 rows and zero fill), the tokens the N side (padded to a
// multiple of 16), and the model width is split across the k_split CTAs of a
// thread-block cluster (split-K), about one CTA per SM streaming weights:
//   * grid (n_tiles, k_split), cluster (1, k_split); CTA (i, z) reduces d over
//     atoms [z A, (z+1) A) of 64 elements;
//   * warp 0: TMA of the 128 x 64 weight box and the Bp x 64 activation box
//     per atom (128-byte swizzle) into a ring of 2-4 stages (96-144 KiB);
//   * warp 1: tcgen05.mma kind::f16 M=128 x N=Bp x K=16, four per atom, into
//     one TMEM accumulator;
//   * warps 2-5: tcgen05.ld of the accumulator into the CTA's shared memory;
//     after a cluster barrier each CTA sums its share of the tile's tokens
//     over the k_split partials through distributed shared memory, in split
//     order (deterministic), and writes q as bf16 and w as fp32.
// Every wait is bounded (about 1 s); a timeout sets an error bit and the roles
// drain and free TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "indexer_kernels.h"
#include "sm103_ptx.cuh"

namespace dsa {
namespace {

// Shared memory for the stage ring: 96 KiB up to 64 tokens (two CTAs per SM, so that the
// clusters of k_split CTAs find room together), more for wider token tiles, whose fp32
// partial tile (128 x Bp x 4 B) reuses the drained ring.
__host__ __device__ constexpr int stage_budget(int bp) { return bp <= 64 ? 96 * 1024 : (bp == 128 ? 128 * 1024 : 144 * 1024); }
constexpr int kAtom = 64;                    // bf16 elements of d per stage (one 128-byte swizzle row)
constexpr int kWBoxBytes = 128 * kAtom * 2;  // 16 KiB
constexpr int kThreadsP = 192;               // producer, MMA, 4 epilogue warps
constexpr int kCtasPerSmP = 2;
constexpr int kMaxSplitP = 8;                // portable cluster size


struct __align__(8) ProjCtl {
    uint64_t full[8];
    uint64_t empty[8];
    uint64_t done;
    uint32_t tmem_base;
    int abort;
};

__host__ __device__ constexpr int x_box_bytes(int bp) { return bp * kAtom * 2; }
__host__ __device__ constexpr int stage_bytes(int bp) { return kWBoxBytes + x_box_bytes(bp); }
__host__ __device__ constexpr int stages_for(int bp) {
    return stage_budget(bp) / stage_bytes(bp) < 8 ? stage_budget(bp) / stage_bytes(bp) : 8;
}

// TMEM columns for a Bp-column fp32 accumulator (power of two >= 32).
__host__ __device__ constexpr uint32_t tmem_cols(int bp) {
    return bp <= 32 ? 32u : (bp <= 64 ? 64u : (bp <= 128 ? 128u : 256u));
}

template <int kBp>
__global__ void __launch_bounds__(kThreadsP, kCtasPerSmP)
    proj_kernel(const __grid_constant__ CUtensorMap wq_map, const __grid_constant__ CUtensorMap ww_map,
                const __grid_constant__ CUtensorMap x_map, const ProjParams p) {
    constexpr int kStagesP_ = stages_for(kBp);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    ProjCtl& ctl = *reinterpret_cast<ProjCtl*>(tiles + size_t(kStagesP_) * stage_bytes(kBp));
    float* red = reinterpret_cast<float*>(tiles);  // [kBp][128] partial tile, over the drained stages
    static_assert(size_t(kStagesP_) * stage_bytes(kBp) >= size_t(kBp) * 128 * 4, "partial tile fits the stages");
    constexpr uint32_t kCols = tmem_cols(kBp);
    constexpr uint32_t kIdescP = idesc_bf16_f32(128, kBp);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tile = blockIdx.x;   // 128 output features
    const int split = blockIdx.y;  // range of d
    const int atoms_total = p.d_model / kAtom;
    const int a0 = int((int64_t(atoms_total) * split) / gridDim.y);
    const int a1 = int((int64_t(atoms_total) * (split + 1)) / gridDim.y);
    const bool is_w_tile = tile == p.q_tiles;  // the last tile holds Ww's 32 rows

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesP_; ++s) {
            mbar_init(&ctl.full[s], 1);
            mbar_init(&ctl.empty[s], 1);
        }
        mbar_init(&ctl.done, 1);
        ctl.abort = 0;
        fence_mbar_init();
        tma_prefetch_map(is_w_tile ? &ww_map : &wq_map);
        tma_prefetch_map(&x_map);
    }
    if (warp == 1) {
        tmem_alloc(&ctl.tmem_base, kCols);
        tmem_relinquish();
    }
    pdl_wait_prior_grid();
    pdl_allow_next_grid();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = ctl.tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_first();  // weights: read once
            const uint64_t pol_x = l2_policy_evict_last();   // activations: every tile reads them
            int stage = 0, issued = 0;
            uint32_t phase = 0;
            bool stop = false;
            for (int a = a0; a < a1; ++a) {
                if (!mbar_wait(&ctl.empty[stage], phase ^ 1u, &ctl.abort)) {
                    stop = true;
                    break;
                }
                uint8_t* st = tiles + size_t(stage) * stage_bytes(kBp);
                mbar_arrive_expect_tx(&ctl.full[stage], uint32_t(stage_bytes(kBp)));
                if (is_w_tile)
                    tma_load_2d(st, &ww_map, &ctl.full[stage], a * kAtom, 0, pol_w);
                else
                    tma_load_2d(st, &wq_map, &ctl.full[stage], a * kAtom, tile * 128, pol_w);
                tma_load_2d(st + kWBoxBytes, &x_map, &ctl.full[stage], a * kAtom, 0, pol_x);
                ++issued;
                if (++stage == kStagesP_) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (stop) {
                atomicOr(p.err, kErrWaitTimeout);
                ctl.abort = 1;
            }
            if (ctl.abort) {  // let the copies in flight land before the CTA may exit
                int s = stage;
                uint32_t ph = phase;
                for (int i = 0; i < min(issued, kStagesP_); ++i) {
                    if (s == 0) {
                        s = kStagesP_ - 1;
                        ph ^= 1u;
                    } else {
                        --s;
                    }
                    const uint32_t addr = smem_u32(&ctl.full[s]);
                    const uint64_t t0 = global_timer_ns();
                    while (!mbar_try_wait(addr, ph) && global_timer_ns() - t0 < kWaitLimitNs) {
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool stop = false;
            for (int a = a0; a < a1; ++a) {
                if (!mbar_wait(&ctl.full[stage], phase, &ctl.abort)) {
                    stop = true;
                    break;
                }
                tc_fence_after_sync();
                uint8_t* st = tiles + size_t(stage) * stage_bytes(kBp);
                const uint64_t a_desc = smem_desc_kmajor_sw128(smem_u32(st));
                const uint64_t b_desc = smem_desc_kmajor_sw128(smem_u32(st + kWBoxBytes));
#pragma unroll
                for (int kk = 0; kk < kAtom / 16; ++kk)
                    umma_bf16_ss(tmem_base, a_desc + 2u * kk, b_desc + 2u * kk, kIdescP,
                                 (a > a0 || kk > 0) ? 1u : 0u);
                umma_commit(&ctl.empty[stage]);
                if (++stage == kStagesP_) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (stop) {
                atomicOr(p.err, kErrWaitTimeout);
                ctl.abort = 1;
            }
            umma_commit(&ctl.done);  // every MMA issued has completed when this arrives
        }
        __syncwarp();
    } else {
        // ================= epilogue: warps 2..5, thread = output feature =================
        const int quad = warp & 3;  // TMEM lanes [32 quad, 32 quad + 32)
        bool ok = true;
        {
            const uint32_t addr = smem_u32(&ctl.done);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(addr, 0)) {
                if (ctl.abort || global_timer_ns() - t0 > kWaitLimitNs) {
                    ok = false;
                    break;
                }
            }
        }
        ok = __all_sync(0xffffffffu, ok);
        tc_fence_after_sync();
        if (ok) {  // the partial tile to shared memory, red[token][row] (the stages are free now)
#pragma unroll 1
            for (int c0 = 0; c0 < kBp; c0 += 32) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(c0), r);
                tmem_ld_wait(r);
#pragma unroll
                for (int j = 0; j < 32; ++j) red[(c0 + j) * 128 + quad * 32 + lane] = __uint_as_float(r[j]);
            }
        } else if (lane == 0) {
            atomicOr(p.err, kErrWaitTimeout);
            ctl.abort = 1;
        }
    }

    tc_fence_before_sync();
    cluster_sync_all();  // every CTA's partial tile is in its shared memory
    if (warp >= 2) {
        // CTA z sums tokens [z Bp / k, (z+1) Bp / k) of the tile over the k partials, thread = row.
        const int row = threadIdx.x - 64;
        const int k = int(gridDim.y);
        const int z = int(cluster_rank());
        const int c_lo = (kBp * z) / k, c_hi = (kBp * (z + 1)) / k;
        const int valid_rows = is_w_tile ? kHeads : 128;
        uint32_t base[kMaxSplitP];
#pragma unroll
        for (int src = 0; src < kMaxSplitP; ++src) base[src] = src < k ? cluster_addr(red, uint32_t(src)) : 0u;
        for (int c = c_lo; c < c_hi && c < p.batch; ++c) {
            const uint32_t off = uint32_t(c * 128 + row) * 4u;
            float v[kMaxSplitP];
#pragma unroll
            for (int src = 0; src < kMaxSplitP; ++src) v[src] = src < k ? ld_cluster_f32(base[src] + off) : 0.f;
            float acc = 0.f;
#pragma unroll
            for (int src = 0; src < kMaxSplitP; ++src) acc += v[src];  // split order: deterministic
            if (row < valid_rows) {
                if (is_w_tile)
                    p.w_out[int64_t(c) * kHeads + row] = acc;
                else
                    p.q_out[int64_t(c) * (p.q_tiles * 128) + tile * 128 + row] =
                        static_cast<__nv_bfloat16_raw>(__float2bfloat16_rn(acc));
            }
        }
    }
    cluster_sync_all();  // no CTA leaves while another still reads its shared memory
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kCols);
    }
}

template <int kBp>
cudaError_t launch_proj_bp(const CUtensorMap& wq_map, const CUtensorMap& ww_map, const CUtensorMap& x_map,
                           const ProjParams& p, cudaStream_t stream) {
    static SmemLimitOnce smem_limit;
    const size_t smem = 1024 + size_t(stages_for(kBp)) * stage_bytes(kBp) + sizeof(ProjCtl);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = smem_limit.apply(dev, proj_kernel<kBp>, int(smem));
    if (e != cudaSuccess) return e;
    if (p.k_split < 1 || p.k_split > kMaxSplitP) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = unsigned(p.k_split);
    attr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(p.q_tiles + 1), unsigned(p.k_split));
    cfg.blockDim = dim3(kThreadsP);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, proj_kernel<kBp>, wq_map, ww_map, x_map, p);
}

}  // namespace

int proj_batch_pad(int batch) { return batch <= 32 ? 32 : (batch <= 64 ? 64 : (batch <= 128 ? 128 : 256)); }

cudaError_t launch_proj(const CUtensorMap& wq_map, const CUtensorMap& ww_map, const CUtensorMap& x_map,
                        const ProjParams& p, cudaStream_t stream) {
    switch (p.batch_pad) {
        case 32: return launch_proj_bp<32>(wq_map, ww_map, x_map, p, stream);
        case 64: return launch_proj_bp<64>(wq_map, ww_map, x_map, p, stream);
        case 128: return launch_proj_bp<128>(wq_map, ww_map, x_map, p, stream);
        case 256: return launch_proj_bp<256>(wq_map, ww_map, x_map, p, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace dsa

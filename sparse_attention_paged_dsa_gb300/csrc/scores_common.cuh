// scores_common.cuh -- pieces shared by the bf16 and fp8 scores kernels:
// per-request live extents, the work-unit schedule, page-id preparation,
// unit metadata, the dead-tail -inf fill and the schedule reset.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "indexer_kernels.h"
#include "sm103_ptx.cuh"

namespace dsa {
namespace scores {

constexpr int kBatch = 32;         // units prepared per warp-wide page-table load
constexpr int kEndOfWork = -1;     // metadata marker: no more units

// Unit metadata: request (10 bits), page pair within the request (15 bits),
// validity of its two pages (2 bits).  Max row width 2^22 C4 positions keeps
// the pair below 2^15; kMaxBatch = 1024 keeps the request below 2^10.
__device__ __forceinline__ int pack_meta(int b, int pair, bool ok0, bool ok1) {
    return (b << 17) | (pair << 2) | (ok1 ? 2 : 0) | (ok0 ? 1 : 0);
}
__device__ __forceinline__ int meta_row(int m) { return m >> 17; }
__device__ __forceinline__ int meta_pair(int m) { return (m >> 2) & 0x7FFF; }

// Live C4 count and first work unit of every request: two arrays in shared
// memory, sized by the launch's batch (placed after a kernel's fixed layout).
struct RowTable {
    int32_t* n_live;      // [batch]
    int32_t* unit_start;  // [batch + 1]
};

// Shared-memory bytes of the table for `batch` requests (a 16-byte multiple).
__host__ __device__ constexpr size_t row_table_bytes(int batch) {
    return (size_t(2 * batch + 1) * sizeof(int32_t) + 15) & ~size_t(15);
}

__device__ __forceinline__ RowTable row_table_at(uint8_t* base, int batch) {
    int32_t* a = reinterpret_cast<int32_t*>(base);
    return RowTable{a, a + batch};
}

// One warp fills the table: n_b = ceil(clamp(seq_len_b, 0, max_context) / 4), units of
// kUnitPositions positions, exclusive prefix of units.  Flags clamped lengths (CTA 0).
__device__ __forceinline__ void build_row_table(const RowTable& t, const ScoresParams& p, int lane) {
    const int batch = p.batch;
    const int per = (batch + 31) / 32;  // lane l owns rows [l*per, (l+1)*per)
    const int b0 = min(lane * per, batch), b1 = min(b0 + per, batch);
    int units = 0;
    bool clamped = false;
    for (int b = b0; b < b1; ++b) {
        int64_t s = p.seq_lens[b];
        if (s < 0 || s > p.max_context) clamped = true;
        s = s < 0 ? 0 : (s > p.max_context ? p.max_context : s);
        const int n = static_cast<int>((s + 3) >> 2);
        t.n_live[b] = n;
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
        t.unit_start[b] = run;
        run += (t.n_live[b] + kUnitPositions - 1) / kUnitPositions;
    }
    if (lane == 31) t.unit_start[batch] = incl;
    if (clamped && blockIdx.x == 0) atomicOr(p.err, kErrSeqLenClamped);
}

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

// Bounded wait used only while draining after an abort.
__device__ __forceinline__ void wait_landed(uint64_t* bar, uint32_t parity) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(a, parity) && global_timer_ns() - t0 < kWaitLimitNs) {
    }
}

// One lane's unit of a batch: its request, page pair and page ids (-2: no live second page).
struct UnitPrep {
    int b = 0;
    int pair = 0;
    int pg0 = -1;
    int pg1 = -2;
};

// Lane l prepares unit u0 + l when l < cnt (page-table loads in flight on return).
__device__ __forceinline__ UnitPrep prepare_units(const RowTable& t, const ScoresParams& p, int u0, int cnt,
                                                  int lane) {
    UnitPrep c;
    if (lane < cnt) {
        const int u = u0 + lane;
        c.b = row_of_unit(t.unit_start, p.batch, u);
        c.pair = u - t.unit_start[c.b];
        const int live_pages = (t.n_live[c.b] + kPageEntries - 1) / kPageEntries;
        const int32_t* row = p.page_table + int64_t(c.b) * p.table_width;
        c.pg0 = __ldg(row + 2 * c.pair);
        c.pg1 = (2 * c.pair + 1 < live_pages) ? __ldg(row + 2 * c.pair + 1) : -2;
    }
    return c;
}

// A CTA's units: the contiguous range [c S, (c + 1) S) with S = floor(U / grid),
// in batches of kBatch, then unit S grid + c when c < U - S grid.  Fixed by
// (U, grid, c) alone, so every producer warp of the CTA walks the same
// sequence without talking to the others.  (A dynamic share handed out from
// a global counter cost more in round trips than it won in balance.)
struct UnitSchedule {
    int sp, se, extra;

    __device__ __forceinline__ explicit UnitSchedule(int total_units) {
        const int grid = gridDim.x;
        const int S = total_units / grid;
        sp = blockIdx.x * S;
        se = sp + S;
        extra = int(blockIdx.x) < total_units - S * grid ? S * grid + int(blockIdx.x) : -1;
    }

    // Next batch [u0, u0 + cnt); cnt == 0 when the CTA has no more units.
    __device__ __forceinline__ void next(int& u0, int& cnt) {
        if (sp < se) {
            u0 = sp;
            cnt = min(kBatch, se - sp);
            sp += cnt;
        } else if (extra >= 0) {
            u0 = extra;
            cnt = 1;
            extra = -1;
        } else {
            u0 = 0;
            cnt = 0;
        }
    }
};

// Stream -inf over every row's positions past its request's live units (all
// `tokens` rows of a request share the extent), done by one warp per CTA
// (lane = `lane`) beside the pipeline: the dead float4s of all rows, taken in
// row order as one flat range, are split into equal contiguous shares, one per
// CTA, and each share is written by the warp with consecutive lanes on
// consecutive float4s.
__device__ __forceinline__ void fill_dead_tails_warp(const RowTable& t, const ScoresParams& p, int lane,
                                                     int tokens = 1) {
    const int64_t M4 = p.row_width / 4;
    const float neg_inf = __int_as_float(0xff800000);
    const float4 ninf4 = make_float4(neg_inf, neg_inf, neg_inf, neg_inf);
    const int batch = p.batch;
    auto dead4 = [&](int b) {  // dead float4s of each of request b's rows
        const int64_t e4 = int64_t(t.unit_start[b + 1] - t.unit_start[b]) * (kUnitPositions / 4);
        return e4 < M4 ? M4 - e4 : int64_t(0);
    };
    // Lane l sums the rows [l * per, (l + 1) * per); a warp scan gives each lane's flat start.
    const int per = (batch + 31) / 32;
    const int r0 = min(lane * per, batch), r1 = min(r0 + per, batch);
    int64_t mine = 0;
    for (int b = r0; b < r1; ++b) mine += dead4(b) * tokens;
    int64_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
    }
    const int64_t total = __shfl_sync(0xffffffffu, incl, 31);  // < 2^31 float4s
    // This CTA's share [lo, hi): floor(total * c / grid) in double is exact (the product is
    // below 2^53 and the quotient is at least 1 / grid away from the next integer).
    const int64_t lo = int64_t(double(total) * blockIdx.x / gridDim.x);
    const int64_t hi = int64_t(double(total) * (blockIdx.x + 1) / gridDim.x);
    const int64_t start = incl - mine;
    uint32_t owners = __ballot_sync(0xffffffffu, mine > 0 && start < hi && start + mine > lo);
    while (owners) {  // lanes whose rows meet the share, in row order
        const int src = __ffs(owners) - 1;
        owners &= owners - 1u;
        int64_t acc = __shfl_sync(0xffffffffu, start, src);
        for (int b = min(src * per, batch); b < min(src * per + per, batch) && acc < hi; ++b) {
            const int64_t d = dead4(b);
            for (int j = 0; j < tokens; ++j, acc += d) {
                const int64_t s0 = acc > lo ? acc : lo, s1 = acc + d < hi ? acc + d : hi;
                float4* row = reinterpret_cast<float4*>(p.out + (int64_t(b) * tokens + j) * p.row_width) + (M4 - d);
                for (int64_t i = s0 + lane; i < s1; i += 32) __stcs(row + (i - acc), ninf4);
            }
        }
    }
}

}  // namespace scores
}  // namespace dsa

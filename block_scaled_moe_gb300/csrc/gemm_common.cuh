// gemm_common.cuh -- pieces of the tcgen05 grouped GEMMs shared by the
// stand-alone GEMM kernels (moe_gemm.cu) and the single-launch fused kernel
// (moe_fused.cu): the global unit list, the routing-plan tables, bounded
// drains and pipeline tracing.
#pragma once
#include "moe_internal.h"
#include "ptx.cuh"

namespace bmoe {
namespace {

// Pipeline tracing (compiled in with -DBMOE_TRACE): clock64 stamps of the first
// kTraceJobs K stages of CTAs 0 and 1, per role, into GemmArgs::trace
// ([2 CTAs][8 events][kTraceJobs] int64): 0 producer got a free stage, 1 producer
// issued it, 2 first MMA warp saw it full, 3 that warp issued its MMAs; per
// unit: 4 epilogue saw the accumulator, 5 epilogue released it; per stage again:
// 6 weight-scale warp got the free stage, 7 it arrived on the full barrier.
__device__ __forceinline__ void trace(const GemmArgs& a, int ev, long idx) {
#ifdef BMOE_TRACE
    constexpr int kTraceJobs = 512;
    if (a.trace && blockIdx.x < 2 && idx < kTraceJobs)
        a.trace[(static_cast<long>(blockIdx.x) * 8 + ev) * kTraceJobs + idx] = clock64();
#else
    (void)a;
    (void)ev;
    (void)idx;
#endif
}

// Tracing builds: globaltimer stamp `which` (0 start, 1 end) of this CTA, after the stage stamps.
__device__ __forceinline__ void trace_cta(const GemmArgs& a, int which) {
#ifdef BMOE_TRACE
    if (a.trace && blockIdx.x < 1024) a.trace[2 * 8 * 512 + 2 * blockIdx.x + which] = static_cast<long long>(globaltimer_ns());
#else
    (void)a;
    (void)which;
#endif
}

struct UnitInfo {
    int e, m, g, row0, n;
};

// Routing plan as read by the GEMM roles: shared-memory copies when E fits the
// tables, else the global arrays.
struct Plan {
    const int32_t* tile_base;  // [E+1]
    const int32_t* rowbase;    // [E+1]
    const int32_t* counts;     // [E]
};

// Unit u of the global list: experts ascending; inside an expert, weight tile m
// major and route tile j minor, so CTAs running consecutive units share a
// weight tile (L2 reuse when an expert has several route tiles).  `ecur` only
// moves forward because every role walks its units in increasing order.
// Unit u of expert e (tile_base[e] <= u / mtiles < tile_base[e + 1]).
__device__ __forceinline__ UnitInfo unit_of_expert(int u, int e, const Plan& pl, int mtiles, int NT) {
    const int tb = pl.tile_base[e];
    const int nt = pl.tile_base[e + 1] - tb;
    const int ul = u - tb * mtiles;
    UnitInfo r;
    r.e = e;
    r.m = ul / nt;
    const int j = ul - r.m * nt;
    r.g = tb + j;
    r.row0 = pl.rowbase[e] + j * NT;
    r.n = min(NT, pl.counts[e] - j * NT);
    return r;
}

__device__ __forceinline__ UnitInfo decode_unit(int u, int& ecur, const Plan& pl, int mtiles, int NT) {
    const int q = u / mtiles;
    while (pl.tile_base[ecur + 1] <= q) ++ecur;
    return unit_of_expert(u, ecur, pl, mtiles, NT);
}

// The expert of unit u by bisection of tile_base[0..E] (no cursor), for decoding a CTA's units once
// up front: the cursor walk costs a dependent shared-memory load per expert passed, which under a
// full stage ring adds up to a few thousand cycles per unit.
__device__ __forceinline__ int expert_of_unit(int u, const Plan& pl, int mtiles, int E) {
    const int q = u / mtiles;
    int lo = 0, hi = E;  // tile_base[lo] <= q < tile_base[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pl.tile_base[mid] <= q)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// Units of a CTA decoded once into shared memory before the pipeline starts (16 bytes each, up to
// kUnitTab of them, fewer where the stage ring leaves less room); later units, if any, are decoded
// with the role's cursor.
constexpr int kUnitTab = 512;

// A decoded unit in one 16-byte shared-memory word: {e, m | n << 16, g, row0}.
__device__ __forceinline__ int4 pack_unit(const UnitInfo& r) { return make_int4(r.e, r.m | (r.n << 16), r.g, r.row0); }
__device__ __forceinline__ UnitInfo unpack_unit(int4 v) {
    UnitInfo r;
    r.e = v.x;
    r.m = v.y & 0xffff;
    r.n = v.y >> 16;
    r.g = v.z;
    r.row0 = v.w;
    return r;
}

// The CTA's unit number ui of a single unit list (GEMM units strided over the grid); the table
// holds the first `ntab` units.
__device__ __forceinline__ UnitInfo unit_ref(int ui, const int4* utab, int ntab, int& ecur, const Plan& pl, int mtiles,
                                             int NT) {
    if (ui < ntab) return unpack_unit(utab[ui]);
    return decode_unit(static_cast<int>(blockIdx.x) + ui * static_cast<int>(gridDim.x), ecur, pl, mtiles, NT);
}

#ifdef MOE_DEBUG_BOUNDS
// Bounds-checking builds: how many of the CTA's n units (unit i from decode(i)) lie inside the
// workspace regions, i.e. a route tile below lim_tiles and rows [row0, row0 + n) below lim_rows with
// 1 <= n <= NT, counted up to the first that does not; the CTA's roles all end their unit lists
// there, so they stay in step.
template <typename Decode>
__device__ __forceinline__ int units_in_bounds(int n, Decode&& decode, int NT, int lim_rows, int lim_tiles,
                                               uint32_t* status, uint32_t* ticket) {
    for (int i = 0; i < n; ++i) {
        const UnitInfo cu = decode(i);
        if (!(bounds_ok(status, ticket, cu.g, lim_tiles, kBsUnit) && bounds_ok(status, ticket, cu.n - 1, NT, kBsUnit) &&
              bounds_ok(status, ticket, cu.row0, lim_rows, kBsUnit) &&
              bounds_ok(status, ticket, static_cast<long long>(cu.row0) + cu.n - 1, lim_rows, kBsUnit)))
            return i;
    }
    return n;
}
#endif

// The loads of the last STAGES jobs this producer issued land before the CTA
// exits (they are consumed already unless another role gave up).  Bounded.
template <int STAGES>
__device__ __forceinline__ void drain_stages(uint64_t* full, int stage, uint32_t phase, long issued,
                                             uint32_t* status) {
    volatile int never = 0;
    for (long i = 0; i < STAGES && i < issued; ++i) {
        if (stage == 0) {
            stage = STAGES - 1;
            phase ^= 1u;
        } else {
            --stage;
        }
        (void)mbar_wait(&full[stage], phase, &never, status, kStTimeout | (1u << (kSiteShift + 1)),
                        kWaitLimitNs / 4);
    }
}

}  // namespace
}  // namespace bmoe

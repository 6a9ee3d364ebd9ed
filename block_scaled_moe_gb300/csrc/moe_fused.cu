// moe_fused.cu -- the single-launch fused path for small token counts
// (ROCm/aiter PR #6881, MegaMoEV2 small-input path, "Technical Details": at
// most 512 tokens, and the whole layer runs inside a single kernel launch so
// that the per-stage launches and their grid-wide hand-offs disappear).
//
// One persistent cooperative CTA per SM runs, in one launch:
//   phase 0  dispatch (fixed-slot or compact) and MXFP8 quantisation + scatter,
//            separated by grid barriers;
//   phase 1  GEMM1 and GEMM2 as ONE unit list (all GEMM1 units, then all GEMM2
//            units, strided over the CTAs): the weight stream does not drain
//            between the GEMMs.  A GEMM2 unit of route tile g starts its row
//            loads once the 4 epilogue warps of each of the I/128 GEMM1 units
//            of g have released their h rows (per-tile readiness counter,
//            release/acquire and proxy fences, bounded wait);
//   phase 2  combine, after a last grid barrier.
// Grid barriers wait for a generation word to CHANGE from the value read before
// arriving (equality, so the 32-bit word may wrap) and are bounded: on expiry
// the CTA sets MOE_ST_TIMEOUT with a site bit and skips the remaining phases.
//
// GEMM tiles are the decode width (N <= 32 routed rows, 2 MMA-issuing warps
// each owning an accumulator chain: GEMM1 gate / up, GEMM2 one W2 tile of a pair
// or half of a stage's K-steps); a stage holds up to two 128x128 weight
// chunks (GEMM1: gate and up; GEMM2: two 128-wide K chunks) and two row chunks.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "gemm_common.cuh"
#include "layer_rows.cuh"
#include "moe_internal.h"
#include "ptx.cuh"

#ifdef BMOE_TRACE
// Phase trace (tracing builds only): per CTA 32 int64 slots of globaltimer ns
// stamps and counters, read back with bmoe_fused_trace_copy; and per K stage of
// CTAs 0 and 1, clock64 stamps [2 CTAs][16 events][4096 stages]: 0 producer got
// a free stage, 1 producer issued it, 2 MMA chain 0 saw it full, 3 chain 0
// issued, 4 weight-scale warp got it, 5 that warp filled it, 6 producer began
// waiting for it, 7 / 8 / 9 chains 1 / 2 / 3 (those there are) issued, 10 chain 0 began
// waiting for it, 11 the last chain saw it full; per unit (index = the CTA's unit number): 12 producer
// entered the unit, 13 producer decoded it, 14 producer issued its prefetch, 15 chain 0
// decoded it (stamps 13 and 15 take an index that depends on the decoded unit, so that
// they follow the decode) (bmoe_fused_stage_trace_copy).
__device__ long long g_fused_trace[1024 * 32];
constexpr int kFusedTraceStages = 4096;
constexpr int kFusedStageEvents = 16;
__device__ long long g_fused_stage_trace[2 * kFusedStageEvents * kFusedTraceStages];
#define FTRACE(ev, val)                                              \
    do {                                                             \
        if (blockIdx.x < 1024) g_fused_trace[blockIdx.x * 32 + (ev)] = (val); \
    } while (0)
#define FSTRACE(ev, idx)                                                                         \
    do {                                                                                         \
        if (blockIdx.x < 2 && (idx) < kFusedTraceStages)                                          \
            g_fused_stage_trace[(blockIdx.x * kFusedStageEvents + (ev)) * kFusedTraceStages + (idx)] = clock64(); \
    } while (0)
#else
#define FTRACE(ev, val) \
    do {                \
    } while (0)
#define FSTRACE(ev, idx) \
    do {                 \
    } while (0)
#endif

namespace bmoe {

namespace {

constexpr int F_NT = 32;                                    // route tile width
constexpr int F_MW = 2;                                     // accumulator chains = MMA-issuing warps
constexpr int F_EW = 4;                                     // epilogue warps (one per TMEM lane quadrant)
constexpr int F_MMA_WARP0 = 2, F_EPI_WARP0 = 2 + F_MW;
constexpr int F_THREADS = 32 * (2 + F_MW + F_EW);
constexpr int F_A_BYTES = 128 * 128;                        // one 128x128 FP4 chunk in smem
constexpr int F_A_TX = 128 * 128 / 2;                       // ... and its transaction bytes
constexpr int F_B_BYTES = F_NT * 128;                       // one row chunk
constexpr int F_STAGE_BYTES = 2 * F_A_BYTES + 2 * F_B_BYTES + 4 * 512;
constexpr int F_TAB_E = 512;                                // the fused path needs E <= 512
constexpr int F_TAB_BYTES = 4 * (3 * F_TAB_E + 4);
constexpr int F_SCR_INTS = 2 * F_TAB_E + 64;                // phase-0 scratch, inside the (idle) stage ring
constexpr int F_STAGES = (220 * 1024 - F_TAB_BYTES) / F_STAGE_BYTES;
constexpr int F_ACC_COLS = F_MW * F_NT;
constexpr int F_SF_SLOT = 8;                                // [weight atom | row atom] of the chain's chunk
constexpr int F_SF_BASE = 512 - F_MW * 2 * F_SF_SLOT;       // two slots per chain (alternating stages)
constexpr int F_NUM_ACC = 2;
constexpr bool kUnitPrefetch = true;  // L2 prefetch of each unit's first weight box one unit ahead
constexpr int F_BAR_BYTES = (2 * F_STAGES + 2 * 2 + 1) * 8 + 16;
constexpr int F_UTAB = kUnitTab;                            // a CTA's first units, decoded once (16 bytes each)
constexpr int F_UTAB_OFF = (F_STAGES * F_STAGE_BYTES + F_TAB_BYTES + F_BAR_BYTES + 15) & ~15;
constexpr int F_SMEM = 1024 + F_UTAB_OFF + F_UTAB * 16;
static_assert(4 * F_SCR_INTS <= F_STAGES * F_STAGE_BYTES, "phase-0 scratch");
static_assert(F_NUM_ACC * F_ACC_COLS <= F_SF_BASE, "TMEM columns");
static_assert(F_SMEM <= 232448, "shared memory");

struct FusedArgs {
    rows::QuantArgs q;     // x, ids, T, K, E, H, mtpr, words, NT, scheme, ws
    const int32_t* nvr;
    const float* wts;
    uint16_t* out;
    const uint8_t* w13s;
    const uint8_t* w2s;
    int I;
    int w13_rs, w13_up;    // W13 scale rows: gate j at j * w13_rs, up j at j * w13_rs + w13_up
    int kc2;               // K chunks per GEMM2 stage of single W2 tiles (2 when I % 256 == 0)
    int w2w;               // GEMM2 units take W2 tiles in pairs (H % 256 == 0): one 256-row box per 128-wide K stage
    uint8_t* y8;           // GEMM2 rows as MXFP8 codes / scales (nullptr: BF16 rows in ws.y)
    uint8_t* ys;
    int nchunks;           // compact dispatch chunks
    int tiles_cap;
    float swiglu_limit;
};

// Grid-wide barrier of a cooperative launch (see the file comment).
__device__ bool grid_sync(uint32_t* count, uint32_t* gen, uint32_t* status, volatile int* abort_smem) {
    __syncthreads();
    if (threadIdx.x == 0 && !*abort_smem) {
        const uint32_t g = ld_acquire_u32(gen);
        __threadfence();
        const uint32_t arrived = atomicAdd(count, 1u) + 1u;
        if (arrived == gridDim.x) {
            atomicExch(count, 0u);
            __threadfence();
            st_release_u32(gen, g + 1u);
        } else {
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_u32(gen) == g) {
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    atomicOr(status, kStTimeout | kSiteGrid);
                    *abort_smem = 1;
                    break;
                }
                __nanosleep(100);
            }
        }
        __threadfence();
    }
    __syncthreads();
    return !*abort_smem;
}

// Exclusive scan of in[0..n) into out[0..n] (out[n] = total) by the whole CTA.
__device__ void cta_exclusive_scan(const int* in, int* out, int n, int* warp_sums) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int start = tid * per;
    int local = 0;
    for (int i = start; i < start + per && i < n; ++i) local += in[i];
    int x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int v = lane < nwarps ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
        }
        warp_sums[lane] = v;
    }
    __syncthreads();
    int run = (warp > 0 ? warp_sums[warp - 1] : 0) + x - local;
    for (int i = start; i < start + per && i < n; ++i) {
        out[i] = run;
        run += in[i];
    }
    if (tid == 0) out[n] = warp_sums[nwarps - 1];
    __syncthreads();
}

// Unit u of the fused list: GEMM1 units [0, U1), then GEMM2 units.
struct FUnit {
    bool g2;
    UnitInfo u;
};
struct FCursor {
    int e1 = 0, e2 = 0;
};
__device__ __forceinline__ FUnit fused_unit(int u, int U1, FCursor& c, const Plan& pl, int mt1, int mt2) {
    FUnit r;
    r.g2 = u >= U1;
    r.u = r.g2 ? decode_unit(u - U1, c.e2, pl, mt2, F_NT) : decode_unit(u, c.e1, pl, mt1, F_NT);
    return r;
}

// The CTA's unit number ui: from the table decoded before phase 1 (the first F_UTAB units), else
// decoded here with the role's cursor.
__device__ __forceinline__ FUnit unit_at(int ui, const int4* utab, int U1, FCursor& c, const Plan& pl, int mt1,
                                         int mt2) {
    const int u = static_cast<int>(blockIdx.x) + ui * static_cast<int>(gridDim.x);
    if (ui >= F_UTAB) return fused_unit(u, U1, c, pl, mt1, mt2);
    FUnit r;
    r.g2 = u >= U1;
    r.u = unpack_unit(utab[ui]);
    return r;
}

// Phase-1 pipeline: the stage ring in shared memory and the TMEM base.
struct P1 {
    uint8_t* sA;     // [stage][2] weight chunks
    uint8_t* sB;     // [stage][2] row chunks
    uint8_t* sSFA;   // [stage][2] weight scale atoms
    uint8_t* sSFB;   // [stage][2] row scale atoms
    uint64_t* full;
    uint64_t* empty;
    volatile int* abort_flag;
    uint32_t* status;
    uint32_t tmem;
};

struct Ring {
    int stage = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void next() {
        if (++stage == F_STAGES) {
            stage = 0;
            phase ^= 1u;
        }
    }
};

// TMA producer, one unit of kt K stages.  GEMM1 (G2 false): the gate and up chunks of weight
// tile m of expert e (one box of the W13 pair view, coordinates (k, m*128, 0, e)), one row
// chunk and its scale atom per stage; GEMM2: KC (W2 chunk, h chunk) pairs and KC h-scale
// atoms per stage (W2 rows from wrow), or, for paired W2 tiles (PAIR2), one 256-row W2 box
// (both tiles, back to back like GEMM1's gate and up chunks), one h chunk and its atom per
// stage.  The row-scale atoms of the unit start at bsf.
template <bool G2, int KC, bool PAIR2 = false>
__device__ __forceinline__ bool produce_unit(const P1& p, Ring& r, long& issued, const CUtensorMap* tw,
                                             const CUtensorMap* tb, int wrow, int e, int row0,
                                             const uint8_t* bsf, int kt, uint64_t pol_w, uint64_t pol_b,
                                             long long& wait_ns, long long& issue_ns) {
    for (int kk = 0; kk < kt; ++kk) {
#ifdef BMOE_TRACE
        const long long tw0 = (long long)globaltimer_ns();
        if (threadIdx.x == 0) FSTRACE(6, issued);
#endif
        const bool got = mbar_wait(&p.empty[r.stage], r.phase ^ 1u, p.abort_flag, p.status,
                                   kStTimeout | (1u << (kSiteShift + 0)), kWaitLimitNs);
        if (!__all_sync(0xffffffffu, got)) return false;  // the warp stays converged for the elected issue
#ifdef BMOE_TRACE
        const long long tw1 = (long long)globaltimer_ns();
        wait_ns += tw1 - tw0;
        if (threadIdx.x == 0) FSTRACE(0, issued);
#else
        (void)wait_ns;
        (void)issue_ns;
#endif
        uint64_t* fb = &p.full[r.stage];
        uint8_t* a0 = p.sA + (r.stage * 2) * F_A_BYTES;
        uint8_t* b0 = p.sB + (r.stage * 2) * F_B_BYTES;
        // the producer's arrival carries the stage's transaction bytes (one elected lane issues)
        if constexpr (!G2) {
            mbar_arrive_expect_tx_w(fb, 2 * F_A_TX + F_B_BYTES + 512);
            tma_load_4d_w(a0, tw, fb, kk * 128, wrow, 0, e, pol_w);
            tma_load_2d_w(b0, tb, fb, kk * 128, row0, pol_b);
            bulk_load_w(p.sSFB + (r.stage * 2) * 512, bsf + static_cast<size_t>(kk) * 512, 512, fb);
        } else if constexpr (PAIR2) {
            mbar_arrive_expect_tx_w(fb, 2 * F_A_TX + F_B_BYTES + 512);
            tma_load_2d_w(a0, tw, fb, kk * 128, wrow, pol_w);
            tma_load_2d_w(b0, tb, fb, kk * 128, row0, pol_b);
            bulk_load_w(p.sSFB + (r.stage * 2) * 512, bsf + static_cast<size_t>(kk) * 512, 512, fb);
        } else {
            mbar_arrive_expect_tx_w(fb, KC * (F_A_TX + F_B_BYTES + 512));
            if constexpr (KC == 2) {  // two-chunk views (the launch passes them for 256-wide stages)
                tma_load_3d_w(a0, tw, fb, 0, wrow, kk * KC, pol_w);
                tma_load_3d_w(b0, tb, fb, 0, row0, kk * KC, pol_b);
            } else {
                tma_load_2d_w(a0, tw, fb, kk * 128, wrow, pol_w);
                tma_load_2d_w(b0, tb, fb, kk * 128, row0, pol_b);
            }
            bulk_load_w(p.sSFB + (r.stage * 2) * 512, bsf + static_cast<size_t>(kk) * KC * 512, KC * 512, fb);
        }
#ifdef BMOE_TRACE
        issue_ns += (long long)globaltimer_ns() - tw1;
        if (threadIdx.x == 0) FSTRACE(1, issued);
#endif
        ++issued;
        r.next();
    }
    return true;
}

// MMA issue of one unit by chain w (its warp, converged, one elected lane issuing).  GEMM1: chain w multiplies operand
// w & 1 (gate / up) over the K-steps k with k % 2 == w >> 1; GEMM2: chain w takes the KC
// consecutive K-steps [w*KC, w*KC + KC) of the stage (k = 4 * chunk + step in chunk), all in
// chunk w*KC/4.  Either way a chain reads one weight atom and one row atom per stage, which
// it copies to its own TMEM slot (two slots, alternating stages).
template <bool G2, int KC>
__device__ __forceinline__ bool mma_unit(const P1& p, Ring& r, long& job, int w, int lane, uint32_t d_tmem, int N,
                                         int kt, long long& wait_ns, long long& issue_ns) {
    constexpr int SPC = 4 * KC / F_MW;   // GEMM2: consecutive K-steps of a chain per stage
    constexpr int KSPLIT = F_MW / 2;     // GEMM1: chains per operand (K-steps split by k % KSPLIT)
    static_assert((F_MW == 2 || F_MW == 4) && (KC == 1 || KC == 2) && SPC >= 1 && SPC <= 4,
                  "each chain's K-steps lie in one chunk");
    const int ach = G2 ? (w * SPC) >> 2 : (w & 1);  // weight chunk (GEMM1: operand) of this chain
    const int bch = G2 ? (w * SPC) >> 2 : 0;        // row chunk of this chain
    for (int kk = 0; kk < kt; ++kk) {
#ifdef BMOE_TRACE
        const long long tw0 = (long long)globaltimer_ns();
        if (w == 0 && lane == 0) FSTRACE(10, job);
#endif
        const bool got = mbar_wait(&p.full[r.stage], r.phase, p.abort_flag, p.status,
                                   kStTimeout | (1u << (kSiteShift + 3)), kWaitLimitNs);
        if (!__all_sync(0xffffffffu, got)) return false;  // the warp stays converged for the elected issue
#ifdef BMOE_TRACE
        const long long tw1 = (long long)globaltimer_ns();
        wait_ns += tw1 - tw0;
        if (w == 0 && lane == 0) FSTRACE(2, job);
        if (w == F_MW - 1 && lane == 0) FSTRACE(11, job);
#else
        (void)wait_ns;
        (void)issue_ns;
#endif
        tc_fence_after();
        {
            const uint32_t sfa = p.tmem + static_cast<uint32_t>(F_SF_BASE + (w * 2 + (job & 1)) * F_SF_SLOT);
            const uint32_t sfb = sfa + 4;
            tc_cp_32x128b_x4_w(sfa, desc_sf_atom(smem_u32(p.sSFA + (r.stage * 2 + ach) * 512)));
            tc_cp_32x128b_x4_w(sfb, desc_sf_atom(smem_u32(p.sSFB + (r.stage * 2 + bch) * 512)));
            const uint64_t da0 = desc_kmajor_sw128(smem_u32(p.sA + (r.stage * 2 + ach) * F_A_BYTES));
            const uint64_t db0 = desc_kmajor_sw128(smem_u32(p.sB + (r.stage * 2 + bch) * F_B_BYTES));
            if constexpr (!G2) {
                const int kq = w >> 1;
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    if (k4 % KSPLIT != kq) continue;
                    tc_mma_mx_w(d_tmem, da0 + static_cast<uint64_t>((k4 * 32) >> 4),
                                db0 + static_cast<uint64_t>((k4 * 32) >> 4), idesc_mx(128, N, 5, 0, k4, k4), sfa, sfb,
                                (kk > 0 || k4 != kq) ? 1u : 0u);
                }
            } else {
#pragma unroll
                for (int j = 0; j < SPC; ++j) {
                    const int k4 = (w * SPC + j) & 3;
                    tc_mma_mx_w(d_tmem, da0 + static_cast<uint64_t>((k4 * 32) >> 4),
                                db0 + static_cast<uint64_t>((k4 * 32) >> 4), idesc_mx(128, N, 5, 0, k4, k4), sfa, sfb,
                                (kk > 0 || j > 0) ? 1u : 0u);
                }
            }
            tc_commit_w(&p.empty[r.stage]);
#ifdef BMOE_TRACE
            issue_ns += (long long)globaltimer_ns() - tw1;
            if (lane == 0) FSTRACE(w == 0 ? 3 : 6 + w, job);
#endif
        }
        __syncwarp();
        ++job;
        r.next();
    }
    return true;
}

// Epilogue of one unit by one warp (TMEM lane quadrant qd = its 32 output features).  The
// chains are summed in the stand-alone GEMMs' order, from +0, so both paths give the same
// bits.  GEMM1: gate/up -> optional clamp -> SwiGLU -> MXFP8 per 32 features (OCP MX rule)
// into the h rows and their scale atom, then this warp's share of tile g is released to the
// GEMM2 units; GEMM2: BF16 rows of y.  The accumulator is handed back before the stores.
// GEMM2 with paired W2 tiles (PAIR2): chains 0 / 2 hold the first tile, 1 / 3 the second (like GEMM1's
// gate and up), summed in the same order; the unit's rows are features m*256 + f and m*256 + 128 + f.
// These are stored as each 16-column slice is read (the pair's 64 values per lane do not fit the
// register budget), so the accumulator goes back after the stores are issued.
template <bool G2, bool PAIR2 = false>
__device__ __forceinline__ void epilogue_unit(const P1& p, uint64_t* acce_b, const Workspace& ws, const UnitInfo& cu,
                                              int acc, int qd, int lane, int I, int H, float L, uint8_t* y8,
                                              uint8_t* ys) {
    const uint32_t tb = p.tmem + (static_cast<uint32_t>(32 * qd) << 16) + static_cast<uint32_t>(acc * F_ACC_COLS);
    const int feat = cu.m * (PAIR2 ? 256 : 128) + 32 * qd + lane;
    float v[PAIR2 ? 1 : F_NT];
#pragma unroll
    for (int j = 0; j < F_NT / 16; ++j) {
        const int c0 = 16 * j;
        if (c0 < cu.n) {
            uint32_t r[F_MW][16];
#pragma unroll
            for (int w = 0; w < F_MW; ++w) tmem_ld16(tb + w * F_NT + c0, r[w]);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float ga = 0.f, ub = 0.f;
#pragma unroll
                for (int w = 0; w < F_MW; ++w) {
                    if ((!G2 || PAIR2) && (w & 1))
                        ub += __uint_as_float(r[w][i]);
                    else
                        ga += __uint_as_float(r[w][i]);
                }
                if constexpr (!G2) {
                    if (ws.g && c0 + i < cu.n) {
                        const size_t prow = static_cast<size_t>(cu.row0 + c0 + i);
                        ws.g[prow * 2 * I + feat] = ga;
                        ws.g[prow * 2 * I + I + feat] = ub;
                    }
                    if (L > 0.f) {
                        ga = fminf(ga, L);
                        ub = fminf(fmaxf(ub, -L), L);
                    }
                    v[c0 + i] = __fdividef(ga, 1.0f + __expf(-ga)) * ub;  // SwiGLU, fast exp / divide intrinsics
                } else if constexpr (PAIR2) {
                    if (c0 + i < cu.n) {
                        const size_t prow = static_cast<size_t>(cu.row0 + c0 + i);
                        if (y8) {  // MXFP8 GEMM2 rows: this warp's 32 features of each tile are one 1x32 block
                            uint8_t sc;
                            y8[prow * H + feat] = rows::quant_block_warp(ga, &sc);
                            if (lane == 0) ys[prow * (H >> 5) + (feat >> 5)] = sc;
                            y8[prow * H + feat + 128] = rows::quant_block_warp(ub, &sc);
                            if (lane == 0) ys[prow * (H >> 5) + ((feat + 128) >> 5)] = sc;
                        } else {
                            ws.y[prow * H + feat] = __bfloat16_as_ushort(__float2bfloat16_rn(ga));
                            ws.y[prow * H + feat + 128] = __bfloat16_as_ushort(__float2bfloat16_rn(ub));
                        }
                    }
                } else {
                    v[c0 + i] = ga;
                }
            }
        }
    }
    tc_fence_before();
    mbar_arrive(acce_b);
    if constexpr (PAIR2) return;
    if (G2 && y8) {  // MXFP8 GEMM2 rows: this warp's 32 features are one 1x32 block
#pragma unroll
        for (int c = 0; c < F_NT; ++c) {
            if (c < cu.n) {
                const size_t prow = static_cast<size_t>(cu.row0 + c);
                uint8_t sc;
                y8[prow * H + feat] = rows::quant_block_warp(v[c], &sc);
                if (lane == 0) ys[prow * (H >> 5) + (feat >> 5)] = sc;
            }
        }
        return;
    }
#pragma unroll
    for (int c = 0; c < F_NT; ++c) {
        if (c < cu.n) {
            const size_t prow = static_cast<size_t>(cu.row0 + c);
            if constexpr (!G2) {
                const float h = v[c];
                const uint32_t amax = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(h)));
                int code = static_cast<int>(amax >> 23) - 8;
                code = code < 0 ? 0 : code;
                const float mul = __uint_as_float(static_cast<uint32_t>(254 - code) << 23);
                ws.hq[prow * I + feat] = __nv_cvt_float_to_fp8(h * mul, __NV_SATFINITE, __NV_E4M3);
                if (lane == 0)
                    ws.hs[((size_t)cu.g * (I >> 7) + cu.m) * 512 + 16 * (c & 31) + 4 * (c >> 5) + qd] =
                        static_cast<uint8_t>(code);
            } else {
                ws.y[prow * H + feat] = __bfloat16_as_ushort(__float2bfloat16_rn(v[c]));
            }
        }
    }
    if constexpr (!G2) {
        // Release this warp's 32 features of tile g's h rows to the GEMM2 units (TMA reads them
        // from any CTA); warps release independently, nobody waits here.
        fence_proxy_async_all();
        __threadfence();
        __syncwarp();
        if (lane == 0) {
            __threadfence();
            atom_add_release_u32(&ws.ready[cu.g], 1u);
        }
    }
}

__global__ void __launch_bounds__(F_THREADS, 1)
    k_fused(const __grid_constant__ CUtensorMap tm_w13p, const __grid_constant__ CUtensorMap tm_aq,
            const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_hq, const FusedArgs f) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = sm;                                       // [stage][2] weight chunks
    uint8_t* sB = sA + F_STAGES * 2 * F_A_BYTES;            // [stage][2] row chunks
    uint8_t* sSFA = sB + F_STAGES * 2 * F_B_BYTES;          // [stage][2] weight scale atoms
    uint8_t* sSFB = sSFA + F_STAGES * 2 * 512;              // [stage][2] row scale atoms
    int32_t* tab = reinterpret_cast<int32_t*>(sSFB + F_STAGES * 2 * 512);
    int32_t* scr = reinterpret_cast<int32_t*>(sA);          // phase-0 scratch (the ring is idle then)
    uint64_t* full = reinterpret_cast<uint64_t*>(tab + 3 * F_TAB_E + 4);
    uint64_t* empty = full + F_STAGES;
    uint64_t* accf = empty + F_STAGES;
    uint64_t* acce = accf + 2;
    uint64_t* drain = acce + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int4* utab = reinterpret_cast<int4*>(sm + F_UTAB_OFF);  // [F_UTAB] decoded units of this CTA

    const rows::QuantArgs& q = f.q;
    const Workspace& ws = q.ws;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = q.E, K = q.K, T = q.T, H = q.H, I = f.I;
    const int nvr = rows::read_nvr(f.nvr, T);
    const int gtid = blockIdx.x * blockDim.x + threadIdx.x, gstride = gridDim.x * blockDim.x;
    uint32_t* bar_count = ws.ticket + 2;
    uint32_t* bar_gen = ws.ticket + 3;
    int32_t* t_tile = tab;                  // [E+1]
    int32_t* t_row = tab + F_TAB_E + 1;     // [E+1]
    int32_t* t_cnt = tab + 2 * F_TAB_E + 2; // [E]
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        FTRACE(0, (long long)globaltimer_ns());
    }
    __syncthreads();

    // ------------------------------------------------------------------ phase 0: dispatch + quant
    for (int i = gtid; i < f.tiles_cap; i += gstride) ws.ready[i] = 0;
    if (q.scheme == 1) {
        // fixed-slot (vLLM PR #61262): slot (e, t), occupancy bits, no prepare step
        for (int i = gtid; i < E * q.words; i += gstride) ws.occ[i] = 0;
        if (!grid_sync(bar_count, bar_gen, ws.status, abort_flag)) goto finish;
        if (threadIdx.x == 0) FTRACE(22, (long long)globaltimer_ns());
        for (int s = gtid; s < T * K; s += gstride) {
            const int t = s / K, e = q.ids[s];
            if (t < nvr && e >= E) atomicOr(ws.status, kStBadId);
            BMOE_BOUNDS_ONLY(if (!bounds_ok(ws.status, ws.ticket, s, ws.lim_slots, kBsSlot)) continue;)
            if (t < nvr && e >= 0 && e < E BMOE_BOUNDS_ONLY(&& bounds_ok(ws.status, ws.ticket, t, q.mtpr, kBsOcc))) {
                atomicOr(&ws.occ[(size_t)e * q.words + (t >> 5)], 1u << (t & 31));
                ws.route_slot[s] = e * q.mtpr + t;
            } else {
                ws.route_slot[s] = -1;
            }
        }
        if (!grid_sync(bar_count, bar_gen, ws.status, abort_flag)) goto finish;
        if (threadIdx.x == 0) FTRACE(23, (long long)globaltimer_ns());
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            int c = 0;
            for (int w = 0; w < q.words; ++w) c += __popc(__ldcg(&ws.occ[(size_t)e * q.words + w]));
            t_cnt[e] = c;
            t_row[e] = e * q.mtpr;
            scr[e] = (c + F_NT - 1) / F_NT;
        }
        if (threadIdx.x == 0) t_row[E] = E * q.mtpr;
        __syncthreads();
        cta_exclusive_scan(scr, t_tile, E, scr + 2 * F_TAB_E);
    } else {
        // compact (vLLM PR #61262): per-chunk histograms, scan, stable pack
        int* cnt = scr;
        // every CTA takes the same branch
        BMOE_BOUNDS_ONLY(if (!bounds_ok(ws.status, ws.ticket, f.nchunks, ws.lim_chunks + 1, kBsChunk)) goto finish;)
        for (int c = blockIdx.x; c < f.nchunks; c += gridDim.x) {
            for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
            __syncthreads();
            for (int i = threadIdx.x; i < kChunk; i += blockDim.x) {
                const int s = c * kChunk + i;
                if (s < T * K) {
                    const int t = s / K, e = q.ids[s];
                    if (t < nvr && e >= E) atomicOr(ws.status, kStBadId);
                    if (t < nvr && e >= 0 && e < E) atomicAdd(&cnt[e], 1);
                }
            }
            __syncthreads();
            for (int e = threadIdx.x; e < E; e += blockDim.x) ws.chunk_base[(size_t)c * E + e] = cnt[e];
            __syncthreads();
        }
        if (!grid_sync(bar_count, bar_gen, ws.status, abort_flag)) goto finish;
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            int run = 0;
            for (int c = 0; c < f.nchunks; ++c) run += __ldcg(&ws.chunk_base[(size_t)c * E + e]);
            t_cnt[e] = run;
            cnt[e] = run;
        }
        __syncthreads();
        cta_exclusive_scan(cnt, t_row, E, scr + 2 * F_TAB_E);
        for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = (t_cnt[e] + F_NT - 1) / F_NT;
        __syncthreads();
        cta_exclusive_scan(cnt, t_tile, E, scr + 2 * F_TAB_E);
        // stable ranks of this CTA's chunks: one warp walks each chunk in order
        for (int c = blockIdx.x; c < f.nchunks; c += gridDim.x) {
            int* run = scr;  // per-expert next row of this chunk
            for (int e = threadIdx.x; e < E; e += blockDim.x) {
                int b = t_row[e];
                for (int c2 = 0; c2 < c; ++c2) b += __ldcg(&ws.chunk_base[(size_t)c2 * E + e]);
                run[e] = b;
            }
            __syncthreads();
            if (warp == 0) {
                const unsigned lt = (1u << lane) - 1u;
                for (int it = 0; it < kChunk / 32; ++it) {
                    const int s = c * kChunk + it * 32 + lane;
                    const bool in = s < T * K;
                    const int e = in ? q.ids[s] : -1;
                    const bool valid = in && (s / K) < nvr && e >= 0 && e < E;
                    const int key = valid ? e : (0x40000000 | lane);
                    const unsigned peers = __match_any_sync(0xffffffffu, key);
                    if (valid) {
                        const int p = run[e] + __popc(peers & lt);
                        BMOE_BOUNDS_ONLY(if (bounds_ok(ws.status, ws.ticket, s, ws.lim_slots, kBsSlot)))
                        ws.route_row[s] = p;
                        BMOE_BOUNDS_ONLY(if (bounds_ok(ws.status, ws.ticket, p, ws.lim_slots, kBsPerm)))
                        ws.perm[p] = s;
                    } else if (in BMOE_BOUNDS_ONLY(&& bounds_ok(ws.status, ws.ticket, s, ws.lim_slots, kBsSlot))) {
                        ws.route_row[s] = -1;
                    }
                    __syncwarp();
                    if (valid && lane == __ffs(peers) - 1) run[e] += __popc(peers);
                    __syncwarp();
                }
            }
            __syncthreads();
        }
        if (!grid_sync(bar_count, bar_gen, ws.status, abort_flag)) goto finish;
    }
    if (blockIdx.x == 0) {  // the plan, for introspection
        for (int e = threadIdx.x; e <= E; e += blockDim.x) {
            ws.tile_base[e] = t_tile[e];
            ws.rowbase[e] = t_row[e];
            if (e < E) ws.counts[e] = t_cnt[e];
        }
    }
    if (threadIdx.x == 0) FTRACE(24, (long long)globaltimer_ns());
    // quantise + scatter: one warp per row segment
    {
        const int items = rows::quant_items(q);
        for (int it = blockIdx.x * (blockDim.x >> 5) + warp; it < items; it += gridDim.x * (blockDim.x >> 5))
            rows::quant_scatter_seg(q, t_row, t_tile, it, nvr, lane);
    }
    fence_proxy_async_all();  // the packed rows and scale atoms are read by TMA / bulk copies
    if (threadIdx.x == 0) FTRACE(25, (long long)globaltimer_ns());
    if (!grid_sync(bar_count, bar_gen, ws.status, abort_flag)) goto finish;

    // ------------------------------------------------------------------ phase 1: GEMM1 + GEMM2
    {
        const int ntiles = t_tile[E];
        const int mt1 = I / 128, mt2 = H / (f.w2w ? 256 : 128);
        const int U1 = ntiles * mt1, U = U1 + ntiles * mt2;
#ifdef MOE_DEBUG_BOUNDS
        const int all_units =
#else
        const int my_units =
#endif
            static_cast<int>(blockIdx.x) < U ? (U - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                                             : 0;
        const int kt1 = H / 128, kt2 = f.w2w ? I / 128 : I / (128 * f.kc2), ktot2 = I / 128;
        const Plan pl{t_tile, t_row, t_cnt};
#ifdef MOE_DEBUG_BOUNDS
        FCursor chk_cur;
        const int my_units = units_in_bounds(
            all_units, [&](int i) { return fused_unit(blockIdx.x + i * gridDim.x, U1, chk_cur, pl, mt1, mt2).u; },
            F_NT, ws.lim_rows, ws.lim_tiles, ws.status, ws.ticket);
#endif
        for (int i = threadIdx.x; i < min(my_units, F_UTAB); i += blockDim.x) {
            const int u = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
            const bool g2 = u >= U1;
            const int uu = g2 ? u - U1 : u, mt = g2 ? mt2 : mt1;
            utab[i] = pack_unit(unit_of_expert(uu, expert_of_unit(uu, pl, mt, E), pl, mt, F_NT));
        }
        if (threadIdx.x == 0) {
            for (int s = 0; s < F_STAGES; ++s) {
                mbar_init(&full[s], 1 + 32);  // the producer's arrive.expect_tx + the scale warp's lanes
                mbar_init(&empty[s], F_MW);
            }
            for (int b = 0; b < 2; ++b) {
                mbar_init(&accf[b], F_MW);
                mbar_init(&acce[b], 32 * F_EW);
            }
            mbar_init(drain, F_MW);
            fence_mbar_init();
        }
        if (warp == F_MMA_WARP0) {
            tmem_alloc(tmem_slot, 512);
            tmem_relinquish();
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        const uint32_t tmem = *tmem_slot;

        if (threadIdx.x == 0) FTRACE(1, (long long)globaltimer_ns());
        P1 p;
        p.sA = sA;
        p.sB = sB;
        p.sSFA = sSFA;
        p.sSFB = sSFB;
        p.full = full;
        p.empty = empty;
        p.abort_flag = abort_flag;
        p.status = ws.status;
        p.tmem = tmem;
        if (warp == 0) {
            // -------------------------------------------------------- TMA producer (one warp, one elected lane issues)
            if (my_units > 0) {
#ifdef BMOE_TRACE
                long long wait_ns = 0;
                bool first_g2 = true;
#endif
                const uint64_t pol_w = policy_evict_first(), pol_b = policy_evict_last();
                Ring ring;
                long issued = 0;
                bool ok = true;
                FCursor cur;
                long long ew1 = 0, ew2 = 0;  // empty-stage wait ns in GEMM1 / GEMM2 units (tracing builds)
                long long pi1 = 0, pi2 = 0;  // issue ns
                fence_proxy_async_all();  // phase-0 rows and scale atoms are read through the async proxy
                FCursor pcur;             // one unit ahead: the next unit's first weight box is prefetched to L2
                for (int ui = 0; ui < my_units && ok; ++ui) {
                    if (threadIdx.x == 0) FSTRACE(12, ui);
                    const FUnit fu = unit_at(ui, utab, U1, cur, pl, mt1, mt2);
                    const UnitInfo& cu = fu.u;
                    if (threadIdx.x == 0) FSTRACE(13, ui + (cu.n > 1000 ? 1 : 0));
                    if (kUnitPrefetch && ui + 1 < my_units) {
                        // a unit's first loads start in weight rows no CTA has touched yet; fetching its first
                        // box one unit early takes that latency off the stage ring
                        const FUnit nu = unit_at(ui + 1, utab, U1, pcur, pl, mt1, mt2);
                        if (!nu.g2)
                            tma_prefetch_4d_w(&tm_w13p, 0, nu.u.m * 128, 0, nu.u.e);
                        else if (f.w2w)
                            tma_prefetch_2d_w(&tm_w2, 0, nu.u.e * H + nu.u.m * 256);
                        else if (f.kc2 == 2)
                            tma_prefetch_3d_w(&tm_w2, 0, nu.u.e * H + nu.u.m * 128, 0);
                        else
                            tma_prefetch_2d_w(&tm_w2, 0, nu.u.e * H + nu.u.m * 128);
                    }
                    if (threadIdx.x == 0) FSTRACE(14, ui);
                    if (!fu.g2) {
                        ok = produce_unit<false, 1>(p, ring, issued, &tm_w13p, &tm_aq, cu.m * 128, cu.e, cu.row0,
                                                    ws.as + (size_t)cu.g * kt1 * 512, kt1, pol_w, pol_b, ew1, pi1);
                        continue;
                    }
                    // the h rows of tile g are complete once all epilogue warps of its I/128 GEMM1
                    // units released them
                    const uint64_t t0 = globaltimer_ns();
#ifdef BMOE_TRACE
                    if (first_g2) FTRACE(2, (long long)t0);
#endif
                    while (ld_acquire_u32(&ws.ready[cu.g]) != static_cast<uint32_t>(mt1 * F_EW)) {
                        if (*abort_flag || globaltimer_ns() - t0 > kWaitLimitNs) {
                            atomicOr(ws.status, kStTimeout | kSiteReady);
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                        __nanosleep(64);
                    }
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
#ifdef BMOE_TRACE
                    {
                        const long long t1 = (long long)globaltimer_ns();
                        if (first_g2) FTRACE(3, t1);
                        first_g2 = false;
                        wait_ns += t1 - (long long)t0;
                    }
#endif
                    fence_proxy_async_all();
                    const int wrow = cu.e * H + cu.m * (f.w2w ? 256 : 128);
                    const uint8_t* bsf = ws.hs + (size_t)cu.g * ktot2 * 512;
                    ok = f.w2w ? produce_unit<true, 1, true>(p, ring, issued, &tm_w2, &tm_hq, wrow, 0, cu.row0, bsf,
                                                             kt2, pol_w, pol_b, ew2, pi2)
                         : f.kc2 == 2 ? produce_unit<true, 2>(p, ring, issued, &tm_w2, &tm_hq, wrow, 0, cu.row0, bsf,
                                                              kt2, pol_w, pol_b, ew2, pi2)
                                      : produce_unit<true, 1>(p, ring, issued, &tm_w2, &tm_hq, wrow, 0, cu.row0, bsf,
                                                              kt2, pol_w, pol_b, ew2, pi2);
                }
#ifdef BMOE_TRACE
                FTRACE(4, wait_ns);
                FTRACE(5, (long long)globaltimer_ns());
                FTRACE(16, ew1);
                FTRACE(17, ew2);
                FTRACE(28, pi1);
                FTRACE(29, pi2);
#endif
                if (lane == 0) drain_stages<F_STAGES>(full, ring.stage, ring.phase, issued, ws.status);
            }
        } else if (warp == 1) {
            // -------------------------------------------------------- weight-scale producer (32 lanes)
            // Lane l writes, per stage, line l of two 128x4 scale atoms (GEMM1: gate and up rows;
            // GEMM2: the two W2 tiles of a pair, or two K chunks of one tile): the 4 K-block bytes
            // of rows l, l+32, l+64, l+96.  Stages are
            // handled in groups of up to 4 of one unit, loaded one group ahead into registers
            // (component j of each uint4 = stage j).  GEMM1 rows whose scale stride is a multiple
            // of 16 bytes take one 16-byte load per row and group: the weight-scale lines then need
            // not stay in L1, which this kernel's shared-memory footprint leaves small.
            const bool g1_vec = (H % 512) == 0;
            const bool g2w_vec = f.w2w && (I % 512) == 0;           // paired W2 tiles: 16-byte scale vectors
            const bool g2_pair = !f.w2w && f.kc2 == 2 && (I / 32) % 8 == 0;  // 8-byte aligned scale rows
            int q_ui = 0, q_kk = 0, q_kt = 0, q_ld = 0, q_rs = 1, q_up = 0;
            bool q_g2 = false, q_two = false, q_vec = false;  // q_two: the two atoms are two tiles' rows
            const uint8_t* q_base = nullptr;
            FCursor qcur;
            auto load_group = [&](uint4(&g)[2][4]) -> int {
                if (q_ui >= my_units) return 0;
                if (q_kk == 0) {
                    const FUnit fu = unit_at(q_ui, utab, U1, qcur, pl, mt1, mt2);
                    q_g2 = fu.g2;
                    q_kt = fu.g2 ? kt2 : kt1;
                    q_ld = fu.g2 ? I / 32 : H / 32;
                    q_rs = fu.g2 ? 1 : f.w13_rs;
                    q_two = !fu.g2 || f.w2w;
                    q_up = fu.g2 ? 128 : f.w13_up;
                    q_vec = fu.g2 ? g2w_vec : g1_vec;
                    const int rrow = fu.g2 ? fu.u.e * H + fu.u.m * (f.w2w ? 256 : 128) + lane
                                           : fu.u.e * 2 * I + (fu.u.m * 128 + lane) * f.w13_rs;
                    q_base = (fu.g2 ? f.w2s : f.w13s) + static_cast<size_t>(rrow) * q_ld;
                }
                const int len = min(4, q_kt - q_kk);
                if (q_two && q_vec) {
#pragma unroll
                    for (int a4 = 0; a4 < 2; ++a4)
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            g[a4][i] = __ldg(reinterpret_cast<const uint4*>(
                                q_base + static_cast<size_t>(a4 * q_up + 32 * i * q_rs) * q_ld + q_kk * 4));
                } else if (q_g2 && g2_pair) {
                    // 256-wide GEMM2 stages: the two K chunks' words of a row are one 8-byte pair
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint2 p4[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            p4[j] = j < len ? __ldg(reinterpret_cast<const uint2*>(
                                                  q_base + static_cast<size_t>(32 * i) * q_ld + (q_kk + j) * 8))
                                            : make_uint2(0u, 0u);
                        g[0][i] = make_uint4(p4[0].x, p4[1].x, p4[2].x, p4[3].x);
                        g[1][i] = make_uint4(p4[0].y, p4[1].y, p4[2].y, p4[3].y);
                    }
                } else {
#pragma unroll
                    for (int a4 = 0; a4 < 2; ++a4) {
                        const bool use = q_two || a4 < f.kc2;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            uint32_t w4[4];
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const int kk = q_kk + j;
                                const uint8_t* src = !q_two ? q_base + (kk * f.kc2 + a4) * 4
                                                            : q_base + static_cast<size_t>(a4 * q_up) * q_ld + kk * 4;
                                w4[j] = (use && j < len) ? __ldg(reinterpret_cast<const uint32_t*>(
                                                               src + static_cast<size_t>(32 * i * q_rs) * q_ld))
                                                         : 0u;
                            }
                            g[a4][i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                        }
                    }
                }
                q_kk += len;
                if (q_kk == q_kt) {
                    q_kk = 0;
                    ++q_ui;
                }
                return len;
            };
            auto word = [](const uint4& v, int j) { return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w; };
            uint4 cur[2][4], nxt[2][4];
            int clen = load_group(cur);
            Ring ring;
            long sjob = 0;
            bool ok = true;
            while (clen > 0 && ok) {
                const int nlen = load_group(nxt);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (j < clen && ok) {
                        if (!mbar_wait(&empty[ring.stage], ring.phase ^ 1u, abort_flag, ws.status,
                                       kStTimeout | (1u << (kSiteShift + 0)), kWaitLimitNs)) {
                            ok = false;
                        } else {
                            if (lane == 0) FSTRACE(4, sjob);
                            uint4* dst = reinterpret_cast<uint4*>(sSFA + (ring.stage * 2) * 512) + lane;
                            dst[0] = make_uint4(word(cur[0][0], j), word(cur[0][1], j), word(cur[0][2], j),
                                                word(cur[0][3], j));
                            dst[32] = make_uint4(word(cur[1][0], j), word(cur[1][1], j), word(cur[1][2], j),
                                                 word(cur[1][3], j));
                            fence_proxy_async_smem();
                            mbar_arrive(&full[ring.stage]);
                            if (lane == 0) FSTRACE(5, sjob);
                            ++sjob;
                            ring.next();
                        }
                    }
                }
#pragma unroll
                for (int a4 = 0; a4 < 2; ++a4)
#pragma unroll
                    for (int i = 0; i < 4; ++i) cur[a4][i] = nxt[a4][i];
                clen = nlen;
            }
        } else if (warp < F_EPI_WARP0) {
            // -------------------------------------------------------- MMA issuers (one chain each)
            const int w = warp - F_MMA_WARP0;
            Ring ring;
            int acc = 0;
            uint32_t acc_phase = 0;
            long job = 0;
            FCursor cur;
            long long fw1 = 0, fw2 = 0;  // stage-ready wait ns (tracing builds)
            long long mi1 = 0, mi2 = 0;  // issue ns
#ifdef BMOE_TRACE
            long long aw1 = 0, aw2 = 0;  // accumulator wait ns
#endif
            for (int ui = 0; ui < my_units; ++ui) {
                const FUnit fu = unit_at(ui, utab, U1, cur, pl, mt1, mt2);
                const int N = (fu.u.n + 15) & ~15;
                if (w == 0 && lane == 0) FSTRACE(15, ui + (N > 1000 ? 1 : 0));
#ifdef BMOE_TRACE
                const long long ta0 = (long long)globaltimer_ns();
#endif
                const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * F_ACC_COLS + w * F_NT);
                const bool got_acc = mbar_wait(&acce[acc], acc_phase ^ 1u, abort_flag, ws.status,
                                               kStTimeout | (1u << (kSiteShift + 2)), kWaitLimitNs);
                if (!__all_sync(0xffffffffu, got_acc)) break;
#ifdef BMOE_TRACE
                (fu.g2 ? aw2 : aw1) += (long long)globaltimer_ns() - ta0;
#endif
                tc_fence_after();
                // paired W2 tiles issue like GEMM1's gate / up pair: chain w takes tile w & 1
                const bool ok = !fu.g2       ? mma_unit<false, 1>(p, ring, job, w, lane, d_tmem, N, kt1, fw1, mi1)
                                : f.w2w      ? mma_unit<false, 1>(p, ring, job, w, lane, d_tmem, N, kt2, fw2, mi2)
                                : f.kc2 == 2 ? mma_unit<true, 2>(p, ring, job, w, lane, d_tmem, N, kt2, fw2, mi2)
                                             : mma_unit<true, 1>(p, ring, job, w, lane, d_tmem, N, kt2, fw2, mi2);
                if (!ok) break;
                tc_commit_w(&accf[acc]);
                __syncwarp();
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            __syncwarp();
            tc_commit_w(drain);
            if (lane == 0 && w == 0) {
                FTRACE(6, (long long)globaltimer_ns());
                FTRACE(18, fw1);
                FTRACE(19, fw2);
                FTRACE(20, aw1);
                FTRACE(21, aw2);
                FTRACE(30, mi1);
                FTRACE(31, mi2);
            }
            __syncwarp();
            volatile int never = 0;
            (void)mbar_wait(drain, 0, &never, ws.status, kStTimeout | (1u << (kSiteShift + 4)), kWaitLimitNs);
        } else {
            // -------------------------------------------------------- epilogue (4 warps)
            const int qd = warp & 3;
            int acc = 0;
            uint32_t acc_phase = 0;
            const float L = f.swiglu_limit;
            FCursor cur;
#ifdef BMOE_TRACE
            bool fused_g2_prev = false;
#endif
            for (int ui = 0; ui < my_units; ++ui) {
                const FUnit fu = unit_at(ui, utab, U1, cur, pl, mt1, mt2);
                if (!mbar_wait(&accf[acc], acc_phase, abort_flag, ws.status, kStTimeout | (1u << (kSiteShift + 5)),
                               kWaitLimitNs))
                    break;
                tc_fence_after();
#ifdef BMOE_TRACE
                if (qd == 0 && lane == 0 && fu.g2 && (ui == 0 || !fused_g2_prev)) FTRACE(8, (long long)globaltimer_ns());
                fused_g2_prev = fu.g2;
#endif
                if (!fu.g2)
                    epilogue_unit<false>(p, &acce[acc], ws, fu.u, acc, qd, lane, I, H, L, f.y8, f.ys);
                else if (f.w2w)
                    epilogue_unit<true, true>(p, &acce[acc], ws, fu.u, acc, qd, lane, I, H, L, f.y8, f.ys);
                else
                    epilogue_unit<true>(p, &acce[acc], ws, fu.u, acc, qd, lane, I, H, L, f.y8, f.ys);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
        }
        if (warp == F_EPI_WARP0 && lane == 0) FTRACE(7, (long long)globaltimer_ns());
#ifdef BMOE_TRACE
        if (threadIdx.x == 0) {
            const int bx = static_cast<int>(blockIdx.x), gx = static_cast<int>(gridDim.x);
            const int n1 = bx < U1 ? (U1 - 1 - bx) / gx + 1 : 0;
            FTRACE(11, n1);
            FTRACE(12, my_units - n1);
        }
#endif
        tc_fence_before();
        __syncthreads();
        if (warp == F_MMA_WARP0) {
            tc_fence_after();
            tmem_dealloc(tmem, 512);
        }
    }
    if (!grid_sync(bar_count, bar_gen, ws.status, abort_flag)) goto finish;
    if (threadIdx.x == 0) FTRACE(9, (long long)globaltimer_ns());

    // ------------------------------------------------------------------ phase 2: combine
    {
        rows::CombineArgs ca;
        ca.y = ws.y;
        ca.yrow = ws.yrow;
        ca.w = f.wts;
        ca.out = f.out;
        ca.T = T;
        ca.K = K;
        ca.H = H;
        ca.y8 = f.y8;
        ca.ys = f.ys;
        BMOE_BOUNDS_ONLY(ca.status = ws.status; ca.ticket = ws.ticket; ca.lim_rows = ws.lim_rows;
                         ca.lim_slots = ws.lim_slots;)
        const int items = rows::combine_items(ca);
        for (int it = blockIdx.x * (blockDim.x >> 5) + warp; it < items; it += gridDim.x * (blockDim.x >> 5))
            rows::combine_item(ca, it, lane);
    }
finish:
    __syncthreads();
    if (threadIdx.x == 0) FTRACE(10, (long long)globaltimer_ns());
}

}  // namespace

bool fused_supported(const Geometry& g) {
    return g.NT == F_NT && g.E <= F_TAB_E && g.cap <= 512 && g.K <= kMaxTopk;
}

cudaError_t fused_set_attributes() {
    return cudaFuncSetAttribute(k_fused, cudaFuncAttributeMaxDynamicSharedMemorySize, F_SMEM);
}

cudaError_t launch_fused(const Geometry& g, const Workspace& ws, const FusedLaunch& fl, const CUtensorMap* tm_w13p,
                         const CUtensorMap* tm_aq, const CUtensorMap* tm_w2, const CUtensorMap* tm_hq, int grid,
                         cudaStream_t s) {
    FusedArgs f{};
    f.q.x = fl.x;
    f.q.ids = fl.ids;
    f.q.T = fl.T;
    f.q.K = g.K;
    f.q.E = g.E;
    f.q.H = g.H;
    f.q.mtpr = g.mtpr;
    f.q.words = g.words;
    f.q.NT = g.NT;
    f.q.nb = g.nb;
    f.q.scheme = g.scheme;
    f.q.ws = ws;
    f.nvr = fl.nvr;
    f.wts = fl.wts;
    f.out = fl.out;
    f.w13s = fl.w13s;
    f.w2s = fl.w2s;
    f.I = g.I;
    f.w13_rs = fl.w13_rs;
    f.w13_up = fl.w13_up;
    f.y8 = fl.y8;
    f.ys = fl.ys;
    f.kc2 = g.I % 256 == 0 ? 2 : 1;
    f.w2w = g.H % 256 == 0 ? 1 : 0;
    f.nchunks = (fl.T * g.K + kChunk - 1) / kChunk;
    f.tiles_cap = static_cast<int>(g.tiles_cap);
    f.swiglu_limit = fl.swiglu_limit;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(F_THREADS);
    cfg.dynamicSmemBytes = F_SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_fused, *tm_w13p, *tm_aq, *tm_w2, *tm_hq, f);
}

}  // namespace bmoe

#ifdef BMOE_TRACE
extern "C" int bmoe_fused_trace_copy(void* dst, size_t bytes) {
    return static_cast<int>(cudaMemcpyFromSymbol(dst, g_fused_trace, bytes < sizeof(g_fused_trace) ? bytes : sizeof(g_fused_trace)));
}
extern "C" int bmoe_fused_stage_trace_copy(void* dst, size_t bytes) {
    return static_cast<int>(cudaMemcpyFromSymbol(
        dst, g_fused_stage_trace, bytes < sizeof(g_fused_stage_trace) ? bytes : sizeof(g_fused_stage_trace)));
}
#endif

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
// GEMM tiles are the decode width (N <= 32 routed rows, 4 MMA-issuing warps
// each owning an accumulator chain); a stage holds up to two 128x128 weight
// chunks (GEMM1: gate and up; GEMM2: two 128-wide K chunks) and two row chunks.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "gemm_common.cuh"
#include "layer_rows.cuh"
#include "moe_internal.h"
#include "ptx.cuh"

namespace bmoe {

namespace {

constexpr int F_NT = 32;                                    // route tile width
constexpr int F_MW = 4;                                     // accumulator chains = MMA-issuing warps
constexpr int F_EW = 4;                                     // epilogue warps (one per TMEM lane quadrant)
constexpr int F_THREADS = 32 * (2 + F_MW + F_EW);
constexpr int F_MMA_WARP0 = 2, F_EPI_WARP0 = 2 + F_MW;
constexpr int F_A_BYTES = 128 * 128;                        // one 128x128 FP4 chunk in smem
constexpr int F_A_TX = 128 * 128 / 2;                       // ... and its transaction bytes
constexpr int F_B_BYTES = F_NT * 128;                       // one row chunk
constexpr int F_STAGE_BYTES = 2 * F_A_BYTES + 2 * F_B_BYTES + 4 * 512;
constexpr int F_TAB_E = 512;                                // the fused path needs E <= 512
constexpr int F_TAB_BYTES = 4 * (3 * F_TAB_E + 4);
constexpr int F_SCR_INTS = 2 * F_TAB_E + 64;                // phase-0 scratch, inside the (idle) stage ring
constexpr int F_STAGES = (220 * 1024 - F_TAB_BYTES) / F_STAGE_BYTES;
constexpr int F_ACC_COLS = F_MW * F_NT;
constexpr int F_SF_SLOT = 16;                               // [A atom 0|A atom 1|B atom 0|B atom 1]
constexpr int F_SF_BASE = 512 - F_MW * 2 * F_SF_SLOT;
constexpr int F_NUM_ACC = 2;
constexpr int F_BAR_BYTES = (2 * F_STAGES + 2 * 2 + 1) * 8 + 16;
constexpr int F_SMEM = 1024 + F_STAGES * F_STAGE_BYTES + F_TAB_BYTES + F_BAR_BYTES;
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
    int kc2;               // K chunks per GEMM2 stage (2 when I % 256 == 0)
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

__global__ void __launch_bounds__(F_THREADS, 1)
    k_fused(const __grid_constant__ CUtensorMap tm_w13, const __grid_constant__ CUtensorMap tm_aq,
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
    if (threadIdx.x == 0) *abort_flag = 0;
    __syncthreads();

    // ------------------------------------------------------------------ phase 0: dispatch + quant
    for (int i = gtid; i < f.tiles_cap; i += gstride) ws.ready[i] = 0;
    if (q.scheme == 1) {
        // fixed-slot (vLLM PR #61262): slot (e, t), occupancy bits, no prepare step
        for (int i = gtid; i < E * q.words; i += gstride) ws.occ[i] = 0;
        if (!grid_sync(bar_count, bar_gen, ws.status, abort_flag)) goto finish;
        for (int s = gtid; s < T * K; s += gstride) {
            const int t = s / K, e = q.ids[s];
            if (t < nvr && e >= E) atomicOr(ws.status, kStBadId);
            if (t < nvr && e >= 0 && e < E) {
                atomicOr(&ws.occ[(size_t)e * q.words + (t >> 5)], 1u << (t & 31));
                ws.route_slot[s] = e * q.mtpr + t;
            } else {
                ws.route_slot[s] = -1;
            }
        }
        if (!grid_sync(bar_count, bar_gen, ws.status, abort_flag)) goto finish;
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
                        ws.route_row[s] = p;
                        ws.perm[p] = s;
                    } else if (in) {
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
    // quantise + scatter: one warp per row
    for (int t = blockIdx.x * (blockDim.x >> 5) + warp; t < T; t += gridDim.x * (blockDim.x >> 5))
        rows::quant_scatter_row(q, t_row, t_tile, t, nvr, lane);
    fence_proxy_async_all();  // the packed rows and scale atoms are read by TMA / bulk copies
    if (!grid_sync(bar_count, bar_gen, ws.status, abort_flag)) goto finish;

    // ------------------------------------------------------------------ phase 1: GEMM1 + GEMM2
    {
        const int ntiles = t_tile[E];
        const int mt1 = I / 128, mt2 = H / 128;
        const int U1 = ntiles * mt1, U = U1 + ntiles * mt2;
        const int my_units = static_cast<int>(blockIdx.x) < U
                                 ? (U - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                                 : 0;
        const int kt1 = H / 128, kt2 = I / (128 * f.kc2), ktot2 = I / 128;
        const Plan pl{t_tile, t_row, t_cnt};
        if (threadIdx.x == 0) {
            for (int s = 0; s < F_STAGES; ++s) {
                mbar_init(&full[s], 1 + 32);
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

        if (warp == 0) {
            // -------------------------------------------------------- TMA producer (one thread)
            if (lane == 0 && my_units > 0) {
                const uint64_t pol_w = policy_evict_first(), pol_b = policy_evict_last();
                int stage = 0;
                uint32_t phase = 0;
                long issued = 0;
                bool ok = true;
                FCursor cur;
                fence_proxy_async_all();  // phase-0 rows and scale atoms are read through the async proxy
                for (int ui = 0; ui < my_units && ok; ++ui) {
                    const FUnit fu = fused_unit(blockIdx.x + ui * gridDim.x, U1, cur, pl, mt1, mt2);
                    const UnitInfo& cu = fu.u;
                    const int kt = fu.g2 ? kt2 : kt1;
                    if (fu.g2) {
                        // the h rows of tile g are complete once all epilogue warps of its I/128 GEMM1
                        // units released them
                        const uint64_t t0 = globaltimer_ns();
                        while (ld_acquire_u32(&ws.ready[cu.g]) != static_cast<uint32_t>(mt1 * F_EW)) {
                            if (*abort_flag || globaltimer_ns() - t0 > kWaitLimitNs) {
                                atomicOr(ws.status, kStTimeout | kSiteReady);
                                *abort_flag = 1;
                                ok = false;
                                break;
                            }
                            __nanosleep(64);
                        }
                        if (!ok) break;
                        fence_proxy_async_all();
                    }
                    for (int kk = 0; kk < kt; ++kk) {
                        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, ws.status,
                                       kStTimeout | (1u << (kSiteShift + 0)), kWaitLimitNs)) {
                            ok = false;
                            break;
                        }
                        if (!fu.g2) {
                            const int wrow = cu.e * 2 * I + cu.m * 128;
                            mbar_expect_tx(&full[stage], 2 * F_A_TX + F_B_BYTES + 512);
                            tma_load_2d(sA + (stage * 2) * F_A_BYTES, &tm_w13, &full[stage], kk * 128, wrow, pol_w);
                            tma_load_2d(sA + (stage * 2 + 1) * F_A_BYTES, &tm_w13, &full[stage], kk * 128, wrow + I,
                                        pol_w);
                            tma_load_2d(sB + (stage * 2) * F_B_BYTES, &tm_aq, &full[stage], kk * 128, cu.row0, pol_b);
                            bulk_load(sSFB + (stage * 2) * 512, ws.as + ((size_t)cu.g * kt1 + kk) * 512, 512,
                                      &full[stage]);
                        } else {
                            const int wrow = cu.e * H + cu.m * 128;
                            mbar_expect_tx(&full[stage], f.kc2 * (F_A_TX + F_B_BYTES + 512));
                            for (int c = 0; c < f.kc2; ++c) {
                                const int k0 = (kk * f.kc2 + c) * 128;
                                tma_load_2d(sA + (stage * 2 + c) * F_A_BYTES, &tm_w2, &full[stage], k0, wrow, pol_w);
                                tma_load_2d(sB + (stage * 2 + c) * F_B_BYTES, &tm_hq, &full[stage], k0, cu.row0,
                                            pol_b);
                            }
                            bulk_load(sSFB + (stage * 2) * 512, ws.hs + ((size_t)cu.g * ktot2 + kk * f.kc2) * 512,
                                      f.kc2 * 512, &full[stage]);
                        }
                        mbar_arrive(&full[stage]);
                        ++issued;
                        if (++stage == F_STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
                drain_stages<F_STAGES>(full, stage, phase, issued, ws.status);
            }
        } else if (warp == 1) {
            // -------------------------------------------------------- weight-scale producer (32 lanes)
            int stage = 0;
            uint32_t phase = 0;
            FCursor cur;
            bool ok = true;
            for (int ui = 0; ui < my_units && ok; ++ui) {
                const FUnit fu = fused_unit(blockIdx.x + ui * gridDim.x, U1, cur, pl, mt1, mt2);
                const UnitInfo& cu = fu.u;
                const int kt = fu.g2 ? kt2 : kt1;
                const uint8_t* wsf = fu.g2 ? f.w2s : f.w13s;
                const int ld = fu.g2 ? I / 32 : H / 32;
                const int wrow = fu.g2 ? cu.e * H + cu.m * 128 : cu.e * 2 * I + cu.m * 128;
                const uint8_t* base = wsf + (static_cast<size_t>(wrow) + lane) * ld;
                for (int kk = 0; kk < kt; ++kk) {
                    uint32_t wv[8];
                    // atom a: GEMM1 -> (gate, up) rows, K chunk kk; GEMM2 -> K chunk kk*kc2 + a
#pragma unroll
                    for (int a4 = 0; a4 < 2; ++a4) {
                        const bool use = !fu.g2 || a4 < f.kc2;
                        const uint8_t* src = fu.g2 ? base + (kk * f.kc2 + a4) * 4
                                                   : base + static_cast<size_t>(a4 * I) * ld + kk * 4;
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            wv[4 * a4 + i] =
                                use ? __ldg(reinterpret_cast<const uint32_t*>(src + static_cast<size_t>(32 * i) * ld))
                                    : 0u;
                    }
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, ws.status,
                                   kStTimeout | (1u << (kSiteShift + 0)), kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    uint4* dst = reinterpret_cast<uint4*>(sSFA + (stage * 2) * 512) + lane;
                    dst[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                    dst[32] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
                    fence_proxy_async_smem();
                    mbar_arrive(&full[stage]);
                    if (++stage == F_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        } else if (warp < F_EPI_WARP0) {
            // -------------------------------------------------------- MMA issuers (one chain each)
            const int w = warp - F_MMA_WARP0;
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            long job = 0;
            bool ok = true;
            FCursor cur;
            for (int ui = 0; ui < my_units && ok; ++ui) {
                const FUnit fu = fused_unit(blockIdx.x + ui * gridDim.x, U1, cur, pl, mt1, mt2);
                const int N = (fu.u.n + 15) & ~15;
                const int kt = fu.g2 ? kt2 : kt1;
                const int kc = fu.g2 ? f.kc2 : 1;
                // GEMM1: chain w = (operand w&1: gate/up, K-steps k%2 == w>>1); GEMM2: K-steps k%4 == w
                const int op = fu.g2 ? 0 : (w & 1);
                const int ks = fu.g2 ? 4 : 2, kq = fu.g2 ? w : (w >> 1);
                const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * F_ACC_COLS + w * F_NT);
                if (!mbar_wait(&acce[acc], acc_phase ^ 1u, abort_flag, ws.status,
                               kStTimeout | (1u << (kSiteShift + 2)), kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kk = 0; kk < kt; ++kk) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, ws.status, kStTimeout | (1u << (kSiteShift + 3)),
                                   kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t sfc =
                            tmem + static_cast<uint32_t>(F_SF_BASE + (w * 2 + (job & 1)) * F_SF_SLOT);
                        if (!fu.g2) {
                            tc_cp_32x128b_x4(sfc, desc_sf_atom(smem_u32(sSFA + (stage * 2 + op) * 512)));
                            tc_cp_32x128b_x4(sfc + 8, desc_sf_atom(smem_u32(sSFB + (stage * 2) * 512)));
                        } else {
                            for (int c = 0; c < kc; ++c) {
                                tc_cp_32x128b_x4(sfc + 4 * c, desc_sf_atom(smem_u32(sSFA + (stage * 2 + c) * 512)));
                                tc_cp_32x128b_x4(sfc + 8 + 4 * c,
                                                 desc_sf_atom(smem_u32(sSFB + (stage * 2 + c) * 512)));
                            }
                        }
                        for (int k = kq; k < 4 * kc; k += ks) {
                            const int c = fu.g2 ? (k >> 2) : 0, k4 = k & 3;
                            const int achunk = fu.g2 ? c : op;
                            const uint64_t da = desc_kmajor_sw128(smem_u32(sA + (stage * 2 + achunk) * F_A_BYTES)) +
                                                static_cast<uint64_t>((k4 * 32) >> 4);
                            const uint64_t db = desc_kmajor_sw128(smem_u32(sB + (stage * 2 + c) * F_B_BYTES)) +
                                                static_cast<uint64_t>((k4 * 32) >> 4);
                            const uint32_t idesc = idesc_mx(128, N, 5, 0, k4, k4);
                            tc_mma_mx(d_tmem, da, db, idesc, sfc + 4 * (fu.g2 ? c : 0), sfc + 8 + 4 * c,
                                      (kk > 0 || k != kq) ? 1u : 0u);
                        }
                        tc_commit(&empty[stage]);
                    }
                    __syncwarp();
                    ++job;
                    if (++stage == F_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (lane == 0) tc_commit(&accf[acc]);
                __syncwarp();
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (lane == 0) tc_commit(drain);
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
            for (int ui = 0; ui < my_units; ++ui) {
                const FUnit fu = fused_unit(blockIdx.x + ui * gridDim.x, U1, cur, pl, mt1, mt2);
                const UnitInfo& cu = fu.u;
                if (!mbar_wait(&accf[acc], acc_phase, abort_flag, ws.status, kStTimeout | (1u << (kSiteShift + 5)),
                               kWaitLimitNs))
                    break;
                tc_fence_after();
                const uint32_t tb =
                    tmem + (static_cast<uint32_t>(32 * qd) << 16) + static_cast<uint32_t>(acc * F_ACC_COLS);
                const int feat = cu.m * 128 + 32 * qd + lane;
                float v[F_NT];
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
                            // chains summed in the multi-kernel path's order, from +0 (same bits)
                            float ga = 0.f, ub = 0.f;
#pragma unroll
                            for (int w = 0; w < F_MW; ++w) {
                                if (!fu.g2 && (w & 1))
                                    ub += __uint_as_float(r[w][i]);
                                else
                                    ga += __uint_as_float(r[w][i]);
                            }
                            if (!fu.g2) {
                                if (ws.g && c0 + i < cu.n) {
                                    const size_t prow = static_cast<size_t>(cu.row0 + c0 + i);
                                    ws.g[prow * 2 * I + feat] = ga;
                                    ws.g[prow * 2 * I + I + feat] = ub;
                                }
                                if (L > 0.f) {
                                    ga = fminf(ga, L);
                                    ub = fminf(fmaxf(ub, -L), L);
                                }
                                v[c0 + i] = ga * (1.0f / (1.0f + expf(-ga))) * ub;
                            } else {
                                v[c0 + i] = ga;
                            }
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&acce[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
#pragma unroll
                for (int c = 0; c < F_NT; ++c) {
                    if (c < cu.n) {
                        const size_t prow = static_cast<size_t>(cu.row0 + c);
                        if (!fu.g2) {
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
                if (!fu.g2) {
                    // Release this warp's 32 features of tile g's h rows to the GEMM2 units (TMA reads
                    // them from any CTA); warps release independently, nobody waits here.
                    fence_proxy_async_all();
                    __threadfence();
                    __syncwarp();
                    if (lane == 0) {
                        __threadfence();
                        atom_add_release_u32(&ws.ready[cu.g], 1u);
                    }
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        if (warp == F_MMA_WARP0) {
            tc_fence_after();
            tmem_dealloc(tmem, 512);
        }
    }
    if (!grid_sync(bar_count, bar_gen, ws.status, abort_flag)) goto finish;

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
        for (int t = blockIdx.x * (blockDim.x >> 5) + warp; t < T; t += gridDim.x * (blockDim.x >> 5))
            rows::combine_row(ca, t, lane);
    }
finish:
    return;
}

}  // namespace

bool fused_supported(const Geometry& g) {
    return g.NT == F_NT && g.E <= F_TAB_E && g.cap <= 512 && g.K <= kMaxTopk;
}

cudaError_t fused_set_attributes() {
    return cudaFuncSetAttribute(k_fused, cudaFuncAttributeMaxDynamicSharedMemorySize, F_SMEM);
}

cudaError_t launch_fused(const Geometry& g, const Workspace& ws, const FusedLaunch& fl, const CUtensorMap* tm_w13,
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
    f.q.scheme = g.scheme;
    f.q.ws = ws;
    f.nvr = fl.nvr;
    f.wts = fl.wts;
    f.out = fl.out;
    f.w13s = fl.w13s;
    f.w2s = fl.w2s;
    f.I = g.I;
    f.kc2 = g.I % 256 == 0 ? 2 : 1;
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
    return cudaLaunchKernelEx(&cfg, k_fused, *tm_w13, *tm_aq, *tm_w2, *tm_hq, f);
}

}  // namespace bmoe

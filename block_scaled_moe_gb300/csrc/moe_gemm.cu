// moe_gemm.cu -- grouped block-scaled GEMMs of the MoE layer on the 5th-generation
// tensor cores (tcgen05.mma kind::mxf8f6f4 with E8M0 block scales).
//
// Orientation ("swap-AB"): the expert weight tile is the M=128 operand A and the
// expert's dispatched rows are the N operand B, so an expert with n routed rows
// runs MMAs of N = roundup(n, 16) instead of padding rows to 128.  For decode,
// where a few rows meet each expert, the layer is a stream over the active
// experts' weights (ROCm/aiter PR #6881 Technical Details: the small-input path
// is dominated by reading expert weights); for prefill the same kernel runs
// route tiles of up to NT=144 rows.
//
//   GEMM1 unit = (route tile, pair m): gate rows [128m,128m+128) and up rows
//     I+[128m,128m+128) of W13[e], K = H.  Epilogue: SwiGLU (optional clamp,
//     ROCm/aiter PR #6154 "clamp-10 SwiGLU") and MXFP8 1x32 re-quantisation of
//     h along I ("FP8 intermediate quantization", aiter #6154 Summary).
//   GEMM2 unit = (route tile, tile m): rows [128m,128m+128) of W2[e], K = I; or,
//     when H % 256 == 0, (route tile, pair m): rows [256m,256m+256), one 256-row
//     box per K stage.  Epilogue: BF16 rows y (aiter #6881: GEMM2 rows go to the
//     combine as BF16).
//
// Pipeline per CTA (persistent, one CTA per SM, units strided over the grid; the
// CTA's units are decoded once into a shared-memory table before the roles start):
//   warp 0      TMA producer (one thread): TMA of the FP4 weight tile
//               (16U4_ALIGN16B expands each 16 codes to 16 bytes in shared
//               memory, the layout kind::mxf8f6f4 reads), TMA of the FP8 row
//               tile and bulk copy of the rows' scale atom.
//   warp 1      scale producer: the weight scales gathered from their natural
//               [rows, K/32] layout into a 128x4 scale atom by the warp's 32
//               lanes, loaded 8 stages ahead into registers and stored with a
//               proxy fence before the stage's arrival.
//   warps 2..   MMA issuers, the whole warp converged and one elected lane
//               issuing (~44 cycles per MMA at N = 32; small-N decode MMAs are
//               still issue bound); MW warps each own an accumulator chain (gate
//               or up, and a residue class of the K-steps) and issue in
//               parallel.  Each copies the stage's scale atoms into its own TMEM
//               columns.
//   last EW     epilogue warps: tcgen05.ld of the MW partial accumulators (lane =
//               output feature, column = routed row) and their fixed-order sum
//               into registers, release of the accumulator, then the
//               SwiGLU/MXFP8 or BF16 epilogue and global stores.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "gemm_common.cuh"
#include "layer_rows.cuh"
#include "moe_internal.h"
#include "ptx.cuh"

namespace bmoe {

namespace {

template <bool G1, int NT, int KC, bool WIDE>
struct Cfg {
    // A K stage is KC chunks of 128 K-elements (one 128-byte swizzle atom each).
    // WIDE (GEMM2, 128-row route tiles): a unit takes two adjacent 128-row W2 tiles
    // against one route tile, like GEMM1's gate/up pair, so that a stage streams
    // 16 KB of weights per 16 KB row chunk instead of 8 KB.
    static constexpr bool PAIR = G1 || WIDE;                // two weight operands per stage
    static constexpr int NA = PAIR ? 2 : 1;                 // weight operands per stage (gate/up, W2 pair or W2)
    static constexpr int A_BYTES = 128 * 128;              // one 128x128 weight chunk in smem (1 byte per code)
    // Transaction bytes of one 128x128 FP4 box: the TMA counts the packed bytes it
    // reads (two codes per byte), not the 16-byte-aligned footprint it writes.
    static constexpr int A_TX = 128 * 128 / 2;
    static constexpr int B_BYTES = NT * 128;               // one row chunk in smem
    static constexpr int NB = (NT + 127) / 128;            // 128-row scale atoms per row chunk
    static constexpr int STAGE_BYTES = KC * (NA * A_BYTES + B_BYTES + (NA + NB) * 512);
    static constexpr int UTAB = 384;                       // the CTA's first units, decoded once (16 bytes each)
    static constexpr int UTAB_BYTES = 16 * UTAB;
    static constexpr int STAGES = (220 * 1024 - UTAB_BYTES) / STAGE_BYTES > 12 ? 12
                                                                              : (220 * 1024 - UTAB_BYTES) / STAGE_BYTES;
    // MMA issuers and their accumulator chains: two for decode tiles (gate / up, the two
    // tiles of a W2 pair, or the halves of a stage's K-steps: each chain copies its own
    // scale atoms per stage, so more chains cost more copies than they save in issue) and
    // for the prefill pairs; one for unpaired 128-wide GEMM2 tiles, so that GEMM2's
    // accumulator can be double-buffered in TMEM.
    static constexpr int MW = NT <= 64 ? 2 : (PAIR ? 2 : 1);
    static constexpr int NI = MW;                          // MMA-issuing warps (chain w is issued by warp w % NI)
    static constexpr int KS = PAIR ? MW / 2 : MW;          // K-steps of a stage split over KS chains per operand
    static constexpr int EW = NT <= 64 ? 4 : 8;            // epilogue warps (EW/4 per TMEM lane quadrant)
    static constexpr int CW = NT / (EW / 4);               // accumulator columns per epilogue warp
    static constexpr int ACC_COLS = MW * NT;               // one accumulator set: MW chains of NT columns
    static constexpr int SF_SLOTS = 2;                     // scale slots per chain (alternating stages)
    // KC weight atoms, then KC x NB row atoms, 4 columns each (row atom b holds rows 128 b .. 128 b + 127)
    static constexpr int SF_SLOT_COLS = 4 * KC * (1 + NB);
    static constexpr int SF_BASE = 512 - MW * SF_SLOTS * SF_SLOT_COLS;
    // 128-row tiles with two chains (GEMM1 gate/up, paired W2 tiles) cannot double-buffer 2 x 256
    // columns next to the scale columns; they rotate three single-chain slots instead: unit u's chain w
    // accumulates in slot (2u + w) % 3, each slot with its own full / free barriers, so the next unit's
    // first chain always finds a free slot and its second waits only for one drained slot.
    static constexpr bool ROT3 = PAIR && NT >= 128;
    static constexpr int NUM_ACC = ROT3 ? 1 : ((2 * ACC_COLS <= SF_BASE) ? 2 : 1);
    // warps: 0 TMA producer, 1 scale producer, 2..1+NI MMA issuers, then EW epilogue warps
    static constexpr int MMA_WARP0 = 2;
    static constexpr int EPI_WARP0 = 2 + NI;
    static constexpr int THREADS = 32 * (2 + NI + EW);
    static constexpr int BAR_BYTES = (2 * STAGES + 4 + 4 + 1) * 8 + 16;
    static constexpr int UTAB_OFF = (STAGES * STAGE_BYTES + BAR_BYTES + 15) & ~15;
    static constexpr int SMEM = 1024 + UTAB_OFF + UTAB_BYTES;
    // the plan's three tables are staged in the stage ring (idle until the pipeline starts) while
    // the units are decoded
    static_assert(STAGES * STAGE_BYTES >= 4 * 3 * (kMaxExperts + 1), "plan staging");
    static_assert(NUM_ACC * ACC_COLS <= SF_BASE, "TMEM columns");
    static_assert(SMEM <= 232448, "shared memory");
    static_assert(4 % KS == 0, "K-steps per stage must split evenly");
    static_assert(!G1 || KC == 1, "GEMM1 stages hold one K chunk (the W13 pair box)");
    static_assert(!WIDE || (!G1 && KC == 1), "wide units: GEMM2 with one K chunk per stage");
    static_assert(!ROT3 || (MW == 2 && NI == 2 && 3 * NT <= SF_BASE), "three rotating slots");
    static_assert(MW <= 4, "barrier slots");
    static_assert(CW % 8 == 0, "epilogue column split");
    static constexpr int LDC = CW % 16 == 0 ? 16 : 8;      // TMEM columns per epilogue load
    static constexpr bool SF_VEC = KC == 1 && NT >= 128;   // prefill tiles: weight scales as 8- or 16-byte vectors
};

// SwiGLU of one (gate, up) pair with the optional clamp (ROCm/aiter PR #6154 "clamp-10 SwiGLU":
// gate <= L, -L <= up <= L), fast exp / divide intrinsics; the clamp is a select, not a branch.
__device__ __forceinline__ float swiglu(float ga, float ub, bool clamp, float L) {
    ga = clamp ? fminf(ga, L) : ga;
    ub = clamp ? fminf(fmaxf(ub, -L), L) : ub;
    return __fdividef(ga, 1.0f + __expf(-ga)) * ub;
}

// BF16 rows of one warp's features: v[j] is row (row0 + j), feature `feat`, for j < n (n may exceed
// CW or be <= 0).  Eight rows per group, branch-free stores for full groups.
template <int CW>
__device__ __forceinline__ void store_rows_bf16(uint16_t* y, const float (&v)[CW], int row0, int n, int H, int feat) {
#pragma unroll
    for (int j0 = 0; j0 < CW; j0 += 8) {
        if (j0 >= n) break;
        uint16_t* yr = y + static_cast<size_t>(row0 + j0) * H + feat;
        if (j0 + 8 <= n) {
#pragma unroll
            for (int i = 0; i < 8; ++i) yr[static_cast<size_t>(i) * H] = __bfloat16_as_ushort(__float2bfloat16_rn(v[j0 + i]));
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (j0 + i < n) yr[static_cast<size_t>(i) * H] = __bfloat16_as_ushort(__float2bfloat16_rn(v[j0 + i]));
        }
    }
}

// 32-bit word j of a vector of weight-scale words
__device__ __forceinline__ uint32_t vword(const uint4& v, int j) {
    return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}
__device__ __forceinline__ uint32_t vword(const uint2& v, int j) { return j == 0 ? v.x : v.y; }

// LDC-column TMEM load (32 lanes x 32 bit) of the epilogue
template <int L>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[L]) {
    if constexpr (L == 16)
        tmem_ld16(taddr, r);
    else
        tmem_ld8(taddr, r);
}

template <bool G1, int NT, int KC, bool WIDE>
__global__ void __launch_bounds__(Cfg<G1, NT, KC, WIDE>::THREADS, 1)
    k_gemm(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_b, const GemmArgs a) {
    using C = Cfg<G1, NT, KC, WIDE>;
    constexpr int STAGES = C::STAGES, NA = C::NA, MW = C::MW, KS = C::KS, NI = C::NI;
    constexpr bool PAIR = C::PAIR;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = sm;
    // per stage: sA [NA][KC] chunks, sB [KC] chunks, sSFA [NA][KC] atoms, sSFB [KC][NB] atoms
    constexpr int NB = C::NB;
    uint8_t* sB = sA + STAGES * NA * KC * C::A_BYTES;
    uint8_t* sSFA = sB + STAGES * KC * C::B_BYTES;
    uint8_t* sSFB = sSFA + STAGES * NA * KC * 512;
    uint64_t* full = reinterpret_cast<uint64_t*>(sSFB + STAGES * KC * NB * 512);
    uint64_t* empty = full + STAGES;
    uint64_t* accf = empty + STAGES;  // accumulator full: [2] sets, or [3] rotating slots (ROT3)
    uint64_t* acce = accf + 4;        // accumulator free, same indexing
    uint64_t* drain = acce + 4;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int4* utab = reinterpret_cast<int4*>(sm + C::UTAB_OFF);  // [UTAB] decoded units of this CTA

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) trace_cta(a, 0);
    const int ntiles = __ldg(a.tile_base + a.E);
    const int n_units = ntiles * a.mtiles;
    if (static_cast<int>(blockIdx.x) >= n_units) return;  // whole CTA
#ifdef MOE_DEBUG_BOUNDS
    const int all_units =
#else
    const int my_units =
#endif
        (n_units - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1;
    const int KT = a.ktiles / KC;  // K stages per unit

    // The CTA's units are decoded once (bisection per unit, one thread each) from a copy of the plan
    // staged in the idle stage ring; units past the table, and the bounds check, read the global plan.
    const Plan pl{a.tile_base, a.rowbase, a.counts};
    {
        int32_t* ptab = reinterpret_cast<int32_t*>(sA);
        const int E = a.E;
        for (int i = threadIdx.x; i <= E; i += blockDim.x) {
            ptab[i] = __ldg(a.tile_base + i);
            ptab[E + 1 + i] = __ldg(a.rowbase + i);
            if (i < E) ptab[2 * E + 2 + i] = __ldg(a.counts + i);
        }
        __syncthreads();
        const Plan sp{ptab, ptab + E + 1, ptab + 2 * E + 2};
#ifdef MOE_DEBUG_BOUNDS
        const int n_tab = min(all_units, C::UTAB);
#else
        const int n_tab = min(my_units, C::UTAB);
#endif
        for (int i = threadIdx.x; i < n_tab; i += blockDim.x) {
            const int u = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
            utab[i] = pack_unit(unit_of_expert(u, expert_of_unit(u, sp, a.mtiles, E), sp, a.mtiles, NT));
        }
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1 + 32);  // TMA issuer + the 32 scale-copying lanes
            mbar_init(&empty[s], NI);
        }
        for (int b = 0; b < 4; ++b) {
            mbar_init(&accf[b], C::ROT3 ? 1 : NI);  // ROT3: one chain (one issuing warp) per slot use
            mbar_init(&acce[b], 32 * C::EW);
        }
        mbar_init(drain, NI);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == C::MMA_WARP0) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
#ifdef MOE_DEBUG_BOUNDS
    int chk_ecur = 0;
    const int my_units = units_in_bounds(
        all_units,
        [&](int i) { return decode_unit(blockIdx.x + i * gridDim.x, chk_ecur, pl, a.mtiles, NT); }, NT, a.lim_rows,
        a.lim_tiles, a.status, a.ticket);
#endif

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (one warp, one elected lane issues)
        {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_b = policy_evict_last();
            if (lane == 0) {
                prefetch_tmap(&tm_w);
                prefetch_tmap(&tm_b);
            }
            __syncwarp();
            int stage = 0, ecur = 0;
            uint32_t phase = 0;
            long issued = 0;
            bool ok = true;
            for (int ui = 0; ui < my_units && ok; ++ui) {
                const UnitInfo cu = unit_ref(ui, utab, C::UTAB, ecur, pl, a.mtiles, NT);
                const int wrow = cu.e * a.w_rows + cu.m * a.m_rows;  // GEMM2 (GEMM1 reads the W13 pair view)
                const uint8_t* b_sf = a.b_sf + static_cast<size_t>(cu.g) * a.ktiles * NB * 512;
                for (int kk = 0; kk < KT; ++kk) {
                    const bool got = mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.status,
                                               kStTimeout | (1u << (kSiteShift + 0)), kWaitLimitNs);
                    if (!__all_sync(0xffffffffu, got)) {  // the lanes agree: the warp stays converged
                        ok = false;
                        break;
                    }
                    if (lane == 0) trace(a, 0, issued);
                    // the producer's arrival carries the stage's transaction bytes; the stage completes
                    // when they have landed and the scale warp has arrived
                    mbar_arrive_expect_tx_w(&full[stage], KC * (NA * C::A_TX + C::B_BYTES + NB * 512));
                    if constexpr (KC == 2) {  // two-chunk views: one box per operand lands both K chunks
                        tma_load_3d_w(sA + (stage * NA) * KC * C::A_BYTES, &tm_w, &full[stage], 0, wrow, kk * KC,
                                      pol_w);
                        tma_load_3d_w(sB + stage * KC * C::B_BYTES, &tm_b, &full[stage], 0, cu.row0, kk * KC, pol_b);
                    } else {
#pragma unroll
                        for (int c = 0; c < KC; ++c) {
                            const int k0 = (kk * KC + c) * 128;
                            if constexpr (G1)  // gate and up tiles of feature tile m: one box {128, 128, 2, 1}
                                tma_load_4d_w(sA + ((stage * NA) * KC + c) * C::A_BYTES, &tm_w, &full[stage], k0,
                                              cu.m * 128, 0, cu.e, pol_w);
                            else  // W2 tile (WIDE: a 256-row box, the unit's two tiles back to back)
                                tma_load_2d_w(sA + ((stage * NA) * KC + c) * C::A_BYTES, &tm_w, &full[stage], k0,
                                              wrow, pol_w);
                            tma_load_2d_w(sB + (stage * KC + c) * C::B_BYTES, &tm_b, &full[stage], k0, cu.row0,
                                          pol_b);
                        }
                    }
                    bulk_load_w(sSFB + stage * KC * NB * 512, b_sf + kk * KC * NB * 512, KC * NB * 512, &full[stage]);
                    if (lane == 0) trace(a, 1, issued);
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (lane == 0) drain_stages<STAGES>(full, stage, phase, issued, a.status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ weight-scale producer (32 lanes)
        // Lane l gathers the 4 K-blocks of the stage for rows l, l+32, l+64, l+96 (one
        // 32-bit word each) and writes them as line l of the 128x4 scale atom.  The
        // words are loaded SD stages ahead of their stage into registers so that
        // their latency stays off this warp's path; the stores are made visible to
        // the tensor core's async proxy here, before the warp arrives on the stage.
        // Prefill tiles leave ~20 KB of L1 beside the stage ring, less than the 32 KB of scale lines a
        // unit touches, so 4-byte gathers per row and stage miss L1 every time and their requests,
        // not the weight stream, set the pace.  When the rows' scale stride allows, each lane loads
        // one 16-byte (else 8-byte) vector per row that holds the scales of 4 (2) consecutive stages,
        // 8 stages ahead.  (Decode tiles keep the 4-byte gathers: their scale lines stay in L1, and
        // 8-byte vectors for the 256-wide GEMM2 stages measured slower.)
        // Vector widths: 16 bytes (uint4) or 8 bytes (uint2) per row, covering SPV = bytes / (4 KC)
        // consecutive K stages, when the scale rows and the unit's stages allow it.
        auto vec_ok = [&](int vb) {
            const int spv = vb / (4 * KC);
            return spv >= 1 && a.ld_sf % vb == 0 && KT % spv == 0 && (reinterpret_cast<uintptr_t>(a.w_sf) % vb) == 0;
        };
        auto vec_loop = [&](auto vtag) {
            using V = decltype(vtag);
            constexpr int WPV = static_cast<int>(sizeof(V)) / 4;  // 32-bit words per vector
            constexpr int SPV = WPV / KC;                         // K stages per vector
            constexpr int GD = 8 / SPV > 1 ? 8 / SPV : 1;          // vector groups loaded ahead (8 stages)
            constexpr int NV = 4 * NA;                            // vectors per lane and group: [op][row group]
            V gring[GD][NV];
            const int GPU = KT / SPV;  // groups per unit
            int q_ui = 0, q_g = 0, q_ecur = 0;
            const uint8_t* q_src = nullptr;
            auto gload = [&](V(&dst)[NV]) {
                if (q_ui >= my_units) return;
                if (q_g == 0) {
                    const UnitInfo pu = unit_ref(q_ui, utab, C::UTAB, q_ecur, pl, a.mtiles, NT);
                    q_src = a.w_sf +
                            (static_cast<size_t>(pu.e) * a.w_rows + (pu.m * a.m_rows + lane) * a.w_rs) * a.ld_sf;
                }
#pragma unroll
                for (int op = 0; op < NA; ++op)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[op * 4 + i] = __ldg(reinterpret_cast<const V*>(
                            q_src + static_cast<size_t>(op * a.up_off + 32 * i * a.w_rs) * a.ld_sf +
                            static_cast<size_t>(q_g) * sizeof(V)));
                if (++q_g == GPU) {
                    q_g = 0;
                    ++q_ui;
                }
            };
#pragma unroll
            for (int d = 0; d < GD; ++d) gload(gring[d]);
            const long ngroups = static_cast<long>(my_units) * GPU;
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            long sjob = 0;
            for (long G0 = 0; G0 < ngroups && ok; G0 += GD) {
#pragma unroll
                for (int d = 0; d < GD; ++d) {
                    if (G0 + d >= ngroups || !ok) continue;
#pragma unroll
                    for (int sq = 0; sq < SPV; ++sq) {
                        if (!ok) continue;
                        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.status,
                                       kStTimeout | (1u << (kSiteShift + 0)), kWaitLimitNs)) {
                            ok = false;
                            continue;
                        }
                        if (lane == 0) trace(a, 6, sjob);
                        uint4* dst = reinterpret_cast<uint4*>(sSFA + stage * NA * KC * 512) + lane;
#pragma unroll
                        for (int op = 0; op < NA; ++op)
#pragma unroll
                            for (int c = 0; c < KC; ++c) {  // atom (op, chunk): word sq * KC + c of each row
                                const V* v = gring[d] + op * 4;
                                const int j = sq * KC + c;
                                dst[32 * (op * KC + c)] =
                                    make_uint4(vword(v[0], j), vword(v[1], j), vword(v[2], j), vword(v[3], j));
                            }
                        fence_proxy_async_smem();
                        mbar_arrive(&full[stage]);
                        if (lane == 0) trace(a, 7, sjob);
                        ++sjob;
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (ok) gload(gring[d]);
                }
            }
        };
        if (C::SF_VEC && vec_ok(16)) {
            vec_loop(uint4{});
        } else if (C::SF_VEC && vec_ok(8)) {
            vec_loop(uint2{});
        } else {
            constexpr int SD = 8;
            constexpr int NW = 4 * NA * KC;  // words per lane per stage: [op][chunk][row group]
            uint32_t ring[SD][NW];
            int p_ui = 0, p_kk = 0, p_ecur = 0;  // load cursor (SD stages ahead)
            const uint8_t* p_src = nullptr;
            auto load_next = [&](uint32_t(&dst)[NW]) {
                if (p_ui >= my_units) return;
                if (p_kk == 0) {
                    const UnitInfo pu = unit_ref(p_ui, utab, C::UTAB, p_ecur, pl, a.mtiles, NT);
                    p_src = a.w_sf + (static_cast<size_t>(pu.e) * a.w_rows + (pu.m * a.m_rows + lane) * a.w_rs) * a.ld_sf;
                }
    #pragma unroll
                for (int op = 0; op < NA; ++op)
    #pragma unroll
                    for (int c = 0; c < KC; ++c) {
                        const uint8_t* src = p_src + static_cast<size_t>(op * a.up_off) * a.ld_sf + (p_kk * KC + c) * 4;
    #pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[(op * KC + c) * 4 + i] =
                                __ldg(reinterpret_cast<const uint32_t*>(src + static_cast<size_t>(32 * i * a.w_rs) * a.ld_sf));
                    }
                if (++p_kk == KT) {
                    p_kk = 0;
                    ++p_ui;
                }
            };
    #pragma unroll
            for (int d = 0; d < SD; ++d) load_next(ring[d]);
            const long njobs = static_cast<long>(my_units) * KT;
            int stage = 0;
            uint32_t phase = 0;
            long issued = 0;
            for (long J0 = 0; J0 < njobs; J0 += SD) {
                bool ok = true;
    #pragma unroll
                for (int d = 0; d < SD; ++d) {
                    if (J0 + d < njobs && ok) {
                        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.status,
                                       kStTimeout | (1u << (kSiteShift + 0)), kWaitLimitNs)) {
                            ok = false;
                        } else {
                            uint4* dst = reinterpret_cast<uint4*>(sSFA + stage * NA * KC * 512) + lane;
    #pragma unroll
                            for (int a4 = 0; a4 < NA * KC; ++a4)  // atom (op, chunk) is 32 uint4 further
                                dst[32 * a4] = make_uint4(ring[d][4 * a4], ring[d][4 * a4 + 1], ring[d][4 * a4 + 2],
                                                          ring[d][4 * a4 + 3]);
                            fence_proxy_async_smem();
                            mbar_arrive(&full[stage]);
                            ++issued;
                            if (++stage == STAGES) {
                                stage = 0;
                                phase ^= 1u;
                            }
                            load_next(ring[d]);
                        }
                    }
                }
                if (!ok) break;
            }
        }
    } else if (warp < C::EPI_WARP0) {
        // ------------------------------------------------------------ MMA issuers
        const int wi = warp - C::MMA_WARP0;  // this warp issues chains wi, wi + NI, ...
        int stage = 0, acc = 0, ecur = 0;
        uint32_t phase = 0, acc_phase = 0;
        long job = 0;
        bool ok = true;
        for (int ui = 0; ui < my_units && ok; ++ui) {
            const UnitInfo cu = unit_ref(ui, utab, C::UTAB, ecur, pl, a.mtiles, NT);
            const int N = (cu.n + 15) & ~15;
            // ROT3: this warp's one chain (w = wi) uses slot (2 ui + wi) % 3, its (2 ui + wi) / 3-th use
            const int rq = 2 * ui + wi, rslot = rq % 3;
            // every lane waits; the warp goes on only if all lanes saw the barrier (a timeout in one
            // lane stops the whole warp), so that it stays converged for the elected issue
            const bool got_acc = C::ROT3 ? mbar_wait(&acce[rslot], ((rq / 3) & 1u) ^ 1u, abort_flag, a.status,
                                                     kStTimeout | (1u << (kSiteShift + 2)), kWaitLimitNs)
                                         : mbar_wait(&acce[acc], acc_phase ^ 1u, abort_flag, a.status,
                                                     kStTimeout | (1u << (kSiteShift + 2)), kWaitLimitNs);
            if (!__all_sync(0xffffffffu, got_acc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            for (int kk = 0; kk < KT; ++kk) {
                const bool got = mbar_wait(&full[stage], phase, abort_flag, a.status,
                                           kStTimeout | (1u << (kSiteShift + 3)), kWaitLimitNs);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                {
                    if (wi == 0 && lane == 0) trace(a, 2, job);
#pragma unroll
                    for (int w = wi; w < MW; w += NI) {
                        // GEMM1: chain w multiplies operand w & 1 (0 gate, 1 up) over the K-steps k with
                        // k % KS == w >> 1; GEMM2: chain w takes the G2S consecutive K-steps from w * G2S
                        // (k = 4 * chunk + step in chunk) and needs only the atoms of their chunks.
                        constexpr int G2S = 4 * KC / MW;
                        // (WIDE: chain w multiplies W2 tile w over every K-step, like an operand of the pair.)
                        const int op = PAIR ? (w & 1) : 0;
                        const int kfirst = PAIR ? (w >> 1) : w * G2S;
                        const int c_lo = PAIR ? 0 : (w * G2S) >> 2, c_hi = PAIR ? KC - 1 : (w * G2S + G2S - 1) >> 2;
                        const uint32_t d_tmem =
                            tmem + static_cast<uint32_t>(C::ROT3 ? rslot * NT : acc * C::ACC_COLS + w * NT);
                        const uint32_t sfc = tmem + static_cast<uint32_t>(
                                                        C::SF_BASE + (w * C::SF_SLOTS + (job & 1)) * C::SF_SLOT_COLS);
#pragma unroll
                        for (int c = 0; c < KC; ++c) {
                            if (c < c_lo || c > c_hi) continue;
                            tc_cp_32x128b_x4_w(sfc + 4 * c,
                                               desc_sf_atom(smem_u32(sSFA + ((stage * NA + op) * KC + c) * 512)));
#pragma unroll
                            for (int b = 0; b < NB; ++b)
                                tc_cp_32x128b_x4_w(sfc + 4 * KC + 4 * (c * NB + b),
                                                   desc_sf_atom(smem_u32(sSFB + ((stage * KC + c) * NB + b) * 512)));
                        }
#pragma unroll
                        for (int k = 0; k < 4 * KC; ++k) {
                            if (PAIR ? (k % KS != kfirst) : (k / G2S != w)) continue;
                            const int c = k >> 2, k4 = k & 3;
                            const uint64_t da =
                                desc_kmajor_sw128(smem_u32(sA + ((stage * NA + op) * KC + c) * C::A_BYTES)) +
                                static_cast<uint64_t>((k4 * 32) >> 4);
                            const uint64_t db = desc_kmajor_sw128(smem_u32(sB + (stage * KC + c) * C::B_BYTES)) +
                                                static_cast<uint64_t>((k4 * 32) >> 4);
                            const uint32_t idesc = idesc_mx(128, N, 5, 0, k4, k4);
                            tc_mma_mx_w(d_tmem, da, db, idesc, sfc + 4 * c, sfc + 4 * KC + 4 * NB * c,
                                        (kk > 0 || k != kfirst) ? 1u : 0u);
                        }
                    }
                    tc_commit_w(&empty[stage]);
                    if (wi == 0 && lane == 0) trace(a, 3, job);
                }
                __syncwarp();
                ++job;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            tc_commit_w(&accf[C::ROT3 ? rslot : acc]);
            __syncwarp();
            if (C::NUM_ACC == 2) {
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            } else {
                acc_phase ^= 1u;
            }
        }
        // Drain: all MMAs issued by this warp complete before TMEM is released.
        __syncwarp();
        tc_commit_w(drain);
        __syncwarp();
        {
            volatile int never = 0;
            (void)mbar_wait(drain, 0, &never, a.status, kStTimeout | (1u << (kSiteShift + 4)), kWaitLimitNs);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // Each warp drains CW columns of its TMEM lane quadrant into registers
        // (summing the MW chains in a fixed order), releases the accumulator so
        // the next unit's MMAs can start, then finishes the columns from registers.
        constexpr int CW = C::CW;
        const int q = warp & 3;                              // TMEM lane quadrant this warp may access
        const int cbase = ((warp - C::EPI_WARP0) >> 2) * CW;  // first column of this warp
        int acc = 0, ecur = 0;
        uint32_t acc_phase = 0;
        const float L = a.swiglu_limit;
        const bool clamp = L > 0.f;
        const bool tracer = warp == C::EPI_WARP0 && lane == 0;
        for (int ui = 0; ui < my_units; ++ui) {
            const UnitInfo cu = unit_ref(ui, utab, C::UTAB, ecur, pl, a.mtiles, NT);
            const int feat = cu.m * 128 + 32 * q + lane;
            float v[CW];  // GEMM1: h = SwiGLU(gate, up); GEMM2: y
            float v2[WIDE && !C::ROT3 ? CW : 1];  // GEMM2 wide units without rotating slots: the second tile's y
            if constexpr (C::ROT3) {
                // chain by chain from its rotating slot; each slot is freed as soon as it is drained
                bool ok = true;
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    const int rq = 2 * ui + w, rslot = rq % 3;
                    if (!mbar_wait(&accf[rslot], (rq / 3) & 1u, abort_flag, a.status,
                                   kStTimeout | (1u << (kSiteShift + 5)), kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (tracer && w == 0) trace(a, 4, ui);
                    const uint32_t tbs = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(rslot * NT);
                    constexpr int LDC = C::LDC;
#pragma unroll
                    for (int j = 0; j < CW / LDC; ++j) {  // LDC columns per load: the gate values stay live
                        const int c0 = cbase + LDC * j;
                        if (c0 < cu.n) {
                            uint32_t r[LDC];
                            tmem_ld_cols<LDC>(tbs + c0, r);
                            tmem_ld_wait();
                            if constexpr (G1) {
                                // (the debug capture stores the chain as read, gate in pass 0, up in pass 1)
                                if (a.g_dbg) {
#pragma unroll
                                    for (int i = 0; i < LDC; ++i)
                                        if (c0 + i < cu.n)
                                            a.g_dbg[static_cast<size_t>(cu.row0 + c0 + i) * 2 * a.I + w * a.I + feat] =
                                                0.f + __uint_as_float(r[i]);
                                }
#pragma unroll
                                for (int i = 0; i < LDC; ++i) {
                                    const int vi = LDC * j + i;
                                    if (w == 0) {
                                        v[vi] = 0.f + __uint_as_float(r[i]);  // gate (+0 like the chain sums)
                                    } else {
                                        v[vi] = swiglu(v[vi], 0.f + __uint_as_float(r[i]), clamp, L);
                                    }
                                }
                            } else {
#pragma unroll
                                for (int i = 0; i < LDC; ++i) v[LDC * j + i] = __uint_as_float(r[i]);
                            }
                        }
                    }
                    tc_fence_before();
                    mbar_arrive(&acce[rslot]);
                    if constexpr (WIDE) {  // chain w = W2 tile w of the pair: store its rows now
                        const int featw = cu.m * a.m_rows + w * 128 + 32 * q + lane;
                        if (a.y8) {  // MXFP8 rows: this warp's 32 features are one 1x32 block
#pragma unroll
                            for (int j = 0; j < CW; ++j) {
                                const int c = cbase + j;
                                if (c < cu.n) {
                                    const size_t prow = static_cast<size_t>(cu.row0 + c);
                                    uint8_t sc;
                                    a.y8[prow * a.H + featw] = rows::quant_block_warp(v[j], &sc);
                                    if (lane == 0) a.ys[prow * (a.H >> 5) + (featw >> 5)] = sc;
                                }
                            }
                        } else {
                            store_rows_bf16<CW>(a.y, v, cu.row0 + cbase, cu.n - cbase, a.H, featw);
                        }
                    }
                }
                if (!ok) break;
                if (tracer) trace(a, 5, ui);
                if constexpr (WIDE) continue;
            } else {
                if (!mbar_wait(&accf[acc], acc_phase, abort_flag, a.status, kStTimeout | (1u << (kSiteShift + 5)),
                               kWaitLimitNs))
                    break;
                tc_fence_after();
                if (tracer) trace(a, 4, ui);
                const uint32_t tb =
                    tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(acc * C::ACC_COLS);
                constexpr int LDC = C::LDC;
#pragma unroll
                for (int j = 0; j < CW / LDC; ++j) {
                    const int c0 = cbase + LDC * j;
                    if (c0 < cu.n) {
                        uint32_t r[MW][LDC];
#pragma unroll
                        for (int w = 0; w < MW; ++w) tmem_ld_cols<LDC>(tb + w * NT + c0, r[w]);
                        tmem_ld_wait();
                        float gav[LDC], ubv[LDC];
#pragma unroll
                        for (int i = 0; i < LDC; ++i) {
                            float ga = 0.f, ub = 0.f;
#pragma unroll
                            for (int w = 0; w < MW; ++w) {
                                if (PAIR && (w & 1))
                                    ub += __uint_as_float(r[w][i]);
                                else
                                    ga += __uint_as_float(r[w][i]);
                            }
                            gav[i] = ga;
                            ubv[i] = ub;
                        }
                        if constexpr (G1) {
                            if (a.g_dbg) {  // debug capture of the chain sums
#pragma unroll
                                for (int i = 0; i < LDC; ++i)
                                    if (c0 + i < cu.n) {
                                        const size_t prow = static_cast<size_t>(cu.row0 + c0 + i);
                                        a.g_dbg[prow * 2 * a.I + feat] = gav[i];
                                        a.g_dbg[prow * 2 * a.I + a.I + feat] = ubv[i];
                                    }
                            }
#pragma unroll
                            for (int i = 0; i < LDC; ++i) v[LDC * j + i] = swiglu(gav[i], ubv[i], clamp, L);
                        } else {
#pragma unroll
                            for (int i = 0; i < LDC; ++i) {
                                v[LDC * j + i] = gav[i];
                                if constexpr (WIDE) v2[LDC * j + i] = ubv[i];  // the pair's second W2 tile
                            }
                        }
                    }
                }
                tc_fence_before();
                if (tracer) trace(a, 5, ui);
                mbar_arrive(&acce[acc]);
                if (C::NUM_ACC == 2) {
                    acc ^= 1;
                    if (acc == 0) acc_phase ^= 1u;
                } else {
                    acc_phase ^= 1u;
                }
            }
            if constexpr (WIDE && !C::ROT3) {  // two W2 tiles: rows of features m*256 + f and m*256 + 128 + f
                const int featw = cu.m * a.m_rows + 32 * q + lane;
                if (a.y8) {
#pragma unroll
                    for (int j = 0; j < CW; ++j) {
                        const int c = cbase + j;
                        if (c < cu.n) {
                            const size_t prow = static_cast<size_t>(cu.row0 + c);
                            uint8_t sc;
                            a.y8[prow * a.H + featw] = rows::quant_block_warp(v[j], &sc);
                            if (lane == 0) a.ys[prow * (a.H >> 5) + (featw >> 5)] = sc;
                            a.y8[prow * a.H + featw + 128] = rows::quant_block_warp(v2[j], &sc);
                            if (lane == 0) a.ys[prow * (a.H >> 5) + ((featw + 128) >> 5)] = sc;
                        }
                    }
                } else {
                    store_rows_bf16<CW>(a.y, v, cu.row0 + cbase, cu.n - cbase, a.H, featw);
                    store_rows_bf16<CW>(a.y, v2, cu.row0 + cbase, cu.n - cbase, a.H, featw + 128);
                }
                continue;
            }
            if (!G1 && a.y8) {  // MXFP8 GEMM2 rows: this warp's 32 features are one 1x32 block
#pragma unroll
                for (int j = 0; j < CW; ++j) {
                    const int c = cbase + j;
                    if (c < cu.n) {
                        const size_t prow = static_cast<size_t>(cu.row0 + c);
                        uint8_t sc;
                        a.y8[prow * a.H + feat] = rows::quant_block_warp(v[j], &sc);
                        if (lane == 0) a.ys[prow * (a.H >> 5) + (feat >> 5)] = sc;
                    }
                }
                continue;
            }
            if constexpr (G1) {
                // MXFP8 1x32 requantisation of h along I: this warp's 32 features of a row are one
                // block.  Eight rows at a time are quantised without branches, then stored.
                uint8_t* hs_tile = a.hs + (static_cast<size_t>(cu.g) * (a.I >> 7) + cu.m) * NB * 512 + q;
#pragma unroll
                for (int j0 = 0; j0 < CW; j0 += 8) {
                    const int c0 = cbase + j0;
                    if (c0 >= cu.n) break;  // warp-uniform: the rest of the columns are past the tile's rows
                    uint8_t q8[8];
                    int cd[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float h = v[j0 + i];
                        const uint32_t amax = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(h)));
                        int code = static_cast<int>(amax >> 23) - 8;
                        code = code < 0 ? 0 : code;
                        const float mul = __uint_as_float(static_cast<uint32_t>(254 - code) << 23);
                        q8[i] = __nv_cvt_float_to_fp8(h * mul, __NV_SATFINITE, __NV_E4M3);
                        cd[i] = code;
                    }
                    uint8_t* hrow = a.hq + static_cast<size_t>(cu.row0 + c0) * a.I + feat;
                    if (c0 + 8 <= cu.n) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) hrow[static_cast<size_t>(i) * a.I] = q8[i];
                        if (lane == 0) {
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const int c = c0 + i;
                                hs_tile[(c >> 7) * 512 + 16 * (c & 31) + 4 * ((c >> 5) & 3)] = static_cast<uint8_t>(cd[i]);
                            }
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int c = c0 + i;
                            if (c < cu.n) {
                                hrow[static_cast<size_t>(i) * a.I] = q8[i];
                                if (lane == 0)
                                    hs_tile[(c >> 7) * 512 + 16 * (c & 31) + 4 * ((c >> 5) & 3)] =
                                        static_cast<uint8_t>(cd[i]);
                            }
                        }
                    }
                }
            } else {
                store_rows_bf16<CW>(a.y, v, cu.row0 + cbase, cu.n - cbase, a.H, feat);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0) trace_cta(a, 1);
    if (warp == C::MMA_WARP0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <bool G1, int NT, int KC, bool WIDE>
cudaError_t set_attr() {
    return cudaFuncSetAttribute(k_gemm<G1, NT, KC, WIDE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg<G1, NT, KC, WIDE>::SMEM);
}

template <bool G1, int NT, int KC, bool WIDE>
cudaError_t launch(const GemmArgs& a, const CUtensorMap* tw, const CUtensorMap* tb, int grid, cudaStream_t s) {
    k_gemm<G1, NT, KC, WIDE><<<grid, Cfg<G1, NT, KC, WIDE>::THREADS, Cfg<G1, NT, KC, WIDE>::SMEM, s>>>(*tw, *tb, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t gemm_set_attributes() {
    cudaError_t e;
    if ((e = set_attr<true, 128, 1, false>()) != cudaSuccess) return e;
    if ((e = set_attr<true, 144, 1, false>()) != cudaSuccess) return e;
    if ((e = set_attr<false, 144, 1, false>()) != cudaSuccess) return e;
    if ((e = set_attr<false, 144, 1, true>()) != cudaSuccess) return e;
    if ((e = set_attr<true, 32, 1, false>()) != cudaSuccess) return e;
    if ((e = set_attr<false, 128, 1, false>()) != cudaSuccess) return e;
    if ((e = set_attr<false, 32, 1, false>()) != cudaSuccess) return e;
    if ((e = set_attr<false, 32, 1, true>()) != cudaSuccess) return e;
    if ((e = set_attr<false, 128, 1, true>()) != cudaSuccess) return e;
    return set_attr<false, 32, 2, false>();
}

cudaError_t launch_gemm1(const GemmArgs& a, const CUtensorMap* tm_w, const CUtensorMap* tm_x, int NT, int grid,
                         cudaStream_t s) {
    if (NT == 32) return launch<true, 32, 1, false>(a, tm_w, tm_x, grid, s);
    return NT == 128 ? launch<true, 128, 1, false>(a, tm_w, tm_x, grid, s)
                     : launch<true, 144, 1, false>(a, tm_w, tm_x, grid, s);
}

cudaError_t launch_gemm2(const GemmArgs& a, const CUtensorMap* tm_w, const CUtensorMap* tm_w_wide,
                         const CUtensorMap* tm_w_k2, const CUtensorMap* tm_h, const CUtensorMap* tm_h_k2, int NT,
                         int grid, cudaStream_t s) {
    // decode tiles: pairs of W2 tiles (a.m_rows == 256) when H allows it, else 256-wide K stages when I
    // allows it (halves the per-stage cost per byte), each operand's two K chunks in one box of its
    // two-chunk view
    if (NT == 32) {
        if (a.m_rows == 256) return launch<false, 32, 1, true>(a, tm_w_wide, tm_h, grid, s);
        return a.ktiles % 2 == 0 ? launch<false, 32, 2, false>(a, tm_w_k2, tm_h_k2, grid, s)
                                 : launch<false, 32, 1, false>(a, tm_w, tm_h, grid, s);
    }
    // prefill route tiles: pairs of W2 tiles (a.m_rows == 256) when H allows it
    if (NT == 128)
        return a.m_rows == 256 ? launch<false, 128, 1, true>(a, tm_w_wide, tm_h, grid, s)
                               : launch<false, 128, 1, false>(a, tm_w, tm_h, grid, s);
    return a.m_rows == 256 ? launch<false, 144, 1, true>(a, tm_w_wide, tm_h, grid, s)
                           : launch<false, 144, 1, false>(a, tm_w, tm_h, grid, s);
}

}  // namespace bmoe

// moe_internal.h -- workspace layout, kernel parameter blocks and launchers
// shared by the host code (moe_api.cu) and the kernels (moe_kernels.cu,
// moe_gemm.cu).  Not part of the public ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace bmoe {

constexpr int kChunk = 512;            // flat slots per compact-dispatch chunk
constexpr int kMaxTopk = 16;
constexpr int kMaxExperts = 4096;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per device-side wait
constexpr uint32_t kStBadId = 0x1u, kStTimeout = 0x2u, kStOverflow = 0x4u, kStBounds = 0x8u;
// Wait sites recorded next to kStTimeout (bit 8 + site): 0 producer/empty,
// 1 producer drain, 2 MMA/accumulator-free, 3 MMA/stage-full, 4 MMA drain,
// 5 epilogue/accumulator-full.
constexpr uint32_t kSiteShift = 8;
constexpr uint32_t kSiteGrid = 1u << (kSiteShift + 6);   // fused path: a grid barrier gave up
constexpr uint32_t kSiteReady = 1u << (kSiteShift + 7);  // fused path: a GEMM1->GEMM2 readiness wait gave up

// Device workspace, carved from one allocation.
struct Workspace {
    int32_t* counts;       // [E]   rows per expert (compact: routes, fixed: occupied slots)
    int32_t* rowbase;      // [E+1] first packed row of each expert
    int32_t* tile_base;    // [E+1] exclusive scan of route tiles per expert; [E] = total tiles
    int32_t* perm;         // [cap*K] compact packed row -> flat slot
    int32_t* route_row;    // [cap*K] compact flat slot -> packed row (-1 invalid)
    int32_t* route_slot;   // [cap*K] fixed flat slot -> e*MTPR+t (-1 invalid)
    int32_t* yrow;         // [cap*K] packed row of the GEMM2 output each slot combines (-1 invalid)
    uint32_t* occ;         // [E*words] fixed-slot occupancy bits
    int32_t* chunk_base;   // [nchunks*E] compact per-chunk counts, then per-chunk base rows
    uint32_t* ticket;      // [8] last-block counters (0, 1), fused grid-barrier count and generation (2, 3),
                           //     first bounds miss: site and index (5, 6; bounds-checking builds)
    uint32_t* status;      // [1] MOE_ST_* bits
    uint8_t* aq;           // [rows_cap][H] packed E4M3 codes of the dispatched rows
    uint8_t* as;           // [tiles_cap][H/128][512] scale atoms of aq, per route tile
    uint8_t* hq;           // [rows_cap][I] E4M3 codes of h
    uint8_t* hs;           // [tiles_cap][I/128][512] scale atoms of hq
    uint16_t* y;           // [rows_cap][H] bf16 GEMM2 outputs
    uint8_t* xq;           // [cap][H] canonical codes (debug capture only)
    uint8_t* xs;           // [cap][H/32] canonical scales (debug capture only)
    float* g;              // [rows_cap][2I] raw GEMM1 outputs (debug capture only)
    uint32_t* ready;       // [tiles_cap] fused path: GEMM1 units finished per route tile
    int32_t* rids;         // [cap*K] router top-k ids (moe_forward_routed)
    float* rw;             // [cap*K] router top-k weights (moe_forward_routed)
#ifdef MOE_DEBUG_BOUNDS
    // region sizes, checked by the bounds-checking build
    int lim_rows;          // packed rows of aq / hq / y
    int lim_tiles;         // route tiles of as / hs / ready
    int lim_slots;         // cap*K entries of perm / route_row / route_slot / yrow
    int lim_chunks;        // compact-dispatch chunks of chunk_base
#endif
};

// Bounds-checking build (-DMOE_DEBUG_BOUNDS, a second library next to the normal one): every index
// a kernel computes into a workspace region or an output row is checked before use.  A miss sets
// kStBounds, records the first miss (site, low 32 bits of the index) in ticket words 5 and 6, and
// the access is skipped, so nothing outside the regions is touched.  The checks, the limits they
// use and their arguments exist only in that build (BMOE_BOUNDS_ONLY): other builds compile the
// unchecked code, token for token.
enum BoundsSite : int {
    kBsOcc = 1,      // occupancy word of (expert, token)
    kBsSlot = 2,     // flat top-k slot of a per-slot array
    kBsPerm = 3,     // packed position of a route
    kBsChunk = 4,    // compact-dispatch chunk
    kBsRow = 5,      // packed row written by the quantise-and-scatter step
    kBsAtom = 6,     // route tile / row of a scale atom written by that step
    kBsYRow = 7,     // packed row read by the combine
    kBsUnit = 8,     // GEMM unit: route tile, first row, row count
};
#ifdef MOE_DEBUG_BOUNDS
#define BMOE_BOUNDS_ONLY(...) __VA_ARGS__
__device__ __forceinline__ bool bounds_ok(uint32_t* status, uint32_t* ticket, long long i, long long n, int site) {
    if (i >= 0 && i < n) return true;
    atomicOr(status, kStBounds);
    if (atomicCAS(ticket + 5, 0u, static_cast<uint32_t>(site)) == 0u) ticket[6] = static_cast<uint32_t>(i);
    return false;
}
#else
#define BMOE_BOUNDS_ONLY(...)
#endif

struct Geometry {
    int H, I, E, K, cap;
    int scheme;            // 1 fixed, 2 compact
    int mtpr;              // fixed-slot capacity per expert (= cap)
    int words;             // ceil(mtpr/32)
    int NT;                // route tile width (MMA N upper bound): 32 decode, 144 prefill (or 128)
    int nb;                // 128-row scale atoms per route tile and K chunk: (NT + 127) / 128
    long long rows_cap;    // packed rows
    long long tiles_cap;   // route tiles
    int nchunks_cap;
    bool debug;
};

size_t workspace_layout(const Geometry& g, char* base, Workspace* ws);  // base may be null (size only)

// ------------------------------------------------------------------ launchers (moe_kernels.cu)
cudaError_t launch_fixed_mark(const Geometry& g, const Workspace& ws, const int32_t* ids, int T,
                              const int32_t* nvr, cudaStream_t s);
cudaError_t launch_compact_dispatch(const Geometry& g, const Workspace& ws, const int32_t* ids, int T,
                                    const int32_t* nvr, cudaStream_t s);
// Shared-memory limit of the compact-dispatch count kernel for up to kMaxExperts experts; once per device
// before the first launch (moe_create, and the allocation-free dispatch's per-device set-up).
cudaError_t dispatch_set_attributes();
cudaError_t launch_quant_scatter(const Geometry& g, const Workspace& ws, const uint16_t* x, const int32_t* ids,
                                 int T, const int32_t* nvr, cudaStream_t s);
// y8/ys non-null: the GEMM2 rows are MXFP8 codes and scales instead of BF16 y.
cudaError_t launch_combine(const Geometry& g, const Workspace& ws, const float* wts, int T,
                           const int32_t* nvr, uint16_t* out, const uint8_t* y8, const uint8_t* ys, cudaStream_t s);

// ------------------------------------------------------------------ GEMMs (moe_gemm.cu)
struct GemmArgs {
    // routing plan
    const int32_t* counts;
    const int32_t* rowbase;
    const int32_t* tile_base;
    int E;
    // weights: codes through the tensor map, scales read directly
    const uint8_t* w_sf;   // natural [E*rows_per_expert][K/32]
    int w_rows;            // weight rows per expert (2I for GEMM1, H for GEMM2)
    int ld_sf;             // K/32
    int up_off;            // GEMM1: row offset of up row j from gate row j (I concatenated, 1 interleaved)
    int w_rs;              // row stride of consecutive output features (1, or 2 for interleaved W13)
    int m_rows;            // weight rows per unit and operand tile index step: 128, or 256 for paired W2 tiles
    uint8_t* y8;           // GEMM2 rows as MXFP8 codes [rows][H] (nullptr: BF16 rows in y)
    uint8_t* ys;           // ... and their E8M0 scales [rows][H/32]
    int ktiles;            // K/128
    int mtiles;            // weight tiles (of 128 rows, or row pairs for GEMM1) per expert
    // activations: codes through the tensor map, scale atoms
    const uint8_t* b_sf;   // [tiles][ktiles][512]
    // outputs
    uint8_t* hq;  uint8_t* hs;  int I;      // GEMM1
    float* g_dbg;                           // GEMM1 debug capture (may be null)
    uint16_t* y;  int H;                    // GEMM2
    float swiglu_limit;
    uint32_t* status;
#ifdef MOE_DEBUG_BOUNDS
    uint32_t* ticket;      // workspace ticket words (bounds-miss record)
    int lim_rows, lim_tiles;  // packed rows of hq / y, route tiles of b_sf / hs
#endif
    long long* trace;      // pipeline trace buffer (tracing builds only), else null
};

cudaError_t launch_gemm1(const GemmArgs& a, const CUtensorMap* tm_w, const CUtensorMap* tm_x, int NT, int grid,
                         cudaStream_t s);
// tm_w_wide: W2 with 256-row boxes, used when a.m_rows == 256 (128-row route tiles, H % 256 == 0)
// tm_w_k2 / tm_h_k2: two-chunk views (one box = two 128-wide K chunks) for 256-wide K stages
cudaError_t launch_gemm2(const GemmArgs& a, const CUtensorMap* tm_w, const CUtensorMap* tm_w_wide,
                         const CUtensorMap* tm_w_k2, const CUtensorMap* tm_h, const CUtensorMap* tm_h_k2, int NT,
                         int grid, cudaStream_t s);
cudaError_t gemm_set_attributes();

// ------------------------------------------------------------------ single-launch fused path (moe_fused.cu)
struct FusedLaunch {
    const uint16_t* x;
    const int32_t* ids;
    const float* wts;
    const int32_t* nvr;
    uint16_t* out;
    const uint8_t* w13s;
    const uint8_t* w2s;
    float swiglu_limit;
    int T;
    int w13_rs;  // W13 scale rows: gate row j of an expert at j * w13_rs, up row j at j * w13_rs + w13_up
    int w13_up;
    uint8_t* y8;  // GEMM2 rows as MXFP8 (nullptr: BF16)
    uint8_t* ys;
};
bool fused_supported(const Geometry& g);
// tm_w13p: the W13 gate/up pair view (K, feature, half, expert), box {128, 128, 2, 1}.
cudaError_t launch_fused(const Geometry& g, const Workspace& ws, const FusedLaunch& f, const CUtensorMap* tm_w13p,
                         const CUtensorMap* tm_aq, const CUtensorMap* tm_w2, const CUtensorMap* tm_hq, int grid,
                         cudaStream_t s);
// Router top-k softmax (moe_route.cu): one warp per row; bf16 != 0 reads BF16 logits.
cudaError_t launch_topk_softmax(const void* logits, int bf16, int T, int E, int K, const int32_t* nvr, int renorm,
                                int32_t* ids, float* w, cudaStream_t s);
cudaError_t fused_set_attributes();

// Error text of a failed call made without a handle (read by moe_last_error(NULL)).
void note_unbound_error(const char* msg);

}  // namespace bmoe

// moe_kernels.cu -- the bandwidth-bound steps of the layer: dispatch (fixed-slot
// and compact), MXFP8 quantisation of the input rows fused with the scatter
// into per-expert packed rows, and the top-k weighted combine.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "layer_rows.cuh"
#include "moe_internal.h"

namespace bmoe {

namespace {

constexpr unsigned kFull = 0xffffffffu;

using rows::read_nvr;

// Exclusive scan of in[0..n) into out[0..n], out[n] = total.  Whole block.
__device__ void block_exclusive_scan(const int* in, int* out, int n, int* warp_sums) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = (blockDim.x + 31) >> 5;
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int start = tid * per;
    int local = 0;
    for (int i = start; i < start + per && i < n; ++i) local += in[i];
    int x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int v = lane < nwarps ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(kFull, v, o);
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

// True in exactly one block: the last one to arrive at `ticket`.
__device__ bool last_block(uint32_t* ticket, bool* flag_smem) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned prev = atomicAdd(ticket, 1u);
        *flag_smem = (prev == gridDim.x - 1);
    }
    __syncthreads();
    if (*flag_smem) __threadfence();
    return *flag_smem;
}

struct DispatchArgs {
    const int32_t* ids;
    const int32_t* nvr;
    int T, K, E, mtpr, words, NT, nchunks;
    Workspace ws;
};

// ---------------------------------------------------------------- fixed-slot
// vLLM PR #61262 (the second, fixed-slot MegaMoEV2 runtime): a token goes
// directly to the slot (e, t) of its expert, capacity MTPR, with no prepare
// step.
// Occupancy bits are ORed atomically (order-independent, so deterministic);
// the last block turns them into per-expert row counts and the route-tile plan.
__global__ void __launch_bounds__(256) k_fixed_mark(DispatchArgs a) {
    extern __shared__ int sm[];
    __shared__ int warp_sums[32];
    __shared__ bool is_last;
    const int s = blockIdx.x * blockDim.x + threadIdx.x;
    const int nvr = read_nvr(a.nvr, a.T);
    if (s < a.T * a.K) {
        const int t = s / a.K, e = a.ids[s];
        if (t < nvr && e >= a.E) atomicOr(a.ws.status, kStBadId);
        BMOE_BOUNDS_ONLY(const Workspace& ws = a.ws; if (!bounds_ok(ws.status, ws.ticket, s, ws.lim_slots, kBsSlot)) {
        } else)
        if (t < nvr && e >= 0 && e < a.E BMOE_BOUNDS_ONLY(&& bounds_ok(ws.status, ws.ticket, t, a.mtpr, kBsOcc))) {
            atomicOr(&a.ws.occ[(size_t)e * a.words + (t >> 5)], 1u << (t & 31));
            a.ws.route_slot[s] = e * a.mtpr + t;
        } else {
            a.ws.route_slot[s] = -1;
        }
    }
    if (!last_block(&a.ws.ticket[0], &is_last)) return;
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
        int c = 0;
        for (int w = 0; w < a.words; ++w) c += __popc(__ldcg(&a.ws.occ[(size_t)e * a.words + w]));
        a.ws.counts[e] = c;
        a.ws.rowbase[e] = e * a.mtpr;
        sm[e] = (c + a.NT - 1) / a.NT;
    }
    if (threadIdx.x == 0) a.ws.rowbase[a.E] = a.E * a.mtpr;
    __syncthreads();
    block_exclusive_scan(sm, sm + a.E, a.E, warp_sums);
    for (int e = threadIdx.x; e <= a.E; e += blockDim.x) a.ws.tile_base[e] = sm[a.E + e];
    if (threadIdx.x == 0) a.ws.ticket[0] = 0;
}

// ---------------------------------------------------------------- compact
// vLLM PR #61262: compact dispatch packs tokens before dispatch.  Canonical
// order: experts ascending, flat slot id t*K+k ascending inside an expert.
// Pass 1: per-chunk expert histograms; the last block scans them into
// per-expert offsets, per-(chunk, expert) base rows and the route-tile plan.
__global__ void __launch_bounds__(512) k_compact_count(DispatchArgs a) {
    extern __shared__ int sm[];  // cnt[E], offs[E+1], ntile[E], tbase[E+1]
    __shared__ int warp_sums[32];
    __shared__ bool is_last;
    int* cnt = sm;
    const int E = a.E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    const int nvr = read_nvr(a.nvr, a.T);
    const int s = blockIdx.x * kChunk + threadIdx.x;
    if (threadIdx.x < kChunk && s < a.T * a.K) {
        const int t = s / a.K, e = a.ids[s];
        if (t < nvr && e >= E) atomicOr(a.ws.status, kStBadId);
        if (t < nvr && e >= 0 && e < E) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    BMOE_BOUNDS_ONLY(if (!bounds_ok(a.ws.status, a.ws.ticket, a.nchunks, a.ws.lim_chunks + 1, kBsChunk)) return;)
    for (int e = threadIdx.x; e < E; e += blockDim.x) a.ws.chunk_base[(size_t)blockIdx.x * E + e] = cnt[e];
    if (!last_block(&a.ws.ticket[1], &is_last)) return;
    int* offs = sm + E;
    int* ntile = offs + E + 1;
    int* tbase = ntile + E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
        for (int c = 0; c < a.nchunks; ++c) {
            int v = __ldcg(&a.ws.chunk_base[(size_t)c * E + e]);
            a.ws.chunk_base[(size_t)c * E + e] = run;
            run += v;
        }
        cnt[e] = run;
        a.ws.counts[e] = run;
        ntile[e] = (run + a.NT - 1) / a.NT;
    }
    __syncthreads();
    block_exclusive_scan(cnt, offs, E, warp_sums);
    block_exclusive_scan(ntile, tbase, E, warp_sums);
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
        a.ws.rowbase[e] = offs[e];
        a.ws.tile_base[e] = tbase[e];
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        for (int c = 0; c < a.nchunks; ++c) a.ws.chunk_base[(size_t)c * E + e] += offs[e];
    if (threadIdx.x == 0) a.ws.ticket[1] = 0;
}

// Pass 2: stable ranks inside each chunk (one warp walks the chunk in order;
// equal experts inside 32 slots are ranked by lane), giving route_row and perm.
__global__ void __launch_bounds__(32) k_compact_rank(DispatchArgs a) {
    extern __shared__ int run[];  // [E]
    const int lane = threadIdx.x;
    const int E = a.E;
    BMOE_BOUNDS_ONLY(const Workspace& ws = a.ws;
                     if (!bounds_ok(ws.status, ws.ticket, a.nchunks, ws.lim_chunks + 1, kBsChunk)) return;)
    for (int e = lane; e < E; e += 32) run[e] = a.ws.chunk_base[(size_t)blockIdx.x * E + e];
    __syncwarp();
    const int nvr = read_nvr(a.nvr, a.T);
    const unsigned lt = (1u << lane) - 1u;
    for (int it = 0; it < kChunk / 32; ++it) {
        const int s = blockIdx.x * kChunk + it * 32 + lane;
        const bool in = s < a.T * a.K;
        const int e = in ? a.ids[s] : -1;
        const bool valid = in && (s / a.K) < nvr && e >= 0 && e < E;
        const int key = valid ? e : (0x40000000 | lane);
        const unsigned peers = __match_any_sync(kFull, key);
        if (valid) {
            const int p = run[e] + __popc(peers & lt);
            BMOE_BOUNDS_ONLY(if (bounds_ok(ws.status, ws.ticket, s, ws.lim_slots, kBsSlot)))
            a.ws.route_row[s] = p;
            BMOE_BOUNDS_ONLY(if (bounds_ok(ws.status, ws.ticket, p, ws.lim_slots, kBsPerm)))
            a.ws.perm[p] = s;
        } else if (in BMOE_BOUNDS_ONLY(&& bounds_ok(ws.status, ws.ticket, s, ws.lim_slots, kBsSlot))) {
            a.ws.route_row[s] = -1;
        }
        __syncwarp();
        if (valid && lane == __ffs(peers) - 1) run[e] += __popc(peers);
        __syncwarp();
    }
}

// ---------------------------------------------------------------- quant + scatter
// One warp per token row (rows::quant_scatter_row).
__global__ void __launch_bounds__(256) k_quant_scatter(rows::QuantArgs a, const int32_t* nvr_ptr) {
    const int lane = threadIdx.x & 31;
    const int item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (item >= rows::quant_items(a)) return;
    rows::quant_scatter_seg(a, a.ws.rowbase, a.ws.tile_base, item, rows::read_nvr(nvr_ptr, a.T), lane);
}

// ---------------------------------------------------------------- combine
// One warp per output row (rows::combine_row).
// Two instances so that the BF16 one keeps its small register footprint (occupancy: the combine
// is bound by memory latency).
template <bool FP8>
__global__ void __launch_bounds__(256) k_combine(rows::CombineArgs a) {
    const int item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (item >= rows::combine_items(a)) return;
    if constexpr (FP8)
        rows::combine_item_fp8(a, item, threadIdx.x & 31);
    else
        rows::combine_item_bf16(a, item, threadIdx.x & 31);
}

DispatchArgs dispatch_args(const Geometry& g, const Workspace& ws, const int32_t* ids, int T, const int32_t* nvr) {
    DispatchArgs a;
    a.ids = ids;
    a.nvr = nvr;
    a.T = T;
    a.K = g.K;
    a.E = g.E;
    a.mtpr = g.mtpr;
    a.words = g.words;
    a.NT = g.NT;
    a.nchunks = (T * g.K + kChunk - 1) / kChunk;
    a.ws = ws;
    return a;
}

}  // namespace

size_t workspace_layout(const Geometry& g, char* base, Workspace* ws) {
    size_t off = 0;
    auto carve = [&](size_t bytes) -> char* {
        off = (off + 255) & ~size_t(255);
        char* p = base ? base + off : nullptr;
        off += bytes;
        return p;
    };
    const size_t slots = (size_t)g.cap * g.K;
    Workspace w{};
    w.counts = reinterpret_cast<int32_t*>(carve(sizeof(int32_t) * g.E));
    w.rowbase = reinterpret_cast<int32_t*>(carve(sizeof(int32_t) * (g.E + 1)));
    w.tile_base = reinterpret_cast<int32_t*>(carve(sizeof(int32_t) * (g.E + 1)));
    w.perm = reinterpret_cast<int32_t*>(carve(sizeof(int32_t) * slots));
    w.route_row = reinterpret_cast<int32_t*>(carve(sizeof(int32_t) * slots));
    w.route_slot = reinterpret_cast<int32_t*>(carve(sizeof(int32_t) * slots));
    w.yrow = reinterpret_cast<int32_t*>(carve(sizeof(int32_t) * slots));
    w.occ = reinterpret_cast<uint32_t*>(carve(sizeof(uint32_t) * (size_t)g.E * g.words));
    w.chunk_base = reinterpret_cast<int32_t*>(carve(sizeof(int32_t) * (size_t)g.nchunks_cap * g.E));
    w.ticket = reinterpret_cast<uint32_t*>(carve(sizeof(uint32_t) * 8));
    w.status = reinterpret_cast<uint32_t*>(carve(sizeof(uint32_t) * 4));
    w.aq = reinterpret_cast<uint8_t*>(carve((size_t)g.rows_cap * g.H));
    w.as = reinterpret_cast<uint8_t*>(carve((size_t)g.tiles_cap * (g.H / 128) * g.nb * 512));
    w.hq = reinterpret_cast<uint8_t*>(carve((size_t)g.rows_cap * g.I));
    w.hs = reinterpret_cast<uint8_t*>(carve((size_t)g.tiles_cap * (g.I / 128) * g.nb * 512));
    w.y = reinterpret_cast<uint16_t*>(carve((size_t)g.rows_cap * g.H * 2));
    w.ready = reinterpret_cast<uint32_t*>(carve(sizeof(uint32_t) * (size_t)g.tiles_cap));
    w.rids = reinterpret_cast<int32_t*>(carve(sizeof(int32_t) * slots));
    w.rw = reinterpret_cast<float*>(carve(sizeof(float) * slots));
    if (g.debug) {
        w.xq = reinterpret_cast<uint8_t*>(carve((size_t)g.cap * g.H));
        w.xs = reinterpret_cast<uint8_t*>(carve((size_t)g.cap * (g.H / 32)));
        w.g = reinterpret_cast<float*>(carve((size_t)g.rows_cap * 2 * g.I * sizeof(float)));
    }
#ifdef MOE_DEBUG_BOUNDS
    w.lim_rows = static_cast<int>(g.rows_cap);
    w.lim_tiles = static_cast<int>(g.tiles_cap);
    w.lim_slots = static_cast<int>(slots);
    w.lim_chunks = g.nchunks_cap;
#endif
    off = (off + 255) & ~size_t(255);
    if (ws) *ws = w;
    return off;
}

cudaError_t launch_fixed_mark(const Geometry& g, const Workspace& ws, const int32_t* ids, int T,
                              const int32_t* nvr, cudaStream_t s) {
    DispatchArgs a = dispatch_args(g, ws, ids, T, nvr);
    const int blocks = (T * g.K + 255) / 256;
    k_fixed_mark<<<blocks, 256, sizeof(int) * (2 * g.E + 1), s>>>(a);
    return cudaGetLastError();
}

cudaError_t dispatch_set_attributes() {
    // k_compact_count keeps 4E+2 int32 in dynamic shared memory: above the default 48 KB for E >= 3072
    return cudaFuncSetAttribute(k_compact_count, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(sizeof(int) * (4 * kMaxExperts + 2)));
}

cudaError_t launch_compact_dispatch(const Geometry& g, const Workspace& ws, const int32_t* ids, int T,
                                    const int32_t* nvr, cudaStream_t s) {
    DispatchArgs a = dispatch_args(g, ws, ids, T, nvr);
    k_compact_count<<<a.nchunks, kChunk, sizeof(int) * (4 * g.E + 2), s>>>(a);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    k_compact_rank<<<a.nchunks, 32, sizeof(int) * g.E, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_quant_scatter(const Geometry& g, const Workspace& ws, const uint16_t* x, const int32_t* ids,
                                 int T, const int32_t* nvr, cudaStream_t s) {
    rows::QuantArgs a;
    a.x = x;
    a.ids = ids;
    a.T = T;
    a.K = g.K;
    a.E = g.E;
    a.H = g.H;
    a.mtpr = g.mtpr;
    a.words = g.words;
    a.NT = g.NT;
    a.nb = g.nb;
    a.scheme = g.scheme;
    a.ws = ws;
    const int items = T * ((g.H / 32 + rows::kQuantBlocks - 1) / rows::kQuantBlocks);
    k_quant_scatter<<<(items + 7) / 8, 256, 0, s>>>(a, nvr);
    return cudaGetLastError();
}

cudaError_t launch_combine(const Geometry& g, const Workspace& ws, const float* wts, int T,
                           const int32_t* /*nvr*/, uint16_t* out, const uint8_t* y8, const uint8_t* ys, cudaStream_t s) {
    rows::CombineArgs a;
    a.y = ws.y;
    a.yrow = ws.yrow;
    a.w = wts;
    a.out = out;
    a.T = T;
    a.K = g.K;
    a.H = g.H;
    a.y8 = y8;
    a.ys = ys;
    BMOE_BOUNDS_ONLY(a.status = ws.status; a.ticket = ws.ticket; a.lim_rows = ws.lim_rows; a.lim_slots = ws.lim_slots;)
    const int items = T * ((g.H / 8 + rows::kCombineVecs - 1) / rows::kCombineVecs);
    if (y8)
        k_combine<true><<<(items + 7) / 8, 256, 0, s>>>(a);
    else
        k_combine<false><<<(items + 7) / 8, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace bmoe

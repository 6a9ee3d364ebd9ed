// layer_rows.cuh -- per-row device code shared by the stand-alone kernels
// (moe_kernels.cu) and the single-launch fused kernel (moe_fused.cu): MXFP8
// quantisation of one token row fused with its scatter into the experts' packed
// rows, and the top-k weighted combine of one output row.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "moe_internal.h"

namespace bmoe {
namespace rows {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ int read_nvr(const int32_t* p, int T) {
    int v = p ? __ldg(p) : T;
    return v < 0 ? 0 : (v > T ? T : v);
}

__device__ __forceinline__ uint32_t pack_fp8x4(float a, float b, float c, float d) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

struct QuantArgs {
    const uint16_t* x;
    const int32_t* ids;
    int T, K, E, H, mtpr, words, NT, scheme;
    int nb;  // 128-row scale atoms per route tile and K chunk
    Workspace ws;
};

// One warp quantises segment `seg` (kQuantBlocks 32-element blocks, one per
// lane) of token row t to MXFP8 (E4M3 codes, one E8M0 scale per 32 along H, OCP
// MX rule: code = max(exponent(amax) - 8, 0), element = RNE_satfinite(x *
// 2^(127-code))) and writes the codes once per valid slot into the expert's
// packed rows, the scale into the route tile's 128x4 scale atom (byte
// 16*(c%32) + 4*(c/32) + kblock%4 for row c of the tile); segment 0 also
// records the packed row each slot combines (yrow, -1 for an invalid slot).
// `rowbase` / `tile_base` may point to global or shared memory.  Routing data
// written earlier by other CTAs is read with L2-coherent loads.
constexpr int kQuantBlocks = 32;

__device__ __forceinline__ int quant_items(const QuantArgs& a) {
    return a.T * ((a.H / 32 + kQuantBlocks - 1) / kQuantBlocks);
}

__device__ __forceinline__ void quant_scatter_seg(const QuantArgs& a, const int32_t* rowbase,
                                                  const int32_t* tile_base, int item, int nvr, int lane) {
    const int segs = (a.H / 32 + kQuantBlocks - 1) / kQuantBlocks;
    const int t = item / segs, seg = item - t * segs;
    const int K = a.K;
    int p = -1, gt = 0, c = 0;
    bool valid = false;
    BMOE_BOUNDS_ONLY(const Workspace& ws = a.ws;)
    if (lane < K) {
        const int e = a.ids[(size_t)t * K + lane];
        if (t < nvr && e >= a.E) atomicOr(a.ws.status, kStBadId);
        valid = t < nvr && e >= 0 && e < a.E;
        BMOE_BOUNDS_ONLY(
            const bool slot_ok = bounds_ok(ws.status, ws.ticket, (long long)t * K + lane, ws.lim_slots, kBsSlot);
            if (valid && !(a.scheme == 1 ? bounds_ok(ws.status, ws.ticket, t, a.mtpr, kBsOcc) : slot_ok)) valid = false;)
        if (valid) {
            int i;
            if (a.scheme == 1) {
                const uint32_t* wb = a.ws.occ + (size_t)e * a.words;
                i = 0;
                for (int w = 0; w < (t >> 5); ++w) i += __popc(__ldcg(wb + w));
                i += __popc(__ldcg(wb + (t >> 5)) & ((1u << (t & 31)) - 1u));
                p = e * a.mtpr + i;
            } else {
                p = __ldcg(a.ws.route_row + (size_t)t * K + lane);
                i = p - rowbase[e];
            }
            gt = tile_base[e] + i / a.NT;
            c = i % a.NT;
        }
        if (seg == 0 BMOE_BOUNDS_ONLY(&& slot_ok)) a.ws.yrow[(size_t)t * K + lane] = valid ? p : -1;
    }
    if (t >= nvr) return;  // warp-uniform
    const unsigned vmask = __ballot_sync(kFull, valid);
    const int H = a.H, nblk = H >> 5, ktiles = H >> 7;
    static_assert(kQuantBlocks == 32, "one 32-element block per lane");
    // Quantise this lane's block once, then store it for each valid slot in turn; the slots'
    // destinations are broadcast from lane k one slot at a time (no per-slot register arrays, so
    // the stand-alone kernel keeps enough warps resident to cover the loads' latency).
    const int blk = seg * kQuantBlocks + lane;
    const bool has = blk < nblk;
    uint4 o0 = make_uint4(0u, 0u, 0u, 0u), o1 = o0;
    int code = 0;
    if (has) {
        const uint4* src = reinterpret_cast<const uint4*>(a.x + (size_t)t * H + blk * 32);
        float f[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 v = __ldg(src + q);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                f[q * 8 + 2 * j] = __uint_as_float(w[j] << 16);
                f[q * 8 + 2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
            }
        }
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(f[j]));
        code = static_cast<int>(__float_as_uint(amax) >> 23) - 8;
        code = code < 0 ? 0 : code;
        const float mul = __uint_as_float(static_cast<uint32_t>(254 - code) << 23);
        uint32_t o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            o[j] = pack_fp8x4(f[4 * j] * mul, f[4 * j + 1] * mul, f[4 * j + 2] * mul, f[4 * j + 3] * mul);
        o0 = make_uint4(o[0], o[1], o[2], o[3]);
        o1 = make_uint4(o[4], o[5], o[6], o[7]);
        if (a.ws.xq) {
            uint4* d = reinterpret_cast<uint4*>(a.ws.xq + (size_t)t * H + blk * 32);
            d[0] = o0;
            d[1] = o1;
            a.ws.xs[(size_t)t * nblk + blk] = static_cast<uint8_t>(code);
        }
    }
#pragma unroll 1
    for (int k = 0; k < K; ++k) {
        if (!((vmask >> k) & 1u)) continue;  // warp-uniform
        const int pk = __shfl_sync(kFull, p, k), gk = __shfl_sync(kFull, gt, k), ci = __shfl_sync(kFull, c, k);
        if (has BMOE_BOUNDS_ONLY(&& bounds_ok(ws.status, ws.ticket, pk, ws.lim_rows, kBsRow) &&
                                 bounds_ok(ws.status, ws.ticket, gk, ws.lim_tiles, kBsAtom) &&
                                 bounds_ok(ws.status, ws.ticket, ci, a.nb * 128, kBsAtom))) {
            uint4* d = reinterpret_cast<uint4*>(a.ws.aq + (size_t)pk * H + blk * 32);
            d[0] = o0;
            d[1] = o1;
            a.ws.as[(((size_t)gk * ktiles + (blk >> 2)) * a.nb + (ci >> 7)) * 512 + 16 * (ci & 31) +
                    4 * ((ci >> 5) & 3) + (blk & 3)] = static_cast<uint8_t>(code);
        }
    }
}

// out[t] = BF16( sum over valid slots, k ascending, of w[t,k] * y[row(t,k)] ),
// float accumulation rounded once (ROCm/ATOM PR #2725: the routed terms are
// added in single precision and rounded one time); -1 slots are skipped (ROCm/aiter PR #6881, Technical
// Details: both paths leave out top-k slots marked -1); rows with no valid slot
// are +0.  Work item = one segment of kCombineVecs 16-byte vectors of one row,
// one warp per item; y is read with L2-coherent loads (the fused kernel
// combines rows other CTAs wrote in the same launch).
constexpr int kCombineVecs = 64;  // 512 BF16 elements per work item
struct CombineArgs {
    const uint16_t* y;
    const int32_t* yrow;
    const float* w;
    uint16_t* out;
    int T, K, H;
    const uint8_t* y8;  // non-null: GEMM2 rows are MXFP8 codes [rows][H] ...
    const uint8_t* ys;  // ... with E8M0 scales [rows][H/32]
#ifdef MOE_DEBUG_BOUNDS
    uint32_t* status;   // workspace status and ticket words (bounds-miss record)
    uint32_t* ticket;
    int lim_rows, lim_slots;  // packed rows of y, entries of yrow
#endif
};

#ifdef MOE_DEBUG_BOUNDS
// The packed row slot k of token t combines (-1: none), where a row outside y or a slot outside yrow
// counts as none.
__device__ __forceinline__ int combine_row(const CombineArgs& a, int t, int k) {
    if (!bounds_ok(a.status, a.ticket, (long long)t * a.K + k, a.lim_slots, kBsSlot)) return -1;
    const int r = __ldcg(a.yrow + (size_t)t * a.K + k);
    return (r < 0 || bounds_ok(a.status, a.ticket, r, a.lim_rows, kBsYRow)) ? r : -1;
}
#define BMOE_COMBINE_ROW(a, t, k) combine_row(a, t, k)
#else
#define BMOE_COMBINE_ROW(a, t, k) __ldcg(a.yrow + (size_t)t * a.K + k)
#endif

// One MXFP8 1x32 block held by a warp, one element per lane (OCP MX rule as for
// the input rows): returns the lane's E4M3 code; *scale receives the E8M0 code.
__device__ __forceinline__ uint8_t quant_block_warp(float v, uint8_t* scale) {
    const uint32_t amax = __reduce_max_sync(kFull, __float_as_uint(fabsf(v)));
    int code = static_cast<int>(amax >> 23) - 8;
    code = code < 0 ? 0 : code;
    *scale = static_cast<uint8_t>(code);
    const float mul = __uint_as_float(static_cast<uint32_t>(254 - code) << 23);
    return __nv_cvt_float_to_fp8(v * mul, __NV_SATFINITE, __NV_E4M3);
}

// 2^(code - 127) for an E8M0 code in [0, 254] (code 0 is the subnormal 2^-127).
__device__ __forceinline__ float e8m0_value(uint32_t code) {
    return code ? __uint_as_float(code << 23) : __uint_as_float(1u << 22);
}

__device__ __forceinline__ int combine_items(const CombineArgs& a) {
    return a.T * ((a.H / 8 + kCombineVecs - 1) / kCombineVecs);
}

__device__ __forceinline__ void combine_item_bf16(const CombineArgs& a, int item, int lane) {
    const int segs = (a.H / 8 + kCombineVecs - 1) / kCombineVecs;
    const int t = item / segs, seg = item - t * segs;
    int r_l = -1;
    float w_l = 0.f;
    if (lane < a.K) {
        r_l = BMOE_COMBINE_ROW(a, t, lane);
        w_l = a.w[(size_t)t * a.K + lane];
    }
    int rows[kMaxTopk];
    float wk[kMaxTopk];
#pragma unroll
    for (int k = 0; k < kMaxTopk; ++k) {
        rows[k] = __shfl_sync(kFull, r_l, k);
        wk[k] = __shfl_sync(kFull, w_l, k);
    }
    const int v1 = min(a.H >> 3, (seg + 1) * kCombineVecs);
    for (int v = seg * kCombineVecs + lane; v < v1; v += 32) {
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.f;
        bool any = false;
#pragma unroll
        for (int k = 0; k < kMaxTopk; ++k) {
            if (k >= a.K || rows[k] < 0) continue;
            any = true;
            const uint4 q = __ldcg(reinterpret_cast<const uint4*>(a.y + (size_t)rows[k] * a.H) + v);
            const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
            const float wv = wk[k];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc[2 * j] = __fadd_rn(acc[2 * j], __fmul_rn(wv, __uint_as_float(w4[j] << 16)));
                acc[2 * j + 1] = __fadd_rn(acc[2 * j + 1], __fmul_rn(wv, __uint_as_float(w4[j] & 0xffff0000u)));
            }
        }
        uint4 o = make_uint4(0, 0, 0, 0);
        if (any) {
            uint32_t ow[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
                ow[j] = *reinterpret_cast<const uint32_t*>(&b);
            }
            o = make_uint4(ow[0], ow[1], ow[2], ow[3]);
        }
        reinterpret_cast<uint4*>(a.out + (size_t)t * a.H)[v] = o;
    }
}

// MXFP8 GEMM2 rows: slots taken one at a time (row and weight shuffled from lane k), so that the
// dequantisation's registers do not add to a per-slot table.
__device__ __forceinline__ void combine_item_fp8(const CombineArgs& a, int item, int lane) {
    constexpr int kPer = kCombineVecs / 32;  // vectors per lane in one item
    const int segs = (a.H / 8 + kCombineVecs - 1) / kCombineVecs;
    const int t = item / segs, seg = item - t * segs;
    int r_l = -1;
    float w_l = 0.f;
    if (lane < a.K) {
        r_l = BMOE_COMBINE_ROW(a, t, lane);
        w_l = a.w[(size_t)t * a.K + lane];
    }
    const int v1 = min(a.H >> 3, (seg + 1) * kCombineVecs);
    float acc[kPer][8];
#pragma unroll
    for (int it = 0; it < kPer; ++it)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[it][j] = 0.f;
    bool any = false;
    for (int k = 0; k < a.K; ++k) {  // slots in ascending k: each element's sum keeps that order
        const int rk = __shfl_sync(kFull, r_l, k);
        const float wv = __shfl_sync(kFull, w_l, k);
        if (rk < 0) continue;
        any = true;
#pragma unroll
        for (int it = 0; it < kPer; ++it) {
            const int v = seg * kCombineVecs + lane + 32 * it;
            if (v >= v1) continue;
            float yv[8];
            {  // MXFP8 row: 8 codes and the scale of their 32-block (exact dequantisation)
                const uint2 q = __ldcg(reinterpret_cast<const uint2*>(a.y8 + (size_t)rk * a.H) + v);
                const float sc = e8m0_value(__ldcg(a.ys + (size_t)rk * (a.H >> 5) + (v >> 2)));
                const uint32_t w2[2] = {q.x, q.y};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(
                        static_cast<__nv_fp8x2_storage_t>((w2[j >> 1] >> (16 * (j & 1))) & 0xffffu), __NV_E4M3);
                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
                    yv[2 * j] = f.x * sc;
                    yv[2 * j + 1] = f.y * sc;
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[it][j] = __fadd_rn(acc[it][j], __fmul_rn(wv, yv[j]));
        }
    }
#pragma unroll
    for (int it = 0; it < kPer; ++it) {
        const int v = seg * kCombineVecs + lane + 32 * it;
        if (v >= v1) continue;
        uint4 o = make_uint4(0, 0, 0, 0);
        if (any) {
            uint32_t ow[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __nv_bfloat162 b = __floats2bfloat162_rn(acc[it][2 * j], acc[it][2 * j + 1]);
                ow[j] = *reinterpret_cast<const uint32_t*>(&b);
            }
            o = make_uint4(ow[0], ow[1], ow[2], ow[3]);
        }
        reinterpret_cast<uint4*>(a.out + (size_t)t * a.H)[v] = o;
    }
}

// Work item -> the combine of one row segment, from BF16 or MXFP8 GEMM2 rows.
__device__ __forceinline__ void combine_item(const CombineArgs& a, int item, int lane) {
    if (a.y8)
        combine_item_fp8(a, item, lane);
    else
        combine_item_bf16(a, item, lane);
}

}  // namespace rows
}  // namespace bmoe

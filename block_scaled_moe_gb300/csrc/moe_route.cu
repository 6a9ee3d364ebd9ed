// moe_route.cu -- router top-k with softmax weights, the step in front of
// dispatch (ROCm/ATOM PR #2725, linked commits on the Triton softmax top-k
// routing driven by the number of valid rows held on the device): every row
// from that number on gets ids -1 and weight 0; each pick takes the largest remaining logit, ties to the
// lowest expert id, and clears it to -inf, so a row that runs out of finite
// logits picks expert 0 again with weight 0; weights are exp(l - max) over the
// picked experts' sum (renormalised) or over the whole row's.
//
// One warp per row.  The picks compare the logits themselves (exact), so the
// ids do not depend on rounding; a lane keeps the picked flags of its experts
// (e = lane + 32 j) in a register bitmask.
#include <cuda_bf16.h>

#include "layer_rows.cuh"
#include "moe_internal.h"

namespace bmoe {
namespace {

constexpr int kRouteWords = kMaxExperts / 32 / 32;  // bitmask words per lane (E <= 4096)

template <bool BF16>
__device__ __forceinline__ float logit(const void* p, size_t i) {
    if constexpr (BF16)
        return __uint_as_float(static_cast<uint32_t>(__ldg(static_cast<const uint16_t*>(p) + i)) << 16);
    else
        return __ldg(static_cast<const float*>(p) + i);
}

template <bool BF16>
__global__ void __launch_bounds__(256) k_topk_softmax(const void* logits, int T, int E, int K, const int32_t* nvr_ptr,
                                                      int renorm, int32_t* ids, float* w) {
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (t >= T) return;
    const int nvr = rows::read_nvr(nvr_ptr, T);
    if (t >= nvr) {
        if (lane < K) {
            ids[(size_t)t * K + lane] = -1;
            w[(size_t)t * K + lane] = 0.f;
        }
        return;
    }
    const size_t base = (size_t)t * E;
    float m = -INFINITY;
    for (int e = lane; e < E; e += 32) m = fmaxf(m, logit<BF16>(logits, base + e));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    uint32_t picked[kRouteWords];
#pragma unroll
    for (int i = 0; i < kRouteWords; ++i) picked[i] = 0u;
    float mynum = 0.f;  // lane k keeps the numerator of pick k
    int myid = 0;
    for (int k = 0; k < K; ++k) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int j = 0, e = lane; e < E; ++j, e += 32) {
            const bool done = (picked[j >> 5] >> (j & 31)) & 1u;
            const float v = done ? -INFINITY : logit<BF16>(logits, base + e);
            if (v > bv || (v == bv && e < bi)) {
                bv = v;
                bi = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane) {
            const int j = bi >> 5;
            picked[j >> 5] |= 1u << (j & 31);
        }
        if (lane == k) {
            myid = bi;
            mynum = bv == -INFINITY ? 0.f : expf(bv - m);
        }
    }
    float den;
    if (renorm) {
        den = lane < K ? mynum : 0.f;
    } else {
        den = 0.f;
        for (int e = lane; e < E; e += 32) den += expf(logit<BF16>(logits, base + e) - m);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    if (lane < K) {
        ids[(size_t)t * K + lane] = myid;
        w[(size_t)t * K + lane] = mynum / den;
    }
}

}  // namespace

cudaError_t launch_topk_softmax(const void* logits, int bf16, int T, int E, int K, const int32_t* nvr, int renorm,
                                int32_t* ids, float* w, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int blocks = (T + 7) / 8;
    if (bf16)
        k_topk_softmax<true><<<blocks, 256, 0, s>>>(logits, T, E, K, nvr, renorm, ids, w);
    else
        k_topk_softmax<false><<<blocks, 256, 0, s>>>(logits, T, E, K, nvr, renorm, ids, w);
    return cudaGetLastError();
}

}  // namespace bmoe

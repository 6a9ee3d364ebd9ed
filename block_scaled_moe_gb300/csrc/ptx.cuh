// ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarrier, TMA (cp.async.bulk),
// tcgen05 (TMEM alloc, smem->TMEM copy, block-scaled MMA, TMEM loads) and the
// shared-memory / instruction descriptors the tensor core reads.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace bmoe {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the phase with parity `parity`.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on the phase with parity `parity`.  Gives up after `limit_ns`
// or as soon as another role of the CTA has given up (*abort != 0); on
// give-up it raises *abort, ORs `flag` into the device status word and
// returns false.  Never traps.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint32_t* status, uint32_t flag, uint64_t limit_ns) {
    if (mbar_test(bar, parity)) return true;
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            *abort = 1;
            atomicOr(status, flag);
            return false;
        }
    }
}


// ------------------------------------------------------------------ fences
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_all() {
    asm volatile("fence.proxy.async;" ::: "memory");
}

// ------------------------------------------------------------------ GPU-scope acquire / release
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_add_release_u32(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.release.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// ------------------------------------------------------------------ L2 policies
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ------------------------------------------------------------------ TMA
// Tiled TMA loads (2D / 3D / 4D box into shared memory, completing on `bar`), the contiguous bulk
// copy (16-byte aligned, size a multiple of 16) and the producer's arrival with its transaction
// bytes, in warp-level form: executed by a whole converged warp, one lane (elected with elect.sync
// over the full mask) issues.  A single thread issuing from a divergent branch
// spends ~440 cycles per box plus barrier operation on GB300; the converged form ~330, and a second
// issuing warp doubles the rate, so the producers issue this way.
#define BMOE_ELECT_ISSUE(body) \
    "{\n\t.reg .pred p;\n\t.reg .b32 e;\n\telect.sync e|p, 0xffffffff;\n\t@p " body ";\n\t}"
__device__ __forceinline__ void mbar_arrive_expect_tx_w(uint64_t* bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b32 e;\n\t.reg .b64 st;\n\telect.sync e|p, 0xffffffff;\n\t"
        "@p mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
        "r"(bytes)
        : "memory");
}
__device__ __forceinline__ void tma_load_2d_w(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                              uint64_t policy) {
    asm volatile(BMOE_ELECT_ISSUE(
                     "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
                     " [%0], [%1, {%3, %4}], [%2], %5") ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(policy)
                 : "memory");
}
__device__ __forceinline__ void tma_load_3d_w(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2,
                                              uint64_t policy) {
    asm volatile(BMOE_ELECT_ISSUE(
                     "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
                     " [%0], [%1, {%3, %4, %5}], [%2], %6") ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
                 : "memory");
}
__device__ __forceinline__ void tma_load_4d_w(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2,
                                              int c3, uint64_t policy) {
    asm volatile(BMOE_ELECT_ISSUE(
                     "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
                     " [%0], [%1, {%3, %4, %5, %6}], [%2], %7") ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
                 "l"(policy)
                 : "memory");
}
__device__ __forceinline__ void bulk_load_w(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(BMOE_ELECT_ISSUE("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3]")
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
// L2 prefetch of one tensor box (no shared memory, no barrier), warp-level like the loads.
__device__ __forceinline__ void tma_prefetch_2d_w(const CUtensorMap* map, int c0, int c1) {
    asm volatile(BMOE_ELECT_ISSUE("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}]")
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void tma_prefetch_3d_w(const CUtensorMap* map, int c0, int c1, int c2) {
    asm volatile(BMOE_ELECT_ISSUE("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}]")
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
__device__ __forceinline__ void tma_prefetch_4d_w(const CUtensorMap* map, int c0, int c1, int c2, int c3) {
    asm volatile(BMOE_ELECT_ISSUE("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}]")
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Warp-level issue: the three helpers below are executed by a whole converged warp and one lane,
// elected with elect.sync over the full mask (the lowest lane, so the same lane every time),
// issues the operation.  Keeping the issuing code warp-uniform lets its operands stay in the
// uniform datapath: on GB300 one warp then issues a block-scaled MMA every ~44 cycles (N = 32)
// and keeps the tensor pipe saturated from N = 128 up, where a divergent single-lane branch
// needs ~100 cycles per MMA.  tcgen05.commit tracks the operations of the issuing thread, so
// the MMAs, the scale copies and their commits of one warp all go through these helpers.
//
// Copy 32 rows x 128 bits from shared memory into TMEM lanes 0-31 (replicated into the four
// 32-lane quadrants), four 32-bit columns starting at taddr.
__device__ __forceinline__ void tc_cp_32x128b_x4_w(uint32_t taddr, uint64_t sdesc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b32 e;\n\t"
        "elect.sync e|p, 0xffffffff;\n\t"
        "@p tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr),
        "l"(sdesc)
        : "memory");
}
// D(tmem) (+)= A(smem) * B(smem)^T with one E8M0 scale per 32 K-elements per row of A and of B,
// the scales read from TMEM (kind::mxf8f6f4); `accumulate` = 0 overwrites D.
__device__ __forceinline__ void tc_mma_mx_w(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t.reg .b32 e;\n\t"
        "elect.sync e|p, 0xffffffff;\n\t"
        "setp.ne.b32 q, %4, 0;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%5], [%6], q;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}
// Arrive on `bar` once every tcgen05 operation the issuing lane issued so far has completed.
__device__ __forceinline__ void tc_commit_w(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b32 e;\n\t"
        "elect.sync e|p, 0xffffffff;\n\t"
        "@p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
            smem_u32(bar))
        : "memory");
}
// Each thread of the warp reads 16 consecutive 32-bit columns of its TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor: K-major operand tile written by TMA with the
// 128-byte swizzle; rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1u) << 16;            // leading byte offset (unused for swizzled K-major)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;    // stride byte offset: next 8-row group
    d |= static_cast<uint64_t>(1u) << 46;            // descriptor version
    d |= static_cast<uint64_t>(2u) << 61;            // 128-byte swizzle
    return d;
}
// Descriptor of one 512-byte scale-factor atom (32 lines of 16 bytes, no
// swizzle; 8-line core matrices 128 bytes apart) as read by tcgen05.cp.
__device__ __forceinline__ uint64_t desc_sf_atom(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(128u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    return d;
}
// Instruction descriptor of kind::mxf8f6f4 with E8M0 scales, both operands K-major.
// fmt codes: 0 = E4M3, 1 = E5M2, 3 = E2M3, 4 = E3M2, 5 = E2M1.
__host__ __device__ constexpr uint32_t idesc_mx(int M, int N, int a_fmt, int b_fmt, int a_sf_id, int b_sf_id) {
    return (static_cast<uint32_t>(b_sf_id & 3) << 4) | (static_cast<uint32_t>(a_fmt) << 7) |
           (static_cast<uint32_t>(b_fmt) << 10) | (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) |
           (static_cast<uint32_t>(M >> 4) << 24) | (static_cast<uint32_t>(a_sf_id & 3) << 29);
}

}  // namespace bmoe

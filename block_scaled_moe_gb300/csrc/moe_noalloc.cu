// moe_noalloc.cu -- compact dispatch for callers that must not allocate device
// memory.
//
// Who needs this: code that runs while a CUDA graph is being captured (where
// cudaMalloc is not allowed), and serving engines that reserve the whole device
// up front for weights and caches and forbid any later allocation.  A handle
// from moe_create owns a cudaMalloc'ed workspace, so such callers cannot build
// one; this entry point instead keeps its scratch in a fixed array compiled into
// the library and writes its results only into the caller's buffers.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "blockmoe.h"
#include "moe_internal.h"

namespace {

// Scratch of the allocation-free dispatch: per-chunk expert counts (nchunks*E
// int32), the route-tile scan (E+1 int32) and the last-block ticket / status
// words.  Every GPU that loads the library holds this array until the process
// exits.  All calls share it, so calls that overlap on the GPU race.
constexpr size_t kScratchBytes = size_t(1) << 20;  // 1 MiB
constexpr size_t kScratchHeader = 256;             // ticket[8] and status[4] words, padded
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};
int fail(int code, const char* msg) {
    bmoe::note_unbound_error(msg);  // readable with moe_last_error(NULL)
    return code;
}

// Device address of the scratch array on the current device; looked up once per
// device (the host-side symbol is only a stand-in and must not reach a kernel),
// together with the dispatch kernel's shared-memory limit.
int scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return fail(MOE_ECUDA, "moe_dispatch_compact_noalloc: no usable current CUDA device");
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            char buf[256];
            snprintf(buf, sizeof(buf), "moe_dispatch_compact_noalloc: cudaGetSymbolAddress failed: %s",
                     cudaGetErrorString(e));
            return fail(MOE_ECUDA, buf);
        }
        e = bmoe::dispatch_set_attributes();  // the count kernel's shared memory for large E, once per device
        if (e != cudaSuccess) {
            char buf[256];
            snprintf(buf, sizeof(buf), "moe_dispatch_compact_noalloc: setting the dispatch kernel's shared memory "
                     "limit failed: %s", cudaGetErrorString(e));
            return fail(MOE_ECUDA, buf);
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}

size_t scratch_needed(int T, int topk, int E) {
    const size_t slots = static_cast<size_t>(T) * topk;
    const size_t nchunks = (slots + bmoe::kChunk - 1) / bmoe::kChunk;
    return kScratchHeader + sizeof(int32_t) * (nchunks * static_cast<size_t>(E) + static_cast<size_t>(E) + 1);
}

}  // namespace

extern "C" {

int moe_dispatch_compact_noalloc(const int32_t* topk_ids, int T, int topk, int E, const int32_t* num_valid_rows,
                                 int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* route_row,
                                 moe_stream_t stream) {
    if (T < 0 || topk < 1 || topk > bmoe::kMaxTopk || E < 1 || E > bmoe::kMaxExperts)
        return fail(MOE_EINVAL, "moe_dispatch_compact_noalloc: need T >= 0, 1 <= topk <= 16, 1 <= E <= 4096");
    const size_t need = scratch_needed(T, topk, E);
    if (need > kScratchBytes) {
        char buf[256];
        snprintf(buf, sizeof(buf),
                 "moe_dispatch_compact_noalloc: T=%d, topk=%d, E=%d needs %zu bytes of scratch; the built-in "
                 "array holds %zu (about (T*topk/512 + 1) * E <= 262000)",
                 T, topk, E, need, kScratchBytes);
        return fail(MOE_ECAPACITY, buf);
    }
    if (!counts || !offsets) return fail(MOE_EINVAL, "moe_dispatch_compact_noalloc: counts and offsets are required");
    if (T > 0 && (!topk_ids || !perm || !route_row))
        return fail(MOE_EINVAL, "moe_dispatch_compact_noalloc: topk_ids, perm and route_row are required when T > 0");
    void* base = nullptr;
    int rc = scratch_address(&base);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned char* sc = static_cast<unsigned char*>(base);
    // the ticket and status words must start at zero on every call
    cudaError_t e = cudaMemsetAsync(sc, 0, kScratchHeader, s);
    if (e != cudaSuccess) return fail(MOE_ECUDA, "moe_dispatch_compact_noalloc: clearing scratch failed");
    if (T == 0) {
        e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s);
        return e == cudaSuccess ? MOE_OK : fail(MOE_ECUDA, "moe_dispatch_compact_noalloc: memset failed");
    }
    bmoe::Geometry g{};
    g.E = E;
    g.K = topk;
    g.cap = T;
    g.NT = 128;
    bmoe::Workspace w{};
    w.ticket = reinterpret_cast<uint32_t*>(sc);       // 8 words
    w.status = reinterpret_cast<uint32_t*>(sc + 32);
    w.chunk_base = reinterpret_cast<int32_t*>(sc + kScratchHeader);
    const size_t nchunks = (static_cast<size_t>(T) * topk + bmoe::kChunk - 1) / bmoe::kChunk;
    w.tile_base = w.chunk_base + nchunks * E;
    w.counts = counts;
    w.rowbase = offsets;
    w.perm = perm;
    w.route_row = route_row;
#ifdef MOE_DEBUG_BOUNDS
    w.lim_slots = T * topk;  // the caller's perm and route_row
    w.lim_chunks = static_cast<int>(nchunks);
#endif
    e = bmoe::launch_compact_dispatch(g, w, topk_ids, T, num_valid_rows, s);
    if (e != cudaSuccess) {
        char buf[256];
        snprintf(buf, sizeof(buf), "moe_dispatch_compact_noalloc: launch failed: %s", cudaGetErrorString(e));
        return fail(MOE_ECUDA, buf);
    }
    return MOE_OK;
}

}  // extern "C"

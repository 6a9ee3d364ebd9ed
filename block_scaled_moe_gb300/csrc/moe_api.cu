// moe_api.cu -- the C ABI of include/blockmoe.h: handle state, argument and
// weight validation, workspace carving, TMA descriptors and the launch order
// of one forward (dispatch -> quant/scatter -> GEMM1 -> GEMM2 -> combine),
// all on the caller's stream with no host synchronisation.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdarg>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "blockmoe.h"
#include "moe_internal.h"

using bmoe::Geometry;
using bmoe::Workspace;

#ifdef BMOE_TRACE
extern "C" {
long long* bmoe_trace_buffer = nullptr;  // device pointer of the pipeline trace (tracing builds)
// Copy the stand-alone GEMMs' trace of the last multi-kernel forward into host memory (synchronous).
int bmoe_gemm_trace_copy(void* dst, size_t bytes) {
    if (!bmoe_trace_buffer) return -1;
    const size_t all = sizeof(long long) * 2 * (2 * 8 * 512 + 2 * 1024);
    return static_cast<int>(cudaMemcpy(dst, bmoe_trace_buffer, bytes < all ? bytes : all, cudaMemcpyDeviceToHost));
}
}
#endif

// One bound layer: the caller's weight buffers (not owned) and their tensor maps.
struct Binding {
    bool bound = false;
    int w13_layout = MOE_W13_CONCAT;
    const uint8_t* w13 = nullptr;
    const uint8_t* w13s = nullptr;
    const uint8_t* w2 = nullptr;
    const uint8_t* w2s = nullptr;
    CUtensorMap tm_w13p{};  // W13 gate/up pair view (K, feature, half, expert)
    CUtensorMap tm_w2{};
    CUtensorMap tm_w2w{};   // W2 with 256-row boxes (paired tiles of prefill GEMM2)
    CUtensorMap tm_w2k2{};  // W2 as (K in chunk, row, K chunk): one box = two 128-wide K chunks (I % 256 == 0)
};

struct moe_ctx {
    int device = -1;
    int num_sms = 0;
    Geometry geo{};
    int opt_dispatch = MOE_DISPATCH_AUTO;
    double swiglu_limit = 0.0;
    int fixed_slot_max = 255;
    int debug = 0;
    int route_tile = 0;
    bool forwarded = false;
    void* ws_mem = nullptr;
    size_t ws_bytes = 0;
    bool ws_owned = false;
    Workspace ws{};
    std::vector<Binding> slots = std::vector<Binding>(1);  // layer slots; forwards use slots[cur]
    int cur = 0;
    int opt_w13_layout = MOE_W13_CONCAT;  // layout the next bind assumes
    int y_format = MOE_Y_BF16;            // GEMM2 rows handed to the combine
    CUtensorMap tm_aq{}, tm_hq{};
    CUtensorMap tm_hqk2{};  // h rows as (K in chunk, row, K chunk), two K chunks per box (I % 256 == 0)
    int last_T = 0;
    int profile = 0;
    bool profiled = false;
    int opt_path = MOE_PATH_AUTO;
    int last_path = 0;
    // T-bucketed path table (bucket T ascending, MOE_PATH_FUSED / MOE_PATH_MULTI); empty = default rule
    std::vector<int32_t> tune_t, tune_path;
    bool coop = false;  // device supports cooperative launches
    cudaEvent_t ev[MOE_PROFILE_STAGES + 1] = {};
    unsigned long long launches = 0;
    std::string err;
};

namespace {

thread_local std::string g_create_err;

int fail(moe_ctx* h, int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    if (h)
        h->err = buf;
    else
        g_create_err = buf;
    return code;
}

int cuda_fail(moe_ctx* h, cudaError_t e, const char* what) {
    return fail(h, MOE_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2D K-major tile map: inner dim = K elements, outer = rows; box 128 x box_rows, 128B swizzle.
int make_map(moe_ctx* h, CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t K, uint64_t rows,
             uint64_t row_bytes, uint32_t box_rows, CUtensorMapL2promotion l2) {
    auto fn = encode_fn();
    if (!fn) return fail(h, MOE_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[2] = {K, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(h, MOE_ECUDA, "cuTensorMapEncodeTiled failed (%d) for a %llu x %llu tensor", (int)r,
                    (unsigned long long)rows, (unsigned long long)K);
    return MOE_OK;
}

// L2 promotion of the weight maps: a box reads 64 bytes of each weight row per K stage.  With
// 256-byte promotion one stage in four fetched four stages of every row from DRAM and the ring
// waited on it, and where the row pitch is not a multiple of 256 bytes (W2 rows of I/2 = 1152
// bytes) a row's last promoted block, shared with the next row, was read twice (~3% extra DRAM
// bytes on the single-launch decode).  128-byte promotion measured faster on every workload
// (decode -1.1%, small-M -0.7%, 8192-row prefill -1.3 to -1.7%, skewed prefill +-0.3%).
CUtensorMapL2promotion weight_promotion(uint64_t /*row_bytes*/) { return CU_TENSOR_MAP_L2_PROMOTION_L2_128B; }

// W13 as a 4D view (K, output feature j, half: gate / up, expert) so that one box
// {128, 128, 2, 1} brings the gate tile and the matching up tile of a unit's K
// chunk: a GEMM1 stage is one TMA.  Concatenated halves: feature stride one row,
// half stride I rows; interleaved rows (gate j at 2j, up j at 2j + 1): feature
// stride two rows, half stride one row.
int make_map_w13_pair(moe_ctx* h, CUtensorMap* m, const void* base, uint64_t H, uint64_t I, uint64_t E,
                      bool interleaved, CUtensorMapL2promotion l2) {
    auto fn = encode_fn();
    if (!fn) return fail(h, MOE_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const uint64_t row = H / 2;
    cuuint64_t dims[4] = {H, I, 2, E};
    cuuint64_t strides[3] = {interleaved ? 2 * row : row, interleaved ? row : I * row, 2 * I * row};
    cuuint32_t box[4] = {128, 128, 2, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 4, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(h, MOE_ECUDA, "cuTensorMapEncodeTiled failed (%d) for the W13 pair view", (int)r);
    return MOE_OK;
}

// K-major rows as a 3D view (128 K-elements of a chunk, row, chunk) so that one box {128, box_rows, 2}
// brings two consecutive 128-wide K chunks, landing chunk-major in shared memory exactly like two
// 2D boxes would: the decode GEMM2's 256-wide K stages take one TMA per operand instead of two.
int make_map_k2(moe_ctx* h, CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t K, uint64_t rows,
                uint64_t row_bytes, uint64_t chunk_bytes, uint32_t box_rows, CUtensorMapL2promotion l2) {
    auto fn = encode_fn();
    if (!fn) return fail(h, MOE_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[3] = {128, rows, K / 128};
    cuuint64_t strides[2] = {row_bytes, chunk_bytes};
    cuuint32_t box[3] = {128, box_rows, 2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(h, MOE_ECUDA, "cuTensorMapEncodeTiled failed (%d) for a two-chunk view", (int)r);
    return MOE_OK;
}

void compute_geometry(moe_ctx* h, Geometry* g) {
    *g = h->geo;
    const bool fixed = h->opt_dispatch == MOE_DISPATCH_FIXED ||
                       (h->opt_dispatch == MOE_DISPATCH_AUTO && g->cap <= h->fixed_slot_max);
    g->scheme = fixed ? 1 : 2;
    g->mtpr = g->cap;
    g->words = (g->cap + 31) / 32;
    int NT = h->route_tile;
    // decode tiles of 32 rows; prefill tiles of 144: most experts of a uniform 8192-row prefill hold
    // 110-150 routes, which 128-row tiles would split into a full tile and a nearly empty one
    if (NT == 0) NT = ((long long)g->cap * g->K <= 8LL * g->E) ? 32 : 144;
    g->NT = NT;
    g->nb = (NT + 127) / 128;
    const long long slots = (long long)g->cap * g->K;
    if (fixed) {
        g->rows_cap = (long long)g->E * g->mtpr;
        g->tiles_cap = (long long)g->E * ((g->mtpr + NT - 1) / NT);
    } else {
        g->rows_cap = slots;
        g->tiles_cap = slots / NT + g->E;
    }
    // the row-tile TMA box is NT rows high: keep the packed tensors at least that tall
    g->rows_cap = (g->rows_cap + NT - 1) / NT * NT;
    if (g->tiles_cap < 1) g->tiles_cap = 1;
    g->nchunks_cap = (int)((slots + bmoe::kChunk - 1) / bmoe::kChunk);
    g->debug = h->debug != 0;
}

int setup_workspace_maps(moe_ctx* h) {
    const Geometry& g = h->geo;
    int rc = make_map(h, &h->tm_aq, CU_TENSOR_MAP_DATA_TYPE_UINT8, h->ws.aq, g.H, g.rows_cap, g.H, g.NT,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
    if (rc) return rc;
    rc = make_map(h, &h->tm_hq, CU_TENSOR_MAP_DATA_TYPE_UINT8, h->ws.hq, g.I, g.rows_cap, g.I, g.NT,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
    if (rc || g.I % 256) return rc;
    return make_map_k2(h, &h->tm_hqk2, CU_TENSOR_MAP_DATA_TYPE_UINT8, h->ws.hq, g.I, g.rows_cap, g.I, 128, g.NT,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
}

void release_workspace(moe_ctx* h) {
    if (h->ws_owned && h->ws_mem) cudaFree(h->ws_mem);
    h->ws_mem = nullptr;
    h->ws_bytes = 0;
    h->ws_owned = false;
    h->ws = Workspace{};
}

// Point the handle at `mem` (bytes) for the current geometry and clear the counters.
int adopt_workspace(moe_ctx* h, void* mem, size_t bytes, bool owned) {
    Workspace w{};
    const size_t need = bmoe::workspace_layout(h->geo, static_cast<char*>(mem), &w);
    if (bytes < need) return fail(h, MOE_ENOMEM, "workspace holds %zu bytes, %zu needed", bytes, need);
    cudaError_t e = cudaMemset(w.ticket, 0, 8 * sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMemset(w.status, 0, 4 * sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_fail(h, e, "clearing workspace counters");
    release_workspace(h);
    h->ws_mem = mem;
    h->ws_bytes = bytes;
    h->ws_owned = owned;
    h->ws = w;
    return setup_workspace_maps(h);
}

int allocate_own_workspace(moe_ctx* h) {
    const size_t need = bmoe::workspace_layout(h->geo, nullptr, nullptr);
    void* mem = nullptr;
    cudaError_t e = cudaMalloc(&mem, need);
    if (e != cudaSuccess) return fail(h, MOE_ENOMEM, "cudaMalloc(%zu) for the workspace: %s", need, cudaGetErrorString(e));
    int rc = adopt_workspace(h, mem, need, true);
    if (rc) cudaFree(mem);
    return rc;
}

// Re-derive the geometry after an option change; reallocate an owned workspace.
int regeometry(moe_ctx* h) {
    Geometry g;
    compute_geometry(h, &g);
    h->geo = g;
    if (h->ws_owned || !h->ws_mem) {
        release_workspace(h);
        return allocate_own_workspace(h);
    }
    const size_t need = bmoe::workspace_layout(g, nullptr, nullptr);
    if (need > h->ws_bytes) {
        h->ws_mem = nullptr;
        h->ws = Workspace{};
        return fail(h, MOE_ENOMEM, "caller workspace too small for the new options (%zu needed)", need);
    }
    return adopt_workspace(h, h->ws_mem, h->ws_bytes, false);
}

int check_device_ptr(moe_ctx* h, const void* p, const char* name, size_t align) {
    if (!p) return fail(h, MOE_EINVAL, "%s is NULL", name);
    if (reinterpret_cast<uintptr_t>(p) % align)
        return fail(h, MOE_EINVAL, "%s is not %zu-byte aligned", name, align);
    cudaPointerAttributes at;
    cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(h, MOE_EINVAL, "%s is not a CUDA pointer (%s)", name, cudaGetErrorString(e));
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
        return fail(h, MOE_EINVAL, "%s is not device memory", name);
    if (at.device != h->device) return fail(h, MOE_EINVAL, "%s lives on device %d, the handle on %d", name, at.device, h->device);
    return MOE_OK;
}

}  // namespace

void bmoe::note_unbound_error(const char* msg) { g_create_err = msg; }

extern "C" {

int moe_create(moe_handle* out, int H, int I, int E, int topk, int capacity) {
    if (!out) return fail(nullptr, MOE_EINVAL, "out is NULL");
    *out = nullptr;
    if (H <= 0 || I <= 0 || H % 128 || I % 128)
        return fail(nullptr, MOE_ESHAPE, "H=%d and I=%d must be positive multiples of 128", H, I);
    if (E < 1 || E > bmoe::kMaxExperts) return fail(nullptr, MOE_ESHAPE, "E=%d outside [1, %d]", E, bmoe::kMaxExperts);
    if (topk < 1 || topk > bmoe::kMaxTopk) return fail(nullptr, MOE_ESHAPE, "topk=%d outside [1, %d]", topk, bmoe::kMaxTopk);
    if (capacity < 1) return fail(nullptr, MOE_EINVAL, "capacity=%d must be >= 1", capacity);
    if ((long long)capacity * topk > (1LL << 30)) return fail(nullptr, MOE_EINVAL, "capacity * topk too large");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(nullptr, MOE_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, dev);
    if (e != cudaSuccess) return fail(nullptr, MOE_ECUDA, "cudaGetDeviceProperties: %s", cudaGetErrorString(e));
    if (!(prop.major == 10 && prop.minor == 3))
        return fail(nullptr, MOE_EDEVICE, "device %d is sm_%d%d; this library is built for sm_103a (GB300)", dev,
                    prop.major, prop.minor);
    e = bmoe::gemm_set_attributes();
    if (e == cudaSuccess) e = bmoe::fused_set_attributes();
    if (e == cudaSuccess) e = bmoe::dispatch_set_attributes();
    if (e != cudaSuccess) return fail(nullptr, MOE_ECUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    int coop = 0;
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    moe_ctx* h = new (std::nothrow) moe_ctx();
    if (!h) return fail(nullptr, MOE_ENOMEM, "host allocation failed");
    h->device = dev;
    h->num_sms = prop.multiProcessorCount;
    h->coop = coop != 0;
    h->geo.H = H;
    h->geo.I = I;
    h->geo.E = E;
    h->geo.K = topk;
    h->geo.cap = capacity;
    Geometry g;
    compute_geometry(h, &g);
    h->geo = g;
    int rc = allocate_own_workspace(h);
    if (rc) {
        g_create_err = h->err;
        delete h;
        return rc;
    }
    *out = h;
    return MOE_OK;
}

void moe_destroy(moe_handle h) {
    if (!h) return;
    for (auto& e : h->ev)
        if (e) cudaEventDestroy(e);
    release_workspace(h);
    delete h;
}

namespace {

// Validate the weights and build their tensor maps into *b; nothing of the handle changes.
int prepare_binding(moe_handle h, Binding* b, const void* w13_fp4, const void* w13_sf, const void* w2_fp4,
                    const void* w2_sf) {
    int rc;
    if ((rc = check_device_ptr(h, w13_fp4, "w13_fp4", 32))) return rc;
    if ((rc = check_device_ptr(h, w13_sf, "w13_sf", 16))) return rc;
    if ((rc = check_device_ptr(h, w2_fp4, "w2_fp4", 32))) return rc;
    if ((rc = check_device_ptr(h, w2_sf, "w2_sf", 16))) return rc;
    const Geometry& g = h->geo;
    const bool inter = h->opt_w13_layout == MOE_W13_INTERLEAVED;
    if ((rc = make_map_w13_pair(h, &b->tm_w13p, w13_fp4, g.H, g.I, g.E, inter, weight_promotion(g.H / 2)))) return rc;
    const CUtensorMapL2promotion w2p = weight_promotion(g.I / 2);
    if ((rc = make_map(h, &b->tm_w2, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w2_fp4, g.I, (uint64_t)g.E * g.H, g.I / 2,
                       128, w2p)))
        return rc;
    if ((rc = make_map(h, &b->tm_w2w, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w2_fp4, g.I, (uint64_t)g.E * g.H, g.I / 2,
                       256, w2p)))
        return rc;
    if (g.I % 256 == 0 &&
        (rc = make_map_k2(h, &b->tm_w2k2, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w2_fp4, g.I, (uint64_t)g.E * g.H,
                          g.I / 2, 64, 128, w2p)))
        return rc;
    b->w13_layout = h->opt_w13_layout;
    b->w13 = static_cast<const uint8_t*>(w13_fp4);
    b->w13s = static_cast<const uint8_t*>(w13_sf);
    b->w2 = static_cast<const uint8_t*>(w2_fp4);
    b->w2s = static_cast<const uint8_t*>(w2_sf);
    b->bound = true;
    return MOE_OK;
}

}  // namespace

int moe_bind_weights(moe_handle h, const void* w13_fp4, const void* w13_sf, const void* w2_fp4, const void* w2_sf) {
    if (!h) return MOE_EINVAL;
    Binding b;
    const int rc = prepare_binding(h, &b, w13_fp4, w13_sf, w2_fp4, w2_sf);
    if (rc) return rc;
    h->slots[h->cur] = b;  // everything validated: switch the binding
    return MOE_OK;
}

int moe_bind_layer(moe_handle h, int slot, const void* w13_fp4, const void* w13_sf, const void* w2_fp4,
                   const void* w2_sf) {
    if (!h) return MOE_EINVAL;
    if (slot < 0 || slot >= static_cast<int>(h->slots.size()))
        return fail(h, MOE_EINVAL, "slot %d outside [0, %d)", slot, static_cast<int>(h->slots.size()));
    Binding b;
    const int rc = prepare_binding(h, &b, w13_fp4, w13_sf, w2_fp4, w2_sf);
    if (rc) return rc;
    h->slots[slot] = b;  // checked slot, then weights, then switch
    h->cur = slot;
    return MOE_OK;
}

int moe_select_layer(moe_handle h, int slot) {
    if (!h) return MOE_EINVAL;
    if (slot < 0 || slot >= static_cast<int>(h->slots.size()))
        return fail(h, MOE_EINVAL, "slot %d outside [0, %d)", slot, static_cast<int>(h->slots.size()));
    if (!h->slots[slot].bound) return fail(h, MOE_ENOTBOUND, "slot %d has no weights bound", slot);
    h->cur = slot;
    return MOE_OK;
}

namespace {

// Path of the table bucket nearest to T (ties: the larger bucket), as the pages' configuration
// lookup does for a token count between measured buckets.
int table_path(const moe_ctx* h, int T) {
    size_t best = 0;
    for (size_t i = 1; i < h->tune_t.size(); ++i) {
        const long d = std::labs((long)h->tune_t[i] - T), db = std::labs((long)h->tune_t[best] - T);
        if (d <= db) best = i;  // ascending buckets: "<=" lets the larger of two equal distances win
    }
    return h->tune_path[best];
}

}  // namespace

int moe_forward(moe_handle h, const void* x, const int32_t* topk_ids, const float* topk_weights,
                const int32_t* num_valid_rows, void* out, int T, moe_stream_t stream) {
    if (!h) return MOE_EINVAL;
    const Geometry& g = h->geo;
    if (T < 0) return fail(h, MOE_EINVAL, "T=%d is negative", T);
    if (T > g.cap) return fail(h, MOE_ECAPACITY, "T=%d exceeds the capacity %d", T, g.cap);
    const Binding& wb = h->slots[h->cur];
    if (!wb.bound) return fail(h, MOE_ENOTBOUND, "no weights bound");
    if (!h->ws_mem) return fail(h, MOE_ENOMEM, "no workspace");
    if (T == 0) return MOE_OK;
    if (!x || !topk_ids || !topk_weights || !out) return fail(h, MOE_EINVAL, "x, topk_ids, topk_weights and out must be non-NULL");
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) & 15)
        return fail(h, MOE_EINVAL, "x and out must be 16-byte aligned");
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device)
        return fail(h, MOE_EINVAL, "current device %d is not the handle's device %d", cur, h->device);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Workspace& ws = h->ws;
    cudaError_t e;
    const bool prof = h->profile != 0;
    auto mark = [&](int i) {
        if (prof) cudaEventRecord(h->ev[i], s);
    };
    // MXFP8 GEMM2 rows live in the y region: codes [rows_cap][H], then scales [rows_cap][H/32]
    uint8_t* y8 = h->y_format == MOE_Y_MXFP8 ? reinterpret_cast<uint8_t*>(ws.y) : nullptr;
    uint8_t* ys = y8 ? y8 + (size_t)g.rows_cap * g.H : nullptr;
    mark(0);
    const bool fused = h->opt_path != MOE_PATH_MULTI && h->coop && bmoe::fused_supported(g) &&
                       (h->opt_path == MOE_PATH_FUSED ||
                        (h->tune_t.empty() ? T <= 512 : table_path(h, T) == MOE_PATH_FUSED));
    if (fused) {
        bmoe::FusedLaunch fl;
        fl.x = static_cast<const uint16_t*>(x);
        fl.ids = topk_ids;
        fl.wts = topk_weights;
        fl.nvr = num_valid_rows;
        fl.out = static_cast<uint16_t*>(out);
        fl.w13s = wb.w13s;
        fl.w2s = wb.w2s;
        fl.w13_rs = wb.w13_layout == MOE_W13_INTERLEAVED ? 2 : 1;
        fl.w13_up = wb.w13_layout == MOE_W13_INTERLEAVED ? 1 : g.I;
        fl.y8 = y8;
        fl.ys = ys;
        fl.swiglu_limit = static_cast<float>(h->swiglu_limit);
        fl.T = T;
        mark(1);
        mark(2);
        // GEMM2 takes W2 tiles in pairs (H % 256 == 0: the 256-row W2 boxes, 128-wide K stages); else
        // 256-wide K stages (I % 256 == 0) read W2 and h through the two-chunk views
        const bool w2w = g.H % 256 == 0, k2 = !w2w && g.I % 256 == 0;
        e = bmoe::launch_fused(g, ws, fl, &wb.tm_w13p, &h->tm_aq,
                               w2w ? &wb.tm_w2w : (k2 ? &wb.tm_w2k2 : &wb.tm_w2), k2 ? &h->tm_hqk2 : &h->tm_hq,
                               h->num_sms, s);
        if (e == cudaErrorCooperativeLaunchTooLarge && h->opt_path != MOE_PATH_FUSED) {
            // the driver could not make the grid co-resident (fewer SMs available to this context than
            // the device reports): nothing was enqueued; take the multi-kernel path from now on
            (void)cudaGetLastError();
            h->coop = false;
        } else if (e != cudaSuccess) {
            return cuda_fail(h, e, "fused launch");
        } else {
            h->launches += 1;
            mark(3);
            mark(4);
            mark(5);
            h->profiled = prof;
            h->forwarded = true;
            h->last_T = T;
            h->last_path = MOE_PATH_FUSED;
            return MOE_OK;
        }
    }
    if (g.scheme == 1) {
        e = cudaMemsetAsync(ws.occ, 0, sizeof(uint32_t) * (size_t)g.E * g.words, s);
        if (e != cudaSuccess) return cuda_fail(h, e, "clearing occupancy");
        e = bmoe::launch_fixed_mark(g, ws, topk_ids, T, num_valid_rows, s);
    } else {
        e = bmoe::launch_compact_dispatch(g, ws, topk_ids, T, num_valid_rows, s);
    }
    if (e != cudaSuccess) return cuda_fail(h, e, "dispatch launch");
    h->launches += g.scheme == 1 ? 1 : 2;
    mark(1);
    e = bmoe::launch_quant_scatter(g, ws, static_cast<const uint16_t*>(x), topk_ids, T, num_valid_rows, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "quant launch");
    h->launches += 1;
    mark(2);

    bmoe::GemmArgs a{};
    a.counts = ws.counts;
    a.rowbase = ws.rowbase;
    a.tile_base = ws.tile_base;
    a.E = g.E;
    a.swiglu_limit = static_cast<float>(h->swiglu_limit);
    a.status = ws.status;
#ifdef MOE_DEBUG_BOUNDS
    a.ticket = ws.ticket;
    a.lim_rows = ws.lim_rows;
    a.lim_tiles = ws.lim_tiles;
#endif
    a.y8 = y8;
    a.ys = ys;
    a.trace = nullptr;
#ifdef BMOE_TRACE
    // per GEMM: [2 CTAs][8][512] clock64 stamps, then [1024 CTAs][2] globaltimer start / end
    static long long* trace_buf = nullptr;
    if (!trace_buf) cudaMalloc(&trace_buf, sizeof(long long) * 2 * (2 * 8 * 512 + 2 * 1024));
    a.trace = trace_buf;
    bmoe_trace_buffer = trace_buf;
#endif
    a.I = g.I;
    a.H = g.H;
    // GEMM1: W13 (gate/up pairs) x dispatched rows, K = H
    a.w_sf = wb.w13s;
    a.w_rows = 2 * g.I;
    a.ld_sf = g.H / 32;
    a.up_off = wb.w13_layout == MOE_W13_INTERLEAVED ? 1 : g.I;
    a.w_rs = wb.w13_layout == MOE_W13_INTERLEAVED ? 2 : 1;
    a.m_rows = 128;
    a.ktiles = g.H / 128;
    a.mtiles = g.I / 128;
    a.b_sf = ws.as;
    a.hq = ws.hq;
    a.hs = ws.hs;
    a.g_dbg = g.debug ? ws.g : nullptr;
    e = bmoe::launch_gemm1(a, &wb.tm_w13p, &h->tm_aq, g.NT, h->num_sms, s);
#ifdef BMOE_TRACE
    a.trace = trace_buf + 2 * 8 * 512 + 2 * 1024;
#endif
    if (e != cudaSuccess) return cuda_fail(h, e, "GEMM1 launch");
    h->launches += 1;
    mark(3);
    // GEMM2: W2 x h rows, K = I
    // W2 tiles go in pairs when H allows it (one 256-row box, alternate accumulator chains per tile)
    const bool w2_pairs = g.H % 256 == 0;
    a.w_sf = wb.w2s;
    a.w_rows = g.H;
    a.ld_sf = g.I / 32;
    a.up_off = w2_pairs ? 128 : 0;
    a.w_rs = 1;
    a.m_rows = w2_pairs ? 256 : 128;
    a.ktiles = g.I / 128;
    a.mtiles = g.H / a.m_rows;
    a.b_sf = ws.hs;
    a.y = ws.y;
    a.g_dbg = nullptr;
    e = bmoe::launch_gemm2(a, &wb.tm_w2, &wb.tm_w2w, &wb.tm_w2k2, &h->tm_hq, &h->tm_hqk2, g.NT, h->num_sms, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "GEMM2 launch");
    h->launches += 1;
    mark(4);
    e = bmoe::launch_combine(g, ws, topk_weights, T, num_valid_rows, static_cast<uint16_t*>(out), y8, ys, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "combine launch");
    h->launches += 1;
    mark(5);
    h->profiled = prof;
    h->forwarded = true;
    h->last_T = T;
    h->last_path = MOE_PATH_MULTI;
    return MOE_OK;
}

int moe_set_option(moe_handle h, int key, double value) {
    if (!h) return MOE_EINVAL;
    switch (key) {
        case MOE_OPT_SWIGLU_LIMIT:
            if (!(value >= 0.0)) return fail(h, MOE_EINVAL, "swiglu limit must be >= 0");
            h->swiglu_limit = value;
            return MOE_OK;
        case MOE_OPT_PROFILE: {
            const int v = value != 0.0 ? 1 : 0;
            if (v)
                for (auto& ev : h->ev)
                    if (!ev) {
                        cudaError_t e = cudaEventCreate(&ev);
                        if (e != cudaSuccess) return cuda_fail(h, e, "cudaEventCreate");
                    }
            h->profile = v;
            h->profiled = false;
            return MOE_OK;
        }
        case MOE_OPT_LAUNCHES:
        case MOE_OPT_LAYER:
            return fail(h, MOE_EINVAL, "option %d is read-only", key);
        case MOE_OPT_W13_LAYOUT: {
            const int v = static_cast<int>(value);
            if (static_cast<double>(v) != value || (v != MOE_W13_CONCAT && v != MOE_W13_INTERLEAVED))
                return fail(h, MOE_EINVAL, "bad W13 layout %g", value);
            h->opt_w13_layout = v;
            return MOE_OK;
        }
        case MOE_OPT_Y_FORMAT: {
            const int v = static_cast<int>(value);
            if (static_cast<double>(v) != value || (v != MOE_Y_BF16 && v != MOE_Y_MXFP8))
                return fail(h, MOE_EINVAL, "bad GEMM2 row format %g", value);
            h->y_format = v;
            return MOE_OK;
        }
        case MOE_OPT_DEBUG_GRID_GEN: {
            if (value < 0 || value >= 4294967296.0 || static_cast<double>(static_cast<uint64_t>(value)) != value)
                return fail(h, MOE_EINVAL, "the generation word takes an integer in [0, 2^32)");
            if (!h->ws_mem) return fail(h, MOE_ENOMEM, "no workspace");
            const uint32_t g = static_cast<uint32_t>(static_cast<uint64_t>(value));
            cudaError_t e = cudaMemcpy(h->ws.ticket + 3, &g, sizeof(g), cudaMemcpyHostToDevice);
            if (e != cudaSuccess) return cuda_fail(h, e, "presetting the grid-barrier word");
            return MOE_OK;
        }
        case MOE_OPT_DEBUG_STALL_GRID: {
            if (value != 1.0) return fail(h, MOE_EINVAL, "the stall takes the value 1");
            if (!h->ws_mem) return fail(h, MOE_ENOMEM, "no workspace");
            // far from the grid size, so that no arrival count ever equals it
            const uint32_t c = 0x80000000u;
            cudaError_t e = cudaMemcpy(h->ws.ticket + 2, &c, sizeof(c), cudaMemcpyHostToDevice);
            if (e != cudaSuccess) return cuda_fail(h, e, "presetting the grid-barrier count");
            return MOE_OK;
        }
        case MOE_OPT_DEBUG_BOUNDS_ROWS: {
#ifdef MOE_DEBUG_BOUNDS
            const long long v = static_cast<long long>(value);
            if (static_cast<double>(v) != value || v < 1 || v > h->geo.rows_cap)
                return fail(h, MOE_EINVAL, "the row limit takes an integer in [1, %lld]", h->geo.rows_cap);
            h->ws.lim_rows = static_cast<int>(v);
            return MOE_OK;
#else
            return fail(h, MOE_ESTATE, "not a bounds-checking build (libblockmoe_bounds.so)");
#endif
        }
        case MOE_OPT_LAYER_SLOTS: {
            const int v = static_cast<int>(value);
            if (static_cast<double>(v) != value || v < 1 || v > 4096)
                return fail(h, MOE_EINVAL, "layer slots must be an integer in [1, 4096]");
            if (h->cur >= v) return fail(h, MOE_EINVAL, "slot %d is the current layer; keep at least %d slots", h->cur, h->cur + 1);
            h->slots.resize(static_cast<size_t>(v));
            return MOE_OK;
        }
        case MOE_OPT_PATH: {
            const int v = static_cast<int>(value);
            if (static_cast<double>(v) != value || v < MOE_PATH_AUTO || v > MOE_PATH_MULTI)
                return fail(h, MOE_EINVAL, "bad path %g", value);
            if (v == MOE_PATH_FUSED && !(h->coop && bmoe::fused_supported(h->geo)))
                return fail(h, MOE_EINVAL, "the fused path needs capacity <= 512, route tile 32, E <= 512 and a "
                                           "cooperative-launch device");
            h->opt_path = v;
            return MOE_OK;
        }
        case MOE_OPT_DISPATCH:
        case MOE_OPT_FIXED_SLOT_MAX:
        case MOE_OPT_DEBUG_CAPTURE:
        case MOE_OPT_ROUTE_TILE: {
            if (h->forwarded) return fail(h, MOE_ESTATE, "option %d changes the workspace layout; set it before the first forward", key);
            const int v = static_cast<int>(value);
            if (static_cast<double>(v) != value) return fail(h, MOE_EINVAL, "option %d takes an integer", key);
            moe_ctx saved = *h;
            if (key == MOE_OPT_DISPATCH) {
                if (v < MOE_DISPATCH_AUTO || v > MOE_DISPATCH_COMPACT) return fail(h, MOE_EINVAL, "bad dispatch scheme %d", v);
                if (v == MOE_DISPATCH_FIXED && h->geo.cap > 4096)
                    return fail(h, MOE_EINVAL, "fixed-slot dispatch needs capacity <= 4096");
                h->opt_dispatch = v;
            } else if (key == MOE_OPT_FIXED_SLOT_MAX) {
                if (v < 0) return fail(h, MOE_EINVAL, "fixed-slot max must be >= 0");
                h->fixed_slot_max = v;
            } else if (key == MOE_OPT_DEBUG_CAPTURE) {
                h->debug = v ? 1 : 0;
            } else {
                if (v != 0 && v != 32 && v != 128 && v != 144)
                    return fail(h, MOE_EINVAL, "route tile must be 0, 32, 128 or 144");
                h->route_tile = v;
            }
            Geometry g;
            compute_geometry(h, &g);
            if (memcmp(&g, &h->geo, sizeof(g)) == 0) return MOE_OK;
            int rc = regeometry(h);
            if (rc) {  // restore the previous options and workspace
                std::string msg = h->err;
                h->opt_dispatch = saved.opt_dispatch;
                h->fixed_slot_max = saved.fixed_slot_max;
                h->debug = saved.debug;
                h->route_tile = saved.route_tile;
                compute_geometry(h, &g);
                h->geo = g;
                if (!h->ws_mem) allocate_own_workspace(h);
                h->err = msg;
            }
            return rc;
        }
        default:
            return fail(h, MOE_EINVAL, "unknown option %d", key);
    }
}

int moe_get_option(moe_handle h, int key, double* value) {
    if (!h || !value) return MOE_EINVAL;
    switch (key) {
        case MOE_OPT_DISPATCH: *value = h->opt_dispatch; return MOE_OK;
        case MOE_OPT_SWIGLU_LIMIT: *value = h->swiglu_limit; return MOE_OK;
        case MOE_OPT_FIXED_SLOT_MAX: *value = h->fixed_slot_max; return MOE_OK;
        case MOE_OPT_DEBUG_CAPTURE: *value = h->debug; return MOE_OK;
        case MOE_OPT_ROUTE_TILE: *value = h->geo.NT; return MOE_OK;
        case MOE_OPT_PROFILE: *value = h->profile; return MOE_OK;
        case MOE_OPT_LAUNCHES: *value = static_cast<double>(h->launches); return MOE_OK;
        case MOE_OPT_PATH: *value = h->opt_path; return MOE_OK;
        case MOE_OPT_W13_LAYOUT: *value = h->opt_w13_layout; return MOE_OK;
        case MOE_OPT_Y_FORMAT: *value = h->y_format; return MOE_OK;
        case MOE_OPT_LAYER_SLOTS: *value = static_cast<double>(h->slots.size()); return MOE_OK;
        case MOE_OPT_LAYER: *value = h->cur; return MOE_OK;
#ifdef MOE_DEBUG_BOUNDS
        case MOE_OPT_BOUNDS_BUILD: *value = 1; return MOE_OK;
#else
        case MOE_OPT_BOUNDS_BUILD: *value = 0; return MOE_OK;
#endif
        default: return fail(h, MOE_EINVAL, "unknown option %d", key);
    }
}

size_t moe_workspace_bytes(moe_handle h) {
    if (!h) return 0;
    return bmoe::workspace_layout(h->geo, nullptr, nullptr);
}

int moe_set_workspace(moe_handle h, void* dev_ptr, size_t bytes) {
    if (!h) return MOE_EINVAL;
    if (h->forwarded) return fail(h, MOE_ESTATE, "set the workspace before the first forward");
    if (!dev_ptr || reinterpret_cast<uintptr_t>(dev_ptr) % 256) return fail(h, MOE_EINVAL, "workspace must be non-NULL and 256-byte aligned");
    int rc = check_device_ptr(h, dev_ptr, "workspace", 256);
    if (rc) return rc;
    return adopt_workspace(h, dev_ptr, bytes, false);
}

int moe_read_status(moe_handle h, uint32_t* flags, moe_stream_t stream) {
    if (!h || !flags) return MOE_EINVAL;
    if (!h->ws_mem) return fail(h, MOE_ENOMEM, "no workspace");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, h->ws.status, sizeof(v), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->ws.status, 0, sizeof(uint32_t), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    // a timed-out fused launch may leave its grid-barrier words mid-count
    if (e == cudaSuccess && (v & MOE_ST_TIMEOUT)) e = cudaMemset(h->ws.ticket + 2, 0, 2 * sizeof(uint32_t));
    // the first-miss record goes with its status bit
    if (e == cudaSuccess && (v & MOE_ST_BOUNDS)) e = cudaMemset(h->ws.ticket + 5, 0, 2 * sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_fail(h, e, "reading the status word");
    *flags = v;
    return MOE_OK;
}

const char* moe_last_error(moe_handle h) {
    return h ? h->err.c_str() : g_create_err.c_str();
}

namespace {

int check_topk_args(moe_ctx* h, const void* logits, int dtype, int T, int E, int K, const void* ids,
                    const void* wts) {
    if (dtype != MOE_DTYPE_F32 && dtype != MOE_DTYPE_BF16) return fail(h, MOE_EINVAL, "bad logits dtype %d", dtype);
    if (T < 0) return fail(h, MOE_EINVAL, "T=%d is negative", T);
    if (E < 1 || E > bmoe::kMaxExperts) return fail(h, MOE_EINVAL, "E=%d outside [1, %d]", E, bmoe::kMaxExperts);
    if (K < 1 || K > bmoe::kMaxTopk || K > E) return fail(h, MOE_EINVAL, "topk=%d outside [1, min(16, E)]", K);
    if (T == 0) return MOE_OK;
    if (!logits || !ids || !wts) return fail(h, MOE_EINVAL, "logits, ids and weights must be non-NULL");
    const uintptr_t a = reinterpret_cast<uintptr_t>(logits);
    if ((dtype == MOE_DTYPE_F32 && (a & 3)) || (a & 1)) return fail(h, MOE_EINVAL, "logits are misaligned for their dtype");
    if ((reinterpret_cast<uintptr_t>(ids) | reinterpret_cast<uintptr_t>(wts)) & 3)
        return fail(h, MOE_EINVAL, "ids and weights must be 4-byte aligned");
    return MOE_OK;
}

}  // namespace

int moe_topk_softmax(const void* logits, int logits_dtype, int T, int E, int topk, const int32_t* num_valid_rows,
                     int renormalize, int32_t* topk_ids, float* topk_weights, moe_stream_t stream) {
    int rc = check_topk_args(nullptr, logits, logits_dtype, T, E, topk, topk_ids, topk_weights);
    if (rc) return rc;
    const cudaError_t e = bmoe::launch_topk_softmax(logits, logits_dtype == MOE_DTYPE_BF16, T, E, topk, num_valid_rows,
                                                    renormalize != 0, topk_ids, topk_weights,
                                                    static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(nullptr, e, "top-k softmax launch");
}

int moe_forward_routed(moe_handle h, const void* x, const void* router_logits, int logits_dtype, int renormalize,
                       const int32_t* num_valid_rows, void* out, int T, moe_stream_t stream) {
    if (!h) return MOE_EINVAL;
    const Geometry& g = h->geo;
    if (T > g.cap) return fail(h, MOE_ECAPACITY, "T=%d exceeds the capacity %d", T, g.cap);
    int rc = check_topk_args(h, router_logits, logits_dtype, T, g.E, g.K, h->ws.rids, h->ws.rw);
    if (rc) return rc;
    if (!h->slots[h->cur].bound) return fail(h, MOE_ENOTBOUND, "no weights bound");
    if (T > 0) {
        const cudaError_t e = bmoe::launch_topk_softmax(router_logits, logits_dtype == MOE_DTYPE_BF16, T, g.E, g.K,
                                                        num_valid_rows, renormalize != 0, h->ws.rids, h->ws.rw,
                                                        static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(h, e, "top-k softmax launch");
        h->launches += 1;
    }
    return moe_forward(h, x, h->ws.rids, h->ws.rw, num_valid_rows, out, T, stream);
}

int moe_last_path(moe_handle h) {
    if (!h) return MOE_EINVAL;
    return h->last_path;
}

int moe_dispatch_scheme(moe_handle h) {
    if (!h) return MOE_EINVAL;
    return h->geo.scheme == 1 ? MOE_DISPATCH_FIXED : MOE_DISPATCH_COMPACT;
}

int moe_profile_read(moe_handle h, float* ms, int n) {
    if (!h || !ms || n < 0) return MOE_EINVAL;
    if (!h->profiled) return fail(h, MOE_ESTATE, "no profiled forward (set MOE_OPT_PROFILE before the forward)");
    cudaError_t e = cudaEventSynchronize(h->ev[MOE_PROFILE_STAGES]);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaEventSynchronize");
    for (int i = 0; i < MOE_PROFILE_STAGES && i < n; ++i) {
        e = cudaEventElapsedTime(&ms[i], h->ev[i], h->ev[i + 1]);
        if (e != cudaSuccess) return cuda_fail(h, e, "cudaEventElapsedTime");
    }
    return MOE_OK;
}

int moe_debug_copy(moe_handle h, int which, void* host_dst, size_t* bytes, moe_stream_t stream) {
    if (!h || !bytes) return MOE_EINVAL;
    const Geometry& g = h->geo;
    const Workspace& w = h->ws;
    const size_t slots = (size_t)h->last_T * g.K;
    const void* src = nullptr;
    size_t n = 0;
    switch (which) {
        case MOE_DBG_COUNTS: src = w.counts; n = sizeof(int32_t) * g.E; break;
        case MOE_DBG_OFFSETS: src = w.rowbase; n = sizeof(int32_t) * (g.E + 1); break;
        case MOE_DBG_PERM: src = w.perm; n = sizeof(int32_t) * slots; break;
        case MOE_DBG_ROUTE_ROW: src = w.route_row; n = sizeof(int32_t) * slots; break;
        case MOE_DBG_ROUTE_SLOT: src = w.route_slot; n = sizeof(int32_t) * slots; break;
        case MOE_DBG_OCC: src = w.occ; n = sizeof(uint32_t) * (size_t)g.E * g.words; break;
        case MOE_DBG_XQ: src = w.xq; n = (size_t)h->last_T * g.H; break;
        case MOE_DBG_XS: src = w.xs; n = (size_t)h->last_T * (g.H / 32); break;
        case MOE_DBG_YROW: src = w.yrow; n = sizeof(int32_t) * slots; break;
        case MOE_DBG_HQ: src = w.hq; n = (size_t)g.rows_cap * g.I; break;
        case MOE_DBG_G: src = w.g; n = (size_t)g.rows_cap * 2 * g.I * sizeof(float); break;
        case MOE_DBG_Y: src = w.y; n = (size_t)g.rows_cap * g.H * 2; break;
        case MOE_DBG_TOPK_IDS: src = w.rids; n = sizeof(int32_t) * (size_t)h->last_T * g.K; break;
        case MOE_DBG_TOPK_WEIGHTS: src = w.rw; n = sizeof(float) * (size_t)h->last_T * g.K; break;
        case MOE_DBG_BOUNDS: src = w.ticket + 5; n = 2 * sizeof(uint32_t); break;
        case MOE_DBG_TILES: {
            std::vector<int32_t> cnt(g.E), rb(g.E + 1), tb(g.E + 1);
            cudaStream_t s = static_cast<cudaStream_t>(stream);
            cudaError_t e = cudaStreamSynchronize(s);
            if (e == cudaSuccess) e = cudaMemcpy(cnt.data(), w.counts, sizeof(int32_t) * g.E, cudaMemcpyDeviceToHost);
            if (e == cudaSuccess) e = cudaMemcpy(rb.data(), w.rowbase, sizeof(int32_t) * (g.E + 1), cudaMemcpyDeviceToHost);
            if (e == cudaSuccess) e = cudaMemcpy(tb.data(), w.tile_base, sizeof(int32_t) * (g.E + 1), cudaMemcpyDeviceToHost);
            if (e != cudaSuccess) return cuda_fail(h, e, "debug copy");
            std::vector<int32_t> v(1 + 3 * (size_t)tb[g.E]);
            v[0] = tb[g.E];
            for (int e2 = 0; e2 < g.E; ++e2)
                for (int j = 0; j < tb[e2 + 1] - tb[e2]; ++j) {
                    const size_t t = tb[e2] + j;
                    v[1 + 3 * t] = e2;
                    v[2 + 3 * t] = rb[e2] + j * g.NT;
                    v[3 + 3 * t] = cnt[e2] - j * g.NT < g.NT ? cnt[e2] - j * g.NT : g.NT;
                }
            n = v.size() * sizeof(int32_t);
            if (host_dst) {
                if (*bytes < n) return fail(h, MOE_EINVAL, "destination holds %zu bytes, %zu needed", *bytes, n);
                memcpy(host_dst, v.data(), n);
            }
            *bytes = n;
            return MOE_OK;
        }
        default: return fail(h, MOE_EINVAL, "unknown debug region %d", which);
    }
    if (!src) return fail(h, MOE_ESTATE, "region %d needs MOE_OPT_DEBUG_CAPTURE", which);
    if (!host_dst) {
        *bytes = n;
        return MOE_OK;
    }
    if (*bytes < n) return fail(h, MOE_EINVAL, "destination holds %zu bytes, %zu needed", *bytes, n);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && n) e = cudaMemcpy(host_dst, src, n, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(h, e, "debug copy");
    *bytes = n;
    return MOE_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ T-bucketed path table
int moe_set_path_table(moe_handle h, const int32_t* t, const int32_t* path, int n) {
    if (!h) return MOE_EINVAL;
    if (n < 0 || n > MOE_TUNE_MAX || (n > 0 && (!t || !path)))
        return fail(h, MOE_EINVAL, "a path table has 0..%d entries and non-NULL arrays", MOE_TUNE_MAX);
    const bool fused_ok = h->coop && bmoe::fused_supported(h->geo);
    for (int i = 0; i < n; ++i) {
        if (t[i] < 1 || t[i] > h->geo.cap || (i > 0 && t[i] <= t[i - 1]))
            return fail(h, MOE_EINVAL, "bucket T values must ascend strictly within [1, capacity=%d]", h->geo.cap);
        if (path[i] != MOE_PATH_FUSED && path[i] != MOE_PATH_MULTI)
            return fail(h, MOE_EINVAL, "entry %d: path %d is neither MOE_PATH_FUSED nor MOE_PATH_MULTI", i, path[i]);
        if (path[i] == MOE_PATH_FUSED && !fused_ok)
            return fail(h, MOE_EINVAL, "entry %d: this handle cannot run the fused path", i);
    }
    h->tune_t.assign(t, t + n);
    h->tune_path.assign(path, path + n);
    return MOE_OK;
}

int moe_get_path_table(moe_handle h, int32_t* t, int32_t* path, int cap) {
    if (!h || cap < 0) return MOE_EINVAL;
    const int n = static_cast<int>(h->tune_t.size());
    for (int i = 0; i < n && i < cap; ++i) {
        if (t) t[i] = h->tune_t[i];
        if (path) path[i] = h->tune_path[i];
    }
    return n;
}

int moe_autotune(moe_handle h, const int32_t* t_buckets, int n, int reps, moe_stream_t stream) {
    if (!h) return MOE_EINVAL;
    if (n < 1 || n > MOE_TUNE_MAX || !t_buckets || reps < 1)
        return fail(h, MOE_EINVAL, "autotune takes 1..%d bucket T values and reps >= 1", MOE_TUNE_MAX);
    const Geometry& g = h->geo;
    for (int i = 0; i < n; ++i)
        if (t_buckets[i] < 1 || t_buckets[i] > g.cap || (i > 0 && t_buckets[i] <= t_buckets[i - 1]))
            return fail(h, MOE_EINVAL, "bucket T values must ascend strictly within [1, capacity=%d]", g.cap);
    if (!h->slots[h->cur].bound) return fail(h, MOE_ENOTBOUND, "no weights bound");
    const bool fused_ok = h->coop && bmoe::fused_supported(g);
    std::vector<int32_t> paths(n, MOE_PATH_MULTI);
    if (!fused_ok) return moe_set_path_table(h, t_buckets, paths.data(), n);

    // Synthetic inputs of the largest bucket: BF16 rows from a fixed linear congruential sequence,
    // K distinct experts per row, equal weights.  A 256 MiB buffer is written before every timed
    // forward so that the weights stream from HBM as they do in a real step.
    const int T = t_buckets[n - 1], K = g.K, E = g.E, H = g.H;
    std::vector<uint16_t> hx((size_t)T * H);
    std::vector<int32_t> hid((size_t)T * K);
    std::vector<float> hw((size_t)T * K, 1.0f / K);
    uint32_t st = 12345u;
    auto next = [&st]() { st = st * 1664525u + 1013904223u; return st; };
    for (auto& v : hx) {
        const float f = (static_cast<int>(next() >> 9) - (1 << 22)) / static_cast<float>(1 << 22);
        uint32_t b;
        std::memcpy(&b, &f, 4);
        v = static_cast<uint16_t>(b >> 16);
    }
    for (int t = 0; t < T; ++t) {
        const int base = static_cast<int>(next() % E), step = 1 + static_cast<int>(next() % std::max(1, E - 1));
        for (int k = 0; k < K; ++k) hid[(size_t)t * K + k] = (base + k * step) % E;
        // (distinct unless step shares a factor with E; a repeated id is a valid input too)
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *dx = nullptr, *did = nullptr, *dw = nullptr, *dout = nullptr, *dflush = nullptr;
    const size_t flush_bytes = 256u << 20;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    int rc = MOE_OK;
    const int saved_path = h->opt_path;
    auto cleanup = [&]() {
        h->opt_path = saved_path;
        cudaFree(dx);
        cudaFree(did);
        cudaFree(dw);
        cudaFree(dout);
        cudaFree(dflush);
        if (e0) cudaEventDestroy(e0);
        if (e1) cudaEventDestroy(e1);
    };
    cudaError_t e = cudaMalloc(&dx, hx.size() * 2);
    if (e == cudaSuccess) e = cudaMalloc(&did, hid.size() * 4);
    if (e == cudaSuccess) e = cudaMalloc(&dw, hw.size() * 4);
    if (e == cudaSuccess) e = cudaMalloc(&dout, hx.size() * 2);
    if (e == cudaSuccess) e = cudaMalloc(&dflush, flush_bytes);
    if (e == cudaSuccess) e = cudaEventCreate(&e0);
    if (e == cudaSuccess) e = cudaEventCreate(&e1);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dx, hx.data(), hx.size() * 2, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(did, hid.data(), hid.size() * 4, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dw, hw.data(), hw.size() * 4, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) {
        cleanup();
        return cuda_fail(h, e, "autotune setup");
    }
    for (int i = 0; i < n && rc == MOE_OK; ++i) {
        float best = 0.f;
        for (int p : {MOE_PATH_FUSED, MOE_PATH_MULTI}) {
            h->opt_path = p;
            float total = 0.f;
            for (int r = -1; r < reps && rc == MOE_OK; ++r) {  // r = -1: untimed warm-up
                e = cudaMemsetAsync(dflush, r & 0xff, flush_bytes, s);
                if (e == cudaSuccess) e = cudaEventRecord(e0, s);
                if (e != cudaSuccess) break;
                rc = moe_forward(h, dx, static_cast<const int32_t*>(did), static_cast<const float*>(dw), nullptr, dout,
                                 t_buckets[i], stream);
                if (rc != MOE_OK) break;
                e = cudaEventRecord(e1, s);
                if (e == cudaSuccess) e = cudaEventSynchronize(e1);
                float ms = 0.f;
                if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
                if (e != cudaSuccess) break;
                if (r >= 0) total += ms;
            }
            if (e != cudaSuccess && rc == MOE_OK) rc = cuda_fail(h, e, "autotune timing");
            if (rc != MOE_OK) break;
            if (p == MOE_PATH_FUSED || total < best) {
                best = total;
                paths[i] = p;
            }
        }
    }
    cleanup();
    if (rc != MOE_OK) return rc;
    return moe_set_path_table(h, t_buckets, paths.data(), n);
}


/*
 * blockmoe.h -- C ABI of the fused block-scaled mixture-of-experts layer for
 * one NVIDIA GB300 (sm_103a).
 *
 * The layer (ROCm/aiter PR #6881 "[FlyDSL] MegaMoEV2: fuse Dispatch, GEMM1,
 * GEMM2 and Combine into one kernel", Title and Technical Details; ROCm/aiter
 * PR #6154 "Add full-expert DeepSeek V4.1 Flash MegaMoE tuning for gfx950",
 * Summary), per token row t < num_valid_rows:
 *   1. quantise the BF16 row to MXFP8: E4M3 codes, one E8M0 scale per 32
 *      elements along H;
 *   2. dispatch the row to each valid top-k expert (fixed-slot or compact
 *      scheme, vLLM PR #61262 (a second, fixed-slot MegaMoEV2 runtime));
 *   3. GEMM1 against the expert's MXFP4 W13 [2I,H] (E2M1 codes, one E8M0 scale
 *      per 32 along H), SwiGLU epilogue (optional clamp), MXFP8 1x32
 *      re-quantisation of the I intermediate values;
 *   4. GEMM2 against the expert's MXFP4 W2 [H,I], rounded to BF16 per route;
 *   5. combine: out[t] = BF16( sum over valid slots k, ascending, of
 *      w[t,k] * y[t,k] ) accumulated in float and rounded once (ROCm/ATOM PR
 *      #2725 "route before the rows move; per-pass real row counts", note on
 *      the mono MoE sum).
 *
 * Conventions shared by every entry point
 *   - Every data pointer is a CUDA device pointer to contiguous row-major
 *     memory unless stated otherwise; the library never copies, frees or
 *     keeps ownership of caller memory.
 *   - Return value 0 is success; a negative MOE_E* code is an error and
 *     moe_last_error() then describes it.  Nothing is thrown across the ABI.
 *     A refused call changes no state of the handle.
 *   - The library targets sm_103a only; moe_create refuses other devices.
 *   - Entry points are not thread-safe on one handle; distinct handles are
 *     independent.
 */
#ifndef BLOCKMOE_H
#define BLOCKMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_ctx* moe_handle;
/* A cudaStream_t; 0 is the legacy default stream (ROCm/aiter PR #6881, commit
 * note on bindings: a null stream handle runs on the default stream, never on
 * a newly created stream). */
typedef void* moe_stream_t;

/* ---------------------------------------------------------------- errors */
#define MOE_OK 0
#define MOE_EINVAL (-1)      /* bad argument (null pointer, bad size, bad option) */
#define MOE_ENOTBOUND (-2)   /* moe_forward before moe_bind_weights */
#define MOE_ESHAPE (-3)      /* H, I, E or topk not supported by the kernels */
#define MOE_ECAPACITY (-4)   /* T larger than the capacity given to moe_create */
#define MOE_ECUDA (-5)       /* a CUDA runtime or driver call failed */
#define MOE_EDEVICE (-6)     /* current device is not an sm_103 GB300 */
#define MOE_ENOMEM (-7)      /* workspace allocation failed or too small */
#define MOE_ESTATE (-8)      /* call not allowed in the handle's state */

/* ------------------------------------------------------ device status bits
 * Written by the kernels into a device word, read with moe_read_status. */
#define MOE_ST_BAD_ID 0x1u      /* a top-k id >= E was seen (skipped like -1) */
#define MOE_ST_TIMEOUT 0x2u     /* a bounded device-side wait gave up */
#define MOE_ST_OVERFLOW 0x4u    /* internal tile list overflow (bug guard) */
#define MOE_ST_BOUNDS 0x8u      /* bounds-checking build: a kernel computed an index outside its region
                                   (the access was skipped; MOE_DBG_BOUNDS holds the first one) */
/* With MOE_ST_TIMEOUT, bits 8..15 name the wait that gave up (diagnostic):
 * 8 producer/stage-free, 9 producer drain, 10 MMA/accumulator-free,
 * 11 MMA/stage-full, 12 MMA drain, 13 epilogue/accumulator-full,
 * 14 fused path grid barrier, 15 fused path GEMM1->GEMM2 readiness.
 * Reading a timeout also resets the fused path's grid-barrier words. */

/* ------------------------------------------------------------- options */
#define MOE_OPT_DISPATCH 1        /* MOE_DISPATCH_* */
#define MOE_OPT_SWIGLU_LIMIT 2    /* clamp L >= 0; 0 = plain SwiGLU (aiter #6154 "clamp-10 SwiGLU") */
#define MOE_OPT_FIXED_SLOT_MAX 3  /* fixed-slot threshold on capacity, default 255
                                     (vLLM PR #61262: FIXED_SLOT_MAX_MTPR) */
#define MOE_OPT_DEBUG_CAPTURE 4   /* 1 = also keep canonical MXFP8 codes of x and raw GEMM1 outputs */
#define MOE_OPT_ROUTE_TILE 5      /* route-tile width NT in {0 (auto: 32 decode, 144 prefill), 32, 128, 144} */
#define MOE_OPT_PROFILE 6         /* 1 = bracket each stage of every forward with CUDA events
                                     (eager use only: keep 0 while capturing a CUDA graph) */
#define MOE_OPT_LAUNCHES 7        /* read-only: CUDA kernels this handle has launched so far */
#define MOE_OPT_PATH 8            /* MOE_PATH_*: which kernels a forward runs */

/* MOE_PATH_AUTO runs the single-launch fused kernel (ROCm/aiter PR #6881,
 * MegaMoEV2 small-input fusion, "Technical Details": for inputs of at most 512
 * tokens every step of the layer happens inside one kernel launch) when the
 * handle allows it: capacity <= 512, route tile 32, E <= 512, and a device
 * that supports cooperative launches; otherwise it runs the multi-kernel path.
 * If the driver refuses the cooperative launch because the grid (one CTA per
 * SM) cannot be co-resident, AUTO takes the multi-kernel path for that forward
 * and every later one on the handle.
 * MOE_PATH_FUSED insists on the fused kernel (setting it is refused when the
 * handle does not allow it, and a refused launch is returned as an error);
 * MOE_PATH_MULTI always runs the separate kernels.  Both paths produce the same
 * bits. */
#define MOE_PATH_AUTO 0
#define MOE_PATH_FUSED 1
#define MOE_PATH_MULTI 2

#define MOE_OPT_W13_LAYOUT 9      /* MOE_W13_*: row order of W13 assumed by the next bind */
#define MOE_OPT_LAYER_SLOTS 10    /* number of layer slots (>= 1, default 1); see moe_bind_layer */
#define MOE_OPT_LAYER 11          /* read-only: the current layer slot */
#define MOE_OPT_Y_FORMAT 12       /* MOE_Y_*: GEMM2 rows handed to the combine */
#define MOE_OPT_DEBUG_GRID_GEN 13 /* test-only, write-only: preset the single-launch kernel's grid-barrier
                                     generation word to a value in [0, 2^32) (the pages test epoch words
                                     preset a few counts short of 2^31 and 2^32; aiter #6881 commit notes).  The
                                     barrier compares the word for a change, so it may wrap.  Synchronous. */
#define MOE_OPT_DEBUG_STALL_GRID 14 /* test-only, write-only, fault injection without a fault: 1 presets the
                                     single-launch kernel's grid-barrier arrival count to 2^31, so that the
                                     next fused forward's first grid barrier can never complete.  Every CTA
                                     gives up after its bounded wait (2 s), sets MOE_ST_TIMEOUT with the
                                     grid-barrier site bit (14) and ends; `out` is not written.  Reading
                                     that status resets the words and the handle works again.  Other paths
                                     do not use the word.  Synchronous. */
#define MOE_OPT_DEBUG_BOUNDS_ROWS 15 /* test-only, write-only, bounds-checking builds only (MOE_ESTATE
                                     otherwise): the packed-row count the kernels check row indices
                                     against, 1 .. the workspace's rows (default).  A smaller value
                                     makes legitimate rows count as misses, which the kernels skip and
                                     record: it shows that the checks run.  Results are then wrong. */
#define MOE_OPT_BOUNDS_BUILD 16   /* read-only: 1 in the bounds-checking build (-DMOE_DEBUG_BOUNDS,
                                     libblockmoe_bounds.so), else 0 */

/* GEMM2 rows.  BF16: one BF16 row per route (default).  MXFP8: the rows go to
 * the combine as 1x32 E4M3 codes with one E8M0 scale per 32 along H (ROCm/aiter
 * PR #6881, Technical Details, small-input path: GEMM2 rows in the main path's
 * 1x32 FP8 format instead of BF16), quantised from the float accumulator with
 * the rule of the input rows and dequantised exactly by the combine.  Takes
 * effect at the next forward; a captured graph keeps the format of capture.
 * MOE_DBG_Y then holds the codes [rows][H] followed by the scales [rows][H/32]. */
#define MOE_Y_BF16 0
#define MOE_Y_MXFP8 1

/* W13 row order.  CONCAT: rows [0,I) gate, rows [I,2I) up.  INTERLEAVED
 * (the gate-up-interleaved experts of the mega_moe reference in ROCm/aiter
 * PR #6881's linked AKLR commit): row 2j is gate row j and row 2j+1 up row j;
 * the reading that gate and up alternate row by row is ours (the pages name
 * the layout without defining its granularity).  Codes and scales follow the
 * same order.  Both layouts give the same bits. */
#define MOE_W13_CONCAT 0
#define MOE_W13_INTERLEAVED 1

#define MOE_DISPATCH_AUTO 0       /* fixed-slot iff capacity <= fixed-slot max */
#define MOE_DISPATCH_FIXED 1
#define MOE_DISPATCH_COMPACT 2

/* --------------------------------------------------------- entry points */

/* Create a layer instance for H (hidden), I (expert intermediate), E experts,
 * top-k = topk, and at most `capacity` token rows per forward (the runtime's
 * max tokens per rank, vLLM PR #61262).  Requirements: H and I multiples of
 * 128 (MMA K-stage and 1x32 scale blocks), 1 <= topk <= 16, 1 <= E <= 4096,
 * 1 <= capacity.  Allocates the device workspace with cudaMalloc on the
 * current device unless moe_set_workspace is used before the first forward.
 * On success *out receives the handle; on error *out is NULL. */
int moe_create(moe_handle* out, int H, int I, int E, int topk, int capacity);

/* Bind expert weights without copying (ROCm/aiter PR #6154, Changes and
 * tuning: one shared workspace takes each layer's prepared weights in place)
 * into the current layer slot:
 *   w13_fp4 u8 [E, 2I, H/2]  E2M1 codes, element 2j in the low nibble of byte j;
 *                            row order per MOE_OPT_W13_LAYOUT (default: rows
 *                            [0,I) gate, rows [I,2I) up)
 *   w13_sf  u8 [E, 2I, H/32] E8M0 scales (uint8 or float8_e8m0fnu bytes)
 *   w2_fp4  u8 [E, H, I/2]
 *   w2_sf   u8 [E, H, I/32]
 * The caller keeps ownership; the memory must outlive the binding and every
 * CUDA graph that captured a forward using it.  Everything is validated
 * before any state changes, so a refused bind leaves the previous binding
 * intact (aiter #6881, commit notes: every check that can refuse runs before a
 * binding changes).  Rebinding is allowed between forwards. */
int moe_bind_weights(moe_handle h, const void* w13_fp4, const void* w13_sf,
                     const void* w2_fp4, const void* w2_sf);

/* Layer slots (ROCm/aiter PR #6881, commit notes on LargeMRuntime.bind_layer:
 * each MoE layer has its own slot on one shared operator; the slot is checked
 * first, then the weights, and only then does the current slot switch).
 * moe_bind_layer binds the weights (as moe_bind_weights) into `slot`, in
 * [0, MOE_OPT_LAYER_SLOTS), and makes it current; MOE_EINVAL for a bad slot,
 * and a refusal leaves both the slot and the current slot unchanged.
 * moe_select_layer makes an already bound slot current without rebuilding its
 * tensor maps (MOE_ENOTBOUND if the slot is empty).  Forwards use the current
 * slot's weights; a captured CUDA graph keeps the slot that was current at
 * capture.  Slots share the handle's workspace, so forwards of different
 * layers on one handle must be stream-ordered. */
int moe_bind_layer(moe_handle h, int slot, const void* w13_fp4, const void* w13_sf,
                   const void* w2_fp4, const void* w2_sf);
int moe_select_layer(moe_handle h, int slot);

/* One forward on `stream`:
 *   x              bf16 [T, H]
 *   topk_ids       int32 [T, topk]; -1 (or any id outside [0,E)) marks an
 *                  invalid slot that claims no slot and adds nothing (ROCm/ATOM
 *                  PR #2725 linked fix: a negative id takes no slot); ids >= E
 *                  also set MOE_ST_BAD_ID
 *   topk_weights   float32 [T, topk]
 *   num_valid_rows device int32, first element = rows to compute, clamped to
 *                  [0,T]; NULL means T.  Read on the device, so a replayed CUDA
 *                  graph follows the value at replay time (ATOM #2725,
 *                  "Per-pass real row counts").  Rows at or past it give +0.
 *   out            bf16 [T, H]; every row is written (T = 0 writes nothing)
 * No host synchronisation, no allocation; enqueues only on `stream`, so the
 * call can be captured in a CUDA graph.  Forwards on one handle share its
 * workspace: issue them on one stream (or order them with events).  Returns MOE_ECAPACITY if T exceeds
 * the capacity, MOE_ENOTBOUND without weights. */
int moe_forward(moe_handle h, const void* x, const int32_t* topk_ids, const float* topk_weights,
                const int32_t* num_valid_rows, void* out, int T, moe_stream_t stream);

/* Release the handle and the workspace it allocated (not caller memory). */
void moe_destroy(moe_handle h);

/* ------------------------------------------------------ supporting calls */

/* Set an option (MOE_OPT_*) before the first forward; MOE_ESTATE afterwards
 * for options that change the workspace layout (dispatch, route tile). */
int moe_set_option(moe_handle h, int key, double value);
int moe_get_option(moe_handle h, int key, double* value);

/* Bytes of device workspace the handle needs with its current options. */
size_t moe_workspace_bytes(moe_handle h);

/* Use caller memory (e.g. from the torch caching allocator) as workspace
 * instead of the library's own allocation.  dev_ptr must be 256-byte aligned
 * and hold moe_workspace_bytes(h) bytes; the caller keeps ownership and must
 * keep it alive while the handle uses it. */
int moe_set_workspace(moe_handle h, void* dev_ptr, size_t bytes);

/* Read and clear the device status word (MOE_ST_* bits).  Synchronises
 * `stream`; never called implicitly by moe_forward. */
int moe_read_status(moe_handle h, uint32_t* flags, moe_stream_t stream);

/* Text of the last error on this handle (or, when h is NULL, of the last
 * failed call on this thread that had no handle: moe_create,
 * moe_dispatch_compact_noalloc).  Valid until the next call on the same handle. */
const char* moe_last_error(moe_handle h);

/* Which dispatch scheme the handle runs: MOE_DISPATCH_FIXED or _COMPACT. */
int moe_dispatch_scheme(moe_handle h);

/* Path the last forward took: MOE_PATH_FUSED or MOE_PATH_MULTI (0 before any forward). */
int moe_last_path(moe_handle h);

/* ------------------------------------------------ T-bucketed path table
 * ROCm/aiter PR #6154, "Changes and tuning": a measured configuration table per
 * source-token bucket M, an arbitrary M taking the nearest bucket with ties to
 * the larger.  Here the per-T choice is the path (the dispatch scheme and the
 * route tile follow the handle's capacity).  With a non-empty table, a forward
 * under MOE_PATH_AUTO takes the path of the bucket nearest to T (ties: the
 * larger bucket); with an empty one (the default) it takes the fused kernel for
 * T <= 512 whenever the handle allows it.  MOE_PATH_FUSED / MOE_PATH_MULTI set
 * by moe_set_option still override the table. */
#define MOE_TUNE_MAX 64
/* Replace the table: n (0..MOE_TUNE_MAX) buckets, t strictly ascending in
 * [1, capacity], path MOE_PATH_FUSED or MOE_PATH_MULTI (FUSED only where the
 * handle allows it).  n = 0 clears it.  Refused tables change nothing. */
int moe_set_path_table(moe_handle h, const int32_t* t, const int32_t* path, int n);
/* Copy up to `cap` entries into t / path (either may be NULL); returns the
 * number of entries (or a negative error). */
int moe_get_path_table(moe_handle h, int32_t* t, int32_t* path, int cap);
/* Measure each path the handle allows for every bucket T (strictly ascending
 * in [1, capacity], n <= MOE_TUNE_MAX) on synthetic inputs and the bound
 * weights: `reps` timed forwards after one warm-up, a 256 MiB buffer written
 * before each so the weights come from HBM; record the faster path per bucket as
 * the table.  Allocates its inputs (device memory for the largest T and the
 * 256 MiB buffer), synchronises `stream`, and is not capturable: run it once
 * after binding.  MOE_ENOTBOUND without weights. */
int moe_autotune(moe_handle h, const int32_t* t_buckets, int n, int reps, moe_stream_t stream);

/* ------------------------------------------------ router top-k in front of dispatch */
#define MOE_DTYPE_F32 0
#define MOE_DTYPE_BF16 1

/* Router top-k with softmax weights (ROCm/ATOM PR #2725, linked commits on
 * the Triton softmax top-k routing that follows the device row count):
 *   router_logits  [T, E] float32 or bf16 (logits_dtype), device memory
 *   num_valid_rows device int32 (first element) or NULL (= T); rows at or
 *                  past it get ids -1 and weights 0 (read on the device, so a
 *                  replayed CUDA graph follows the value at replay)
 *   topk_ids       out int32 [T, topk]; topk_weights out float32 [T, topk]
 * Per row: pick topk times the expert with the largest remaining logit (ties:
 * lowest id) and clear it to -inf, so a row with fewer finite logits than topk
 * picks expert 0 again with weight 0; weight = exp(logit - row max) divided by
 * the sum over the picked experts (renormalize != 0) or over the whole row.  A
 * row of -inf logits gets NaN weights.  1 <= E <= 4096, 1 <= topk <= min(16, E).
 * One kernel launch on `stream`; errors are readable with moe_last_error(NULL). */
int moe_topk_softmax(const void* router_logits, int logits_dtype, int T, int E, int topk,
                     const int32_t* num_valid_rows, int renormalize, int32_t* topk_ids,
                     float* topk_weights, moe_stream_t stream);

/* moe_topk_softmax into the handle's workspace (E and topk of the handle),
 * then moe_forward with those ids and weights: the router output feeds the
 * dispatch directly, with no buffer of the caller's in between.  Same
 * arguments, errors and stream semantics as the two calls; the ids and weights
 * of the last call are readable with MOE_DBG_TOPK_IDS / MOE_DBG_TOPK_WEIGHTS. */
int moe_forward_routed(moe_handle h, const void* x, const void* router_logits, int logits_dtype,
                       int renormalize, const int32_t* num_valid_rows, void* out, int T,
                       moe_stream_t stream);

/* Stage times in milliseconds of the last forward run with MOE_OPT_PROFILE=1,
 * measured by CUDA events recorded on the forward's stream:
 *   ms[0] dispatch, ms[1] quantisation + scatter, ms[2] GEMM1, ms[3] GEMM2,
 *   ms[4] combine.  A forward on the fused path reports its single kernel in
 *   ms[2] and 0 elsewhere.  Waits for the last event; n = entries ms can hold (<= 5
 * written).  MOE_ESTATE if profiling is off or no profiled forward ran. */
#define MOE_PROFILE_STAGES 5
int moe_profile_read(moe_handle h, float* ms, int n);

/* ------------------------------------------- allocation-free dispatch
 * The pages have no counterpart of this call; it serves callers that may not
 * allocate device memory: code running while a CUDA graph is captured (where
 * cudaMalloc is not allowed) and serving engines that reserve the whole GPU up
 * front and forbid later allocations.  It runs the compact dispatch of
 * moe_forward on its own, with the same results (counts, offsets = exclusive
 * scan of counts with E+1 entries, perm, route_row; see MOE_DBG_* below for
 * their layouts), and allocates nothing: its scratch is a 1 MiB array built
 * into the library (every GPU that loads the library keeps it until the
 * process exits), so it accepts only sizes that need at most
 * 256 + 4 * (ceil(T*topk/512) * E + E + 1) bytes of scratch within 1 MiB, and
 * refuses larger ones with MOE_ECAPACITY.  All calls share that array, so calls that overlap on the GPU
 * (other streams, other threads) race and must be serialised by the caller.
 * The first call on a device looks up the array's device address; make that
 * first call before any stream capture.  Outputs: counts int32 [E],
 * offsets int32 [E+1], perm int32 [T*topk] (first offsets[E] entries
 * written), route_row int32 [T*topk]; all device memory of the caller.
 * num_valid_rows as in moe_forward.  Ids outside [0, E) claim no slot, as in
 * moe_forward, but this call reports nothing about ids >= E (it has no status
 * word a caller can read).  The first call on a device also sets the dispatch
 * kernel's shared-memory limit there.  Errors: moe_last_error(NULL). */
int moe_dispatch_compact_noalloc(const int32_t* topk_ids, int T, int topk, int E, const int32_t* num_valid_rows,
                                 int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* route_row,
                                 moe_stream_t stream);

/* ------------------------------------------- test-only introspection
 * Copies one internal array of the last forward into host memory
 * (synchronises `stream`).  `which` is a MOE_DBG_* id; *bytes receives the
 * region size when host_dst is NULL.  The layouts are those documented next
 * to each id; they exist so that tests can compare the dispatch and the MXFP8
 * codes bit-exactly with an independent implementation. */
#define MOE_DBG_COUNTS 1        /* int32 [E]: routes (compact) / occupied slots (fixed) per expert */
#define MOE_DBG_OFFSETS 2       /* int32 [E+1]: compact exclusive scan of counts */
#define MOE_DBG_PERM 3          /* int32 [T*topk]: compact packed position -> flat slot t*topk+k */
#define MOE_DBG_ROUTE_ROW 4     /* int32 [T*topk]: compact slot -> packed position, -1 invalid */
#define MOE_DBG_ROUTE_SLOT 5    /* int32 [T*topk]: fixed slot -> e*capacity+t, -1 invalid */
#define MOE_DBG_OCC 6           /* uint32 [E][ceil(capacity/32)]: fixed-slot occupancy bits */
#define MOE_DBG_XQ 7            /* uint8 [T][H]: canonical E4M3 codes of x, rows < num_valid_rows (needs DEBUG_CAPTURE) */
#define MOE_DBG_XS 8            /* uint8 [T][H/32]: canonical E8M0 scales of x, rows < num_valid_rows (needs DEBUG_CAPTURE) */
#define MOE_DBG_YROW 9          /* int32 [T*topk]: row of the GEMM2 output each slot combines, -1 invalid */
#define MOE_DBG_HQ 10           /* uint8 [rows][I]: E4M3 codes of h per packed row */
#define MOE_DBG_G 11            /* float [rows][2I]: raw GEMM1 outputs (needs DEBUG_CAPTURE) */
#define MOE_DBG_Y 12            /* bf16 [rows][H]: GEMM2 outputs per packed row */
#define MOE_DBG_TILES 13        /* int32 [1 + 3*tiles]: tile count, then (expert, row0, n) per tile */
#define MOE_DBG_TOPK_IDS 14     /* int32 [T][topk]: router ids of the last moe_forward_routed */
#define MOE_DBG_TOPK_WEIGHTS 15 /* float [T][topk]: router weights of the last moe_forward_routed */
#define MOE_DBG_BOUNDS 16       /* uint32 [2]: site (1 occupancy word, 2 top-k slot, 3 packed position,
                                   4 dispatch chunk, 5 scattered row, 6 scale atom, 7 combined row,
                                   8 GEMM unit) and low 32 bits of the index of the first bounds miss;
                                   zeros if none.  moe_read_status clears it with MOE_ST_BOUNDS. */
int moe_debug_copy(moe_handle h, int which, void* host_dst, size_t* bytes, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* BLOCKMOE_H */

/*
 * lora_linear.h -- shared-base, per-request LoRA projection on one GB300 (sm_103a).
 *
 * For a batch of token rows grouped into request segments, one call computes
 *
 *     Y[t,:] = X[t,:] W^T + s_a (X[t,:] A_a^T) B_a^T    rows of a segment naming adapter a >= 1
 *     Y[t,:] = X[t,:] W^T                              rows of a segment naming no adapter (0)
 *
 * Source: "Two 27B models on a single RTX 5090", section 3 (each changed matrix of the
 * fine-tuned model equals the base matrix plus B.A, rank 256) and section 4 (a request
 * that names the adapter runs the adapter's two thin matrices beside each changed matrix
 * and adds their output; every other request in the same batch uses the base weights).
 *
 * Layouts (all row-major, bf16 = IEEE binary32 upper half, little endian):
 *   X   [T, d_in]        W   [d_out, d_in]  (nn.Linear layout: row n is output feature n)
 *   A_a [rank, d_in]     B_a [d_out, rank]  Y   [T, d_out]
 * Arithmetic: bf16 operands, fp32 accumulation on the tensor cores. The shrink output
 * U = s_a X A_a^T is rounded to bf16 (round to nearest even) before the expand; Y is
 * rounded from fp32 to bf16 (round to nearest even). The summation order is not
 * specified, so results are not bitwise equal to any other implementation; on one handle a
 * row's output does not depend on the other rows of its batch (the same bits in any batch,
 * launch shape or host-buffer chunking). A handle may sum the base product in parts of K
 * (LORA_OPT_K_SPLIT); it decides that once, at create, from its shape and max_tokens, so two
 * handles of one shape but different max_tokens may differ in the last bit.
 *
 * Errors: every function returns LORA_OK (0) or a negative code below. Argument checks
 * run on the host before any launch; a failed check launches nothing and leaves every
 * output buffer untouched. The library never prints, never aborts the process and never
 * falls back to another implementation.
 */
#ifndef LORA_LINEAR_H
#define LORA_LINEAR_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct lora_linear lora_linear; /* opaque handle */

enum {
    LORA_OK = 0,
    LORA_EINVAL = -1,       /* bad argument (sizes, segments, ids, pointers, alignment, aliasing) */
    LORA_ENOMEM = -2,       /* a device or pinned-host allocation failed in lora_linear_create */
    LORA_ECUDA = -3,        /* a CUDA runtime/driver call failed */
    LORA_ETIMEOUT = -4,     /* a kernel's bounded wait ran out (read by lora_linear_status) */
    LORA_EUNSUPPORTED = -5, /* valid request this library does not run (e.g. a capture of a call whose work list is uploaded) */
    LORA_ENODEV = -6        /* the device is not an sm_103 GPU or cannot be used */
};

/* Limits of this library. */
#define LORA_MAX_RANK 256   /* adapter rank: the shrink writes at most one 256-column tile */
#define LORA_TILE_ROWS 128  /* rows per tile of the planner (the tensor-core tile height) */
#define LORA_MAX_FEATURES (1 << 20)  /* d_in, d_out */
#define LORA_MAX_TOKENS (1 << 24)    /* max_tokens: keeps every row and tile count in int range */
#define LORA_MAX_SEGMENTS (1 << 20)  /* max_segments */

/*
 * lora_linear_create -- make a handle for one projection shape on one device.
 *   out          receives the handle (set to NULL on failure).
 *   d_in, d_out  input / output features; each a multiple of 8 (16-byte rows) in
 *                [8, LORA_MAX_FEATURES].
 *   rank         adapter rank r, a multiple of 8 in [8, LORA_MAX_RANK].
 *   max_tokens   largest T a forward call will pass, in [1, LORA_MAX_TOKENS].
 *   max_segments largest n_seg a forward call will pass, in [1, LORA_MAX_SEGMENTS].
 *   device       CUDA device ordinal; it must be an sm_103 GPU.
 * The handle owns its workspace: the shrink output U (bf16 [max_tokens + 128, rank]),
 * a ring of work-list buffers (device and pinned host), a device status word and CUDA
 * events. The caller keeps the current device unchanged across the call.
 * Returns LORA_OK, LORA_EINVAL, LORA_ENODEV, LORA_ENOMEM or LORA_ECUDA.
 * Source: the shapes of "Two 27B models on a single RTX 5090", sections 2-3 (hidden
 * size 5,120, rank 256).
 */
int lora_linear_create(lora_linear** out, int d_in, int d_out, int rank,
                       int max_tokens, int max_segments, int device);

/*
 * lora_linear_forward -- Y for one batch, enqueued on `stream`; returns without waiting.
 *   x               device bf16 [T, d_in], 16-byte aligned.
 *   T               rows (0 <= T <= max_tokens). T = 0 returns LORA_OK and launches nothing.
 *   seg_offsets     HOST int32 [n_seg + 1]: seg_offsets[0] = 0, seg_offsets[n_seg] = T,
 *                   nondecreasing. Segment i is rows [seg_offsets[i], seg_offsets[i+1]),
 *                   one request; empty segments are allowed.
 *   seg_adapter_ids HOST int32 [n_seg]: 0 = no adapter, k >= 1 = adapter k (A[k-1], ...).
 *   n_seg           1 <= n_seg <= max_segments (0 allowed only when T = 0).
 *   W               device bf16 [d_out, d_in], 16-byte aligned.
 *   A, B            HOST arrays [n_adapters] of device pointers: A[k] bf16 [rank, d_in],
 *                   B[k] bf16 [d_out, rank], each 16-byte aligned. Only adapters named
 *                   by a segment are read; the others may be NULL.
 *   scale           HOST float [n_adapters]: s for each adapter (finite).
 *   n_adapters      >= 0; every id must be <= n_adapters.
 *   y               device bf16 [T, d_out], 16-byte aligned; fully overwritten. It must
 *                   not overlap x, W or any named A/B.
 *   stream          a cudaStream_t (NULL = the legacy default stream).
 * Host arrays are read before the call returns. Device buffers must stay valid until
 * the stream reaches the end of the call. Calls on one handle must be ordered on one
 * stream (they share the handle's workspace); the handle is not thread-safe.
 * Returns LORA_OK, LORA_EINVAL (nothing launched) or LORA_ECUDA. A bounded wait that
 * ran out inside a kernel is reported later by lora_linear_status.
 * CUDA graphs: a call may be recorded by stream capture when its work list travels in the
 * kernel parameters (at most 64 row tiles over both passes, SM-pair padding included, 48
 * merged segments and 4 named adapters; a 2,048-row batch of a few requests fits); a larger
 * call returns LORA_EUNSUPPORTED while the stream is capturing and records nothing. Each launch
 * leaves the handle's workspace as it found it, so a graph can be replayed any number of
 * times (the host arrays are read at capture; device buffers are read at every replay).
 * Make one call of the same shape before capturing: it caches the launch shape.
 * A call with adapter rows runs its shrink and fused passes in one cooperative launch, which
 * starts only when its whole grid can be resident, so calls on different handles and streams
 * may run side by side; profilers that reject cooperative launches can set
 * LORA_LINEAR_NONCOOPERATIVE=1 in the environment (they run one kernel at a time).
 * Source: "Two 27B models on a single RTX 5090", section 4 (per-request adapter in a
 * shared batch) and section 3 (W + B.A).
 */
int lora_linear_forward(lora_linear* h, const void* x, int T,
                        const int32_t* seg_offsets, const int32_t* seg_adapter_ids, int n_seg,
                        const void* W, const void* const* A, const void* const* B,
                        const float* scale, int n_adapters, void* y, void* stream);

/*
 * lora_linear_forward_host -- the same projection from and to HOST memory.
 *   x_host [T, d_in] and y_host [T, d_out] are host bf16 buffers (pinned memory gives the
 *   fastest copies); W, A, B stay device pointers (resident weights). The call copies X
 *   to a device staging buffer owned by the handle, runs lora_linear_forward, copies Y
 *   back and waits for the stream before returning. The staging buffers are allocated on
 *   the first call and grow to max_tokens rows. Returns as lora_linear_forward, plus
 *   LORA_ENOMEM if staging cannot be allocated and LORA_ETIMEOUT if a kernel's bounded
 *   wait ran out. Large T runs as row chunks whose copies overlap the kernels; on any error
 *   the call still waits for the copies it has queued, so x_host and y_host are not touched
 *   after it returns.
 * Source: as lora_linear_forward.
 */
int lora_linear_forward_host(lora_linear* h, const void* x_host, int T,
                             const int32_t* seg_offsets, const int32_t* seg_adapter_ids, int n_seg,
                             const void* W, const void* const* A, const void* const* B,
                             const float* scale, int n_adapters, void* y_host, void* stream);

/*
 * lora_linear_w4_repack -- convert a 4-bit base weight from the plain layout to the kernel
 * layout that lora_linear_forward_w4 reads. Run once when the weight is loaded.
 *   src  device uint8 [d_out, d_in / 2], plain layout: signed 4-bit weights q in [-8, 7]
 *        (two's complement nibbles); byte j of row n holds input feature 2j in its low
 *        nibble and 2j + 1 in its high one.
 *   dst  device, same size; may equal src (in place). Kernel layout, per 32-bit
 *        little-endian word of a row (input features 8c .. 8c+7): offset-binary nibbles
 *        q + 8, feature 8c+2j in nibble j and feature 8c+2j+1 in nibble j+4 (j = 0..3).
 *   n_bytes  size of the weight in bytes: a multiple of 4, both pointers 4-byte aligned
 *        (else LORA_EINVAL). Enqueued on `stream`; returns once launched.
 * Source: no counterpart on the pages (the layout is this library's: the converter warps of
 * lora_linear_forward_w4 turn one word into four bf16 pairs with a mask, an or and two
 * bf16 operations per pair).
 */
int lora_linear_w4_repack(const void* src, void* dst, long long n_bytes, void* stream);

/*
 * lora_linear_forward_w4 -- lora_linear_forward with a 4-bit base weight.
 *   Wq  device uint8 [d_out, d_in / 2], in the kernel layout written by
 *       lora_linear_w4_repack from the plain layout (signed 4-bit q[n, k], see there).
 *   Ws  device bf16 [d_in / 128, d_out]: one scale per output row and group of 128 inputs.
 *   The base weight is W[n, k] = q[n, k] * Ws[k / 128, n]; on the GPU each weight is
 *   rounded to bf16 (round to nearest even) before the bf16 tensor-core product. The
 *   adapters (A, B) stay bf16. Requires d_in to be a multiple of 128 (else LORA_EINVAL);
 *   all other arguments, layouts and errors as lora_linear_forward.
 * Source: "Two 27B models on a single RTX 5090", section 4 (the memory budget: a 4-bit base
 * of 18.1 GiB with a bf16 adapter of 1.3 GiB) and "Qwen3.8-27B on one RTX 3090 with patched
 * vLLM + DFlash2" (the W4A16 base); the group size and symmetric form are this library's.
 */
int lora_linear_forward_w4(lora_linear* h, const void* x, int T,
                           const int32_t* seg_offsets, const int32_t* seg_adapter_ids, int n_seg,
                           const void* Wq, const void* Ws, const void* const* A, const void* const* B,
                           const float* scale, int n_adapters, void* y, void* stream);

/*
 * lora_linear_forward_host_w4 -- lora_linear_forward_host with the 4-bit base of
 * lora_linear_forward_w4 (Wq, Ws device pointers; X and Y host buffers).
 * Source: as lora_linear_forward_w4.
 */
int lora_linear_forward_host_w4(lora_linear* h, const void* x_host, int T,
                                const int32_t* seg_offsets, const int32_t* seg_adapter_ids, int n_seg,
                                const void* Wq, const void* Ws, const void* const* A, const void* const* B,
                                const float* scale, int n_adapters, void* y_host, void* stream);

/* lora_linear_destroy -- wait for the handle's work, free everything it owns. NULL-safe. */
int lora_linear_destroy(lora_linear* h);

/*
 * lora_linear_status -- LORA_OK, or LORA_ETIMEOUT if any kernel launched by this handle
 * gave up a bounded wait (it then stopped early and its output is incomplete). Waits for
 * the device first. reset != 0 clears the status word afterwards.
 */
int lora_linear_status(lora_linear* h, int reset);

/*
 * lora_linear_plan -- the token-segment planner, on the host (no GPU needed).
 *   Tiles for the fused base+expand pass: walk the rows in order; a new tile starts when
 *   the current one holds LORA_TILE_ROWS rows or when the next row names an adapter that
 *   differs from one already in the tile. Rows with id 0 join the tile they fall in.
 *   Shrink tiles: the fused tiles with a nonzero id, stably ordered by id.
 *   fused_tiles / shrink_tiles receive int32 triples (row0, nrows, adapter_id); their
 *   capacity in triples is *n_fused / *n_shrink on entry, the count written on return.
 * Returns LORA_EINVAL for bad segments or too small a capacity.
 * Source: "Two 27B models on a single RTX 5090", section 4 (requests that name the
 * adapter and requests that do not share batches).
 */
int lora_linear_plan(const int32_t* seg_offsets, const int32_t* seg_adapter_ids, int n_seg, int T,
                     int32_t* fused_tiles, int* n_fused, int32_t* shrink_tiles, int* n_shrink);

/*
 * lora_linear_validate -- the host checks lora_linear_forward runs first, without a
 * handle or a GPU: the handle's shape (d_in, d_out, rank, max_tokens, max_segments) and
 * the call's arguments. Pointers are checked for NULL, 16-byte alignment and overlap only.
 * Returns LORA_OK or LORA_EINVAL.
 */
int lora_linear_validate(int d_in, int d_out, int rank, int max_tokens, int max_segments,
                         const void* x, int T, const int32_t* seg_offsets,
                         const int32_t* seg_adapter_ids, int n_seg, const void* W,
                         const void* const* A, const void* const* B, const float* scale,
                         int n_adapters, const void* y);

/* Tunables and diagnostics (tests, benchmarks). */
enum {
    LORA_OPT_TILE_N = 1,        /* force the output-tile width (multiple of 16, 16..256; 272..512 runs
                                   wide row tiles on SM pairs of the bf16 base with whole K, see
                                   LORA_OPT_WIDE_TILES, else 256); 0 = auto */
    LORA_OPT_WAIT_LIMIT_US = 2, /* bound of every in-kernel wait, microseconds (default 4,000,000) */
    LORA_OPT_DEBUG_STALL = 3,   /* 1 = the load warp never issues: every wait runs out (tests only) */
    LORA_OPT_TIMING = 4,        /* 1 = record CUDA events around each kernel launch */
    LORA_OPT_RASTER = 5,        /* 0 = auto, 1 = row tiles fastest, 2 = column tiles fastest,
                                   3 = groups of LORA_OPT_RASTER_GROUP column tiles, row tiles fastest;
                                   4-bit base: 1 = token groups fastest, 2 = feature tiles fastest,
                                   0 or 3 = auto */
    LORA_OPT_TWO_LAUNCH = 6,    /* 1 = shrink and fused pass as two launches (default 0: one launch) */
    LORA_OPT_CLUSTER = 7,       /* 0 = auto, 1 = one CTA per tile, 2 = SM pairs run M = 256 MMAs (tcgen05 cta_group::2) */
    LORA_OPT_RASTER_GROUP = 8,  /* column tiles per group for LORA_OPT_RASTER = 3 (default 4) */
    /* 9: retired (L2 eviction hints measured no gain and were removed; rejected with LORA_EINVAL) */
    LORA_OPT_TILE_K = 10,       /* K per pipeline stage: 0 = auto, 32 or 64 */
    LORA_OPT_INLINE_WORK_LIST = 11, /* 1 (default) = small work lists travel in the kernel parameters,
                                      0 = always upload them to device memory */
    LORA_OPT_MMA_GROUP = 12,    /* pipeline stages the MMA warp waits for at once: 0 = auto (2 for SM
                                   pairs and for batches of one tile, 1 otherwise), 1 or 2 */
    LORA_OPT_DEBUG_PUBLISH_DELAY_US = 13, /* tests only: each shrink unit of a one-launch call publishes
                                   its U rows this many microseconds late (0..1,000,000; default 0) */
    LORA_OPT_K_SPLIT = 14,      /* bf16 base: 0 = the handle's own choice (made at create), 1 = whole K per
                                   output block, 2 or 4 = K in that many parts: each block runs as that many
                                   work units; every part but the last to finish stores its fp32 sums, the
                                   last adds all of them in part order before the bf16 rounding (the same sum
                                   whichever part ends last). Fills the GPU when long-K, narrow projections
                                   leave too few or too ragged waves of blocks; fewer parts are used where K
                                   is too short for every part to get a 64-wide K-step. Changes the
                                   summation for later calls; may allocate (LORA_ENOMEM) */
    LORA_OPT_MAX_CTAS = 15,     /* at most this many CTAs (one per SM) per launch, >= 2; 0 = every SM (default).
                                   Leaves the other SMs to calls on other streams; the launch shape is chosen
                                   for the SMs it may use. Does not change any result */
    LORA_OPT_PDL = 16,          /* 1 = programmatic dependent launch for calls without adapter rows (bf16 base,
                                   one launch): the launch may start on SMs the previous kernel of the stream
                                   leaves, requests its first W tiles, and waits for that kernel before it
                                   reads or writes anything else; it lets the next kernel start early in turn.
                                   The previous kernel must not write this call's W. 0 (default) = off.
                                   Does not change any result */
    LORA_OPT_TOKEN_COLUMNS = 17, /* bf16 base: token-column units for batches of at most 512 rows whose rows
                                   all name one adapter (or none), on handles that sum whole K: each unit of
                                   an SM pair computes 256 output features for every token row of the batch
                                   (features on the MMA's M, tokens on its N), so each W tile is read once
                                   and no 128-row tile is padded. 0 (default) = when the launch-shape model
                                   expects them to finish sooner, 1 = never, 2 = whenever the batch allows
                                   them. Does not change any result */
    LORA_OPT_W4_K_SPLIT = 18,   /* 4-bit base: 0 = the handle's own choice (made at create: decode-sized
                                   handles of at most 128 rows whose one-tile units would leave most SMs
                                   idle split K in 2 to 4 parts), 1 = whole K, 2..4 = K in that many parts
                                   (each a multiple of 4 K-steps, at least 8; fewer where K is too short).
                                   Every part but the last to finish stores its fp32 sums, the last adds
                                   them in part order before the bf16 rounding. Changes the summation for
                                   later calls; may allocate (LORA_ENOMEM) */
    LORA_OPT_WIDE_TILES = 19    /* bf16 base, SM pairs, whole K: wide row tiles of 288 to 320 output columns
                                   (each 16-wide K step a second MMA over the columns past 256, one
                                   accumulator per unit), so that a projection's units fill whole waves of
                                   SM pairs. 0 (default) = when the launch-shape model expects them to
                                   finish sooner, 1 = never. Does not change any result */
};

/* lora_linear_set_option -- set one option above. Returns LORA_OK or LORA_EINVAL. */
int lora_linear_set_option(lora_linear* h, int option, long long value);

/*
 * lora_linear_timing -- with LORA_OPT_TIMING on: synchronises on the recorded events and
 * returns, per kernel kind, the summed device time in milliseconds and the launch count
 * since the option was last set. kind 0 = a separate shrink launch (two-launch mode
 * only), 1 = the launch that computes Y (in the default one-launch mode it also runs the
 * shrink). Also returns
 * the total number of kernels this handle has launched (any option state).
 */
int lora_linear_timing(lora_linear* h, int kind, double* total_ms, long long* launches,
                       long long* all_launches);

/*
 * lora_linear_describe -- the launch shape forward would use for T rows and these
 * segments, without launching: output-tile width, number of fused tiles, work units (fused
 * and shrink), grid size, pipeline stages, whether a shrink runs, and the unit order (as
 * lora_linear_shape reports it; 3 = token-column units). Any pointer may be NULL.
 */
int lora_linear_describe(lora_linear* h, int T, const int32_t* seg_offsets,
                         const int32_t* seg_adapter_ids, int n_seg, int* tile_n, int* n_tiles,
                         int* n_units, int* grid, int* stages, int* has_shrink, int* unit_order);

/*
 * lora_linear_shape -- the launch shape lora_linear_forward (w4 = 0) or
 * lora_linear_forward_w4 (w4 = 1) would choose, computed on the host alone (no device, no
 * handle): for d_in, d_out, rank as in lora_linear_create, a GPU with num_sms SMs (>= 2), the
 * default options, and T rows in these segments (checked as by lora_linear_plan). Outputs
 * (any may be NULL): cluster (2 = SM pairs, 1 = single CTAs), tile_n (output columns per
 * fused unit), bk (K per pipeline stage), stages, unit_order (0 = column (feature) tiles
 * first, 1 = row tiles (token groups) first, 2 = groups of column tiles, 3 = token-column units:
 * each covers every token row, see LORA_OPT_TOKEN_COLUMNS), fused_units (work
 * units of the fused launch, or of the 4-bit kernel) and shrink_units (shrink work units).
 * T = 0 gives zeros. Returns LORA_OK or LORA_EINVAL. Diagnostics and tests.
 */
int lora_linear_shape(int d_in, int d_out, int rank, int num_sms, int T, const int32_t* seg_offsets,
                      const int32_t* seg_adapter_ids, int n_seg, int w4, int* cluster, int* tile_n, int* bk,
                      int* stages, int* unit_order, int* fused_units, int* shrink_units);

/*
 * lora_linear_k_split -- the K parts (1 or 2, see LORA_OPT_K_SPLIT) a handle of this shape
 * and max_tokens would choose at create on a GPU with num_sms SMs, computed on the host alone.
 * Returns LORA_OK or LORA_EINVAL. Diagnostics and tests.
 */
int lora_linear_k_split(int d_in, int d_out, int rank, int max_tokens, int num_sms, int* k_split);

/*
 * lora_linear_host_chunks -- the row chunks lora_linear_forward_host runs T rows in (its
 * copies of one chunk overlap the kernel of the next): writes the n + 1 chunk bounds (0 first,
 * T last) to bounds, which must have room for LORA_MAX_HOST_CHUNKS + 1 values, and n to *n.
 * Returns LORA_OK or LORA_EINVAL (T < 0, NULL pointers).
 */
#define LORA_MAX_HOST_CHUNKS 16
int lora_linear_host_chunks(int T, int32_t* bounds, int* n);

/*
 * lora_linear_forward_noalloc -- the same projection without a handle and without
 * allocating any memory, for callers that cannot call cudaMalloc: code that runs while
 * another component owns all device memory (a serving engine whose pools were reserved
 * up front, so a raw allocation fails or fragments them), code on a latency-critical
 * path where cudaMalloc's implicit device-wide synchronisation would stall other
 * streams, and plugins whose host process forbids allocations after start-up.
 * The source pages describe no such entry point; it exists for these callers.
 *
 * Scratch: the shrink output U, the work list and a status word live in one file-scope
 * __device__ array of LORA_NOALLOC_SCRATCH_BYTES (about 2.2 MB), which every GPU that
 * loads this library holds until the process exits. Limits: T <= LORA_NOALLOC_MAX_TOKENS,
 * n_seg <= LORA_NOALLOC_MAX_SEGMENTS, rank <= LORA_MAX_RANK; larger requests return
 * LORA_EINVAL and launch nothing.
 * Arguments are those of lora_linear_forward plus the shape (d_in, d_out, rank), with the
 * same layouts, alignment rules and checks; the caller still owns x, W, A, B and y. It sums
 * each output over the whole of K in one unit, as a handle does with LORA_OPT_K_SPLIT = 1,
 * and gives the same bits as such a handle.
 * The first call on a device looks up the scratch array's device address there
 * (cudaGetSymbolAddress) and sets the kernels' shared-memory limit; make that first call
 * before any stream capture. Every call shares the one scratch array and leaves its
 * contents behind: calls that overlap on the GPU (on different streams, or from several
 * threads) race and give wrong results; order them on one stream. A work list of at most
 * 64 row tiles (shrink and fused), 48 merged segments and 4 named adapters travels in the
 * kernel parameters; a larger one is copied from a buffer on the call's stack into the
 * scratch array with cudaMemcpyAsync. While `stream` is capturing, the call returns
 * LORA_EUNSUPPORTED and enqueues nothing. Every tensor map is encoded before anything is
 * enqueued, so a call that fails enqueues nothing. A kernel wait that runs out stops that
 * kernel early (Y incomplete); this entry point has no way to report it afterwards.
 * Returns LORA_OK, LORA_EINVAL, LORA_ENODEV, LORA_EUNSUPPORTED or LORA_ECUDA.
 */
#define LORA_NOALLOC_MAX_TOKENS 4096
#define LORA_NOALLOC_MAX_SEGMENTS 64
#define LORA_NOALLOC_SCRATCH_BYTES (((LORA_NOALLOC_MAX_TOKENS + 128) * LORA_MAX_RANK * 2) + 65536)
int lora_linear_forward_noalloc(const void* x, int T, const int32_t* seg_offsets,
                                const int32_t* seg_adapter_ids, int n_seg, int d_in, int d_out,
                                int rank, const void* W, const void* const* A,
                                const void* const* B, const float* scale, int n_adapters,
                                void* y, void* stream);

/* lora_linear_error_string -- a short static description of a return code. */
const char* lora_linear_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* LORA_LINEAR_H */

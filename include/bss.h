/*
 * bss.h -- C ABI of the block-sparse spatio-temporal attention library for
 * one NVIDIA GB300 GPU (sm_103a).
 *
 * The method follows the blog "Accelerating Spatio-Temporal Attention for
 * Video Diffusion on TPUs" (Google Developers).  Each head of a video
 * diffusion transformer is routed by a boolean flag to a spatial mask (a band
 * of nearby frames) or a temporal mask (a band of nearby raster positions
 * across all frames); both masks also keep full attention to the first frame
 * (Figure 3).  Attention is computed tile by tile; tiles are full, boundary
 * or skipped (section "Logical sparsity is not physical sparsity"), full tiles
 * run without any mask (section "Avoid intra-tile masking when there is
 * nothing to mask"), and optionally the mask is rounded to the tile grid so
 * that only padding needs masking (section "Align the sparse mask with final
 * execution").  Temporal heads are permuted from frame-major (F,H,W) to
 * temporal-major (H,W,F) token order so their band becomes contiguous
 * (section "Arrange tokens for efficient temporal access", Figure 9).
 *
 * Conventions for every call:
 *  - Tensors are caller-owned device memory, contiguous [H][N][d] bf16
 *    (head-major, then token, then channel), 16-byte aligned.  N = F*Hs*Ws.
 *  - Calls are asynchronous on `stream` unless marked "synchronous".
 *  - Host-detectable errors are returned before anything is launched, and a
 *    message is available from bss_last_error_message() (thread-local).
 *  - Device-side problems (a pipeline wait that exceeded its time limit) are
 *    recorded in a per-device status word read by bss_get_device_status();
 *    the kernel then returns normally instead of hanging.
 *  - No call allocates device memory except bss_build_tile_map,
 *    bss_step_workspace_create and bss_route_heads (stream-ordered pool).
 *  - Handles are not thread-safe; one GPU, one stream per call.
 */
#ifndef BSS_H_
#define BSS_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    BSS_OK = 0,
    BSS_ERR_INVALID_ARG = 1, /* null / misaligned pointer, bad size, stale handle */
    BSS_ERR_UNSUPPORTED = 2, /* valid but not implemented (tile shape, head_dim, ...) */
    BSS_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed */
    BSS_ERR_TIMEOUT = 4,     /* a device-side pipeline wait gave up (status word) */
    BSS_ERR_OOM = 5          /* device memory allocation failed */
} bss_status;

/* Mask kinds selected per head by the routing flag (section "Support dynamic
 * routing with fixed tensor shapes": one boolean per head). */
enum { BSS_KIND_SPATIAL = 0, BSS_KIND_TEMPORAL = 1 };

/* Tile classes stored in the top two bits of a tile-map entry.
 *   FULL      every pair retained: no mask
 *   BOUNDARY  evaluates the coordinate predicate per row
 *   PAD       kept tile of a tile-aligned mask with padding key columns: only
 *             the padding is masked
 *   COLUMNS   kept sink-segment tile of a tile-aligned map of permuted temporal
 *             heads, some of whose frame-0 keys also sit in a kept band tile of
 *             the same q tile: those columns (and padding) are masked, the same
 *             for every row, so each physical key counts once */
enum { BSS_CLASS_FULL = 0, BSS_CLASS_BOUNDARY = 1, BSS_CLASS_PAD = 2, BSS_CLASS_COLUMNS = 3 };
#define BSS_CLASS_SHIFT 30
#define BSS_TILE_INDEX_MASK 0x3FFFFFFF

/* Indices of the statistics returned by bss_tile_map_stats. */
enum {
    BSS_STAT_FULL = 0,          /* tiles run without a mask */
    BSS_STAT_BOUNDARY = 1,      /* tiles that evaluate the coordinate predicate */
    BSS_STAT_PAD = 2,           /* kept tiles that mask padding columns only */
    BSS_STAT_SKIP = 3,          /* tiles never visited */
    BSS_STAT_RETAINED = 4,      /* distinct query-key pairs the result is defined over */
    BSS_STAT_EXACT_RETAINED = 5,/* pairs retained by the exact (unrounded) mask */
    BSS_STAT_COLUMNS = 6,       /* kept tiles masked by a column set (BSS_CLASS_COLUMNS) */
    BSS_STAT_COUNT = 7
};

/* Video geometry and mask parameters.
 *   F, Hs, Ws          latent frames, height and width; S = Hs*Ws, N = F*S.
 *   head_dim           64 or 128.
 *   spatial_frame_window   spatial heads keep keys with |f_k - f_q| <= window
 *                          (a local frame band, Figure 3 left).
 *   temporal_raster_window temporal heads keep keys with |s_k - s_q| <= window
 *                          in the raster index s = h*Ws + w, across all frames
 *                          (Figure 3 right; the band shape is this library's
 *                          reading of "a small spatial region").
 *   sink_frames        frames kept by every query (the first-frame attention
 *                      sink, F00); only 1 is supported.
 *   temporal_permuted  1: temporal heads are in (H,W,F) order and their keys
 *                      are addressed as a sink segment (the frame-0 keys,
 *                      S rounded up to BKV columns) followed by the N permuted
 *                      rows; 0: temporal heads stay in (F,H,W) order and the
 *                      kernel evaluates the striped predicate (the blog's
 *                      "handling temporal access inside the kernel").
 *   rounding           0: exact mask (full / boundary / skip tiles; the
 *                      blog's B2);
 *                      1: tile-aligned mask, a tile is kept iff at least half
 *                      of its real pairs are retained, then only padding
 *                      columns are masked (B3); the result is attention over
 *                      the set of physical pairs the kept tiles cover, so on
 *                      permuted temporal heads a frame-0 key kept both in the
 *                      sink segment and in a band tile is masked in the sink
 *                      tile (BSS_CLASS_COLUMNS);
 *                      2: exact mask evaluated in every visited tile (the
 *                      blog's naive traversal B1, kept for comparison: every
 *                      non-skipped tile is classed BOUNDARY). */
typedef struct {
    int32_t F, Hs, Ws;
    int32_t head_dim;
    int32_t spatial_frame_window;
    int32_t temporal_raster_window;
    int32_t sink_frames;
    int32_t temporal_permuted;
    int32_t rounding;
} bss_mask_params;

/* Opaque tile map: per mask kind, a CSR list of non-skipped kv tiles for every
 * q tile (ascending kv index, class in bits 30..31), its statistics, a
 * longest-first q-tile order and, for tile-aligned maps of permuted temporal
 * heads, the retained-column bitmask of every (q tile, sink-segment tile).
 * Owns device memory; free with bss_destroy_tile_map. */
typedef struct bss_tile_map_s* bss_tile_map;

/* Build the tile maps of both mask kinds for tiles of BQ query rows by BKV key
 * columns (section "Logical sparsity is not physical sparsity": full, boundary
 * and skipped tiles; section "Align the sparse mask with final execution":
 * tile-aligned rounding).  Counts retained pairs per tile on the GPU, compacts
 * non-skipped tiles to CSR.  Any BQ, BKV in [16, 65536] builds a map (for
 * statistics); bss_sparse_attention runs maps with BKV = 128 (the default) or
 * 64 and BQ = 256 (two 128-row MMA halves per CTA, the default) or BQ = 128
 * (one half); the fused permutation needs BKV = 128.
 * Synchronous: it allocates the map's device memory, synchronizes `stream`
 * and returns the map in *out.  Errors: INVALID_ARG (null, non-positive or
 * inconsistent sizes, windows < 0), UNSUPPORTED (sink_frames != 1,
 * head_dim not 64/128), OOM, CUDA. */
bss_status bss_build_tile_map(const bss_mask_params* params, int32_t BQ, int32_t BKV, bss_tile_map* out,
                              cudaStream_t stream);

/* Copy statistics of one kind into host out[BSS_STAT_COUNT] (indices above).
 * Host-only, no device work.  Errors: INVALID_ARG (null, stale handle, kind). */
bss_status bss_tile_map_stats(bss_tile_map map, int32_t kind, int64_t* out);

/* Host out[4] = { number of q tiles, number of kv tiles, number of CSR
 * entries, number of key columns (N, or S_pad + N for permuted temporal) }. */
bss_status bss_tile_map_dims(bss_tile_map map, int32_t kind, int32_t* out);

/* Copy the CSR of one kind to HOST buffers: row_ptr[nq + 1] and entries[nnz]
 * (sizes from bss_tile_map_dims).  Synchronous.  Errors: INVALID_ARG, CUDA. */
bss_status bss_tile_map_copy_csr(bss_tile_map map, int32_t kind, int32_t* row_ptr, int32_t* entries);

/* Free a tile map (no-op for NULL).  The caller must make sure no launch that
 * uses it is still running.  Using the handle afterwards returns INVALID_ARG. */
void bss_destroy_tile_map(bss_tile_map map);

/* Flag-driven token permutation (section "Arrange tokens for efficient
 * temporal access", Figure 9; section "Support dynamic routing with fixed
 * tensor shapes").  For head h with head_is_temporal[h] != 0:
 *   forward (inverse = 0):  out[h][s*F + f] = in[h][f*S + s]   (F,H,W)->(H,W,F)
 *   inverse (inverse = 1):  out[h][f*S + s] = in[h][s*F + f]
 * heads with flag 0 are copied unchanged.  in, out: device [H][N][d] bf16,
 * non-overlapping; head_is_temporal: device uint8[H] (NULL = all spatial).
 * Errors: INVALID_ARG (null / misaligned / overlapping, H <= 0), UNSUPPORTED. */
bss_status bss_permute(const void* in, void* out, const uint8_t* head_is_temporal, int32_t H,
                       const bss_mask_params* params, int32_t inverse, cudaStream_t stream);

/* The same permutation for the flagged (temporal) heads only: heads with
 * head_is_temporal[h] == 0 are not read and their rows of `out` are left as
 * they are.  head_is_temporal must not be NULL.  Used with
 * bss_sparse_attention_split so that spatial heads are never copied. */
bss_status bss_permute_flagged(const void* in, void* out, const uint8_t* head_is_temporal, int32_t H,
                               const bss_mask_params* params, int32_t inverse, cudaStream_t stream);

/* bss_permute_flagged of `count` (1..3) tensors with the same flags in one
 * launch (the step's Q, K and V): in[i] -> out[i], host arrays of device
 * pointers.  No output may overlap an input or another output.
 * Errors: INVALID_ARG, UNSUPPORTED. */
bss_status bss_permute_flagged_multi(const void* const* in, void* const* out, int32_t count,
                                     const uint8_t* head_is_temporal, int32_t H, const bss_mask_params* params,
                                     int32_t inverse, cudaStream_t stream);

/* Block-sparse attention O = softmax(Q K^T * scale) V over the retained pairs
 * of each head's mask (blog: tiles of Q[i1:i2] K[j1:j2]^T with running softmax
 * statistics; full tiles mask-free, boundary tiles masked, skipped tiles never
 * visited; both paths combined through the softmax normalisation).
 *   Q, K, V, O  device [H][N][d] bf16; temporal heads already permuted when
 *               the map was built with temporal_permuted = 1.
 *   lse         optional device float[H][N], natural-log log-sum-exp per row
 *               (-inf for a row with no retained key, whose O row is 0).
 *   map         built for this geometry with BKV = 128 (default) or 64 and
 *               BQ = 256 (default) or 128.
 *   head_is_temporal  device uint8[H] (NULL = all spatial); changing flags
 *               needs no map rebuild.
 *   softmax_scale    <= 0 selects 1/sqrt(head_dim).
 * Errors: INVALID_ARG, UNSUPPORTED (map tile shape), CUDA.  A device-side
 * timeout is reported by bss_get_device_status. */
bss_status bss_sparse_attention(const void* Q, const void* K, const void* V, void* O, float* lse,
                                bss_tile_map map, const uint8_t* head_is_temporal, int32_t H,
                                float softmax_scale, cudaStream_t stream);

/* bss_sparse_attention with the two head kinds in separate buffers: heads with
 * head_is_temporal[h] == 0 read Q, K, V and write O, heads with flag 1 read Qt,
 * Kt, Vt and write Ot (all device [H][N][d] bf16, only each kind's heads are
 * touched).  With Qt, Kt, Vt the bss_permute_flagged images of Q, K, V and O
 * restored by the inverse bss_permute_flagged of Ot, the step permutes only
 * the temporal heads.  Ot may be NULL: the temporal heads' output rows are
 * then written straight to O at their (F,H,W) positions (row s*F + f of the
 * permuted layout goes to row f*S + s), so no inverse permutation is needed
 * and O holds every head in (F,H,W) order (bit for bit what the inverse
 * bss_permute_flagged of Ot would give); this needs a map built with
 * temporal_permuted = 1, else Ot = NULL writes O in the heads' own layout.
 * lse as in bss_sparse_attention (each head in its own layout, also with
 * Ot = NULL).  Errors as bss_sparse_attention. */
bss_status bss_sparse_attention_split(const void* Q, const void* K, const void* V, void* O, const void* Qt,
                                      const void* Kt, const void* Vt, void* Ot, float* lse, bss_tile_map map,
                                      const uint8_t* head_is_temporal, int32_t H, float softmax_scale,
                                      cudaStream_t stream);

/* The same attention with the token permutation fused into the kernel (blog,
 * section "Arrange tokens for efficient temporal access": the (H,W,F) order
 * makes a temporal head's window one contiguous band; here the kernel reads
 * that order straight from (F,H,W) memory instead of a separate permute pass).
 *   Q, K, V, O  device [H][N][d] bf16 in (F,H,W) token order for EVERY head
 *               (no permute before, no unpermute after).  For heads with
 *               head_is_temporal[h] != 0 and a map built with
 *               temporal_permuted = 1 the kernel walks the permuted tile map
 *               and gathers its query / key rows (row s*F + f of the permuted
 *               order is row f*S + s of the input) with 16-byte cp.async
 *               copies, and writes each output row to its (F,H,W) position.
 *               Measured slower than bss_attention_step (permute first).
 *   lse         optional device float[H][N] in (F,H,W) order.
 * Results are bit-identical to bss_permute -> bss_sparse_attention ->
 * inverse bss_permute of O (and of lse) with the same flags.  H*N must be
 * below 2^31; the map must have 128-key tiles (BKV = 128; a 64-key map gives
 * UNSUPPORTED).  Errors as bss_sparse_attention. */
bss_status bss_sparse_attention_fused(const void* Q, const void* K, const void* V, void* O, float* lse,
                                      bss_tile_map map, const uint8_t* head_is_temporal, int32_t H,
                                      float softmax_scale, cudaStream_t stream);

/* Dense attention control (the blog's B0 dense baseline): the same kernel
 * visiting every tile, masking only padding columns of the last kv tile.
 * Q, K, V, O: device [H][N][d] bf16, d = 64 or 128; lse optional. */
bss_status bss_dense_attention(const void* Q, const void* K, const void* V, void* O, float* lse, int32_t H,
                               int32_t N, int32_t d, float softmax_scale, cudaStream_t stream);

/* Per-head routing from sampled queries (section "Speeding up attention":
 * Sparse VideoGen samples a few queries, computes their outputs under dense,
 * spatial and temporal attention and routes each head to the sparse mask whose
 * output deviates least from the dense one; Figure 8: one flag per head).
 * Reading: deviation = squared L2 distance to the dense output summed over the
 * sampled rows and channels; a head is temporal iff its temporal deviation is
 * strictly smaller.  Masks in (F,H,W) order.  The three outputs come from the
 * attention kernel (tensor cores; bf16 P, fp32 accumulation and output), the
 * kv range split across CTAs and merged through the log-sum-exps.
 *   Q, K, V           device [H][N][d] bf16 in (F,H,W) order, 16-byte aligned.
 *   rows              device int32[R], 1 <= R <= 65535: sampled query tokens
 *                     ((F,H,W) index), the same rows for every head; a row
 *                     outside [0, N) is skipped and recorded as
 *                     BSS_ERR_INVALID_ARG in the status word.
 *   head_is_temporal  device uint8[H] output (1 = temporal).
 *   errors            device float[2 * H] output: per head the spatial and the
 *                     temporal deviation.
 * Asynchronous on `stream`.  Scratch of 3*H*R*d*2 + 3*H*R*(d+1)*4*splits +
 * 2*H*R*4 bytes (splits <= number of SMs / (H * ceil(3R / 256)), at least 1) is
 * taken from and returned to the device's stream-ordered memory pool
 * (cudaMallocAsync).
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA. */
bss_status bss_route_heads(const void* Q, const void* K, const void* V, int32_t H, const bss_mask_params* params,
                           const int32_t* rows, int32_t R, uint8_t* head_is_temporal, float* errors,
                           cudaStream_t stream);

/* The per-layer path on device buffers (the blog's Figure 8; section "Support
 * dynamic routing with fixed tensor shapes"): with a map built with
 * temporal_permuted = 1, the temporal heads' Q, K, V are permuted into the
 * workspaces Qp, Kp, Vp (bss_permute_flagged_multi, one launch), then
 * bss_sparse_attention_split reads the spatial heads in place and stores every
 * temporal head's output row straight to its (F,H,W) row of O; with
 * temporal_permuted = 0, or
 * head_is_temporal = NULL (every head spatial), it is bss_sparse_attention on
 * Q, K, V.  Q, K, V, O: device [H][N][d] bf16 in (F,H,W) order; Qp, Kp, Vp:
 * device [H][N][d] workspaces (only the temporal heads' rows are written; may
 * be NULL when nothing is permuted); lse: optional device float[H][N], each
 * head in its own layout (permuted temporal heads in (H,W,F) order).  Two
 * launches on `stream`, no allocation.  Errors: those of the calls it makes. */
bss_status bss_attention_step(const void* Q, const void* K, const void* V, void* O, float* lse, bss_tile_map map,
                              const uint8_t* head_is_temporal, int32_t H, void* Qp, void* Kp, void* Vp,
                              cudaStream_t stream);

/* Opaque workspace of bss_attention_step_host: `depth` device buffer sets (Q,
 * K, V, O and the three permutation workspaces, [H][N][d] bf16 each, plus the
 * flags), two copy streams and events.  Owns device memory. */
typedef struct bss_step_workspace_s* bss_step_workspace;

/* Create a workspace for H heads of the geometry in params (F, Hs, Ws,
 * head_dim; the windows are not used).  depth in [1, 8] buffer sets: a call
 * uses the next set in turn, so with depth >= 2 the copies of one call overlap
 * the kernels of the previous one (3 sets let the H2D copy of call i+1 start
 * while the D2H copy of call i-1 still runs).  heads_per_group in [1, H]:
 * heads copied in, computed and copied out together.  Allocates
 * depth * (7 * H * N * d * 2 + H) bytes of device memory.  Synchronous.
 * Errors: INVALID_ARG, UNSUPPORTED, OOM, CUDA. */
bss_status bss_step_workspace_create(const bss_mask_params* params, int32_t H, int32_t depth,
                                     int32_t heads_per_group, bss_step_workspace* out);

/* Wait for the workspace's work to finish, then free it (no-op for NULL). */
void bss_step_workspace_destroy(bss_step_workspace ws);

/* Order the workspace's copy streams after all work enqueued on `stream` so
 * far (e.g. after an event that opens a timed region). */
bss_status bss_step_workspace_wait_stream(bss_step_workspace ws, cudaStream_t stream);

/* bss_attention_step from HOST buffers, pipelined.  hQ, hK, hV: host [H][N][d]
 * bf16 inputs in (F,H,W) order; hO: host output of the same shape;
 * h_head_is_temporal: host uint8[H] flags, copied each call.  Host buffers
 * should be page-locked (cudaHostAlloc / cudaHostRegister): pageable memory
 * works, but its copies do not overlap anything.  Per group of heads: H2D
 * copies of Q, K, V on the workspace's copy-in stream, the step's kernels once
 * they have landed (even groups on `stream`, odd groups on a workspace stream
 * that starts after `stream`'s earlier work, so that a group's kernels can
 * start while the previous group's drain; `stream` is ordered after all of
 * them when the call returns), the D2H copy of O on the copy-out stream once
 * they are done.  Returns once everything is enqueued; `done` (optional,
 * a caller-created event) is recorded after the last D2H copy: do not read hO,
 * or change the inputs, before it completes.  The map must be of the
 * workspace's geometry (H, N, d).  Not thread-safe per workspace.
 * Errors: INVALID_ARG (NULL buffer, stale handle, geometry), those of the
 * calls it makes, CUDA. */
bss_status bss_attention_step_host(const void* hQ, const void* hK, const void* hV, void* hO,
                                   const uint8_t* h_head_is_temporal, bss_tile_map map, bss_step_workspace ws,
                                   cudaEvent_t done, cudaStream_t stream);

/* Scratch held by bss_build_tile_map_csr_noalloc (bytes): one byte per tile
 * plus one int32 per q tile (256-byte aligned) must fit in it: about 8.3M
 * tiles.  It holds the 302,400-token geometry (21 x 90 x 160) of either kind
 * with 128 x 128 tiles (2,363 x 2,476 = 5.85M tiles), 256 x 128 or 256 x 64
 * tiles, but not with 128 x 64 tiles (2,363 x 4,950 = 11.7M tiles). */
#define BSS_NOALLOC_SCRATCH_BYTES ((int64_t)8 << 20)

/* Tile-map build that allocates no device memory.  The blog has no counterpart
 * to this call: it exists for callers that cannot allocate device memory
 * themselves -- a framework whose caching allocator owns the GPU's memory and
 * enforces its own limit, where a stray cudaMalloc can fail or fragment the
 * pool, or a latency-critical loop where cudaMalloc / cudaFree would
 * synchronize the device.
 * Builds the CSR map of ONE mask kind (0 spatial, 1 temporal) into
 * caller-owned device buffers, with the same contents as the map that
 * bss_build_tile_map builds for that kind (no longest-first order):
 *   row_ptr   int32[nq + 1], nq = ceil(N / BQ)
 *   entries   int32[entries_capacity]; entries_capacity >= nq * nkv, with
 *             nkv = ceil(ncols / BKV), ncols = N (spatial heads, and temporal
 *             heads when temporal_permuted = 0) or S_pad + N (permuted temporal
 *             heads, S_pad = S rounded up to BKV); the first row_ptr[nq] are set
 *   stats     int64[BSS_STAT_COUNT] (indices BSS_STAT_*)
 * Its scratch is a file-scope __device__ array of BSS_NOALLOC_SCRATCH_BYTES
 * that every GPU loading this library holds until the process exits; a map too
 * large for it returns BSS_ERR_UNSUPPORTED before anything is launched.
 * Asynchronous on `stream`; calls no cudaMalloc, cudaFree or allocating
 * library routine.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress), so make that first call before any stream
 * capture.  The address is kept for the process: it belongs to the context
 * current at that first call (the primary context for runtime-API callers)
 * and must not be used after that context is destroyed (cudaDeviceReset, or
 * a driver-API context destroyed), so do not call this after either.  Every
 * call uses the same array and it keeps the last call's contents: calls whose
 * work overlaps on the GPU (other streams or threads) race and corrupt each
 * other's maps, so serialize them.
 * Errors: INVALID_ARG (null / misaligned buffer, kind, tile sizes, capacity),
 * UNSUPPORTED (map larger than the scratch), CUDA. */
bss_status bss_build_tile_map_csr_noalloc(const bss_mask_params* params, int32_t kind, int32_t BQ, int32_t BKV,
                                          int32_t* row_ptr, int32_t* entries, int64_t entries_capacity,
                                          int64_t* stats, cudaStream_t stream);

/* Synchronizes `stream`, returns the current device's status word (BSS_OK or
 * the first device-side error since the last call) and clears it. */
bss_status bss_get_device_status(cudaStream_t stream);

/* Static text for a status code. */
const char* bss_status_string(bss_status status);

/* Text of the last host-side error on the calling thread ("" if none). */
const char* bss_last_error_message(void);

/* Library version (major*10000 + minor*100 + patch). */
int32_t bss_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BSS_H_ */

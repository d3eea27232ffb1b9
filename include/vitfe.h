/*
 * vitfe.h — C ABI of libvitfe, the GB300 (sm_103a) front end of a Qwen-VL
 * style vision tower: FusedInputNorm + merge-order patchify + Conv3d patch
 * embedding (as one tcgen05 GEMM with fused bias) + 2D-RoPE cos/sin tables.
 *
 * Sources of the operations (web pages, cited by title and section):
 *  - "PR #55370 完整报告" ([Bugfix] Make mm_device_do_normalize
 *    encoder-cudagraph safe, vLLM): 实现拆解 items 1-2 (normalisation is
 *    owned by the vision tower's forward: integer pixels -> rescale ->
 *    normalise -> model dtype), 评论区精华 item 1 (uint8-only input),
 *    风险与影响 items 2-4 (no silent identity default; padding rows; the
 *    per-replay cast and fp32 temporaries the fused path avoids).
 *  - "vLLM 多模态推理｜ViT 性能优化": §2.2 (patchify in merge order,
 *    flatten_patches, grid_thw, Conv3d patch embedding), §3.2 (the Conv3d as
 *    an img2col GEMM; flatten_patches shapes), §3.3 (2D-RoPE cos/sin cache,
 *    position ids in merge order, [H || W] concatenation).
 *
 * Conventions shared by every call:
 *  - All tensors are caller-owned DEVICE memory unless a parameter says
 *    "host".  Nothing here allocates, frees, synchronises or copies between
 *    host and device except vitfe_create / vitfe_destroy, so vitfe_embed,
 *    vitfe_rope, vitfe_normalize_patchify, vitfe_pos_ids and vitfe_cu_seqlens
 *    can be captured in a CUDA graph: per-call metadata (the item table and
 *    its count) is read on the device at run time.
 *  - A handle serialises its own work: calls that share a handle must be
 *    ordered (one stream, or events between streams).
 *  - The embedding calls (vitfe_embed, vitfe_embed_rope, vitfe_embed_folded)
 *    launch with programmatic stream serialization: when the kernel before
 *    one on its stream is another embedding launch, the call may start (read
 *    its pixels, items and weights, produce and multiply) while that kernel
 *    finishes, and every write it makes (outputs and status) waits for it.
 *    So stream order holds for everything a call writes; inputs must not be
 *    written by that previous embedding launch (none of them are), and a
 *    kernel of the caller's before the call is waited for in full.
 *  - Host-side argument errors return a status and launch nothing.
 *    Device-side errors are written to the optional `status` word pair
 *    (int32[2] = {code, item index or -1}); every device call overwrites it
 *    ({0, -1} on success).  Rows of an item found invalid on the device are
 *    written as the pad value; nothing is read out of range and nothing traps.
 *  - Every wait inside a kernel is bounded (1 s, or VITFE_WAIT_LIMIT_MS at
 *    vitfe_create); on expiry the launch drains its asynchronous work, frees
 *    what it holds and reports VITFE_EDEVICE_TIMEOUT (outputs invalid), and the
 *    context stays usable.  VITFE_TEST_STALL_W_LOADS=1 at vitfe_create makes
 *    the embed kernel load no weights, to exercise that path in tests.
 *  - Bucket padding: rows at or past sum(t*h*w) up to `rows` are written as
 *    embedding 0, cos 1, sin 0, position id -1, flatten_patches 0.
 *  - Pixel reads: the library reads whole aligned words of 4, 8 or 16 bytes
 *    that each hold at least one of an item's bytes, so it may touch up to 15
 *    bytes past `pixel_bytes` (inside the same 16-byte-aligned block of the
 *    16-byte-aligned buffer) but never a word that holds none of them.
 */
#ifndef VITFE_H
#define VITFE_H

#include <stdint.h>
#include <cuda_runtime_api.h>   /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

#define VITFE_MAX_ITEMS 256      /* items per call (max_items bound)            */
#define VITFE_ROPE_MAX_SIDE 4096 /* largest h or w (in patches) vitfe_rope takes */
#define VITFE_ROPE_MAX_HEAD_DIM 512
#define VITFE_MAX_HOST_ITEMS 65536 /* items per vitfe_embed_rope_host call         */

typedef struct vitfe_ctx* vitfe_t;

typedef enum {
  VITFE_OK = 0,
  VITFE_EINVAL = 1,           /* host: bad argument, nothing launched            */
  VITFE_ENOMEM = 2,           /* host: device allocation failed (create only)    */
  VITFE_ECUDA = 3,            /* host: a CUDA runtime call failed                */
  VITFE_EDEVICE_DESC = 4,     /* device: an item descriptor is inconsistent      */
  VITFE_EDEVICE_RANGE = 5,    /* device: pixels past pixel_bytes, or rows > bucket */
  VITFE_EDEVICE_TIMEOUT = 6,  /* device: a pipeline wait ran out; output invalid */
  VITFE_EUNSUPPORTED = 7      /* host: shape the kernels do not implement        */
} vitfe_status;

/* One image or video (device-resident array, 24 bytes, 8-byte aligned).
 * grid_thw = (t, h, w) in patches ("vLLM 多模态推理｜ViT 性能优化" §2.2).
 * Pixels: uint8 [frames][h*patch][w*patch][3], HWC, contiguous, starting at
 * `pixels + pixel_offset`.  frames == 1 marks a still (needs t == 1) that the
 * temporal patch replicates; a video stores frames == t * tpatch.  h and w must
 * be multiples of the merge size.  pixel_offset must be a multiple of 16. */
typedef struct {
  int64_t pixel_offset;
  int32_t t, h, w;
  int32_t frames;
} vitfe_item;

/* Create a handle for one model's front end.
 * mean[3], std[3] (host): per-channel statistics; rescale: pixel scale (1/255).
 *   x = (v * rescale - mean_c) / std_c  ("PR #55370 完整报告", 实现拆解 item 2).
 *   std_c must be finite and > 0; there is no identity default.
 * patch, tpatch, merge: P, T, m of the patchify (§2.2); hidden: N.
 * W (device, bf16): Conv3d weight [hidden][3][tpatch][patch][patch] flattened to
 *   [hidden][K], K = 3*tpatch*patch*patch (§3.2).  Copied: the caller may free it
 *   after this returns.  b (device, bf16 [hidden]) or NULL for no bias.
 * Limits: hidden % 16 == 0, 16 <= hidden <= 8192; patch 1..32; tpatch 1..4;
 *   merge 1..8.  The call synchronises `stream` before returning.
 * Returns VITFE_OK and *out, or an error (and *out = NULL). */
vitfe_status vitfe_create(vitfe_t* out, const float mean[3], const float std[3], float rescale,
                          int patch, int tpatch, int merge, int hidden,
                          const void* W, const void* b, cudaStream_t stream);

/* Release a handle (synchronises the device work it owns). NULL is ignored. */
void vitfe_destroy(vitfe_t h);

/* Fused FusedInputNorm + patchify + patch-embed GEMM + bias ("PR #55370
 * 完整报告" 实现拆解 item 2; "vLLM 多模态推理｜ViT 性能优化" §2.2, §3.2).
 * pixels (device uint8, 16-byte aligned), pixel_bytes: the pixel buffer.
 * items (device vitfe_item[max_items]); n_items (device int32): live count,
 *   0 <= *n_items <= max_items <= VITFE_MAX_ITEMS.
 * rows: output rows (the bucket), >= 0.  out (device bf16 [rows][hidden],
 *   16-byte aligned), row r = the r-th patch in item order, merge order inside
 *   each item.  status (device int32[2]) or NULL.
 * Normalised pixels and flatten_patches never reach device memory.
 * Implemented for patch 14 or 16 and hidden % 64 == 0 (else VITFE_EUNSUPPORTED). */
vitfe_status vitfe_embed(vitfe_t h, const uint8_t* pixels, int64_t pixel_bytes,
                         const vitfe_item* items, const int32_t* n_items, int32_t max_items,
                         int64_t rows, void* out, int32_t* status, cudaStream_t stream);

/* 2D-RoPE tables ("vLLM 多模态推理｜ViT 性能优化" §3.3): rotary width
 * d = head_dim / 2, inverse frequencies w_i = theta^(-2i/d), i < head_dim/4;
 * cos[r] = [cos(hpos*w_i)]_i || [cos(wpos*w_i)]_i, sin likewise.
 * cos, sin: device float32 [rows][head_dim/2], 16-byte aligned.
 * head_dim % 8 == 0, 8 <= head_dim <= VITFE_ROPE_MAX_HEAD_DIM; theta > 0.
 * Items with h or w > VITFE_ROPE_MAX_SIDE are rejected on the device.
 * The handle builds the axis table of a (head_dim, theta) pair once, over every
 * position below VITFE_ROPE_MAX_SIDE, and keeps it for its lifetime; it keeps up
 * to 4 pairs, and a call with a further pair rebuilds a transient table each time.
 * A table first needed inside a stream capture is built by the graph on every
 * replay; one eager call before the capture keeps that build out of the graph. */
vitfe_status vitfe_rope(vitfe_t h, const vitfe_item* items, const int32_t* n_items,
                        int32_t max_items, int64_t rows, int head_dim, float theta,
                        float* cos, float* sin, int32_t* status, cudaStream_t stream);

/* vitfe_embed_rope from HOST buffers, with the copies overlapped: the items are cut
 * into `chunks` runs of consecutive items with about equal rows (at most
 * VITFE_MAX_ITEMS items each); each run's pixels and descriptors go up, the fused
 * launch runs and its results come down on three streams of the handle, so one
 * run's upload and launch overlap the previous run's download.
 * pixels (host, pixel_bytes), items (host, n_items <= VITFE_MAX_HOST_ITEMS): as
 *   for vitfe_embed, but validated on the host (every item's pixels must lie
 *   inside the buffer; otherwise VITFE_EINVAL and nothing is copied).
 * out (host bf16 [rows][hidden]), cos, sin (host fp32 [rows][head_dim/2]),
 *   rows = sum of t*h*w (no bucket padding); status (host int32[2], optional):
 *   the first device error, its item index counted over all items.
 * Page-locked host memory is what lets the copies overlap.  The handle keeps
 * device staging for two runs (grown on demand, freed by vitfe_destroy).
 * Returns when every result is in host memory.  Not capturable. */
vitfe_status vitfe_embed_rope_host(vitfe_t h, const uint8_t* pixels, int64_t pixel_bytes,
                                   const vitfe_item* items, int32_t n_items, void* out,
                                   int head_dim, float theta, float* cos, float* sin,
                                   int32_t* status, int32_t chunks);

/* Folded-still variant of vitfe_embed (NOT the method's exact result): a still's
 * temporal slices of A are equal, so it multiplies one slice by W' = the sum of
 * the weight's temporal slices, computed exactly and rounded once to bf16 at
 * vitfe_create.  This halves a still's multiply-adds; only W''s rounding differs
 * from vitfe_embed.  Tiles that hold video rows are computed exactly as by
 * vitfe_embed.  Same arguments and conventions as vitfe_embed;
 * VITFE_EUNSUPPORTED when tpatch == 1. */
vitfe_status vitfe_embed_folded(vitfe_t h, const uint8_t* pixels, int64_t pixel_bytes,
                                const vitfe_item* items, const int32_t* n_items,
                                int32_t max_items, int64_t rows, void* out, int32_t* status,
                                cudaStream_t stream);

/* vitfe_embed and vitfe_rope over the same items in one launch: the embed
 * kernel's epilogue warps write each tile's cos/sin rows after draining the tile's
 * second N pass, while the MMAs of its later passes run.  Arguments, outputs, pad rows and errors are those of
 * the two calls, with one status word; items with h or w > VITFE_ROPE_MAX_SIDE
 * are rejected on the device for both outputs.  The first call with a
 * (head_dim, theta) pair also launches the table build (see vitfe_rope). */
vitfe_status vitfe_embed_rope(vitfe_t h, const uint8_t* pixels, int64_t pixel_bytes,
                              const vitfe_item* items, const int32_t* n_items,
                              int32_t max_items, int64_t rows, void* out, int head_dim,
                              float theta, float* cos, float* sin, int32_t* status,
                              cudaStream_t stream);

/* Standalone FusedInputNorm + patchify: writes flatten_patches, bf16
 * [rows][K] in the canonical (C, T, P, P) feature order of §3.2 (the order
 * the Conv3d weight is flattened in).  Same inputs as vitfe_embed. */
vitfe_status vitfe_normalize_patchify(vitfe_t h, const uint8_t* pixels, int64_t pixel_bytes,
                                      const vitfe_item* items, const int32_t* n_items,
                                      int32_t max_items, int64_t rows, void* out,
                                      int32_t* status, cudaStream_t stream);

/* Position ids (§3.3 step 2): int32 [rows][2] = (hpos, wpos) per patch in merge
 * order, repeated over t; pad rows (-1, -1). */
vitfe_status vitfe_pos_ids(vitfe_t h, const vitfe_item* items, const int32_t* n_items,
                           int32_t max_items, int64_t rows, int32_t* pos, int32_t* status,
                           cudaStream_t stream);

/* RoPE applied to Q and K ("vLLM 多模态推理｜ViT 性能优化" §3.3 step 6), in place,
 * in the rotate-half form: for every row r, head and i < head_dim/2,
 *   y[i]              = x[i] * cos[r][i] - x[i + head_dim/2] * sin[r][i]
 *   y[i + head_dim/2] = x[i + head_dim/2] * cos[r][i] + x[i] * sin[r][i]
 * in fp32, rounded to nearest-even bf16.  cos, sin: the [rows][head_dim/2] tables
 * of vitfe_rope (device fp32, 16-byte aligned).  q: device bf16, row r head h at
 * q + r * q_row_stride + h * head_dim (elements; stride a multiple of 4, at least
 * heads_q * head_dim; 8-byte aligned), so Q may be a view into a packed QKV
 * buffer; k likewise.  heads_q or heads_k may be 0 (that pointer is then
 * unused).  head_dim % 8 == 0, 8 <= head_dim <= VITFE_ROPE_MAX_HEAD_DIM.
 * Needs no handle; capturable. */
vitfe_status vitfe_rope_apply(const float* cos, const float* sin, int64_t rows, int head_dim,
                              void* q, int32_t heads_q, int64_t q_row_stride, void* k,
                              int32_t heads_k, int64_t k_row_stride, cudaStream_t stream);

/* Attention sequence boundaries ("vLLM 多模态推理｜ViT 性能优化" §3.4): the
 * encoder's attention keeps images apart, and its variable-length kernels take
 * the first row of every sequence.  Each temporal group of an item (a still: the
 * image) is one sequence of h*w rows, in item order, clipped to `rows`.
 * cu_seqlens (device int32 [max_seqs + 1]): cu_seqlens[0] = 0, cu_seqlens[s + 1]
 *   = end row of sequence s; entries past the last sequence repeat its end.
 * seq_info (device int32 [2]): {number of sequences, longest sequence}.
 * More than max_seqs sequences: the first max_seqs are written and the status
 * word reports VITFE_EDEVICE_RANGE.  One small launch; capturable. */
vitfe_status vitfe_cu_seqlens(vitfe_t h, const vitfe_item* items, const int32_t* n_items,
                              int32_t max_items, int64_t rows, int32_t max_seqs,
                              int32_t* cu_seqlens, int32_t* seq_info, int32_t* status,
                              cudaStream_t stream);

/* Allocation-free 2D-RoPE tables, for callers that cannot allocate device memory:
 * code whose device memory is all reserved up front by a pool it does not own (a
 * serving runtime that carves up the GPU at start-up), or a process that may not call
 * cudaMalloc once it is serving, where an allocation can fail or stall the other work
 * on the GPU.  Creating a handle allocates, so they cannot use vitfe_rope.  No
 * counterpart in the pages; it computes exactly what vitfe_rope computes, without a
 * handle (tpatch and merge are passed directly).
 * Scratch: a 1 MiB file-scope device array that every GPU loading the library
 * keeps until exit; it bounds head_dim to 128 (VITFE_EUNSUPPORTED above that, up
 * to VITFE_ROPE_MAX_HEAD_DIM) and h, w to VITFE_ROPE_MAX_SIDE (checked on the
 * device, VITFE_EDEVICE_DESC).  The call allocates and frees nothing.
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  All calls
 * share the array: calls that overlap on the GPU (other streams, other threads)
 * race and must be ordered by the caller.  Arguments, layouts and errors are
 * otherwise those of vitfe_rope. */
vitfe_status vitfe_rope_noalloc(int tpatch, int merge, const vitfe_item* items, const int32_t* n_items,
                                int32_t max_items, int64_t rows, int head_dim, float theta,
                                float* cos, float* sin, int32_t* status, cudaStream_t stream);

/* Host helper: build packed item descriptors from grid_thw.
 * grid_thw (host int32 [n][3]); is_still (host uint8 [n], nonzero = a still
 * stored as one frame; NULL = every item with t == 1 is a still).
 * Writes items_out (host [n]) with 16-byte aligned offsets of a packed pixel
 * buffer, *total_rows = sum t*h*w, *pixel_bytes = bytes that buffer needs. */
vitfe_status vitfe_items_from_grid(const int32_t* grid_thw, const uint8_t* is_still, int32_t n,
                                   int patch, int tpatch, vitfe_item* items_out,
                                   int64_t* total_rows, int64_t* pixel_bytes);

/* Feature width K = 3*tpatch*patch*patch of a handle (0 for NULL). */
int vitfe_feature_dim(vitfe_t h);

/* Static description of a status code. */
const char* vitfe_status_str(vitfe_status s);

#ifdef __cplusplus
}
#endif
#endif /* VITFE_H */

/*
 * dflash.h - C ABI of the GB300 (sm_103a) DFlash 2 drafter pass.
 *
 * The pass, as the cortiq-engine pages define it (src/cortiq_engine/dflash.rs,
 * module doc and `Drafter`; src/gpu_cuda/hyb/dflash.rs, `Dev`):
 *
 *   settle   t   = rms(FC . f16(taps), hidden_norm)              per context row
 *            K_l = rot(rms_head(Wk_l . t, k_norm_l)),  V_l = Wv_l . t   into the cache
 *   block    rows [anchor, MASK, ...] at positions a, a+1, ...:
 *            x = rms(h); d = Pr . f16(x); x = conv(stage 0, x, d); q, k, v = W . x;
 *            per-head q/k norms and rotation; attention over the layer's windowed
 *            context and the block's own rows (not causal); h += conv(stage 1, Wo . y, d);
 *            the SwiGLU MLP wrapped the same way; hn = rms(h, norm)
 *   head     logits[j] = Head[0:width] . hn[j],  hp[j] = S . f16(hn[j])   for rows j = 1..k
 *   select   per row: top candidates re-scored in order, score = logit + (P[prev] * hp) . C[cand]
 *
 * Conventions for every call:
 *  - Device pointers are plain CUDA device addresses; the caller owns all
 *    device memory (weights, caches, workspace, inputs, outputs). The library
 *    allocates no device memory and keeps only small host state.
 *  - Calls that take a stream only enqueue work on it (no host synchronisation,
 *    no device-to-host copy); they can be captured in a CUDA graph.
 *  - Every call that can fail returns 0 on success or a DFLASH_E_* code, with a
 *    thread-local message in dflash_last_error(). On failure nothing is enqueued
 *    unless the code is DFLASH_E_CUDA (a launch failed after earlier launches).
 *  - The library fails loudly: there is no host fallback of any step.
 *  - A drafter handle keeps host state (each sequence's settled range, the
 *    caches' tensor maps): calls on one handle come from one thread at a time.
 *    Separate handles may be driven from separate threads and devices; the
 *    one-time set-up of each kernel is done once per device and is safe when
 *    threads race to it.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DFLASH_MAX_LAYERS 64
#define DFLASH_SETTLE_MAX 1024    /* rows per settle call (gpu_cuda/hyb/dflash.rs, SETTLE_MAX, is 256 there) */
#define DFLASH_MAX_BLOCK 16       /* rows of a block this build takes */

enum {
  DFLASH_OK = 0,
  DFLASH_E_GEOMETRY = 1,   /* the geometry breaks a rule of Geometry::of or a limit of this build */
  DFLASH_E_ARG = 2,        /* a bad argument: null or misaligned pointer, size out of range */
  DFLASH_E_CAPACITY = 3,   /* the context cache or the workspace is too small */
  DFLASH_E_CUDA = 4,       /* a CUDA call failed */
  DFLASH_E_NOMEM = 5       /* a host allocation failed */
};

/* What a DFlash 2 checkpoint fixes (dflash.rs, `Geometry`). `windows[l]` is the
 * positions a block row of layer l sees back, 0 = all; `no_rope[l]` = 1 for a
 * layer without rotary position. `quant_group` is the four-bit group along the
 * input dimension (32, 64 or 128). `conv_group` is channels per group of the
 * row convolution (groups = hidden / conv_group). */
typedef struct dflash_geometry {
  int32_t hidden, intermediate, layers, heads, kv_heads, head_dim, vocab, block;
  uint32_t mask_token;
  int32_t conv_group, conv_kernel, selector_rank, selector_top, taps, quant_group;
  int32_t windows[DFLASH_MAX_LAYERS];
  uint8_t no_rope[DFLASH_MAX_LAYERS];
  double rope_theta, eps;
} dflash_geometry;

/* A matrix in the library's packed layout (dflash_pack_int4 / dflash_pack_f16). */
typedef struct dflash_matrix {
  const void *data;      /* device; int4: tiles of codes; f16: tiles of values */
  const void *scales;    /* device; int4 only: packed f16 scales; NULL for f16 */
} dflash_matrix;

/* One layer (dflash.rs `Layer`): f32 device vectors, packed matrices. */
typedef struct dflash_layer_weights {
  const float *in_norm, *post_norm;        /* [hidden] */
  const float *q_norm, *k_norm;            /* [head_dim] */
  const float *attn_base, *mlp_base;       /* [2][conv_kernel][hidden] */
  dflash_matrix attn_proj, mlp_proj;       /* f16 [2*conv_kernel*groups][hidden] */
  dflash_matrix q, k, v, o, gate, up, down;/* int4 [rows][cols] as in Drafter::new */
} dflash_layer_weights;

typedef struct dflash_weights {
  dflash_matrix fc;                /* f16 [hidden][taps*hidden] */
  const float *hidden_norm, *norm; /* [hidden] */
  dflash_matrix sel;               /* f16 [selector_rank][hidden] */
  const uint16_t *pred_book;       /* f16 [vocab][selector_rank], row-major, unpacked */
  const uint16_t *succ_book;       /* f16 [vocab][selector_rank], row-major, unpacked */
  dflash_matrix head;              /* int4 [vocab][hidden] (the target's head) */
  const dflash_layer_weights *layers; /* host array of `layers` entries */
} dflash_weights;

typedef struct dflash_t dflash_t;

/* ---- context caches --------------------------------------------------------- */

#define DFLASH_KV_PLANES 0  /* two f16 planes an element (hi, lo): 4 bytes, about 21 bits (dflash_create) */
#define DFLASH_KV_F16 1     /* one f16 an element: 2 bytes, 11 bits */

/* How the K and V caches of every (sequence, layer) are laid out. `format` is
 * DFLASH_KV_PLANES or DFLASH_KV_F16 (the element's form, per row and KV head:
 * hi[head_dim] then lo[head_dim], or one f16[head_dim]). ring[l] = 0: a linear
 * cache of ctx_cap rows, row = position - first. ring[l] = C > 0, only for a
 * layer with a window w (C >= 2 * w): a ring of C rows, row = (position -
 * first) % C, followed by w more rows that repeat its first w rows, so that
 * every range a block reads (fewer than w rows) is contiguous. A ring holds
 * every row the layer keeps: after each settle the window trim of dflash.rs
 * `Drafter::settle_rows` leaves a layer at most 2 * w rows (the ring of
 * dory.rs `struct Slot` holds a sliding layer's rows the same way). */
typedef struct dflash_cache_config {
  int32_t format;
  int32_t ring[DFLASH_MAX_LAYERS];
} dflash_cache_config;

/* Rows, and bytes, of layer `layer`'s K cache (the V cache is the same) of one
 * sequence under `cache` (NULL: DFLASH_KV_PLANES, no rings); 0 for a bad
 * argument or a ring the layer cannot take. */
int64_t dflash_cache_rows(const dflash_geometry *g, const dflash_cache_config *cache, int32_t layer, int64_t ctx_cap);
size_t dflash_cache_bytes(const dflash_geometry *g, const dflash_cache_config *cache, int32_t layer, int64_t ctx_cap);

/* ---- packing (the library's matrix layouts) -------------------------------- */

/* Bytes of the packed codes and of the packed scales of a four-bit matrix
 * [rows][cols]; cols % 64 == 0, group in {32, 64, 128}, rows padded to 128.
 * Returns 0 for a shape the library does not take. */
size_t dflash_int4_packed_bytes(int64_t rows, int64_t cols, int32_t group);
size_t dflash_int4_scale_bytes(int64_t rows, int64_t cols, int32_t group);

/* Repack a four-bit matrix from the interchange format (codes u8 [rows][cols/2],
 * q+8 offset-binary, the even column in the low nibble; scales f16
 * [rows][cols/group]) into the library's tile layout. All pointers are device
 * pointers, 16-byte aligned; dst_codes/dst_scales hold the sizes above.
 * Enqueued on `stream`. Errors: DFLASH_E_ARG. */
int dflash_pack_int4(const uint8_t *codes, const uint16_t *scales, int64_t rows, int64_t cols,
                     int32_t group, void *dst_codes, void *dst_scales, void *stream);

/* The f16 matrices' tile layout: bytes, and the repack from row-major f16. */
size_t dflash_f16_packed_bytes(int64_t rows, int64_t cols);
int dflash_pack_f16(const uint16_t *src, int64_t rows, int64_t cols, void *dst, void *stream);

/* The exact values of a packed four-bit matrix, f32 [rows][cols] (q * scale):
 * the drafter's own dequantisation, exposed for checking. */
int dflash_dequant_int4(const void *codes, const void *scales, int64_t rows, int64_t cols,
                        int32_t group, float *out, void *stream);

/* The drafter's product of a packed matrix W [rows][cols] with T rows of X:
 * Y[t][r] = sum_c X[t][c] W[r][c], f32 X [T][cols] and Y [T][rows] (device,
 * row-major). `kind` 4: a four-bit matrix (group `group`; X enters at full f32
 * precision as f16 hi + lo planes); `kind` 16: an f16 matrix (X rounded to f16,
 * as the card arm's `to_half` before its f16 GEMM). `workspace` (device,
 * 16-byte aligned) receives the packed rows of X: at least
 * dflash_gemm_workspace_bytes(kind, cols, T) bytes. Exposed for checking the
 * kernels the pass uses. Errors: ARG, CAPACITY, CUDA. */
size_t dflash_gemm_workspace_bytes(int32_t kind, int64_t cols, int32_t T);
int dflash_gemm(const dflash_matrix *w, int32_t kind, int64_t rows, int64_t cols, int32_t group, const float *x,
                int32_t T, float *y, void *workspace, size_t workspace_bytes, void *stream);

/* The GEMM kernel of dflash_gemm alone, for T <= 32 rows: it reads the token
 * tiles that a dflash_gemm call with the same kind, cols, T and workspace
 * packed before (so that the kernel can be timed without its packing). When
 * the launch splits its k-range, y is cleared first on the stream. Errors:
 * ARG (T > 32 or a bad shape), CUDA. */
int dflash_gemm_packed(const dflash_matrix *w, int32_t kind, int64_t rows, int64_t cols, int32_t group, int32_t T,
                       float *y, const void *workspace, void *stream);

/* The library's device error word: bit 0 (value 1) is set when one of its
 * kernels gave up a bounded wait (the kernel then stopped early and its outputs
 * are not to be trusted); bit 1 (value 2) when a settle or a block wrote a K or
 * V value that is not finite or at least 65,536 in magnitude, beyond the range
 * of the cache's hi plane (that element then reads as infinity). Reads the word
 * (synchronising the device) and clears it if `reset`. */
int dflash_device_error(uint32_t *error, int32_t reset);

/* ---- the drafter ----------------------------------------------------------- */

/* Workspace bytes for up to `max_batch` sequences in one block call. */
size_t dflash_workspace_bytes(const dflash_geometry *g, int32_t max_batch);

/* Check the geometry (Geometry::of's rules and this build's limits: hidden % 64,
 * heads*head_dim % 64, intermediate % 64, head_dim in {64, 128}, block <= 16,
 * selector_top <= 32, vocab % 16) and bind the weights, the per-sequence
 * context caches and the workspace. `ctx_k` / `ctx_v` are host arrays of
 * max_batch*layers device pointers, indexed [seq*layers + layer], each a
 * cache of ctx_cap * kv_heads * head_dim * 4 bytes, 16-byte aligned: per
 * (position - first, KV head), in the card arm's `[position - first][kv]`
 * order, the row's f32 values as two f16 planes, hi[head_dim] then
 * lo[head_dim], with hi = x with its low 13 mantissa bits cleared (exact in
 * f16 for 2^-14 <= |x| < 65536; below that range hi + lo is off by at most
 * 2^-24, at or above it the planes overflow to infinity) and lo = f16(x - hi),
 * so that hi + lo carries about 21 bits of x (the form the attention's tensor
 * cores read); a value out of that range sets bit 1 of the device error word
 * (dflash_device_error). Every sequence starts empty at
 * first = 0. Nothing is enqueued. Errors: GEOMETRY, ARG, CAPACITY (workspace),
 * NOMEM. */
int dflash_create(dflash_t **out, const dflash_geometry *g, const dflash_weights *w,
                  int32_t max_batch, void *const *ctx_k, void *const *ctx_v, int64_t ctx_cap,
                  void *workspace, size_t workspace_bytes);

/* dflash_create with the caches laid out by `cache` (dflash_cache_config):
 * ctx_k / ctx_v[seq * layers + l] hold dflash_cache_bytes(g, cache, l, ctx_cap)
 * bytes each. Errors as dflash_create. */
int dflash_create_ex(dflash_t **out, const dflash_geometry *g, const dflash_weights *w, int32_t max_batch,
                     const dflash_cache_config *cache, void *const *ctx_k, void *const *ctx_v, int64_t ctx_cap,
                     void *workspace, size_t workspace_bytes);

/* ---- the context of a sequence (dflash.rs `Drafter`: first, len, pending,
 * and per layer `Ctx::dropped`). The context covers positions first ..
 * first + len; `pending` rows of positions first + len .. wait to be settled;
 * layer l holds positions first + dropped[l] .. first + len. */

/* Context of sequence `seq` = empty, starting at position `first`. Host only. */
int dflash_reset(dflash_t *d, int32_t seq, int64_t first);

/* The settled context of `seq`: first position and row count. Host only. */
int dflash_context(const dflash_t *d, int32_t seq, int64_t *first, int64_t *len);

/* dflash_context plus the rows waiting to be settled and, per layer, the rows
 * the window trim let go (`dropped`: a host array of `layers`, or NULL). */
int dflash_context_ex(const dflash_t *d, int32_t seq, int64_t *first, int64_t *len, int64_t *pending,
                      int64_t *dropped);

/* Add `n` (1..1024) tap rows of sequence `seq` at positions pos..pos+n-1 to the
 * context (dflash.rs `Drafter::push_context`: `queue_context`, then `settle`;
 * the rows computed as gpu_cuda/hyb/dflash.rs `Dev::settle` does). `taps` is a
 * device f32 [n][taps*hidden], joined in tap order. A position already held
 * (first <= pos <= the next position) drops what follows it first
 * (`Drafter::truncate`); any other pos (a gap) starts the context over at
 * pos. Rows that waited settle with these; when they and these are more than
 * dflash_pending_limit, the oldest (a multiple of 64 rows) settle first, in a
 * settle of their own. After each settle a windowed layer holding more than
 * twice its window rows lets go of all but its last `window` rows
 * (`Drafter::settle_rows`). Errors: ARG (n), CAPACITY (a linear cache past
 * ctx_cap), CUDA. */
int dflash_settle(dflash_t *d, int32_t seq, int64_t pos, const float *taps, int32_t n, void *stream);

/* Rows that may wait unsettled in a sequence (dflash.rs `Drafter::queue_context`,
 * the limit of its CUDA arm): max(512, widest window + 256) when every layer
 * has a window, else 512. */
int64_t dflash_pending_limit(const dflash_geometry *g);

/* Give sequence `seq` the device buffer its waiting tap rows are kept in:
 * 16-byte aligned, `rows` * taps * hidden * 4 bytes, rows >= the pending limit
 * (NULL: none; then dflash_queue fails). The buffer stays the caller's; rows
 * waiting in an earlier buffer are dropped. Host only. Errors: ARG, CAPACITY. */
int dflash_bind_pending(dflash_t *d, int32_t seq, void *buf, int64_t rows);

/* Queue `n` (1..1024) tap rows at pos.. (dflash.rs `Drafter::queue_context`):
 * the position rule of dflash_settle; the rows are copied into the pending
 * buffer and wait, except that past the pending limit the oldest (a multiple
 * of 64 rows) settle at once. A block reads no waiting rows: settle them first.
 * Errors: ARG (n, no pending buffer), CAPACITY, CUDA. */
int dflash_queue(dflash_t *d, int32_t seq, int64_t pos, const float *taps, int32_t n, void *stream);

/* Every waiting row of `seq` becomes context, in one settle (dflash.rs
 * `Drafter::settle`). Errors: CAPACITY, CUDA. */
int dflash_settle_pending(dflash_t *d, int32_t seq, void *stream);

/* Forget the context of `seq` from position `pos` on (dflash.rs
 * `Drafter::truncate`, a rewind of the target): waiting rows past pos,
 * settled rows at or past it; nothing is enqueued. Host only. */
int dflash_truncate(dflash_t *d, int32_t seq, int64_t pos);

/* Keys and values made elsewhere as the context rows of positions
 * pos..pos+n-1 (n 1..1024) of every layer (gpu_cuda/hyb/dflash.rs
 * `Dev::push_rows`, here for every layer at once): k[l], v[l] are device f32
 * [n][kv_heads][head_dim], keys already normalised and rotated. The position
 * rule, the waiting rows and the window trim are dflash_settle's; the rows are
 * written in the cache format. Errors: ARG, CAPACITY, CUDA. */
int dflash_push_rows(dflash_t *d, int32_t seq, int64_t pos, int32_t n, const float *const *k, const float *const *v,
                     void *stream);

/* One block of `batch` sequences 0..batch-1 (dflash.rs `Drafter::block` +
 * the head and selector GEMMs of `Dev::block`). `anchor_pos` is a host array
 * [batch]; `h` a device f32 [batch][block][hidden] of the rows' embeddings
 * (read only). Writes logits f32 [batch][k][width] (rows 1..k over the head's
 * first `width` rows) and hp f32 [batch][k][selector_rank]. 0 < k < block,
 * selector_top <= width <= vocab. Layer l of sequence s reads its context
 * range by `Drafter::block`'s rule, from first + dropped[l] on. Errors: ARG
 * (also: rows of a sequence wait to be settled), CUDA. */
int dflash_block(dflash_t *d, int32_t batch, const int64_t *anchor_pos, const float *h, int32_t k,
                 int32_t width, float *logits, float *hp, void *stream);

/* The selector (dflash.rs `Drafter::select_with`, `top_k`) for `batch`
 * sequences: logits f32 [batch][k][width], hp f32 [batch][k][rank],
 * anchor_tok u32 [batch] (device). Writes chosen u32 [batch][k] and
 * plain u32 [batch][k] (each row's own top token). An anchor token >= vocab
 * (device data, so not checked on the host) makes every output of its
 * sequence 0xFFFFFFFF. Errors: ARG, CUDA. */
int dflash_select(dflash_t *d, int32_t batch, const float *logits, const float *hp,
                  const uint32_t *anchor_tok, int32_t k, int32_t width, uint32_t *chosen,
                  uint32_t *plain, void *stream);

/* dflash_block then dflash_select in one call, with the same arguments and
 * results (logits and hp are written as dflash_block writes them; chosen and
 * plain are the tokens dflash_select would return for them). When the head's
 * GEMM gives every CTA whole row tiles over the full hidden width (at most 32
 * draft rows, and at least two row-tile pairs a CTA, as with a full
 * vocabulary), the GEMM also finds each row's largest key (logit, then lower
 * index) of every 2048 logits, the selector's first stage, from the values it
 * writes, so that the logits are not read back for it; otherwise the selector
 * runs its own first stage. Errors: those of dflash_block and dflash_select. */
int dflash_draft(dflash_t *d, int32_t batch, const int64_t *anchor_pos, const float *h, int32_t k,
                 int32_t width, const uint32_t *anchor_tok, float *logits, float *hp, uint32_t *chosen,
                 uint32_t *plain, void *stream);

/* The selector for callers that cannot allocate device memory: code running
 * under another framework's memory pool (which owns the device heap and does
 * not let a plug-in call cudaMalloc), decode loops that must not take
 * cudaMalloc's implicit device-wide synchronisation mid-token, and
 * foreign-function callers with no device allocator. The pages have no
 * counterpart of this call; it computes what dflash_select computes (same
 * arguments and outputs, the codebooks f16 [vocab][rank] and the sizes passed
 * directly, no drafter handle) and needs no workspace: its candidate scratch
 * is a fixed 8 MiB array inside the library, held by every GPU that loads the
 * library until the process exits, so a call's chunk maxima, candidate lists
 * and score tables, batch * k * (ceil(width / 2048) * 8 + 8200 + top * 4 +
 * top * top * 4) + 256 bytes, must fit in 8 MiB (else DFLASH_E_CAPACITY;
 * dflash_select has no such limit). The first call
 * on a device looks up that device's address of the array
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * Every call on a device shares the one array, so calls that overlap on the
 * GPU (other streams, other threads) race; serialise them. The one part that
 * must start at zero (a per-row candidate counter) is cleared by each call itself;
 * everything else a call reads it wrote itself.
 * It calls no cudaMalloc, cudaFree or allocating library routine.
 * Errors: ARG, CAPACITY, CUDA. */
int dflash_select_static(const float *logits, const float *hp, const uint32_t *anchor_tok,
                         const uint16_t *pred_book, const uint16_t *succ_book, int32_t batch, int32_t k,
                         int32_t width, int32_t vocab, int32_t rank, int32_t top, uint32_t *chosen,
                         uint32_t *plain, void *stream);

/* ---- the router ------------------------------------------------------------ */

/* A sidecar's router (dflash.rs `RouteFit` / `Route`): for the rounds the block
 * drafter won and for those the target's own chain won, a fitted subspace of
 * the target's rows, its mean f16 [hidden] and basis rows f16 [rank][hidden]
 * (orthonormal as fitted); device pointers, the caller's. */
typedef struct dflash_route {
  const uint16_t *block_mean, *block_basis;
  const uint16_t *chain_mean, *chain_basis;
  int32_t block_rank, chain_rank;   /* 0..256; a basis may be NULL at rank 0 */
} dflash_route;

/* `Route::margin` of `n` rows (device f32 [n][hidden], the target's rows at the
 * tip) into margin (device f32 [n]): each row scaled to unit length (its norm
 * at least 1e-12), then the chain subspace's reconstruction error minus the
 * block subspace's, an error being the squared length of d - B^T (B d) with
 * d = unit - mean (the pages call `router::recon_error` without printing it;
 * this is its plain reading). Above zero the round is the block drafter's.
 * Enqueued on `stream`. Errors: ARG (hidden 1..16384, ranks 0..256), CUDA. */
int dflash_route_margin(const dflash_route *r, int32_t hidden, const float *rows, int32_t n, float *margin,
                        void *stream);

void dflash_destroy(dflash_t *d);

/* The message of the calling thread's last failure ("" if none). */
const char *dflash_last_error(void);

/* Kernels the library has enqueued in this process so far (launch accounting). */
uint64_t dflash_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H */

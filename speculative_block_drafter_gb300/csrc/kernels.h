// Host-side launchers of the drafter's kernels (internal to the library).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <string>
#include <utility>

#include "common.cuh"

namespace dfl {

// Kernel launches enqueued by the library in this process.
extern std::atomic<unsigned long long> g_launches;
inline void count_launch(int n = 1) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }
// Set the calling thread's dflash_last_error() message; returns `code`.
int dflash_fail(int code, const std::string &msg);

// Launch `kern` so that it may start while the previous kernel of the stream
// finishes (programmatic dependent launch); the kernel orders itself with
// pdl_wait() (common.cuh). cluster > 1 launches thread-block clusters of that
// many CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, int cluster,
                       Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (cluster > 1) {
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = (unsigned)cluster;
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = at;
  cfg.numAttrs = n;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
  count_launch(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// One-time set-up of a kernel on each device (its dynamic shared-memory limit,
// a cached occupancy figure), safe when several host threads launch at once:
// one slot a device, 0 until set. Declare these `static` (zero-initialised).
struct PerDevice {
  std::atomic<int> slot[64];
};
// The calling thread's current device, within PerDevice's 64 slots.
inline cudaError_t device_slot(int &dev) {
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  return dev >= 0 && dev < 64 ? cudaSuccess : cudaErrorInvalidDevice;
}
// Raise `kern`'s dynamic shared-memory limit to `bytes`, once per device.
template <typename KERN>
cudaError_t smem_limit(KERN kern, int bytes, PerDevice &done) {
  int dev = 0;
  cudaError_t e = device_slot(dev);
  if (e != cudaSuccess) return e;
  if (done.slot[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.slot[dev].store(1, std::memory_order_release);
  return e;
}

// -------------------------------------------------------------- tensor-core GEMMs (tc_gemm.cu)
// Packed layouts: four-bit codes in 4 KiB tiles of 128 rows x 64 columns plus
// per-row f16 scales per 32-or-64-column unit; f16 matrices in 16 KiB tiles of
// 128 rows x 64 columns, 128-byte swizzled. Rows are padded to 128.
size_t tc_int4_codes_bytes(int64_t rows, int64_t cols);
size_t tc_int4_scale_bytes(int64_t rows, int64_t cols, int group);
size_t tc_f16_bytes(int64_t rows, int64_t cols);
cudaError_t tc_pack_int4(const uint8_t *codes, const uint16_t *scales, int64_t rows, int64_t cols, int group,
                         void *dst, void *dst_scales, cudaStream_t st);
cudaError_t tc_pack_f16(const uint16_t *src, int64_t rows, int64_t cols, void *dst, cudaStream_t st);
cudaError_t tc_dequant_int4(const void *codes, const void *scales, int64_t rows, int64_t cols, int group, float *out,
                            cudaStream_t st);

// One matrix of a GEMM launch: Y[t][r] (r < n) = sum_k X[t][k] W[r][k].
struct TcJob {
  const void *w;        // packed codes or f16 tiles
  const void *scales;   // packed scales (four-bit), else null
  float *y;             // [T][ldy]
  int n;                // rows
  int ldy;
};
// Bytes of the packed token tiles a GEMM of T rows over K columns needs.
size_t tc_act_bytes(int T, int K, bool int4);
// Up to 4 matrices over the same X [T][ldx] (K columns) in one launch. `act`
// receives the packed token tiles (tc_act_bytes). When the k-range is split,
// the outputs are cleared and accumulated with atomics.
cudaError_t tc_gemm_int4(const TcJob *jobs, int njobs, int group, const float *X, int ldx, int T, int K, void *act,
                         int num_sms, cudaStream_t st);
cudaError_t tc_gemm_f16(const TcJob *jobs, int njobs, const float *X, int ldx, int T, int K, void *act, int num_sms,
                        cudaStream_t st);

// -------------------------------------------------------------- wide GEMMs (tc_wide.cu)
// Many tokens (T > 32): X [T][ldx] is packed into token tiles of up to 256
// rows (`act`, wide_act_bytes) and the (token tile, row tile, k-tile) units of
// all jobs are split evenly over the SMs. A run of units over a row tile's
// whole k-range stores its outputs; the row tiles split between two runs are
// cleared first and accumulated with atomics. Jobs share K; `tile0` (set
// here) is a job's first row tile in the concatenation of all jobs' 128-row
// tiles. The jobs travel by value in the launch (K and V of up to 64 layers).
constexpr int SELECT_CHUNK = 2048;   // logits per chunk of the selector's first stage
constexpr int WIDE_MAX_N = 256;      // token rows of one MMA
constexpr int WIDE_MAX_JOBS = 128;
constexpr int WIDE_MAX_CTAS = 320;   // CTAs a launch may list its ranges for (WideArgs::bnd)
struct WideJob {
  const void *w;   // packed codes or f16 tiles
  const void *s;   // packed scales (four-bit), else null
  float *y;        // [T][ldy] (y_off added)
  int n;           // rows
  int ldy;
  int tile0;
};
struct WideArgs {
  int njobs, mtiles;
  int64_t y_off;
  const uint8_t *bpack;
  int K, KT, T, N, ntt;
  int64_t units;
  // CTA q's units are [bnd[q], bnd[q + 1]) when nbnd > 0, else [q U / Q, (q + 1) U / Q)
  int nbnd;
  int bnd[WIDE_MAX_CTAS + 1];
  WideJob job[WIDE_MAX_JOBS];
};
void wide_tiles(int T, int &ntt, int &N);
size_t wide_act_bytes(int T, int K, bool int4);
// With `norm_w`, the rows of X enter as rms(X[t], norm_w) (eps), the norm taken
// by the kernel that packs them.
// With `x_ready` (X does not come from a kernel before this one in the stream,
// and `act` and the outputs are this GEMM's alone), the packing runs before its
// dependency wait, overlapping the kernels before it.
cudaError_t wide_gemm(const WideJob *jobs, int njobs, int64_t y_off, bool int4, int group, const float *X, int ldx,
                      int T, int K, void *act, int num_sms, cudaStream_t st, const float *norm_w = nullptr,
                      float eps = 0.f, bool x_ready = false);

// Narrow GEMMs (T <= 32) on token tiles a producer kernel has packed: the
// tiles' rows, whether the launch will split its k-range (its outputs must then
// be cleared by the producer), and the launches. `bstride` is the bytes from
// one k-tile of the f16 GEMM's tiles to the next (TT * 128, or twice that to
// read the hi plane of a two-plane pack).
int tc_tile_rows(int T, bool int4);
bool tc_splits_int4(const TcJob *jobs, int njobs, int T, int K, int num_sms);
bool tc_splits_f16(const TcJob *jobs, int njobs, int T, int K, int num_sms);
// With `cmax` (one job whose launch takes whole k-ranges: tc_int4_whole), the
// kernel also adds each token's largest key of every SELECT_CHUNK rows into
// cmax[token * nchunks + chunk] (atomicMax; cleared beforehand): the
// selector's first stage, from the values it stores.
bool tc_int4_whole(const TcJob *jobs, int njobs, int T, int K, int num_sms);
cudaError_t tc_gemm_int4_packed(const TcJob *jobs, int njobs, int group, const void *act, int T, int K, int num_sms,
                                cudaStream_t st, unsigned long long *cmax = nullptr, int nchunks = 0);
cudaError_t tc_gemm_f16_packed(const TcJob *jobs, int njobs, const void *act, int bstride, int T, int K, int num_sms,
                               cudaStream_t st);

// The device error word (DFL_ERR_* bits, common.cuh): the union of the words of
// the files whose kernels wait on mbarriers or write the cache planes.
cudaError_t read_device_error(unsigned *out, bool reset);
cudaError_t wide_read_error(unsigned *out, bool reset);
cudaError_t attn_read_error(unsigned *out, bool reset);
cudaError_t rows_read_error(unsigned *out, bool reset);

// -------------------------------------------------------------- row kernels (rows.cu)
// out[map(t)] = x[t] * rsqrt(mean(x[t]^2) + eps) * w for rows t < T. If
// `keep_from/keep_to` are set (>= 0), only rows whose position in their block
// (t % block) lies in [keep_from, keep_to] are written, packed per sequence.
cudaError_t rmsnorm(const float *x, const float *w, float *out, int T, int hs, float eps, int block,
                    int keep_from, int keep_to, cudaStream_t st);
// Stage 0 of the row convolution: y[t] = sum_o (base[0][o] + d[t][0][o][g]) * x[t-o], o <= t % block.
cudaError_t conv_stage0(const float *x, const float *d, const float *base, float *y, int T, int hs, int kn,
                        int gs, int block, cudaStream_t st);
// Stage 1 with the residual: h[t] += sum_o (base[1][o] + d[t][1][o][g]) * x[t-o].
cudaError_t conv_stage1_residual(const float *x, const float *d, const float *base, float *h, int T, int hs,
                                 int kn, int gs, int block, cudaStream_t st);
constexpr int MAX_BATCH = 64;
// K and V rows of every layer into the context caches, in the cache format
// (planes = 2: per row and head hi[hd] then lo[hd], hi + lo carrying about 21
// bits; planes = 1: one f16 per element). With `norm`, K is normalised per head
// and, on rotary layers, rotated to pos_base + t (a settle); without, the rows
// are taken as they are (imported rows). Row t goes to cache row at + t, or for
// a ring of C rows to (at + t) % C (also C rows further on when below the
// layer's mirror); k/v[l] are f32 [T][heads][hd].
struct CtxWrite {
  const float *k[64], *v[64];
  __half *ck[64], *cv[64];
  const float *w[64];
  int rotary[64], ring[64], mirror[64];
};
cudaError_t ctx_planes(const CtxWrite &W, int nlayers, int T, int heads, int hd, int planes, float eps,
                       const float *inv_freq, int64_t pos_base, int64_t at, bool norm, cudaStream_t st);
// Fused producers of a GEMM's packed token tiles (rows.cu). Each writes its
// result into P (the following GEMM's token tiles) and clears Z (that GEMM's
// outputs, when it splits its k-range).
// rms_pack: optionally h[t] += the stage-1 convolution of (cx, cd, cbase)
// first; then x = rms(h[t], w) into xout (may be null) and P, rows outside
// [keep_from, keep_to] of their block left out when keep_from >= 0.
cudaError_t rms_pack(float *h, const float *cx, const float *cd, const float *cbase, int kn, int gs, const float *w,
                     float *xout, int T, int hs, float eps, int block, int keep_from, int keep_to, const PackDst &P,
                     const ZeroSet &Z, cudaStream_t st);
cudaError_t conv0_pack(const float *x, const float *d, const float *base, int T, int hs, int kn, int gs, int block,
                       const PackDst &P, const ZeroSet &Z, cudaStream_t st);
cudaError_t silu_pack(const float *g, const float *u, int T, int n, const PackDst &P, const ZeroSet &Z,
                      cudaStream_t st);
// The block's q, k and v, one launch: q normalised per head and rotated to
// pos0[t / block] + t % block in place; k the same and v as it is, written in
// the cache format [T][hk][planes][hd] to kp and vp (the attention's format).
cudaError_t qk_norm_rope(float *q, int ldq, const float *wq, int hq, const float *k, int ldk, const float *wk,
                         const float *v, int ldv, int hk, __half *kp, __half *vp, const float *inv_freq, int T, int hd,
                         float eps, bool rotary, const int64_t *pos0, int nseq, int block, int planes,
                         cudaStream_t st);
// m = silu(g) * u, elementwise over n values.
cudaError_t silu_mul(const float *g, const float *u, float *m, int64_t n, cudaStream_t st);

// -------------------------------------------------------------- attention (attention.cu)
// The kernel loads K and V with tensor copies: a cache of f16 values
// [rows][kv][planes][hd] (per row and head: hi[hd], lo[hd] for two planes) is
// described by a map of boxes of 64 halves x 1 plane x 1 head x `box_rows`
// rows, 128-byte swizzled. Encoding is host-only work; false if the driver cannot.
bool attn_kv_map(CUtensorMap *m, const void *base, int64_t rows, int kv, int hd, int planes, int box_rows);
// A map over bytes of `rank` (<= 5) dimensions (dims[0] innermost, strides in
// bytes for dims 1..), boxes of `box`, no swizzle, zero fill outside; false if
// the driver cannot encode it (unaligned base or strides, a box over 256).
bool byte_map(CUtensorMap *m, const void *base, int rank, const uint64_t *dims, const uint64_t *strides,
              const uint32_t *box);
struct AttnSeq {          // per sequence and layer
  CUtensorMap kmap, vmap; // the layer's K and V cache of the sequence (box_rows 64)
  int64_t row0;           // cache row of the first context row read
  int64_t lo;             // its position
  int64_t anchor;         // position of block row 0
  int n;                  // context rows read
};
size_t attn_partial_bytes(int max_batch, int kv_heads, int heads, int block, int hd);
// `seqs` is a host array of `batch` entries (passed by value). q is [batch *
// block][heads][hd] f32 (normalised and rotated); own_k / own_v map the block's
// own K and V planes [batch * block][kv][2][hd] (box_rows = block). With `pack` set, the merged rows go straight
// into those token tiles (for the output projection; `zero` its outputs to
// clear) instead of y.
cudaError_t attention(const float *q, const CUtensorMap &own_k, const CUtensorMap &own_v, const AttnSeq *seqs,
                      int batch, int heads, int kv_heads, int hd, int planes, int block, int window, float scale,
                      float *partials, float *y, int num_sms, const PackDst *pack, const ZeroSet *zero,
                      cudaStream_t st);

// -------------------------------------------------------------- selector (select.cu)
size_t select_scratch_bytes(int max_rows, int width, int top);
// `stage1_done`: the chunk maxima (and the cleared candidate counts) are
// already in the scratch (the head GEMM wrote them): the first stage is skipped.
cudaError_t select_tokens(const float *logits, const float *hp, const uint32_t *anchor_tok,
                          const uint16_t *pred, const uint16_t *succ, int batch, int k, int width, int rank,
                          int top, int vocab, void *scratch, uint32_t *chosen, uint32_t *plain, int num_sms,
                          cudaStream_t st, bool stage1_done = false);
// Where a call over `rows` rows of `width` logits keeps its chunk maxima
// ([rows][nchunks] keys) and candidate counts ([rows] ints) in `scratch`.
void select_stage1(void *scratch, int rows, int width, unsigned long long **cmax, int **cnt, int *nchunks);

}  // namespace dfl

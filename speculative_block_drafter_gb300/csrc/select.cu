// The selector (cortiq-engine src/cortiq_engine/dflash.rs, `Drafter::select_with`
// and `top_k`): per draft row, the `top` largest logits (larger first, the lower
// index first among equals), then the candidates re-scored in order against the
// token chosen before: score = logit + (P[prev] * hp) . C[cand], the first
// strictly greater score winning, the chain starting at the anchor token.
//
// Stage 1 (chunks x rows CTAs): each chunk of 2048 logits yields its own top `top`.
// Stage 2 (one CTA per row): the chunks' candidates merge into the row's top `top`.
// Stage 3 (one CTA per sequence): the chain. Row j's predecessor is the anchor
// (j = 0) or one of row j-1's candidates, so every score the chain can ask for is
// computed first, in parallel; the chain itself then only compares numbers.
#include <mutex>
#include <string>

#include "common.cuh"
#include "dflash.h"
#include "kernels.h"

namespace dfl {

constexpr int SEL_THREADS = 256;
constexpr int SEL_PER = 8;                         // logits per thread in stage 1
constexpr int SEL_CHUNK = SEL_THREADS * SEL_PER;   // logits per chunk
constexpr int MERGE_PER = 16;                      // candidates per thread in stage 2
constexpr int TOP_MAX = 32;
constexpr int RANK_MAX = 256;
constexpr int CHAIN_THREADS = 512;
constexpr int KMAX = 15;

static inline int sel_chunks(int width) { return (width + SEL_CHUNK - 1) / SEL_CHUNK; }

// Scratch of one call: per row the chunks' candidates (u64), the row's
// candidates (u32) and its score table (f32 [top][top]); one counter per row
// (sequences <= rows).
size_t select_scratch_bytes(int max_rows, int width, int top) {
  return (size_t)max_rows * ((size_t)sel_chunks(width) * top * 8 + (size_t)top * 4 + (size_t)top * top * 4 + 4) + 256;
}

// The `top` largest keys of a warp (N keys per lane in `keys`), largest first,
// written by lane 0 to out[0..top). Keys are unique except 0 (= none).
template <int N>
__device__ __forceinline__ void warp_top(unsigned long long (&keys)[N], int top, unsigned long long *out) {
  const int lane = threadIdx.x & 31;
  for (int t = 0; t < top; ++t) {
    unsigned long long mine = 0;
#pragma unroll
    for (int i = 0; i < N; ++i) mine = keys[i] > mine ? keys[i] : mine;
    const unsigned long long best = warp_max_u64(mine);
    if (best != 0ull && mine == best) {
#pragma unroll
      for (int i = 0; i < N; ++i)
        if (keys[i] == best) keys[i] = 0ull;
    }
    if (lane == 0) out[t] = best;
  }
}

// One CTA per (chunk, row): every warp takes 256 logits and keeps its top; one
// warp then takes the top of the warps' lists.
__global__ void __launch_bounds__(SEL_THREADS) k_topk_chunks(const float *__restrict__ logits, int width, int top,
                                                             unsigned long long *__restrict__ cand) {
  __shared__ unsigned long long wl[SEL_THREADS / 32][TOP_MAX];
  const int chunk = blockIdx.x, row = blockIdx.y;
  const int nchunks = gridDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float *lr = logits + (int64_t)row * width;
  unsigned long long keys[SEL_PER];
#pragma unroll
  for (int i = 0; i < SEL_PER; ++i) {
    const int idx = chunk * SEL_CHUNK + warp * 256 + i * 32 + lane;
    keys[i] = idx < width ? cand_key(lr[idx], (uint32_t)idx) : 0ull;
  }
  warp_top<SEL_PER>(keys, top, wl[warp]);
  __syncthreads();
  if (warp == 0) {
    constexpr int M = SEL_THREADS / 32 * TOP_MAX / 32;  // keys per lane in the final round
    unsigned long long k2[M];
#pragma unroll
    for (int i = 0; i < M; ++i) {
      const int idx = i * 32 + lane;  // over [warps][top]
      const int w = idx / TOP_MAX, t = idx % TOP_MAX;
      k2[i] = t < top ? wl[w][t] : 0ull;
    }
    warp_top<M>(k2, top, cand + ((int64_t)row * nchunks + chunk) * top);
  }
}

// The row's top `top` from the chunks' lists, largest first, into ctok (smem).
__device__ void merge_row(const unsigned long long *__restrict__ cr, int ncand, int top, unsigned long long (*wl)[TOP_MAX],
                          uint32_t *ctok) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned long long keys[MERGE_PER];
#pragma unroll
  for (int i = 0; i < MERGE_PER; ++i) {
    const int idx = (warp * MERGE_PER + i) * 32 + lane;
    keys[i] = idx < ncand ? cr[idx] : 0ull;
  }
  warp_top<MERGE_PER>(keys, top, wl[warp]);
  __syncthreads();
  if (warp == 0) {
    constexpr int M = SEL_THREADS / 32 * TOP_MAX / 32;
    unsigned long long k2[M];
#pragma unroll
    for (int i = 0; i < M; ++i) {
      const int idx = i * 32 + lane;
      const int w = idx / TOP_MAX, t = idx % TOP_MAX;
      k2[i] = t < top ? wl[w][t] : 0ull;
    }
    __shared__ unsigned long long fin[TOP_MAX];
    warp_top<M>(k2, top, fin);
    __syncwarp();
    for (int t = lane; t < top; t += 32) ctok[t] = cand_index(fin[t]);
  }
  __syncthreads();
}

// One CTA per (sequence, row j): row j's candidates, the predecessors it can
// have (the anchor for row 0, else row j-1's candidates, merged again here),
// and every score[p][c] = logit[c] + sum_i (P[prev_p][i] * hp[i]) * C[cand_c][i].
// The CTA that finishes a sequence last runs its chain: the first strictly
// greater score in candidate order wins, its token is the next predecessor.
__global__ void __launch_bounds__(SEL_THREADS) k_row_scores(
    const float *__restrict__ logits, const float *__restrict__ hp, const uint32_t *__restrict__ anchor_tok,
    const uint16_t *__restrict__ pred, const uint16_t *__restrict__ succ, int k, int width, int rank, int top,
    int vocab, int nchunks, const unsigned long long *__restrict__ cand, uint32_t *__restrict__ ctok_g,
    float *__restrict__ score_g, unsigned int *__restrict__ done, uint32_t *__restrict__ chosen,
    uint32_t *__restrict__ plain) {
  __shared__ unsigned long long wl[SEL_THREADS / 32][TOP_MAX];
  __shared__ uint32_t cur[TOP_MAX], prv[TOP_MAX];
  __shared__ float clog[TOP_MAX];
  __shared__ __align__(16) uint16_t Ps[TOP_MAX * RANK_MAX];
  __shared__ __align__(16) uint16_t Cs[TOP_MAX * RANK_MAX];
  __shared__ float hs[RANK_MAX];
  __shared__ bool last;
  const int row = blockIdx.x, b = row / k, j = row % k;
  const uint32_t anchor = anchor_tok[b];
  const bool bad = anchor >= (uint32_t)vocab;
  const int ncand = nchunks * top;
  if (!bad) {
    merge_row(cand + (int64_t)row * ncand, ncand, top, wl, cur);
    if (j > 0) merge_row(cand + (int64_t)(row - 1) * ncand, ncand, top, wl, prv);
    const int np = j > 0 ? top : 1;
    if (j == 0 && threadIdx.x == 0) prv[0] = anchor;
    __syncthreads();
    const int r2 = rank / 2;
    for (int i = threadIdx.x; i < top * r2; i += SEL_THREADS) {
      const int c = i / r2, e = i % r2;
      ((uint32_t *)Cs)[c * r2 + e] = ((const uint32_t *)(succ + (int64_t)cur[c] * rank))[e];
      if (c < np) ((uint32_t *)Ps)[c * r2 + e] = ((const uint32_t *)(pred + (int64_t)prv[c] * rank))[e];
    }
    for (int i = threadIdx.x; i < rank; i += SEL_THREADS) hs[i] = hp[(int64_t)row * rank + i];
    for (int c = threadIdx.x; c < top; c += SEL_THREADS) clog[c] = logits[(int64_t)row * width + cur[c]];
    __syncthreads();
    for (int it = threadIdx.x; it < np * top; it += SEL_THREADS) {
      const int p = it / top, c = it % top;
      const __half2 *pr = (const __half2 *)(Ps + p * rank);
      const __half2 *cr = (const __half2 *)(Cs + c * rank);
      float acc = 0.f;
      for (int e = 0; e < r2; ++e) {
        const float2 pv = __half22float2(pr[e]);
        const float2 cv = __half22float2(cr[e]);
        acc = fmaf(pv.x * hs[2 * e], cv.x, acc);
        acc = fmaf(pv.y * hs[2 * e + 1], cv.y, acc);
      }
      score_g[((int64_t)row * top + p) * top + c] = clog[c] + acc;
    }
    for (int c = threadIdx.x; c < top; c += SEL_THREADS) ctok_g[(int64_t)row * top + c] = cur[c];
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(done + b, 1u) == (unsigned)(k - 1);
  __syncthreads();
  if (!last || threadIdx.x != 0) return;
  __threadfence();
  done[b] = 0;  // ready for the next call
  if (bad) {
    for (int jj = 0; jj < k; ++jj) chosen[b * k + jj] = plain[b * k + jj] = 0xFFFFFFFFu;
    return;
  }
  int slot = 0;  // the predecessor's slot among the previous row's candidates
  for (int jj = 0; jj < k; ++jj) {
    const int rr = b * k + jj;
    const float *sr = score_g + ((int64_t)rr * top + slot) * top;
    float bs = -INFINITY;
    int bc = 0;
    for (int c = 0; c < top; ++c) {
      const float sc = __ldcg(sr + c);
      if (sc > bs) {
        bs = sc;
        bc = c;
      }
    }
    chosen[rr] = __ldcg(ctok_g + (int64_t)rr * top + bc);
    plain[rr] = __ldcg(ctok_g + (int64_t)rr * top);
    slot = bc;
  }
}

cudaError_t select_tokens(const float *logits, const float *hp, const uint32_t *anchor_tok, const uint16_t *pred,
                          const uint16_t *succ, int batch, int k, int width, int rank, int top, int vocab, void *scratch,
                          uint32_t *chosen, uint32_t *plain, cudaStream_t st) {
  if (top > TOP_MAX || rank > RANK_MAX || top < 1 || k > KMAX || rank % 2) return cudaErrorInvalidValue;
  const int nchunks = sel_chunks(width);
  if (nchunks * top > MERGE_PER * SEL_THREADS) return cudaErrorInvalidValue;
  const int rows = batch * k;
  unsigned long long *cand = (unsigned long long *)scratch;
  uint32_t *ctok = (uint32_t *)(cand + (size_t)rows * nchunks * top);
  float *score = (float *)(ctok + (size_t)rows * top);
  unsigned int *done = (unsigned int *)(score + (size_t)rows * top * top);
  cudaError_t e = cudaMemsetAsync(done, 0, (size_t)batch * sizeof(unsigned int), st);
  if (e != cudaSuccess) return e;
  dim3 g1(nchunks, rows);
  k_topk_chunks<<<g1, SEL_THREADS, 0, st>>>(logits, width, top, cand);
  k_row_scores<<<rows, SEL_THREADS, 0, st>>>(logits, hp, anchor_tok, pred, succ, k, width, rank, top, vocab, nchunks,
                                             cand, ctok, score, done, chosen, plain);
  count_launch(2);
  return cudaGetLastError();
}

}  // namespace dfl

// ---------------------------------------------------------------------------
// The selector for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library scratch memory: code that runs
// under another framework's memory pool (which owns the device heap and does
// not let a plug-in call cudaMalloc), decode loops that must not take
// cudaMalloc's implicit device-wide synchronisation in the middle of a token,
// and foreign-function callers with no device allocator of their own. For
// them the selector's candidate scratch lives in a fixed array below, part of
// the library image: every GPU that loads the library holds it until the
// process exits.

namespace dfl {
namespace {

constexpr size_t kStaticSelectScratch = 8u << 20;  // bytes: 32 sequences x 15 rows at a 151,936 vocabulary
static __device__ __align__(256) unsigned char g_select_scratch[kStaticSelectScratch];

// Host code cannot use g_select_scratch as a device address (in host code the
// name is a host-side stand-in), so each device's address is looked up once.
std::mutex g_scratch_mu;
void *g_scratch_addr[64] = {};

cudaError_t static_scratch(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_select_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

}  // namespace dfl

extern "C" int dflash_select_static(const float *logits, const float *hp, const uint32_t *anchor_tok,
                                    const uint16_t *pred_book, const uint16_t *succ_book, int32_t batch, int32_t k,
                                    int32_t width, int32_t vocab, int32_t rank, int32_t top, uint32_t *chosen,
                                    uint32_t *plain, void *stream) {
  using namespace dfl;
  if (!logits || !hp || !anchor_tok || !pred_book || !succ_book || !chosen || !plain)
    return dflash_fail(DFLASH_E_ARG, "select_static: null pointer");
  if (batch < 1 || k < 1 || k > KMAX || top < 1 || top > TOP_MAX || width < top || width > vocab ||
      rank < 16 || rank > RANK_MAX || rank % 16)
    return dflash_fail(DFLASH_E_ARG, "select_static: batch >= 1, 1 <= k <= 15, 1 <= top <= 32, "
                                     "top <= width <= vocab, rank a multiple of 16 in 16..256");
  if (sel_chunks(width) * top > MERGE_PER * SEL_THREADS)
    return dflash_fail(DFLASH_E_ARG, "select_static: width / top beyond the selector's merge");
  const size_t need = select_scratch_bytes(batch * k, width, top);
  if (need > kStaticSelectScratch)
    return dflash_fail(DFLASH_E_CAPACITY, "select_static: the call's candidates and score tables exceed the fixed "
                                          "8 MiB scratch; use dflash_select");
  void *scratch = nullptr;
  cudaError_t e = static_scratch(&scratch);
  if (e != cudaSuccess)
    return dflash_fail(DFLASH_E_CUDA, std::string("select_static: cudaGetSymbolAddress: ") + cudaGetErrorString(e));
  e = select_tokens(logits, hp, anchor_tok, pred_book, succ_book, batch, k, width, rank, top, vocab, scratch,
                    chosen, plain, (cudaStream_t)stream);
  if (e != cudaSuccess) return dflash_fail(DFLASH_E_CUDA, std::string("select_static: ") + cudaGetErrorString(e));
  return DFLASH_OK;
}

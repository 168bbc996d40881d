// The selector (cortiq-engine src/cortiq_engine/dflash.rs, `Drafter::select_with`
// and `top_k`): per draft row, the `top` largest logits (larger first, the lower
// index first among equals), then the candidates re-scored in order against the
// token chosen before: score = logit + (P[prev] * hp) . C[cand], the first
// strictly greater score winning, the chain starting at the anchor token.
//
// Stage 1 (chunks x rows CTAs): the largest key (value, then lower index) of
// each chunk of 2048 logits.
// Stage 2 (chunks x rows CTAs): tau = the top-th largest of the row's chunk
// maxima. The top chunk maxima are `top` distinct logits of the row, so the
// row's top-th largest key is at least tau, and every key >= tau is a
// candidate: the chunks append theirs to the row's list (typically a few
// dozen entries).
// Stage 3 (one CTA per row): the list ranked among itself gives the row's top
// `top` in order (a list past its capacity, from many equal logits, falls back
// to `top` exact passes over the row); the CTA also ranks the previous row's
// list and computes every score the chain can ask of the row (row j's
// predecessors are the anchor for j = 0, else row j-1's candidates).
// Stage 4 (one CTA per sequence): the chain itself, over the tables copied
// into shared memory.
#include <mutex>
#include <string>

#include "common.cuh"
#include "dflash.h"
#include "kernels.h"

namespace dfl {

constexpr int SEL_THREADS = 256;
constexpr int SEL_CHUNK = SELECT_CHUNK;            // logits per chunk of stage 1
constexpr int ROW_THREADS = 512;
constexpr int CAND_CAP = 1024;                     // candidates (and chunk maxima) a row CTA holds
constexpr int MAX_CHUNKS = CAND_CAP;               // width <= 2 M
constexpr int TOP_MAX = 32;
constexpr int RANK_MAX = 256;
constexpr int CHAIN_THREADS = 512;
constexpr int KMAX = 15;

static inline int sel_chunks(int width) { return (width + SEL_CHUNK - 1) / SEL_CHUNK; }

// Scratch of one call, per row: the chunk maxima (u64), the candidate count and
// list (u64, CAND_CAP), the row's top (u32) and its score table (f32 [top][top]).
static size_t row_scratch(int width, int top) {
  return (size_t)sel_chunks(width) * 8 + 8 + (size_t)CAND_CAP * 8 + (size_t)top * 4 + (size_t)top * top * 4;
}
size_t select_scratch_bytes(int max_rows, int width, int top) { return (size_t)max_rows * row_scratch(width, top) + 256; }


// Stage 1: a CTA per (group of cpb chunks, row), eight logits a thread per chunk.
__global__ void __launch_bounds__(SEL_THREADS) k_chunk_max(const float *__restrict__ logits, int width, int nchunks,
                                                           int cpb, unsigned long long *__restrict__ cmax,
                                                           int *__restrict__ cnt) {
  pdl_wait();
  __shared__ unsigned long long red[SEL_THREADS / 32];
  const int row = blockIdx.y;
  const float *lr = logits + (int64_t)row * width;
  const int c0 = blockIdx.x * cpb, c1 = min(nchunks, c0 + cpb);
  for (int chunk = c0; chunk < c1; ++chunk) {
    unsigned long long best = 0ull;
#pragma unroll
    for (int i = 0; i < SEL_CHUNK / SEL_THREADS; ++i) {
      const int idx = chunk * SEL_CHUNK + i * SEL_THREADS + threadIdx.x;
      if (idx < width) best = umax64(best, cand_key(__ldg(lr + idx), (uint32_t)idx));
    }
    best = warp_max_u64(best);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
    __syncthreads();
    if (threadIdx.x < 32) {
      unsigned long long v = threadIdx.x < SEL_THREADS / 32 ? red[threadIdx.x] : 0ull;
      v = warp_max_u64(v);
      if (threadIdx.x == 0) cmax[(int64_t)row * nchunks + chunk] = v;
    }
    __syncthreads();
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) cnt[row] = 0;
}

// Stage 2: a CTA per (group of cpb chunks, row): tau = the row's top-th
// largest chunk maximum (the top chunk maxima are `top` distinct logits of the
// row, so the row's top-th key is at least tau); the chunks' keys >= tau join
// the row's candidate list.
__global__ void __launch_bounds__(SEL_THREADS) k_chunk_filter(const float *__restrict__ logits, int width, int top,
                                                              int nchunks, int cpb,
                                                              const unsigned long long *__restrict__ cmax,
                                                              int *__restrict__ cnt,
                                                              unsigned long long *__restrict__ cands) {
  pdl_wait();
  __shared__ unsigned long long cm[MAX_CHUNKS];
  __shared__ unsigned long long tau;
  const int row = blockIdx.y;
  for (int i = threadIdx.x; i < nchunks; i += SEL_THREADS) cm[i] = cmax[(int64_t)row * nchunks + i];
  if (threadIdx.x == 0) tau = 0ull;  // fewer chunks than `top`: every logit is a candidate
  __syncthreads();
  if (nchunks >= top)
    for (int i = threadIdx.x; i < nchunks; i += SEL_THREADS) {
      const unsigned long long k = cm[i];
      int above = 0;
      for (int m = 0; m < nchunks; ++m) above += cm[m] > k;
      if (above == top - 1) tau = k;  // keys are unique: exactly one thread
    }
  __syncthreads();
  const unsigned long long t = tau;
  const float *lr = logits + (int64_t)row * width;
  unsigned long long *out = cands + (int64_t)row * CAND_CAP;
  const int c0 = blockIdx.x * cpb, c1 = min(nchunks, c0 + cpb);
  for (int chunk = c0; chunk < c1; ++chunk) {
    if (cm[chunk] < t) continue;  // nothing in this chunk reaches tau
#pragma unroll
    for (int i = 0; i < SEL_CHUNK / SEL_THREADS; ++i) {
      const int idx = chunk * SEL_CHUNK + i * SEL_THREADS + threadIdx.x;
      if (idx < width) {
        const unsigned long long k = cand_key(__ldg(lr + idx), (uint32_t)idx);
        if (k >= t) {
          const int at = atomicAdd(cnt + row, 1);
          if (at < CAND_CAP) out[at] = k;
        }
      }
    }
  }
}

// The largest key below `below` in the row (block-wide), for the exact fallback.
__device__ unsigned long long row_max_below(const float *__restrict__ lr, int width, unsigned long long below,
                                            unsigned long long *red) {
  unsigned long long best = 0ull;
  for (int idx = threadIdx.x; idx < width; idx += ROW_THREADS) {
    const unsigned long long k = cand_key(lr[idx], (uint32_t)idx);
    if (k < below) best = umax64(best, k);
  }
  best = warp_max_u64(best);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
  __syncthreads();
  unsigned long long v = 0ull;
  for (int w = 0; w < ROW_THREADS / 32; ++w) v = umax64(v, red[w]);
  return v;
}

// The row's top `top` keys' indices, in order, into out (shared memory): its
// candidate list ranked among itself, or, when the list overflowed (many equal
// logits), `top` exact passes over the row.
__device__ void row_top(const float *__restrict__ lr, int width, int top, int n,
                        const unsigned long long *__restrict__ list, unsigned long long *keys, unsigned long long *red,
                        uint32_t *out) {
  __syncthreads();
  if (n <= CAND_CAP) {
    for (int i = threadIdx.x; i < n; i += ROW_THREADS) keys[i] = list[i];
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += ROW_THREADS) {
      const unsigned long long k = keys[i];
      int above = 0;
      for (int m = 0; m < n; ++m) above += keys[m] > k;
      if (above < top) out[above] = cand_index(k);
    }
  } else {
    unsigned long long below = ~0ull;
    for (int r = 0; r < top; ++r) {
      below = row_max_below(lr, width, below, red);
      if (threadIdx.x == 0) out[r] = cand_index(below);
    }
  }
  __syncthreads();
}

// Stage 3: one CTA per row j of a sequence: its candidates, its possible
// predecessors (the anchor, or row j-1's candidates, ranked again here) and the
// score table score[p][c] = logit[cand_c] + sum_i (P[prev_p][i] * hp[i]) * C[cand_c][i].
__global__ void __launch_bounds__(ROW_THREADS) k_row_select(
    const float *__restrict__ logits, const float *__restrict__ hp, const uint32_t *__restrict__ anchor_tok,
    const uint16_t *__restrict__ pred, const uint16_t *__restrict__ succ, int k, int width, int rank, int top,
    int vocab, const int *__restrict__ cnt, const unsigned long long *__restrict__ cands, uint32_t *__restrict__ ctok,
    float *__restrict__ score) {
  pdl_wait();
  __shared__ unsigned long long keys[CAND_CAP];
  __shared__ unsigned long long red[ROW_THREADS / 32];
  __shared__ uint32_t cur[TOP_MAX], prv[TOP_MAX];
  __shared__ __align__(16) uint16_t Ps[TOP_MAX * RANK_MAX];
  __shared__ __align__(16) uint16_t Cs[TOP_MAX * RANK_MAX];
  __shared__ float hs[RANK_MAX];
  __shared__ float clog[TOP_MAX];
  const int row = blockIdx.x, b = row / k, j = row % k;
  const uint32_t anchor = anchor_tok[b];
  if (anchor >= (uint32_t)vocab) return;  // the chain reports it
  row_top(logits + (int64_t)row * width, width, top, cnt[row], cands + (int64_t)row * CAND_CAP, keys, red, cur);
  if (j > 0)
    row_top(logits + (int64_t)(row - 1) * width, width, top, cnt[row - 1], cands + (int64_t)(row - 1) * CAND_CAP,
            keys, red, prv);
  else if (threadIdx.x == 0)
    prv[0] = anchor;
  __syncthreads();
  const int np = j > 0 ? top : 1;
  const int r2 = rank / 2;
  for (int i = threadIdx.x; i < top * r2; i += ROW_THREADS) {
    const int c = i / r2, e = i % r2;
    ((uint32_t *)Cs)[c * r2 + e] = __ldg((const uint32_t *)(succ + (int64_t)cur[c] * rank) + e);
    if (c < np) ((uint32_t *)Ps)[c * r2 + e] = __ldg((const uint32_t *)(pred + (int64_t)prv[c] * rank) + e);
  }
  for (int i = threadIdx.x; i < rank; i += ROW_THREADS) hs[i] = hp[(int64_t)row * rank + i];
  for (int c = threadIdx.x; c < top; c += ROW_THREADS) {
    clog[c] = logits[(int64_t)row * width + cur[c]];
    ctok[(int64_t)row * top + c] = cur[c];
  }
  __syncthreads();
  for (int it = threadIdx.x; it < np * top; it += ROW_THREADS) {
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
    score[((int64_t)row * top + p) * top + c] = clog[c] + acc;
  }
}

// Stage 4: one CTA per sequence runs the chain over the rows' tables: the first
// strictly greater score in candidate order wins and is the next predecessor.
__global__ void __launch_bounds__(CHAIN_THREADS) k_chain(const uint32_t *__restrict__ anchor_tok, int k, int top,
                                                         int vocab, const uint32_t *__restrict__ ctok,
                                                         const float *__restrict__ score, uint32_t *__restrict__ chosen,
                                                         uint32_t *__restrict__ plain) {
  pdl_wait();
  extern __shared__ __align__(16) uint8_t chain_sm[];
  float *sc = (float *)chain_sm;                    // [k][top][top]
  uint32_t *cand = (uint32_t *)(sc + k * top * top);  // [k][top]
  const int b = blockIdx.x;
  if (anchor_tok[b] >= (uint32_t)vocab) {
    for (int j = threadIdx.x; j < k; j += CHAIN_THREADS) chosen[b * k + j] = plain[b * k + j] = 0xFFFFFFFFu;
    return;
  }
  const float *sg = score + (int64_t)b * k * top * top;
  for (int i = threadIdx.x; i < k * top * top; i += CHAIN_THREADS) {
    const int j = i / (top * top);
    const int p = (i / top) % top;
    if (j > 0 || p == 0) sc[i] = sg[i];  // row 0 has one predecessor, the anchor
  }
  for (int i = threadIdx.x; i < k * top; i += CHAIN_THREADS) cand[i] = ctok[(int64_t)b * k * top + i];
  __syncthreads();
  if (threadIdx.x == 0) {
    int slot = 0;  // the predecessor's place among the previous row's candidates
    for (int j = 0; j < k; ++j) {
      const float *r = sc + (j * top + slot) * top;
      float bs = -INFINITY;
      int bc = 0;
      for (int c = 0; c < top; ++c)
        if (r[c] > bs) {
          bs = r[c];
          bc = c;
        }
      chosen[b * k + j] = cand[j * top + bc];
      plain[b * k + j] = cand[j * top];
      slot = bc;
    }
  }
}

void select_stage1(void *scratch, int rows, int width, unsigned long long **cmax, int **cnt, int *nchunks) {
  *nchunks = sel_chunks(width);
  *cmax = (unsigned long long *)scratch;
  unsigned long long *cands = *cmax + (size_t)rows * *nchunks;
  *cnt = (int *)(cands + (size_t)rows * CAND_CAP);
}

cudaError_t select_tokens(const float *logits, const float *hp, const uint32_t *anchor_tok, const uint16_t *pred,
                          const uint16_t *succ, int batch, int k, int width, int rank, int top, int vocab, void *scratch,
                          uint32_t *chosen, uint32_t *plain, int num_sms, cudaStream_t st, bool stage1_done) {
  if (top > TOP_MAX || rank > RANK_MAX || top < 1 || k > KMAX || rank % 2) return cudaErrorInvalidValue;
  const int nchunks = sel_chunks(width);
  if (nchunks > MAX_CHUNKS) return cudaErrorInvalidValue;
  const int rows = batch * k;
  unsigned long long *cmax = (unsigned long long *)scratch;
  unsigned long long *cands = cmax + (size_t)rows * nchunks;
  int *cnt = (int *)(cands + (size_t)rows * CAND_CAP);
  uint32_t *ctok = (uint32_t *)(cnt + ((rows + 1) & ~1));
  float *score = (float *)(ctok + (size_t)rows * top);
  static PerDevice configured;
  const size_t smem = (size_t)k * top * top * 4 + (size_t)k * top * 4;
  const size_t most = (size_t)KMAX * TOP_MAX * TOP_MAX * 4 + (size_t)KMAX * TOP_MAX * 4;
  if (cudaError_t e = smem_limit(k_chain, (int)most, configured)) return e;
  // chunks a CTA so that stages 1 and 2 are about one wave (8 CTAs an SM)
  const int cpb = std::max(1, (int)(((int64_t)nchunks * rows + 8 * num_sms - 1) / (8 * num_sms)));
  const dim3 g12((nchunks + cpb - 1) / cpb, rows);
  cudaError_t e = cudaSuccess;
  if (!stage1_done) {
    e = launch_pdl(k_chunk_max, g12, dim3(SEL_THREADS), 0, st, 1, logits, width, nchunks, cpb, cmax, cnt);
    if (e != cudaSuccess) return e;
  }
  e = launch_pdl(k_chunk_filter, g12, dim3(SEL_THREADS), 0, st, 1, logits, width, top, nchunks, cpb, cmax, cnt,
                 cands);
  if (e != cudaSuccess) return e;
  e = launch_pdl(k_row_select, dim3(rows), dim3(ROW_THREADS), 0, st, 1, logits, hp, anchor_tok, pred, succ, k, width,
                 rank, top, vocab, cnt, cands, ctok, score);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_chain, dim3(batch), dim3(CHAIN_THREADS), smem, st, 1, anchor_tok, k, top, vocab, ctok, score,
                    chosen, plain);
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

constexpr size_t kStaticSelectScratch = 8u << 20;  // bytes: 9,888 a row at a 151,936 vocabulary and top 16
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
  if (sel_chunks(width) > MAX_CHUNKS) return dflash_fail(DFLASH_E_ARG, "select_static: width beyond 2 M");
  const size_t need = select_scratch_bytes(batch * k, width, top);
  if (need > kStaticSelectScratch)
    return dflash_fail(DFLASH_E_CAPACITY, "select_static: the call's candidates and score tables exceed the fixed "
                                          "8 MiB scratch; use dflash_select");
  void *scratch = nullptr;
  cudaError_t e = static_scratch(&scratch);
  if (e != cudaSuccess)
    return dflash_fail(DFLASH_E_CUDA, std::string("select_static: cudaGetSymbolAddress: ") + cudaGetErrorString(e));
  int sms = 148, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  e = select_tokens(logits, hp, anchor_tok, pred_book, succ_book, batch, k, width, rank, top, vocab, scratch,
                    chosen, plain, sms, (cudaStream_t)stream);
  if (e != cudaSuccess) return dflash_fail(DFLASH_E_CUDA, std::string("select_static: ") + cudaGetErrorString(e));
  return DFLASH_OK;
}

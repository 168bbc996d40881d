// The selector (cortiq-engine src/cortiq_engine/dflash.rs, `Drafter::select_with`
// and `top_k`): per draft row, the `top` largest logits (larger first, the lower
// index first among equals), then the candidates re-scored in order against the
// token chosen before: score = logit + (P[prev] * hp) . C[cand], the first
// strictly greater score winning, the chain starting at the anchor token.
//
// Stage 1 (many CTAs): each chunk of a row's logits yields its own top `top`.
// Stage 2 (one CTA per sequence): per row, the chunks' candidates merge into the
// row's top `top`, then the row's choice, which the next row needs.
#include "common.cuh"
#include "kernels.h"

namespace dfl {

constexpr int SEL_THREADS = 256;
constexpr int SEL_PER = 8;                       // logits per thread in stage 1
constexpr int SEL_CHUNK = SEL_THREADS * SEL_PER;  // logits per chunk
constexpr int MERGE_PER = 16;                    // candidates per thread in stage 2
constexpr int TOP_MAX = 32;
constexpr int RANK_MAX = 256;

static inline int sel_chunks(int width) { return (width + SEL_CHUNK - 1) / SEL_CHUNK; }

size_t select_scratch_bytes(int max_rows, int width, int top) {
  return (size_t)max_rows * sel_chunks(width) * top * sizeof(unsigned long long);
}

// Block-wide maximum of one key per thread; every thread gets it.
__device__ __forceinline__ unsigned long long block_max_u64(unsigned long long v, unsigned long long *red) {
  v = warp_max_u64(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  unsigned long long m = 0;
  if (threadIdx.x < 32) {
    m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0ull;
    m = warp_max_u64(m);
    if (threadIdx.x == 0) red[32] = m;
  }
  __syncthreads();
  m = red[32];
  __syncthreads();
  return m;
}

__global__ void __launch_bounds__(SEL_THREADS) k_topk_chunks(const float *__restrict__ logits, int width, int top,
                                                             unsigned long long *__restrict__ cand) {
  __shared__ unsigned long long red[33];
  const int chunk = blockIdx.x, row = blockIdx.y;
  const int nchunks = gridDim.x;
  const float *lr = logits + (int64_t)row * width;
  unsigned long long keys[SEL_PER];
#pragma unroll
  for (int i = 0; i < SEL_PER; ++i) {
    const int idx = chunk * SEL_CHUNK + i * SEL_THREADS + threadIdx.x;
    keys[i] = idx < width ? cand_key(lr[idx], (uint32_t)idx) : 0ull;
  }
  unsigned long long* out = cand + ((int64_t)row * nchunks + chunk) * top;
  for (int t = 0; t < top; ++t) {
    unsigned long long mine = 0;
#pragma unroll
    for (int i = 0; i < SEL_PER; ++i) mine = keys[i] > mine ? keys[i] : mine;
    const unsigned long long best = block_max_u64(mine, red);
    if (best != 0ull && mine == best) {
#pragma unroll
      for (int i = 0; i < SEL_PER; ++i)
        if (keys[i] == best) keys[i] = 0ull;
    }
    if (threadIdx.x == 0) out[t] = best;
  }
}

__global__ void __launch_bounds__(SEL_THREADS) k_select(const float *__restrict__ logits, const float *__restrict__ hp,
                                                        const uint32_t *__restrict__ anchor_tok,
                                                        const uint16_t *__restrict__ pred,
                                                        const uint16_t *__restrict__ succ, int k, int width, int rank,
                                                        int top, int nchunks, int vocab,
                                                        const unsigned long long *__restrict__ cand,
                                                        uint32_t *__restrict__ chosen, uint32_t *__restrict__ plain) {
  __shared__ unsigned long long red[33];
  __shared__ uint32_t ctok[TOP_MAX];
  __shared__ float cscore[TOP_MAX];
  __shared__ float pc[RANK_MAX];
  __shared__ uint32_t prev_s;
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ncand = nchunks * top;
  if (threadIdx.x == 0) prev_s = anchor_tok[b];
  __syncthreads();
  if (prev_s >= (uint32_t)vocab) {  // not a token: the sequence's outputs say so
    for (int j = threadIdx.x; j < k; j += SEL_THREADS) chosen[b * k + j] = plain[b * k + j] = 0xFFFFFFFFu;
    return;
  }
  for (int j = 0; j < k; ++j) {
    const int row = b * k + j;
    const unsigned long long *cr = cand + (int64_t)row * ncand;
    unsigned long long keys[MERGE_PER];
#pragma unroll
    for (int i = 0; i < MERGE_PER; ++i) {
      const int idx = i * SEL_THREADS + threadIdx.x;
      keys[i] = idx < ncand ? cr[idx] : 0ull;
    }
    for (int t = 0; t < top; ++t) {
      unsigned long long mine = 0;
#pragma unroll
      for (int i = 0; i < MERGE_PER; ++i) mine = keys[i] > mine ? keys[i] : mine;
      const unsigned long long best = block_max_u64(mine, red);
      if (best != 0ull && mine == best) {
#pragma unroll
        for (int i = 0; i < MERGE_PER; ++i)
          if (keys[i] == best) keys[i] = 0ull;
      }
      if (threadIdx.x == 0) ctok[t] = cand_index(best);
    }
    const uint32_t prev = prev_s;
    for (int i = threadIdx.x; i < rank; i += SEL_THREADS)
      pc[i] = __half2float(__ushort_as_half(pred[(int64_t)prev * rank + i])) * hp[(int64_t)row * rank + i];
    __syncthreads();
    for (int c = warp; c < top; c += SEL_THREADS / 32) {
      const uint32_t tok = ctok[c];
      float acc = 0.f;
      for (int i = lane; i < rank; i += 32)
        acc = fmaf(pc[i], __half2float(__ushort_as_half(succ[(int64_t)tok * rank + i])), acc);
      acc = warp_sum(acc);
      if (lane == 0) cscore[c] = logits[(int64_t)row * width + tok] + acc;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float best = -INFINITY;
      uint32_t bt = ctok[0];
      for (int c = 0; c < top; ++c) {
        if (cscore[c] > best) {
          best = cscore[c];
          bt = ctok[c];
        }
      }
      chosen[row] = bt;
      plain[row] = ctok[0];
      prev_s = bt;
    }
    __syncthreads();
  }
}

cudaError_t select_tokens(const float *logits, const float *hp, const uint32_t *anchor_tok, const uint16_t *pred,
                          const uint16_t *succ, int batch, int k, int width, int rank, int top, int vocab, void *scratch,
                          uint32_t *chosen, uint32_t *plain, cudaStream_t st) {
  if (top > TOP_MAX || rank > RANK_MAX || top < 1) return cudaErrorInvalidValue;
  const int nchunks = sel_chunks(width);
  if (nchunks * top > MERGE_PER * SEL_THREADS) return cudaErrorInvalidValue;
  unsigned long long *cand = (unsigned long long *)scratch;
  dim3 g1(nchunks, batch * k);
  k_topk_chunks<<<g1, SEL_THREADS, 0, st>>>(logits, width, top, cand);
  k_select<<<batch, SEL_THREADS, 0, st>>>(logits, hp, anchor_tok, pred, succ, k, width, rank, top, nchunks, vocab, cand,
                                          chosen, plain);
  count_launch(2);
  return cudaGetLastError();
}

}  // namespace dfl

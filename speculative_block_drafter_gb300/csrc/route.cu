// The router's margin (cortiq-engine src/cortiq_engine/dflash.rs, `Route::margin`):
// which drafter a round is for, read from the target's row at the tip. The row
// is scaled to unit length (its norm at least 1e-12); each fitted subspace
// (mean, basis rows) then leaves a reconstruction error, the squared length of
// d - B^T (B d) with d = unit - mean; the margin is the chain subspace's error
// minus the block subspace's (above zero: the block's round).
//
// One CTA per row. d lives in shared memory; p = B d takes one warp per basis
// row (a dot product of f16 basis values with d); the residual pass walks the
// columns, each thread summing p_i B[i][j] over the basis rows for its columns
// (coalesced reads of the basis row by row).
#include "common.cuh"
#include "dflash.h"
#include "kernels.h"

namespace dfl {

constexpr int RT_THREADS = 256;
constexpr int RT_RANK_MAX = 256;

struct RouteArgs {
  const __half *mean[2], *basis[2];  // [0] chain, [1] block
  int rank[2];
};

__device__ __forceinline__ float rt_block_sum(float v, float *red) {
  v = warp_sum(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < RT_THREADS / 32; ++w) t += red[w];
  return t;
}

__global__ void __launch_bounds__(RT_THREADS) k_route_margin(const float *__restrict__ rows, int hidden, RouteArgs A,
                                                             float *__restrict__ margin) {
  pdl_wait();
  extern __shared__ float rt_sm[];
  float *d = rt_sm;                      // [hidden]
  float *p = rt_sm + hidden;             // [RT_RANK_MAX]
  __shared__ float red[RT_THREADS / 32];
  const float *x = rows + (int64_t)blockIdx.x * hidden;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float ss = 0.f;
  for (int j = threadIdx.x; j < hidden; j += RT_THREADS) ss = fmaf(x[j], x[j], ss);
  const float inv = 1.f / fmaxf(sqrtf(rt_block_sum(ss, red)), 1e-12f);
  float err[2];
  for (int s = 0; s < 2; ++s) {
    const __half *mean = A.mean[s], *B = A.basis[s];
    const int rank = A.rank[s];
    for (int j = threadIdx.x; j < hidden; j += RT_THREADS) d[j] = x[j] * inv - __half2float(mean[j]);
    __syncthreads();
    for (int i = warp; i < rank; i += RT_THREADS / 32) {
      const __half *b = B + (int64_t)i * hidden;
      float acc = 0.f;
      for (int j = lane; j < hidden; j += 32) acc = fmaf(__half2float(b[j]), d[j], acc);
      acc = warp_sum(acc);
      if (lane == 0) p[i] = acc;
    }
    __syncthreads();
    float e = 0.f;
    for (int j = threadIdx.x; j < hidden; j += RT_THREADS) {
      float r = d[j];
      for (int i = 0; i < rank; ++i) r = fmaf(-p[i], __half2float(B[(int64_t)i * hidden + j]), r);
      e = fmaf(r, r, e);
    }
    err[s] = rt_block_sum(e, red);
    __syncthreads();  // d and p are rewritten for the next subspace
  }
  if (threadIdx.x == 0) margin[blockIdx.x] = err[0] - err[1];
}

}  // namespace dfl

extern "C" int dflash_route_margin(const dflash_route *r, int32_t hidden, const float *rows, int32_t n, float *margin,
                                   void *stream) {
  using namespace dfl;
  if (!r || !rows || !margin || n < 1) return dflash_fail(DFLASH_E_ARG, "route_margin: null pointer or no rows");
  if (hidden < 1 || hidden > 16384) return dflash_fail(DFLASH_E_ARG, "route_margin: hidden must be 1..16384");
  if (r->block_rank < 0 || r->block_rank > RT_RANK_MAX || r->chain_rank < 0 || r->chain_rank > RT_RANK_MAX)
    return dflash_fail(DFLASH_E_ARG, "route_margin: a rank must be 0..256");
  if (!r->block_mean || !r->chain_mean || (r->block_rank && !r->block_basis) || (r->chain_rank && !r->chain_basis))
    return dflash_fail(DFLASH_E_ARG, "route_margin: a null mean or basis");
  RouteArgs A;
  A.mean[0] = (const __half *)r->chain_mean;
  A.basis[0] = (const __half *)r->chain_basis;
  A.rank[0] = r->chain_rank;
  A.mean[1] = (const __half *)r->block_mean;
  A.basis[1] = (const __half *)r->block_basis;
  A.rank[1] = r->block_rank;
  const size_t smem = ((size_t)hidden + RT_RANK_MAX) * sizeof(float);
  static PerDevice configured;
  cudaError_t e = smem_limit(k_route_margin, (int)smem, configured);
  if (e == cudaSuccess)
    e = launch_pdl(k_route_margin, dim3((unsigned)n), dim3(RT_THREADS), smem, (cudaStream_t)stream, 1, rows, hidden, A,
                   margin);
  if (e != cudaSuccess) return dflash_fail(DFLASH_E_CUDA, std::string("route_margin: ") + cudaGetErrorString(e));
  return DFLASH_OK;
}

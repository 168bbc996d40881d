// Row-wise stages of the drafter pass: RMSNorm, the grouped causal row
// convolution (both stages), the per-head q/k norm with the rotation, SiLU.
// Cited passages: cortiq-engine src/cortiq_engine/dflash.rs, `rms`,
// `Drafter::conv`, `Drafter::rotate`, `Drafter::mlp`, `Drafter::block`.
#include "common.cuh"
#include "kernels.h"

namespace dfl {

// ---------------------------------------------------------------- rms
// x * (mean(x^2) + eps)^-1/2 * w, one CTA per row.
__global__ void k_rmsnorm(const float *__restrict__ x, const float *__restrict__ w, float *__restrict__ out, int hs,
                          float eps, int block, int keep_from, int keep_to) {
  const int t = blockIdx.x;
  int orow = t;
  if (keep_from >= 0) {
    const int s = t / block, r = t % block;
    if (r < keep_from || r > keep_to) return;
    orow = s * (keep_to - keep_from + 1) + (r - keep_from);
  }
  const float *xr = x + (int64_t)t * hs;
  float ss = 0.f;
  for (int i = threadIdx.x; i < hs; i += blockDim.x) ss = fmaf(xr[i], xr[i], ss);
  __shared__ float red[32];
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    v = warp_sum(v);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float s = 1.0f / sqrtf(red[0] / (float)hs + eps);
  float *o = out + (int64_t)orow * hs;
  for (int i = threadIdx.x; i < hs; i += blockDim.x) o[i] = xr[i] * s * w[i];
}

cudaError_t rmsnorm(const float *x, const float *w, float *out, int T, int hs, float eps, int block, int keep_from,
                    int keep_to, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  k_rmsnorm<<<T, 256, 0, st>>>(x, w, out, hs, eps, block, keep_from, keep_to);
  count_launch(1);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- row convolution
// y[t][i] = sum_{o <= min(kn-1, t % block)} (base[stage][o][i] + d[t][stage][o][i/gs]) * x[t-o][i]
template <int STAGE>
__global__ void k_conv(const float *__restrict__ x, const float *__restrict__ d, const float *__restrict__ base,
                       float *__restrict__ y, int hs, int kn, int gs, int block) {
  const int t = blockIdx.y;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= hs) return;
  const int groups = hs / gs, g = i / gs;
  const int r = t % block;
  const float *dr = d + (int64_t)t * (2 * kn * groups) + STAGE * kn * groups;
  const float *br = base + (int64_t)STAGE * kn * hs;
  float acc = 0.f;
  const int nmax = min(kn, r + 1);
  for (int o = 0; o < nmax; ++o) acc = fmaf(br[(int64_t)o * hs + i] + dr[o * groups + g], x[(int64_t)(t - o) * hs + i], acc);
  if (STAGE == 0) y[(int64_t)t * hs + i] = acc;
  else y[(int64_t)t * hs + i] += acc;
}

cudaError_t conv_stage0(const float *x, const float *d, const float *base, float *y, int T, int hs, int kn, int gs,
                        int block, cudaStream_t st) {
  dim3 grid((hs + 255) / 256, T);
  k_conv<0><<<grid, 256, 0, st>>>(x, d, base, y, hs, kn, gs, block);
  count_launch(1);
  return cudaGetLastError();
}

cudaError_t conv_stage1_residual(const float *x, const float *d, const float *base, float *h, int T, int hs, int kn,
                                 int gs, int block, cudaStream_t st) {
  dim3 grid((hs + 255) / 256, T);
  k_conv<1><<<grid, 256, 0, st>>>(x, d, base, h, hs, kn, gs, block);
  count_launch(1);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- head norm + rotation
struct PosArgs {
  int64_t pos0[MAX_BATCH];
  float inv[64];  // inv_freq, head_dim <= 128
};

// One warp normalises one head of HD values at p (weight w) and, if rotary,
// rotates it to `pos`. HD/32 values per lane: lane owns i = lane + 32m
// (m < HD/64) of the low half and its partner i + HD/2.
template <int HD>
__device__ __forceinline__ void norm_rope_head(float *__restrict__ p, const float *__restrict__ w, float eps,
                                               bool rotary, int64_t pos, const float *inv, int lane) {
  constexpr int M = HD / 64;  // pairs per lane
  float lo[M], hi[M];
  float ss = 0.f;
#pragma unroll
  for (int m = 0; m < M; ++m) {
    lo[m] = p[lane + 32 * m];
    hi[m] = p[lane + 32 * m + HD / 2];
    ss = fmaf(lo[m], lo[m], ss);
    ss = fmaf(hi[m], hi[m], ss);
  }
  ss = warp_sum(ss);
  const float s = 1.0f / sqrtf(ss / (float)HD + eps);
#pragma unroll
  for (int m = 0; m < M; ++m) {
    lo[m] = lo[m] * s * w[lane + 32 * m];
    hi[m] = hi[m] * s * w[lane + 32 * m + HD / 2];
  }
  if (rotary) {
    const float fp = (float)pos;
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const float ang = __fmul_rn(fp, inv[lane + 32 * m]);
      float sn, cs;
      sincosf(ang, &sn, &cs);
      const float a = lo[m], b = hi[m];
      lo[m] = a * cs - b * sn;
      hi[m] = b * cs + a * sn;
    }
  }
#pragma unroll
  for (int m = 0; m < M; ++m) {
    p[lane + 32 * m] = lo[m];
    p[lane + 32 * m + HD / 2] = hi[m];
  }
}

// One warp per (row, head).
template <int HD>
__global__ void k_head_norm_rope(float *__restrict__ x, int ld, const float *__restrict__ w, int T, int heads,
                                 float eps, int rotary, PosArgs pa,
                                 int use_pos0, int block, int64_t pos_base) {
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= T * heads) return;
  const int t = wid / heads, h = wid % heads;
  const int64_t pos = use_pos0 ? pa.pos0[t / block] + (t % block) : pos_base + t;
  norm_rope_head<HD>(x + (int64_t)t * ld + h * HD, w, eps, rotary != 0, pos, pa.inv, lane);
}

struct CtxRope {
  float *k[64];
  const float *w[64];
  int rotary[64];
  float inv[64];
};

// One warp per (row, head) of layer blockIdx.y's context K.
template <int HD>
__global__ void k_ctx_norm_rope(CtxRope R, int T, int heads, float eps, int64_t pos_base) {
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= T * heads) return;
  const int l = blockIdx.y;
  const int t = wid / heads, h = wid % heads;
  norm_rope_head<HD>(R.k[l] + ((int64_t)t * heads + h) * HD, R.w[l], eps, R.rotary[l] != 0, pos_base + t, R.inv, lane);
}

cudaError_t ctx_norm_rope(float *const *k, const float *const *w, const int *rotary, int nlayers, int T, int heads,
                          int hd, float eps, const float *inv_freq, int64_t pos_base, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (nlayers < 1 || nlayers > 64) return cudaErrorInvalidValue;
  CtxRope R{};
  for (int l = 0; l < nlayers; ++l) {
    R.k[l] = k[l];
    R.w[l] = w[l];
    R.rotary[l] = rotary[l];
  }
  for (int i = 0; i < 64; ++i) R.inv[i] = i < hd / 2 ? inv_freq[i] : 0.f;
  const int warps = T * heads;
  dim3 grid((unsigned)((warps * 32 + 255) / 256), nlayers);
  if (hd == 128) k_ctx_norm_rope<128><<<grid, 256, 0, st>>>(R, T, heads, eps, pos_base);
  else if (hd == 64) k_ctx_norm_rope<64><<<grid, 256, 0, st>>>(R, T, heads, eps, pos_base);
  else return cudaErrorInvalidValue;
  count_launch(1);
  return cudaGetLastError();
}

cudaError_t head_norm_rope(float *x, int ld, const float *w, const float *inv_freq, int T, int heads, int hd,
                           float eps, bool rotary, const int64_t *pos0, int nseq, int block, int64_t pos_base,
                           cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (hd > 128) return cudaErrorInvalidValue;
  PosArgs pa;
  for (int i = 0; i < MAX_BATCH; ++i) pa.pos0[i] = (pos0 && i < nseq) ? pos0[i] : 0;
  for (int i = 0; i < 64; ++i) pa.inv[i] = i < hd / 2 ? inv_freq[i] : 0.f;
  const int warps = T * heads;
  const unsigned grid = (unsigned)((warps * 32 + 255) / 256);
  if (hd == 128)
    k_head_norm_rope<128><<<grid, 256, 0, st>>>(x, ld, w, T, heads, eps, rotary, pa, pos0 != nullptr,
                                                block, pos_base);
  else if (hd == 64)
    k_head_norm_rope<64><<<grid, 256, 0, st>>>(x, ld, w, T, heads, eps, rotary, pa, pos0 != nullptr,
                                               block, pos_base);
  else
    return cudaErrorInvalidValue;
  count_launch(1);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- SiLU gate
__global__ void k_silu_mul(const float *__restrict__ g, const float *__restrict__ u, float *__restrict__ m, int64_t n) {
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float a = g[i];
  m[i] = a / (1.0f + expf(-a)) * u[i];
}

cudaError_t silu_mul(const float *g, const float *u, float *m, int64_t n, cudaStream_t st) {
  k_silu_mul<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(g, u, m, n);
  count_launch(1);
  return cudaGetLastError();
}

}  // namespace dfl

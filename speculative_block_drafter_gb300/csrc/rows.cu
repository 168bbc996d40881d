// Row-wise stages of the drafter pass: RMSNorm, the grouped causal row
// convolution (both stages), the per-head q/k norm with the rotation, SiLU.
// Cited passages: cortiq-engine src/cortiq_engine/dflash.rs, `rms`,
// `Drafter::conv`, `Drafter::rotate`, `Drafter::mlp`, `Drafter::block`.
#include "common.cuh"
#include "kernels.h"

namespace dfl {

// ---------------------------------------------------------------- rms
// x * (mean(x^2) + eps)^-1/2 * w, one CTA per row. V4: rows, weight and output
// 16-byte aligned and hs a multiple of 4 (float4 accesses, the row kept in
// registers between the two passes when it fits).
constexpr int RMS_THREADS = 256;
constexpr int RMS_KEEP = 8;  // float4 a thread keeps: rows up to 8192

__device__ __forceinline__ float block_sum(float v, float *red) {
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    t = warp_sum(t);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  return red[0];
}

template <bool V4>
__global__ void __launch_bounds__(RMS_THREADS) k_rmsnorm(const float *__restrict__ x, const float *__restrict__ w,
                                                         float *__restrict__ out, int hs, float eps, int block,
                                                         int keep_from, int keep_to) {
  pdl_wait();
  const int t = blockIdx.x;
  int orow = t;
  if (keep_from >= 0) {
    const int s = t / block, r = t % block;
    if (r < keep_from || r > keep_to) return;
    orow = s * (keep_to - keep_from + 1) + (r - keep_from);
  }
  __shared__ float red[32];
  const float *xr = x + (int64_t)t * hs;
  float *o = out + (int64_t)orow * hs;
  if (V4) {
    const int n4 = hs / 4;
    const float4 *x4 = (const float4 *)xr;
    float4 keep[RMS_KEEP];
    float ss = 0.f;
#pragma unroll
    for (int m = 0; m < RMS_KEEP; ++m) {
      const int i = threadIdx.x + m * RMS_THREADS;
      keep[m] = i < n4 ? x4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
      ss = fmaf(keep[m].x, keep[m].x, fmaf(keep[m].y, keep[m].y, fmaf(keep[m].z, keep[m].z, fmaf(keep[m].w, keep[m].w, ss))));
    }
    for (int i = threadIdx.x + RMS_KEEP * RMS_THREADS; i < n4; i += RMS_THREADS) {
      const float4 v = x4[i];
      ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
    }
    const float sc = 1.0f / sqrtf(block_sum(ss, red) / (float)hs + eps);
    const float4 *w4 = (const float4 *)w;
    float4 *o4 = (float4 *)o;
#pragma unroll
    for (int m = 0; m < RMS_KEEP; ++m) {
      const int i = threadIdx.x + m * RMS_THREADS;
      if (i < n4) {
        const float4 g = w4[i];
        o4[i] = make_float4(keep[m].x * sc * g.x, keep[m].y * sc * g.y, keep[m].z * sc * g.z, keep[m].w * sc * g.w);
      }
    }
    for (int i = threadIdx.x + RMS_KEEP * RMS_THREADS; i < n4; i += RMS_THREADS) {
      const float4 v = x4[i], g = w4[i];
      o4[i] = make_float4(v.x * sc * g.x, v.y * sc * g.y, v.z * sc * g.z, v.w * sc * g.w);
    }
  } else {
    float ss = 0.f;
    for (int i = threadIdx.x; i < hs; i += RMS_THREADS) ss = fmaf(xr[i], xr[i], ss);
    const float sc = 1.0f / sqrtf(block_sum(ss, red) / (float)hs + eps);
    for (int i = threadIdx.x; i < hs; i += RMS_THREADS) o[i] = xr[i] * sc * w[i];
  }
}

cudaError_t rmsnorm(const float *x, const float *w, float *out, int T, int hs, float eps, int block, int keep_from,
                    int keep_to, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  const bool v4 = (hs % 4 == 0) && ((((uintptr_t)x) | ((uintptr_t)w) | ((uintptr_t)out)) & 15) == 0;
  if (v4)
    return launch_pdl(k_rmsnorm<true>, dim3(T), dim3(RMS_THREADS), 0, st, 1, x, w, out, hs, eps, block, keep_from,
                      keep_to);
  return launch_pdl(k_rmsnorm<false>, dim3(T), dim3(RMS_THREADS), 0, st, 1, x, w, out, hs, eps, block, keep_from,
                    keep_to);
}

// ---------------------------------------------------------------- row convolution
// y[t][i] = sum_{o <= min(kn-1, t % block)} (base[stage][o][i] + d[t][stage][o][i/gs]) * x[t-o][i]
template <int STAGE>
__global__ void k_conv(const float *__restrict__ x, const float *__restrict__ d, const float *__restrict__ base,
                       float *__restrict__ y, int hs, int kn, int gs, int block) {
  pdl_wait();
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
  return launch_pdl(k_conv<0>, grid, dim3(256), 0, st, 1, x, d, base, y, hs, kn, gs, block);
}

cudaError_t conv_stage1_residual(const float *x, const float *d, const float *base, float *h, int T, int hs, int kn,
                                 int gs, int block, cudaStream_t st) {
  dim3 grid((hs + 255) / 256, T);
  return launch_pdl(k_conv<1>, grid, dim3(256), 0, st, 1, x, d, base, h, hs, kn, gs, block);
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
  pdl_wait();
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
  pdl_wait();
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
  if (hd == 128) return launch_pdl(k_ctx_norm_rope<128>, grid, dim3(256), 0, st, 1, R, T, heads, eps, pos_base);
  if (hd == 64) return launch_pdl(k_ctx_norm_rope<64>, grid, dim3(256), 0, st, 1, R, T, heads, eps, pos_base);
  return cudaErrorInvalidValue;
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
  const int up0 = pos0 != nullptr;
  if (hd == 128)
    return launch_pdl(k_head_norm_rope<128>, dim3(grid), dim3(256), 0, st, 1, x, ld, w, T, heads, eps, (int)rotary, pa,
                      up0, block, pos_base);
  if (hd == 64)
    return launch_pdl(k_head_norm_rope<64>, dim3(grid), dim3(256), 0, st, 1, x, ld, w, T, heads, eps, (int)rotary, pa,
                      up0, block, pos_base);
  return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------- SiLU gate
__global__ void k_silu_mul(const float *__restrict__ g, const float *__restrict__ u, float *__restrict__ m, int64_t n) {
  pdl_wait();
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float a = g[i];
  m[i] = a / (1.0f + expf(-a)) * u[i];
}

cudaError_t silu_mul(const float *g, const float *u, float *m, int64_t n, cudaStream_t st) {
  return launch_pdl(k_silu_mul, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, 1, g, u, m, n);
}

}  // namespace dfl

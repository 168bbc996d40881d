// Row-wise stages of the drafter pass: RMSNorm, the grouped causal row
// convolution (both stages), the per-head q/k norm with the rotation, SiLU.
// Cited passages: cortiq-engine src/cortiq_engine/dflash.rs, `rms`,
// `Drafter::conv`, `Drafter::rotate`, `Drafter::mlp`, `Drafter::block`.
#include <algorithm>

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
__device__ __forceinline__ void norm_rope_regs(float (&lo)[HD / 64], float (&hi)[HD / 64], const float *__restrict__ w,
                                               float eps, bool rotary, int64_t pos, const float *inv, int lane) {
  constexpr int M = HD / 64;  // pairs per lane
  float ss = 0.f;
#pragma unroll
  for (int m = 0; m < M; ++m) {
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
}

template <int HD>
__device__ __forceinline__ void norm_rope_head(float *__restrict__ p, const float *__restrict__ w, float eps,
                                               bool rotary, int64_t pos, const float *inv, int lane) {
  constexpr int M = HD / 64;
  float lo[M], hi[M];
#pragma unroll
  for (int m = 0; m < M; ++m) {
    lo[m] = p[lane + 32 * m];
    hi[m] = p[lane + 32 * m + HD / 2];
  }
  norm_rope_regs<HD>(lo, hi, w, eps, rotary, pos, inv, lane);
#pragma unroll
  for (int m = 0; m < M; ++m) {
    p[lane + 32 * m] = lo[m];
    p[lane + 32 * m + HD / 2] = hi[m];
  }
}

// This file's device error word: DFL_ERR_RANGE when a K or V value written to
// a cache was not finite or beyond the range of the cache's f16 values (it
// then reads as infinity).
static __device__ unsigned int g_rows_error = 0;

// The cache formats (per row and KV head). PL = 2: two f16 planes, hi[HD] then
// lo[HD], hi = x with its low 13 mantissa bits cleared (exact below 65,536 in
// magnitude), lo = f16(x - hi); hi + lo carries about 21 bits of x. PL = 1:
// one f16 plane, f16(x) rounded to nearest (11 bits; infinite from 65,520).
template <int PL>
__device__ __forceinline__ void kv_pair(float x, __half &h, __half &l, bool &bad) {
  if constexpr (PL == 2) {
    const float t = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
    h = __float2half_rn(t);
    l = __float2half_rn(x - t);
    bad |= !(fabsf(x) < 65536.f);
  } else {
    h = __float2half_rn(x);
    bad |= !(fabsf(x) < 65520.f);
  }
}
__device__ __forceinline__ void flag_range(bool bad) {
  if (bad) atomicOr(&g_rows_error, DFL_ERR_RANGE);
}
// A head row into the cache format at dst (lane owns i = lane + 32m and i + HD/2).
template <int HD, int PL>
__device__ __forceinline__ void store_kv(__half *__restrict__ dst, const float (&lo)[HD / 64],
                                         const float (&hi)[HD / 64], int lane) {
  bool bad = false;
#pragma unroll
  for (int m = 0; m < HD / 64; ++m) {
    __half h, l;
    kv_pair<PL>(lo[m], h, l, bad);
    dst[lane + 32 * m] = h;
    if (PL == 2) dst[HD + lane + 32 * m] = l;
    kv_pair<PL>(hi[m], h, l, bad);
    dst[lane + 32 * m + HD / 2] = h;
    if (PL == 2) dst[HD + lane + 32 * m + HD / 2] = l;
  }
  flag_range(bad);
}

struct CtxPlanes {
  const float *k[64], *v[64];   // per layer f32 [T][heads][HD]: the settle's K and V, or imported rows
  __half *ck[64], *cv[64];      // per layer: the cache (row r at ck + r * heads * PL * HD)
  const float *w[64];           // k norms
  int rotary[64];
  int ring[64];                 // 0: a linear cache (row = at + t); else the ring's rows C
  int mirror[64];               // ring rows below this are also written C rows further on
  float inv[64];
};

// E consecutive floats (one vector load when E == 2).
template <int E>
__device__ __forceinline__ void load_e(const float *__restrict__ p, float (&v)[E]) {
  if constexpr (E == 2) {
    const float2 a = *(const float2 *)p;
    v[0] = a.x;
    v[1] = a.y;
  } else {
#pragma unroll
    for (int j = 0; j < E; ++j) v[j] = p[j];
  }
}
// E consecutive halves (one 4-byte store when E == 2).
template <int E>
__device__ __forceinline__ void store_e(__half *p, const __half (&v)[E]) {
  if constexpr (E == 2) {
    *(__half2 *)p = __halves2half2(v[0], v[1]);
  } else {
#pragma unroll
    for (int j = 0; j < E; ++j) p[j] = v[j];
  }
}

// E consecutive elements of each half of a head into the cache format at dst.
template <int HD, int PL, int E>
__device__ __forceinline__ void store_kv_e(__half *__restrict__ dst, const float (&x0)[E], const float (&x1)[E], int i0,
                                           bool &bad) {
  __half h[E], l[E];
#pragma unroll
  for (int j = 0; j < E; ++j) kv_pair<PL>(x0[j], h[j], l[j], bad);
  store_e<E>(dst + i0, h);
  if (PL == 2) store_e<E>(dst + HD + i0, l);
#pragma unroll
  for (int j = 0; j < E; ++j) kv_pair<PL>(x1[j], h[j], l[j], bad);
  store_e<E>(dst + HD / 2 + i0, h);
  if (PL == 2) store_e<E>(dst + HD + HD / 2 + i0, l);
}

// One warp per (row t, head) of layer blockIdx.y: with `norm`, the head's K
// normalised and rotated to pos_base + t (a settle); without, K taken as given
// (imported rows); then K and V into the cache row at + t, or, for a ring of C
// rows, into row (at + t) % C (and C rows further on when that is below the
// layer's mirror). In a ring, rows that a later row of the same call replaces
// (t < T - C) are not written, so that no two warps write one row. A lane
// holds E = HD/64 consecutive elements of each half of the head, i = E*lane + j
// and i + HD/2 (the rotation's pairs), so that its loads and stores are vectors
// and both rows' loads are in flight together.
template <int HD, int PL>
__global__ void k_ctx_planes(CtxPlanes P, int T, int heads, float eps, int64_t pos_base, int64_t at, int norm) {
  pdl_wait();
  // the next settle's packing of its taps (which needs nothing of this) may run
  // meanwhile; every kernel after this one waits for it before touching its data
  pdl_trigger();
  constexpr int E = HD / 64;
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= T * heads) return;
  const int l = blockIdx.y;
  const int t = wid / heads, hh = wid - t * heads;
  const int C = P.ring[l];
  int64_t row = at + t;
  if (C > 0) {
    if (t < T - C) return;
    row %= C;
  }
  const int64_t off = (int64_t)wid * HD;  // (t * heads + h) * HD
  const int i0 = E * lane;
  float k0[E], k1[E], v0[E], v1[E];
  load_e<E>(P.k[l] + off + i0, k0);
  load_e<E>(P.k[l] + off + HD / 2 + i0, k1);
  load_e<E>(P.v[l] + off + i0, v0);
  load_e<E>(P.v[l] + off + HD / 2 + i0, v1);
  if (norm) {
    float w0[E], w1[E];  // the norm's weights: plain loads (the caller's vector is only 4-byte aligned)
#pragma unroll
    for (int j = 0; j < E; ++j) {
      w0[j] = P.w[l][i0 + j];
      w1[j] = P.w[l][HD / 2 + i0 + j];
    }
    // K: the per-head RMS norm, then the rotation
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < E; ++j) {
      ss = fmaf(k0[j], k0[j], ss);
      ss = fmaf(k1[j], k1[j], ss);
    }
    ss = warp_sum(ss);
    const float s = 1.0f / sqrtf(ss / (float)HD + eps);
#pragma unroll
    for (int j = 0; j < E; ++j) {
      k0[j] = k0[j] * s * w0[j];
      k1[j] = k1[j] * s * w1[j];
    }
    if (P.rotary[l]) {
      const float fp = (float)(pos_base + t);
#pragma unroll
      for (int j = 0; j < E; ++j) {
        const float ang = __fmul_rn(fp, P.inv[i0 + j]);
        float sn, cs;
        sincosf(ang, &sn, &cs);
        const float a = k0[j], b = k1[j];
        k0[j] = a * cs - b * sn;
        k1[j] = b * cs + a * sn;
      }
    }
  }
  bool bad = false;
  for (int copy = 0; copy < 2; ++copy) {
    const int64_t r = row + (int64_t)copy * C;
    const int64_t dst = (r * heads + hh) * PL * HD;
    store_kv_e<HD, PL, E>(P.ck[l] + dst, k0, k1, i0, bad);
    store_kv_e<HD, PL, E>(P.cv[l] + dst, v0, v1, i0, bad);
    if (C == 0 || row >= P.mirror[l]) break;
  }
  flag_range(bad);
}

cudaError_t ctx_planes(const CtxWrite &W, int nlayers, int T, int heads, int hd, int planes, float eps,
                       const float *inv_freq, int64_t pos_base, int64_t at, bool norm, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (nlayers < 1 || nlayers > 64 || (planes != 1 && planes != 2)) return cudaErrorInvalidValue;
  CtxPlanes P{};
  for (int l = 0; l < nlayers; ++l) {
    P.k[l] = W.k[l];
    P.v[l] = W.v[l];
    P.ck[l] = W.ck[l];
    P.cv[l] = W.cv[l];
    P.w[l] = W.w[l];
    P.rotary[l] = W.rotary[l];
    P.ring[l] = W.ring[l];
    P.mirror[l] = W.mirror[l];
  }
  for (int i = 0; i < 64; ++i) P.inv[i] = i < hd / 2 ? inv_freq[i] : 0.f;
  const int warps = T * heads;
  dim3 grid((unsigned)((warps * 32 + 255) / 256), nlayers);
  const int nm = norm ? 1 : 0;
  if (hd == 128 && planes == 2)
    return launch_pdl(k_ctx_planes<128, 2>, grid, dim3(256), 0, st, 1, P, T, heads, eps, pos_base, at, nm);
  if (hd == 128)
    return launch_pdl(k_ctx_planes<128, 1>, grid, dim3(256), 0, st, 1, P, T, heads, eps, pos_base, at, nm);
  if (hd == 64 && planes == 2)
    return launch_pdl(k_ctx_planes<64, 2>, grid, dim3(256), 0, st, 1, P, T, heads, eps, pos_base, at, nm);
  if (hd == 64)
    return launch_pdl(k_ctx_planes<64, 1>, grid, dim3(256), 0, st, 1, P, T, heads, eps, pos_base, at, nm);
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


// ---------------------------------------------------------------- fused producers of a GEMM's token tiles
// Each writes its result straight into the packed token tiles of the GEMM that
// follows (PackDst) and, when that GEMM will split its k-range, clears the
// GEMM's outputs (ZeroSet) with its blocks past the work grid. Threads own 8
// consecutive columns of a row.

constexpr int FP_THREADS = 256;
constexpr int FP_KEEP = 4;  // 8-column groups a thread keeps between the two passes of a row past 8192 columns

__device__ __forceinline__ void load8(const float *p, float (&v)[8]) {
  const float4 a = ((const float4 *)p)[0], b = ((const float4 *)p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void store8(float *p, const float (&v)[8]) {
  ((float4 *)p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  ((float4 *)p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// Stage 1 of the row convolution with the residual for 8 channels i0.. of row t:
// h[t][i] += sum_{o <= min(kn-1, t % block)} (base[1][o][i] + d[t][1][o][i/gs]) * x[t-o][i].
__device__ __forceinline__ void conv1_8(const float *__restrict__ x, const float *__restrict__ d,
                                        const float *__restrict__ base, float (&h)[8], int t, int i0, int hs, int kn,
                                        int gs, int block) {
  const int groups = hs / gs, r = t % block;
  const float *dr = d + (int64_t)t * (2 * kn * groups) + kn * groups;
  const float *br = base + (int64_t)kn * hs;
  const int nmax = min(kn, r + 1);
#pragma unroll 4
  for (int o = 0; o < nmax; ++o) {  // unrolled: the taps' loads go out together
    float xv[8], bv[8];
    load8(x + (int64_t)(t - o) * hs + i0, xv);
    load8(br + (int64_t)o * hs + i0, bv);
    if (gs % 8 == 0) {
      const float dv = dr[o * groups + i0 / gs];
#pragma unroll
      for (int e = 0; e < 8; ++e) h[e] = fmaf(bv[e] + dv, xv[e], h[e]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) h[e] = fmaf(bv[e] + dr[o * groups + (i0 + e) / gs], xv[e], h[e]);
    }
  }
}

// One CTA per row t (blocks >= T clear). If `conv` is set, first h[t] += the
// stage-1 convolution of (cx, cd, cbase) (the residual); then x = rms(h[t], w)
// into xout (if set) and into the token tiles at the row's packed index
// (rows outside [keep_from, keep_to] of their block are left out, packed per
// sequence, when keep_from >= 0).
template <int KEEP>
__global__ void __launch_bounds__(1024) k_rms_pack(float *__restrict__ h, const float *__restrict__ cx,
                                                         const float *__restrict__ cd, const float *__restrict__ cbase,
                                                         int kn, int gs, const float *__restrict__ w,
                                                         float *__restrict__ xout, int T, int hs, float eps, int block,
                                                         int keep_from, int keep_to, PackDst P, ZeroSet Z) {
  pdl_wait();
  pdl_trigger();  // the GEMM this feeds may fetch its weights meanwhile
  if ((int)blockIdx.x >= T) {
    zero_set_clear(Z, blockIdx.x - T, gridDim.x - T);
    return;
  }
  const int t = blockIdx.x;
  const int ng = hs / 8, nt = blockDim.x;
  float v[KEEP][8], w0[8];
  float ss = 0.f;
  float *hr = h + (int64_t)t * hs;
  if ((int)threadIdx.x < ng) load8(w + 8 * threadIdx.x, w0);  // the first group's weights, fetched early
#pragma unroll
  for (int m = 0; m < KEEP; ++m) {
    const int gi = threadIdx.x + m * nt;
    if (gi < ng) {
      load8(hr + 8 * gi, v[m]);
      if (cx) {
        conv1_8(cx, cd, cbase, v[m], t, 8 * gi, hs, kn, gs, block);
        store8(hr + 8 * gi, v[m]);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(v[m][e], v[m][e], ss);
    }
  }
  __shared__ float red[32];
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float q = threadIdx.x < (nt >> 5) ? red[threadIdx.x] : 0.f;
    q = warp_sum(q);
    if (threadIdx.x == 0) red[0] = q;
  }
  __syncthreads();
  const float sc = 1.0f / sqrtf(red[0] / (float)hs + eps);
  int orow = t;
  bool keep = true;
  if (keep_from >= 0) {
    const int sq = t / block, r = t % block;
    keep = r >= keep_from && r <= keep_to;
    orow = sq * (keep_to - keep_from + 1) + (r - keep_from);
  }
  if (!keep) return;
#pragma unroll
  for (int m = 0; m < KEEP; ++m) {
    const int gi = threadIdx.x + m * nt;
    if (gi < ng) {
      float o[8], wv[8];
      if (m == 0) {
#pragma unroll
        for (int e = 0; e < 8; ++e) wv[e] = w0[e];
      } else {
        load8(w + 8 * gi, wv);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = v[m][e] * sc * wv[e];
      if (xout) store8(xout + (int64_t)orow * hs + 8 * gi, o);
      pack_store8(P, orow, 8 * gi, o);
    }
  }
}

// Stage 0 of the row convolution into the token tiles: one thread per 8 channels of a row.
__global__ void __launch_bounds__(FP_THREADS) k_conv0_pack(const float *__restrict__ x, const float *__restrict__ d,
                                                           const float *__restrict__ base, int T, int hs, int kn,
                                                           int gs, int block, int work_blocks, PackDst P, ZeroSet Z) {
  pdl_wait();
  pdl_trigger();  // the GEMM this feeds may fetch its weights meanwhile
  if ((int)blockIdx.x >= work_blocks) {
    zero_set_clear(Z, blockIdx.x - work_blocks, gridDim.x - work_blocks);
    return;
  }
  const int ng = hs / 8;
  const int id = blockIdx.x * FP_THREADS + threadIdx.x;
  if (id >= T * ng) return;
  const int t = id / ng, i0 = 8 * (id - t * ng);
  const int groups = hs / gs, r = t % block;
  const float *dr = d + (int64_t)t * (2 * kn * groups);
  const int nmax = min(kn, r + 1);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int o = 0; o < nmax; ++o) {  // unrolled: the taps' loads go out together
    float xv[8], bv[8];
    load8(x + (int64_t)(t - o) * hs + i0, xv);
    load8(base + (int64_t)o * hs + i0, bv);
    if (gs % 8 == 0) {
      const float dv = dr[o * groups + i0 / gs];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(bv[e] + dv, xv[e], acc[e]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(bv[e] + dr[o * groups + (i0 + e) / gs], xv[e], acc[e]);
    }
  }
  pack_store8(P, t, i0, acc);
}

// m = silu(g) * u into the token tiles: one thread per 8 columns of a row.
__global__ void __launch_bounds__(FP_THREADS) k_silu_pack(const float *__restrict__ g, const float *__restrict__ u,
                                                          int T, int n, int work_blocks, PackDst P, ZeroSet Z) {
  pdl_wait();
  pdl_trigger();  // the GEMM this feeds may fetch its weights meanwhile
  if ((int)blockIdx.x >= work_blocks) {
    zero_set_clear(Z, blockIdx.x - work_blocks, gridDim.x - work_blocks);
    return;
  }
  const int ng = n / 8;
  const int id = blockIdx.x * FP_THREADS + threadIdx.x;
  if (id >= T * ng) return;
  const int t = id / ng, i0 = 8 * (id - t * ng);
  float gv[8], uv[8], m[8];
  load8(g + (int64_t)t * n + i0, gv);
  load8(u + (int64_t)t * n + i0, uv);
#pragma unroll
  for (int e = 0; e < 8; ++e) m[e] = gv[e] / (1.0f + expf(-gv[e])) * uv[e];
  pack_store8(P, t, i0, m);
}

// The block's q, k and v in one launch: q normalised and rotated in place; k
// normalised and rotated, and v as it is, written in the cache format
// [T][hk][PL][HD] (the attention's format) to kp and vp.
template <int HD, int PL>
__global__ void k_qk_norm_rope(float *__restrict__ q, int ldq, const float *__restrict__ wq, int hq,
                               const float *__restrict__ k, int ldk, const float *__restrict__ wk,
                               const float *__restrict__ v, int ldv, int hk, __half *__restrict__ kp,
                               __half *__restrict__ vp, int T, float eps, int rotary, PosArgs pa, int block) {
  pdl_wait();
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int nq = T * hq, nk = T * hk;
  if (wid >= nq + 2 * nk) return;
  const int kind = wid < nq ? 0 : wid < nq + nk ? 1 : 2;  // q, k, v
  const int w2 = kind == 0 ? wid : kind == 1 ? wid - nq : wid - nq - nk;
  const int heads = kind == 0 ? hq : hk;
  const int t = w2 / heads, h = w2 % heads;
  const int64_t pos = pa.pos0[t / block] + (t % block);
  if (kind == 0) {
    norm_rope_head<HD>(q + (int64_t)t * ldq + h * HD, wq, eps, rotary != 0, pos, pa.inv, lane);
    return;
  }
  const float *src = kind == 1 ? k + (int64_t)t * ldk + h * HD : v + (int64_t)t * ldv + h * HD;
  constexpr int M = HD / 64;
  float lo[M], hi[M];
#pragma unroll
  for (int m = 0; m < M; ++m) {
    lo[m] = src[lane + 32 * m];
    hi[m] = src[lane + 32 * m + HD / 2];
  }
  if (kind == 1) norm_rope_regs<HD>(lo, hi, wk, eps, rotary != 0, pos, pa.inv, lane);
  store_kv<HD, PL>((kind == 1 ? kp : vp) + ((int64_t)t * hk + h) * PL * HD, lo, hi, lane);
}

static unsigned zero_blocks_for(const ZeroSet &Z) {
  int64_t most = 0;
  for (int j = 0; j < Z.count; ++j) most = std::max<int64_t>(most, (int64_t)Z.n[j]);
  return Z.count ? (unsigned)std::min<int64_t>((most + 1023) / 1024, 128) : 0u;
}

cudaError_t rms_pack(float *h, const float *cx, const float *cd, const float *cbase, int kn, int gs, const float *w,
                     float *xout, int T, int hs, float eps, int block, int keep_from, int keep_to, const PackDst &P,
                     const ZeroSet &Z, cudaStream_t st) {
  // a thread per 8-column group of the row (at most FP_KEEP groups a thread)
  const int ng = hs / 8;
  const int nt = std::min(1024, std::max(32, (ng + 31) / 32 * 32));
  if (hs % 8 || ng > nt * FP_KEEP) return cudaErrorInvalidValue;
  // one 8-column group a thread up to 8192 columns (fewer live registers)
  return launch_pdl(ng <= nt ? k_rms_pack<1> : k_rms_pack<FP_KEEP>, dim3(T + zero_blocks_for(Z)), dim3(nt), 0, st, 1,
                    h, cx, cd, cbase, kn, gs, w, xout, T, hs, eps, block, keep_from, keep_to, P, Z);
}

cudaError_t conv0_pack(const float *x, const float *d, const float *base, int T, int hs, int kn, int gs, int block,
                       const PackDst &P, const ZeroSet &Z, cudaStream_t st) {
  if (hs % 8) return cudaErrorInvalidValue;
  const int work = (T * (hs / 8) + FP_THREADS - 1) / FP_THREADS;
  return launch_pdl(k_conv0_pack, dim3(work + zero_blocks_for(Z)), dim3(FP_THREADS), 0, st, 1, x, d, base, T, hs, kn,
                    gs, block, work, P, Z);
}

cudaError_t silu_pack(const float *g, const float *u, int T, int n, const PackDst &P, const ZeroSet &Z,
                      cudaStream_t st) {
  if (n % 8) return cudaErrorInvalidValue;
  const int work = (T * (n / 8) + FP_THREADS - 1) / FP_THREADS;
  return launch_pdl(k_silu_pack, dim3(work + zero_blocks_for(Z)), dim3(FP_THREADS), 0, st, 1, g, u, T, n, work, P, Z);
}

cudaError_t qk_norm_rope(float *q, int ldq, const float *wq, int hq, const float *k, int ldk, const float *wk,
                         const float *v, int ldv, int hk, __half *kp, __half *vp, const float *inv_freq, int T, int hd,
                         float eps, bool rotary, const int64_t *pos0, int nseq, int block, int planes,
                         cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (planes != 1 && planes != 2) return cudaErrorInvalidValue;
  PosArgs pa;
  for (int i = 0; i < MAX_BATCH; ++i) pa.pos0[i] = (pos0 && i < nseq) ? pos0[i] : 0;
  for (int i = 0; i < 64; ++i) pa.inv[i] = i < hd / 2 ? inv_freq[i] : 0.f;
  const int warps = T * (hq + 2 * hk);
  const unsigned grid = (unsigned)((warps * 32 + 255) / 256);
  auto kern = hd == 128 ? (planes == 2 ? k_qk_norm_rope<128, 2> : k_qk_norm_rope<128, 1>)
                        : (planes == 2 ? k_qk_norm_rope<64, 2> : k_qk_norm_rope<64, 1>);
  if (hd == 128 || hd == 64)
    return launch_pdl(kern, dim3(grid), dim3(256), 0, st, 1, q, ldq, wq, hq, k, ldk, wk, v, ldv, hk, kp, vp, T, eps,
                      (int)rotary, pa, block);
  return cudaErrorInvalidValue;
}

// This file's device error word (a value out of the cache planes' range).
cudaError_t rows_read_error(unsigned *out, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_rows_error, sizeof(unsigned));
  if (e == cudaSuccess && reset) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_rows_error, &zero, sizeof(unsigned));
  }
  return e;
}

}  // namespace dfl

// Weight-streaming GEMMs of the drafter: Y = X . W^T with few rows of X (a
// block's 16 rows, a settle's 256) against a four-bit or f16 weight matrix.
//
// The four-bit matrices are q/k/v/o/gate/up/down and the head; the f16 ones fc,
// the kernel projections and the selector's projection (cortiq-engine
// src/gpu_cuda/hyb/dflash.rs, module doc and `Dev::new`). The codes enter the
// tensor cores exactly (q in -7..7 is exact in f16) and each group's f16 scale
// multiplies the f32 partial sum of its columns, so the dequantisation is exact.
// Activations: for four-bit matrices, f32 rows as f16 hi + lo planes (about 22
// significant bits); for f16 matrices, the rows rounded to f16 (the card arm's
// `to_half` before its f16 GEMM).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace dfl {

constexpr int GW = 8;        // warps per CTA
constexpr int KC_MAX = 32;   // column tiles staged per CTA

// ---------------------------------------------------------------- packing

size_t int4_packed_bytes(int64_t rows, int64_t cols) { return (size_t)rows * cols / 2; }
size_t int4_scale_bytes(int64_t rows, int64_t cols, int group) {
  return (size_t)(rows / 16) * (cols / group) * 8 * 4;
}
size_t f16_packed_bytes(int64_t rows, int64_t cols) { return (size_t)rows * cols * 2; }

__constant__ int kNibbleElem[8] = {0, 2, 4, 6, 1, 3, 5, 7};

// (row, col) inside a tile of the A-fragment element e (0..7) of lane (g, c), column step j.
__device__ __forceinline__ void frag_pos(int e, int g, int c, int j, int &r, int &col) {
  r = g + 8 * ((e >> 1) & 1);
  col = j * 16 + 2 * c + (e & 1) + 8 * (e >> 2);
}

__global__ void k_pack_int4(const uint8_t *__restrict__ codes, int64_t rows, int64_t cols, uint4 *__restrict__ dst) {
  int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t KT = cols / 64;
  const int64_t total = (rows / 16) * KT * 32;
  if (t >= total) return;
  const int lane = (int)(t & 31);
  const int64_t tile = t >> 5;
  const int64_t rb = tile / KT, kt = tile % KT;
  const int g = lane >> 2, c = lane & 3;
  uint32_t out[4];
  for (int j = 0; j < 4; ++j) {
    uint32_t w = 0;
    for (int i = 0; i < 8; ++i) {
      int r, col;
      frag_pos(kNibbleElem[i], g, c, j, r, col);
      const int64_t row = rb * 16 + r, cc = kt * 64 + col;
      uint8_t byte = codes[row * (cols / 2) + cc / 2];
      uint32_t nib = (cc & 1) ? (byte >> 4) : (byte & 15);
      w |= nib << (4 * i);
    }
    out[j] = w;
  }
  dst[t] = make_uint4(out[0], out[1], out[2], out[3]);
}

__global__ void k_pack_scales(const uint16_t *__restrict__ scales, int64_t rows, int64_t ngroups,
                              uint32_t *__restrict__ dst) {
  int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = (rows / 16) * ngroups * 8;
  if (t >= total) return;
  const int g = (int)(t & 7);
  const int64_t rest = t >> 3;
  const int64_t rb = rest / ngroups, grp = rest % ngroups;
  uint32_t lo = scales[(rb * 16 + g) * ngroups + grp];
  uint32_t hi = scales[(rb * 16 + g + 8) * ngroups + grp];
  dst[t] = lo | (hi << 16);
}

__global__ void k_pack_f16(const uint16_t *__restrict__ src, int64_t rows, int64_t cols, uint4 *__restrict__ dst) {
  int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t KT = cols / 64;
  const int64_t total = (rows / 16) * KT * 4 * 32;
  if (t >= total) return;
  const int lane = (int)(t & 31);
  const int j = (int)((t >> 5) & 3);
  const int64_t tile = t >> 7;
  const int64_t rb = tile / KT, kt = tile % KT;
  const int g = lane >> 2, c = lane & 3;
  uint32_t out[4];
  for (int m = 0; m < 4; ++m) {
    const int64_t row = rb * 16 + g + 8 * (m & 1);
    const int64_t col = kt * 64 + j * 16 + 2 * c + 8 * (m >> 1);
    out[m] = (uint32_t)src[row * cols + col] | ((uint32_t)src[row * cols + col + 1] << 16);
  }
  dst[t] = make_uint4(out[0], out[1], out[2], out[3]);
}

__global__ void k_dequant_int4(const uint4 *__restrict__ w, const uint32_t *__restrict__ s, int64_t rows,
                               int64_t cols, int group, float *__restrict__ out) {
  int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t KT = cols / 64;
  const int64_t total = (rows / 16) * KT * 32;
  if (t >= total) return;
  const int lane = (int)(t & 31);
  const int64_t tile = t >> 5;
  const int64_t rb = tile / KT, kt = tile % KT;
  const int g = lane >> 2, c = lane & 3;
  const int64_t NG = cols / group;
  const uint4 v = w[t];
  const uint32_t words[4] = {v.x, v.y, v.z, v.w};
  for (int j = 0; j < 4; ++j) {
    uint32_t a[4];
    dequant8(words[j], a);
    for (int e = 0; e < 8; ++e) {
      int r, col;
      frag_pos(e, g, c, j, r, col);
      const int64_t cc = kt * 64 + col;
      const uint32_t sp = s[(rb * NG + cc / group) * 8 + g];
      const uint16_t sbits = (uint16_t)(r < 8 ? (sp & 0xFFFF) : (sp >> 16));
      const uint16_t qbits = (uint16_t)((e & 1) ? (a[e >> 1] >> 16) : (a[e >> 1] & 0xFFFF));
      const float q = __half2float(__ushort_as_half(qbits));
      const float sc = __half2float(__ushort_as_half(sbits));
      out[(rb * 16 + r) * cols + cc] = __fmul_rn(q, sc);
    }
  }
}

static inline unsigned nblocks(int64_t n, int b) { return (unsigned)((n + b - 1) / b); }

cudaError_t pack_int4(const uint8_t *codes, const uint16_t *scales, int64_t rows, int64_t cols, int group,
                      void *dst, void *dst_scales, cudaStream_t st) {
  int64_t n = (rows / 16) * (cols / 64) * 32;
  k_pack_int4<<<nblocks(n, 256), 256, 0, st>>>(codes, rows, cols, (uint4 *)dst);
  int64_t ns = (rows / 16) * (cols / group) * 8;
  k_pack_scales<<<nblocks(ns, 256), 256, 0, st>>>(scales, rows, cols / group, (uint32_t *)dst_scales);
  count_launch(2);
  return cudaGetLastError();
}

cudaError_t pack_f16(const uint16_t *src, int64_t rows, int64_t cols, void *dst, cudaStream_t st) {
  int64_t n = (rows / 16) * (cols / 64) * 128;
  k_pack_f16<<<nblocks(n, 256), 256, 0, st>>>(src, rows, cols, (uint4 *)dst);
  count_launch(1);
  return cudaGetLastError();
}

cudaError_t dequant_int4(const void *codes, const void *scales, int64_t rows, int64_t cols, int group,
                         float *out, cudaStream_t st) {
  int64_t n = (rows / 16) * (cols / 64) * 32;
  k_dequant_int4<<<nblocks(n, 256), 256, 0, st>>>((const uint4 *)codes, (const uint32_t *)scales, rows, cols,
                                                  group, out);
  count_launch(1);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- the GEMM

// Stage X[tok0 .. tok0+16)[col0 .. col0 + 16*nsteps) as B fragments in shared
// memory. Four-bit: per column step, 32 lanes x uint4 of hi, then 32 of lo.
// f16: per column step, 32 lanes x uint4. uint4 = (t0 r0, t0 r1, t1 r0, t1 r1),
// t = tokens 0-7 / 8-15, r = columns 2c,2c+1 / 2c+8,2c+9.
template <bool INT4>
__device__ __forceinline__ void stage_x(uint4 *sm, const float *__restrict__ X, int ldx, int T, int tok0, int col0,
                                        int nsteps) {
  for (int i = threadIdx.x; i < nsteps * 32; i += blockDim.x) {
    const int s = i >> 5, lane = i & 31, g = lane >> 2, c = lane & 3;
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int tok = tok0 + t * 8 + g;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int col = col0 + s * 16 + 2 * c + 8 * r;
        float2 v = make_float2(0.f, 0.f);
        if (tok < T) v = *reinterpret_cast<const float2 *>(X + (int64_t)tok * ldx + col);
        if (INT4) {
          split2(v.x, v.y, hi[t * 2 + r], lo[t * 2 + r]);
        } else {
          hi[t * 2 + r] = pack_half2(__float2half_rn(v.x), __float2half_rn(v.y));
        }
      }
    }
    if (INT4) {
      sm[(s * 2 + 0) * 32 + lane] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      sm[(s * 2 + 1) * 32 + lane] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    } else {
      sm[s * 32 + lane] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    }
  }
}

__device__ __forceinline__ uint4 ldg_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// out_mode: 0 store, 1 atomic add, 2 plain add (each element owned by one thread)
template <bool INT4, int NB, int PF>
__global__ void __launch_bounds__(GW * 32, INT4 ? 2 : 1) k_gemm(const uint4 *__restrict__ W, const uint32_t *__restrict__ S,
                                                  int group, int N, int K, const float *__restrict__ X, int ldx,
                                                  float *__restrict__ Y, int ldy, int T, int kc, int out_mode) {
  extern __shared__ uint4 sm[];
  constexpr int WV = INT4 ? 1 : 4;  // uint4 per lane per column tile
  const int KT = K / 64;
  const int tok0 = blockIdx.x * 16;
  const int kt0 = blockIdx.z * kc, kt1 = min(KT, kt0 + kc);
  if (kt0 >= kt1) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int RB = (N + 15) / 16;
  const int rb0 = (blockIdx.y * GW + warp) * NB;
  const bool active = rb0 < RB;
  const int NG = INT4 ? K / group : 0;

  const uint4 *wp[NB];
  bool live[NB];
#pragma unroll
  for (int i = 0; i < NB; ++i) {
    live[i] = rb0 + i < RB;
    const int rb = live[i] ? rb0 + i : (active ? rb0 : 0);
    wp[i] = W + ((int64_t)rb * KT) * (32 * WV) + lane;
  }

  // the first weight tiles are in flight while the activations are staged
  uint4 buf[PF][NB][WV];
#pragma unroll
  for (int p = 0; p < PF; ++p)
#pragma unroll
    for (int i = 0; i < NB; ++i)
#pragma unroll
      for (int v = 0; v < WV; ++v)
        buf[p][i][v] = (active && kt0 + p < kt1) ? ldg_stream(wp[i] + (int64_t)(kt0 + p) * (32 * WV) + v * 32)
                                                 : make_uint4(0, 0, 0, 0);

  stage_x<INT4>(sm, X, ldx, T, tok0, kt0 * 64, (kt1 - kt0) * 4);
  __syncthreads();
  if (!active) return;

  float acc[NB][2][4];
#pragma unroll
  for (int i = 0; i < NB; ++i)
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][t][e] = 0.f;

  for (int kt = kt0; kt < kt1; kt += PF) {
#pragma unroll
    for (int p = 0; p < PF; ++p) {
      const int ktp = kt + p;
      if (ktp < kt1) {
        uint4 cur[NB][WV];
#pragma unroll
        for (int i = 0; i < NB; ++i)
#pragma unroll
          for (int v = 0; v < WV; ++v) cur[i][v] = buf[p][i][v];
        if (ktp + PF < kt1) {
#pragma unroll
          for (int i = 0; i < NB; ++i)
#pragma unroll
            for (int v = 0; v < WV; ++v) buf[p][i][v] = ldg_stream(wp[i] + (int64_t)(ktp + PF) * (32 * WV) + v * 32);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int s = (ktp - kt0) * 4 + j;
          if (INT4) {
            const uint4 bh = sm[(s * 2 + 0) * 32 + lane];
            const uint4 bl = sm[(s * 2 + 1) * 32 + lane];
            const int grp = (ktp * 64 + j * 16) / group;
#pragma unroll
            for (int i = 0; i < NB; ++i) {
              const uint32_t word = j == 0 ? cur[i][0].x : j == 1 ? cur[i][0].y : j == 2 ? cur[i][0].z : cur[i][0].w;
              uint32_t a[4];
              dequant8(word, a);
              float t0[4] = {0.f, 0.f, 0.f, 0.f}, t1[4] = {0.f, 0.f, 0.f, 0.f};
              mma16816(t0, a, bh.x, bh.y);
              mma16816(t1, a, bh.z, bh.w);
              mma16816(t0, a, bl.x, bl.y);
              mma16816(t1, a, bl.z, bl.w);
              const int rb = live[i] ? rb0 + i : rb0;
              const uint32_t sp = __ldg(S + ((int64_t)rb * NG + grp) * 8 + g);
              const float s0 = __half2float(__ushort_as_half((uint16_t)(sp & 0xFFFF)));
              const float s1 = __half2float(__ushort_as_half((uint16_t)(sp >> 16)));
              acc[i][0][0] = fmaf(s0, t0[0], acc[i][0][0]);
              acc[i][0][1] = fmaf(s0, t0[1], acc[i][0][1]);
              acc[i][0][2] = fmaf(s1, t0[2], acc[i][0][2]);
              acc[i][0][3] = fmaf(s1, t0[3], acc[i][0][3]);
              acc[i][1][0] = fmaf(s0, t1[0], acc[i][1][0]);
              acc[i][1][1] = fmaf(s0, t1[1], acc[i][1][1]);
              acc[i][1][2] = fmaf(s1, t1[2], acc[i][1][2]);
              acc[i][1][3] = fmaf(s1, t1[3], acc[i][1][3]);
            }
          } else {
            const uint4 b = sm[s * 32 + lane];
#pragma unroll
            for (int i = 0; i < NB; ++i) {
              const uint4 av = cur[i][WV > 1 ? j : 0];
              const uint32_t a[4] = {av.x, av.y, av.z, av.w};
              mma16816(acc[i][0], a, b.x, b.y);
              mma16816(acc[i][1], a, b.z, b.w);
            }
          }
        }
      }
    }
  }

#pragma unroll
  for (int i = 0; i < NB; ++i) {
    if (!live[i]) continue;
    const int f0 = (rb0 + i) * 16 + g;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int n0 = tok0 + t * 8 + 2 * c;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int f = f0 + 8 * (e >> 1), n = n0 + (e & 1);
        if (n < T && f < N) {
          float *p = Y + (int64_t)n * ldy + f;
          const float v = acc[i][t][e];
          if (out_mode == 1) atomicAdd(p, v);
          else if (out_mode == 2) *p += v;
          else *p = v;
        }
      }
    }
  }
}

template <bool INT4, int NB, int PF>
static cudaError_t launch_gemm(const Gemm &a, int num_sms, cudaStream_t st) {
  const int KT = a.K / 64;
  const int RB = (a.N + 15) / 16;
  const int tx = (a.T + 15) / 16;
  const int gy = (RB + GW * NB - 1) / (GW * NB);
  const int64_t base = (int64_t)tx * gy;
  const int64_t want = 2 * (int64_t)num_sms;
  int splits = 1;
  if (base < want) splits = (int)std::min<int64_t>(KT, (want + base - 1) / base);
  int kc = (KT + splits - 1) / splits;
  kc = std::min(kc, KC_MAX);
  splits = (KT + kc - 1) / kc;
  int mode = 0;
  if (a.accumulate) {
    mode = splits > 1 ? 1 : 2;
  } else if (splits > 1) {
    mode = 1;
    cudaError_t e = cudaMemset2DAsync(a.Y, (size_t)a.ldy * 4, 0, (size_t)a.N * 4, a.T, st);
    if (e != cudaSuccess) return e;
  }
  const size_t smem = (size_t)kc * 4 * (INT4 ? 2 : 1) * 32 * sizeof(uint4);
  auto kern = k_gemm<INT4, NB, PF>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(KC_MAX * 4 * (INT4 ? 2 : 1) * 32 * sizeof(uint4)));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(tx, gy, splits);
  kern<<<grid, GW * 32, smem, st>>>((const uint4 *)a.w, (const uint32_t *)a.scales, a.group, a.N, a.K, a.X, a.ldx,
                                    a.Y, a.ldy, a.T, kc, mode);
  count_launch(1);
  return cudaGetLastError();
}

cudaError_t gemm_int4(const Gemm &g, int num_sms, cudaStream_t st) { return launch_gemm<true, 2, 4>(g, num_sms, st); }
cudaError_t gemm_f16(const Gemm &g, int num_sms, cudaStream_t st) { return launch_gemm<false, 1, 2>(g, num_sms, st); }

}  // namespace dfl

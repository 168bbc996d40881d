// Shared device helpers of the DFlash 2 drafter library (sm_103a).
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dfl {

// Bits of the library's device error word (dflash_device_error).
constexpr unsigned DFL_ERR_TIMEOUT = 1u;  // a kernel gave up a bounded wait
constexpr unsigned DFL_ERR_RANGE = 2u;    // a K/V value out of the cache planes' range

// ---------------------------------------------------------------- programmatic dependent launch
// Every kernel of the pass is launched so that it may start while the kernel
// before it in the stream finishes (launch_pdl). Such a kernel calls pdl_wait()
// before it touches any buffer an earlier kernel reads or writes (weights are
// never written during a pass and may be read before), in every thread and
// before any early return, so that the chain of waits orders the whole stream.
// pdl_trigger() lets the next kernel start before this one ends. Only the
// kernels that pack a GEMM's token tiles call it early (the GEMM then fetches
// its first weight tiles meanwhile); the GEMMs call it when their own work is
// done; the others not at all (the next kernel starts as they exit). A kernel
// started early shares the SMs with the one still running: a few heavy CTAs
// would be packed onto the SMs that happen to be free.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- small math
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
  return r;
}

__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// Eight nibbles (q + 8) -> the four f16x2 registers of an A fragment holding q,
// exactly: 0x6400 | n is the f16 1024 + n; 0x6400 | 16n is 1024 + 16n.
__device__ __forceinline__ void dequant8(uint32_t w, uint32_t (&a)[4]) {
  const uint32_t lo_mask = 0x000F000Fu, hi_mask = 0x00F000F0u, magic = 0x64006400u;
  const uint32_t k1032 = 0x64086408u;          // 1032 = 1024 + 8
  const uint32_t k1_16 = 0x2C002C00u;          // 1/16
  const uint32_t km72 = 0xD480D480u;           // -72 = -(1024/16 + 8)
  uint32_t w2 = w >> 8;
  a[0] = hsub2_u(lop3_and_or(w, lo_mask, magic), k1032);
  a[1] = hfma2_u(lop3_and_or(w, hi_mask, magic), k1_16, km72);
  a[2] = hsub2_u(lop3_and_or(w2, lo_mask, magic), k1032);
  a[3] = hfma2_u(lop3_and_or(w2, hi_mask, magic), k1_16, km72);
}

// D = A . B + C, m16n8k16, f16 inputs, f32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_half2(__half lo, __half hi) {
  return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

// f32 pair -> (hi, lo) f16 planes: hi = f16(x), lo = f16(x - hi).
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
  __half l0 = __float2half_rn(x0 - __half2float(h0)), l1 = __float2half_rn(x1 - __half2float(h1));
  hi = pack_half2(h0, h1);
  lo = pack_half2(l0, l1);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Order-preserving map of a float onto u32 (larger float -> larger integer).
__device__ __forceinline__ uint32_t f32_ordered(float f) {
  uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float f32_from_ordered(uint32_t u) {
  uint32_t b = (u & 0x80000000u) ? (u & 0x7fffffffu) : ~u;
  return __uint_as_float(b);
}

// Candidate key: larger value first, then the lower index first. 0 = no candidate.
__device__ __forceinline__ unsigned long long cand_key(float v, uint32_t idx) {
  return ((unsigned long long)f32_ordered(v) << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}
__device__ __forceinline__ uint32_t cand_index(unsigned long long k) { return 0xFFFFFFFFu - (uint32_t)k; }

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) { return a > b ? a : b; }
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// ---------------------------------------------------------------- packed token tiles
// Byte offset of (row r, 16-byte chunk c) in a K-major tile of 64 f16 per row, 128-byte swizzle.
__host__ __device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// ---------------------------------------------------------------- token tiles
// One 16-byte chunk (8 columns of one token row) of the packed token tiles:
// per (token tile tt, k-tile kt, plane p) TT rows x 64 columns f16, K-major
// with the 128-byte swizzle. Plane 0 = f16(x); plane 1 = f16(x - f16(x)).
// Chunk t < ceil(T/TT) * (K/64) * TT * 8; rows past T are zero.
// Its two halves, so that a caller can have several chunks' loads in flight
// before the stores: the 8 values of chunk t (zeros past T), then their store.
__device__ __forceinline__ void pack_chunk_load(const float *__restrict__ X, int ldx, int T, int K, int TT, int64_t t,
                                                float (&x)[8]) {
  const int KT = K / 64;
  const int c = (int)(t & 7);
  const int r = (int)((t >> 3) % TT);
  const int64_t rest = (t >> 3) / TT;
  const int kt = (int)(rest % KT);
  const int tt = (int)(rest / KT);
  const int tok = tt * TT + r;
  if (tok < T) {
    const float *src = X + (int64_t)tok * ldx + kt * 64 + c * 8;
    if ((((uintptr_t)src) & 15) == 0) {
      const float4 a = __ldg((const float4 *)src), b = __ldg((const float4 *)src + 1);
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
      x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = src[i];
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = 0.f;
  }
}
template <int PLANES>
__device__ __forceinline__ void pack_chunk_store(int K, int TT, int64_t t, const float (&x)[8],
                                                 uint4 *__restrict__ dst) {
  const int KT = K / 64;
  const int c = (int)(t & 7);
  const int r = (int)((t >> 3) % TT);
  const int64_t rest = (t >> 3) / TT;
  const int kt = (int)(rest % KT);
  const int tt = (int)(rest / KT);
  uint32_t hi[4], lo[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (PLANES == 2) {
      split2(x[2 * i], x[2 * i + 1], hi[i], lo[i]);
    } else {
      hi[i] = pack_half2(__float2half_rn(x[2 * i]), __float2half_rn(x[2 * i + 1]));
    }
  }
  const int64_t base = (((int64_t)tt * KT + kt) * PLANES) * TT * 8;  // in 16-byte chunks
  dst[base + sw128_off(r, c) / 16] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  if (PLANES == 2) dst[base + TT * 8 + sw128_off(r, c) / 16] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}
template <int PLANES>
__device__ __forceinline__ void pack_act_chunk(const float *__restrict__ X, int ldx, int T, int K, int TT,
                                               uint4 *__restrict__ dst, int64_t t) {
  float x[8];
  pack_chunk_load(X, ldx, T, K, TT, t, x);
  pack_chunk_store<PLANES>(K, TT, t, x, dst);
}

// A GEMM's packed token tiles as a producer kernel writes them: 8 consecutive
// columns of one token row at a time (the layout of pack_act_chunk).
struct PackDst {
  uint4 *dst;
  int TT;      // token rows a tile
  int planes;  // 1: f16(x); 2: hi and lo
  int KT;      // 64-column k-tiles
};
__device__ __forceinline__ void pack_store8(const PackDst &P, int tok, int col, const float (&x)[8]) {
  const int tt = tok / P.TT, r = tok - tt * P.TT, kt = col >> 6, c = (col & 63) >> 3;
  const int64_t base = ((int64_t)tt * P.KT + kt) * P.planes * P.TT * 8;
  uint32_t hi[4], lo[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (P.planes == 2) split2(x[2 * i], x[2 * i + 1], hi[i], lo[i]);
    else hi[i] = pack_half2(__float2half_rn(x[2 * i]), __float2half_rn(x[2 * i + 1]));
  }
  P.dst[base + sw128_off(r, c) / 16] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  if (P.planes == 2) P.dst[base + P.TT * 8 + sw128_off(r, c) / 16] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

// Outputs that the GEMM fed by a producer accumulates into when its k-range is
// split: the producer clears T rows of n floats of each (grid-stride over blocks).
constexpr int ZERO_MAX = 4;
struct ZeroSet {
  float *y[ZERO_MAX];
  int ldy[ZERO_MAX];
  int n[ZERO_MAX];
  int count;
  int T;
};
__device__ __forceinline__ void zero_set_clear(const ZeroSet &Z, int block, int nblocks) {
  for (int j = 0; j < Z.count; ++j)
    for (int t = 0; t < Z.T; ++t) {
      float *y = Z.y[j] + (int64_t)t * Z.ldy[j];
      for (int c = (block * blockDim.x + threadIdx.x) * 4; c < Z.n[j]; c += nblocks * blockDim.x * 4) {
        if (c + 3 < Z.n[j] && (((uintptr_t)(y + c)) & 15) == 0) *(float4 *)(y + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        else
          for (int e = 0; e < 4 && c + e < Z.n[j]; ++e) y[c + e] = 0.f;
      }
    }
}

}  // namespace dfl

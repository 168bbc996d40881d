// Shared device helpers of the DFlash 2 drafter library (sm_103a).
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dfl {

// ---------------------------------------------------------------- packed layouts
//
// Four-bit matrices [rows][cols]: tiles of 16 rows x 64 columns, 512 bytes,
// ordered [row block][column tile]. Inside a tile, lane l (0..31) owns 16 bytes:
// u32 j (0..3) is the mma.m16n8k16 A fragment of the lane for columns
// 16j..16j+15, eight nibbles (q + 8) in the order a0 a2 a4 a6 a1 a3 a5 a7, where
// with g = l/4, c = l%4:  a0 (g, 2c)  a1 (g, 2c+1)  a2 (g+8, 2c)  a3 (g+8, 2c+1)
//                         a4 (g, 2c+8) a5 (g, 2c+9) a6 (g+8, 2c+8) a7 (g+8, 2c+9).
// Scales: u32 [row block][group][g] = f16 scale of row g | f16 of row g+8 << 16.
//
// f16 matrices: the same tiles, 2 KiB each; lane l owns 64 bytes, u32 4j+m is
// the pair (a_{2m}, a_{2m+1}) of column step j, laid out [tile][j][lane][4 u32]
// so that one step of one tile is 512 contiguous bytes.
constexpr int TILE_ROWS = 16;
constexpr int TILE_COLS = 64;

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

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

}  // namespace dfl

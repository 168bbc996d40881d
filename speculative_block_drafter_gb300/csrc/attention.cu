// Non-causal grouped-query attention of a block's rows over the layer's
// windowed context and the block's own rows (cortiq-engine
// src/cortiq_engine/dflash.rs, `Drafter::block`: the scores of every (head,
// row) over the context and the block's rows, a row further on seeing less
// far back when the layer has a window, a max-subtracted softmax).
//
// Split-K: the context rows of a sequence are cut into splits of whole 64-key
// chunks, one CTA per (split, KV head, sequence); the last split of a sequence
// takes the block's own rows (alone when the splits are short). Each keeps a
// running maximum m, sum l and unnormalised output o per query (the rep =
// heads/kv_heads query heads of the KV head times the block rows) and a second
// kernel merges the splits.
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace dfl {

constexpr int ATT_THREADS = 256;
constexpr int CH = 64;              // keys per chunk
constexpr int QMAX = 64;            // queries per CTA (rep * block)
// A split's partial row in global memory: o[hd], m, l, two floats of padding so
// that every row starts on 16 bytes (the merge reads o with vector loads).
__host__ __device__ constexpr int part_row(int hd) { return hd + 4; }

struct AttnArgs {
  AttnSeq seq[MAX_BATCH];
  CUtensorMap own_k, own_v;
};

// Splits per (sequence, KV head) and chunks per split: the split count whose
// waves of CTAs (one an SM) finish first, counting a split's fixed cost (its
// pipeline fill and merge) as two chunks; at most 1024 + 2 * pairs CTAs.
static void plan_splits(int pairs, int max_n, int num_sms, int &ns, int &cps) {
  const int chunks = std::max(1, (max_n + CH - 1) / CH);
  int64_t best = INT64_MAX;
  ns = 1;
  cps = chunks;
  for (int want = 1; want <= chunks && (int64_t)pairs * want <= 1024 + 2 * (int64_t)pairs; ++want) {
    const int c = (chunks + want - 1) / want, n = (chunks + c - 1) / c;
    const int64_t waves = ((int64_t)pairs * n + num_sms - 1) / num_sms;
    const int64_t cost = waves * (c + 2);
    if (cost < best) {
      best = cost;
      ns = n;
      cps = c;
    }
  }
}

size_t attn_partial_bytes(int max_batch, int kv_heads, int heads, int block, int hd) {
  const int Q = heads / kv_heads * block;
  // one partial per CTA: at most 1024 + 2 * batch * kv of them (plan_splits), plus the
  // own rows' split
  const size_t worst = (size_t)1024 + 3 * (size_t)max_batch * kv_heads;
  return worst * Q * (hd + 4) * sizeof(float);
}

// ---------------------------------------------------------------- tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return (PFN_cuTensorMapEncodeTiled_v12000)f;
  }();
  return fn;
}

bool attn_kv_map(CUtensorMap *m, const void *base, int64_t rows, int kv, int hd, int planes, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc || rows < 1 || rows > INT32_MAX || box_rows < 1 || box_rows > 256 || hd % 64 || (planes != 1 && planes != 2))
    return false;
  // (dimension, plane, head, row) of halves; 64 halves (128 bytes) a box row
  const cuuint64_t dims[4] = {(cuuint64_t)hd, (cuuint64_t)planes, (cuuint64_t)kv, (cuuint64_t)rows};
  const cuuint64_t strides[3] = {(cuuint64_t)hd * 2, (cuuint64_t)hd * 2 * planes, (cuuint64_t)kv * hd * 2 * planes};
  const cuuint32_t box[4] = {64, 1, 1, (cuuint32_t)box_rows};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, (void *)base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

__device__ __forceinline__ void tma_load4(uint32_t dst, const CUtensorMap *m, int x, int p, int h, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(dst),
      "l"((uint64_t)m), "r"(x), "r"(p), "r"(h), "r"(z), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm4t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// f32 pair -> f16 hi/lo pairs without the conversion unit: hi keeps the top 11
// significant bits (truncation, exact in f16 over its normal range), lo = x - hi
// rounded to f16; hi + lo carries about 21 bits. Two packed conversions a pair.
__device__ __forceinline__ uint32_t f16x2_rn(float first, float second) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(second), "f"(first));
  return r;
}
__device__ __forceinline__ void split_hl(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  const float h0 = __uint_as_float(__float_as_uint(x0) & 0xFFFFE000u);
  const float h1 = __uint_as_float(__float_as_uint(x1) & 0xFFFFE000u);
  hi = f16x2_rn(h0, h1);
  lo = f16x2_rn(x0 - h0, x1 - h1);
}

// Three-term product of f16 hi/lo pairs: acc += ah.bh + ah.bl + al.bh (about 22 bits).
__device__ __forceinline__ void mma3(float (&acc)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4], uint32_t bh0,
                                     uint32_t bh1, uint32_t bl0, uint32_t bl1) {
  mma16816(acc, ah, bh0, bh1);
  mma16816(acc, ah, bl0, bl1);
  mma16816(acc, al, bh0, bh1);
}

// ---------------------------------------------------------------- the split kernel
//
// One CTA per (split, KV head, sequence): the rep*R queries of the KV head over
// the split's context keys in chunks of 64 (the last split takes the block's
// own R rows as a final chunk). The context caches and the block's own K/V hold
// f16 values per row and head in PL planes (PL = 2: hi, lo; PL = 1: one f16),
// written once when the rows were settled or projected. Warp 0 loads each
// chunk's K and V planes with tensor copies (boxes of 64 rows x 64 halves,
// 128-byte swizzled) into a ring of stages; the warps read their B fragments
// with ldmatrix (K as stored, V transposed) and hold the queries' hi/lo
// fragments in registers. The products: q.k as qh.kh + qh.kl + ql.kh (PL = 2)
// or qh.k + ql.k (PL = 1), p.v likewise with p split into hi and lo. Warp w
// takes query block w % QW and key group w / QW of every chunk; each keeps a
// running (m, l, o), merged in the CTA at the end. Rows past a chunk's keys
// (the context's end, or the block's own R rows) hold whatever the copy or an
// earlier chunk left: their scores are masked and, before P.V, the warps whose
// key range reaches them zero their V planes.
template <int PL>
struct AttnRing {
  static constexpr int BOX = CH * 128;       // 64 rows x 64 halves
  static constexpr int REGION = 2 * BOX;     // one plane of K or V of a chunk (hd <= 128)
  static constexpr int STAGE = 2 * PL * REGION;  // K planes, then V planes
  static constexpr int STAGES = PL == 2 ? 3 : 5;
  static constexpr size_t BYTES = (size_t)STAGES * STAGE + 1024 + 16 * STAGES;  // + alignment, barriers
};

// Byte offset of 16-byte chunk j (8 halves: dimensions 8j..8j+7) of row r in a
// plane region: box j / 8, swizzled within the row's 128 bytes.
__device__ __forceinline__ uint32_t plane_off(int r, int j) {
  return (uint32_t)((j >> 3) * (CH * 128) + r * 128 + (((j & 7) ^ (r & 7)) << 4));
}

template <int HD, int KG, int PL>
__global__ void __launch_bounds__(ATT_THREADS, 1) k_attn(const float *__restrict__ q, const __grid_constant__ AttnArgs args,
                                                         int heads, int kv, int R, int window, float scale, int nsplit,
                                                         int cps, float *__restrict__ part) {
  using RG = AttnRing<PL>;
  constexpr int S = RG::STAGES;
  constexpr int H2 = HD / 64;        // boxes of a row
  constexpr int KW = CH / KG;        // keys per warp per chunk
  constexpr int NT = KW / 8;         // n8 tiles of scores
  constexpr int KS = KW / 16;        // k16 steps of P . V
  constexpr int OT = HD / 8;         // n8 tiles of the output
  static_assert(NT % 2 == 0 && OT % 2 == 0 && KS >= 1, "fragments load in pairs of tiles");
  extern __shared__ __align__(16) uint8_t smraw[];
  uint8_t *sm = smraw + ((1024 - (smem_u32(smraw) & 1023)) & 1023);
  const uint32_t ring = smem_u32(sm);
  const uint32_t full0 = ring + S * RG::STAGE, empty0 = full0 + 8 * S;

  const int sp = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int rep = heads / kv, Q = rep * R;
  const int QW = (Q + 15) / 16;
  const AttnSeq &Sq = args.seq[b];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, cq = lane & 3;
  const int qb = warp % QW, kgi = warp / QW;
  const bool busy = kgi < KG && warp < QW * KG;
  const int nwarps = ATT_THREADS / 32;

  // this CTA's chunks: context chunks [c0, c1), then the block's own rows if last
  const int n = Sq.n;
  const int nctx = (n + CH - 1) / CH;
  const int c0 = min(nctx, sp * cps), c1 = min(nctx, c0 + cps);
  const bool own = sp == nsplit - 1;
  const int nch = (c1 - c0) + (own ? 1 : 0);

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, nwarps);
    }
    mbar_fence_init();
  }
  pdl_wait();
  __syncthreads();

  // warp 0, lane 0: the 4 * H2 tensor copies of chunk j into stage st
  auto fill = [&](int j, int st) {
    if (lane != 0) return;
    const bool is_own = own && j == nch - 1;
    const CUtensorMap *km = is_own ? &args.own_k : &Sq.kmap;
    const CUtensorMap *vm = is_own ? &args.own_v : &Sq.vmap;
    const int z = is_own ? b * R : (int)(Sq.row0 + (int64_t)(c0 + j) * CH);
    const uint32_t rows = is_own ? R : CH;
    const uint32_t bar = full0 + 8 * st, base = ring + st * RG::STAGE;
    mbar_expect_tx(bar, 2 * PL * H2 * rows * 128);
#pragma unroll
    for (int h = 0; h < H2; ++h)
#pragma unroll
      for (int p = 0; p < PL; ++p) {
        tma_load4(base + p * RG::REGION + h * RG::BOX, km, 64 * h, p, g, z, bar);
        tma_load4(base + (PL + p) * RG::REGION + h * RG::BOX, vm, 64 * h, p, g, z, bar);
      }
  };
  int issued = 0;  // chunks warp 0 has filled
  if (warp == 0)
    for (; issued < S && issued < nch; ++issued) fill(issued, issued);

  // the queries' hi/lo A fragments (rows qb*16 + gq and + 8)
  uint32_t qh[HD / 16][4], ql[HD / 16][4];
  const int qi0 = qb * 16 + gq, qi1 = qi0 + 8;
  {
    const float *q0 = nullptr, *q1 = nullptr;
    if (qi0 < Q) q0 = q + ((int64_t)b * R + qi0 % R) * heads * HD + (g * rep + qi0 / R) * HD;
    if (qi1 < Q) q1 = q + ((int64_t)b * R + qi1 % R) * heads * HD + (g * rep + qi1 / R) * HD;
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
      const int c = ks * 16 + 2 * cq;
      const float2 x00 = q0 ? *(const float2 *)(q0 + c) : make_float2(0.f, 0.f);
      const float2 x10 = q1 ? *(const float2 *)(q1 + c) : make_float2(0.f, 0.f);
      const float2 x01 = q0 ? *(const float2 *)(q0 + c + 8) : make_float2(0.f, 0.f);
      const float2 x11 = q1 ? *(const float2 *)(q1 + c + 8) : make_float2(0.f, 0.f);
      split_hl(x00.x, x00.y, qh[ks][0], ql[ks][0]);
      split_hl(x10.x, x10.y, qh[ks][1], ql[ks][1]);
      split_hl(x01.x, x01.y, qh[ks][2], ql[ks][2]);
      split_hl(x11.x, x11.y, qh[ks][3], ql[ks][3]);
    }
  }
  const int r0 = qi0 % R, r1 = qi1 % R;
  // ldmatrix lane roles: row within an 8x8 matrix and which of the four matrices
  const int mr = lane & 7, mi = lane >> 3;

  float o[OT][4];
#pragma unroll
  for (int t = 0; t < OT; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  bool ok = true;

  for (int j = 0; j < nch && ok; ++j) {
    const int st = j % S;
    ok = mbar_wait(full0 + 8 * st, (j / S) & 1);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    const bool is_own = own && j == nch - 1;
    const int kb = (c0 + j) * CH;
    const int cnt = is_own ? R : min(CH, n - kb);
    uint8_t *stp = sm + st * RG::STAGE;
    // K planes at regions 0..PL-1, V planes at PL..2PL-1 (klo, vlo unused with one plane)
    const uint32_t khi = smem_u32(stp), klo = khi + RG::REGION, vhi = khi + PL * RG::REGION, vlo = vhi + RG::REGION;
    const int kk0 = kgi * KW;
    if (busy && cnt < kk0 + KW) {
      // zero the V rows of this warp's keys past the chunk's (both planes, every box)
      const int z0 = max(kk0, cnt), nz = kk0 + KW - z0;
      for (int idx = lane; idx < nz * PL * H2 * 8; idx += 32) {
        const int row = z0 + idx / (PL * H2 * 8), rest = idx % (PL * H2 * 8);
        const int pl = rest / (H2 * 8), bx = (rest / 8) % H2, ch = rest % 8;
        *(uint4 *)(stp + (PL + pl) * RG::REGION + bx * RG::BOX + row * 128 + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // before the stage's next tensor copy
      __syncwarp();
    }
    if (busy) {
      float sc[NT][4];
      // S = Q . K^T: per k16 step and pair of key tiles the four 8x8 matrices
      // (tile t, dims 16ks..+8), (t, +8..+16), (t+1, ..), (t+1, ..) of each plane.
      // The three products go to separate accumulators (two with four tiles),
      // so that the MMAs of a step do not wait on one another.
      constexpr int NA = (PL == 2 && NT == 2) ? 3 : 2;
      float sa[NA][NT][4];
#pragma unroll
      for (int a = 0; a < NA; ++a)
#pragma unroll
        for (int t = 0; t < NT; ++t) sa[a][t][0] = sa[a][t][1] = sa[a][t][2] = sa[a][t][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < HD / 16; ++ks) {
#pragma unroll
        for (int t = 0; t < NT; t += 2) {
          const uint32_t off = plane_off(kk0 + 8 * (t + (mi >> 1)) + mr, 2 * ks + (mi & 1));
          uint32_t h0, h1, h2, h3;
          ldsm4(khi + off, h0, h1, h2, h3);
          mma16816(sa[0][t], qh[ks], h0, h1);
          mma16816(sa[0][t + 1], qh[ks], h2, h3);
          if constexpr (PL == 2) {
            uint32_t w0, w1, w2, w3;
            ldsm4(klo + off, w0, w1, w2, w3);
            mma16816(sa[1][t], qh[ks], w0, w1);
            mma16816(sa[1][t + 1], qh[ks], w2, w3);
          }
          mma16816(sa[NA - 1][t], ql[ks], h0, h1);
          mma16816(sa[NA - 1][t + 1], ql[ks], h2, h3);
        }
      }
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[t][e] = sa[0][t][e] + (NA == 3 ? sa[1][t][e] + sa[2][t][e] : sa[1][t][e]);
      // mask, scale, online softmax (rows gq, gq+8; the 4 lanes of a row hold its 2*NT keys)
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = kk0 + t * 8 + 2 * cq + (e & 1);
          const int qi = (e < 2) ? qi0 : qi1;
          const int rr = (e < 2) ? r0 : r1;
          bool vis = key < cnt && qi < Q;
          if (vis && !is_own && window > 0) vis = Sq.lo + kb + key >= Sq.anchor + rr + 1 - window;
          const float x = vis ? sc[t][e] * scale : -INFINITY;
          sc[t][e] = x;
          if (e < 2) mx0 = fmaxf(mx0, x);
          else mx1 = fmaxf(mx1, x);
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
      const float a0 = n0 == -INFINITY ? 1.f : expf(m0 - n0);
      const float a1 = n1 == -INFINITY ? 1.f : expf(m1 - n1);
      m0 = n0;
      m1 = n1;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        sc[t][0] = sc[t][0] == -INFINITY ? 0.f : expf(sc[t][0] - n0);
        sc[t][1] = sc[t][1] == -INFINITY ? 0.f : expf(sc[t][1] - n0);
        sc[t][2] = sc[t][2] == -INFINITY ? 0.f : expf(sc[t][2] - n1);
        sc[t][3] = sc[t][3] == -INFINITY ? 0.f : expf(sc[t][3] - n1);
        s0 += sc[t][0] + sc[t][1];
        s1 += sc[t][2] + sc[t][3];
      }
      l0 = l0 * a0 + s0;
      l1 = l1 * a1 + s1;
      if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {  // a row's maximum moved
#pragma unroll
        for (int t = 0; t < OT; ++t) {
          o[t][0] *= a0;
          o[t][1] *= a0;
          o[t][2] *= a1;
          o[t][3] *= a1;
        }
      }
      // O += P . V: P as hi/lo A fragments from the scores; V by transposed
      // ldmatrix: (keys +0..8, dims tile t), (keys +8..16, t), (.., t+1), (.., t+1)
#pragma unroll
      for (int js = 0; js < KS; ++js) {
        uint32_t ph[4], pl[4];
        split_hl(sc[2 * js][0], sc[2 * js][1], ph[0], pl[0]);
        split_hl(sc[2 * js][2], sc[2 * js][3], ph[1], pl[1]);
        split_hl(sc[2 * js + 1][0], sc[2 * js + 1][1], ph[2], pl[2]);
        split_hl(sc[2 * js + 1][2], sc[2 * js + 1][3], ph[3], pl[3]);
        const int row = kk0 + 16 * js + 8 * (mi & 1) + mr;
#pragma unroll
        for (int t = 0; t < OT; t += 2) {
          const uint32_t off = plane_off(row, t + (mi >> 1));
          uint32_t h0, h1, h2, h3;
          ldsm4t(vhi + off, h0, h1, h2, h3);
          if constexpr (PL == 2) {
            uint32_t w0, w1, w2, w3;
            ldsm4t(vlo + off, w0, w1, w2, w3);
            mma3(o[t], ph, pl, h0, h1, w0, w1);
            mma3(o[t + 1], ph, pl, h2, h3, w2, w3);
          } else {
            mma16816(o[t], ph, h0, h1);
            mma16816(o[t + 1], ph, h2, h3);
            mma16816(o[t], pl, h0, h1);
            mma16816(o[t + 1], pl, h2, h3);
          }
        }
      }
    }
    // release the stage; warp 0 refills it with the chunk S ahead
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * st);
    if (warp == 0 && j + S < nch) {
      ok = mbar_wait(empty0 + 8 * st, (j / S) & 1);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        fill(j + S, st);
        ++issued;
      }
    }
  }
  // every copy issued has landed before the ring becomes the merge scratch (on
  // the error path too: each stage's latest fill, a bounded wait each)
  if (warp == 0)
    for (int j = max(0, issued - S); j < issued; ++j) mbar_wait(full0 + 8 * (j % S), (j / S) & 1);
  __syncthreads();

  // in-CTA merge of the key groups: per warp 16 rows x (o, m, l) in the scratch
  float *scr = (float *)sm;
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  if (busy) {
    float *w = scr + warp * 16 * (HD + 2);
#pragma unroll
    for (int t = 0; t < OT; ++t) {
      w[gq * (HD + 2) + t * 8 + 2 * cq] = o[t][0];
      w[gq * (HD + 2) + t * 8 + 2 * cq + 1] = o[t][1];
      w[(gq + 8) * (HD + 2) + t * 8 + 2 * cq] = o[t][2];
      w[(gq + 8) * (HD + 2) + t * 8 + 2 * cq + 1] = o[t][3];
    }
    if (cq == 0) {
      w[gq * (HD + 2) + HD] = m0;
      w[gq * (HD + 2) + HD + 1] = l0;
      w[(gq + 8) * (HD + 2) + HD] = m1;
      w[(gq + 8) * (HD + 2) + HD + 1] = l1;
    }
  }
  __syncthreads();
  float *out = part + ((int64_t)(b * kv + g) * nsplit + sp) * Q * part_row(HD);
  // one warp per query row at a time: the key groups' weights once, then the row
  for (int qi = warp; qi < Q; qi += ATT_THREADS / 32) {
    const int qbk = qi / 16, rr = qi % 16;
    float M = -INFINITY;
#pragma unroll
    for (int kg = 0; kg < KG; ++kg) M = fmaxf(M, scr[(kg * QW + qbk) * 16 * (HD + 2) + rr * (HD + 2) + HD]);
    float wt[KG];
#pragma unroll
    for (int kg = 0; kg < KG; ++kg) {
      const float mk = scr[(kg * QW + qbk) * 16 * (HD + 2) + rr * (HD + 2) + HD];
      wt[kg] = mk == -INFINITY ? 0.f : expf(mk - M);
    }
    float *orow = out + (int64_t)qi * part_row(HD);
    for (int c = lane; c < HD + 2; c += 32) {
      float acc = 0.f;
      if (c == HD) {
        acc = M;
      } else {
#pragma unroll
        for (int kg = 0; kg < KG; ++kg)
          acc = fmaf(scr[(kg * QW + qbk) * 16 * (HD + 2) + rr * (HD + 2) + c], wt[kg], acc);  // o, or l at HD + 1
      }
      orow[c] = acc;
    }
  }
}

// y[b*R + r][h*HD + d] = sum_s o_s e^(m_s - M) / sum_s l_s e^(m_s - M), one warp a
// query row: lane s reads split s's (m, l) (a loop past 32 splits), the warp
// reduces M and L, then each lane sums 4 dimensions over the splits with the
// splits' loads independent of one another (a few L2 round trips in all).
// PACK writes the row into the output projection's token tiles (hi/lo planes;
// even lanes take their neighbour's 4 values) and the blocks past the work
// grid clear that GEMM's outputs when it splits; else the row goes to y.
constexpr int MERGE_WARPS = 4;

template <int HD, bool PACK>
__global__ void __launch_bounds__(32 * MERGE_WARPS) k_attn_merge(const float *__restrict__ part, int heads, int kv,
                                                                 int R, int ns, int work_blocks,
                                                                 float *__restrict__ y, PackDst P, ZeroSet Z) {
  static_assert(HD == 4 * 32 || HD == 2 * 32, "head dimension");
  constexpr int DL = HD / 32;  // dimensions a lane
  pdl_wait();
  if (PACK) pdl_trigger();  // the GEMM this feeds may fetch its weights meanwhile
  if ((int)blockIdx.x >= work_blocks) {
    if (PACK && blockIdx.y == 0) zero_set_clear(Z, blockIdx.x - work_blocks, gridDim.x - work_blocks);
    return;
  }
  const int b = blockIdx.y, lane = threadIdx.x & 31;
  const int rep = heads / kv, Q = rep * R;
  const int row = blockIdx.x * MERGE_WARPS + (threadIdx.x >> 5);
  if (row >= kv * Q) return;
  const int g = row / Q, qi = row - g * Q;
  const int hrep = qi / R, r = qi - hrep * R;
  const int64_t sstride = (int64_t)Q * part_row(HD);
  const float *base = part + (int64_t)(b * kv + g) * ns * sstride + (int64_t)qi * part_row(HD);
  // M and L over the splits: lane s holds split s's (m, l) and weight e^(m - M)
  // (more than 32 splits: a loop, the weights recomputed in the sum below)
  float M = -INFINITY, L = 0.f, ws = 0.f;
  if (ns <= 32) {
    float ms = -INFINITY, ls = 0.f;
    if (lane < ns) {
      ms = base[lane * sstride + HD];
      ls = base[lane * sstride + HD + 1];
    }
    M = warp_max(ms);
    ws = ms == -INFINITY ? 0.f : expf(ms - M);
    L = warp_sum(ls * ws);
  } else {
    for (int s = lane; s < ns; s += 32) M = fmaxf(M, base[s * sstride + HD]);
    M = warp_max(M);
    for (int s = lane; s < ns; s += 32) {
      const float m = base[s * sstride + HD];
      if (m != -INFINITY) L = fmaf(base[s * sstride + HD + 1], expf(m - M), L);
    }
    L = warp_sum(L);
  }
  // the row: lane's DL dimensions over the splits (independent vector loads)
  float acc[DL];
#pragma unroll
  for (int e = 0; e < DL; ++e) acc[e] = 0.f;
#pragma unroll 8
  for (int s = 0; s < ns; ++s) {
    const float *ps = base + s * sstride;
    float w;
    if (ns <= 32) {
      w = __shfl_sync(0xffffffffu, ws, s);
    } else {
      const float m = ps[HD];
      w = m == -INFINITY ? 0.f : expf(m - M);
    }
    if constexpr (DL == 4) {
      const float4 o = *(const float4 *)(ps + 4 * lane);
      acc[0] = fmaf(o.x, w, acc[0]);
      acc[1] = fmaf(o.y, w, acc[1]);
      acc[2] = fmaf(o.z, w, acc[2]);
      acc[3] = fmaf(o.w, w, acc[3]);
    } else {
      const float2 o = *(const float2 *)(ps + 2 * lane);
      acc[0] = fmaf(o.x, w, acc[0]);
      acc[1] = fmaf(o.y, w, acc[1]);
    }
  }
  const float inv = 1.f / L;
#pragma unroll
  for (int e = 0; e < DL; ++e) acc[e] *= inv;
  const int col = (g * rep + hrep) * HD;
  if constexpr (PACK) {
    // 8 consecutive columns a store: lanes 8/DL apart hand theirs to the first
    constexpr int LPC = 8 / DL;  // lanes a store
    float x8[8];
#pragma unroll
    for (int j = 0; j < LPC; ++j)
#pragma unroll
      for (int e = 0; e < DL; ++e) x8[j * DL + e] = __shfl_sync(0xffffffffu, acc[e], (lane / LPC) * LPC + j);
    if (lane % LPC == 0) pack_store8(P, b * R + r, col + DL * lane, x8);
  } else {
    float *out = y + ((int64_t)b * R + r) * heads * HD + col + DL * lane;
    if constexpr (DL == 4) *(float4 *)out = make_float4(acc[0], acc[1], acc[2], acc[3]);
    else *(float2 *)out = make_float2(acc[0], acc[1]);
  }
}

template <int HD, int KG, int PL>
static cudaError_t launch_attn(const float *q, const AttnArgs &args, int batch, int max_n, int heads, int kv, int R,
                               int window, float scale, float *part, float *y, int num_sms, const PackDst *pack,
                               const ZeroSet *zero, cudaStream_t st) {
  const size_t smem = AttnRing<PL>::BYTES;
  static PerDevice configured;
  if (cudaError_t e = smem_limit(k_attn<HD, KG, PL>, (int)smem, configured)) return e;
  int ns, cps;
  plan_splits(batch * kv, max_n, num_sms, ns, cps);
  // With short splits the block's own rows get a split of their own (the last
  // one, past every context chunk), so that no CTA does twice the others' work.
  if (cps <= 4 && max_n > 0) ++ns;
  dim3 grid(ns, kv, batch);
  cudaError_t e = launch_pdl(k_attn<HD, KG, PL>, grid, dim3(ATT_THREADS), smem, st, 1, q, args, heads, kv, R, window,
                             scale, ns, cps, part);
  if (e != cudaSuccess) return e;
  const int Q = heads / kv * R;
  const int work = (kv * Q + MERGE_WARPS - 1) / MERGE_WARPS;
  if (pack) {
    int64_t most = 0;
    for (int j = 0; j < zero->count; ++j) most = std::max<int64_t>(most, zero->n[j]);
    const int zb =
        zero->count ? (int)std::min<int64_t>((most + 4 * 32 * MERGE_WARPS - 1) / (4 * 32 * MERGE_WARPS), 256) : 0;
    return launch_pdl(k_attn_merge<HD, true>, dim3(work + zb, batch), dim3(32 * MERGE_WARPS), 0, st, 1, part, heads,
                      kv, R, ns, work, (float *)nullptr, *pack, *zero);
  }
  return launch_pdl(k_attn_merge<HD, false>, dim3(work, batch), dim3(32 * MERGE_WARPS), 0, st, 1, part, heads, kv, R,
                    ns, work, y, PackDst{}, ZeroSet{});
}

template <int HD, int PL>
static cudaError_t launch_attn_hd(const float *q, const AttnArgs &args, int batch, int max_n, int heads, int kv, int R,
                                  int window, float scale, float *part, float *y, int num_sms, const PackDst *pack,
                                  const ZeroSet *zero, cudaStream_t st) {
  const int QW = (heads / kv * R + 15) / 16;
  if (QW >= 3)
    return launch_attn<HD, 2, PL>(q, args, batch, max_n, heads, kv, R, window, scale, part, y, num_sms, pack, zero, st);
  return launch_attn<HD, 4, PL>(q, args, batch, max_n, heads, kv, R, window, scale, part, y, num_sms, pack, zero, st);
}

cudaError_t attention(const float *q, const CUtensorMap &own_k, const CUtensorMap &own_v, const AttnSeq *seqs,
                      int batch, int heads, int kv_heads, int hd, int planes, int block, int window, float scale,
                      float *partials, float *y, int num_sms, const PackDst *pack, const ZeroSet *zero,
                      cudaStream_t st) {
  if (batch < 1 || batch > MAX_BATCH || heads / kv_heads * block > QMAX || (planes != 1 && planes != 2))
    return cudaErrorInvalidValue;
  AttnArgs args;  // entries past batch are not read
  int max_n = 0;
  for (int i = 0; i < batch; ++i) {
    args.seq[i] = seqs[i];
    max_n = std::max(max_n, seqs[i].n);
  }
  args.own_k = own_k;
  args.own_v = own_v;
  num_sms = std::max(1, std::min(num_sms, 1024));
  if (hd == 128 && planes == 2)
    return launch_attn_hd<128, 2>(q, args, batch, max_n, heads, kv_heads, block, window, scale, partials, y, num_sms,
                                  pack, zero, st);
  if (hd == 128)
    return launch_attn_hd<128, 1>(q, args, batch, max_n, heads, kv_heads, block, window, scale, partials, y, num_sms,
                                  pack, zero, st);
  if (hd == 64 && planes == 2)
    return launch_attn_hd<64, 2>(q, args, batch, max_n, heads, kv_heads, block, window, scale, partials, y, num_sms,
                                 pack, zero, st);
  if (hd == 64)
    return launch_attn_hd<64, 1>(q, args, batch, max_n, heads, kv_heads, block, window, scale, partials, y, num_sms,
                                 pack, zero, st);
  return cudaErrorInvalidValue;
}

// This file's device error word (a bounded wait that gave up).
cudaError_t attn_read_error(unsigned *out, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_dev_error, sizeof(unsigned));
  if (e == cudaSuccess && reset) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_dev_error, &zero, sizeof(unsigned));
  }
  return e;
}

}  // namespace dfl

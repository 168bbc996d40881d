// Weight GEMMs over many tokens (a settle chunk of up to 1024 rows, a batch of
// blocks) on the tcgen05 tensor cores: Y[t][r] = sum_k X[t][k] W[r][k].
//
// At these sizes a 128-row weight tile meets up to 256 tokens in one MMA
// (M = 128, N = tokens, K = 16), so the weights are no longer the whole cost:
// the work is split over the SMs ("stream-K"). The (token tile, row tile,
// 64-column k-tile) units of all matrices are laid end to end and each CTA
// takes one contiguous range of them, in runs that each stay inside one tile.
// A run over part of a tile adds its partial sums into Y with atomics (Y is
// cleared first). The f16 kernel's ranges are equal; the four-bit kernel's
// are equal in cost, a run's read-back of its one accumulator counted as a
// few units (wide_bounds). When the tiles about fill the resident CTAs, each
// CTA takes one whole tile instead (launch_wide), which splits none. Every
// CTA bulk-copies its own operands.
//
//   warp 4      bulk-copies each unit's operands into a shared-memory ring
//   warp 5      issues the MMAs (one thread)
//   warps 0-3   four-bit matrices: turn the unit's codes into the A operand in
//               tensor memory; at the end of a run: read the accumulator back
//               and add it to Y
//
// f16 matrices (fc, the kernel projections, the selector's projection): the
// weight tiles go to shared memory as packed and the tokens enter rounded to
// f16, as the card arm does (`to_half`, cortiq-engine
// src/gpu_cuda/hyb/dflash.rs, `Dev::settle`).
//
// Four-bit matrices: every weight q * s is written exactly as hi + lo, two
// f16 values, after scaling the row by a power of two 2^p chosen from its
// largest scale in the run (so that lo stays a normal f16); the tokens enter
// as f16 planes x = xh + xl. One accumulator spans the whole run:
//   D = Wh xh + Wh xl + Wl xh   (three MMAs a k-step; Wl xl is below 2^-22)
// and the run's partial sums are multiplied by 2^-p when added to Y.
#include <algorithm>
#include <climits>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace dfl {

constexpr int W_THREADS = 192;
constexpr int W_PRODUCER = 4;
constexpr int W_MMA = 5;
constexpr int W_KIND_F16 = 0;
constexpr int W_KIND_I4 = 1;

template <int KIND, int DU>
struct WCfg {
  // shared-memory stage: B (token planes, N x 128 B each) first, then
  // f16: the weight tile (16 KiB); four-bit: codes (4 KiB) and scales (DU x 256 B)
  static constexpr int PLANES = KIND == W_KIND_F16 ? 1 : 2;
  static constexpr int A_BYTES = KIND == W_KIND_F16 ? 16384 : 4096 + DU * 256;
  static constexpr int STAGE_MAX = (PLANES * WIDE_MAX_N * 128 + A_BYTES + 1023) / 1024 * 1024;
  static constexpr int STAGES = KIND == W_KIND_F16 ? 4 : 3;
  static constexpr int SA = 2;                     // tensor-memory A slots (four-bit)
  static constexpr int NBUF = KIND == W_KIND_F16 ? 2 : 1;
  static constexpr int A_COL = 256;                // A slots after the accumulator (four-bit)
  static constexpr int NBAR = 2 * STAGES + 2 * SA + 2 * NBUF;
  static constexpr int STAGING = 4 * 16 * 32 * 4;  // a slice of 16 tokens x 32 rows f32 a warp (the epilogue)
  static constexpr int SMEM = STAGES * STAGE_MAX + STAGING + 1024 + 8 * NBAR + 64;
};

__device__ __forceinline__ WideJob wjob(const WideArgs &A, int j) { return A.job[j]; }

// The job holding global row tile mt (jobs in order of tile0).
__device__ __forceinline__ int wjob_of(const WideArgs &A, int mt) {
  int lo = 0, hi = A.njobs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (wjob(A, mid).tile0 <= mt) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// The units [u0, u1) of CTA q of Q.
__device__ __forceinline__ void wrange(const WideArgs &A, int64_t q, int64_t Q, int64_t &u0, int64_t &u1) {
  if (A.nbnd > 0) {
    u0 = A.bnd[q];
    u1 = A.bnd[q + 1];
  } else {
    u0 = q * A.units / Q;
    u1 = (q + 1) * A.units / Q;
  }
}

// A unit: token tile, row tile, k-tile.
struct WUnit {
  int tt, mt, kt;
};
__device__ __forceinline__ WUnit wunit(const WideArgs &A, int64_t u) {
  const int64_t per_tt = (int64_t)A.mtiles * A.KT;
  WUnit r;
  r.tt = (int)(u / per_tt);
  const int64_t rest = u - (int64_t)r.tt * per_tt;
  r.mt = (int)(rest / A.KT);
  r.kt = (int)(rest - (int64_t)r.mt * A.KT);
  return r;
}

// the end (exclusive) of the run that starts at unit u: the end of its k-range or of the CTA's range
__device__ __forceinline__ int64_t wrun_end(const WideArgs &A, int64_t u, int64_t u1) {
  const int64_t tile_end = (u / A.KT + 1) * A.KT;
  return tile_end < u1 ? tile_end : u1;
}

// A walk over consecutive units of one CTA: the token tile, the k-tile and the
// address of the CTA's weight tile, advanced without divisions.
struct WCursor {
  int tt, mt, kt;
  int64_t tile0;              // the row tile's first k-tile in its matrix's packed tiles
  const uint8_t *w, *s;       // the matrix's codes (or f16 tiles) and scales
  __device__ __forceinline__ void locate(const WideArgs &A) {
    const WideJob J = wjob(A, wjob_of(A, mt));
    tile0 = (int64_t)(mt - J.tile0) * A.KT;
    w = (const uint8_t *)J.w;
    s = (const uint8_t *)J.s;
  }
  __device__ __forceinline__ void start(const WideArgs &A, int64_t u) {
    const int64_t tg = u / A.KT;
    kt = (int)(u - tg * A.KT);
    mt = (int)(tg % A.mtiles);
    tt = (int)(tg / A.mtiles);
    locate(A);
  }
  __device__ __forceinline__ void next(const WideArgs &A) {
    if (++kt == A.KT) {
      kt = 0;
      if (++mt == A.mtiles) {
        mt = 0;
        ++tt;
      }
      locate(A);
    }
  }
  // the weights are read once: evict them from L2 first
  template <int KIND, int DU>
  __device__ __forceinline__ void load_a(const WideArgs &A, uint32_t dst, uint32_t bar, uint64_t pol) const {
    if (KIND == W_KIND_F16) {
      bulk_g2s_hint(dst, w + (tile0 + kt) * 16384, 16384, bar, pol);
    } else {
      bulk_g2s_hint(dst, w + (tile0 + kt) * 4096, 4096, bar, pol);
      bulk_g2s_hint(dst + 4096, s + (tile0 + kt) * DU * 256, DU * 256, bar, pol);
    }
  }
};

// Four-bit: the power of two 2^p that row r of the CTA's row tile is scaled by
// over the run [u, ue): smax * 2^p < 2^12 for the row's largest scale smax in
// the run, so |q| * s * 2^p < 2^15. The run's DU * (ue - u) scales of the row
// sit 128 halves apart; they are read eight at a time into separate maxima so
// that the loads are in flight together.
template <int DU>
__device__ __forceinline__ int run_pow2(const WideArgs &A, int64_t u, int64_t ue, int r) {
  const WUnit w0 = wunit(A, u);
  const WideJob J = wjob(A, wjob_of(A, w0.mt));
  const int m = w0.mt - J.tile0;
  const uint16_t *sc = (const uint16_t *)J.s + ((int64_t)m * A.KT + w0.kt) * DU * 128 + r;
  const int n = (int)(ue - u) * DU;
  float mx[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int i = 0;
  for (; i + 8 <= n; i += 8) {
    uint16_t v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = __ldg(sc + (int64_t)(i + e) * 128);
#pragma unroll
    for (int e = 0; e < 8; ++e) mx[e] = fmaxf(mx[e], fabsf(__half2float(__ushort_as_half(v[e]))));
  }
  for (; i < n; ++i) mx[0] = fmaxf(mx[0], fabsf(__half2float(__ushort_as_half(__ldg(sc + (int64_t)i * 128)))));
  float smax = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) smax = fmaxf(smax, mx[e]);
  int p = 0;
  if (smax > 0.f) {
    int e;
    frexpf(smax, &e);                  // smax in [2^(e-1), 2^e)
    p = max(-100, min(100, 12 - e));
  }
  return p;
}

template <int KIND, int DU>
__global__ void __launch_bounds__(W_THREADS, 1) k_wide(WideArgs A) {
  using C = WCfg<KIND, DU>;
  constexpr int S = C::STAGES;
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t *sm = smraw + ((1024 - (smem_u32(smraw) & 1023)) & 1023);
  const int N = A.N;
  const int b_bytes = C::PLANES * N * 128;
  const int stage = (b_bytes + C::A_BYTES + 1023) & ~1023;
  float *staging = (float *)(sm + S * stage);
  uint64_t *bars = (uint64_t *)(sm + S * stage + C::STAGING);
  uint32_t *tslot = (uint32_t *)(bars + C::NBAR);
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * S, afull0 = empty0 + 8 * S;
  const uint32_t afree0 = afull0 + 8 * C::SA, dfull0 = afree0 + 8 * C::SA, dfree0 = dfull0 + 8 * C::NBUF;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // this CTA's units
  int64_t u0, u1;
  wrange(A, blockIdx.x, gridDim.x, u0, u1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(full0 + 8 * i, 1);
      // released by the MMAs (B) and, four-bit, the dequantisers (codes)
      mbar_init(empty0 + 8 * i, KIND == W_KIND_F16 ? 1 : 1 + 128);
    }
    for (int i = 0; i < C::SA; ++i) {
      mbar_init(afull0 + 8 * i, 128);
      mbar_init(afree0 + 8 * i, 1);
    }
    for (int i = 0; i < C::NBUF; ++i) {
      mbar_init(dfull0 + 8 * i, 1);
      mbar_init(dfree0 + 8 * i, 128);
    }
    mbar_fence_init();
  }
  __syncthreads();
  // The weights do not depend on the kernels before this one: the first stages'
  // weight tiles are fetched before waiting for them. The producer walks its
  // units with counters (a division per unit would slow the one thread that
  // feeds the pipeline).
  WCursor cur;
  int npre = 0;
  if (warp == W_PRODUCER && lane == 0) {
    const uint64_t wpol = l2_evict_first();
    cur.start(A, u0);
    for (; npre < S && u0 + npre < u1; ++npre, cur.next(A)) {
      mbar_expect_tx(full0 + 8 * npre, b_bytes + C::A_BYTES);
      cur.load_a<KIND, DU>(A, smem_u32(sm + npre * stage) + b_bytes, full0 + 8 * npre, wpol);
    }
  }
  // Four-bit: the first run's row scaling, from the weights' scales (which do
  // not depend on the kernels before this one either).
  int p_next = 0;
  if (KIND == W_KIND_I4 && warp < 4 && u0 < u1) p_next = run_pow2<DU>(A, u0, wrun_end(A, u0, u1), threadIdx.x);
  pdl_wait();
  if (warp == 0) tmem_alloc(smem_u32(tslot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp == W_PRODUCER) {
    if (lane == 0) {
      WCursor bc;  // the units' token tiles
      bc.start(A, u0);
      // the token tiles are read by every row tile: keep them in L2
      const uint64_t wpol = l2_evict_first(), bpol = l2_evict_last();
      int i = 0;
      bool ok = true;
      for (int64_t u = u0; u < u1; ++u, ++i, bc.next(A)) {
        const int s = i % S;
        const uint32_t st = smem_u32(sm + s * stage);
        if (i >= npre) {
          if (i >= S && !mbar_wait(empty0 + 8 * s, ((i / S) - 1) & 1)) {
            ok = false;
            break;
          }
          mbar_expect_tx(full0 + 8 * s, b_bytes + C::A_BYTES);
          cur.load_a<KIND, DU>(A, st + b_bytes, full0 + 8 * s, wpol);
          cur.next(A);
        }
        const uint8_t *bp = A.bpack + ((int64_t)bc.tt * A.KT + bc.kt) * b_bytes;
        bulk_g2s_hint(st, bp, b_bytes, full0 + 8 * s, bpol);
      }
      // every stage released by every consumer (no copy still bound for this CTA)
      if (ok)
        for (int k = (i > S ? i - S : 0); k < i; ++k)
          if (!mbar_wait(empty0 + 8 * (k % S), (k / S) & 1)) break;
    }
  } else if (warp == W_MMA) {
    if (lane == 0) {
      const uint32_t idesc = f16_idesc(128, N);
      int i = 0, run = 0;
      bool ok = true;
      for (int64_t u = u0; u < u1 && ok; ++run) {
        const int64_t ue = wrun_end(A, u, u1);
        const int d = run % C::NBUF;
        if (run >= C::NBUF && !mbar_wait(dfree0 + 8 * d, ((run / C::NBUF) - 1) & 1)) break;
        tc_fence_after();
        const uint32_t dcol = tbase + d * 256;
        for (int64_t v = u; v < ue; ++v, ++i) {
          const int s = i % S;
          if (!mbar_wait(full0 + 8 * s, (i / S) & 1)) {
            ok = false;
            break;
          }
          const uint32_t st = smem_u32(sm + s * stage);
          if (KIND == W_KIND_F16) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_ss(dcol, sw128_desc(st + b_bytes + ks * 32), sw128_desc(st + ks * 32), idesc, (v > u || ks > 0));
          } else {
            const int a = i % C::SA;
            if (!mbar_wait(afull0 + 8 * a, (i / C::SA) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t ah = tbase + C::A_COL + a * 64, al = ah + 32;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint64_t bh = sw128_desc(st + ks * 32), bl = sw128_desc(st + N * 128 + ks * 32);
              mma_ts(dcol, ah + ks * 8, bh, idesc, (v > u || ks > 0));
              mma_ts(dcol, ah + ks * 8, bl, idesc, 1);
              mma_ts(dcol, al + ks * 8, bh, idesc, 1);
            }
            mma_commit(afree0 + 8 * a);
          }
          mma_commit(empty0 + 8 * s);
        }
        mma_commit(dfull0 + 8 * d);
        u = ue;
      }
    }
  } else if (warp < 4) {
    const int r = warp * 32 + lane;
    const uint32_t lrow = (uint32_t)(warp * 32) << 16;
    int i = 0, run = 0;
    bool ok = true;
    for (int64_t u = u0; u < u1 && ok; ++run) {
      const int64_t ue = wrun_end(A, u, u1);
      const WUnit w0 = wunit(A, u);
      const WideJob J = wjob(A, wjob_of(A, w0.mt));
      const int m = w0.mt - J.tile0;
      // four-bit: the row's power-of-two scaling for this run (found before
      // the run's first unit, see run_pow2)
      float unscale = 1.f;
      if (KIND == W_KIND_I4) {
        const int p = p_next;
        unscale = ldexpf(1.f, -p);
        for (int64_t v = u; v < ue && ok; ++v, ++i) {
          const int s = i % S, a = i % C::SA;
          if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * s, (i / S) & 1))) {
            ok = false;
            break;
          }
          if (i >= C::SA && !__all_sync(0xffffffffu, mbar_wait(afree0 + 8 * a, ((i / C::SA) - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t *st = sm + s * stage;
          const uint4 c0 = *(const uint4 *)(st + b_bytes + r * 16);
          const uint4 c1 = *(const uint4 *)(st + b_bytes + 2048 + r * 16);
          __half2 s2[DU];
#pragma unroll
          for (int du = 0; du < DU; ++du) {
            const float sv = __half2float(__ushort_as_half(*(const uint16_t *)(st + b_bytes + 4096 + du * 256 + r * 2)));
            s2[du] = __float2half2_rn(ldexpf(sv, p));
          }
          mbar_arrive(empty0 + 8 * s);
          const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
          uint32_t vh[32], vl[32];
#pragma unroll
          for (int jw = 0; jw < 8; ++jw) {
            uint32_t q4[4];
            dequant8(words[jw], q4);
            const __half2 sc2 = s2[DU == 2 ? jw / 4 : 0];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __half2 qv = *(const __half2 *)&q4[e];
              const __half2 h = __hmul2(qv, sc2);
              const __half2 l = __hfma2(qv, sc2, __hneg2(h));
              vh[4 * jw + e] = *(const uint32_t *)&h;
              vl[4 * jw + e] = *(const uint32_t *)&l;
            }
          }
          tmem_st32(tbase + lrow + C::A_COL + a * 64, vh);
          tmem_st32(tbase + lrow + C::A_COL + a * 64 + 32, vl);
          tc_wait_st();
          tc_fence_before();
          mbar_arrive(afull0 + 8 * a);
        }
        if (!ok) break;
        // the next run's scaling while the MMAs finish this run's last units
        if (ue < u1) p_next = run_pow2<DU>(A, ue, wrun_end(A, ue, u1), r);
      }
      // the run's partial sums into Y
      const int d = run % C::NBUF;
      if (!__all_sync(0xffffffffu, mbar_wait(dfull0 + 8 * d, (run / C::NBUF) & 1))) break;
      tc_fence_after();
      // a run over the whole k-range owns its outputs; the others add into cleared ones
      const bool whole = (ue - u) == A.KT;
      const int row0 = m * 128;
      const int rows = min(128, J.n - row0);
      float *ybase = J.y + A.y_off + row0;
      const int tok0 = w0.tt * N;
      const int ntok = min(N, A.T - tok0);
      const bool bulk = (rows & 3) == 0 && (J.ldy & 3) == 0 && (((uintptr_t)ybase) & 15) == 0;
      if (bulk) {
        // 16 tokens at a time: TMEM -> registers -> this warp's [token][32 rows]
        // slice in shared memory -> 16 bytes a lane, four tokens an instruction
        // (vector stores, or vector atomic adds for a split tile). Each warp
        // turns its own rows around, so the warps never wait for one another.
        float *stg = staging + warp * 16 * 32;
        const int rq = 4 * (lane & 7), eq = lane >> 3;  // a lane's 4 rows, and its token of each 4
        const bool rlive = warp * 32 + rq < rows;
        for (int c0 = 0; c0 < N; c0 += 16) {
          uint32_t v16[16];
          tmem_ld16(tbase + lrow + d * 256 + c0, v16);
          tc_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) stg[e * 32 + lane] = __uint_as_float(v16[e]) * unscale;
          __syncwarp();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int e = 4 * q + eq;
            if (rlive && c0 + e < ntok) {
              const float4 v = *(const float4 *)(stg + e * 32 + rq);
              float4 *dst = (float4 *)(ybase + (int64_t)(tok0 + c0 + e) * J.ldy + warp * 32 + rq);
              if (whole) *dst = v;
              else atomicAdd(dst, v);
            }
          }
          __syncwarp();
        }
      } else {
        const bool live = r < rows;
        float *y = ybase + r;
        for (int c0 = 0; c0 < N; c0 += 16) {
          uint32_t v16[16];
          tmem_ld16(tbase + lrow + d * 256 + c0, v16);
          tc_wait_ld();
          if (live)
            for (int e = 0; e < 16 && c0 + e < ntok; ++e) {
              const float v = __uint_as_float(v16[e]) * unscale;
              if (whole) y[(int64_t)(tok0 + c0 + e) * J.ldy] = v;
              else atomicAdd(y + (int64_t)(tok0 + c0 + e) * J.ldy, v);
            }
        }
      }
      tc_fence_before();
      mbar_arrive(dfree0 + 8 * d);
      u = ue;
    }
  }
  pdl_trigger();  // this CTA's work is done
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// ---------------------------------------------------------------- launch

// Token tiles of a wide GEMM: as few as fit 256 rows, of equal height (a multiple of 16).
void wide_tiles(int T, int &ntt, int &N) {
  ntt = (T + WIDE_MAX_N - 1) / WIDE_MAX_N;
  const int per = (T + ntt - 1) / ntt;
  N = (per + 15) / 16 * 16;
}

size_t wide_act_bytes(int T, int K, bool int4) {
  int ntt, N;
  wide_tiles(T, ntt, N);
  return (size_t)ntt * N * K * 2 * (int4 ? 2 : 1);
}

// The token tiles (blocks < pack_blocks) and the clearing of the row tiles
// that a boundary between two CTAs' ranges splits (their runs add into the
// outputs; runs over a whole k-range store). Clearing block b takes boundary
// b / WZ_PARTS and a part of that tile's token rows.
constexpr int WZ_PARTS = 8;

// Clearing block zb: boundary q = zb / WZ_PARTS + 1 between two CTAs' ranges,
// when it falls inside a row tile's k-range, and part zb % WZ_PARTS of that
// tile's token rows (the runs on either side add into them).
__device__ void wide_clear(const WideArgs &A, int Q, int zb) {
  const int part = zb % WZ_PARTS, q = zb / WZ_PARTS + 1;
  int64_t u, up, un;
  wrange(A, q, Q, u, un);
  if (u % A.KT == 0 || u >= A.units) return;
  // the tile was cleared for the boundary before if that one split it too
  wrange(A, q - 1, Q, up, un);
  if (q > 1 && up % A.KT != 0 && up / A.KT == u / A.KT) return;
  const int64_t tg = u / A.KT;
  const int tt = (int)(tg / A.mtiles), mt = (int)(tg % A.mtiles);
  const WideJob J = A.job[wjob_of(A, mt)];
  const int row0 = (mt - J.tile0) * 128;
  const int rows = min(128, J.n - row0);
  const int toks = min(A.N, A.T - tt * A.N);
  const int per = (toks + WZ_PARTS - 1) / WZ_PARTS;
  const int t0 = part * per, t1 = min(toks, t0 + per);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  float *base = J.y + A.y_off + (int64_t)(tt * A.N) * J.ldy + row0;
  const bool v4 = rows == 128 && (J.ldy & 3) == 0 && (((uintptr_t)base) & 15) == 0;
  for (int t = t0 + warp; t < t1; t += nw) {
    float *y = base + (int64_t)t * J.ldy;
    if (v4) ((float4 *)y)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
    else
      for (int r = lane; r < rows; r += 32) y[r] = 0.f;
  }
}

// With x_ready (X and dst depend on no kernel before this one), the packing
// blocks do their work before the dependency wait and wait at the end, so that
// the kernel still completes only after the one before it; the clearing blocks
// always wait first (the outputs may still be read before).
template <int PLANES>
__global__ void k_wide_pack(const float *__restrict__ X, int ldx, WideArgs A, int Q, uint4 *__restrict__ dst,
                            int pack_blocks, int x_ready) {
  if (!x_ready) pdl_wait();
  pdl_trigger();
  if ((int)blockIdx.x < pack_blocks) {
    const int64_t total = (int64_t)A.ntt * A.KT * A.N * 8;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t < total) pack_act_chunk<PLANES>(X, ldx, A.T, A.K, A.N, dst, t);
    if (x_ready) pdl_wait();
    return;
  }
  if (x_ready) pdl_wait();
  wide_clear(A, Q, blockIdx.x - pack_blocks);
}

// The token tiles of rows that still need their RMS norm (the settle's t before
// the K/V GEMM): block b < ntt * N takes token row b, x * (mean(x^2) + eps)^-1/2
// * w into its packed chunks (zeros past T); the blocks past them clear split
// tiles as k_wide_pack does. One launch and one round trip of the rows fewer
// than a norm kernel before the packing.
constexpr int WR_THREADS = 256;
constexpr int WR_CHUNKS = 3;  // 8-column chunks a thread holds: rows of up to 6,144 columns in registers
template <int PLANES>
__global__ void __launch_bounds__(WR_THREADS) k_wide_rms_pack(const float *__restrict__ X, int ldx,
                                                              const float *__restrict__ w, float eps, WideArgs A, int Q,
                                                              uint4 *__restrict__ dst, int pack_blocks) {
  pdl_wait();
  pdl_trigger();
  if ((int)blockIdx.x >= pack_blocks) {
    // the split tiles' outputs: the clearing blocks of k_wide_pack
    wide_clear(A, Q, blockIdx.x - pack_blocks);
    return;
  }
  const int tok = blockIdx.x;
  const PackDst P{dst, A.N, PLANES, A.KT};
  const int nc = A.K / 8;  // 8-column chunks of a row
  if (tok >= A.T) {
    const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int c = threadIdx.x; c < nc; c += WR_THREADS) pack_store8(P, tok, 8 * c, z);
    return;
  }
  const float *xr = X + (int64_t)tok * ldx;
  __shared__ float red[WR_THREADS / 32];
  const bool aligned = (((uintptr_t)xr) & 15) == 0;
  if (nc <= WR_CHUNKS * WR_THREADS && aligned) {
    // the row stays in registers between its sum of squares and its packing
    // (chunk c = threadIdx.x + j * WR_THREADS, all loads in flight together)
    float v[WR_CHUNKS][8];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < WR_CHUNKS; ++j) {
      const int c = threadIdx.x + j * WR_THREADS;
      if (c < nc) {
        const float4 a = __ldg((const float4 *)(xr + 8 * c)), b = __ldg((const float4 *)(xr + 8 * c) + 1);
        v[j][0] = a.x; v[j][1] = a.y; v[j][2] = a.z; v[j][3] = a.w;
        v[j][4] = b.x; v[j][5] = b.y; v[j][6] = b.z; v[j][7] = b.w;
      }
    }
#pragma unroll
    for (int j = 0; j < WR_CHUNKS; ++j)
      if (threadIdx.x + j * WR_THREADS < nc)
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(v[j][e], v[j][e], ss);
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < WR_THREADS / 32; ++i) tot += red[i];
    const float sc = 1.0f / sqrtf(tot / (float)A.K + eps);
#pragma unroll
    for (int j = 0; j < WR_CHUNKS; ++j) {
      const int c = threadIdx.x + j * WR_THREADS;
      if (c < nc) {
        float o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = v[j][e] * sc * __ldg(w + 8 * c + e);
        pack_store8(P, tok, 8 * c, o);
      }
    }
    return;
  }
  float ss = 0.f;
  for (int i = threadIdx.x; i < A.K; i += WR_THREADS) ss = fmaf(xr[i], xr[i], ss);
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < WR_THREADS / 32; ++i) tot += red[i];
  const float sc = 1.0f / sqrtf(tot / (float)A.K + eps);
  for (int c = threadIdx.x; c < nc; c += WR_THREADS) {
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = xr[8 * c + e] * sc * w[8 * c + e];
    pack_store8(P, tok, 8 * c, v);
  }
}

// Runs of at least this many units: a run ends with a read-back of its accumulator.
constexpr int W_MIN_RUN = 4;
// What a run's read-back and atomic add of its partial sums cost, in units.
constexpr int W_RUN_COST = 6;

// Ranges of equal cost: a CTA's units plus `run_cost` units for each run it
// holds (a run ends with a read-back of its accumulator, which, with one
// accumulator, the next run's MMAs wait for). The smallest cost C for which
// CTAs that each take as many units as C allows cover them all; the CTAs past
// the last units get none. A CTA's range is walked a tile at a time, and the
// ranges of a shape are kept (the settle asks for the same few shapes again
// and again).
static bool wide_cover(int64_t U, int64_t KT, int Q, int run_cost, int64_t C, int *bnd) {
  int64_t u = 0;
  for (int q = 0; q < Q; ++q) {
    if (bnd) bnd[q] = (int)u;
    int64_t budget = C;
    while (u < U && budget > run_cost) {
      if (u % KT == 0) {  // whole tiles at once, each a run
        const int64_t whole = std::min(budget / (KT + run_cost), (U - u) / KT);
        if (whole > 0) {
          u += whole * KT;
          budget -= whole * (KT + run_cost);
          continue;
        }
      }
      budget -= run_cost;  // a run begins at u
      const int64_t take = std::min(std::min(budget, (u / KT + 1) * KT - u), U - u);
      u += take;
      budget -= take;
      if (u % KT != 0) break;  // the budget ended inside the tile
    }
  }
  if (bnd) bnd[Q] = (int)U;
  return u >= U;
}

static void wide_bounds(WideArgs &A, int Q, int run_cost) {
  static std::mutex mu;
  static std::map<std::tuple<int64_t, int, int, int>, std::vector<int>> cache;
  const auto key = std::make_tuple(A.units, A.KT, Q, run_cost);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it == cache.end()) {
    const int64_t U = A.units, KT = A.KT;
    int64_t lo = (U + Q - 1) / Q, hi = U + (int64_t)run_cost * (U / KT + Q + 1);
    while (lo < hi) {
      const int64_t mid = (lo + hi) / 2;
      if (wide_cover(U, KT, Q, run_cost, mid, nullptr)) hi = mid;
      else lo = mid + 1;
    }
    std::vector<int> b(Q + 1);
    wide_cover(U, KT, Q, run_cost, lo, b.data());
    if (cache.size() > 256) cache.clear();
    it = cache.emplace(key, std::move(b)).first;
  }
  std::copy(it->second.begin(), it->second.end(), A.bnd);
  A.nbnd = Q + 1;
}

template <int KIND, int DU>
static cudaError_t launch_wide(WideArgs &A, const float *X, int ldx, const float *norm_w, float eps, void *act,
                               int num_sms, cudaStream_t st, bool x_ready) {
  using C = WCfg<KIND, DU>;
  static PerDevice smem_set, resident;   // per device: the limit raised; the resident CTAs (0 = not yet)
  auto kern = k_wide<KIND, DU>;
  int dev = 0;
  if (cudaError_t e = device_slot(dev)) return e;
  int max_ctas = resident.slot[dev].load(std::memory_order_acquire);
  if (max_ctas == 0) {
    cudaError_t e = smem_limit(kern, C::SMEM, smem_set);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, W_THREADS, C::SMEM);
    if (e != cudaSuccess) return e;
    max_ctas = std::max(1, per_sm) * num_sms;
    resident.slot[dev].store(max_ctas, std::memory_order_release);
  }
  A.units = (int64_t)A.ntt * A.mtiles * A.KT;
  // With no more (token tile, row tile) tiles than resident CTAs, each CTA may
  // take one tile over its whole k-range: no split tile (no clearing of Y, no
  // second read-back, plain stores instead of atomics), but KT units a CTA.
  // An even split costs units / Q a CTA plus, for each run it holds, a
  // read-back and atomic add of the run's partial sums, worth about W_RUN_COST
  // units. The cheaper one is taken (measured: whole tiles for the 0.6B K/V
  // and the batched projections, k-ranges of 16; split for the FCs and the
  // 27B K/V, k-ranges of 80 to 400).
  const int64_t tiles = (int64_t)A.ntt * A.mtiles;
  const int64_t q_split = std::max<int64_t>(1, std::min<int64_t>(max_ctas, A.units / W_MIN_RUN));
  const int64_t per = (A.units + q_split - 1) / q_split;
  const int64_t split_cost = per + W_RUN_COST * (1 + (per + A.KT - 1) / A.KT);
  const bool whole = tiles <= max_ctas && A.KT <= split_cost;
  const int Q = whole ? (int)tiles : (int)q_split;
  // four-bit split runs: ranges balanced by cost (a run's read-back blocks the
  // next run's MMAs; the f16 kernel drains one accumulator while it fills the other)
  A.nbnd = 0;
  if (KIND == W_KIND_I4 && !whole && Q <= WIDE_MAX_CTAS && A.units < INT32_MAX) wide_bounds(A, Q, W_RUN_COST);
  const int64_t chunks = (int64_t)A.ntt * A.KT * A.N * 8;
  const int zero_blocks = whole ? 0 : (Q - 1) * WZ_PARTS;
  cudaError_t e;
  if (norm_w) {
    const int pack_blocks = A.ntt * A.N;  // one block a token row
    e = launch_pdl(k_wide_rms_pack<C::PLANES>, dim3(pack_blocks + zero_blocks), dim3(WR_THREADS), 0, st, 1, X, ldx,
                   norm_w, eps, A, Q, (uint4 *)act, pack_blocks);
  } else {
    const int pack_blocks = (int)((chunks + 255) / 256);
    e = launch_pdl(k_wide_pack<C::PLANES>, dim3(pack_blocks + zero_blocks), dim3(256), 0, st, 1, X, ldx, A, Q,
                   (uint4 *)act, pack_blocks, (int)x_ready);
  }
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3((unsigned)Q), dim3(W_THREADS), C::SMEM, st, 1, A);
}

cudaError_t wide_gemm(const WideJob *jobs, int njobs, int64_t y_off, bool int4, int group, const float *X, int ldx,
                      int T, int K, void *act, int num_sms, cudaStream_t st, const float *norm_w, float eps,
                      bool x_ready) {
  if (x_ready && norm_w) return cudaErrorInvalidValue;  // the norm's packing waits first
  if (njobs < 1 || njobs > WIDE_MAX_JOBS || T < 1 || K % 64) return cudaErrorInvalidValue;
  WideArgs A{};
  A.njobs = njobs;
  A.mtiles = 0;
  for (int j = 0; j < njobs; ++j) {
    A.job[j] = jobs[j];
    A.job[j].tile0 = A.mtiles;
    A.mtiles += (jobs[j].n + 127) / 128;
  }
  A.y_off = y_off;
  A.bpack = (const uint8_t *)act;
  A.K = K;
  A.KT = K / 64;
  A.T = T;
  wide_tiles(T, A.ntt, A.N);
  if (!int4) return launch_wide<W_KIND_F16, 1>(A, X, ldx, norm_w, eps, act, num_sms, st, x_ready);
  return group >= 64 ? launch_wide<W_KIND_I4, 1>(A, X, ldx, norm_w, eps, act, num_sms, st, x_ready)
                     : launch_wide<W_KIND_I4, 2>(A, X, ldx, norm_w, eps, act, num_sms, st, x_ready);
}

// This file's device error word (a bounded wait that gave up).
cudaError_t wide_read_error(unsigned *out, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_dev_error, sizeof(unsigned));
  if (e == cudaSuccess && reset) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_dev_error, &zero, sizeof(unsigned));
  }
  return e;
}

}  // namespace dfl

// Weight GEMMs of the drafter on the 5th-generation tensor cores (tcgen05):
// Y[t][n] = sum_k X[t][k] W[n][k] for the four-bit matrices (q, k, v, o, gate,
// up, down, head) and the f16 ones (fc, the kernel projections, the selector's
// projection); cortiq-engine src/gpu_cuda/hyb/dflash.rs (`Dev::settle`,
// `Dev::block`) names which is which.
//
// One CTA owns a 128-row tile of one matrix, a tile of TT tokens and a range of
// 64-column k-tiles. Warp 4 streams the k-tiles into a shared-memory ring with
// bulk copies; warp 5 issues tcgen05.mma (M = 128 weight rows, N = TT tokens,
// K = 16) into tensor memory.
//
// Four-bit matrices: warps 0-3 own one weight row each. They turn the row's
// codes into exact f16 integers (-7..7) and store them in tensor memory, where
// the MMA reads its A operand; the tokens enter as two f16 planes, hi = f16(x)
// and lo = f16(x - hi), both accumulated into the same tensor-memory columns.
// Each quantisation group has its own accumulator, which the same warps read
// back, multiply by the group's f16 scale in f32 and add up in registers: the
// dequantisation is exact and no shared-memory bandwidth is spent on A.
//
// f16 matrices: the weight tiles go to shared memory by bulk copy as they are
// (pre-swizzled by the packer) and the tokens enter rounded to f16 (the card
// arm's `to_half`); one accumulator spans the CTA's k-range.
#include <algorithm>
#include <climits>
#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace dfl {

constexpr int TC_THREADS = 192;  // warps 0-3 rows / epilogue, 4 producer, 5 MMA
constexpr int TC_PRODUCER = 4;
constexpr int TC_MMA = 5;
constexpr int TC_STAGES = 4;
constexpr uint32_t TC_TMEM_COLS = 256;

// ---------------------------------------------------------------- packed layouts

size_t tc_int4_codes_bytes(int64_t rows, int64_t cols) { return (size_t)((rows + 127) / 128) * 128 * cols / 2; }
static int drain_units(int group) { return group >= 64 ? 1 : 2; }
size_t tc_int4_scale_bytes(int64_t rows, int64_t cols, int group) {
  return (size_t)((rows + 127) / 128) * (cols / 64) * drain_units(group) * 256;
}
size_t tc_f16_bytes(int64_t rows, int64_t cols) { return (size_t)((rows + 127) / 128) * 128 * cols * 2; }

// Codes: per (row tile m, k-tile kt) 4 KiB = [half h][row r][16 B]; the 16 B of
// (r, h) hold columns 32h .. 32h+31 as four u32 of eight nibbles (q + 8) in the
// order c0 c2 c4 c6 c1 c3 c5 c7 of their eight columns, so that two lop3 give
// the f16 pairs (c0,c1), (c2,c3), ... Rows past the matrix are code 8 (q = 0).
__global__ void k_tc_pack_int4(const uint8_t *__restrict__ codes, int64_t rows, int64_t cols,
                               uint32_t *__restrict__ dst) {
  const int64_t KT = cols / 64;
  const int64_t MT = (rows + 127) / 128;
  const int64_t total = MT * KT * 2 * 128 * 4;  // u32 words
  int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= total) return;
  const int j = (int)(t & 3);
  const int r = (int)((t >> 2) & 127);
  const int h = (int)((t >> 9) & 1);
  const int64_t tile = t >> 10;
  const int64_t m = tile / KT, kt = tile % KT;
  const int64_t row = m * 128 + r;
  uint32_t w = 0;
  for (int i = 0; i < 8; ++i) {
    const int e = (i < 4) ? 2 * i : 2 * (i - 4) + 1;  // nibble i holds column e of the eight
    const int64_t col = kt * 64 + 32 * h + 8 * j + e;
    uint32_t nib = 8;
    if (row < rows) {
      const uint8_t byte = codes[row * (cols / 2) + col / 2];
      nib = (col & 1) ? (byte >> 4) : (byte & 15);
    }
    w |= nib << (4 * i);
  }
  dst[t] = w;
}

// Scales: per (m, kt) [drain unit u][row r] f16; unit u covers columns
// kt*64 + 32u .. (both units share the group's scale when the group is >= 64).
__global__ void k_tc_pack_scales(const uint16_t *__restrict__ scales, int64_t rows, int64_t cols, int group,
                                 uint16_t *__restrict__ dst) {
  const int64_t KT = cols / 64;
  const int64_t MT = (rows + 127) / 128;
  const int DU = group >= 64 ? 1 : 2;
  const int64_t total = MT * KT * DU * 128;
  int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= total) return;
  const int r = (int)(t & 127);
  const int u = (int)((t >> 7) % DU);
  const int64_t tile = (t >> 7) / DU;
  const int64_t m = tile / KT, kt = tile % KT;
  const int64_t row = m * 128 + r;
  const int64_t col = kt * 64 + 32 * u;
  dst[t] = row < rows ? scales[row * (cols / group) + col / group] : (uint16_t)0;
}

// f16 matrix: per (m, kt) 16 KiB, 128 rows x 64 columns, K-major with the
// 128-byte swizzle; rows past the matrix are zero.
__global__ void k_tc_pack_f16(const uint16_t *__restrict__ src, int64_t rows, int64_t cols, uint4 *__restrict__ dst) {
  const int64_t KT = cols / 64;
  const int64_t MT = (rows + 127) / 128;
  const int64_t total = MT * KT * 128 * 8;  // 16-byte chunks
  int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= total) return;
  const int c = (int)(t & 7);
  const int r = (int)((t >> 3) & 127);
  const int64_t tile = t >> 10;
  const int64_t m = tile / KT, kt = tile % KT;
  const int64_t row = m * 128 + r;
  uint32_t v[4] = {0, 0, 0, 0};
  if (row < rows) {
    const uint16_t *p = src + row * cols + kt * 64 + c * 8;
    for (int i = 0; i < 4; ++i) v[i] = (uint32_t)p[2 * i] | ((uint32_t)p[2 * i + 1] << 16);
  }
  dst[tile * 1024 + sw128_off(r, c) / 16] = make_uint4(v[0], v[1], v[2], v[3]);
}

// Outputs a split-K launch accumulates into, cleared first: T rows of n floats.
constexpr int MAX_JOBS = 4;
struct ZeroJobs {
  float *y[MAX_JOBS];
  int ldy[MAX_JOBS];
  int n[MAX_JOBS];
  int njobs;
};

// The token tiles of a GEMM (blocks < pack_blocks) and the clearing of its
// outputs (the other blocks).
template <int PLANES>
__global__ void k_tc_pack_act(const float *__restrict__ X, int ldx, int T, int K, int TT, uint4 *__restrict__ dst,
                              ZeroJobs Z, int pack_blocks) {
  pdl_wait();
  pdl_trigger();
  if ((int)blockIdx.x >= pack_blocks) {
    // segments of 2048 outputs of one token row, round robin over the clearing blocks
    const int zb = blockIdx.x - pack_blocks, nzb = gridDim.x - pack_blocks;
    int seg0 = 0;
    for (int j = 0; j < Z.njobs; ++j) {
      const int per_row = (Z.n[j] + 2047) / 2048;
      const int segs = T * per_row;
      int first = zb - seg0 % nzb;
      if (first < 0) first += nzb;
      for (int sg = first; sg < segs; sg += nzb) {
        const int t = sg / per_row, c0 = (sg - t * per_row) * 2048;
        float *y = Z.y[j] + (int64_t)t * Z.ldy[j];
        const int c1 = min(Z.n[j], c0 + 2048);
        for (int c = c0 + threadIdx.x; c < c1; c += blockDim.x) y[c] = 0.f;
      }
      seg0 += segs;
    }
    return;
  }
  const int64_t total = (int64_t)((T + TT - 1) / TT) * (K / 64) * TT * 8;
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t < total) pack_act_chunk<PLANES>(X, ldx, T, K, TT, dst, t);
}

// ---------------------------------------------------------------- jobs
struct TcJobs {
  const void *w[MAX_JOBS];        // packed codes / f16 tiles
  const uint16_t *s[MAX_JOBS];    // packed scales (four-bit)
  float *y[MAX_JOBS];
  int n[MAX_JOBS];                // rows
  int ldy[MAX_JOBS];
  int tile0[MAX_JOBS + 1];        // first row tile of each job in the grid's y
  int njobs;
};

__device__ __forceinline__ int job_of(const TcJobs &J, int mt) {
  int j = 0;
#pragma unroll
  for (int i = 1; i < MAX_JOBS; ++i)
    if (i < J.njobs && mt >= J.tile0[i]) j = i;
  return j;
}

// ---------------------------------------------------------------- four-bit kernel
// The shape used: two CTAs an SM (256 tensor-memory columns each), stages of
// two k-tiles, four dequantising warps, two issuing warps a row tile, both
// activation planes into one accumulator. Measured on the head (151,936 x
// 5,120, 15 rows): one CTA an SM with 512 columns, eight dequantising warps or
// four-k-tile stages were each slower; see the kernel comment for why the
// issuing warps matter.
constexpr int I4_CPS = 2, I4_KS = 2, I4_NDQ = 4, I4_P = 2, I4_FOLD = 1;
//
// Persistent CTAs walk a list of items (MT row tiles of one matrix, a token
// tile, a k-range); the k-tiles of consecutive items flow through one pipeline:
//   producer      copies a stage of KS k-tiles: one tensor copy of the MT row
//                 tiles' codes, one of their scales (boxes of MT tiles x KS
//                 k-tiles; past a matrix's last tile or k-tile they read zeros),
//                 one bulk copy of the tokens' hi/lo planes
//   NDQ warps     dequantise each k-tile's codes into a tensor-memory A slot
//                 (8 warps: two a lane quarter, one half of the columns each)
//   MT x P warps  issue the MMAs: P warps a row tile, taking its k-tiles in
//                 turn; with FOLD the hi and the lo plane go into the same
//                 accumulator (two MMAs of N = TT), else one MMA of N = 2 TT
//   4 warps       read each accumulator back, scale it and add it up; at the
//                 end of an item they write the item's rows, and they free a
//                 stage once its last k-tile is drained
// Measured on this GPU: an MMA of M = 128, K = 16 holds its issuing thread for
// about 150 cycles whatever its N, while MMAs issued from different warps
// overlap; so the issue is spread over several warps. A CTA's bulk copies are
// served nearly one after another at a cost that hardly depends on their size
// up to 16 KiB, so a stage is a few large copies; A slots and accumulators still
// turn over per k-tile.
template <int TT, int DU, int MT, int KS, int CPS, int NDQ, int P, int FOLD>
struct I4 {
  static constexpr int DRAIN0 = NDQ;                           // 4 drain warps
  static constexpr int PRODUCER = NDQ + 4;
  static constexpr int MMA0 = NDQ + 5;                         // MT x P issuing warps
  static constexpr int THREADS = 32 * (MMA0 + MT * P);
  static constexpr uint32_t TMEM_COLS = CPS == 1 ? 512 : 256;  // CPS CTAs an SM share its 512 columns
  static constexpr int B1 = 2 * TT * 128;                      // hi + lo planes of one k-tile
  static constexpr int CODE_OFF = KS * B1;                     // MT x KS x 4 KiB
  static constexpr int SCALE_OFF = CODE_OFF + MT * KS * 4096;  // MT x KS x DU x 256 B
  static constexpr int STAGE = ((SCALE_OFF + MT * KS * DU * 256) + 1023) / 1024 * 1024;
  static constexpr int S_FIT = (CPS == 1 ? 196 : 108) * 1024 / STAGE;
  static constexpr int S = S_FIT < 16 ? S_FIT : 16;            // shared-memory stages
  static_assert(S >= 2, "shared memory");
  static constexpr int AW = MT * 32;                           // A columns of a slot
  static constexpr int SA = CPS == 1 ? 4 : 2;                  // tensor-memory A slots
  static constexpr int DW = MT * TT * (FOLD ? 1 : 2);          // accumulator columns of a unit
  static constexpr int DCOL = SA * AW;
  static constexpr int NDU_FIT = ((int)TMEM_COLS - DCOL) / DW;
  static constexpr int NDU = NDU_FIT < 8 ? NDU_FIT : 8;        // accumulators in flight
  static_assert(NDU >= 2, "tensor memory");
  static constexpr int NBAR = 2 * S + 2 * SA + 2 * NDU;
  static constexpr int SMEM = S * STAGE + 1024 + 512;
};

// The units of a launch, (token tile, group of MT row tiles, k-tile), laid end
// to end; CTA b takes units [b U / grid, (b + 1) U / grid) ("stream-K"), as runs
// that each stay inside one group's k-range. A run over the whole k-range
// stores its rows; a shorter one adds them into outputs cleared beforehand.
// Per job: the codes as bytes (256, 16, k-tile, row tile), boxes (256, 16, KS,
// MT), and the scales as bytes (256, DU, k-tile, row tile), boxes (256, DU, KS,
// MT), so that one copy brings a stage's codes (or scales) of all MT tiles.
// A box spans min(KS, k-tiles) k-tiles and min(MT, row tiles) tiles of its
// matrix; wbox is the bytes of the two boxes, ksb the k-tiles of a box (the
// stride of a tile's codes in the stage).
struct I4Maps {
  CUtensorMap code[MAX_JOBS], scale[MAX_JOBS];
  int wbox[MAX_JOBS];
  int ksb;
};

struct I4Items {
  int groups;       // row-tile groups over all jobs
  int gtile0[MAX_JOBS + 1];
  int ntt;
  int units;        // < 2^31 (checked at launch)
  int whole;        // CTA ranges at group boundaries (when there are as many groups as CTAs)
  // With whole runs and one job (the head): the selector's first stage, the
  // largest key (value, then lower row) of each chunk of I4_KEY_CHUNK rows per
  // token, added with atomicMax into cmax[token * nchunks + chunk] (cleared
  // by the producer before); null: none.
  unsigned long long *cmax;
  int nchunks;
};
constexpr int I4_KEY_CHUNK = 2048;

// The run that starts at unit u and ends at the group's last k-tile or at u1.
__device__ __forceinline__ void i4_run(const TcJobs &J, const I4Items &P, int MT, int KT, int u, int u1, int &job,
                                       int &m0, int &mtv, int &tt, int &kt0, int &kt1) {
  const int tg = u / KT;
  kt0 = u - tg * KT;
  const int mg = tg % P.groups;
  tt = tg / P.groups;
  kt1 = min(KT, kt0 + (u1 - u));
  job = 0;
#pragma unroll
  for (int i = 1; i < MAX_JOBS; ++i)
    if (i < J.njobs && mg >= P.gtile0[i]) job = i;
  m0 = (mg - P.gtile0[job]) * MT;
  const int tiles = J.tile0[job + 1] - J.tile0[job];
  mtv = min(MT, tiles - m0);
}

template <int TT, int DU, int MT, int KS, int CPS, int NDQ, int NP, int FOLD>
__global__ void __launch_bounds__(32 * (NDQ + 5 + MT * NP), CPS)
    k_tc_int4(const __grid_constant__ I4Maps M, TcJobs J, I4Items P, const uint8_t *__restrict__ bpack, int K, int T) {
  using C = I4<TT, DU, MT, KS, CPS, NDQ, NP, FOLD>;
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t *sm = smraw + ((1024 - (smem_u32(smraw) & 1023)) & 1023);
  uint64_t *bars = (uint64_t *)(sm + C::S * C::STAGE);
  uint32_t *tslot = (uint32_t *)(bars + C::NBAR);
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * C::S, afull0 = empty0 + 8 * C::S;
  const uint32_t afree0 = afull0 + 8 * C::SA, dfull0 = afree0 + 8 * C::SA, dfree0 = dfull0 + 8 * C::NDU;
  const int KT = K / 64;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int ru0, ru1;
  if (P.whole) {
    const int ng = P.units / KT;
    ru0 = (int)((int64_t)blockIdx.x * ng / gridDim.x) * KT;
    ru1 = (int)((int64_t)(blockIdx.x + 1) * ng / gridDim.x) * KT;
  } else {
    ru0 = (int)((int64_t)blockIdx.x * P.units / gridDim.x);
    ru1 = (int)((int64_t)(blockIdx.x + 1) * P.units / gridDim.x);
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::S; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, 4);  // one arrive per drain warp
    }
    for (int i = 0; i < C::SA; ++i) {
      mbar_init(afull0 + 8 * i, NDQ);  // one arrive per dequantising warp
      mbar_init(afree0 + 8 * i, MT);
    }
    for (int i = 0; i < C::NDU; ++i) {
      mbar_init(dfull0 + 8 * i, MT);
      mbar_init(dfree0 + 8 * i, 4);
    }
    mbar_fence_init();
  }
  __syncthreads();
  // The weights do not depend on the kernels before this one: the first stages'
  // codes and scales are fetched before waiting for them.
  int npre = 0;
  if (warp == C::PRODUCER && lane == 0) {
    int job, m0, mtv, tt, kt0, kt1;
    for (int pu = ru0; pu < ru1 && npre < C::S; pu += kt1 - kt0) {
      i4_run(J, P, MT, KT, pu, ru1, job, m0, mtv, tt, kt0, kt1);
      for (int kt = kt0; kt < kt1 && npre < C::S; kt += KS, ++npre) {
        const int n = min(KS, kt1 - kt);
        const uint32_t st = smem_u32(sm + npre * C::STAGE), fb = full0 + 8 * npre;
        mbar_expect_tx(fb, n * C::B1 + M.wbox[job]);
        tma_load4(st + C::CODE_OFF, &M.code[job], 0, 0, kt, m0, fb);
        tma_load4(st + C::SCALE_OFF, &M.scale[job], 0, 0, kt, m0, fb);
      }
    }
  }
  pdl_wait();
  if (warp == 0) tmem_alloc(smem_u32(tslot), C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp == C::PRODUCER) {
    if (lane == 0) {
      int g = 0;
      bool ok = true;
      int job, m0, mtv, tt, kt0, kt1;
      for (int pu = ru0; pu < ru1 && ok; pu += kt1 - kt0) {
        i4_run(J, P, MT, KT, pu, ru1, job, m0, mtv, tt, kt0, kt1);
        const uint8_t *bp = bpack + (int64_t)tt * KT * C::B1;
        for (int kt = kt0; kt < kt1; kt += KS, ++g) {
          const int n = min(KS, kt1 - kt), s = g % C::S;
          const uint32_t st = smem_u32(sm + s * C::STAGE), fb = full0 + 8 * s;
          if (g >= npre) {
            if (g >= C::S && !mbar_wait(empty0 + 8 * s, ((g / C::S) - 1) & 1)) {
              ok = false;
              break;
            }
            mbar_expect_tx(fb, n * C::B1 + M.wbox[job]);
            tma_load4(st + C::CODE_OFF, &M.code[job], 0, 0, kt, m0, fb);
            tma_load4(st + C::SCALE_OFF, &M.scale[job], 0, 0, kt, m0, fb);
          }
          bulk_g2s(st, bp + (int64_t)kt * C::B1, n * C::B1, fb);
        }
      }
    }
  } else if (warp >= C::MMA0) {
    if (lane == 0) {
      // this warp's row tile of the item, and its share of the k-tiles (those
      // with i % NP == pw): an MMA holds its issuing thread for about 150
      // cycles whatever its N, so several warps issue side by side
      const int jj = (warp - C::MMA0) % MT, pw = (warp - C::MMA0) / MT;
      constexpr uint32_t idesc = f16_idesc(128, FOLD ? TT : 2 * TT);
      constexpr int KSU = 4 / DU;
      int g = 0, i = 0, u = 0;
      bool ok = true;
      int job, m0, mtv, tt, kt0, kt1;
      for (int pu = ru0; pu < ru1 && ok; pu += kt1 - kt0) {
        i4_run(J, P, MT, KT, pu, ru1, job, m0, mtv, tt, kt0, kt1);
        const bool live = jj < mtv;
        for (int kt = kt0; kt < kt1 && ok; kt += KS, ++g) {
          const int n = min(KS, kt1 - kt), s = g % C::S;
          if (!mbar_wait(full0 + 8 * s, (g / C::S) & 1)) {
            ok = false;
            break;
          }
          const uint32_t st = smem_u32(sm + s * C::STAGE);
          for (int sub = 0; sub < n && ok; ++sub, ++i) {
            if (NP > 1 && i % NP != pw) {
              u += DU;
              continue;
            }
            const int a = i % C::SA;
            if (!mbar_wait(afull0 + 8 * a, (i / C::SA) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t bsub = st + sub * C::B1;
            for (int du = 0; du < DU; ++du, ++u) {
              const int d = u % C::NDU;
              if (u >= C::NDU && !mbar_wait(dfree0 + 8 * d, ((u / C::NDU) - 1) & 1)) {
                ok = false;
                break;
              }
              tc_fence_after();
              if (live) {
                // both activation planes into one accumulator: the hi rows of the
                // B tile, then its lo rows (TT rows = TT * 128 bytes further on)
                const uint32_t dcol = tbase + C::DCOL + d * C::DW + jj * (C::DW / MT);
                // the descriptor's start address counts 16-byte units: a k-step
                // (32 bytes) is +2, the lo plane (TT rows of 128 bytes) + TT * 8
                const uint64_t bdesc = sw128_desc(bsub + du * KSU * 32);
                const uint32_t acol0 = tbase + a * C::AW + jj * 32 + du * KSU * 8;
#pragma unroll
                for (int ks = 0; ks < KSU; ++ks) {
                  mma_ts(dcol, acol0 + ks * 8, bdesc + 2 * ks, idesc, ks > 0);
                  if (FOLD) mma_ts(dcol, acol0 + ks * 8, bdesc + 2 * ks + TT * 8, idesc, 1);
                }
              }
              mma_commit(dfull0 + 8 * d);
            }
            mma_commit(afree0 + 8 * a);
          }
        }
      }
    }
  } else if (warp < NDQ) {
    // dequantise: thread r of lane quarter warp % 4 owns row r of each of the
    // item's tiles; with 8 warps, warp / 4 picks the half of the 64 columns
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lrow = (uint32_t)((warp & 3) * 32) << 16;
    constexpr int HALVES = NDQ == 8 ? 1 : 2;  // column halves a thread dequantises
    const int h0 = NDQ == 8 ? warp >> 2 : 0;
    int g = 0, i = 0;
    bool ok = true;
    int job, m0, mtv, tt, kt0, kt1;
    for (int pu = ru0; pu < ru1 && ok; pu += kt1 - kt0) {
      i4_run(J, P, MT, KT, pu, ru1, job, m0, mtv, tt, kt0, kt1);
      for (int kt = kt0; kt < kt1 && ok; kt += KS, ++g) {
        const int n = min(KS, kt1 - kt), s = g % C::S;
        if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * s, (g / C::S) & 1))) {
          ok = false;
          break;
        }
        const uint8_t *st = sm + s * C::STAGE;
        for (int sub = 0; sub < n; ++sub, ++i) {
          const int a = i % C::SA;
          if (i >= C::SA && !__all_sync(0xffffffffu, mbar_wait(afree0 + 8 * a, ((i / C::SA) - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int jj = 0; jj < MT; ++jj) {
            if (jj < mtv) {
              const uint8_t *cp = st + C::CODE_OFF + (jj * M.ksb + sub) * 4096 + r * 16;
#pragma unroll
              for (int hh = 0; hh < HALVES; ++hh) {
                const int h = h0 + hh;
                const uint4 c = *(const uint4 *)(cp + h * 2048);
                const uint32_t words[4] = {c.x, c.y, c.z, c.w};
                uint32_t v[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  uint32_t a4[4];
                  dequant8(words[j], a4);
                  v[4 * j + 0] = a4[0];
                  v[4 * j + 1] = a4[1];
                  v[4 * j + 2] = a4[2];
                  v[4 * j + 3] = a4[3];
                }
                tmem_st16(tbase + lrow + a * C::AW + jj * 32 + h * 16, v);
              }
            }
          }
          tc_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(afull0 + 8 * a);
        }
      }
    }
  } else if (warp < C::DRAIN0 + 4) {
    // drain: 4 warps read the accumulators of their lane quarter
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lrow = (uint32_t)((warp & 3) * 32) << 16;
    float acc[MT][TT];
#pragma unroll
    for (int jj = 0; jj < MT; ++jj)
#pragma unroll
      for (int t = 0; t < TT; ++t) acc[jj][t] = 0.f;
    int g = 0, i = 0, u = 0;
    bool ok = true;
    int job, m0, mtv, tt, kt0, kt1;
    for (int pu = ru0; pu < ru1 && ok; pu += kt1 - kt0) {
      i4_run(J, P, MT, KT, pu, ru1, job, m0, mtv, tt, kt0, kt1);
      for (int kt = kt0; kt < kt1 && ok; kt += KS, ++g) {
        const int n = min(KS, kt1 - kt), s = g % C::S;
        if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * s, (g / C::S) & 1))) {
          ok = false;
          break;
        }
        const uint8_t *st = sm + s * C::STAGE;
        for (int sub = 0; sub < n && ok; ++sub, ++i) {
          float sc[MT][DU];
#pragma unroll
          for (int jj = 0; jj < MT; ++jj)
#pragma unroll
            for (int du = 0; du < DU; ++du)
              sc[jj][du] = jj < mtv ? __half2float(__ushort_as_half(*(const uint16_t *)(
                                          st + C::SCALE_OFF + ((jj * M.ksb + sub) * DU + du) * 256 + r * 2)))
                                    : 0.f;
#pragma unroll
          for (int du = 0; du < DU; ++du, ++u) {
            const int d = u % C::NDU;
            if (!__all_sync(0xffffffffu, mbar_wait(dfull0 + 8 * d, (u / C::NDU) & 1))) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int jj = 0; jj < MT; ++jj) {
              if (jj < mtv) {
#pragma unroll
                for (int c0 = 0; c0 < TT; c0 += 16) {
                  const uint32_t col = tbase + lrow + C::DCOL + d * C::DW + jj * (C::DW / MT) + c0;
                  uint32_t w[16];
                  tmem_ld16(col, w);
                  if (FOLD) {
                    tc_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) acc[jj][c0 + e] = fmaf(sc[jj][du], __uint_as_float(w[e]), acc[jj][c0 + e]);
                  } else {
                    uint32_t wl[16];
                    tmem_ld16(col + TT, wl);
                    tc_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                      acc[jj][c0 + e] =
                          fmaf(sc[jj][du], __uint_as_float(w[e]) + __uint_as_float(wl[e]), acc[jj][c0 + e]);
                  }
                }
              }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dfree0 + 8 * d);
          }
        }
        // the stage's codes, scales and tokens are no longer read (its MMAs
        // completed before their accumulators were drained)
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
      }
      if (!ok) break;
      // the item's rows
      float *y = J.y[job];
      const int ldy = J.ldy[job], n = J.n[job];
      if (P.cmax && kt1 - kt0 == KT) {
        // the chunk maxima of the values stored below: the item's MT tiles
        // start on an even tile, so they lie in one chunk of 2048 rows
        const int chunk = (m0 * 128) / I4_KEY_CHUNK;
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          const int tok = tt * TT + t;
          if (tok >= T) break;
          unsigned long long key = 0ull;
#pragma unroll
          for (int jj = 0; jj < MT; ++jj) {
            const int row = (m0 + jj) * 128 + r;
            if (jj < mtv && row < n) key = umax64(key, cand_key(acc[jj][t], (uint32_t)row));
          }
          key = warp_max_u64(key);
          if (lane == 0 && key) atomicMax(P.cmax + (int64_t)tok * P.nchunks + chunk, key);
        }
      }
#pragma unroll
      for (int jj = 0; jj < MT; ++jj) {
        const int row = (m0 + jj) * 128 + r;
        if (jj < mtv && row < n) {
#pragma unroll
          for (int t = 0; t < TT; ++t) {
            const int tok = tt * TT + t;
            if (tok < T) {
              if (kt1 - kt0 < KT) atomicAdd(y + (int64_t)tok * ldy + row, acc[jj][t]);
              else y[(int64_t)tok * ldy + row] = acc[jj][t];
            }
          }
        }
#pragma unroll
        for (int t = 0; t < TT; ++t) acc[jj][t] = 0.f;
      }
    }
  }
  pdl_trigger();  // this CTA's work is done
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- f16 kernel
template <int TT>
struct F16Cfg {
  static constexpr int B_BYTES = TT * 128;
  static constexpr int A_OFF = B_BYTES;
  static constexpr int STAGE = B_BYTES + 16384;
  static constexpr int STAGES = TT >= 128 ? 4 : 6;
  static constexpr int SMEM = STAGES * STAGE + 1024 + 256;
  static constexpr uint32_t COLS = TT <= 32 ? 32 : TT;
};

template <int TT>
__global__ void __launch_bounds__(TC_THREADS) k_tc_f16(TcJobs J, const uint8_t *__restrict__ bpack, int bstride, int K,
                                                       int T, int kc, int atomic_out) {
  using C = F16Cfg<TT>;
  constexpr int S = C::STAGES;
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t *sm = smraw + ((1024 - (smem_u32(smraw) & 1023)) & 1023);
  uint64_t *bars = (uint64_t *)(sm + S * C::STAGE);
  uint32_t *tslot = (uint32_t *)(bars + 2 * S + 1);
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * S, done = empty0 + 8 * S;

  const int KT = K / 64;
  const int tt = blockIdx.x, mt = blockIdx.y;
  const int kt0 = blockIdx.z * kc, kt1 = min(KT, kt0 + kc);
  const int n = kt1 - kt0;
  if (n <= 0) {
    pdl_wait();
    pdl_trigger();
    return;
  }
  const int job = job_of(J, mt);
  const int m = mt - J.tile0[job];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, 1);
    }
    mbar_init(done, 1);
    mbar_fence_init();
  }
  __syncthreads();
  // the first stages' weight tiles before waiting for the kernels this one follows
  const uint8_t *wa = (const uint8_t *)J.w[job] + ((int64_t)m * KT) * 16384;
  const int npre = n < S ? n : S;
  if (warp == TC_PRODUCER && lane == 0)
    for (int i = 0; i < npre; ++i) {
      mbar_expect_tx(full0 + 8 * i, C::B_BYTES + 16384);
      bulk_g2s(smem_u32(sm + i * C::STAGE) + C::A_OFF, wa + (int64_t)(kt0 + i) * 16384, 16384, full0 + 8 * i);
    }
  pdl_wait();
  if (warp == 0) tmem_alloc(smem_u32(tslot), C::COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp == TC_PRODUCER) {
    if (lane == 0) {
      const uint8_t *bp = bpack + ((int64_t)tt * KT) * bstride;
      for (int i = 0; i < n; ++i) {
        const int s = i % S, kt = kt0 + i;
        const uint32_t st = smem_u32(sm + s * C::STAGE);
        if (i >= npre) {
          if (i >= S && !mbar_wait(empty0 + 8 * s, ((i / S) - 1) & 1)) break;
          mbar_expect_tx(full0 + 8 * s, C::B_BYTES + 16384);
          bulk_g2s(st + C::A_OFF, wa + (int64_t)kt * 16384, 16384, full0 + 8 * s);
        }
        bulk_g2s(st, bp + (int64_t)kt * bstride, C::B_BYTES, full0 + 8 * s);
      }
    }
  } else if (warp == TC_MMA) {
    if (lane == 0) {
      constexpr uint32_t idesc = f16_idesc(128, TT);
      for (int i = 0; i < n; ++i) {
        const int s = i % S;
        if (!mbar_wait(full0 + 8 * s, (i / S) & 1)) break;
        tc_fence_after();
        const uint32_t st = smem_u32(sm + s * C::STAGE);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_ss(tbase, sw128_desc(st + C::A_OFF + ks * 32), sw128_desc(st + ks * 32), idesc, (i > 0 || ks > 0));
        mma_commit(empty0 + 8 * s);
      }
      mma_commit(done);
    }
  } else {
    const int r = warp * 32 + lane;
    const uint32_t lrow = (uint32_t)(warp * 32) << 16;
    const bool ok = __all_sync(0xffffffffu, mbar_wait(done, 0));
    tc_fence_after();
    const int row = m * 128 + r;
    if (ok) {
      float *y = J.y[job];
      const int ldy = J.ldy[job];
      const bool live = row < J.n[job];
#pragma unroll 1
      for (int c0 = 0; c0 < TT; c0 += 16) {
        uint32_t w16[16];
        tmem_ld16(tbase + lrow + c0, w16);
        tc_wait_ld();
        if (live) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int tok = tt * TT + c0 + e;
            if (tok < T) {
              if (atomic_out) atomicAdd(y + (int64_t)tok * ldy + row, __uint_as_float(w16[e]));
              else y[(int64_t)tok * ldy + row] = __uint_as_float(w16[e]);
            }
          }
        }
      }
    }
  }
  pdl_trigger();  // this CTA's work is done
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, C::COLS);
  }
}

// The exact values of packed four-bit codes, f32 [rows][cols]: the kernels'
// own dequantisation (dequant8) and scale layout, exposed for checking.
__global__ void k_tc_dequant(const uint4 *__restrict__ codes, const uint16_t *__restrict__ scales, int64_t rows,
                             int64_t cols, int DU, float *__restrict__ out) {
  const int64_t KT = cols / 64;
  const int64_t MT = (rows + 127) / 128;
  const int64_t total = MT * KT * 2 * 128;  // (tile, half, row)
  int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= total) return;
  const int r = (int)(t & 127);
  const int h = (int)((t >> 7) & 1);
  const int64_t tile = t >> 8;
  const int64_t m = tile / KT, kt = tile % KT;
  const int64_t row = m * 128 + r;
  if (row >= rows) return;
  const uint4 v = codes[tile * 256 + h * 128 + r];
  const uint32_t words[4] = {v.x, v.y, v.z, v.w};
  const int u = DU == 2 ? h : 0;
  const float sc = __half2float(__ushort_as_half(scales[(tile * DU + u) * 128 + r]));
  for (int j = 0; j < 4; ++j) {
    uint32_t a[4];
    dequant8(words[j], a);
    for (int p = 0; p < 4; ++p) {
      const int64_t col = kt * 64 + 32 * h + 8 * j + 2 * p;
      const float q0 = __half2float(__ushort_as_half((uint16_t)(a[p] & 0xFFFF)));
      const float q1 = __half2float(__ushort_as_half((uint16_t)(a[p] >> 16)));
      out[row * cols + col] = __fmul_rn(q0, sc);
      out[row * cols + col + 1] = __fmul_rn(q1, sc);
    }
  }
}

// ---------------------------------------------------------------- launchers

static unsigned blocks_for(int64_t n, int b) { return (unsigned)((n + b - 1) / b); }

cudaError_t tc_pack_int4(const uint8_t *codes, const uint16_t *scales, int64_t rows, int64_t cols, int group,
                         void *dst, void *dst_scales, cudaStream_t st) {
  const int64_t MT = (rows + 127) / 128, KT = cols / 64;
  k_tc_pack_int4<<<blocks_for(MT * KT * 1024, 256), 256, 0, st>>>(codes, rows, cols, (uint32_t *)dst);
  k_tc_pack_scales<<<blocks_for(MT * KT * drain_units(group) * 128, 256), 256, 0, st>>>(scales, rows, cols, group,
                                                                                       (uint16_t *)dst_scales);
  count_launch(2);
  return cudaGetLastError();
}

cudaError_t tc_dequant_int4(const void *codes, const void *scales, int64_t rows, int64_t cols, int group, float *out,
                            cudaStream_t st) {
  const int64_t MT = (rows + 127) / 128, KT = cols / 64;
  k_tc_dequant<<<blocks_for(MT * KT * 256, 256), 256, 0, st>>>((const uint4 *)codes, (const uint16_t *)scales, rows,
                                                              cols, drain_units(group), out);
  count_launch(1);
  return cudaGetLastError();
}

cudaError_t tc_pack_f16(const uint16_t *src, int64_t rows, int64_t cols, void *dst, cudaStream_t st) {
  const int64_t MT = (rows + 127) / 128, KT = cols / 64;
  k_tc_pack_f16<<<blocks_for(MT * KT * 1024, 256), 256, 0, st>>>(src, rows, cols, (uint4 *)dst);
  count_launch(1);
  return cudaGetLastError();
}

// Up to 32 tokens: the kernels of this file; more: the wide GEMMs (tc_wide.cu).
constexpr int NARROW_MAX_T = 32;
static int tt_int4(int T) { return T <= 16 ? 16 : 32; }
static int tt_f16(int T) { return T <= 16 ? 16 : 32; }

size_t tc_act_bytes(int T, int K, bool int4) {
  if (T > NARROW_MAX_T) return wide_act_bytes(T, K, int4);
  const int TT = int4 ? tt_int4(T) : tt_f16(T);
  return (size_t)((T + TT - 1) / TT) * TT * K * 2 * (int4 ? 2 : 1);
}

// Pack X into token tiles of TT rows and, for a split-K launch, clear its outputs.
static cudaError_t launch_pack(const float *X, int ldx, int T, int K, int TT, int planes, void *act,
                               const TcJob *jobs, int njobs, bool clear, cudaStream_t st) {
  const int64_t chunks = (int64_t)((T + TT - 1) / TT) * (K / 64) * TT * 8;
  const int pack_blocks = (int)blocks_for(chunks, 256);
  ZeroJobs Z{};
  int zero_blocks = 0;
  if (clear) {
    Z.njobs = njobs;
    int64_t most = 0;
    for (int j = 0; j < njobs; ++j) {
      Z.y[j] = jobs[j].y;
      Z.ldy[j] = jobs[j].ldy;
      Z.n[j] = jobs[j].n;
      most = std::max<int64_t>(most, (int64_t)T * jobs[j].n);
    }
    zero_blocks = (int)std::min<int64_t>(blocks_for(most, 2048), 256);
  }
  if (planes == 2)
    return launch_pdl(k_tc_pack_act<2>, dim3(pack_blocks + zero_blocks), dim3(256), 0, st, 1, X, ldx, T, K, TT,
                      (uint4 *)act, Z, pack_blocks);
  return launch_pdl(k_tc_pack_act<1>, dim3(pack_blocks + zero_blocks), dim3(256), 0, st, 1, X, ldx, T, K, TT,
                    (uint4 *)act, Z, pack_blocks);
}

// The wide path for up to 4 matrices given as TcJobs.
static cudaError_t wide_jobs(const TcJob *jobs, int njobs, bool int4, int group, const float *X, int ldx, int T,
                             int K, void *act, int num_sms, cudaStream_t st) {
  if (njobs < 1 || njobs > MAX_JOBS) return cudaErrorInvalidValue;
  WideJob w[MAX_JOBS];
  for (int j = 0; j < njobs; ++j) w[j] = WideJob{jobs[j].w, jobs[j].scales, jobs[j].y, jobs[j].n, jobs[j].ldy, 0};
  return wide_gemm(w, njobs, 0, int4, group, X, ldx, T, K, act, num_sms, st);
}

// Grid over (token tiles, row tiles of all jobs, k splits): splits fill the
// GPU, but a CTA keeps at least `kc_min` k-tiles so that its set-up and its
// output atomics stay small beside its stream.
static void plan(int ntt, int mtiles, int KT, int num_sms, int kc_min, int &kc, int &splits) {
  const int64_t base = (int64_t)ntt * mtiles;
  const int64_t want = 2 * (int64_t)num_sms;
  splits = 1;
  if (base < want) splits = (int)std::min<int64_t>(KT, (want + base - 1) / base);
  kc = (KT + splits - 1) / splits;
  kc = std::max(kc, std::min(kc_min, KT));
  splits = (KT + kc - 1) / kc;
}

static cudaError_t fill_jobs(const TcJob *jobs, int njobs, TcJobs &J, int &mtiles) {
  if (njobs < 1 || njobs > MAX_JOBS) return cudaErrorInvalidValue;
  J = TcJobs{};
  J.njobs = njobs;
  mtiles = 0;
  for (int j = 0; j < njobs; ++j) {
    J.w[j] = jobs[j].w;
    J.s[j] = (const uint16_t *)jobs[j].scales;
    J.y[j] = jobs[j].y;
    J.n[j] = jobs[j].n;
    J.ldy[j] = jobs[j].ldy;
    J.tile0[j] = mtiles;
    mtiles += (jobs[j].n + 127) / 128;
  }
  J.tile0[njobs] = mtiles;
  return cudaSuccess;
}

// ---- four-bit: the partition of a launch
template <int MT, int CPS>
static void plan_int4(const TcJobs &J, int njobs, int ntt, int K, int num_sms, I4Items &P, int &grid, bool &split) {
  P = I4Items{};
  P.groups = 0;
  for (int j = 0; j < njobs; ++j) {
    P.gtile0[j] = P.groups;
    P.groups += (J.tile0[j + 1] - J.tile0[j] + MT - 1) / MT;
  }
  P.gtile0[njobs] = P.groups;
  P.ntt = ntt;
  const int KT = K / 64;
  P.units = (int)std::min<int64_t>((int64_t)ntt * P.groups * KT, INT32_MAX - 1);
  // two CTAs an SM, each at least 2 units long (a small GEMM is latency-bound: more CTAs, shorter
  // chains); whole groups a CTA when there are enough of them
  const int ngroups = ntt * P.groups;
  split = false;
  if (ngroups >= CPS * num_sms) {
    P.whole = 1;
    grid = CPS * num_sms;
  } else {
    P.whole = 0;
    grid = (int)std::max<int64_t>(1, std::min<int64_t>(CPS * num_sms, P.units / 2));
    for (int b = 1; b < grid && !split; ++b) split = ((int64_t)b * P.units / grid) % KT != 0;
  }
}

// The jobs' tensor maps, encoded once per (matrix, box shape) and kept: the
// weights of a drafter stay where they are between calls.
static bool i4_maps(const TcJobs &J, int njobs, int KT, int KS, int MT, int DU, I4Maps &M) {
  using Key = std::tuple<const void *, const void *, int, int, int, int, int>;
  static std::mutex mu;
  static std::map<Key, std::pair<CUtensorMap, CUtensorMap>> cache;
  std::lock_guard<std::mutex> lock(mu);
  M.ksb = std::min(KS, KT);
  for (int j = 0; j < njobs; ++j) {
    const int mt = J.tile0[j + 1] - J.tile0[j];
    const int mtb = std::min(MT, mt);
    M.wbox[j] = mtb * M.ksb * (4096 + DU * 256);
    const Key key{J.w[j], J.s[j], mt, KT, M.ksb, mtb, DU};
    auto it = cache.find(key);
    if (it == cache.end()) {
      if (cache.size() > 4096) cache.clear();
      std::pair<CUtensorMap, CUtensorMap> maps;
      const uint64_t cd[4] = {256, 16, (uint64_t)KT, (uint64_t)mt};
      const uint64_t cs[3] = {256, 4096, (uint64_t)KT * 4096};
      const uint32_t cb[4] = {256, 16, (uint32_t)M.ksb, (uint32_t)mtb};
      const uint64_t sd[4] = {256, (uint64_t)DU, (uint64_t)KT, (uint64_t)mt};
      const uint64_t ss[3] = {256, (uint64_t)DU * 256, (uint64_t)KT * DU * 256};
      const uint32_t sb[4] = {256, (uint32_t)DU, (uint32_t)M.ksb, (uint32_t)mtb};
      if (!byte_map(&maps.first, J.w[j], 4, cd, cs, cb) || !byte_map(&maps.second, J.s[j], 4, sd, ss, sb))
        return false;
      it = cache.emplace(key, maps).first;
    }
    M.code[j] = it->second.first;
    M.scale[j] = it->second.second;
  }
  return true;
}

template <int TT, int DU, int MT>
static cudaError_t launch_int4(const TcJobs &J, int njobs, const void *act, int K, int T, int ntt, int num_sms,
                               cudaStream_t st, unsigned long long *cmax, int nchunks) {
  using C = I4<TT, DU, MT, I4_KS, I4_CPS, I4_NDQ, I4_P, I4_FOLD>;
  static PerDevice configured;
  cudaError_t e = smem_limit(k_tc_int4<TT, DU, MT, I4_KS, I4_CPS, I4_NDQ, I4_P, I4_FOLD>, C::SMEM, configured);
  if (e != cudaSuccess) return e;
  I4Maps M{};
  if (!i4_maps(J, njobs, K / 64, I4_KS, MT, DU, M)) return cudaErrorInvalidValue;
  I4Items P;
  int grid;
  bool split;
  plan_int4<MT, I4_CPS>(J, njobs, ntt, K, num_sms, P, grid, split);
  if (cmax && (!P.whole || njobs != 1)) return cudaErrorInvalidValue;  // the caller asks tc_int4_whole first
  P.cmax = cmax;
  P.nchunks = nchunks;
  return launch_pdl(k_tc_int4<TT, DU, MT, I4_KS, I4_CPS, I4_NDQ, I4_P, I4_FOLD>, dim3(grid), dim3(C::THREADS), C::SMEM, st, 1, M, J, P,
                    (const uint8_t *)act, K, T);
}

// (token tile, quantisation units a k-tile, 128-row tiles an item, tensor-memory A slots)
static cudaError_t dispatch_int4(const TcJobs &J, int njobs, int group, const void *act, int K, int T, int num_sms,
                                 cudaStream_t st, unsigned long long *cmax = nullptr, int nchunks = 0) {
  const int TT = tt_int4(T);
  const int ntt = (T + TT - 1) / TT;
  const int DU = drain_units(group);
  if (TT == 16) return DU == 1 ? launch_int4<16, 1, 2>(J, njobs, act, K, T, ntt, num_sms, st, cmax, nchunks)
                               : launch_int4<16, 2, 2>(J, njobs, act, K, T, ntt, num_sms, st, cmax, nchunks);
  return DU == 1 ? launch_int4<32, 1, 1>(J, njobs, act, K, T, ntt, num_sms, st, cmax, nchunks)
                 : launch_int4<32, 2, 1>(J, njobs, act, K, T, ntt, num_sms, st, cmax, nchunks);
}

int tc_tile_rows(int T, bool int4) { return int4 ? tt_int4(T) : tt_f16(T); }

bool tc_splits_int4(const TcJob *jobs, int njobs, int T, int K, int num_sms) {
  TcJobs J;
  int mtiles;
  if (T > NARROW_MAX_T || fill_jobs(jobs, njobs, J, mtiles) != cudaSuccess) return false;
  const int TT = tt_int4(T), ntt = (T + TT - 1) / TT;
  I4Items P;
  int grid;
  bool split;
  if (TT == 16) plan_int4<2, I4_CPS>(J, njobs, ntt, K, num_sms, P, grid, split);
  else plan_int4<1, I4_CPS>(J, njobs, ntt, K, num_sms, P, grid, split);
  return split;
}

bool tc_int4_whole(const TcJob *jobs, int njobs, int T, int K, int num_sms) {
  TcJobs J;
  int mtiles;
  if (T > NARROW_MAX_T || fill_jobs(jobs, njobs, J, mtiles) != cudaSuccess) return false;
  const int TT = tt_int4(T), ntt = (T + TT - 1) / TT;
  I4Items P;
  int grid;
  bool split;
  if (TT == 16) plan_int4<2, I4_CPS>(J, njobs, ntt, K, num_sms, P, grid, split);
  else plan_int4<1, I4_CPS>(J, njobs, ntt, K, num_sms, P, grid, split);
  return P.whole != 0;
}

bool tc_splits_f16(const TcJob *jobs, int njobs, int T, int K, int num_sms) {
  TcJobs J;
  int mtiles;
  if (T > NARROW_MAX_T || fill_jobs(jobs, njobs, J, mtiles) != cudaSuccess) return false;
  const int TT = tt_f16(T), ntt = (T + TT - 1) / TT;
  int kc, splits;
  plan(ntt, mtiles, K / 64, num_sms, 2, kc, splits);
  return splits > 1;
}

cudaError_t tc_gemm_int4_packed(const TcJob *jobs, int njobs, int group, const void *act, int T, int K, int num_sms,
                                cudaStream_t st, unsigned long long *cmax, int nchunks) {
  if (T > NARROW_MAX_T) return cudaErrorInvalidValue;
  TcJobs J;
  int mtiles;
  cudaError_t e = fill_jobs(jobs, njobs, J, mtiles);
  if (e != cudaSuccess) return e;
  return dispatch_int4(J, njobs, group, act, K, T, num_sms, st, cmax, nchunks);
}

cudaError_t tc_gemm_int4(const TcJob *jobs, int njobs, int group, const float *X, int ldx, int T, int K, void *act,
                         int num_sms, cudaStream_t st) {
  if (T > NARROW_MAX_T) return wide_jobs(jobs, njobs, true, group, X, ldx, T, K, act, num_sms, st);
  TcJobs J;
  int mtiles;
  cudaError_t e = fill_jobs(jobs, njobs, J, mtiles);
  if (e != cudaSuccess) return e;
  e = launch_pack(X, ldx, T, K, tt_int4(T), 2, act, jobs, njobs, tc_splits_int4(jobs, njobs, T, K, num_sms), st);
  if (e != cudaSuccess) return e;
  return dispatch_int4(J, njobs, group, act, K, T, num_sms, st);
}

// ---- f16
template <int TT>
static cudaError_t launch_f16(const TcJobs &J, int mtiles, const void *act, int bstride, int K, int T, int ntt,
                              int num_sms, cudaStream_t st) {
  using C = F16Cfg<TT>;
  static PerDevice configured;
  cudaError_t e = smem_limit(k_tc_f16<TT>, C::SMEM, configured);
  if (e != cudaSuccess) return e;
  int kc, splits;
  plan(ntt, mtiles, K / 64, num_sms, 2, kc, splits);
  dim3 grid(ntt, mtiles, splits);
  return launch_pdl(k_tc_f16<TT>, grid, dim3(TC_THREADS), C::SMEM, st, 1, J, (const uint8_t *)act, bstride, K, T, kc,
                    (int)(splits > 1));
}

cudaError_t tc_gemm_f16_packed(const TcJob *jobs, int njobs, const void *act, int bstride, int T, int K, int num_sms,
                               cudaStream_t st) {
  if (T > NARROW_MAX_T) return cudaErrorInvalidValue;
  TcJobs J;
  int mtiles;
  cudaError_t e = fill_jobs(jobs, njobs, J, mtiles);
  if (e != cudaSuccess) return e;
  const int TT = tt_f16(T), ntt = (T + TT - 1) / TT;
  return TT == 16 ? launch_f16<16>(J, mtiles, act, bstride, K, T, ntt, num_sms, st)
                  : launch_f16<32>(J, mtiles, act, bstride, K, T, ntt, num_sms, st);
}

cudaError_t tc_gemm_f16(const TcJob *jobs, int njobs, const float *X, int ldx, int T, int K, void *act, int num_sms,
                        cudaStream_t st) {
  if (T > NARROW_MAX_T) return wide_jobs(jobs, njobs, false, 0, X, ldx, T, K, act, num_sms, st);
  const int TT = tt_f16(T);
  cudaError_t e = launch_pack(X, ldx, T, K, TT, 1, act, jobs, njobs, tc_splits_f16(jobs, njobs, T, K, num_sms), st);
  if (e != cudaSuccess) return e;
  return tc_gemm_f16_packed(jobs, njobs, act, TT * 128, T, K, num_sms, st);
}

// Each translation unit that waits on mbarriers has its own copy of the word
// (tc.cuh); the library's is their union.
static cudaError_t gemm_read_error(unsigned *out, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_dev_error, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  if (reset) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_dev_error, &zero, sizeof(unsigned));
  }
  return e;
}

cudaError_t read_device_error(unsigned *out, bool reset) {
  unsigned a = 0, b = 0, c = 0, r = 0;
  cudaError_t e = gemm_read_error(&a, reset);
  if (e == cudaSuccess) e = wide_read_error(&b, reset);
  if (e == cudaSuccess) e = attn_read_error(&c, reset);
  if (e == cudaSuccess) e = rows_read_error(&r, reset);
  *out = a | b | c | r;
  return e;
}

}  // namespace dfl

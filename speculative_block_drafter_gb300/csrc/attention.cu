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

bool byte_map(CUtensorMap *m, const void *base, int rank, const uint64_t *dims, const uint64_t *strides,
              const uint32_t *box) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i > 0) st[i - 1] = strides[i - 1];
  }
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, (void *)base, d, st, bx, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


// ---------------------------------------------------------------- the split kernel
//
// One CTA per (split, KV head, sequence): the Q = rep * R queries of the KV
// head over the split's context keys in chunks of 64 (the last split takes the
// block's own R rows as a final chunk of 16), on the 5th-generation tensor
// cores with everything the products need in tensor memory (512 columns, one
// CTA an SM; lanes = query rows, the Q real ones first, the rest zero):
//   QH, QL   the queries as f16 hi/lo planes (the A operand of S = Q K^T)
//   SA, SB   the scores' two partial sums (64 columns each): the products
//            over the first and over the second half of the head dimension
//   P0, P1   two probability buffers, hi and lo planes (A of O += P V)
//   O        the output accumulator (HD columns)
// The context caches and the block's own K/V hold f16 values in PL planes per
// row and head (PL = 2: hi, lo; PL = 1: one f16), written once when the rows
// were settled or projected.
//   warp 8    tensor copies of each chunk's K and V planes (boxes of 64 rows x
//             64 halves, 128-byte swizzled) into a ring of stages
//   warps 9, 11  the score MMAs, one thread each, one half of the head
//             dimension each into its partial sum: S = Qh Kh + Qh Kl + Ql Kh
//             (PL = 2) or Qh K + Ql K (PL = 1), K read K-major from the stage.
//             A chunk's partials are taken once the softmax has read the
//             previous chunk's
//   warp 10   the output MMAs, one thread: once the chunk's P is written,
//             O += Ph Vh + Ph Vl + Pl Vh (or Ph V + Pl V), V read MN-major from
//             the same stage. An MMA holds its issuing thread for about 150
//             cycles whatever its N, so the MMAs are spread over three
//             threads; the softmax of one chunk runs while the next chunk's
//             scores are taken. A stage is released by the three threads'
//             commits.
//   warps 0-7 two threads a query row, each with half of a chunk's keys (warp w
//             takes the rows of tensor-memory lanes 32 (w % 4).. and key half
//             w / 4): the scores from tensor memory (the two partials added),
//             the window mask, the row's
//             largest score exchanged with the partner through shared memory,
//             an online softmax, P as hi/lo planes into tensor memory; at the
//             end the row's (o, m, l) to the partials. Warps whose rows are all
//             past the Q queries skip the arithmetic.
// Online softmax in the base-2 domain with a lazy reference: P = 2^(x - m) with
// m the largest score seen when it last moved by more than TAU, so that P <=
// 2^TAU stays in f16's range and O (in tensor memory) is rescaled only when m
// moves that far; O and l always share m, so the result is exact. Keys past a
// chunk's end are masked and their V rows zeroed in the stage before the P.V
// products read them. The softmax warps meet at a named barrier with an AND
// of their wait results, so that a wait that gave up ends all of them together.
template <int HD, int PL>
struct AttnTc {
  static constexpr int QH = 0, QL = HD / 2;          // HD/2 columns a plane (f16 pairs)
  static constexpr int S0 = HD;                      // + 64 * partial
  static constexpr int P0 = HD + 128;                // + 64 * buffer: hi 32 columns, lo 32 columns
  static constexpr int OC = HD + 256;                // HD columns
  static_assert(OC + HD <= 512, "tensor memory");
  static constexpr int BOX = CH * 128;               // 64 rows x 64 halves
  static constexpr int REGION = (HD / 64) * BOX;     // one plane of K or V of a chunk
  static constexpr int STAGE = 2 * PL * REGION;      // K planes, then V planes
  static constexpr int STAGES = (192 * 1024) / STAGE < 6 ? (192 * 1024) / STAGE : 6;
  // kvfull, kvempty (a stage each), qfull, sfull, sfree (+1 unused each), pfull[2], pfree[2], obar, fin
  static constexpr int NBAR = 2 * STAGES + 11;
  // + alignment, barriers, the tensor-memory address; and 20 KB past them that no
  // operand descriptor of the last stage can reach beyond
  static constexpr size_t BYTES = (size_t)STAGES * STAGE + 1024 + 8 * NBAR + 16 + 20 * 1024;
};
constexpr int ATT_TC_THREADS = 384;
constexpr int ATT_SM_THREADS = 256;  // the softmax warps 0-7
constexpr float ATT_TAU = 11.f;      // P <= 2^11 between rescales

// bar.red.and over the softmax warps (named barrier 1): every thread waits for
// all ATT_SM_THREADS and gets the AND of their `p`.
__device__ __forceinline__ bool sm_and(bool p) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred a, b;\n setp.ne.u32 a, %1, 0;\n bar.red.and.pred b, 1, %2, a;\n selp.u32 %0, 1, 0, b;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)p), "n"(ATT_SM_THREADS)
      : "memory");
  return r != 0;
}

// 2^x, the hardware's approximation (relative error about 2^-22; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

template <int HD, int PL>
__global__ void __launch_bounds__(ATT_TC_THREADS, 1)
    k_attn_tc(const float *__restrict__ q, const __grid_constant__ AttnArgs args, int heads, int kv, int R, int window,
              float scale, int nsplit, int cps, float *__restrict__ part) {
  using C = AttnTc<HD, PL>;
  constexpr int S = C::STAGES;
  constexpr int H2 = HD / 64;
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t *sm = smraw + ((1024 - (smem_u32(smraw) & 1023)) & 1023);
  const uint32_t ring = smem_u32(sm);
  uint64_t *bars = (uint64_t *)(sm + S * C::STAGE);
  uint32_t *tslot = (uint32_t *)(bars + C::NBAR);
  const uint32_t kvfull = smem_u32(bars), kvempty = kvfull + 8 * S, qfull = kvempty + 8 * S;
  const uint32_t sfull = qfull + 8, sfree = sfull + 16, pfull = sfree + 16, pfree = pfull + 16, obar = pfree + 16;
  const uint32_t fin = obar + 8;

  const int sp = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int rep = heads / kv, Q = rep * R;
  const AttnSeq &Sq = args.seq[b];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this CTA's chunks: context chunks [c0, c1), then the block's own rows if last
  const int n = Sq.n;
  const int nctx = (n + CH - 1) / CH;
  const int c0 = min(nctx, sp * cps), c1 = min(nctx, c0 + cps);
  const bool own = sp == nsplit - 1;
  const int nch = (c1 - c0) + (own ? 1 : 0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(kvfull + 8 * i, 1);
      mbar_init(kvempty + 8 * i, 3);  // released by the two halves' Q K and the P V products
    }
    mbar_init(qfull, 128);
    mbar_init(sfull, 2);               // both partials of a chunk's scores
    mbar_init(sfree, ATT_SM_THREADS);  // read by the softmax
    for (int i = 0; i < 2; ++i) {
      mbar_init(pfull + 8 * i, ATT_SM_THREADS);
      mbar_init(pfree + 8 * i, 1);
    }
    mbar_init(obar, 1);
    mbar_init(fin, 3);  // the three issuing threads' last commits
    mbar_fence_init();
  }
  pdl_wait();
  if (warp == 0) tmem_alloc(smem_u32(tslot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = *tslot;

  if (warp == 8) {
    // the K and V planes of chunk j into stage j % S
    if (lane == 0) {
      int issued = 0;
      for (int j = 0; j < nch; ++j, ++issued) {
        const int st = j % S;
        if (j >= S && !mbar_wait(kvempty + 8 * st, ((j / S) - 1) & 1)) break;
        const bool is_own = own && j == nch - 1;
        const CUtensorMap *km = is_own ? &args.own_k : &Sq.kmap;
        const CUtensorMap *vm = is_own ? &args.own_v : &Sq.vmap;
        const int z = is_own ? b * R : (int)(Sq.row0 + (int64_t)(c0 + j) * CH);
        const uint32_t rows = is_own ? R : CH;
        const uint32_t bar = kvfull + 8 * st, base = ring + st * C::STAGE;
        mbar_expect_tx(bar, 2 * PL * H2 * rows * 128);
#pragma unroll
        for (int h = 0; h < H2; ++h)
#pragma unroll
          for (int p = 0; p < PL; ++p) {
            tma_load4(base + p * C::REGION + h * C::BOX, km, 64 * h, p, g, z, bar);
            tma_load4(base + (PL + p) * C::REGION + h * C::BOX, vm, 64 * h, p, g, z, bar);
          }
      }
      // no copy still bound for this CTA's shared memory when it leaves (the
      // copies of the last stages issued; a bounded wait each)
      for (int j = (issued > S ? issued - S : 0); j < issued; ++j) mbar_wait(kvfull + 8 * (j % S), (j / S) & 1);
    }
  } else if (warp == 9 || warp == 11) {
    // the partial S_h = Q K^T over half h of the head dimension into its 64
    // columns. An MMA holds its issuing thread for about 150 cycles whatever
    // its N, so the scores have two warps and the P V products a third.
    if (lane == 0 && nch > 0) {
      const int h = warp == 9 ? 0 : 1;
      constexpr int KS = HD / 32;  // k-steps of a half
      bool ok = mbar_wait(qfull, 0);
      tc_fence_after();
      const uint32_t dS = tb + C::S0 + h * 64;
      for (int j = 0; j < nch && ok; ++j) {
        const int st = j % S;
        if (!mbar_wait_spin(kvfull + 8 * st, (j / S) & 1)) break;
        // the softmax has read the previous chunk's partials
        if (j >= 1 && !mbar_wait_spin(sfree, (j - 1) & 1)) break;
        tc_fence_after();
        const bool is_own = own && j == nch - 1;
        const uint32_t idesc = f16_idesc(128, is_own ? 16 : CH);
        const uint32_t kh = ring + st * C::STAGE, kl = kh + C::REGION;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const int ks = h * KS + kk;
          const uint32_t off = (ks >> 2) * C::BOX + (ks & 3) * 32;
          mma_ts(dS, tb + C::QH + ks * 8, sw128_desc(kh + off), idesc, kk > 0);
          if (PL == 2) mma_ts(dS, tb + C::QH + ks * 8, sw128_desc(kl + off), idesc, 1);
          mma_ts(dS, tb + C::QL + ks * 8, sw128_desc(kh + off), idesc, 1);
        }
        mma_commit(sfull);
        mma_commit(kvempty + 8 * st);  // K read (the stage's other releases: the other half, P V)
      }
      // every MMA of this thread completed before the tensor memory is freed
      mma_commit(fin);
      mbar_wait(fin, 0);
    }
  } else if (warp == 10) {
    // O += P V of each chunk, once its P is written
    if (lane == 0 && nch > 0) {
      for (int jj = 0; jj < nch; ++jj) {
        const int st = jj % S, pb = jj & 1;
        if (!mbar_wait_spin(kvfull + 8 * st, (jj / S) & 1)) break;
        if (!mbar_wait_spin(pfull + 8 * pb, (jj >> 1) & 1)) break;
        tc_fence_after();
        const bool is_own = own && jj == nch - 1;
        const int ksteps = is_own ? 1 : CH / 16;
        const uint32_t idesc = f16_idesc_bmn(128, HD);
        const uint32_t vh = ring + st * C::STAGE + PL * C::REGION, vl = vh + C::REGION;
        const uint32_t ph = tb + C::P0 + pb * 64, pl = ph + 32;
        for (int kk = 0; kk < ksteps; ++kk) {
          const uint64_t bh = sw128_mn_desc(vh + kk * 2048, C::BOX), bl = sw128_mn_desc(vl + kk * 2048, C::BOX);
          mma_ts(tb + C::OC, ph + kk * 8, bh, idesc, (jj > 0 || kk > 0));
          if (PL == 2) mma_ts(tb + C::OC, ph + kk * 8, bl, idesc, 1);
          mma_ts(tb + C::OC, pl + kk * 8, bh, idesc, 1);
        }
        mma_commit(obar);
        mma_commit(pfree + 8 * pb);
        mma_commit(kvempty + 8 * st);
      }
      mma_commit(fin);
      mbar_wait(fin, 0);
    }
  } else {
    // warps 0-7: query row `row` (tensor-memory lane), key half `kh` of each chunk
    // the rows' largest scores per key half, by chunk parity (a slot is written
    // again two chunks later, after both halves passed the barrier between); the sums
    __shared__ float xch[2][2][128], lsum[2][128];
    const int row = threadIdx.x & 127, kh = warp >> 2;
    const uint32_t lrow = (uint32_t)((warp & 3) * 32) << 16;
    const bool live = row < Q;
    const bool dead = (warp & 3) * 32 >= Q;  // every row of this warp past the queries
    const int rr = row % R;
    const float sl2 = scale * 1.4426950408889634f;  // scores to the base-2 domain
    if (kh == 0) {
      // the row's query (normalised, rotated) as hi/lo planes into tensor memory
      const float *qr = live ? q + ((int64_t)b * R + rr) * heads * HD + (g * rep + row / R) * HD : nullptr;
#pragma unroll
      for (int half = 0; half < H2; ++half) {
        uint32_t vh[32], vl[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float2 x = make_float2(0.f, 0.f);
          if (live) x = *(const float2 *)(qr + half * 64 + 2 * e);
          split_hl(x.x, x.y, vh[e], vl[e]);
        }
        tmem_st32(tb + lrow + C::QH + half * 32, vh);
        tmem_st32(tb + lrow + C::QL + half * 32, vl);
      }
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(qfull);
    }
    float mref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nch; ++j) {
      const int sb = j & 1, st = j % S;
      const bool is_own = own && j == nch - 1;
      const int kb = (c0 + j) * CH;
      const int cnt = is_own ? R : min(CH, n - kb);
      const int N = is_own ? 16 : CH;
      const int k0 = kh * 32;  // this thread's keys k0 .. k0 + 31 of the chunk
      bool w_ok = __all_sync(0xffffffffu, mbar_wait_spin(sfull, j & 1));
      tc_fence_after();
      // raw scores of the visible keys [kmin, kmax) of the chunk, -inf elsewhere
      float x[32];
      float mh = -INFINITY;
      if (!dead && w_ok) {
        // the two partial sums of the scores
        uint32_t r0[32];
        tmem_ld32(tb + lrow + C::S0 + k0, r0);
        tc_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(r0[e]);
        tmem_ld32(tb + lrow + C::S0 + 64 + k0, r0);
        tc_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) r0[e] = __float_as_uint(x[e] + __uint_as_float(r0[e]));
        const int kmax = live ? cnt : 0;
        int kmin = 0;
        if (!is_own && window > 0) {
          const int64_t first_vis = Sq.anchor + rr + 1 - window - (Sq.lo + kb);  // as a key of this chunk
          kmin = first_vis <= 0 ? 0 : (first_vis >= CH ? CH : (int)first_vis);
        }
        if (kmin <= k0 && kmax >= k0 + 32) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            x[e] = __uint_as_float(r0[e]);
            mh = fmaxf(mh, x[e]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int k = k0 + e;
            x[e] = (k >= kmin && k < kmax) ? __uint_as_float(r0[e]) : -INFINITY;
            mh = fmaxf(mh, x[e]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(sfree);
      // keys past the chunk's end: their V rows zeroed before the P.V products read them
      if (cnt < N && w_ok) {
        const int nz = N - cnt;
        uint8_t *vst = sm + st * C::STAGE + PL * C::REGION;
        for (int idx = threadIdx.x; idx < nz * PL * H2 * 8; idx += ATT_SM_THREADS) {
          const int r = cnt + idx / (PL * H2 * 8), rest = idx % (PL * H2 * 8);
          const int pl = rest / (H2 * 8), bx = (rest / 8) % H2, ch = rest % 8;
          *(uint4 *)(vst + pl * C::REGION + bx * C::BOX + r * 128 + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
      xch[sb][kh][row] = mh;
      ok = sm_and(ok && w_ok);
      if (!ok) break;
      const float mx = fmaxf(xch[sb][0][row], xch[sb][1][row]) * sl2;  // the base-2 domain
      // the reference moves (both halves of a row decide alike); O's half `kh` of
      // the columns is rescaled once the products of the chunks before are done
      const bool up = mx > mref + ATT_TAU;
      if (__any_sync(0xffffffffu, up)) {
        float alpha = 1.f;
        if (up) {
          alpha = mref == -INFINITY ? 0.f : ex2(mref - mx);
          l *= alpha;
          mref = mx;
        }
        if (j > 0 && !dead) {
          // O holds the products of chunks 0 .. j-1 once obar completed its phase
          // j-1. The P V products have their own issuing thread, so first make
          // sure that chunk j-2's completed (it frees P buffer j & 1): obar is
          // then at most one phase behind and the parity wait cannot pass early
          if (j >= 2) ok = __all_sync(0xffffffffu, mbar_wait(pfree + 8 * sb, ((j >> 1) - 1) & 1));
          ok = ok && __all_sync(0xffffffffu, mbar_wait(obar, (j - 1) & 1));
          tc_fence_after();
          if (ok) {
#pragma unroll
            for (int c = 0; c < HD / 64; ++c) {
              uint32_t o[32];
              const uint32_t col = tb + lrow + C::OC + kh * (HD / 2) + c * 32;
              tmem_ld32(col, o);
              tc_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tmem_st32(col, o);
            }
            tc_wait_st();
          }
        }
      }
      // P = 2^(x - m) of this thread's keys, as hi/lo planes (16 columns each)
      uint32_t ph[16], pw[16];
      if (!dead) {
        // 2^(x sl2 - m): a masked key's -inf gives 0 (and no row has a visible
        // key while m is still -inf)
        const float negm = mref == -INFINITY ? 0.f : -mref;
        float sum = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = ex2(fmaf(x[2 * e], sl2, negm));
          const float p1 = ex2(fmaf(x[2 * e + 1], sl2, negm));
          sum += p0 + p1;
          split_hl(p0, p1, ph[e], pw[e]);
        }
        l += sum;
      }
      if (j >= 2) {
        ok = ok && __all_sync(0xffffffffu, mbar_wait(pfree + 8 * sb, ((j >> 1) - 1) & 1));
        tc_fence_after();
      }
      if (!dead && ok) {
        tmem_st16(tb + lrow + C::P0 + sb * 64 + kh * 16, ph);
        tmem_st16(tb + lrow + C::P0 + sb * 64 + 32 + kh * 16, pw);
        tc_wait_st();
      }
      tc_fence_before();
      mbar_arrive(pfull + 8 * sb);
    }
    // the row's partial: o (unnormalised, against m), m (natural base), l; key
    // half kh writes o's columns kh * HD/2 ..
    lsum[kh][row] = l;
    const bool all_ok = sm_and(ok);
    l = lsum[0][row] + lsum[1][row];
    float *out = part + ((int64_t)(b * kv + g) * nsplit + sp) * Q * part_row(HD) + (int64_t)row * part_row(HD);
    // O is final once every MMA has completed (`fin`, committed after the last
    // P V): obar may still be two phases behind here, where a wait on the
    // parity of its last phase would pass at once
    const bool have = all_ok && nch > 0 && !dead && __all_sync(0xffffffffu, mbar_wait(fin, 0));
    if (have) {
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < HD / 64; ++c) {
        uint32_t o[32];
        tmem_ld32(tb + lrow + C::OC + kh * (HD / 2) + c * 32, o);
        tc_wait_ld();
        if (live)
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *(float4 *)(out + kh * (HD / 2) + c * 32 + e) = make_float4(
                __uint_as_float(o[e]), __uint_as_float(o[e + 1]), __uint_as_float(o[e + 2]), __uint_as_float(o[e + 3]));
      }
    } else if (live) {
      for (int c = 0; c < HD / 2; ++c) out[kh * (HD / 2) + c] = 0.f;
      mref = -INFINITY;
      l = 0.f;
    }
    if (live && kh == 0) {
      out[HD] = mref == -INFINITY ? -INFINITY : mref * 0.6931471805599453f;
      out[HD + 1] = l;
    }
  }
  pdl_trigger();  // this CTA's work is done
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
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

template <int HD, int PL>
static cudaError_t launch_attn(const float *q, const AttnArgs &args, int batch, int max_n, int heads, int kv, int R,
                               int window, float scale, float *part, float *y, int num_sms, const PackDst *pack,
                               const ZeroSet *zero, cudaStream_t st) {
  const size_t smem = AttnTc<HD, PL>::BYTES;
  static PerDevice configured;
  if (cudaError_t e = smem_limit(k_attn_tc<HD, PL>, (int)smem, configured)) return e;
  int ns, cps;
  plan_splits(batch * kv, max_n, num_sms, ns, cps);
  // With short splits the block's own rows get a split of their own (the last
  // one, past every context chunk), so that no CTA does twice the others' work.
  if (cps <= 4 && max_n > 0) ++ns;
  dim3 grid(ns, kv, batch);
  cudaError_t e = launch_pdl(k_attn_tc<HD, PL>, grid, dim3(ATT_TC_THREADS), smem, st, 1, q, args, heads, kv, R,
                             window, scale, ns, cps, part);
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
  return launch_attn<HD, PL>(q, args, batch, max_n, heads, kv, R, window, scale, part, y, num_sms, pack, zero, st);
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

// Non-causal grouped-query attention of a block's rows over the layer's
// windowed context and the block's own rows (cortiq-engine
// src/cortiq_engine/dflash.rs, `Drafter::block`: the scores of every (head,
// row) over the context and the block's rows, a row further on seeing less
// far back when the layer has a window, a max-subtracted softmax).
//
// Split-K: the context rows of a sequence are cut into chunks, one CTA per
// (chunk, KV head, sequence), plus one CTA per (KV head, sequence) for the
// block's own rows. Each keeps a running maximum m, sum l and unnormalised
// output o per query (the rep = heads/kv_heads query heads of the KV head times
// the block rows) and a second kernel merges the chunks.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace dfl {

constexpr int ATT_THREADS = 256;
constexpr int CH = 64;              // keys per chunk
constexpr int QMAX = 64;            // queries per CTA (rep * block)
// Split-K aims at one wave: a CTA (about 170 KB of shared memory) per SM.

struct AttnArgs {
  AttnSeq seq[MAX_BATCH];
};

// Chunks a split takes: one wave of the context's CTAs over the SMs that the
// block's own CTAs (one per sequence and KV head) leave free.
static int chunks_per_split(int batch, int kv, int max_n, int num_sms) {
  const int chunks = (max_n + CH - 1) / CH;
  const int units = batch * kv * chunks;
  const int ctas = std::max(num_sms - batch * kv, batch * kv);
  return std::max(1, (units + ctas - 1) / ctas);
}

size_t attn_partial_bytes(int max_batch, int kv_heads, int heads, int block, int hd) {
  const int Q = heads / kv_heads * block;
  // per (sequence, KV head): at most ceil(units / ctas) + 1 context splits (ctas >= batch * kv), plus
  // the block's own; bounded for any SM count up to 1024
  const size_t worst = (size_t)1024 + 3 * (size_t)max_batch * kv_heads;
  return worst * Q * (hd + 2) * sizeof(float);
}

// ---- fragments (mma.sync m16n8k16, f16 in, f32 accumulate)
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
__device__ __forceinline__ uint32_t cvta_smem(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0));
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Three-term product of f16 hi/lo pairs: acc += ah.bh + ah.bl + al.bh (about 22 bits).
__device__ __forceinline__ void mma3(float (&acc)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4], uint32_t bh0,
                                     uint32_t bh1, uint32_t bl0, uint32_t bl1) {
  mma16816(acc, ah, bh0, bh1);
  mma16816(acc, ah, bl0, bl1);
  mma16816(acc, al, bh0, bh1);
}

template <int HD>
struct AttnSmem {
  static constexpr int LD = HD + 8;                       // halves per row (16-byte pad: no ldmatrix conflicts)
  static constexpr int QPLANE = QMAX * LD;                // halves
  static constexpr int KPLANE = CH * LD;
  static constexpr int STAGE_F = 2 * CH * HD;             // f32 staging of K and V
  static constexpr int MERGE_F = 8 * 16 * (HD + 2);       // per-warp partials for the in-CTA merge
  static constexpr int SCRATCH_F = STAGE_F > MERGE_F ? STAGE_F : MERGE_F;
  static constexpr size_t BYTES = (size_t)(2 * QPLANE + 4 * KPLANE) * 2 + (size_t)SCRATCH_F * 4;
};

// One CTA per (split, KV head, sequence): the rep*R queries of the KV head over
// the split's keys, in chunks of 64. Warp w takes query block w % QW and key
// group w / QW (a quarter or half of each chunk); each keeps a running (m, l, o)
// that the CTA merges at the end.
template <int HD, int KG>
__global__ void __launch_bounds__(ATT_THREADS) k_attn(const float *__restrict__ q, const float *__restrict__ k,
                                                      const float *__restrict__ v, AttnArgs args, int heads, int kv,
                                                      int R, int window, float scale, int nsplit, int cps,
                                                      float *__restrict__ part) {
  pdl_wait();
  using SM = AttnSmem<HD>;
  constexpr int KW = CH / KG;      // keys per warp per chunk
  constexpr int NT = KW / 8;       // n8 tiles of scores
  constexpr int KS = KW / 16;      // k16 steps of P . V
  constexpr int OT = HD / 8;       // n8 tiles of the output
  extern __shared__ __align__(16) uint8_t smb[];
  __half *Qh = (__half *)smb, *Ql = Qh + SM::QPLANE;
  __half *Kh = Ql + SM::QPLANE, *Kl = Kh + SM::KPLANE, *Vh = Kl + SM::KPLANE, *Vl = Vh + SM::KPLANE;
  float *scr = (float *)(Vl + SM::KPLANE);

  const int sp = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int rep = heads / kv, Q = rep * R;
  const int QW = (Q + 15) / 16;
  const AttnSeq S = args.seq[b];
  const bool own = sp == nsplit;
  const int kbeg = own ? 0 : sp * cps * CH;
  const int kend = own ? R : min(S.n, kbeg + cps * CH);
  const float *kbase = own ? k + (int64_t)b * R * kv * HD : S.ck;
  const float *vbase = own ? v + (int64_t)b * R * kv * HD : S.cv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, cq = lane & 3;
  const int qb = warp % QW, kgi = warp / QW;
  const bool busy = kgi < KG && warp < QW * KG;

  // f32 rows of one chunk into the staging area
  auto stage = [&](int kb) {
    for (int i = tid; i < 2 * CH * (HD / 4); i += ATT_THREADS) {
      const int which = i / (CH * (HD / 4)), rem = i % (CH * (HD / 4));
      const int j = rem / (HD / 4), c4 = rem % (HD / 4);
      const int key = kb + j;
      const bool ok = key < kend;
      const float *src = (which ? vbase : kbase) + ((int64_t)(ok ? key : kbeg) * kv + g) * HD + c4 * 4;
      cp_async16(cvta_smem(scr + which * CH * HD + j * HD + c4 * 4), src, ok);
    }
    asm volatile("cp.async.commit_group;");
  };
  if (kbeg < kend) stage(kbeg);

  // the queries, hi/lo: every load of the thread first, then the conversions
  {
    constexpr int PER = QMAX * HD / 4 / ATT_THREADS;  // float4 a thread
    float4 xv[PER];
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const int i = tid + m * ATT_THREADS;
      const int qi = i / (HD / 4), d4 = i % (HD / 4);
      xv[m] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (qi < Q) {
        const int hrep = qi / R, r = qi - hrep * R;
        xv[m] = *(const float4 *)(q + ((int64_t)b * R + r) * heads * HD + (g * rep + hrep) * HD + 4 * d4);
      }
    }
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const int i = tid + m * ATT_THREADS;
      const int qi = i / (HD / 4), d4 = i % (HD / 4);
      uint32_t h0, l0, h1, l1;
      split2(xv[m].x, xv[m].y, h0, l0);
      split2(xv[m].z, xv[m].w, h1, l1);
      *(uint2 *)(Qh + qi * SM::LD + 4 * d4) = make_uint2(h0, h1);
      *(uint2 *)(Ql + qi * SM::LD + 4 * d4) = make_uint2(l0, l1);
    }
  }

  float o[OT][4];
#pragma unroll
  for (int t = 0; t < OT; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows gq and gq + 8 of the warp's block
  const int qi0 = qb * 16 + gq, qi1 = qi0 + 8;
  const int r0 = qi0 % R, r1 = qi1 % R;

  for (int kb = kbeg; kb < kend; kb += CH) {
    cp_async_wait_all();
    __syncthreads();
    // staging -> hi/lo planes
    for (int i = tid; i < 2 * CH * HD / 2; i += ATT_THREADS) {
      const int which = i / (CH * HD / 2), rem = i % (CH * HD / 2);
      const int j = rem / (HD / 2), d2 = rem % (HD / 2);
      const float2 x = *(const float2 *)(scr + which * CH * HD + j * HD + 2 * d2);
      uint32_t hi, lo;
      split2(x.x, x.y, hi, lo);
      __half *ph = which ? Vh : Kh, *pl = which ? Vl : Kl;
      *(uint32_t *)(ph + j * SM::LD + 2 * d2) = hi;
      *(uint32_t *)(pl + j * SM::LD + 2 * d2) = lo;
    }
    __syncthreads();
    if (kb + CH < kend) stage(kb + CH);

    if (busy) {
      // scores S = Q . K^T over the warp's keys
      float sc[NT][4];
#pragma unroll
      for (int t = 0; t < NT; ++t) sc[t][0] = sc[t][1] = sc[t][2] = sc[t][3] = 0.f;
      const int kk0 = kgi * KW;
#pragma unroll
      for (int ks = 0; ks < HD / 16; ++ks) {
        uint32_t ah[4], al[4];
        const int qrow = qb * 16 + (lane & 7) + 8 * ((lane >> 3) & 1), qcol = ks * 16 + 8 * (lane >> 4);
        ldsm4(cvta_smem(Qh + qrow * SM::LD + qcol), ah[0], ah[1], ah[2], ah[3]);
        ldsm4(cvta_smem(Ql + qrow * SM::LD + qcol), al[0], al[1], al[2], al[3]);
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
          const int krow = kk0 + np * 16 + (lane & 7) + 8 * (lane >> 4), kcol = ks * 16 + 8 * ((lane >> 3) & 1);
          uint32_t h0, h1, h2, h3, w0, w1, w2, w3;
          ldsm4(cvta_smem(Kh + krow * SM::LD + kcol), h0, h1, h2, h3);
          ldsm4(cvta_smem(Kl + krow * SM::LD + kcol), w0, w1, w2, w3);
          mma3(sc[2 * np], ah, al, h0, h1, w0, w1);
          mma3(sc[2 * np + 1], ah, al, h2, h3, w2, w3);
        }
      }
      // mask, scale, online softmax (rows gq, gq+8; the 4 lanes of a row hold its 2*NT keys)
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = kb + kk0 + t * 8 + 2 * cq + (e & 1);
          const int qi = (e < 2) ? qi0 : qi1;
          const int rr = (e < 2) ? r0 : r1;
          bool ok = key < kend && qi < Q;
          if (ok && !own && window > 0) ok = S.lo + key >= S.anchor + rr + 1 - window;
          const float x = ok ? sc[t][e] * scale : -INFINITY;
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
#pragma unroll
      for (int t = 0; t < OT; ++t) {
        o[t][0] *= a0;
        o[t][1] *= a0;
        o[t][2] *= a1;
        o[t][3] *= a1;
      }
      // O += P . V, P as hi/lo A fragments straight from the score registers
#pragma unroll
      for (int js = 0; js < KS; ++js) {
        uint32_t ph[4], pl[4];
        split2(sc[2 * js][0], sc[2 * js][1], ph[0], pl[0]);
        split2(sc[2 * js][2], sc[2 * js][3], ph[1], pl[1]);
        split2(sc[2 * js + 1][0], sc[2 * js + 1][1], ph[2], pl[2]);
        split2(sc[2 * js + 1][2], sc[2 * js + 1][3], ph[3], pl[3]);
        const int vrow = kk0 + js * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
        for (int tp = 0; tp < OT / 2; ++tp) {
          const int vcol = tp * 16 + 8 * (lane >> 4);
          uint32_t h0, h1, h2, h3, w0, w1, w2, w3;
          ldsm4t(cvta_smem(Vh + vrow * SM::LD + vcol), h0, h1, h2, h3);
          ldsm4t(cvta_smem(Vl + vrow * SM::LD + vcol), w0, w1, w2, w3);
          mma3(o[2 * tp], ph, pl, h0, h1, w0, w1);
          mma3(o[2 * tp + 1], ph, pl, h2, h3, w2, w3);
        }
      }
    }
  }
  cp_async_wait_all();
  __syncthreads();

  // in-CTA merge of the key groups: per warp 16 rows x (o, m, l) in the scratch
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
  float *out = part + ((int64_t)(b * kv + g) * (nsplit + 1) + sp) * Q * (HD + 2);
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
    float *orow = out + (int64_t)qi * (HD + 2);
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

// y[b*R + r][h*HD + d] = sum_s o_s e^(m_s - M) / sum_s l_s e^(m_s - M)
template <int HD>
__global__ void k_attn_merge(const float *__restrict__ part, int heads, int kv, int R, int nsplit,
                             float *__restrict__ y) {
  pdl_wait();
  const int qi_all = blockIdx.x;  // over kv * Q
  const int b = blockIdx.y;
  const int rep = heads / kv, Q = rep * R;
  const int g = qi_all / Q, qi = qi_all % Q;
  const int hrep = qi / R, r = qi % R;
  const int d = threadIdx.x;
  const float *base = part + (int64_t)(b * kv + g) * (nsplit + 1) * Q * (HD + 2) + (int64_t)qi * (HD + 2);
  const int64_t sstride = (int64_t)Q * (HD + 2);
  float M = -INFINITY;
  for (int s = 0; s <= nsplit; ++s) M = fmaxf(M, base[s * sstride + HD]);
  float L = 0.f, acc = 0.f;
  for (int s = 0; s <= nsplit; ++s) {
    const float m = base[s * sstride + HD];
    if (m == -INFINITY) continue;
    const float e = expf(m - M);
    L = fmaf(base[s * sstride + HD + 1], e, L);
    acc = fmaf(base[s * sstride + d], e, acc);
  }
  y[((int64_t)b * R + r) * heads * HD + (g * rep + hrep) * HD + d] = acc / L;
}

// The same merge written straight into the token tiles of the output
// projection (hi/lo planes; a thread per 8 columns of a query row), with the
// projection's outputs cleared by the blocks past the work grid when it splits.
constexpr int MERGE_THREADS = 32;  // small CTAs: the work is a few thousand threads of dependent loads

template <int HD>
__global__ void __launch_bounds__(MERGE_THREADS) k_attn_merge_pack(const float *__restrict__ part, int heads, int kv, int R,
                                                         int nsplit, int work_blocks, PackDst P, ZeroSet Z) {
  pdl_wait();
  pdl_trigger();  // the GEMM this feeds may fetch its weights meanwhile
  if ((int)blockIdx.x >= work_blocks) {
    if (blockIdx.y == 0) zero_set_clear(Z, blockIdx.x - work_blocks, gridDim.x - work_blocks);
    return;
  }
  constexpr int D8 = HD / 8;
  const int b = blockIdx.y;
  const int rep = heads / kv, Q = rep * R;
  const int id = blockIdx.x * MERGE_THREADS + threadIdx.x;
  if (id >= kv * Q * D8) return;
  const int qa = id / D8, d8 = id - qa * D8;
  const int g = qa / Q, qi = qa - g * Q;
  const int hrep = qi / R, r = qi - hrep * R;
  const float *base = part + (int64_t)(b * kv + g) * (nsplit + 1) * Q * (HD + 2) + (int64_t)qi * (HD + 2);
  const int64_t sstride = (int64_t)Q * (HD + 2);
  float M = -INFINITY;
  for (int s = 0; s <= nsplit; ++s) M = fmaxf(M, base[s * sstride + HD]);
  float L = 0.f, acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int s = 0; s <= nsplit; ++s) {
    const float *ps = base + s * sstride;
    const float m = ps[HD];
    if (m == -INFINITY) continue;
    const float e = expf(m - M);
    L = fmaf(ps[HD + 1], e, L);
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = fmaf(ps[8 * d8 + c], e, acc[c]);
  }
#pragma unroll
  for (int c = 0; c < 8; ++c) acc[c] = acc[c] / L;
  pack_store8(P, b * R + r, (g * rep + hrep) * HD + 8 * d8, acc);
}

template <int HD, int KG>
static cudaError_t launch_attn(const float *q, const float *k, const float *v, const AttnArgs &args, int batch,
                               int max_n, int heads, int kv, int R, int window, float scale, float *part, float *y,
                               int num_sms, const PackDst *pack, const ZeroSet *zero, cudaStream_t st) {
  const size_t smem = AttnSmem<HD>::BYTES;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k_attn<HD, KG>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int cps = chunks_per_split(batch, kv, max_n, num_sms);
  const int ns = max_n > 0 ? ((max_n + CH - 1) / CH + cps - 1) / cps : 0;
  dim3 grid(ns + 1, kv, batch);
  cudaError_t e = launch_pdl(k_attn<HD, KG>, grid, dim3(ATT_THREADS), smem, st, 1, q, k, v, args, heads, kv, R, window,
                             scale, ns, cps, part);
  if (e != cudaSuccess) return e;
  const int Q = heads / kv * R;
  if (pack) {
    const int work = (kv * Q * (HD / 8) + MERGE_THREADS - 1) / MERGE_THREADS;
    int64_t most = 0;
    for (int j = 0; j < zero->count; ++j) most = std::max<int64_t>(most, zero->n[j]);
    const int zb = zero->count ? (int)std::min<int64_t>((most + 4 * MERGE_THREADS - 1) / (4 * MERGE_THREADS), 256) : 0;
    return launch_pdl(k_attn_merge_pack<HD>, dim3(work + zb, batch), dim3(MERGE_THREADS), 0, st, 1, part, heads, kv, R,
                      ns, work, *pack, *zero);
  }
  dim3 g2(kv * Q, batch);
  return launch_pdl(k_attn_merge<HD>, g2, dim3(HD), 0, st, 1, part, heads, kv, R, ns, y);
}

template <int HD>
static cudaError_t launch_attn_hd(const float *q, const float *k, const float *v, const AttnArgs &args, int batch,
                                  int max_n, int heads, int kv, int R, int window, float scale, float *part, float *y,
                                  int num_sms, const PackDst *pack, const ZeroSet *zero, cudaStream_t st) {
  const int QW = (heads / kv * R + 15) / 16;
  if (QW >= 3)
    return launch_attn<HD, 2>(q, k, v, args, batch, max_n, heads, kv, R, window, scale, part, y, num_sms, pack, zero,
                              st);
  return launch_attn<HD, 4>(q, k, v, args, batch, max_n, heads, kv, R, window, scale, part, y, num_sms, pack, zero,
                            st);
}

cudaError_t attention(const float *q, const float *k, const float *v, const AttnSeq *seqs, int batch, int max_ctx,
                      int heads, int kv_heads, int hd, int block, int window, float scale, float *partials, float *y,
                      int num_sms, const PackDst *pack, const ZeroSet *zero, cudaStream_t st) {
  (void)max_ctx;
  if (batch > MAX_BATCH || heads / kv_heads * block > QMAX) return cudaErrorInvalidValue;
  AttnArgs args;
  int max_n = 0;
  for (int i = 0; i < MAX_BATCH; ++i) {
    if (i < batch) {
      args.seq[i] = seqs[i];
      max_n = std::max(max_n, seqs[i].n);
    } else {
      args.seq[i] = AttnSeq{nullptr, nullptr, 0, 0, 0};
    }
  }
  num_sms = std::max(1, std::min(num_sms, 1024));
  if (hd == 128)
    return launch_attn_hd<128>(q, k, v, args, batch, max_n, heads, kv_heads, block, window, scale, partials, y, num_sms,
                               pack, zero, st);
  if (hd == 64)
    return launch_attn_hd<64>(q, k, v, args, batch, max_n, heads, kv_heads, block, window, scale, partials, y, num_sms,
                              pack, zero, st);
  return cudaErrorInvalidValue;
}

}  // namespace dfl

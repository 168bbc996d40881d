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
constexpr int KEYS = 32;        // keys per step
constexpr int QMAX = 64;        // queries per CTA (rep * block)
constexpr int SPLIT_CTAS = 1024;
constexpr int MIN_SPLIT_KEYS = 128;  // keys a split takes at least

struct AttnArgs {
  AttnSeq seq[MAX_BATCH];
};

static int splits_for(int batch, int kv, int max_n) {
  if (max_n <= 0) return 0;
  int s = SPLIT_CTAS / std::max(1, batch * kv);
  s = std::max(1, std::min(s, 128));
  s = std::min(s, (max_n + MIN_SPLIT_KEYS - 1) / MIN_SPLIT_KEYS);
  return s;
}

size_t attn_partial_bytes(int max_batch, int kv_heads, int heads, int block, int hd) {
  const int Q = heads / kv_heads * block;
  size_t worst = 0;
  for (int b = 1; b <= max_batch; ++b) {
    const int s = std::max(1, std::min(128, SPLIT_CTAS / std::max(1, b * kv_heads)));
    worst = std::max(worst, (size_t)b * kv_heads * (s + 1));
  }
  return worst * Q * (hd + 2) * sizeof(float);
}

template <int HD>
__global__ void __launch_bounds__(ATT_THREADS) k_attn(const float *__restrict__ q, const float *__restrict__ k,
                                                      const float *__restrict__ v, AttnArgs args, int heads, int kv,
                                                      int R, int window, float scale, int nsplit, int chunk,
                                                      float *__restrict__ part) {
  extern __shared__ float smf[];
  const int sp = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int rep = heads / kv, Q = rep * R;
  const AttnSeq S = args.seq[b];
  float *Qs = smf;                          // [Q][HD]
  float *Ks = Qs + QMAX * HD;               // [KEYS][HD + 1]
  float *Vs = Ks + KEYS * (HD + 1);         // [KEYS][HD]
  float *P = Vs + KEYS * HD;                // [Q][KEYS]
  float *ms = P + QMAX * KEYS;              // [Q]
  float *ls = ms + QMAX;
  float *al = ls + QMAX;

  const bool own = sp == nsplit;            // the block's own rows
  int kbeg, kend;
  if (own) {
    kbeg = 0;
    kend = R;
  } else {
    kbeg = sp * chunk;
    kend = min(S.n, kbeg + chunk);
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  for (int i = tid; i < Q * HD; i += ATT_THREADS) {
    const int qi = i / HD, d = i % HD;
    const int hrep = qi / R, r = qi % R;
    Qs[i] = q[((int64_t)b * R + r) * heads * HD + (g * rep + hrep) * HD + d];
  }
  for (int i = tid; i < Q; i += ATT_THREADS) {
    ms[i] = -INFINITY;
    ls[i] = 0.f;
  }
  constexpr int OPT = QMAX * HD / ATT_THREADS;  // outputs per thread at most
  constexpr int QSTEP = ATT_THREADS / HD;       // query stride of a thread
  const int od = tid % HD, oq0 = tid / HD;
  float o[OPT];
#pragma unroll
  for (int i = 0; i < OPT; ++i) o[i] = 0.f;
  __syncthreads();

  for (int kb = kbeg; kb < kend; kb += KEYS) {
    for (int i = tid; i < KEYS * HD; i += ATT_THREADS) {
      const int j = i / HD, d = i % HD;
      const int key = kb + j;
      float kk = 0.f, vv = 0.f;
      if (key < kend) {
        if (own) {
          kk = k[((int64_t)b * R + key) * kv * HD + g * HD + d];
          vv = v[((int64_t)b * R + key) * kv * HD + g * HD + d];
        } else {
          kk = S.ck[((int64_t)key * kv + g) * HD + d];
          vv = S.cv[((int64_t)key * kv + g) * HD + d];
        }
      }
      Ks[j * (HD + 1) + d] = kk;
      Vs[j * HD + d] = vv;
    }
    __syncthreads();
    // scores: warp w takes queries w, w+8, ...; lane = key
    for (int qi = warp; qi < Q; qi += ATT_THREADS / 32) {
      const int key = kb + lane;
      float s = -INFINITY;
      if (key < kend) {
        float acc = 0.f;
        const float *qr = Qs + qi * HD;
        const float *kr = Ks + lane * (HD + 1);
#pragma unroll 8
        for (int d = 0; d < HD; ++d) acc = fmaf(qr[d], kr[d], acc);
        s = acc * scale;
        if (!own && window > 0) {
          const int r = qi % R;
          const int64_t pos = S.lo + key;
          if (pos < S.anchor + r + 1 - window) s = -INFINITY;
        }
      }
      const float mx = warp_max(s);
      const float mo = ms[qi];
      const float mn = fmaxf(mo, mx);
      float p = 0.f, alpha = 1.f;
      if (mn != -INFINITY) {
        p = s == -INFINITY ? 0.f : expf(s - mn);
        alpha = mo == -INFINITY ? 0.f : expf(mo - mn);
      }
      const float ps = warp_sum(p);
      P[qi * KEYS + lane] = p;
      __syncwarp();
      if (lane == 0) {
        ms[qi] = mn;
        ls[qi] = ls[qi] * alpha + ps;
        al[qi] = alpha;
      }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < OPT; ++i) {
      const int qi = oq0 + QSTEP * i;
      if (qi < Q) {
        float acc = o[i] * al[qi];
        const float *pr = P + qi * KEYS;
#pragma unroll 8
        for (int j = 0; j < KEYS; ++j) acc = fmaf(pr[j], Vs[j * HD + od], acc);
        o[i] = acc;
      }
    }
    __syncthreads();
  }

  float *out = part + ((int64_t)(b * kv + g) * (nsplit + 1) + sp) * Q * (HD + 2);
#pragma unroll
  for (int i = 0; i < OPT; ++i) {
    const int qi = oq0 + QSTEP * i;
    if (qi < Q) out[qi * (HD + 2) + od] = o[i];
  }
  for (int i = tid; i < Q; i += ATT_THREADS) {
    out[i * (HD + 2) + HD] = ms[i];
    out[i * (HD + 2) + HD + 1] = ls[i];
  }
}

// y[b*R + r][h*HD + d] = sum_s o_s e^(m_s - M) / sum_s l_s e^(m_s - M)
template <int HD>
__global__ void k_attn_merge(const float *__restrict__ part, int heads, int kv, int R, int nsplit,
                             float *__restrict__ y) {
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

template <int HD>
static cudaError_t launch_attn(const float *q, const float *k, const float *v, const AttnArgs &args, int batch,
                               int max_n, int heads, int kv, int R, int window, float scale, float *part, float *y,
                               cudaStream_t st) {
  const int nsplit = splits_for(batch, kv, max_n);
  int chunk = nsplit > 0 ? (max_n + nsplit - 1) / nsplit : 0;
  chunk = (chunk + KEYS - 1) / KEYS * KEYS;
  const int ns = nsplit > 0 ? (max_n + chunk - 1) / chunk : 0;
  const size_t smem = (size_t)(QMAX * HD + KEYS * (HD + 1) + KEYS * HD + QMAX * KEYS + 3 * QMAX) * sizeof(float);
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k_attn<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(ns + 1, kv, batch);
  k_attn<HD><<<grid, ATT_THREADS, smem, st>>>(q, k, v, args, heads, kv, R, window, scale, ns, chunk, part);
  const int Q = heads / kv * R;
  dim3 g2(kv * Q, batch);
  k_attn_merge<HD><<<g2, HD, 0, st>>>(part, heads, kv, R, ns, y);
  count_launch(2);
  return cudaGetLastError();
}

cudaError_t attention(const float *q, const float *k, const float *v, const AttnSeq *seqs, int batch, int max_ctx,
                      int heads, int kv_heads, int hd, int block, int window, float scale, float *partials, float *y,
                      cudaStream_t st) {
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
  if (hd == 128) return launch_attn<128>(q, k, v, args, batch, max_n, heads, kv_heads, block, window, scale, partials, y, st);
  if (hd == 64) return launch_attn<64>(q, k, v, args, batch, max_n, heads, kv_heads, block, window, scale, partials, y, st);
  return cudaErrorInvalidValue;
}

}  // namespace dfl

// The C ABI of the drafter (include/dflash.h) and the host driver that
// enqueues a settle, a block and a selection. The pass follows cortiq-engine
// src/gpu_cuda/hyb/dflash.rs (`Dev::settle`, `Dev::block`) and
// src/cortiq_engine/dflash.rs (`Drafter::block`, `Drafter::select_with`); the
// context bookkeeping follows the host drafter (`Drafter::queue_context`,
// `settle`, `truncate`, the window trim of `settle_rows`). The host keeps each
// sequence's (first, len, dropped per layer, waiting rows); the device memory
// is the caller's.
#include <algorithm>
#include <cmath>
#include <climits>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "dflash.h"
#include "kernels.h"

namespace dfl {
std::atomic<unsigned long long> g_launches{0};
}

namespace {

thread_local std::string g_err;

int fail(int code, const std::string &msg) {
  g_err = msg;
  return code;
}

#define DF_CUDA(call)                                                                            \
  do {                                                                                           \
    cudaError_t e_ = (call);                                                                     \
    if (e_ != cudaSuccess) return fail(DFLASH_E_CUDA, std::string(#call) + ": " + cudaGetErrorString(e_)); \
  } while (0)

constexpr size_t ALIGN = 256;
size_t up(size_t n) { return (n + ALIGN - 1) / ALIGN * ALIGN; }

bool aligned16(const void *p) { return ((uintptr_t)p & 15) == 0; }

// A sequence's context (dflash.rs `Drafter`: first, len, `Ctx::dropped` per
// layer, the pending rows). The pending rows live in the caller's buffer as a
// ring of `pcap` rows: `pcount` rows from slot `phead` on, of positions
// first + len ...
struct Seq {
  int64_t first = 0, len = 0;
  int64_t dropped[DFLASH_MAX_LAYERS] = {};
  float *pbuf = nullptr;
  int64_t pcap = 0, phead = 0, pcount = 0;
};

// Rows of the host drafter's bookkeeping (dflash.rs, module constants).
constexpr int64_t PENDING_ROWS = 512;
constexpr int64_t BLOCK_SLACK = 256;
constexpr int64_t CONTEXT_CHUNK = 64;

// Workspace carve; sizes in bytes.
struct Carve {
  size_t h, x, xc, d, d2, q, k, v, y, o, gt, up, part, sel, act, act_fc, kvs, kp, vp, total;
};

Carve carve_of(const dflash_geometry &g, int max_batch) {
  const int R = g.block;
  const size_t T = (size_t)max_batch * R;                           // block rows
  const size_t Tx = std::max(T, (size_t)DFLASH_SETTLE_MAX);          // x also holds a settle's rows
  const size_t G = (size_t)g.hidden / g.conv_group;
  const size_t pr = 2 * (size_t)g.conv_kernel * G;
  const size_t f = sizeof(float);
  Carve c{};
  c.h = up(T * g.hidden * f);
  c.x = up(Tx * g.hidden * f);
  c.xc = up(T * g.hidden * f);
  c.d = up(T * pr * f);
  c.d2 = c.d;  // the MLP's kernel projection (the attention's d is still read when it is written)
  c.q = up(T * (size_t)g.heads * g.head_dim * f);
  c.k = up(T * (size_t)g.kv_heads * g.head_dim * f);
  c.v = c.k;
  c.y = c.q;
  c.o = up(T * g.hidden * f);
  c.gt = up(T * (size_t)g.intermediate * f);
  c.up = c.gt;
  c.part = up(dfl::attn_partial_bytes(max_batch, g.kv_heads, g.heads, R, g.head_dim));
  const size_t kvd = (size_t)g.kv_heads * g.head_dim;
  c.kvs = up((size_t)2 * g.layers * DFLASH_SETTLE_MAX * kvd * f);  // a settle's K and V before their planes
  c.kp = up(T * kvd * 4);                                          // the block's own K and V as f16 planes
  c.vp = c.kp;
  c.sel = up(dfl::select_scratch_bytes(max_batch * (R - 1), g.vocab, g.selector_top));
  // packed token tiles of the largest GEMM (block rows, a settle chunk, the fc's taps)
  const int Tb = max_batch * R;
  const int kmax = std::max(std::max(g.hidden, g.intermediate), g.heads * g.head_dim);
  c.act = up(std::max({dfl::tc_act_bytes(Tb, kmax, true), dfl::tc_act_bytes(DFLASH_SETTLE_MAX, g.hidden, true),
                       dfl::tc_act_bytes(Tb, g.hidden, false)}));
  // the settle's fc has token tiles of its own, which it packs from the taps while
  // the previous settle's last kernel runs
  c.act_fc = up(dfl::tc_act_bytes(DFLASH_SETTLE_MAX, g.taps * g.hidden, false));
  c.total = c.h + c.x + c.xc + c.d + c.d2 + c.q + c.k + c.v + c.y + c.o + c.gt + c.up + c.part + c.sel + c.act +
            c.act_fc + c.kvs + c.kp + c.vp;
  return c;
}

std::string check_geometry(const dflash_geometry &g) {
  // Geometry::of's rules (src/cortiq_engine/dflash.rs)
  if (g.layers < 1 || g.layers > DFLASH_MAX_LAYERS) return "layers must be 1..64";
  if (g.block < 2) return "block must be at least 2";
  if (g.taps < 1) return "no taps";
  if (g.kv_heads < 1) return "kv_heads must be at least 1";
  if (g.heads % g.kv_heads != 0) return "heads must be a multiple of kv_heads";
  if (g.head_dim % 2 != 0) return "head_dim must be even";
  if (g.conv_group < 1) return "conv_group must be at least 1";
  if (g.hidden % g.conv_group != 0) return "hidden must be a multiple of conv_group";
  for (int l = 0; l < g.layers; ++l)
    if (g.windows[l] < 0) return "a negative window";
  // this build's limits
  if (g.block > DFLASH_MAX_BLOCK) return "block must be at most 16";
  if (g.head_dim != 64 && g.head_dim != 128) return "head_dim must be 64 or 128";
  if (g.hidden % 64 || g.intermediate % 64 || (g.heads * g.head_dim) % 64)
    return "hidden, intermediate and heads*head_dim must be multiples of 64";
  if ((g.kv_heads * g.head_dim) % 16) return "kv_heads*head_dim must be a multiple of 16";
  if (g.vocab < 16 || g.vocab % 16) return "vocab must be a positive multiple of 16";
  if (g.vocab > (1 << 21)) return "vocab must be at most 2,097,152";
  if ((2 * g.conv_kernel * (g.hidden / g.conv_group)) % 16) return "2*conv_kernel*groups must be a multiple of 16";
  if (g.conv_kernel < 1 || g.conv_kernel > DFLASH_MAX_BLOCK) return "conv_kernel must be 1..16";
  if (g.selector_rank < 16 || g.selector_rank > 256 || g.selector_rank % 16) return "selector_rank must be 16..256, a multiple of 16";
  if (g.selector_top < 1 || g.selector_top > 32 || g.selector_top > g.vocab) return "selector_top must be 1..32";
  if (g.quant_group != 32 && g.quant_group != 64 && g.quant_group != 128) return "quant_group must be 32, 64 or 128";
  if (g.hidden % g.quant_group || g.intermediate % g.quant_group || (g.heads * g.head_dim) % g.quant_group)
    return "every four-bit matrix's columns must be a multiple of quant_group";
  if (g.heads / g.kv_heads * g.block > 64) return "heads/kv_heads * block must be at most 64";
  if (!(g.eps >= 0.0) || !(g.rope_theta > 0.0)) return "eps must be >= 0 and rope_theta > 0";
  return "";
}

}  // namespace

namespace dfl {
// Record a failure message for dflash_last_error() from another file of the library.
int dflash_fail(int code, const std::string &msg) { return fail(code, msg); }
}  // namespace dfl

namespace {

bool int4_ok(const dflash_matrix &m) { return m.data && m.scales && aligned16(m.data) && aligned16(m.scales); }
bool f16_ok(const dflash_matrix &m) { return m.data && aligned16(m.data); }

}  // namespace

struct dflash_t {
  dflash_geometry g;
  dflash_weights w;
  std::vector<dflash_layer_weights> layers;
  int max_batch = 0;
  std::vector<__half *> ck, cv;   // context caches [seq * layers + l], [rows][kv][planes][hd]
  int64_t cap = 0;                // rows of a linear cache
  int planes = 2;                 // 2: DFLASH_KV_PLANES, 1: DFLASH_KV_F16
  int ring[DFLASH_MAX_LAYERS] = {};    // a layer's ring rows C (0: linear)
  int mirror[DFLASH_MAX_LAYERS] = {};  // rows past the ring repeating its first ones (the window)
  char *ws = nullptr;
  Carve c{};
  float *h, *x, *xc, *d, *d2, *q, *k, *v, *y, *o, *gt, *up, *part, *kvs;
  __half *kp, *vp;
  void *sel, *act, *act_fc;
  std::vector<Seq> seqs;
  std::vector<float> inv;
  int num_sms = 148;
  // tensor maps of the context caches [seq * layers + layer] and of the block's
  // own K and V, encoded at the first block (host-only work)
  std::vector<CUtensorMap> kmap, vmap;
  CUtensorMap own_k, own_v;
  bool maps = false;
};

namespace {
// Rows of layer l's cache: a linear cache's ctx_cap, or a ring and its mirror.
int64_t layer_rows(const dflash_t *d, int l) { return d->ring[l] ? (int64_t)d->ring[l] + d->mirror[l] : d->cap; }

bool encode_maps(dflash_t *d) {
  if (d->maps) return true;
  const dflash_geometry &g = d->g;
  const size_t n = (size_t)d->max_batch * g.layers;
  d->kmap.resize(n);
  d->vmap.resize(n);
  for (size_t i = 0; i < n; ++i) {
    const int64_t rows = layer_rows(d, (int)(i % g.layers));
    if (!dfl::attn_kv_map(&d->kmap[i], d->ck[i], rows, g.kv_heads, g.head_dim, d->planes, 64) ||
        !dfl::attn_kv_map(&d->vmap[i], d->cv[i], rows, g.kv_heads, g.head_dim, d->planes, 64))
      return false;
  }
  const int64_t rows = (int64_t)d->max_batch * g.block;
  if (!dfl::attn_kv_map(&d->own_k, d->kp, rows, g.kv_heads, g.head_dim, d->planes, g.block) ||
      !dfl::attn_kv_map(&d->own_v, d->vp, rows, g.kv_heads, g.head_dim, d->planes, g.block))
    return false;
  d->maps = true;
  return true;
}

int64_t pending_limit(const dflash_geometry &g) {
  int64_t widest = 0;
  bool all = true;
  for (int l = 0; l < g.layers; ++l) {
    all = all && g.windows[l] > 0;
    widest = std::max<int64_t>(widest, g.windows[l]);
  }
  return all ? std::max(PENDING_ROWS, widest + BLOCK_SLACK) : PENDING_ROWS;
}

// dflash.rs `Drafter::truncate`: waiting rows past pos, settled rows at or past it.
void truncate_seq(dflash_t *d, Seq &s, int64_t pos) {
  const int64_t held = s.first + s.len;
  s.pcount = std::min(s.pcount, std::max<int64_t>(pos - held, 0));
  const int64_t keep = std::min(std::max<int64_t>(pos - s.first, 0), s.len);
  for (int l = 0; l < d->g.layers; ++l) s.dropped[l] = std::min(s.dropped[l], keep);
  s.len = keep;
}

// The position rule of `Drafter::queue_context`: a gap starts the context over at
// pos; a held position (first <= pos <= the next position) truncates there.
void restart_or_truncate(dflash_t *d, Seq &s, int64_t pos) {
  if (pos > s.first + s.len + s.pcount || pos < s.first) {
    truncate_seq(d, s, 0);
    s.pcount = 0;
    s.phead = 0;
    s.first = pos;
  } else {
    truncate_seq(d, s, pos);
  }
}

// The end of `Drafter::settle_rows`: a windowed layer holding more than twice its
// window lets go of all but its last `window` rows.
void window_trim(dflash_t *d, Seq &s) {
  for (int l = 0; l < d->g.layers; ++l) {
    const int64_t w = d->g.windows[l], held = s.len - s.dropped[l];
    if (w > 0 && held > 2 * w) s.dropped[l] += held - w;
  }
}

// Whether the linear caches take rows up to (not including) cache row `end`.
bool fits(const dflash_t *d, int64_t end) {
  for (int l = 0; l < d->g.layers; ++l)
    if (!d->ring[l] && end > d->cap) return false;
  return true;
}

// Cache rows of every layer of `seq`, for ctx_planes.
void cache_rows(const dflash_t *d, int seq, dfl::CtxWrite &W) {
  const dflash_geometry &g = d->g;
  for (int l = 0; l < g.layers; ++l) {
    W.ck[l] = d->ck[(size_t)seq * g.layers + l];
    W.cv[l] = d->cv[(size_t)seq * g.layers + l];
    W.ring[l] = d->ring[l];
    W.mirror[l] = d->mirror[l];
    W.w[l] = d->layers[l].k_norm;
    W.rotary[l] = g.no_rope[l] == 0;
  }
}
}  // namespace

namespace {
// gpu_cuda/hyb/dflash.rs `Dev::settle`: n (<= 1024) tap rows of positions
// first + len .. into every layer's cache at row index len: t = rms(fc .
// f16(taps), hidden_norm); per layer K = rot(rms_head(Wk t, k_norm)), V = Wv t.
int settle_call(dflash_t *d, int seq, const float *taps, int n, cudaStream_t st) {
  Seq &s = d->seqs[seq];
  const dflash_geometry &g = d->g;
  const int hs = g.hidden, tw = g.taps * g.hidden, kvd = g.kv_heads * g.head_dim;
  const dfl::TcJob fc{d->w.fc.data, nullptr, d->x, hs, hs};
  if (n > 32) {
    // the taps come from the caller: their packing needs no kernel before it
    const dfl::WideJob fj{d->w.fc.data, nullptr, d->x, hs, hs, 0};
    DF_CUDA(dfl::wide_gemm(&fj, 1, 0, false, 0, taps, tw, n, tw, d->act_fc, d->num_sms, st, nullptr, 0.f, true));
  } else {
    DF_CUDA(dfl::tc_gemm_f16(&fc, 1, taps, tw, n, tw, d->act, d->num_sms, st));
  }
  // the hidden norm is taken by the K/V GEMM's packing of t (below)
  // k = Wk rms(t), v = Wv rms(t) of every layer in one GEMM (into the
  // workspace), then k normed and rotated and both written into the caches
  dfl::WideJob kv[dfl::WIDE_MAX_JOBS];
  dfl::CtxWrite W{};
  cache_rows(d, seq, W);
  for (int l = 0; l < g.layers; ++l) {
    const dflash_layer_weights &L = d->layers[l];
    float *yk = d->kvs + (size_t)(2 * l) * DFLASH_SETTLE_MAX * kvd, *yv = yk + (size_t)DFLASH_SETTLE_MAX * kvd;
    W.k[l] = yk;
    W.v[l] = yv;
    kv[2 * l] = dfl::WideJob{L.k.data, L.k.scales, yk, kvd, kvd, 0};
    kv[2 * l + 1] = dfl::WideJob{L.v.data, L.v.scales, yv, kvd, kvd, 0};
  }
  DF_CUDA(dfl::wide_gemm(kv, 2 * g.layers, 0, true, g.quant_group, d->x, hs, n, hs, d->act, d->num_sms, st,
                          d->w.hidden_norm, (float)g.eps));
  DF_CUDA(dfl::ctx_planes(W, g.layers, n, g.kv_heads, g.head_dim, d->planes, (float)g.eps, d->inv.data(),
                           s.first + s.len, s.len, true, st));
  s.len += n;
  return DFLASH_OK;
}

// A run of rows for one settle (`Drafter::settle_rows`): device tap rows.
struct Seg {
  const float *taps;
  int64_t n;
};

// `Drafter::settle_rows` over the rows of `segs` in order (positions first + len ..),
// in calls of at most DFLASH_SETTLE_MAX rows, then the window trim.
int settle_rows(dflash_t *d, int seq, const Seg *segs, int nseg, cudaStream_t st) {
  const size_t tw = (size_t)d->g.taps * d->g.hidden;
  for (int i = 0; i < nseg; ++i)
    for (int64_t r = 0; r < segs[i].n; r += DFLASH_SETTLE_MAX) {
      const int n = (int)std::min<int64_t>(DFLASH_SETTLE_MAX, segs[i].n - r);
      if (int e = settle_call(d, seq, segs[i].taps + (size_t)r * tw, n, st)) return e;
    }
  window_trim(d, d->seqs[seq]);
  return DFLASH_OK;
}

// The `take` oldest waiting rows as up to two runs of the pending ring.
int pending_segs(const Seq &s, int64_t take, size_t tw, Seg *out) {
  if (take <= 0) return 0;
  const int64_t first = std::min(take, s.pcap - s.phead);
  out[0] = Seg{s.pbuf + (size_t)s.phead * tw, first};
  if (first == take) return 1;
  out[1] = Seg{s.pbuf, take - first};
  return 2;
}

// `Drafter::queue_context` (queue = true: the rows left under the limit wait in
// the pending buffer) or `push_context` (queue = false: they settle now).
int add_context(dflash_t *d, int seq, int64_t pos, const float *taps, int n, bool queue, cudaStream_t st) {
  Seq &s = d->seqs[seq];
  const size_t tw = (size_t)d->g.taps * d->g.hidden;
  const int64_t limit = pending_limit(d->g);
  Seq after = s;
  restart_or_truncate(d, after, pos);
  // rows up to the end of these must fit the linear caches
  if (!fits(d, pos - after.first + n)) return fail(DFLASH_E_CAPACITY, "context rows do not fit the cache");
  if (queue && !s.pbuf) return fail(DFLASH_E_ARG, "queue: no pending buffer (dflash_bind_pending)");
  s = after;
  int64_t total = s.pcount + n;
  int64_t used = 0;  // of the new rows
  if (total > limit) {
    const int64_t over = std::min((total - limit + CONTEXT_CHUNK - 1) / CONTEXT_CHUNK * CONTEXT_CHUNK, total);
    Seg segs[3];
    const int64_t from_pending = std::min(over, s.pcount);
    int ns = pending_segs(s, from_pending, tw, segs);
    used = over - from_pending;
    if (used > 0) segs[ns++] = Seg{taps, used};
    s.phead = s.pcap ? (s.phead + from_pending) % s.pcap : 0;
    s.pcount -= from_pending;
    if (int e = settle_rows(d, seq, segs, ns, st)) return e;
  }
  const int64_t rest = n - used;
  if (!queue) {
    Seg segs[3];
    int ns = pending_segs(s, s.pcount, tw, segs);
    if (rest > 0) segs[ns++] = Seg{taps + (size_t)used * tw, rest};
    s.pcount = 0;
    s.phead = 0;
    return ns ? settle_rows(d, seq, segs, ns, st) : DFLASH_OK;
  }
  // the rest wait: copied behind the pending rows (up to two runs of the ring)
  int64_t done = 0;
  while (done < rest) {
    const int64_t slot = (s.phead + s.pcount) % s.pcap;
    const int64_t m = std::min(rest - done, s.pcap - slot);
    DF_CUDA(cudaMemcpyAsync(s.pbuf + (size_t)slot * tw, taps + (size_t)(used + done) * tw, (size_t)m * tw * 4,
                             cudaMemcpyDeviceToDevice, st));
    s.pcount += m;
    done += m;
  }
  return DFLASH_OK;
}
}  // namespace

extern "C" {

const char *dflash_last_error(void) { return g_err.c_str(); }

uint64_t dflash_launch_count(void) { return dfl::g_launches.load(); }

size_t dflash_int4_packed_bytes(int64_t rows, int64_t cols, int32_t group) {
  if (rows <= 0 || cols <= 0 || cols % 64 || (group != 32 && group != 64 && group != 128) || cols % group)
    return 0;
  return dfl::tc_int4_codes_bytes(rows, cols);
}

size_t dflash_int4_scale_bytes(int64_t rows, int64_t cols, int32_t group) {
  if (dflash_int4_packed_bytes(rows, cols, group) == 0) return 0;
  return dfl::tc_int4_scale_bytes(rows, cols, group);
}

size_t dflash_f16_packed_bytes(int64_t rows, int64_t cols) {
  if (rows <= 0 || cols <= 0 || cols % 64) return 0;
  return dfl::tc_f16_bytes(rows, cols);
}

int dflash_pack_int4(const uint8_t *codes, const uint16_t *scales, int64_t rows, int64_t cols, int32_t group,
                     void *dst_codes, void *dst_scales, void *stream) {
  if (dflash_int4_packed_bytes(rows, cols, group) == 0) return fail(DFLASH_E_ARG, "pack_int4: unsupported shape");
  if (!codes || !scales || !dst_codes || !dst_scales) return fail(DFLASH_E_ARG, "pack_int4: null pointer");
  if (!aligned16(dst_codes) || !aligned16(dst_scales)) return fail(DFLASH_E_ARG, "pack_int4: misaligned output");
  DF_CUDA(dfl::tc_pack_int4(codes, scales, rows, cols, group, dst_codes, dst_scales, (cudaStream_t)stream));
  return DFLASH_OK;
}

int dflash_pack_f16(const uint16_t *src, int64_t rows, int64_t cols, void *dst, void *stream) {
  if (dflash_f16_packed_bytes(rows, cols) == 0) return fail(DFLASH_E_ARG, "pack_f16: unsupported shape");
  if (!src || !dst) return fail(DFLASH_E_ARG, "pack_f16: null pointer");
  if (!aligned16(dst)) return fail(DFLASH_E_ARG, "pack_f16: misaligned output");
  DF_CUDA(dfl::tc_pack_f16(src, rows, cols, dst, (cudaStream_t)stream));
  return DFLASH_OK;
}

int dflash_dequant_int4(const void *codes, const void *scales, int64_t rows, int64_t cols, int32_t group, float *out,
                        void *stream) {
  if (dflash_int4_packed_bytes(rows, cols, group) == 0) return fail(DFLASH_E_ARG, "dequant_int4: unsupported shape");
  if (!codes || !scales || !out) return fail(DFLASH_E_ARG, "dequant_int4: null pointer");
  if (!aligned16(codes) || !aligned16(scales)) return fail(DFLASH_E_ARG, "dequant_int4: misaligned input");
  DF_CUDA(dfl::tc_dequant_int4(codes, scales, rows, cols, group, out, (cudaStream_t)stream));
  return DFLASH_OK;
}

size_t dflash_gemm_workspace_bytes(int32_t kind, int64_t cols, int32_t T) {
  if ((kind != 4 && kind != 16) || cols <= 0 || cols % 64 || cols > INT32_MAX || T < 1) return 0;
  return dfl::tc_act_bytes(T, (int)cols, kind == 4);
}

int dflash_gemm(const dflash_matrix *w, int32_t kind, int64_t rows, int64_t cols, int32_t group, const float *x,
                int32_t T, float *y, void *workspace, size_t workspace_bytes, void *stream) {
  if (!w || !x || !y || T < 1) return fail(DFLASH_E_ARG, "gemm: null pointer or no rows");
  if (((uintptr_t)x & 3) || ((uintptr_t)y & 3)) return fail(DFLASH_E_ARG, "gemm: misaligned x or y");
  if (rows > INT32_MAX || cols > INT32_MAX) return fail(DFLASH_E_ARG, "gemm: matrix too large");
  const size_t need = dflash_gemm_workspace_bytes(kind, cols, T);
  if (need == 0) return fail(DFLASH_E_ARG, "gemm: kind must be 4 or 16, cols a multiple of 64");
  if (!workspace || ((uintptr_t)workspace & 15)) return fail(DFLASH_E_ARG, "gemm: null or misaligned workspace");
  if (workspace_bytes < need) return fail(DFLASH_E_CAPACITY, "gemm: workspace smaller than dflash_gemm_workspace_bytes");
  int sms = 148, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  dfl::TcJob job{w->data, w->scales, y, (int)rows, (int)rows};
  if (kind == 4) {
    if (dflash_int4_packed_bytes(rows, cols, group) == 0) return fail(DFLASH_E_ARG, "gemm: unsupported int4 shape");
    if (!int4_ok(*w)) return fail(DFLASH_E_ARG, "gemm: null or misaligned matrix");
    DF_CUDA(dfl::tc_gemm_int4(&job, 1, group, x, (int)cols, T, (int)cols, workspace, sms, (cudaStream_t)stream));
  } else {
    if (!f16_ok(*w)) return fail(DFLASH_E_ARG, "gemm: null or misaligned matrix");
    DF_CUDA(dfl::tc_gemm_f16(&job, 1, x, (int)cols, T, (int)cols, workspace, sms, (cudaStream_t)stream));
  }
  return DFLASH_OK;
}

int dflash_gemm_packed(const dflash_matrix *w, int32_t kind, int64_t rows, int64_t cols, int32_t group, int32_t T,
                       float *y, const void *workspace, void *stream) {
  if (!w || !y || !workspace || T < 1 || T > 32) return fail(DFLASH_E_ARG, "gemm_packed: null pointer or T not 1..32");
  if (((uintptr_t)y & 3) || ((uintptr_t)workspace & 15)) return fail(DFLASH_E_ARG, "gemm_packed: misaligned y or workspace");
  if (rows > INT32_MAX || cols > INT32_MAX || dflash_gemm_workspace_bytes(kind, cols, T) == 0)
    return fail(DFLASH_E_ARG, "gemm_packed: kind must be 4 or 16, cols a multiple of 64");
  int sms = 148, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaStream_t st = (cudaStream_t)stream;
  dfl::TcJob job{w->data, w->scales, y, (int)rows, (int)rows};
  if (kind == 4) {
    if (dflash_int4_packed_bytes(rows, cols, group) == 0) return fail(DFLASH_E_ARG, "gemm_packed: unsupported int4 shape");
    if (!int4_ok(*w)) return fail(DFLASH_E_ARG, "gemm_packed: null or misaligned matrix");
    if (dfl::tc_splits_int4(&job, 1, T, (int)cols, sms))
      DF_CUDA(cudaMemsetAsync(y, 0, (size_t)T * rows * sizeof(float), st));
    DF_CUDA(dfl::tc_gemm_int4_packed(&job, 1, group, workspace, T, (int)cols, sms, st));
  } else {
    if (!f16_ok(*w)) return fail(DFLASH_E_ARG, "gemm_packed: null or misaligned matrix");
    if (dfl::tc_splits_f16(&job, 1, T, (int)cols, sms))
      DF_CUDA(cudaMemsetAsync(y, 0, (size_t)T * rows * sizeof(float), st));
    DF_CUDA(dfl::tc_gemm_f16_packed(&job, 1, workspace, dfl::tc_tile_rows(T, false) * 128, T, (int)cols, sms, st));
  }
  return DFLASH_OK;
}

int dflash_device_error(uint32_t *error, int32_t reset) {
  if (!error) return fail(DFLASH_E_ARG, "device_error: null pointer");
  unsigned v = 0;
  DF_CUDA(dfl::read_device_error(&v, reset != 0));
  *error = v;
  return DFLASH_OK;
}

size_t dflash_workspace_bytes(const dflash_geometry *g, int32_t max_batch) {
  if (!g || max_batch < 1 || max_batch > dfl::MAX_BATCH || !check_geometry(*g).empty()) return 0;
  return carve_of(*g, max_batch).total;
}

int64_t dflash_cache_rows(const dflash_geometry *g, const dflash_cache_config *cache, int32_t layer, int64_t ctx_cap) {
  if (!g || layer < 0 || layer >= g->layers || layer >= DFLASH_MAX_LAYERS || ctx_cap < 1) return 0;
  const int64_t C = cache ? cache->ring[layer] : 0;
  if (C == 0) return ctx_cap;
  const int64_t w = g->windows[layer];
  if (w <= 0 || C < 2 * w || C > INT32_MAX / 2) return 0;
  return C + w;
}

size_t dflash_cache_bytes(const dflash_geometry *g, const dflash_cache_config *cache, int32_t layer, int64_t ctx_cap) {
  const int64_t rows = dflash_cache_rows(g, cache, layer, ctx_cap);
  if (rows == 0) return 0;
  const int fmt = cache ? cache->format : DFLASH_KV_PLANES;
  if (fmt != DFLASH_KV_PLANES && fmt != DFLASH_KV_F16) return 0;
  return (size_t)rows * g->kv_heads * g->head_dim * (fmt == DFLASH_KV_PLANES ? 4 : 2);
}

int dflash_create(dflash_t **out, const dflash_geometry *g, const dflash_weights *w, int32_t max_batch,
                  void *const *ctx_k, void *const *ctx_v, int64_t ctx_cap, void *workspace,
                  size_t workspace_bytes) {
  dflash_cache_config cache{};
  cache.format = DFLASH_KV_PLANES;
  return dflash_create_ex(out, g, w, max_batch, &cache, ctx_k, ctx_v, ctx_cap, workspace, workspace_bytes);
}

int dflash_create_ex(dflash_t **out, const dflash_geometry *g, const dflash_weights *w, int32_t max_batch,
                     const dflash_cache_config *cache, void *const *ctx_k, void *const *ctx_v, int64_t ctx_cap,
                     void *workspace, size_t workspace_bytes) {
  if (!out || !g || !w || !cache) return fail(DFLASH_E_ARG, "create: null argument");
  *out = nullptr;
  const std::string why = check_geometry(*g);
  if (!why.empty()) return fail(DFLASH_E_GEOMETRY, "unsupported DFlash geometry: " + why);
  if (max_batch < 1 || max_batch > dfl::MAX_BATCH) return fail(DFLASH_E_ARG, "create: max_batch must be 1..64");
  if (!ctx_k || !ctx_v || ctx_cap < 1) return fail(DFLASH_E_ARG, "create: context caches");
  if (ctx_cap > INT32_MAX) return fail(DFLASH_E_ARG, "create: ctx_cap must be below 2^31");
  if (cache->format != DFLASH_KV_PLANES && cache->format != DFLASH_KV_F16)
    return fail(DFLASH_E_ARG, "create: cache format must be DFLASH_KV_PLANES or DFLASH_KV_F16");
  for (int l = 0; l < g->layers; ++l)
    if (dflash_cache_rows(g, cache, l, ctx_cap) == 0)
      return fail(DFLASH_E_ARG, "create: a ring needs a windowed layer and at least twice its window rows (layer " +
                                    std::to_string(l) + ")");
  if (!workspace || !aligned16(workspace)) return fail(DFLASH_E_ARG, "create: null or misaligned workspace");
  const Carve c = carve_of(*g, max_batch);
  if (workspace_bytes < c.total) return fail(DFLASH_E_CAPACITY, "create: workspace smaller than dflash_workspace_bytes");
  if (!w->layers) return fail(DFLASH_E_ARG, "create: no layers");
  if (!f16_ok(w->fc) || !f16_ok(w->sel) || !int4_ok(w->head) || !w->hidden_norm || !w->norm || !w->pred_book ||
      !w->succ_book)
    return fail(DFLASH_E_ARG, "create: a null or misaligned weight");
  for (int l = 0; l < g->layers; ++l) {
    const dflash_layer_weights &L = w->layers[l];
    if (!L.in_norm || !L.post_norm || !L.q_norm || !L.k_norm || !L.attn_base || !L.mlp_base ||
        !f16_ok(L.attn_proj) || !f16_ok(L.mlp_proj) || !int4_ok(L.q) || !int4_ok(L.k) || !int4_ok(L.v) ||
        !int4_ok(L.o) || !int4_ok(L.gate) || !int4_ok(L.up) || !int4_ok(L.down))
      return fail(DFLASH_E_ARG, "create: a null or misaligned weight of layer " + std::to_string(l));
  }
  for (int i = 0; i < max_batch * g->layers; ++i)
    if (!ctx_k[i] || !ctx_v[i] || !aligned16(ctx_k[i]) || !aligned16(ctx_v[i]))
      return fail(DFLASH_E_ARG, "create: a null or misaligned context cache");

  dflash_t *d = new (std::nothrow) dflash_t;
  if (!d) return fail(DFLASH_E_NOMEM, "create: out of host memory");
  d->g = *g;
  d->w = *w;
  d->layers.assign(w->layers, w->layers + g->layers);
  d->w.layers = d->layers.data();
  d->max_batch = max_batch;
  for (int i = 0; i < max_batch * g->layers; ++i) {
    d->ck.push_back((__half *)ctx_k[i]);
    d->cv.push_back((__half *)ctx_v[i]);
  }
  d->cap = ctx_cap;
  d->planes = cache->format == DFLASH_KV_PLANES ? 2 : 1;
  for (int l = 0; l < g->layers; ++l) {
    d->ring[l] = cache->ring[l];
    d->mirror[l] = cache->ring[l] ? g->windows[l] : 0;
  }
  d->ws = (char *)workspace;
  d->c = c;
  char *p = d->ws;
  auto take = [&](size_t n) {
    char *r = p;
    p += n;
    return r;
  };
  d->h = (float *)take(c.h);
  d->x = (float *)take(c.x);
  d->xc = (float *)take(c.xc);
  d->d = (float *)take(c.d);
  d->d2 = (float *)take(c.d2);
  d->q = (float *)take(c.q);
  d->k = (float *)take(c.k);
  d->v = (float *)take(c.v);
  d->y = (float *)take(c.y);
  d->o = (float *)take(c.o);
  d->gt = (float *)take(c.gt);
  d->up = (float *)take(c.up);
  d->part = (float *)take(c.part);
  d->kvs = (float *)take(c.kvs);
  d->kp = (__half *)take(c.kp);
  d->vp = (__half *)take(c.vp);
  d->sel = take(c.sel);
  d->act = take(c.act);
  d->act_fc = take(c.act_fc);
  d->seqs.assign(max_batch, Seq{});
  // inv_freq = f32(theta^(-2i/hd)) (src/cortiq_engine/dflash.rs, Drafter::new)
  d->inv.resize(g->head_dim / 2);
  for (int i = 0; i < g->head_dim / 2; ++i)
    d->inv[i] = (float)std::pow(g->rope_theta, -(2.0 * i) / (double)g->head_dim);
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0) d->num_sms = n;
  }
  *out = d;
  return DFLASH_OK;
}

void dflash_destroy(dflash_t *d) { delete d; }

int dflash_reset(dflash_t *d, int32_t seq, int64_t first) {
  if (!d || seq < 0 || seq >= d->max_batch || first < 0) return fail(DFLASH_E_ARG, "reset: bad sequence or position");
  Seq &s = d->seqs[seq];
  float *buf = s.pbuf;
  const int64_t cap = s.pcap;
  s = Seq{};
  s.pbuf = buf;
  s.pcap = cap;
  s.first = first;
  return DFLASH_OK;
}

int dflash_context(const dflash_t *d, int32_t seq, int64_t *first, int64_t *len) {
  return dflash_context_ex(d, seq, first, len, nullptr, nullptr);
}

int dflash_context_ex(const dflash_t *d, int32_t seq, int64_t *first, int64_t *len, int64_t *pending,
                      int64_t *dropped) {
  if (!d || seq < 0 || seq >= d->max_batch) return fail(DFLASH_E_ARG, "context: bad sequence");
  const Seq &s = d->seqs[seq];
  if (first) *first = s.first;
  if (len) *len = s.len;
  if (pending) *pending = s.pcount;
  if (dropped)
    for (int l = 0; l < d->g.layers; ++l) dropped[l] = s.dropped[l];
  return DFLASH_OK;
}

int64_t dflash_pending_limit(const dflash_geometry *g) {
  if (!g || g->layers < 1 || g->layers > DFLASH_MAX_LAYERS) return 0;
  return pending_limit(*g);
}

int dflash_bind_pending(dflash_t *d, int32_t seq, void *buf, int64_t rows) {
  if (!d || seq < 0 || seq >= d->max_batch) return fail(DFLASH_E_ARG, "bind_pending: bad sequence");
  Seq &s = d->seqs[seq];
  if (buf && (!aligned16(buf) || rows < 1)) return fail(DFLASH_E_ARG, "bind_pending: misaligned buffer or no rows");
  if (buf && rows < pending_limit(d->g))
    return fail(DFLASH_E_CAPACITY, "bind_pending: fewer rows than dflash_pending_limit");
  s.pbuf = (float *)buf;
  s.pcap = buf ? rows : 0;
  s.phead = s.pcount = 0;
  return DFLASH_OK;
}

static int context_call_checks(dflash_t *d, int32_t seq, int64_t pos, const void *rows, int32_t n, const char *who) {
  if (!d) return fail(DFLASH_E_ARG, std::string(who) + ": null drafter");
  if (seq < 0 || seq >= d->max_batch) return fail(DFLASH_E_ARG, std::string(who) + ": bad sequence");
  if (n < 1 || n > DFLASH_SETTLE_MAX) return fail(DFLASH_E_ARG, std::string(who) + ": 1 to 1024 rows a call");
  if (pos < 0) return fail(DFLASH_E_ARG, std::string(who) + ": a negative position");
  if (!rows || ((uintptr_t)rows & 7)) return fail(DFLASH_E_ARG, std::string(who) + ": null or misaligned rows");
  return DFLASH_OK;
}

int dflash_settle(dflash_t *d, int32_t seq, int64_t pos, const float *taps, int32_t n, void *stream) {
  if (int e = context_call_checks(d, seq, pos, taps, n, "settle")) return e;
  return add_context(d, seq, pos, taps, n, false, (cudaStream_t)stream);
}

int dflash_queue(dflash_t *d, int32_t seq, int64_t pos, const float *taps, int32_t n, void *stream) {
  if (int e = context_call_checks(d, seq, pos, taps, n, "queue")) return e;
  return add_context(d, seq, pos, taps, n, true, (cudaStream_t)stream);
}

int dflash_settle_pending(dflash_t *d, int32_t seq, void *stream) {
  if (!d || seq < 0 || seq >= d->max_batch) return fail(DFLASH_E_ARG, "settle_pending: bad sequence");
  Seq &s = d->seqs[seq];
  if (s.pcount == 0) return DFLASH_OK;
  Seg segs[2];
  const int ns = pending_segs(s, s.pcount, (size_t)d->g.taps * d->g.hidden, segs);
  s.pcount = 0;
  s.phead = 0;
  return settle_rows(d, seq, segs, ns, (cudaStream_t)stream);
}

int dflash_truncate(dflash_t *d, int32_t seq, int64_t pos) {
  if (!d || seq < 0 || seq >= d->max_batch || pos < 0) return fail(DFLASH_E_ARG, "truncate: bad sequence or position");
  truncate_seq(d, d->seqs[seq], pos);
  return DFLASH_OK;
}

int dflash_push_rows(dflash_t *d, int32_t seq, int64_t pos, int32_t n, const float *const *k, const float *const *v,
                     void *stream) {
  if (int e = context_call_checks(d, seq, pos, k, n, "push_rows")) return e;
  const dflash_geometry &g = d->g;
  if (!v) return fail(DFLASH_E_ARG, "push_rows: null rows");
  for (int l = 0; l < g.layers; ++l)
    if (!k[l] || !v[l] || ((uintptr_t)k[l] & 7) || ((uintptr_t)v[l] & 7))
      return fail(DFLASH_E_ARG, "push_rows: a null or misaligned layer's rows");
  cudaStream_t st = (cudaStream_t)stream;
  Seq &s = d->seqs[seq];
  Seq after = s;
  restart_or_truncate(d, after, pos);
  if (!fits(d, pos - after.first + n)) return fail(DFLASH_E_CAPACITY, "push_rows: context rows do not fit the cache");
  s = after;
  // the waiting rows before pos settle first, then the rows are the context's next ones
  if (int e = dflash_settle_pending(d, seq, stream)) return e;
  dfl::CtxWrite W{};
  cache_rows(d, seq, W);
  for (int l = 0; l < g.layers; ++l) {
    W.k[l] = k[l];
    W.v[l] = v[l];
  }
  DF_CUDA(dfl::ctx_planes(W, g.layers, n, g.kv_heads, g.head_dim, d->planes, (float)g.eps, d->inv.data(),
                          s.first + s.len, s.len, false, st));
  s.len += n;
  window_trim(d, s);
  return DFLASH_OK;
}

}  // extern "C"

// The block pass. With `stage1` set, and when the head GEMM takes whole k-ranges
// (the narrow path over the full head), the head also writes the selector's
// chunk maxima into the drafter's selector scratch, cleared by the pass's last
// norm: *stage1 is then left true, else false.
static int block_pass(dflash_t *d, int32_t batch, const int64_t *anchor_pos, const float *h, int32_t k, int32_t width,
                      float *logits, float *hp, void *stream, bool *stage1) {
  const bool want_stage1 = stage1 && *stage1;
  if (stage1) *stage1 = false;
  if (!d) return fail(DFLASH_E_ARG, "block: null drafter");
  const dflash_geometry &g = d->g;
  const int R = g.block;
  if (batch < 1 || batch > d->max_batch) return fail(DFLASH_E_ARG, "block: batch must be 1..max_batch");
  if (!anchor_pos || !h || !logits || !hp || ((uintptr_t)h & 15)) return fail(DFLASH_E_ARG, "block: null or misaligned pointer");
  if (k < 1 || k >= R) return fail(DFLASH_E_ARG, "block: k must be 1..block-1");
  if (width < g.selector_top || width > g.vocab) return fail(DFLASH_E_ARG, "block: width must be selector_top..vocab");
  for (int b = 0; b < batch; ++b) {
    if (anchor_pos[b] < 0) return fail(DFLASH_E_ARG, "block: a negative anchor position");
    if (d->seqs[b].pcount > 0)
      return fail(DFLASH_E_ARG, "block: rows of sequence " + std::to_string(b) + " wait to be settled");
  }
  if (!encode_maps(d)) return fail(DFLASH_E_CUDA, "block: the driver could not encode the context caches' tensor maps");
  cudaStream_t st = (cudaStream_t)stream;
  const int T = batch * R;
  const int hs = g.hidden, nh = g.heads, kv = g.kv_heads, hd = g.head_dim, ffn = g.intermediate;
  const int qd = nh * hd, kvd = kv * hd, kn = g.conv_kernel, gs = g.conv_group;
  const int pr = 2 * kn * (hs / gs);
  const float eps = (float)g.eps;
  const float scale = std::pow((float)hd, -0.5f);
  const int grp = g.quant_group;
  const int sms = d->num_sms;
  DF_CUDA(cudaMemcpyAsync(d->h, h, (size_t)T * hs * sizeof(float), cudaMemcpyDeviceToDevice, st));
  std::vector<dfl::AttnSeq> seqs(batch);
  auto ranges = [&](int l, int W) {
    // the layer's context range (src/cortiq_engine/dflash.rs, Drafter::block): the
    // layer holds positions first + dropped .. first + len; a ring's rows start
    // at (position - first) % C, and a range (fewer than W rows) runs on into the
    // rows past the ring that repeat its first ones
    for (int b = 0; b < batch; ++b) {
      const Seq &s = d->seqs[b];
      const int64_t a = anchor_pos[b];
      const int64_t base = s.first + s.dropped[l];
      const int64_t hi = std::max(std::min(a, s.first + s.len), base);
      int64_t lo = base;
      if (W > 0) lo = std::min(std::max(std::max<int64_t>(a + 1 - W, 0), base), hi);
      seqs[b].kmap = d->kmap[(size_t)b * g.layers + l];
      seqs[b].vmap = d->vmap[(size_t)b * g.layers + l];
      seqs[b].row0 = d->ring[l] ? (lo - s.first) % d->ring[l] : lo - s.first;
      seqs[b].n = (int)(hi - lo);
      seqs[b].lo = lo;
      seqs[b].anchor = a;
    }
  };
  const int Tk = batch * k;
  bool fuse = false;
  unsigned long long *cmax = nullptr;
  int nchunks = 0;

  if (T <= 32) {
    // Up to 32 rows: every GEMM reads token tiles that the kernel before it
    // wrote (norm, convolution, SiLU or the attention merge), which also clears
    // the GEMM's outputs when the GEMM splits its k-range.
    const int tf = dfl::tc_tile_rows(T, false), ti = dfl::tc_tile_rows(T, true);
    auto pack_for = [&](int planes, int tt, int K) { return dfl::PackDst{(uint4 *)d->act, tt, planes, K / 64}; };
    auto zero_for = [&](const dfl::TcJob *jobs, int n, bool split, int rows) {
      dfl::ZeroSet z{};
      if (split) {
        z.count = n;
        z.T = rows;
        for (int j = 0; j < n; ++j) {
          z.y[j] = jobs[j].y;
          z.ldy[j] = jobs[j].ldy;
          z.n[j] = jobs[j].n;
        }
      }
      return z;
    };
    for (int l = 0; l < g.layers; ++l) {
      const dflash_layer_weights &L = d->layers[l];
      const int W = g.windows[l];
      const bool rot = g.no_rope[l] == 0;
      const dfl::TcJob ap{L.attn_proj.data, nullptr, d->d, pr, pr};
      const dfl::TcJob qkv[3] = {{L.q.data, L.q.scales, d->q, qd, qd}, {L.k.data, L.k.scales, d->k, kvd, kvd},
                                 {L.v.data, L.v.scales, d->v, kvd, kvd}};
      const dfl::TcJob oj{L.o.data, L.o.scales, d->o, hs, hs};
      const dfl::TcJob mp{L.mlp_proj.data, nullptr, d->d2, pr, pr};
      const dfl::TcJob gu[2] = {{L.gate.data, L.gate.scales, d->gt, ffn, ffn},
                                {L.up.data, L.up.scales, d->up, ffn, ffn}};
      const dfl::TcJob dn{L.down.data, L.down.scales, d->o, hs, hs};
      // attention: x = norm(h) (for layers after the first, the previous layer's
      // last convolution already did it); d = Pr_attn . f16(x); xc = conv_in(x, d); q, k, v
      if (l == 0)
        DF_CUDA(dfl::rms_pack(d->h, nullptr, nullptr, nullptr, kn, gs, L.in_norm, d->x, T, hs, eps, R, -1, -1,
                              pack_for(1, tf, hs), zero_for(&ap, 1, dfl::tc_splits_f16(&ap, 1, T, hs, sms), T), st));
      DF_CUDA(dfl::tc_gemm_f16_packed(&ap, 1, d->act, tf * 128, T, hs, sms, st));
      DF_CUDA(dfl::conv0_pack(d->x, d->d, L.attn_base, T, hs, kn, gs, R, pack_for(2, ti, hs),
                              zero_for(qkv, 3, dfl::tc_splits_int4(qkv, 3, T, hs, sms), T), st));
      DF_CUDA(dfl::tc_gemm_int4_packed(qkv, 3, grp, d->act, T, hs, sms, st));
      DF_CUDA(dfl::qk_norm_rope(d->q, qd, L.q_norm, nh, d->k, kvd, L.k_norm, d->v, kvd, kv, d->kp, d->vp,
                                d->inv.data(), T, hd, eps, rot, anchor_pos, batch, R, d->planes, st));
      ranges(l, W);
      const dfl::PackDst po = pack_for(2, ti, qd);
      const dfl::ZeroSet zo = zero_for(&oj, 1, dfl::tc_splits_int4(&oj, 1, T, qd, sms), T);
      DF_CUDA(dfl::attention(d->q, d->own_k, d->own_v, seqs.data(), batch, nh, kv, hd, d->planes, R, W, scale,
                             d->part, d->y, sms, &po, &zo, st));
      DF_CUDA(dfl::tc_gemm_int4_packed(&oj, 1, grp, d->act, T, qd, sms, st));
      // h += conv_out(o, d); x = norm(h); the MLP the same way
      DF_CUDA(dfl::rms_pack(d->h, d->o, d->d, L.attn_base, kn, gs, L.post_norm, d->x, T, hs, eps, R, -1, -1,
                            pack_for(1, tf, hs), zero_for(&mp, 1, dfl::tc_splits_f16(&mp, 1, T, hs, sms), T), st));
      DF_CUDA(dfl::tc_gemm_f16_packed(&mp, 1, d->act, tf * 128, T, hs, sms, st));
      DF_CUDA(dfl::conv0_pack(d->x, d->d2, L.mlp_base, T, hs, kn, gs, R, pack_for(2, ti, hs),
                              zero_for(gu, 2, dfl::tc_splits_int4(gu, 2, T, hs, sms), T), st));
      DF_CUDA(dfl::tc_gemm_int4_packed(gu, 2, grp, d->act, T, hs, sms, st));
      DF_CUDA(dfl::silu_pack(d->gt, d->up, T, ffn, pack_for(2, ti, ffn),
                             zero_for(&dn, 1, dfl::tc_splits_int4(&dn, 1, T, ffn, sms), T), st));
      DF_CUDA(dfl::tc_gemm_int4_packed(&dn, 1, grp, d->act, T, ffn, sms, st));
      // h += conv_out(down, d) and the next norm: the next layer's input norm, or the last norm (rows 1..k)
      if (l + 1 < g.layers) {
        const dflash_layer_weights &N = d->layers[l + 1];
        const dfl::TcJob ap2{N.attn_proj.data, nullptr, d->d, pr, pr};
        DF_CUDA(dfl::rms_pack(d->h, d->o, d->d2, L.mlp_base, kn, gs, N.in_norm, d->x, T, hs, eps, R, -1, -1,
                              pack_for(1, tf, hs), zero_for(&ap2, 1, dfl::tc_splits_f16(&ap2, 1, T, hs, sms), T),
                              st));
      } else {
        const dfl::TcJob ends[2] = {{d->w.head.data, d->w.head.scales, logits, width, width},
                                    {d->w.sel.data, nullptr, hp, g.selector_rank, g.selector_rank}};
        const bool split = dfl::tc_splits_int4(&ends[0], 1, Tk, hs, sms) || dfl::tc_splits_f16(&ends[1], 1, Tk, hs, sms);
        dfl::ZeroSet z = zero_for(ends, 2, split, Tk);
        // the selector's chunk maxima and candidate counts, when the head computes the former
        fuse = want_stage1 && dfl::tc_int4_whole(&ends[0], 1, Tk, hs, sms);
        if (fuse) {
          int *cnt;
          dfl::select_stage1(d->sel, Tk, width, &cmax, &cnt, &nchunks);
          z.T = Tk;
          z.y[z.count] = (float *)cmax;
          z.ldy[z.count] = 2 * nchunks;
          z.n[z.count++] = 2 * nchunks;
          z.y[z.count] = (float *)cnt;
          z.ldy[z.count] = 1;
          z.n[z.count++] = 1;
        }
        DF_CUDA(dfl::rms_pack(d->h, d->o, d->d2, L.mlp_base, kn, gs, d->w.norm, nullptr, T, hs, eps, R, 1, k,
                              pack_for(2, dfl::tc_tile_rows(Tk, true), hs), z, st));
      }
    }
    // the head and the selector's projection over rows 1..k (the selector reads the hi plane)
    const int th = dfl::tc_tile_rows(Tk, true);
    const dfl::TcJob hj{d->w.head.data, d->w.head.scales, logits, width, width};
    DF_CUDA(dfl::tc_gemm_int4_packed(&hj, 1, grp, d->act, Tk, hs, sms, st, fuse ? cmax : nullptr, nchunks));
    if (stage1) *stage1 = fuse;
    const dfl::TcJob sj{d->w.sel.data, nullptr, hp, g.selector_rank, g.selector_rank};
    DF_CUDA(dfl::tc_gemm_f16_packed(&sj, 1, d->act, 2 * th * 128, Tk, hs, sms, st));
    return DFLASH_OK;
  }

  for (int l = 0; l < g.layers; ++l) {
    const dflash_layer_weights &L = d->layers[l];
    const int W = g.windows[l];
    const bool rot = g.no_rope[l] == 0;
    // attention: x = norm(h); x, d = conv_in(x); q, k, v
    DF_CUDA(dfl::rmsnorm(d->h, L.in_norm, d->x, T, hs, eps, R, -1, -1, st));
    const dfl::TcJob ap{L.attn_proj.data, nullptr, d->d, pr, pr};
    DF_CUDA(dfl::tc_gemm_f16(&ap, 1, d->x, hs, T, hs, d->act, sms, st));
    DF_CUDA(dfl::conv_stage0(d->x, d->d, L.attn_base, d->xc, T, hs, kn, gs, R, st));
    const dfl::TcJob qkv[3] = {{L.q.data, L.q.scales, d->q, qd, qd}, {L.k.data, L.k.scales, d->k, kvd, kvd},
                               {L.v.data, L.v.scales, d->v, kvd, kvd}};
    DF_CUDA(dfl::tc_gemm_int4(qkv, 3, grp, d->xc, hs, T, hs, d->act, sms, st));
    DF_CUDA(dfl::qk_norm_rope(d->q, qd, L.q_norm, nh, d->k, kvd, L.k_norm, d->v, kvd, kv, d->kp, d->vp,
                              d->inv.data(), T, hd, eps, rot, anchor_pos, batch, R, d->planes, st));
    ranges(l, W);
    DF_CUDA(dfl::attention(d->q, d->own_k, d->own_v, seqs.data(), batch, nh, kv, hd, d->planes, R, W, scale, d->part,
                           d->y, sms, nullptr, nullptr, st));
    const dfl::TcJob oj{L.o.data, L.o.scales, d->o, hs, hs};
    DF_CUDA(dfl::tc_gemm_int4(&oj, 1, grp, d->y, qd, T, qd, d->act, sms, st));
    DF_CUDA(dfl::conv_stage1_residual(d->o, d->d, L.attn_base, d->h, T, hs, kn, gs, R, st));
    // the MLP the same way
    DF_CUDA(dfl::rmsnorm(d->h, L.post_norm, d->x, T, hs, eps, R, -1, -1, st));
    const dfl::TcJob mp{L.mlp_proj.data, nullptr, d->d, pr, pr};
    DF_CUDA(dfl::tc_gemm_f16(&mp, 1, d->x, hs, T, hs, d->act, sms, st));
    DF_CUDA(dfl::conv_stage0(d->x, d->d, L.mlp_base, d->xc, T, hs, kn, gs, R, st));
    const dfl::TcJob gu[2] = {{L.gate.data, L.gate.scales, d->gt, ffn, ffn}, {L.up.data, L.up.scales, d->up, ffn, ffn}};
    DF_CUDA(dfl::tc_gemm_int4(gu, 2, grp, d->xc, hs, T, hs, d->act, sms, st));
    DF_CUDA(dfl::silu_mul(d->gt, d->up, d->gt, (int64_t)T * ffn, st));
    const dfl::TcJob dn{L.down.data, L.down.scales, d->o, hs, hs};
    DF_CUDA(dfl::tc_gemm_int4(&dn, 1, grp, d->gt, ffn, T, ffn, d->act, sms, st));
    DF_CUDA(dfl::conv_stage1_residual(d->o, d->d, L.mlp_base, d->h, T, hs, kn, gs, R, st));
  }
  // the last norm; the head and the selector's projection over rows 1..k
  DF_CUDA(dfl::rmsnorm(d->h, d->w.norm, d->x, T, hs, eps, R, 1, k, st));
  const dfl::TcJob hj{d->w.head.data, d->w.head.scales, logits, width, width};
  DF_CUDA(dfl::tc_gemm_int4(&hj, 1, grp, d->x, hs, Tk, hs, d->act, sms, st));
  const dfl::TcJob sj{d->w.sel.data, nullptr, hp, g.selector_rank, g.selector_rank};
  DF_CUDA(dfl::tc_gemm_f16(&sj, 1, d->x, hs, Tk, hs, d->act, sms, st));
  return DFLASH_OK;
}

extern "C" {

int dflash_block(dflash_t *d, int32_t batch, const int64_t *anchor_pos, const float *h, int32_t k, int32_t width,
                 float *logits, float *hp, void *stream) {
  return block_pass(d, batch, anchor_pos, h, k, width, logits, hp, stream, nullptr);
}

int dflash_draft(dflash_t *d, int32_t batch, const int64_t *anchor_pos, const float *h, int32_t k, int32_t width,
                 const uint32_t *anchor_tok, float *logits, float *hp, uint32_t *chosen, uint32_t *plain,
                 void *stream) {
  if (!d) return fail(DFLASH_E_ARG, "draft: null drafter");
  if (!anchor_tok || !chosen || !plain) return fail(DFLASH_E_ARG, "draft: null pointer");
  bool stage1 = true;
  int rc = block_pass(d, batch, anchor_pos, h, k, width, logits, hp, stream, &stage1);
  if (rc != DFLASH_OK) return rc;
  const dflash_geometry &g = d->g;
  DF_CUDA(dfl::select_tokens(logits, hp, anchor_tok, d->w.pred_book, d->w.succ_book, batch, k, width, g.selector_rank,
                             g.selector_top, g.vocab, d->sel, chosen, plain, d->num_sms, (cudaStream_t)stream,
                             stage1));
  return DFLASH_OK;
}

int dflash_select(dflash_t *d, int32_t batch, const float *logits, const float *hp, const uint32_t *anchor_tok,
                  int32_t k, int32_t width, uint32_t *chosen, uint32_t *plain, void *stream) {
  if (!d) return fail(DFLASH_E_ARG, "select: null drafter");
  const dflash_geometry &g = d->g;
  if (batch < 1 || batch > d->max_batch) return fail(DFLASH_E_ARG, "select: batch must be 1..max_batch");
  if (k < 1 || k >= g.block) return fail(DFLASH_E_ARG, "select: k must be 1..block-1");
  if (width < g.selector_top || width > g.vocab) return fail(DFLASH_E_ARG, "select: width must be selector_top..vocab");
  if (!logits || !hp || !anchor_tok || !chosen || !plain) return fail(DFLASH_E_ARG, "select: null pointer");
  DF_CUDA(dfl::select_tokens(logits, hp, anchor_tok, d->w.pred_book, d->w.succ_book, batch, k, width, g.selector_rank,
                             g.selector_top, g.vocab, d->sel, chosen, plain, d->num_sms, (cudaStream_t)stream));
  return DFLASH_OK;
}

}  // extern "C"

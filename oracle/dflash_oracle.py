"""CPU oracle of the DFlash 2 drafter pass: context settle, block forward, head and selector.

TEST INFRASTRUCTURE ONLY. This module is the slow, plain definition the CUDA
library is checked against. Only ``tests/``, ``__graft_entry__.smoke()`` and the
bench's ``cpu_baseline`` / ``--impl reference`` legs may import or run it; the
product path never does. It shares no code with the CUDA library: it reads the
same synthetic inputs (``dflash_inputs``) and nothing else.

Source followed: the cortiq-engine pages, "src/cortiq_engine/dflash.rs" (the
host drafter: ``rms``, ``Drafter::new`` inv_freq, ``Drafter::rotate``,
``Drafter::settle_rows``, ``Drafter::conv_in`` / ``conv``, ``Drafter::block``,
``Drafter::mlp``, ``Drafter::select_with``, ``top_k``) and, where the card
arm fixes a step the host leaves to its matrix type, "src/gpu_cuda/hyb/dflash.rs"
(``Dev::settle``, ``Dev::block``).

Arithmetic: every value is kept in f64 and every dot product, norm and softmax
is taken in f64. Inputs keep their stored precision (f16 matrices and
codebooks, four-bit codes with f16 scales, f32 norms, base kernels, taps and
embeddings). Readings fixed where the pages leave a step open:

* four-bit matrices: the value of a code is ``(nibble - 8) * scale``, exact
  (interchange format of ``dflash_inputs``); they multiply the activations at
  full precision (the card arm feeds them f16 "planes" of the f32 rows);
* f16 matrices (fc, the kernel projections, the selector's projection)
  multiply the activations rounded to f16, as the card arm does with
  ``to_half`` before its f16 GEMM (``Dev::settle``, ``Dev::block``);
* rotary angle: ``f32(f32(pos) * inv_freq_f32)`` as in ``Drafter::rotate``;
  its cosine and sine are taken in f64;
* the attention scale is the f32 value of ``head_dim^-1/2`` (``Drafter::block``);
* context bookkeeping follows the host drafter: ``Drafter::truncate``,
  ``Drafter::queue_context`` (a gap starts the context over; past the pending
  limit the oldest rows settle in multiples of ``CONTEXT_CHUNK``), ``settle``
  and the window trim at the end of ``Drafter::settle_rows`` (a layer holding
  more than twice its window keeps its last ``window`` rows, ``dropped`` grows
  by the rest); the pending limit is the one the page gives when CUDA is
  active; a layer's context range is ``Drafter::block``'s rule with the base
  ``first + dropped``.

Parity pins: every function here is pinned by a ``-m "not gpu"`` test against
a closed form, the page's worked example, a brute-force evaluation or an
invariant (tests/test_oracle_pins.py). The composition is pinned too: the
block rows the head and the selector's projection read (a closed form on
one-hot matrices), the settle's order (a closed form: the norm after the fc,
the key norm before the rotation), which kernel each stage-1 convolution uses
(linearity in its signal and which projection rows reach it), and the
checker's scores against ``select_with``. No printed end-to-end value exists
on the pages, so the whole pass is otherwise pinned through these parts.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence

import numpy as np

__all__ = [
    "dequant_int4", "int4_matmul", "f16_matmul", "rms", "inv_freq", "rotate", "conv",
    "context_range", "attention", "mlp", "top_k", "select_with", "pending_limit", "recon_error",
    "route_margin", "Oracle",
]

# Context bookkeeping constants of the host drafter (dflash.rs, module constants).
BLOCK_SLACK = 256       # positions past a layer's window still kept for the next anchors
CONTEXT_CHUNK = 64      # the over-limit settle takes a multiple of this many rows
PENDING_ROWS = 512      # rows that may wait unsettled


# ---------------------------------------------------------------- matrices

def dequant_int4(codes: np.ndarray, scales: np.ndarray, group: int) -> np.ndarray:
    """Values of a four-bit matrix: ``(nibble - 8) * scale``, f64 ``[rows][cols]``.

    Low nibble = even column; scale ``[rows][cols/group]`` f16. The product of
    a code in -7..7 and an f16 scale is exact in f32 and in f64.
    """
    rows, half = codes.shape
    cols = 2 * half
    q = np.empty((rows, cols), dtype=np.float64)
    q[:, 0::2] = (codes & 0x0F).astype(np.float64) - 8.0
    q[:, 1::2] = (codes >> 4).astype(np.float64) - 8.0
    s = np.repeat(scales.astype(np.float64), group, axis=1)
    return q * s


def int4_matmul(m, x: np.ndarray, row_lo: int = 0, row_hi: Optional[int] = None) -> np.ndarray:
    """``x @ W[row_lo:row_hi].T`` for a four-bit matrix ``m`` (``dflash_inputs.Int4``), in f64.

    ``x`` is ``[n][cols]``; the matrix is dequantised a slab of rows at a time.
    """
    row_hi = m.rows if row_hi is None else row_hi
    x = np.asarray(x, dtype=np.float64)
    out = np.empty((x.shape[0], row_hi - row_lo), dtype=np.float64)
    per = max(1, (1 << 22) // m.cols)
    for r0 in range(row_lo, row_hi, per):
        r1 = min(row_hi, r0 + per)
        w = dequant_int4(m.codes[r0:r1], m.scales[r0:r1], m.group)
        out[:, r0 - row_lo:r1 - row_lo] = x @ w.T
    return out


def f16_matmul(w16: np.ndarray, x: np.ndarray) -> np.ndarray:
    """``f16(x) @ W.T`` for an f16 matrix ``W`` ``[rows][cols]``, products and sums in f64."""
    xh = np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)
    return xh @ w16.astype(np.float64).T


# ---------------------------------------------------------------- norms, rotation

def rms(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """``x * (mean(x^2) + eps)^-1/2 * w`` over each run of ``len(w)`` values (dflash.rs ``rms``)."""
    x = np.asarray(x, dtype=np.float64)
    n = len(w)
    r = x.reshape(-1, n)
    ms = (r * r).sum(axis=1) / n
    s = 1.0 / np.sqrt(ms + eps)
    return (r * s[:, None] * np.asarray(w, dtype=np.float64)[None, :]).reshape(x.shape)


def inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """``f32(theta^(-2i/head_dim))`` for ``i < head_dim/2`` (dflash.rs ``Drafter::new``)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return (theta ** (-(2.0 * i) / head_dim)).astype(np.float32)


def rotate(x: np.ndarray, heads: int, positions: Sequence[int], inv: np.ndarray) -> np.ndarray:
    """Half-split rotation of every head of row r to position ``positions[r]`` (dflash.rs ``Drafter::rotate``).

    ``x`` is ``[rows][heads*head_dim]``. For pair ``(i, i + hd/2)``:
    ``lo' = a cos - b sin``, ``hi' = b cos + a sin`` with the angle the f32
    product ``f32(pos) * inv[i]``.
    """
    x = np.asarray(x, dtype=np.float64)
    rows = x.shape[0]
    half = len(inv)
    hd = 2 * half
    out = x.reshape(rows, heads, hd).copy()
    for r in range(rows):
        ang = (np.float32(positions[r]) * inv).astype(np.float32).astype(np.float64)
        c, s = np.cos(ang), np.sin(ang)
        a = out[r, :, :half].copy()
        b = out[r, :, half:].copy()
        out[r, :, :half] = a * c - b * s
        out[r, :, half:] = b * c + a * s
    return out.reshape(rows, heads * hd)


# ---------------------------------------------------------------- row convolution

def conv(base: np.ndarray, d: np.ndarray, x: np.ndarray, stage: int, kn: int, gs: int) -> np.ndarray:
    """Grouped causal row convolution (dflash.rs ``Drafter::conv``).

    ``y[r][i] = sum_{o < min(kn, r+1)} (base[stage][o][i] + d[r][stage][o][i // gs]) * x[r - o][i]``.
    ``base`` is ``[2][kn][hidden]``; ``d`` is ``[rows][2][kn][groups]`` flattened per row.
    """
    x = np.asarray(x, dtype=np.float64)
    rows, hs = x.shape
    groups = hs // gs
    d = np.asarray(d, dtype=np.float64).reshape(rows, 2, kn, groups)
    base = np.asarray(base, dtype=np.float64).reshape(2, kn, hs)
    y = np.zeros((rows, hs), dtype=np.float64)
    for r in range(rows):
        for o in range(min(kn, r + 1)):
            k = base[stage, o] + np.repeat(d[r, stage, o], gs)
            y[r] += k * x[r - o]
    return y


# ---------------------------------------------------------------- attention

def pending_limit(g) -> int:
    """Rows that may wait unsettled (dflash.rs ``Drafter::queue_context``, the CUDA arm's limit):
    as many as the widest window reads plus ``BLOCK_SLACK`` when every layer is windowed, else
    ``PENDING_ROWS``; never fewer than ``PENDING_ROWS``."""
    if all(g.window_of(l) > 0 for l in range(g.layers)):
        return max(PENDING_ROWS, max(g.window_of(l) for l in range(g.layers)) + BLOCK_SLACK)
    return PENDING_ROWS


def context_range(first: int, length: int, anchor_pos: int, window: int, dropped: int = 0):
    """Context positions ``[lo, hi)`` a layer's block reads (dflash.rs ``Drafter::block``): the
    layer holds ``first + dropped .. first + length``."""
    base = first + dropped
    hi = max(min(anchor_pos, first + length), base)
    if window > 0:
        lo = min(max(max(anchor_pos + 1 - window, 0), base), hi)
    else:
        lo = base
    return lo, hi


def attention(q, k, v, ctx_k, ctx_v, lo: int, anchor_pos: int, window: int, heads: int,
              kv_heads: int, head_dim: int, scale: float) -> np.ndarray:
    """Non-causal grouped-query attention of the block rows (dflash.rs ``Drafter::block``).

    Query head h reads KV head ``h // (heads/kv_heads)``. Row r's keys are the
    context rows ``ctx_k`` (positions ``lo ..``), those before position
    ``anchor_pos + r + 1 - window`` masked when ``window > 0``, then all block
    rows. Scores are scaled by ``scale``; softmax subtracts the row maximum.
    ``ctx_k``/``ctx_v`` are ``[n][kv_heads][head_dim]``; q ``[rows][heads*hd]``,
    k, v ``[rows][kv_heads*hd]``. Returns y ``[rows][heads*hd]``.
    """
    rows = q.shape[0]
    n = ctx_k.shape[0]
    rep = heads // kv_heads
    q = np.asarray(q, np.float64).reshape(rows, heads, head_dim)
    k = np.asarray(k, np.float64).reshape(rows, kv_heads, head_dim)
    v = np.asarray(v, np.float64).reshape(rows, kv_heads, head_dim)
    ck = np.asarray(ctx_k, np.float64)
    cv = np.asarray(ctx_v, np.float64)
    y = np.zeros((rows, heads, head_dim), dtype=np.float64)
    for h in range(heads):
        g = h // rep
        keys = np.concatenate([ck[:, g, :], k[:, g, :]], axis=0)      # [n + rows][hd]
        vals = np.concatenate([cv[:, g, :], v[:, g, :]], axis=0)
        s = (q[:, h, :] @ keys.T) * scale                               # [rows][n + rows]
        if window > 0:
            for r in range(rows):
                start = max(anchor_pos + r + 1 - window, 0)
                s[r, :min(max(start - lo, 0), n)] = -np.inf
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        y[:, h, :] = p @ vals
    return y.reshape(rows, heads * head_dim)


def mlp(L: dict, x: np.ndarray) -> np.ndarray:
    """``down . (silu(gate . x) * (up . x))``, ``silu(a) = a / (1 + exp(-a))`` (dflash.rs ``Drafter::mlp``)."""
    a = int4_matmul(L["gate"], x)
    u = int4_matmul(L["up"], x)
    m = a / (1.0 + np.exp(-a)) * u
    return int4_matmul(L["down"], m)


# ---------------------------------------------------------------- selector

def top_k(x: np.ndarray, k: int):
    """The ``k`` largest values with their indices, largest first; among equal values the lower index first (dflash.rs ``top_k``)."""
    x = np.asarray(x)
    order = np.argsort(-x, kind="stable")[:k]
    return [(x[i], int(i)) for i in order]


def select_with(hp: np.ndarray, logits: np.ndarray, anchor: int, pred_book: np.ndarray,
                succ_book: np.ndarray, top: int):
    """The selector's in-order re-score (dflash.rs ``Drafter::select_with``).

    Row j: candidates = ``top_k(logits[j], top)``; ``pc = P[prev] * hp[j]``;
    score = logit + ``pc . C[cand]``; the first strictly greater score wins,
    starting from ``(-inf, cand[0])``; ``prev`` starts at the anchor token.
    Returns ``(chosen, plain)``; ``plain[j]`` is row j's own top token.
    """
    n = logits.shape[0]
    prev = int(anchor)
    chosen, plain = [], []
    for j in range(n):
        cand = top_k(logits[j], top)
        plain.append(cand[0][1])
        pc = pred_book[prev].astype(np.float64) * np.asarray(hp[j], np.float64)
        best_s, best_t = -np.inf, cand[0][1]
        for unary, tok in cand:
            s = float(unary) + float(pc @ succ_book[tok].astype(np.float64))
            if s > best_s:
                best_s, best_t = s, tok
        prev = best_t
        chosen.append(prev)
    return chosen, plain


# ---------------------------------------------------------------- router

def recon_error(unit: np.ndarray, mean: np.ndarray, basis: np.ndarray) -> float:
    """How badly a subspace holds a row: the squared length of what is left of ``unit - mean``
    after taking away its projection on the basis rows, ``d - B^T (B d)`` (the basis rows of a
    fitted descriptor are orthonormal). The pages call ``router::recon_error`` without
    printing it; this is the plain reading of a reconstruction error."""
    d = np.asarray(unit, np.float64) - np.asarray(mean, np.float64)
    B = np.asarray(basis, np.float64).reshape(-1, d.shape[0])
    r = d - B.T @ (B @ d)
    return float(r @ r)


def route_margin(row: np.ndarray, block_mean, block_basis, chain_mean, chain_basis) -> float:
    """``Route::margin`` (dflash.rs): the row scaled to unit length (its norm at least 1e-12),
    then the chain subspace's reconstruction error minus the block subspace's; above zero
    the round is the block's. Means and bases are f16 ``[hidden]``, ``[rank][hidden]``."""
    row = np.asarray(row, np.float64)
    unit = row / max(float(np.sqrt(row @ row)), 1e-12)
    return recon_error(unit, chain_mean, chain_basis) - recon_error(unit, block_mean, block_basis)


def select_scores(hp: np.ndarray, logits: np.ndarray, prev_tokens: Sequence[int], pred_book, succ_book, top: int):
    """Every candidate's score of each row given that row's predecessor (for near-tie checks)."""
    out = []
    for j in range(logits.shape[0]):
        cand = top_k(logits[j], top)
        pc = pred_book[int(prev_tokens[j])].astype(np.float64) * np.asarray(hp[j], np.float64)
        out.append([(tok, float(u) + float(pc @ succ_book[tok].astype(np.float64))) for u, tok in cand])
    return out


# ---------------------------------------------------------------- the drafter

class Oracle:
    """One sequence of the drafter: weights, the per-layer context and the pass.

    ``w`` is ``dflash_inputs.make_weights``' dict; ``g`` its ``Geometry``.
    """

    def __init__(self, g, w: dict):
        self.g = g
        self.w = w
        self.inv = inv_freq(g.head_dim, g.rope_theta)
        self.first = 0
        self.len = 0
        self.dropped = [0] * g.layers           # per layer: rows let go by the window trim
        self.pending: List[np.ndarray] = []     # tap rows waiting to be settled, from first + len on
        kvd = (0, g.kv_heads, g.head_dim)
        self.ctx_k: List[np.ndarray] = [np.zeros(kvd) for _ in range(g.layers)]
        self.ctx_v: List[np.ndarray] = [np.zeros(kvd) for _ in range(g.layers)]

    # -- context
    def reset(self, first: int = 0):
        """The context empty, starting at ``first`` (dflash.rs ``Drafter::reset`` starts at 0)."""
        self.first, self.len = first, 0
        self.dropped = [0] * self.g.layers
        self.pending = []
        for i in range(self.g.layers):
            self.ctx_k[i] = self.ctx_k[i][:0]
            self.ctx_v[i] = self.ctx_v[i][:0]

    def settle_rows(self, pos: int, taps: np.ndarray, layers: Optional[Sequence[int]] = None):
        """Keys and values of tap rows at positions ``pos ..`` (dflash.rs ``Drafter::settle_rows``; gpu_cuda ``Dev::settle``).

        ``t = rms(fc . f16(taps), hidden_norm)``; per layer ``k = rms_head(Wk . t, k_norm)``
        rotated to ``pos + r`` when the layer is rotary, ``v = Wv . t``. Returns
        ``(t, [(k, v) per layer])`` with k, v ``[n][kv_heads][head_dim]``.
        """
        g, w = self.g, self.w
        t = f16_matmul(w["fc"], taps)
        t = rms(t, w["hidden_norm"], g.eps)
        out = []
        for li in (range(g.layers) if layers is None else layers):
            L = w["layers"][li]
            k = int4_matmul(L["k"], t)
            v = int4_matmul(L["v"], t)
            k = rms(k, L["k_norm"], g.eps)
            if g.rotary(li):
                k = rotate(k, g.kv_heads, [pos + r for r in range(len(taps))], self.inv)
            out.append((k.reshape(-1, g.kv_heads, g.head_dim), v.reshape(-1, g.kv_heads, g.head_dim)))
        return t, out

    def next_position(self) -> int:
        """The position the next context row belongs to (dflash.rs ``Drafter::next_position``)."""
        return self.first + self.len + len(self.pending)

    def truncate(self, pos: int):
        """Forget the context from position ``pos`` on (dflash.rs ``Drafter::truncate``): waiting rows
        past it, settled rows at or past it; a layer that let rows go keeps ``dropped <= len``."""
        held = self.first + self.len
        self.pending = self.pending[:max(pos - held, 0)]
        keep = min(max(pos - self.first, 0), self.len)
        for li in range(self.g.layers):
            rows = max(keep - self.dropped[li], 0)
            self.ctx_k[li] = self.ctx_k[li][:rows]
            self.ctx_v[li] = self.ctx_v[li][:rows]
            self.dropped[li] = min(self.dropped[li], keep)
        self.len = keep

    def _append(self, pos: int, rows):
        """Rows of positions ``pos ..`` (= first + len) into every layer's context, then the window
        trim (the end of dflash.rs ``Drafter::settle_rows``). ``rows`` is tap rows ``[n][tw]`` or,
        for imported rows, a list of per-layer ``(k, v)`` ``[n][kv_heads][head_dim]``."""
        if isinstance(rows, np.ndarray):
            if len(rows) == 0:
                return
            _, kv = self.settle_rows(pos, rows)
        else:
            kv = rows
        n = len(kv[0][0])
        for li, (k, v) in enumerate(kv):
            self.ctx_k[li] = np.concatenate([self.ctx_k[li], np.asarray(k, np.float64)], axis=0)
            self.ctx_v[li] = np.concatenate([self.ctx_v[li], np.asarray(v, np.float64)], axis=0)
        self.len += n
        for li in range(self.g.layers):
            w, held = self.g.window_of(li), self.len - self.dropped[li]
            if w > 0 and held > 2 * w:
                cut = held - w
                self.ctx_k[li] = self.ctx_k[li][cut:]
                self.ctx_v[li] = self.ctx_v[li][cut:]
                self.dropped[li] += cut

    def _restart_or_truncate(self, pos: int):
        # a gap starts the context over; a held position replaces what follows
        if pos > self.next_position() or pos < self.first:
            self.truncate(0)
            self.first = pos
        else:
            self.truncate(pos)

    def queue(self, pos: int, taps: np.ndarray):
        """Tap rows of positions ``pos ..`` wait to become context (dflash.rs ``Drafter::queue_context``);
        past ``pending_limit`` the oldest settle at once, a multiple of ``CONTEXT_CHUNK`` rows."""
        self._restart_or_truncate(pos)
        self.pending.extend(np.asarray(taps))
        held = len(self.pending)
        limit = pending_limit(self.g)
        if held > limit:
            over = min(-(-(held - limit) // CONTEXT_CHUNK) * CONTEXT_CHUNK, held)
            rows = np.stack(self.pending[:over])
            self.pending = self.pending[over:]
            self._append(self.first + self.len, rows)

    def settle_pending(self):
        """Every waiting row becomes context (dflash.rs ``Drafter::settle``)."""
        if self.pending:
            rows = np.stack(self.pending)
            self.pending = []
            self._append(self.first + self.len, rows)

    def settle(self, pos: int, taps: np.ndarray):
        """Add tap rows of positions ``pos ..`` to the context (dflash.rs ``Drafter::push_context``):
        queue them, then settle every waiting row. Rows at held positions replace them and what
        follows; a gap starts the context over."""
        self.queue(pos, taps)
        self.settle_pending()

    def push_rows(self, pos: int, kv):
        """Keys and values made elsewhere (per layer ``(k, v)`` ``[n][kv_heads][head_dim]``, keys
        already normed and rotated) as the context rows of positions ``pos ..``: the bookkeeping
        of a settle at ``pos`` (gap, truncate, window trim), the rows taken as given (the
        card arm's ``Dev::push_rows`` import, for every layer at once)."""
        self._restart_or_truncate(pos)
        self.settle_pending()
        self._append(self.first + self.len, kv)

    # -- block
    def block(self, anchor_pos: int, h: np.ndarray, trace: Optional[Dict] = None) -> np.ndarray:
        """The block forward over ``h`` (rows ``[anchor, MASK, ...]`` at ``anchor_pos ..``) (dflash.rs ``Drafter::block``).

        Returns every row after the last norm, f64 ``[block][hidden]``.
        """
        g, w = self.g, self.w
        hs, hd, nh, kv, R = g.hidden, g.head_dim, g.heads, g.kv_heads, g.block
        kn, gs = g.conv_kernel, g.conv_group
        scale = float(np.float32(hd) ** np.float32(-0.5))
        h = np.asarray(h, dtype=np.float64).copy()
        pos = [anchor_pos + r for r in range(R)]
        for li, L in enumerate(w["layers"]):
            win = g.window_of(li)
            assert not self.pending, "rows wait to become context (settle_pending)"
            base = self.first + self.dropped[li]
            lo, hi = context_range(self.first, self.len, anchor_pos, win, self.dropped[li])
            ck = self.ctx_k[li][lo - base:hi - base]
            cv = self.ctx_v[li][lo - base:hi - base]
            # attention sub-layer: x = norm(h); x, d = conv_in(x); q, k, v
            x = rms(h, L["in_norm"], g.eps)
            ad = f16_matmul(L["attn_proj"], x)
            xc = conv(L["attn_base"], ad, x, 0, kn, gs)
            q = int4_matmul(L["q"], xc)
            k = int4_matmul(L["k"], xc)
            v = int4_matmul(L["v"], xc)
            q = rms(q, L["q_norm"], g.eps)
            k = rms(k, L["k_norm"], g.eps)
            if g.rotary(li):
                q = rotate(q, nh, pos, self.inv)
                k = rotate(k, kv, pos, self.inv)
            y = attention(q, k, v, ck, cv, lo, anchor_pos, win, nh, kv, hd, scale)
            o = int4_matmul(L["o"], y)
            h = h + conv(L["attn_base"], ad, o, 1, kn, gs)
            # the MLP the same way
            x2 = rms(h, L["post_norm"], g.eps)
            md = f16_matmul(L["mlp_proj"], x2)
            xc2 = conv(L["mlp_base"], md, x2, 0, kn, gs)
            dn = mlp(L, xc2)
            h = h + conv(L["mlp_base"], md, dn, 1, kn, gs)
            if trace is not None:
                trace.setdefault("layers", []).append(dict(
                    x=x, ad=ad, xc=xc, q=q, k=k, v=v, y=y, o=o, x2=x2, md=md, xc2=xc2, dn=dn, h=h.copy(),
                    lo=lo, hi=hi))
        return rms(h, w["norm"], g.eps)

    # -- head and selector
    def head_logits(self, hn: np.ndarray, k: int, width: int) -> np.ndarray:
        """Logits of block rows ``1 ..= k`` over the head's first ``width`` rows (gpu_cuda ``Dev::block``)."""
        return int4_matmul(self.w["head"], hn[1:k + 1], 0, width)

    def selector_projection(self, hn: np.ndarray, k: int) -> np.ndarray:
        """``hp = S . f16(hn)`` of block rows ``1 ..= k`` (gpu_cuda ``Dev::block``, the selector GEMM)."""
        return f16_matmul(self.w["sel"], hn[1:k + 1])

    def select(self, hp: np.ndarray, logits: np.ndarray, anchor: int):
        return select_with(hp, logits, anchor, self.w["pred_book"], self.w["succ_book"], self.g.selector_top)

    def draft(self, anchor_pos: int, h: np.ndarray, anchor: int, k: Optional[int] = None,
              width: Optional[int] = None, trace: Optional[Dict] = None):
        """Block, head, selector projection and selection: ``(hn, logits, hp, chosen, plain)``."""
        g = self.g
        k = g.block - 1 if k is None else k
        width = g.vocab if width is None else width
        hn = self.block(anchor_pos, h, trace)
        logits = self.head_logits(hn, k, width)
        hp = self.selector_projection(hn, k)
        chosen, plain = self.select(hp, logits, anchor)
        return hn, logits, hp, chosen, plain

"""The drafter on one GPU through the C ABI, with PyTorch holding the device memory.

``Drafter`` uploads a weight set (the dict of ``dflash_inputs.make_weights``),
packs its matrices with the library's own packers, allocates the per-sequence
context caches and the workspace, and forwards settle / block / select to
libdflash.so on the current CUDA stream. All compute is in the library.
"""
from __future__ import annotations

import ctypes as C
from typing import List, Optional, Sequence

import numpy as np
import torch

from . import _lib as L


def geometry_struct(g) -> L.Geometry:
    s = L.Geometry()
    for f in ("hidden", "intermediate", "layers", "heads", "kv_heads", "head_dim", "vocab", "block",
              "mask_token", "conv_group", "conv_kernel", "selector_rank", "selector_top", "taps", "quant_group"):
        setattr(s, f, int(getattr(g, f)))
    for i in range(g.layers):
        s.windows[i] = int(g.windows[i])
        s.no_rope[i] = 1 if i in g.no_rope else 0
    s.rope_theta = float(g.rope_theta)
    s.eps = float(g.eps)
    return s


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


class Drafter:
    """``cache_format``: "planes" (two f16 planes an element, about 21 bits) or "f16" (one f16).
    ``rings``: None (linear caches of ``ctx_cap`` rows), "window" (every windowed layer a ring
    of twice its window rows) or a list of ring rows per layer (0 = linear)."""

    def __init__(self, g, weights: dict, max_batch: int = 1, ctx_cap: int = 4096, device: str = "cuda",
                 cache_format: str = "planes", rings=None):
        self.g = g
        self.dev = torch.device(device)
        self.max_batch = max_batch
        self.ctx_cap = ctx_cap
        self.cache = L.CacheConfig()
        self.cache.format = {"planes": L.KV_PLANES, "f16": L.KV_F16}[cache_format]
        self.planes = 2 if cache_format == "planes" else 1
        if rings == "window":
            rings = [2 * g.windows[l] for l in range(g.layers)]
        for l, r in enumerate(rings or []):
            self.cache.ring[l] = int(r)
        self.rings = [int(self.cache.ring[l]) for l in range(g.layers)]
        self._pending = {}
        self._keep: List[torch.Tensor] = []
        self.geom = geometry_struct(g)
        st = _stream()
        tmp: List[torch.Tensor] = []

        def keep(t: torch.Tensor) -> int:
            self._keep.append(t)
            return t.data_ptr()

        def vec(a: np.ndarray) -> int:
            return keep(torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(self.dev))

        def int4(m) -> L.Matrix:
            codes = torch.from_numpy(np.ascontiguousarray(m.codes)).to(self.dev)
            scales = torch.from_numpy(np.ascontiguousarray(m.scales).view(np.int16)).to(self.dev)
            tmp.extend([codes, scales])
            nb = L.dflash_int4_packed_bytes(m.rows, m.cols, m.group)
            ns = L.dflash_int4_scale_bytes(m.rows, m.cols, m.group)
            if nb == 0:
                raise ValueError(f"a four-bit matrix [{m.rows}][{m.cols}] g{m.group} the library does not take")
            dst = torch.empty(nb, dtype=torch.uint8, device=self.dev)
            dsc = torch.empty(ns, dtype=torch.uint8, device=self.dev)
            L.dflash_pack_int4(codes.data_ptr(), scales.data_ptr(), m.rows, m.cols, m.group, dst.data_ptr(),
                               dsc.data_ptr(), st)
            return L.Matrix(keep(dst), keep(dsc))

        def f16(a: np.ndarray) -> L.Matrix:
            rows, cols = a.shape
            src = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(self.dev)
            tmp.append(src)
            nb = L.dflash_f16_packed_bytes(rows, cols)
            if nb == 0:
                raise ValueError(f"an f16 matrix [{rows}][{cols}] the library does not take")
            dst = torch.empty(nb, dtype=torch.uint8, device=self.dev)
            L.dflash_pack_f16(src.data_ptr(), rows, cols, dst.data_ptr(), st)
            return L.Matrix(keep(dst), None)

        layers = (L.LayerWeights * g.layers)()
        for i, lw in enumerate(weights["layers"]):
            x = layers[i]
            x.in_norm, x.post_norm = vec(lw["in_norm"]), vec(lw["post_norm"])
            x.q_norm, x.k_norm = vec(lw["q_norm"]), vec(lw["k_norm"])
            x.attn_base, x.mlp_base = vec(lw["attn_base"]), vec(lw["mlp_base"])
            x.attn_proj, x.mlp_proj = f16(lw["attn_proj"]), f16(lw["mlp_proj"])
            for name in ("q", "k", "v", "o", "gate", "up", "down"):
                setattr(x, name, int4(lw[name]))
        self._layers = layers
        w = L.Weights()
        w.fc = f16(weights["fc"])
        w.hidden_norm, w.norm = vec(weights["hidden_norm"]), vec(weights["norm"])
        w.sel = f16(weights["sel"])
        w.pred_book = keep(torch.from_numpy(np.ascontiguousarray(weights["pred_book"]).view(np.int16)).to(self.dev))
        w.succ_book = keep(torch.from_numpy(np.ascontiguousarray(weights["succ_book"]).view(np.int16)).to(self.dev))
        w.head = int4(weights["head"])
        w.layers = C.cast(layers, C.POINTER(L.LayerWeights))
        self._weights = w

        # the caches: per (position, head) the f16 planes hi[hd] then lo[hd], or one
        # f16[hd] (held_kv decodes them); a ring layer's rows past the ring repeat its first ones
        kv, hd = g.kv_heads, g.head_dim
        rows = [L.dflash_cache_rows(self.geom, self.cache, l, ctx_cap) for l in range(g.layers)]
        if not all(rows):
            raise ValueError("a ring needs a windowed layer and at least twice its window rows")
        self.ctx_k = [[torch.zeros(rows[l], kv, self.planes, hd, dtype=torch.float16, device=self.dev)
                       for l in range(g.layers)] for _ in range(max_batch)]
        self.ctx_v = [[torch.zeros(rows[l], kv, self.planes, hd, dtype=torch.float16, device=self.dev)
                       for l in range(g.layers)] for _ in range(max_batch)]
        ks = [t.data_ptr() for row in self.ctx_k for t in row]
        vs = [t.data_ptr() for row in self.ctx_v for t in row]
        self.ws_bytes = L.dflash_workspace_bytes(self.geom, max_batch)
        if self.ws_bytes == 0:
            raise ValueError("the library does not take this geometry / batch")
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.dev)
        torch.cuda.synchronize()
        del tmp
        self.h = L.dflash_create_ex(self.geom, self._weights, max_batch, self.cache, ks, vs, ctx_cap,
                                    self.workspace.data_ptr(), self.ws_bytes)

    # ------------------------------------------------------------------ calls
    def reset(self, seq: int = 0, first: int = 0):
        L.dflash_reset(self.h, seq, first)

    def context(self, seq: int = 0):
        return L.dflash_context(self.h, seq)

    def context_ex(self, seq: int = 0):
        """(first, len, pending rows, dropped rows per layer)."""
        return L.dflash_context_ex(self.h, seq, self.g.layers)

    def held_kv(self, seq: int, layer: int):
        """The K and V rows layer `layer` of `seq` holds (positions first + dropped .. first + len),
        decoded to f32 [rows][kv][hd] (hi + lo of the planes, or the f16 values)."""
        _, n, _, dropped = self.context_ex(seq)
        idx = torch.arange(dropped[layer], n, device=self.dev)
        if self.rings[layer]:
            idx = idx % self.rings[layer]
        k, v = self.ctx_k[seq][layer][idx].float(), self.ctx_v[seq][layer][idx].float()
        return k.sum(dim=2), v.sum(dim=2)

    def context_kv(self, seq: int, layer: int, n: int):
        """The first n cached K and V rows of (seq, layer) of a linear cache with nothing dropped."""
        k, v = self.ctx_k[seq][layer][:n].float(), self.ctx_v[seq][layer][:n].float()
        return k.sum(dim=2), v.sum(dim=2)

    def bind_pending(self, seq: int, rows: Optional[int] = None):
        """A pending buffer for `seq` of `rows` tap rows (default: the pending limit)."""
        rows = L.dflash_pending_limit(self.geom) if rows is None else rows
        buf = torch.empty(rows, self.g.taps * self.g.hidden, dtype=torch.float32, device=self.dev)
        L.dflash_bind_pending(self.h, seq, buf.data_ptr(), rows)
        self._pending[seq] = buf

    def queue(self, seq: int, pos: int, taps: torch.Tensor, chunk: int = L.SETTLE_MAX):
        """Queue tap rows [n][tw] (device f32) at positions pos.., `chunk` rows a call."""
        assert taps.dtype == torch.float32 and taps.is_cuda and taps.is_contiguous()
        st = _stream()
        for i in range(0, taps.shape[0], chunk):
            m = min(chunk, taps.shape[0] - i)
            L.dflash_queue(self.h, seq, pos + i, taps[i:i + m].data_ptr(), m, st)

    def settle_pending(self, seq: int):
        L.dflash_settle_pending(self.h, seq, _stream())

    def truncate(self, seq: int, pos: int):
        L.dflash_truncate(self.h, seq, pos)

    def push_rows(self, seq: int, pos: int, k: Sequence[torch.Tensor], v: Sequence[torch.Tensor]):
        """Every layer's K and V rows of positions pos.. (device f32 [n][kv][hd], keys normed and rotated)."""
        n = k[0].shape[0]
        for t in list(k) + list(v):
            assert t.dtype == torch.float32 and t.is_cuda and t.is_contiguous() and t.shape[0] == n
        L.dflash_push_rows(self.h, seq, pos, n, [t.data_ptr() for t in k], [t.data_ptr() for t in v], _stream())

    def settle(self, seq: int, pos: int, taps: torch.Tensor, chunk: int = L.SETTLE_MAX):
        """Settle tap rows [n][tw] (device f32) at positions pos.., `chunk` (1..1024) rows a call."""
        assert taps.dtype == torch.float32 and taps.is_cuda and taps.is_contiguous()
        assert 1 <= chunk <= L.SETTLE_MAX
        n = taps.shape[0]
        st = _stream()
        for i in range(0, n, chunk):
            m = min(chunk, n - i)
            L.dflash_settle(self.h, seq, pos + i, taps[i:i + m].data_ptr(), m, st)

    def block(self, anchor_pos: Sequence[int], h: torch.Tensor, k: Optional[int] = None, width: Optional[int] = None,
              out: Optional[tuple] = None):
        g = self.g
        batch = len(anchor_pos)
        k = g.block - 1 if k is None else k
        width = g.vocab if width is None else width
        assert h.dtype == torch.float32 and h.is_cuda and h.is_contiguous() and h.numel() == batch * g.block * g.hidden
        if out is None:
            logits = torch.empty(batch, k, width, dtype=torch.float32, device=self.dev)
            hp = torch.empty(batch, k, g.selector_rank, dtype=torch.float32, device=self.dev)
        else:
            logits, hp = out
        L.dflash_block(self.h, batch, anchor_pos, h.data_ptr(), k, width, logits.data_ptr(), hp.data_ptr(), _stream())
        return logits, hp

    def select(self, logits: torch.Tensor, hp: torch.Tensor, anchor_tok: torch.Tensor, out: Optional[tuple] = None):
        batch, k, width = logits.shape
        assert anchor_tok.dtype == torch.int32 and anchor_tok.is_cuda and anchor_tok.numel() == batch
        if out is None:
            chosen = torch.empty(batch, k, dtype=torch.int32, device=self.dev)
            plain = torch.empty(batch, k, dtype=torch.int32, device=self.dev)
        else:
            chosen, plain = out
        L.dflash_select(self.h, batch, logits.data_ptr(), hp.data_ptr(), anchor_tok.data_ptr(), k, width,
                        chosen.data_ptr(), plain.data_ptr(), _stream())
        return chosen, plain

    def draft(self, anchor_pos: Sequence[int], h: torch.Tensor, anchor_tok: torch.Tensor, k: Optional[int] = None,
              width: Optional[int] = None, out: Optional[tuple] = None):
        """block() then select() in one call (dflash_draft): (logits, hp, chosen, plain)."""
        g = self.g
        batch = len(anchor_pos)
        k = g.block - 1 if k is None else k
        width = g.vocab if width is None else width
        assert h.dtype == torch.float32 and h.is_cuda and h.is_contiguous() and h.numel() == batch * g.block * g.hidden
        assert anchor_tok.dtype == torch.int32 and anchor_tok.is_cuda and anchor_tok.numel() == batch
        if out is None:
            logits = torch.empty(batch, k, width, dtype=torch.float32, device=self.dev)
            hp = torch.empty(batch, k, g.selector_rank, dtype=torch.float32, device=self.dev)
            chosen = torch.empty(batch, k, dtype=torch.int32, device=self.dev)
            plain = torch.empty(batch, k, dtype=torch.int32, device=self.dev)
        else:
            logits, hp, chosen, plain = out
        L.dflash_draft(self.h, batch, anchor_pos, h.data_ptr(), k, width, anchor_tok.data_ptr(), logits.data_ptr(),
                       hp.data_ptr(), chosen.data_ptr(), plain.data_ptr(), _stream())
        return logits, hp, chosen, plain

    def close(self):
        if getattr(self, "h", None):
            L.dflash_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def dequant_int4(m, device="cuda") -> np.ndarray:
    """The library's dequantisation of a four-bit matrix (packed on the GPU), f32 [rows][cols]."""
    dev = torch.device(device)
    st = _stream()
    codes = torch.from_numpy(np.ascontiguousarray(m.codes)).to(dev)
    scales = torch.from_numpy(np.ascontiguousarray(m.scales).view(np.int16)).to(dev)
    dst = torch.empty(L.dflash_int4_packed_bytes(m.rows, m.cols, m.group), dtype=torch.uint8, device=dev)
    dsc = torch.empty(L.dflash_int4_scale_bytes(m.rows, m.cols, m.group), dtype=torch.uint8, device=dev)
    out = torch.empty(m.rows, m.cols, dtype=torch.float32, device=dev)
    L.dflash_pack_int4(codes.data_ptr(), scales.data_ptr(), m.rows, m.cols, m.group, dst.data_ptr(), dsc.data_ptr(), st)
    L.dflash_dequant_int4(dst.data_ptr(), dsc.data_ptr(), m.rows, m.cols, m.group, out.data_ptr(), st)
    torch.cuda.synchronize()
    return out.cpu().numpy()


class PackedMatrix:
    """A matrix packed on the GPU by the library (four-bit ``Int4`` or an f16 array)."""

    def __init__(self, m, device="cuda"):
        dev = torch.device(device)
        st = _stream()
        if isinstance(m, np.ndarray):
            self.kind, self.rows, self.cols, self.group = 16, m.shape[0], m.shape[1], 64
            src = torch.from_numpy(np.ascontiguousarray(m).view(np.int16)).to(dev)
            self.data = torch.empty(L.dflash_f16_packed_bytes(self.rows, self.cols), dtype=torch.uint8, device=dev)
            L.dflash_pack_f16(src.data_ptr(), self.rows, self.cols, self.data.data_ptr(), st)
            self.scales = None
            self.mat = L.Matrix(self.data.data_ptr(), None)
        else:
            self.kind, self.rows, self.cols, self.group = 4, m.rows, m.cols, m.group
            codes = torch.from_numpy(np.ascontiguousarray(m.codes)).to(dev)
            scales = torch.from_numpy(np.ascontiguousarray(m.scales).view(np.int16)).to(dev)
            self.data = torch.empty(L.dflash_int4_packed_bytes(m.rows, m.cols, m.group), dtype=torch.uint8, device=dev)
            self.scales = torch.empty(L.dflash_int4_scale_bytes(m.rows, m.cols, m.group), dtype=torch.uint8, device=dev)
            L.dflash_pack_int4(codes.data_ptr(), scales.data_ptr(), m.rows, m.cols, m.group, self.data.data_ptr(),
                               self.scales.data_ptr(), st)
            self.mat = L.Matrix(self.data.data_ptr(), self.scales.data_ptr())
        torch.cuda.synchronize()

    def matmul(self, x: torch.Tensor) -> torch.Tensor:
        """Y [T][rows] = X [T][cols] . W^T on the GPU."""
        assert x.dtype == torch.float32 and x.is_cuda and x.is_contiguous() and x.shape[1] == self.cols
        y = torch.empty(x.shape[0], self.rows, dtype=torch.float32, device=x.device)
        nb = L.dflash_gemm_workspace_bytes(self.kind, self.cols, x.shape[0])
        if getattr(self, "_ws", None) is None or self._ws.numel() < nb:
            self._ws = torch.empty(nb, dtype=torch.uint8, device=x.device)
        L.dflash_gemm(self.mat, self.kind, self.rows, self.cols, self.group, x.data_ptr(), x.shape[0], y.data_ptr(),
                      self._ws.data_ptr(), self._ws.numel(), _stream())
        self._packed_T = x.shape[0]
        return y

    def matmul_packed(self, y: torch.Tensor) -> torch.Tensor:
        """The GEMM kernel alone on the token tiles the last `matmul` packed (up to 32 rows), into y."""
        T = getattr(self, "_packed_T", None)
        if T is None:
            raise RuntimeError("matmul_packed needs a matmul call first (it packs the token tiles)")
        assert y.dtype == torch.float32 and y.is_cuda and y.is_contiguous() and y.shape == (T, self.rows)
        L.dflash_gemm_packed(self.mat, self.kind, self.rows, self.cols, self.group, T, y.data_ptr(),
                             self._ws.data_ptr(), _stream())
        return y


class Router:
    """A router's two fitted subspaces (means f16 [hidden], bases f16 [rank][hidden]) on the GPU;
    ``margin(rows)`` is `Route::margin` of each row (device f32 [n][hidden])."""

    def __init__(self, block_mean, block_basis, chain_mean, chain_basis, device="cuda"):
        dev = torch.device(device)

        def up(a):
            return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float16).view(np.int16)).to(dev)

        self._t = [up(block_mean), up(block_basis), up(chain_mean), up(chain_basis)]
        self.hidden = int(np.asarray(block_mean).shape[0])
        self.r = L.Route(self._t[0].data_ptr(), self._t[1].data_ptr() if self._t[1].numel() else None,
                         self._t[2].data_ptr(), self._t[3].data_ptr() if self._t[3].numel() else None,
                         int(np.asarray(block_basis).reshape(-1, self.hidden).shape[0]),
                         int(np.asarray(chain_basis).reshape(-1, self.hidden).shape[0]))

    def margin(self, rows: torch.Tensor) -> torch.Tensor:
        assert rows.dtype == torch.float32 and rows.is_cuda and rows.is_contiguous() and rows.shape[1] == self.hidden
        out = torch.empty(rows.shape[0], dtype=torch.float32, device=rows.device)
        L.dflash_route_margin(self.r, self.hidden, rows.data_ptr(), rows.shape[0], out.data_ptr(), _stream())
        return out

"""Seeded synthetic inputs for the DFlash 2 drafter pass.

This module is shared by the CPU oracle (``oracle/``), the tests and the bench.
It holds no arithmetic of the drafter pass itself: it only draws weights,
context tap rows and block embeddings from fixed distributions, and stores the
four-bit matrices in their interchange format.

Interchange format of a four-bit matrix ``[rows][cols]`` (group ``g`` along
``cols``, the input dimension):

* ``scales``  f16 ``[rows][cols / g]``: ``f16(max|w| / 7)`` of the group, rounded
  to nearest even; a group of zeros has scale 0;
* ``codes``   u8 ``[rows][cols / 2]``: ``q = clamp(rint(w / scale), -7, 7)``
  stored offset-binary as ``q + 8``, two per byte, the even column in the low
  nibble. A zero-scale group stores ``q = 0``.

The value a code stands for is ``q * scale``. Drawing and quantising the
synthetic weights happens here; reading the codes back is the drafter's job.

Geometry names follow the cortiq-engine ``Geometry`` struct of the DFlash
drafter page (src/cortiq_engine/dflash.rs, ``Geometry``).
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os
import zlib
from typing import Dict, List, Optional

import numpy as np

__all__ = [
    "Geometry", "Workload", "Int4", "WORKLOADS", "workload",
    "quantize_int4", "make_weights", "make_taps", "make_embedding_rows",
    "block_rows", "anchor_token", "weight_shapes",
]


@dataclasses.dataclass(frozen=True)
class Geometry:
    """What a DFlash 2 checkpoint fixes (dflash.rs, ``Geometry``)."""
    hidden: int
    intermediate: int
    layers: int
    heads: int
    kv_heads: int
    head_dim: int
    vocab: int
    block: int
    mask_token: int
    conv_group: int          # channels per group of the row convolution
    conv_kernel: int
    selector_rank: int
    selector_top: int
    taps: int                # tapped target layers joined per context row
    windows: tuple           # per layer, 0 = every position
    no_rope: tuple           # layers without rotary position
    rope_theta: float = 1e6
    eps: float = 1e-6
    quant_group: int = 64    # four-bit group along the input dimension

    @property
    def tap_width(self) -> int:
        return self.taps * self.hidden

    @property
    def groups(self) -> int:
        return self.hidden // self.conv_group

    @property
    def proj_rows(self) -> int:
        """Rows of a kernel projection: two stages x kernel x groups."""
        return 2 * self.conv_kernel * self.groups

    def window_of(self, layer: int) -> int:
        return self.windows[layer]

    def rotary(self, layer: int) -> bool:
        return layer not in self.no_rope


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    geometry: Geometry
    context: int             # positions settled before the block, per sequence
    batch: int = 1           # independent sequences
    seed: int = 0            # weights seed; sequence s uses seed + s for its data
    width: int = 0           # head rows scored (0 = vocab)
    description: str = ""

    @property
    def head_width(self) -> int:
        return self.width or self.geometry.vocab


def _g(**kw) -> Geometry:
    return Geometry(**kw)


_TINY = _g(hidden=256, intermediate=768, layers=1, heads=4, kv_heads=2, head_dim=64,
           vocab=4096, block=16, mask_token=0, conv_group=8, conv_kernel=4,
           selector_rank=16, selector_top=8, taps=2, windows=(0,), no_rope=(),
           quant_group=32)
_Q06 = _g(hidden=1024, intermediate=3072, layers=2, heads=16, kv_heads=8, head_dim=128,
          vocab=151936, block=16, mask_token=0, conv_group=16, conv_kernel=4,
          selector_rank=64, selector_top=16, taps=3, windows=(0, 0), no_rope=(),
          quant_group=64)
_B27 = _g(hidden=5120, intermediate=17408, layers=5, heads=32, kv_heads=8, head_dim=128,
          vocab=151936, block=16, mask_token=0, conv_group=32, conv_kernel=4,
          selector_rank=64, selector_top=16, taps=5, windows=(2048, 2048, 0, 2048, 2048),
          no_rope=(2,), quant_group=64)

WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", _TINY, context=128,
                     description="tiny drafter: 1 layer, hidden 256, 128 context positions"),
    "qwen3-0.6b": Workload("qwen3-0.6b", _Q06, context=1024,
                           description="Qwen3-0.6B-shaped drafter: 2 layers, hidden 1024, 1024 context positions"),
    "27b": Workload("27b", _B27, context=4096,
                    description="27B-target-shaped drafter: 5 layers, hidden 5120, 4096 context positions, "
                                "windows [2048,2048,0,2048,2048], no_rope [2]"),
    "settle-heavy": Workload("settle-heavy", dataclasses.replace(_B27, windows=(0, 0, 0, 0, 0)),
                             context=32768,
                             description="27B-shaped geometry settling 32768 positions, block at 32768 with window 0"),
    "batched": Workload("batched", _Q06, context=8192, batch=32,
                        description="32 independent Qwen3-0.6B-shaped sequences, 8192 context positions each"),
}


def workload(name: str) -> Workload:
    return WORKLOADS[name]


@dataclasses.dataclass
class Int4:
    """A four-bit matrix in the interchange format (module docstring)."""
    codes: np.ndarray        # u8 [rows][cols/2]
    scales: np.ndarray       # f16 [rows][cols/group]
    rows: int
    cols: int
    group: int


# --------------------------------------------------------------------------
# seeded streams: one per (seed, tensor name, chunk), so that chunks can be
# drawn on several threads and the result does not depend on the thread count
# --------------------------------------------------------------------------

_CHUNK = 1 << 22


def _rng(seed: int, name: str, chunk: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([seed, zlib.crc32(name.encode()), chunk]))


_POOL: Optional[_cf.ThreadPoolExecutor] = None


def _pool() -> _cf.ThreadPoolExecutor:
    global _POOL
    if _POOL is None:
        _POOL = _cf.ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1)))
    return _POOL


def _normal_rows(seed: int, name: str, rows: int, cols: int, std: float, fn=None):
    """``[rows][cols]`` f32 draws of N(0, std^2), chunked by rows.

    ``fn`` (optional) maps each f32 chunk to its stored form; the results are
    concatenated along rows.
    """
    per = max(1, _CHUNK // max(cols, 1))
    starts = list(range(0, rows, per))

    def one(ci: int):
        r0 = starts[ci]
        r1 = min(rows, r0 + per)
        x = _rng(seed, name, ci).standard_normal((r1 - r0, cols), dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        return fn(x) if fn is not None else x

    if len(starts) == 1:
        parts = [one(0)]
    else:
        parts = list(_pool().map(one, range(len(starts))))
    if isinstance(parts[0], tuple):
        return tuple(np.concatenate([p[i] for p in parts], axis=0) for i in range(len(parts[0])))
    return np.concatenate(parts, axis=0)


def quantize_int4(w: np.ndarray, group: int):
    """Symmetric four-bit group quantisation of an f32 ``[rows][cols]`` block.

    Returns ``(codes u8 [rows][cols/2], scales f16 [rows][cols/group])`` in the
    interchange format. Input preparation only: it makes the synthetic weights.
    """
    rows, cols = w.shape
    assert cols % group == 0 and cols % 2 == 0 and group % 2 == 0
    g = w.reshape(rows, cols // group, group).astype(np.float32, copy=False)
    amax = np.abs(g).max(axis=2)
    scales = (amax / np.float32(7.0)).astype(np.float16)
    s32 = scales.astype(np.float32)
    safe = np.where(s32 > 0, s32, np.float32(1.0))
    q = np.rint(g / safe[:, :, None])
    q = np.clip(q, -7, 7)
    q[s32 == 0] = 0
    u = (q.astype(np.int16) + 8).astype(np.uint8).reshape(rows, cols)
    codes = (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)
    return codes, scales


def _int4(seed: int, name: str, rows: int, cols: int, group: int) -> Int4:
    std = 1.0 / np.sqrt(cols)
    codes, scales = _normal_rows(seed, name, rows, cols, std, fn=lambda x: quantize_int4(x, group))
    return Int4(codes=codes, scales=scales, rows=rows, cols=cols, group=group)


def _f16(seed: int, name: str, rows: int, cols: int, std: float) -> np.ndarray:
    return _normal_rows(seed, name, rows, cols, std, fn=lambda x: x.astype(np.float16))


def _vec(seed: int, name: str, n: int, mean: float, std: float) -> np.ndarray:
    x = _rng(seed, name, 0).standard_normal(n, dtype=np.float32) * np.float32(std)
    return (x + np.float32(mean)).astype(np.float32)


def _base_kernel(seed: int, name: str, g: Geometry) -> np.ndarray:
    """``[stage][offset][hidden]`` f32: 1 + N(0, 0.05) at offset 0, N(0, 0.05) after."""
    kn, hs = g.conv_kernel, g.hidden
    x = _rng(seed, name, 0).standard_normal((2, kn, hs), dtype=np.float32) * np.float32(0.05)
    x[:, 0, :] += np.float32(1.0)
    return x.astype(np.float32)


def weight_shapes(g: Geometry) -> Dict[str, tuple]:
    """Per-layer matrix shapes ``[rows][cols]`` (dflash.rs, ``Drafter::new``)."""
    qd, kd = g.heads * g.head_dim, g.kv_heads * g.head_dim
    return {"q": (qd, g.hidden), "k": (kd, g.hidden), "v": (kd, g.hidden), "o": (g.hidden, qd),
            "gate": (g.intermediate, g.hidden), "up": (g.intermediate, g.hidden),
            "down": (g.hidden, g.intermediate)}


def make_weights(g: Geometry, seed: int = 0, with_head: bool = True) -> dict:
    """Every tensor of a synthetic drafter (plus the target's head).

    Distributions: four-bit matrices from N(0, 1/fan_in) quantised per the
    interchange format; fc, the kernel projections and the selector's
    projection f16 from N(0, 1/fan_in); codebooks f16 from N(0, rank^-1/2);
    norm weights 1 + N(0, 0.05); base kernels per ``_base_kernel``.
    """
    hs, hd = g.hidden, g.head_dim
    layers = []
    for i in range(g.layers):
        p = f"layers.{i}"
        L = {
            "in_norm": _vec(seed, p + ".input_layernorm", hs, 1.0, 0.05),
            "post_norm": _vec(seed, p + ".post_attention_layernorm", hs, 1.0, 0.05),
            "q_norm": _vec(seed, p + ".q_norm", hd, 1.0, 0.05),
            "k_norm": _vec(seed, p + ".k_norm", hd, 1.0, 0.05),
            "attn_base": _base_kernel(seed, p + ".attention_conv.base_kernel", g),
            "mlp_base": _base_kernel(seed, p + ".mlp_conv.base_kernel", g),
            "attn_proj": _f16(seed, p + ".attention_conv.kernel_projection", g.proj_rows, hs, 1.0 / np.sqrt(hs)),
            "mlp_proj": _f16(seed, p + ".mlp_conv.kernel_projection", g.proj_rows, hs, 1.0 / np.sqrt(hs)),
        }
        for name, (r, c) in weight_shapes(g).items():
            L[name] = _int4(seed, f"{p}.{name}_proj", r, c, g.quant_group)
        layers.append(L)
    w = {
        "layers": layers,
        "fc": _f16(seed, "fc", hs, g.tap_width, 1.0 / np.sqrt(g.tap_width)),
        "hidden_norm": _vec(seed, "hidden_norm", hs, 1.0, 0.05),
        "norm": _vec(seed, "norm", hs, 1.0, 0.05),
        "sel": _f16(seed, "candidate_selector.hidden_projection", g.selector_rank, hs, 1.0 / np.sqrt(hs)),
        "pred_book": _f16(seed, "candidate_selector.predecessor_codebook", g.vocab, g.selector_rank,
                          g.selector_rank ** -0.25),
        "succ_book": _f16(seed, "candidate_selector.successor_codebook", g.vocab, g.selector_rank,
                          g.selector_rank ** -0.25),
    }
    if with_head:
        w["head"] = _int4(seed, "head", g.vocab, hs, g.quant_group)
    return w


def make_taps(g: Geometry, seed: int, n: int, start: int = 0) -> np.ndarray:
    """Context tap rows of positions ``start .. start + n``: f32 ``[n][taps*hidden]`` of N(0, 1).

    Row p is drawn from its own stream, so any slice of positions can be made alone.
    """
    tw = g.tap_width
    out = np.empty((n, tw), dtype=np.float32)
    per = 64
    # positions are drawn in fixed blocks of `per` rows so a slice matches the whole
    firsts = []
    p = start
    while p < start + n:
        nxt = min(start + n, (p // per + 1) * per)
        firsts.append((p, nxt))
        p = nxt

    def blk(a_b):
        a, b = a_b
        base = (a // per) * per
        x = _rng(seed, "taps", a // per).standard_normal((per, tw), dtype=np.float32)
        out[a - start:b - start] = x[a - base:b - base]

    if len(firsts) == 1:
        blk(firsts[0])
    else:
        list(_pool().map(blk, firsts))
    return out


def make_embedding_rows(g: Geometry, seed: int, tokens) -> np.ndarray:
    """The synthetic embedding rows of ``tokens``: f32 ``[len][hidden]`` of N(0, 1), a stream per token."""
    return np.stack([_rng(seed, "embedding", int(t)).standard_normal(g.hidden, dtype=np.float32)
                     for t in tokens]).astype(np.float32)


def anchor_token(g: Geometry, seed: int) -> int:
    """The anchor token of a sequence: uniform over the vocabulary."""
    return int(_rng(seed, "anchor", 0).integers(0, g.vocab))


def block_rows(g: Geometry, seed: int, anchor: int) -> np.ndarray:
    """The block's input rows ``[anchor, MASK, ..., MASK]`` as embeddings: f32 ``[block][hidden]``."""
    emb = make_embedding_rows(g, seed, [anchor, g.mask_token])
    h = np.empty((g.block, g.hidden), dtype=np.float32)
    h[0] = emb[0]
    h[1:] = emb[1]
    return h

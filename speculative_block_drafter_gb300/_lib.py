"""ctypes binding of libdflash.so (include/dflash.h): argument marshalling only.

Every function here forwards to the C entry point of the same name. The
library must have been built (``speculative_block_drafter_gb300.build``); a
missing library raises, there is no other path.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libdflash.so")

MAX_LAYERS = 64
SETTLE_MAX = 1024

E_NAMES = {0: "OK", 1: "E_GEOMETRY", 2: "E_ARG", 3: "E_CAPACITY", 4: "E_CUDA", 5: "E_NOMEM"}


class DflashError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{E_NAMES.get(code, code)}: {msg}")
        self.code = code


class Geometry(C.Structure):
    _fields_ = [
        ("hidden", C.c_int32), ("intermediate", C.c_int32), ("layers", C.c_int32), ("heads", C.c_int32),
        ("kv_heads", C.c_int32), ("head_dim", C.c_int32), ("vocab", C.c_int32), ("block", C.c_int32),
        ("mask_token", C.c_uint32),
        ("conv_group", C.c_int32), ("conv_kernel", C.c_int32), ("selector_rank", C.c_int32),
        ("selector_top", C.c_int32), ("taps", C.c_int32), ("quant_group", C.c_int32),
        ("windows", C.c_int32 * MAX_LAYERS), ("no_rope", C.c_uint8 * MAX_LAYERS),
        ("rope_theta", C.c_double), ("eps", C.c_double),
    ]


KV_PLANES = 0   # two f16 planes an element (4 bytes, about 21 bits)
KV_F16 = 1      # one f16 an element (2 bytes)


class CacheConfig(C.Structure):
    _fields_ = [("format", C.c_int32), ("ring", C.c_int32 * MAX_LAYERS)]


class Route(C.Structure):
    _fields_ = [("block_mean", C.c_void_p), ("block_basis", C.c_void_p), ("chain_mean", C.c_void_p),
                ("chain_basis", C.c_void_p), ("block_rank", C.c_int32), ("chain_rank", C.c_int32)]


class Matrix(C.Structure):
    _fields_ = [("data", C.c_void_p), ("scales", C.c_void_p)]


class LayerWeights(C.Structure):
    _fields_ = [
        ("in_norm", C.c_void_p), ("post_norm", C.c_void_p), ("q_norm", C.c_void_p), ("k_norm", C.c_void_p),
        ("attn_base", C.c_void_p), ("mlp_base", C.c_void_p),
        ("attn_proj", Matrix), ("mlp_proj", Matrix),
        ("q", Matrix), ("k", Matrix), ("v", Matrix), ("o", Matrix), ("gate", Matrix), ("up", Matrix), ("down", Matrix),
    ]


class Weights(C.Structure):
    _fields_ = [
        ("fc", Matrix), ("hidden_norm", C.c_void_p), ("norm", C.c_void_p), ("sel", Matrix),
        ("pred_book", C.c_void_p), ("succ_book", C.c_void_p), ("head", Matrix),
        ("layers", C.POINTER(LayerWeights)),
    ]


_lib = None

EXPORTS = {
    "dflash_int4_packed_bytes": (C.c_size_t, [C.c_int64, C.c_int64, C.c_int32]),
    "dflash_int4_scale_bytes": (C.c_size_t, [C.c_int64, C.c_int64, C.c_int32]),
    "dflash_pack_int4": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int64, C.c_int64, C.c_int32, C.c_void_p,
                                   C.c_void_p, C.c_void_p]),
    "dflash_f16_packed_bytes": (C.c_size_t, [C.c_int64, C.c_int64]),
    "dflash_pack_f16": (C.c_int, [C.c_void_p, C.c_int64, C.c_int64, C.c_void_p, C.c_void_p]),
    "dflash_dequant_int4": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int64, C.c_int64, C.c_int32, C.c_void_p,
                                      C.c_void_p]),
    "dflash_gemm_workspace_bytes": (C.c_size_t, [C.c_int32, C.c_int64, C.c_int32]),
    "dflash_gemm_packed": (C.c_int, [C.POINTER(Matrix), C.c_int32, C.c_int64, C.c_int64, C.c_int32, C.c_int32,
                                     C.c_void_p, C.c_void_p, C.c_void_p]),
    "dflash_gemm": (C.c_int, [C.POINTER(Matrix), C.c_int32, C.c_int64, C.c_int64, C.c_int32, C.c_void_p, C.c_int32,
                              C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]),
    "dflash_device_error": (C.c_int, [C.POINTER(C.c_uint32), C.c_int32]),
    "dflash_workspace_bytes": (C.c_size_t, [C.POINTER(Geometry), C.c_int32]),
    "dflash_create": (C.c_int, [C.POINTER(C.c_void_p), C.POINTER(Geometry), C.POINTER(Weights), C.c_int32,
                                C.POINTER(C.c_void_p), C.POINTER(C.c_void_p), C.c_int64, C.c_void_p, C.c_size_t]),
    "dflash_cache_rows": (C.c_int64, [C.POINTER(Geometry), C.POINTER(CacheConfig), C.c_int32, C.c_int64]),
    "dflash_cache_bytes": (C.c_size_t, [C.POINTER(Geometry), C.POINTER(CacheConfig), C.c_int32, C.c_int64]),
    "dflash_create_ex": (C.c_int, [C.POINTER(C.c_void_p), C.POINTER(Geometry), C.POINTER(Weights), C.c_int32,
                                   C.POINTER(CacheConfig), C.POINTER(C.c_void_p), C.POINTER(C.c_void_p), C.c_int64,
                                   C.c_void_p, C.c_size_t]),
    "dflash_reset": (C.c_int, [C.c_void_p, C.c_int32, C.c_int64]),
    "dflash_context": (C.c_int, [C.c_void_p, C.c_int32, C.POINTER(C.c_int64), C.POINTER(C.c_int64)]),
    "dflash_context_ex": (C.c_int, [C.c_void_p, C.c_int32, C.POINTER(C.c_int64), C.POINTER(C.c_int64),
                                    C.POINTER(C.c_int64), C.POINTER(C.c_int64)]),
    "dflash_settle": (C.c_int, [C.c_void_p, C.c_int32, C.c_int64, C.c_void_p, C.c_int32, C.c_void_p]),
    "dflash_pending_limit": (C.c_int64, [C.POINTER(Geometry)]),
    "dflash_bind_pending": (C.c_int, [C.c_void_p, C.c_int32, C.c_void_p, C.c_int64]),
    "dflash_queue": (C.c_int, [C.c_void_p, C.c_int32, C.c_int64, C.c_void_p, C.c_int32, C.c_void_p]),
    "dflash_settle_pending": (C.c_int, [C.c_void_p, C.c_int32, C.c_void_p]),
    "dflash_truncate": (C.c_int, [C.c_void_p, C.c_int32, C.c_int64]),
    "dflash_push_rows": (C.c_int, [C.c_void_p, C.c_int32, C.c_int64, C.c_int32, C.POINTER(C.c_void_p),
                                   C.POINTER(C.c_void_p), C.c_void_p]),
    "dflash_block": (C.c_int, [C.c_void_p, C.c_int32, C.POINTER(C.c_int64), C.c_void_p, C.c_int32, C.c_int32,
                               C.c_void_p, C.c_void_p, C.c_void_p]),
    "dflash_select": (C.c_int, [C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32,
                                C.c_void_p, C.c_void_p, C.c_void_p]),
    "dflash_draft": (C.c_int, [C.c_void_p, C.c_int32, C.POINTER(C.c_int64), C.c_void_p, C.c_int32, C.c_int32,
                               C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]),
    "dflash_select_static": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32,
                                       C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_void_p,
                                       C.c_void_p, C.c_void_p]),
    "dflash_route_margin": (C.c_int, [C.POINTER(Route), C.c_int32, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p]),
    "dflash_destroy": (None, [C.c_void_p]),
    "dflash_last_error": (C.c_char_p, []),
    "dflash_launch_count": (C.c_uint64, []),
}


def lib():
    """The loaded library; raises if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build the CUDA library first "
                               "(python -m speculative_block_drafter_gb300.build)")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in EXPORTS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(code: int):
    if code != 0:
        raise DflashError(code, lib().dflash_last_error().decode())


def last_error() -> str:
    return lib().dflash_last_error().decode()


# --- one wrapper per entry point (same names, marshalling only) -------------------

def dflash_int4_packed_bytes(rows, cols, group):
    return lib().dflash_int4_packed_bytes(rows, cols, group)


def dflash_int4_scale_bytes(rows, cols, group):
    return lib().dflash_int4_scale_bytes(rows, cols, group)


def dflash_f16_packed_bytes(rows, cols):
    return lib().dflash_f16_packed_bytes(rows, cols)


def dflash_pack_int4(codes, scales, rows, cols, group, dst, dst_scales, stream):
    _check(lib().dflash_pack_int4(codes, scales, rows, cols, group, dst, dst_scales, stream))


def dflash_pack_f16(src, rows, cols, dst, stream):
    _check(lib().dflash_pack_f16(src, rows, cols, dst, stream))


def dflash_dequant_int4(codes, scales, rows, cols, group, out, stream):
    _check(lib().dflash_dequant_int4(codes, scales, rows, cols, group, out, stream))


def dflash_gemm_workspace_bytes(kind, cols, T):
    return lib().dflash_gemm_workspace_bytes(kind, cols, T)


def dflash_gemm(w: Matrix, kind, rows, cols, group, x, T, y, workspace, ws_bytes, stream):
    _check(lib().dflash_gemm(C.byref(w), kind, rows, cols, group, x, T, y, workspace, ws_bytes, stream))


def dflash_gemm_packed(w: Matrix, kind, rows, cols, group, T, y, workspace, stream):
    _check(lib().dflash_gemm_packed(C.byref(w), kind, rows, cols, group, T, y, workspace, stream))


def dflash_device_error(reset: bool = True) -> int:
    v = C.c_uint32()
    _check(lib().dflash_device_error(C.byref(v), 1 if reset else 0))
    return v.value


def dflash_workspace_bytes(geom: Geometry, max_batch: int) -> int:
    return lib().dflash_workspace_bytes(C.byref(geom), max_batch)


def dflash_create(geom: Geometry, weights: Weights, max_batch, ctx_k, ctx_v, ctx_cap, workspace, ws_bytes):
    h = C.c_void_p()
    ks = (C.c_void_p * len(ctx_k))(*ctx_k)
    vs = (C.c_void_p * len(ctx_v))(*ctx_v)
    _check(lib().dflash_create(C.byref(h), C.byref(geom), C.byref(weights), max_batch, ks, vs, ctx_cap,
                               workspace, ws_bytes))
    return h


def dflash_cache_rows(geom: Geometry, cache: CacheConfig, layer, ctx_cap) -> int:
    return lib().dflash_cache_rows(C.byref(geom), C.byref(cache) if cache is not None else None, layer, ctx_cap)


def dflash_cache_bytes(geom: Geometry, cache: CacheConfig, layer, ctx_cap) -> int:
    return lib().dflash_cache_bytes(C.byref(geom), C.byref(cache) if cache is not None else None, layer, ctx_cap)


def dflash_create_ex(geom: Geometry, weights: Weights, max_batch, cache: CacheConfig, ctx_k, ctx_v, ctx_cap, workspace,
                     ws_bytes):
    h = C.c_void_p()
    ks = (C.c_void_p * len(ctx_k))(*ctx_k)
    vs = (C.c_void_p * len(ctx_v))(*ctx_v)
    _check(lib().dflash_create_ex(C.byref(h), C.byref(geom), C.byref(weights), max_batch, C.byref(cache), ks, vs,
                                  ctx_cap, workspace, ws_bytes))
    return h


def dflash_reset(h, seq, first):
    _check(lib().dflash_reset(h, seq, first))


def dflash_context_ex(h, seq, layers):
    """(first, len, pending, dropped per layer)."""
    f, n, p = C.c_int64(), C.c_int64(), C.c_int64()
    dr = (C.c_int64 * max(1, layers))()
    _check(lib().dflash_context_ex(h, seq, C.byref(f), C.byref(n), C.byref(p), dr))
    return f.value, n.value, p.value, [dr[i] for i in range(layers)]


def dflash_pending_limit(geom: Geometry) -> int:
    return lib().dflash_pending_limit(C.byref(geom))


def dflash_bind_pending(h, seq, buf, rows):
    _check(lib().dflash_bind_pending(h, seq, buf, rows))


def dflash_queue(h, seq, pos, taps, n, stream):
    _check(lib().dflash_queue(h, seq, pos, taps, n, stream))


def dflash_settle_pending(h, seq, stream):
    _check(lib().dflash_settle_pending(h, seq, stream))


def dflash_truncate(h, seq, pos):
    _check(lib().dflash_truncate(h, seq, pos))


def dflash_push_rows(h, seq, pos, n, k_ptrs, v_ptrs, stream):
    ks = (C.c_void_p * len(k_ptrs))(*k_ptrs)
    vs = (C.c_void_p * len(v_ptrs))(*v_ptrs)
    _check(lib().dflash_push_rows(h, seq, pos, n, ks, vs, stream))


def dflash_context(h, seq):
    f, n = C.c_int64(), C.c_int64()
    _check(lib().dflash_context(h, seq, C.byref(f), C.byref(n)))
    return f.value, n.value


def dflash_settle(h, seq, pos, taps, n, stream):
    _check(lib().dflash_settle(h, seq, pos, taps, n, stream))


def dflash_block(h, batch, anchor_pos, hrows, k, width, logits, hp, stream):
    ap = (C.c_int64 * batch)(*[int(a) for a in anchor_pos])
    _check(lib().dflash_block(h, batch, ap, hrows, k, width, logits, hp, stream))


def dflash_select(h, batch, logits, hp, anchor_tok, k, width, chosen, plain, stream):
    _check(lib().dflash_select(h, batch, logits, hp, anchor_tok, k, width, chosen, plain, stream))


def dflash_draft(h, batch, anchor_pos, hrows, k, width, anchor_tok, logits, hp, chosen, plain, stream):
    ap = (C.c_int64 * batch)(*[int(a) for a in anchor_pos])
    _check(lib().dflash_draft(h, batch, ap, hrows, k, width, anchor_tok, logits, hp, chosen, plain, stream))


def dflash_select_static(logits, hp, anchor_tok, pred_book, succ_book, batch, k, width, vocab, rank, top, chosen,
                         plain, stream):
    """The selector with its scratch inside the library (for callers that cannot allocate device memory)."""
    _check(lib().dflash_select_static(logits, hp, anchor_tok, pred_book, succ_book, batch, k, width, vocab, rank,
                                      top, chosen, plain, stream))


def dflash_route_margin(route: Route, hidden, rows, n, margin, stream):
    _check(lib().dflash_route_margin(C.byref(route), hidden, rows, n, margin, stream))


def dflash_destroy(h):
    lib().dflash_destroy(h)


def dflash_launch_count() -> int:
    return lib().dflash_launch_count()

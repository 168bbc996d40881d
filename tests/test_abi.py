"""The C ABI without a GPU: the library loads, exports every declared entry point,
and its host-side checks reject bad geometry and arguments before any launch."""
import ctypes as C
import dataclasses
import os
import re

import pytest

import dflash_inputs as di

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from speculative_block_drafter_gb300 import build, _lib
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    _lib.lib()
    return _lib


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(dflash_[a-z0-9_]+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert "dflash_create" in names and "dflash_block" in names
    lib = L.lib()
    for n in sorted(names):
        assert hasattr(lib, n), n
    assert names <= set(L.EXPORTS), names - set(L.EXPORTS)


def _geom(L, **over):
    from speculative_block_drafter_gb300.drafter import geometry_struct
    g = dataclasses.replace(di.workload("tiny").geometry, **over)
    return geometry_struct(g)


def test_workspace_bytes_for_every_workload(L):
    from speculative_block_drafter_gb300.drafter import geometry_struct
    for name, wl in di.WORKLOADS.items():
        n = L.dflash_workspace_bytes(geometry_struct(wl.geometry), wl.batch)
        assert n > 0, name


@pytest.mark.parametrize("over", [dict(layers=0), dict(block=1), dict(taps=0), dict(kv_heads=0), dict(heads=3),
                                  dict(conv_group=0), dict(conv_group=7), dict(head_dim=96), dict(block=17),
                                  dict(quant_group=48), dict(selector_top=33), dict(hidden=200, conv_group=8),
                                  dict(vocab=4100), dict(selector_rank=8)])
def test_geometry_rules(L, over):
    g = _geom(L, **over)
    if "layers" in over and over["layers"] == 0:
        pass
    assert L.dflash_workspace_bytes(g, 1) == 0
    h = C.c_void_p()
    w = L.Weights()
    one = (C.c_void_p * 1)(C.c_void_p(4096))
    code = L.lib().dflash_create(C.byref(h), C.byref(g), C.byref(w), 1, one, one, 16, C.c_void_p(4096), 1 << 30)
    assert code == 1, L.last_error()
    assert "geometry" in L.last_error()


def _fake_create(L, max_batch=1, cap=64):
    """A drafter bound to aligned fake addresses: valid for host-only calls, never for launches."""
    g = _geom(L)
    addr = [1 << 20]

    def nxt():
        addr[0] += 4096
        return addr[0]

    layers = (L.LayerWeights * g.layers)()
    for i in range(g.layers):
        x = layers[i]
        for f in ("in_norm", "post_norm", "q_norm", "k_norm", "attn_base", "mlp_base"):
            setattr(x, f, nxt())
        x.attn_proj = L.Matrix(nxt(), None)
        x.mlp_proj = L.Matrix(nxt(), None)
        for f in ("q", "k", "v", "o", "gate", "up", "down"):
            setattr(x, f, L.Matrix(nxt(), nxt()))
    w = L.Weights()
    w.fc, w.sel, w.head = L.Matrix(nxt(), None), L.Matrix(nxt(), None), L.Matrix(nxt(), nxt())
    w.hidden_norm, w.norm, w.pred_book, w.succ_book = nxt(), nxt(), nxt(), nxt()
    w.layers = C.cast(layers, C.POINTER(L.LayerWeights))
    caches = [nxt() for _ in range(max_batch * g.layers)]
    ws = L.dflash_workspace_bytes(g, max_batch)
    return L.dflash_create(g, w, max_batch, caches, caches, cap, nxt(), ws), (g, w, layers)


def test_create_and_host_state(L):
    h, keep = _fake_create(L, max_batch=2)
    assert L.dflash_context(h, 0) == (0, 0)
    L.dflash_reset(h, 1, 500)
    assert L.dflash_context(h, 1) == (500, 0)
    with pytest.raises(L.DflashError):
        L.dflash_reset(h, 2, 0)
    L.dflash_destroy(h)


def test_settle_and_block_argument_errors_before_any_launch(L):
    h, keep = _fake_create(L, max_batch=1, cap=64)
    taps = 1 << 24
    for n in (0, L.SETTLE_MAX + 1):
        with pytest.raises(L.DflashError) as e:
            L.dflash_settle(h, 0, 0, taps, n, None)
        assert e.value.code == 2
    with pytest.raises(L.DflashError) as e:               # the cache holds 64 rows
        L.dflash_settle(h, 0, 0, taps, 65, None)
    assert e.value.code == 3
    with pytest.raises(L.DflashError) as e:               # a gap starts over at 1000: 65 rows still do not fit
        L.dflash_settle(h, 0, 1000, taps, 65, None)
    assert e.value.code == 3
    assert L.dflash_context(h, 0) == (0, 0)               # a refused call leaves the context as it was
    for pos in (-1,):
        with pytest.raises(L.DflashError) as e:
            L.dflash_settle(h, 0, pos, taps, 1, None)
        assert e.value.code == 2
    out = 1 << 25
    for k, width in ((0, 4096), (16, 4096), (15, 7), (15, 4097)):
        with pytest.raises(L.DflashError) as e:
            L.dflash_block(h, 1, [0], taps, k, width, out, out, None)
        assert e.value.code == 2
    with pytest.raises(L.DflashError) as e:
        L.dflash_block(h, 2, [0, 0], taps, 15, 4096, out, out, None)
    assert e.value.code == 2
    L.dflash_destroy(h)


def test_draft_argument_errors_before_any_launch(L):
    """dflash_draft refuses what dflash_block or dflash_select would refuse, and null
    token pointers, on the host."""
    h, keep = _fake_create(L, max_batch=1, cap=64)
    rows, p = 1 << 24, 1 << 25
    for k, width in ((0, 4096), (16, 4096), (15, 7), (15, 4097)):
        with pytest.raises(L.DflashError) as e:
            L.dflash_draft(h, 1, [0], rows, k, width, p, p, p, p, p, None)
        assert e.value.code == 2
    with pytest.raises(L.DflashError) as e:               # batch above max_batch
        L.dflash_draft(h, 2, [0, 0], rows, 15, 4096, p, p, p, p, p, None)
    assert e.value.code == 2
    for null in range(3):                                 # anchor tokens, chosen, plain
        ptrs = [p, p, p]
        ptrs[null] = 0
        with pytest.raises(L.DflashError) as e:
            L.dflash_draft(h, 1, [0], rows, 15, 4096, ptrs[0], p, p, ptrs[1], ptrs[2], None)
        assert e.value.code == 2
    L.dflash_destroy(h)


def test_create_rejects_small_workspace_and_null_weights(L):
    g = _geom(L)
    h = C.c_void_p()
    w = L.Weights()
    one = (C.c_void_p * 1)(C.c_void_p(4096))
    code = L.lib().dflash_create(C.byref(h), C.byref(g), C.byref(w), 1, one, one, 16, C.c_void_p(4096), 1024)
    assert code == 3
    ws = L.dflash_workspace_bytes(g, 1)
    code = L.lib().dflash_create(C.byref(h), C.byref(g), C.byref(w), 1, one, one, 16, C.c_void_p(4096), ws)
    assert code == 2


def test_packed_sizes(L):
    # rows pad to tiles of 128; codes are half a byte, scales one f16 per row and 64 (or 32) columns
    assert L.dflash_int4_packed_bytes(32, 128, 64) == 128 * 64
    assert L.dflash_int4_packed_bytes(256, 128, 64) == 256 * 64
    assert L.dflash_int4_scale_bytes(256, 128, 64) == 2 * 2 * 256
    assert L.dflash_int4_scale_bytes(256, 128, 32) == 2 * 2 * 2 * 256
    assert L.dflash_int4_packed_bytes(32, 96, 32) == 0
    assert L.dflash_int4_packed_bytes(32, 128, 48) == 0
    assert L.dflash_f16_packed_bytes(16, 64) == 128 * 64 * 2
    assert L.dflash_gemm_workspace_bytes(4, 1024, 16) == 16 * 1024 * 4
    # more than 32 rows: token tiles of at most 256 rows, equal heights rounded up to 16
    assert L.dflash_gemm_workspace_bytes(16, 1024, 200) == 208 * 1024 * 2
    assert L.dflash_gemm_workspace_bytes(4, 1024, 480) == 2 * 240 * 1024 * 2 * 2
    assert L.dflash_gemm_workspace_bytes(5, 1024, 16) == 0


def test_gemm_packed_argument_errors_before_any_launch(L):
    """dflash_gemm_packed refuses more than 32 rows, null pointers, misalignment and bad shapes
    on the host (no device work is enqueued)."""
    m = L.Matrix(1 << 20, 1 << 20)
    for args in ((4, 256, 1024, 64, 33, 1 << 24, 1 << 24),   # T > 32
                 (4, 256, 1024, 64, 0, 1 << 24, 1 << 24),    # no rows
                 (4, 256, 1000, 64, 16, 1 << 24, 1 << 24),   # cols not a multiple of 64
                 (5, 256, 1024, 64, 16, 1 << 24, 1 << 24),   # kind
                 (4, 256, 1024, 64, 16, 0, 1 << 24),         # y null
                 (4, 256, 1024, 64, 16, 1 << 24, (1 << 24) + 4)):  # workspace misaligned
        kind, rows, cols, group, T, y, ws = args
        with pytest.raises(L.DflashError) as e:
            L.dflash_gemm_packed(m, kind, rows, cols, group, T, y, ws, None)
        assert e.value.code == 2, args


def test_select_argument_errors_before_any_launch(L):
    h, keep = _fake_create(L, max_batch=2)
    g = keep[0]
    p = 1 << 24
    bad = [dict(batch=0), dict(batch=3), dict(k=0), dict(k=g.block), dict(width=g.selector_top - 1),
           dict(width=g.vocab + 1), dict(logits=0), dict(hp=0), dict(anchor=0), dict(chosen=0), dict(plain=0)]
    for over in bad:
        a = dict(batch=1, logits=p, hp=p, anchor=p, k=g.block - 1, width=g.vocab, chosen=p, plain=p)
        a.update(over)
        with pytest.raises(L.DflashError) as e:
            L.dflash_select(h, a["batch"], a["logits"], a["hp"], a["anchor"], a["k"], a["width"], a["chosen"],
                            a["plain"], None)
        assert e.value.code == 2, over
    L.dflash_destroy(h)


def test_select_static_argument_and_capacity_errors_before_any_launch(L):
    """The fixed-scratch selector checks its sizes on the host; a call whose tables pass
    the 8 MiB array gets CAPACITY before it looks the array up on any device."""
    p = 1 << 24
    base = dict(batch=1, k=15, width=151936, vocab=151936, rank=64, top=16)
    bad = [dict(batch=0), dict(k=0), dict(k=16), dict(top=0), dict(top=33), dict(width=15), dict(width=151937),
           dict(rank=8), dict(rank=24), dict(rank=272)]
    for over in bad:
        a = dict(base, **over)
        with pytest.raises(L.DflashError) as e:
            L.dflash_select_static(p, p, p, p, p, a["batch"], a["k"], a["width"], a["vocab"], a["rank"], a["top"],
                                   p, p, None)
        assert e.value.code == 2, over
    for ptr in range(7):
        ptrs = [p] * 7
        ptrs[ptr] = 0
        with pytest.raises(L.DflashError) as e:
            L.dflash_select_static(ptrs[0], ptrs[1], ptrs[2], ptrs[3], ptrs[4], 1, 15, 151936, 151936, 64, 16,
                                   ptrs[5], ptrs[6], None)
        assert e.value.code == 2, ptr
    # rows * (chunks * 8 + 8200 + top * 4 + top^2 * 4) + 256 bytes against 8 MiB: 56 sequences fit, 64 do not
    with pytest.raises(L.DflashError) as e:
        L.dflash_select_static(p, p, p, p, p, 64, 15, 151936, 151936, 64, 16, p, p, None)
    assert e.value.code == 3


def test_pack_and_dequant_argument_errors_before_any_launch(L):
    p = 1 << 24
    for rows, cols, group in ((32, 96, 32), (32, 128, 48), (0, 128, 64)):
        with pytest.raises(L.DflashError) as e:
            L.dflash_pack_int4(p, p, rows, cols, group, p, p, None)
        assert e.value.code == 2
        with pytest.raises(L.DflashError) as e:
            L.dflash_dequant_int4(p, p, rows, cols, group, p, None)
        assert e.value.code == 2
    for args in ((0, p, p, p), (p, 0, p, p), (p, p, 0, p), (p, p, p, 0), (p, p, p + 8, p), (p, p, p, p + 4)):
        with pytest.raises(L.DflashError) as e:
            L.dflash_pack_int4(args[0], args[1], 256, 128, 64, args[2], args[3], None)
        assert e.value.code == 2, args
    for src, dst in ((0, p), (p, 0), (p, p + 8)):
        with pytest.raises(L.DflashError) as e:
            L.dflash_pack_f16(src, 256, 128, dst, None)
        assert e.value.code == 2
    with pytest.raises(L.DflashError) as e:
        L.dflash_pack_f16(p, 256, 100, p, None)
    assert e.value.code == 2
    for codes, scales, out in ((0, p, p), (p, 0, p), (p, p, 0), (p + 4, p, p), (p, p + 4, p)):
        with pytest.raises(L.DflashError) as e:
            L.dflash_dequant_int4(codes, scales, 256, 128, 64, out, None)
        assert e.value.code == 2


def test_gemm_argument_errors_before_any_launch(L):
    p = 1 << 24
    m = L.Matrix(p, p)
    ws = L.dflash_gemm_workspace_bytes(4, 1024, 16)
    for kind, rows, cols, group, x, T, y, w, wb, code in (
            (4, 256, 1024, 64, 0, 16, p, p, ws, 2),          # x null
            (4, 256, 1024, 64, p, 0, p, p, ws, 2),           # no rows
            (4, 256, 1024, 64, p + 2, 16, p, p, ws, 2),      # x misaligned
            (4, 256, 1000, 64, p, 16, p, p, ws, 2),          # cols
            (7, 256, 1024, 64, p, 16, p, p, ws, 2),          # kind
            (4, 256, 1024, 64, p, 16, p, 0, ws, 2),          # workspace null
            (4, 256, 1024, 64, p, 16, p, p + 8, ws, 2),      # workspace misaligned
            (4, 256, 1024, 64, p, 16, p, p, ws - 16, 3)):    # workspace too small
        with pytest.raises(L.DflashError) as e:
            L.dflash_gemm(m, kind, rows, cols, group, x, T, y, w, wb, None)
        assert e.value.code == code, (kind, rows, cols, x, T, w, wb)


def test_context_and_reset_argument_errors(L):
    h, keep = _fake_create(L, max_batch=1)
    for seq in (-1, 1):
        with pytest.raises(L.DflashError):
            L.dflash_context(h, seq)
        with pytest.raises(L.DflashError):
            L.dflash_reset(h, seq, 0)
    with pytest.raises(L.DflashError):
        L.dflash_reset(h, 0, -1)
    L.dflash_destroy(h)


def test_cache_layouts(L):
    """Linear caches hold ctx_cap rows; a ring needs a windowed layer and at least twice its
    window, and holds its ring plus `window` rows repeating its first ones; planes take 4
    bytes an element, one f16 two."""
    g = _geom(L, windows=(100,))
    lin = L.CacheConfig()
    assert L.dflash_cache_rows(g, lin, 0, 4096) == 4096
    assert L.dflash_cache_bytes(g, lin, 0, 4096) == 4096 * 2 * 64 * 4
    assert L.dflash_cache_rows(g, None, 0, 4096) == 4096
    ring = L.CacheConfig()
    ring.ring[0] = 200
    assert L.dflash_cache_rows(g, ring, 0, 4096) == 300
    ring.format = L.KV_F16
    assert L.dflash_cache_bytes(g, ring, 0, 4096) == 300 * 2 * 64 * 2
    ring.ring[0] = 199                                     # less than twice the window
    assert L.dflash_cache_rows(g, ring, 0, 4096) == 0
    ring.ring[0] = 200
    assert L.dflash_cache_rows(_geom(L), ring, 0, 4096) == 0   # window 0: no ring
    bad = L.CacheConfig()
    bad.format = 7
    assert L.dflash_cache_bytes(g, bad, 0, 4096) == 0
    assert L.dflash_cache_rows(g, lin, 1, 4096) == 0           # no such layer


def test_pending_limit_follows_the_widest_window(L):
    # dflash.rs Drafter::queue_context (CUDA arm): 512, or the widest window + 256 when every layer has one
    assert L.dflash_pending_limit(_geom(L)) == 512
    assert L.dflash_pending_limit(_geom(L, windows=(100,))) == 512
    assert L.dflash_pending_limit(_geom(L, windows=(600,))) == 856


def test_bookkeeping_argument_errors_before_any_launch(L):
    h, keep = _fake_create(L, max_batch=1, cap=64)
    taps = 1 << 24
    assert L.dflash_context_ex(h, 0, 1) == (0, 0, 0, [0])
    with pytest.raises(L.DflashError) as e:                   # no pending buffer bound
        L.dflash_queue(h, 0, 0, taps, 1, None)
    assert e.value.code == 2
    with pytest.raises(L.DflashError) as e:                   # fewer rows than the pending limit
        L.dflash_bind_pending(h, 0, 1 << 26, 511)
    assert e.value.code == 3
    with pytest.raises(L.DflashError) as e:
        L.dflash_bind_pending(h, 0, (1 << 26) + 8, 512)
    assert e.value.code == 2
    L.dflash_bind_pending(h, 0, None, 0)
    L.dflash_settle_pending(h, 0, None)                      # nothing waits: nothing to do
    L.dflash_truncate(h, 0, 10)
    assert L.dflash_context_ex(h, 0, 1) == (0, 0, 0, [0])
    with pytest.raises(L.DflashError):
        L.dflash_truncate(h, 1, 0)
    with pytest.raises(L.DflashError) as e:                   # rows past the 64-row cache
        L.dflash_push_rows(h, 0, 0, 65, [taps], [taps], None)
    assert e.value.code == 3
    with pytest.raises(L.DflashError) as e:                   # a layer's rows missing
        L.dflash_push_rows(h, 0, 0, 4, [taps], [None], None)
    assert e.value.code == 2
    L.dflash_destroy(h)


def test_create_ex_rejects_bad_cache_layouts(L):
    from speculative_block_drafter_gb300.drafter import geometry_struct
    g = geometry_struct(dataclasses.replace(di.workload("tiny").geometry, windows=(100,)))
    h = C.c_void_p()
    w = L.Weights()
    one = (C.c_void_p * 1)(C.c_void_p(4096))
    cache = L.CacheConfig()
    cache.ring[0] = 150
    code = L.lib().dflash_create_ex(C.byref(h), C.byref(g), C.byref(w), 1, C.byref(cache), one, one, 16,
                                    C.c_void_p(4096), 1 << 30)
    assert code == 2 and "ring" in L.last_error()
    cache.ring[0] = 0
    cache.format = 3
    code = L.lib().dflash_create_ex(C.byref(h), C.byref(g), C.byref(w), 1, C.byref(cache), one, one, 16,
                                    C.c_void_p(4096), 1 << 30)
    assert code == 2 and "format" in L.last_error()


def test_route_margin_argument_errors_before_any_launch(L):
    p = 1 << 20
    for r, hidden, n, code in ((L.Route(p, p, p, p, 257, 4), 64, 1, 2),   # rank past 256
                               (L.Route(None, p, p, p, 4, 4), 64, 1, 2),  # no block mean
                               (L.Route(p, None, p, p, 4, 4), 64, 1, 2),  # a basis missing at rank 4
                               (L.Route(p, p, p, p, 4, 4), 0, 1, 2),      # hidden
                               (L.Route(p, p, p, p, 4, 4), 64, 0, 2)):    # no rows
        with pytest.raises(L.DflashError) as e:
            L.dflash_route_margin(r, hidden, p, n, p, None)
        assert e.value.code == code

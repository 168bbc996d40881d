"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test ties an oracle function to something other than itself: the page's
worked example, a closed form, a library routine on a special case, brute
force on a tiny input, or an invariant of the method. They run without a GPU.
"""
import dataclasses
import math
import os

import numpy as np
import pytest

import dflash_inputs as di
from oracle import dflash_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ four-bit matrices

def _pack(q: np.ndarray) -> np.ndarray:
    """Codes -7..7 [rows][cols] -> interchange bytes (test-side packer, by the format's text)."""
    u = (q + 8).astype(np.uint8)
    return (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)


def test_dequant_hand_group():
    # byte 0x19: low nibble 9 -> +1 at the even column, high nibble 1 -> -7 at the odd one
    codes = np.array([[0x19, 0x8F]], dtype=np.uint8)
    scales = np.array([[0.5]], dtype=np.float16)
    w = O.dequant_int4(codes, scales, 4)
    assert w.tolist() == [[0.5, -3.5, 3.5, 0.0]]


def test_dequant_roundtrip_exact():
    rng = np.random.default_rng(1)
    rows, cols, group = 37, 256, 32
    q = rng.integers(-7, 8, size=(rows, cols))
    # every group holds a code of magnitude 7, so its scale is recovered exactly
    for r in range(rows):
        for g0 in range(0, cols, group):
            q[r, g0 + rng.integers(0, group)] = 7 * (1 if rng.random() < 0.5 else -1)
    scales = (rng.random((rows, cols // group)) * 0.1 + 1e-3).astype(np.float16)
    codes = _pack(q)
    w = O.dequant_int4(codes, scales, group)
    c2, s2 = di.quantize_int4(w.astype(np.float32), group)
    assert np.array_equal(c2, codes)
    assert np.array_equal(s2.view(np.uint16), scales.view(np.uint16))


def test_dequant_zero_group():
    codes, scales = di.quantize_int4(np.zeros((2, 64), np.float32), 32)
    assert np.all(O.dequant_int4(codes, scales, 32) == 0.0)
    assert np.all(codes == 0x88)


def test_int4_matmul_brute_force():
    rng = np.random.default_rng(2)
    rows, cols, group, n = 5, 64, 16, 3
    q = rng.integers(-7, 8, size=(rows, cols))
    scales = (rng.random((rows, cols // group)) + 0.1).astype(np.float16)
    m = di.Int4(codes=_pack(q), scales=scales, rows=rows, cols=cols, group=group)
    x = rng.standard_normal((n, cols))
    y = O.int4_matmul(m, x)
    for i in range(n):
        for r in range(rows):
            acc = 0.0
            for c in range(cols):
                acc += float(q[r, c]) * float(scales[r, c // group]) * x[i, c]
            assert abs(y[i, r] - acc) <= 1e-12 * max(1.0, abs(acc))
    # a slab of rows
    assert np.allclose(O.int4_matmul(m, x, 1, 4), y[:, 1:4], rtol=0, atol=1e-13)


def test_int4_single_code_gives_scale_times_x():
    q = np.zeros((3, 32), dtype=np.int64)
    q[1, 5] = 1
    scales = np.full((3, 1), 0.375, dtype=np.float16)
    m = di.Int4(codes=_pack(q), scales=scales, rows=3, cols=32, group=32)
    x = np.arange(32, dtype=np.float64)[None, :] * 0.25
    y = O.int4_matmul(m, x)
    assert y.tolist() == [[0.0, 0.375 * 5 * 0.25, 0.0]]


def test_f16_matmul_rounds_activations_to_f16():
    w = np.array([[1.0, 1.0]], dtype=np.float16)
    x = np.array([[1.0 + 2.0 ** -12, 3.0]])          # 1 + 2^-12 rounds to 1 in f16
    assert O.f16_matmul(w, x).tolist() == [[4.0]]
    rng = np.random.default_rng(3)
    w = rng.standard_normal((4, 24)).astype(np.float16)
    x = rng.standard_normal((2, 24))
    ref = [[sum(float(np.float16(x[i, c])) * float(w[r, c]) for c in range(24)) for r in range(4)] for i in range(2)]
    assert np.allclose(O.f16_matmul(w, x), ref, rtol=0, atol=1e-12)


def test_mlp_closed_form_on_scaled_identities():
    """gate = 2I, up = I, down = the swap of the first two rows: the output is the
    swapped vector of silu(2x) * x, with silu(a) = a / (1 + e^-a). Swapping gate and
    up (silu(x) * 2x), applying silu to up, or reading down transposed each fail."""
    n = 32
    eye = np.eye(n, dtype=np.int64)
    swap = eye.copy()
    swap[[0, 1]] = swap[[1, 0]]
    swap[0, 5] = 1                       # down row 0 also reads column 5: not symmetric
    one = np.ones((n, 1), dtype=np.float16)
    mat = lambda q, s: di.Int4(codes=_pack(q), scales=s, rows=n, cols=n, group=n)
    L = {"gate": mat(2 * eye, one), "up": mat(eye, one), "down": mat(swap, np.full((n, 1), 0.5, np.float16))}
    x = np.linspace(-3.0, 2.5, n)[None, :]
    m = [2 * v / (1 + math.exp(-2 * v)) * v for v in x[0]]
    want = [0.5 * m[i] for i in range(n)]
    want[0], want[1] = 0.5 * (m[1] + m[5]), 0.5 * m[0]
    assert np.allclose(O.mlp(L, x)[0], want, rtol=1e-13, atol=1e-15)


# ------------------------------------------------------------------ norms and rotation

def test_rms_constant_row_closed_form():
    w = np.array([1.0, 2.0, -0.5, 3.0])
    for c, eps in [(2.0, 0.0), (-0.3, 1e-6), (1e-4, 1e-6)]:
        y = O.rms(np.full(4, c), w, eps)
        assert np.allclose(y, c / math.sqrt(c * c + eps) * w, rtol=1e-14, atol=0)


def test_rms_unit_mean_square_and_scale_invariance():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 64))
    y = O.rms(x, np.ones(64), 0.0)
    assert np.allclose((y * y).mean(axis=1), 1.0, rtol=1e-13)
    assert np.allclose(O.rms(-7.5 * x, np.ones(64), 0.0), -y, rtol=1e-13)
    # per head: a [rows][heads*hd] input normalises each run of hd alone
    z = O.rms(x.reshape(3, 64), np.ones(16), 0.0).reshape(3, 4, 16)
    assert np.allclose((z * z).mean(axis=2), 1.0, rtol=1e-13)


def test_inv_freq_closed_form():
    inv = O.inv_freq(128, 1e6)
    assert inv.dtype == np.float32 and len(inv) == 64
    assert inv[0] == 1.0
    assert inv[32] == np.float32(1e-3)          # theta^(-64/128) = 1e6^-0.5
    assert inv[16] == np.float32(10 ** -1.5)


def test_rotate_is_complex_multiplication_on_half_split_pairs():
    inv = np.array([1.0, 0.25], dtype=np.float32)     # head_dim 4
    x = np.array([[1.0, 2.0, 3.0, -1.0]])
    p = 3
    y = O.rotate(x, 1, [p], inv)
    for i, f in enumerate(inv):
        ang = float(np.float32(p) * f)
        z = complex(x[0, i], x[0, i + 2]) * complex(math.cos(ang), math.sin(ang))
        assert abs(y[0, i] - z.real) < 1e-14 and abs(y[0, i + 2] - z.imag) < 1e-14
    # the pair is (i, i + hd/2): a unit vector in slot 0 turns into slot 2, not slot 1
    e = O.rotate(np.array([[1.0, 0.0, 0.0, 0.0]]), 1, [p], inv)
    assert abs(e[0, 1]) == 0.0 and abs(e[0, 2] - math.sin(3.0)) < 1e-15


def test_rotate_position_zero_identity_norms_and_relative_position():
    rng = np.random.default_rng(5)
    inv = O.inv_freq(64, 1e6)
    x = rng.standard_normal((2, 3 * 64))
    assert np.array_equal(O.rotate(x, 3, [0, 0], inv), x)
    y = O.rotate(x, 3, [7, 1000], inv)
    pairs = lambda v: v.reshape(2, 3, 2, 32)
    assert np.allclose((pairs(y) ** 2).sum(2), (pairs(x) ** 2).sum(2), rtol=1e-13)
    q, k = rng.standard_normal((1, 64)), rng.standard_normal((1, 64))
    d0 = (O.rotate(q, 1, [10], inv) * O.rotate(k, 1, [3], inv)).sum()
    d1 = (O.rotate(q, 1, [110], inv) * O.rotate(k, 1, [103], inv)).sum()
    assert abs(d0 - d1) < 1e-5 * (np.abs(q).sum() * np.abs(k).sum()) ** 0.5


def test_rotate_composes_by_adding_positions():
    """Rotating by p2 and then by p1 is rotating by p1 + p2, up to the f32 rounding of
    the angles; rotating by p then by -p returns the input."""
    rng = np.random.default_rng(21)
    inv = O.inv_freq(128, 1e6)
    x = rng.standard_normal((3, 2 * 128))
    p1, p2 = [5, 300, 4000], [17, 2, 123]
    twice = O.rotate(O.rotate(x, 2, p2, inv), 2, p1, inv)
    once = O.rotate(x, 2, [a + b for a, b in zip(p1, p2)], inv)
    assert np.allclose(twice, once, rtol=0, atol=2e-3 * np.abs(x).max())
    assert not np.allclose(twice, O.rotate(x, 2, p1, inv), rtol=0, atol=1e-3)
    back = O.rotate(O.rotate(x, 2, p1, inv), 2, [-p for p in p1], inv)
    assert np.allclose(back, x, rtol=0, atol=1e-12)


# ------------------------------------------------------------------ row convolution

def _base(kn, hs, rng):
    return rng.standard_normal((2, kn, hs))


def test_conv_identity_kernel():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((5, 8))
    base = np.zeros((2, 1, 8)); base[:, 0, :] = 1.0
    d = np.zeros((5, 2 * 1 * 2))
    for stage in (0, 1):
        assert np.array_equal(O.conv(base, d, x, stage, 1, 4), x)


def test_conv_static_kernel_is_causal_fir():
    rng = np.random.default_rng(7)
    rows, hs, kn = 9, 12, 4
    x = rng.standard_normal((rows, hs))
    base = _base(kn, hs, rng)
    d = np.zeros((rows, 2 * kn * (hs // 3)))
    for stage in (0, 1):
        y = O.conv(base, d, x, stage, kn, 3)
        for i in range(hs):
            ref = np.convolve(x[:, i], base[stage, :, i])[:rows]
            assert np.allclose(y[:, i], ref, rtol=0, atol=1e-13)


def test_conv_dynamic_term_reaches_only_its_group_row_and_offset():
    rng = np.random.default_rng(8)
    rows, hs, kn, gs = 6, 8, 3, 2
    groups = hs // gs
    x = rng.standard_normal((rows, hs))
    base = np.zeros((2, kn, hs))
    d = np.zeros((rows, 2, kn, groups))
    r, stage, o, g = 4, 1, 2, 3
    d[r, stage, o, g] = 0.5
    y = O.conv(base, d.reshape(rows, -1), x, stage, kn, gs)
    want = np.zeros((rows, hs))
    want[r, g * gs:(g + 1) * gs] = 0.5 * x[r - o, g * gs:(g + 1) * gs]
    assert np.array_equal(y, want)
    # the other stage does not see it
    assert np.all(O.conv(base, d.reshape(rows, -1), x, 0, kn, gs) == 0)


def test_conv_row_zero_sees_only_itself():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((4, 6)); x2 = x.copy(); x2[1:] = rng.standard_normal((3, 6))
    base = _base(4, 6, rng); d = rng.standard_normal((4, 2 * 4 * 3))
    assert np.array_equal(O.conv(base, d, x, 0, 4, 2)[0], O.conv(base, d, x2, 0, 4, 2)[0])


# ------------------------------------------------------------------ attention

def _softmax_attention_brute(q, keys, vals, scale):
    out = []
    for qi in q:
        s = [scale * sum(a * b for a, b in zip(qi, k)) for k in keys]
        m = max(s)
        e = [math.exp(v - m) for v in s]
        z = sum(e)
        out.append([sum(e[j] * vals[j][c] for j in range(len(keys))) / z for c in range(len(vals[0]))])
    return np.array(out)


def test_attention_without_context_is_plain_softmax_attention():
    rng = np.random.default_rng(10)
    rows, hd = 4, 6
    q, k, v = (rng.standard_normal((rows, hd)) for _ in range(3))
    empty = np.zeros((0, 1, hd))
    y = O.attention(q, k, v, empty, empty, 0, 0, 0, 1, 1, hd, 0.4)
    assert np.allclose(y, _softmax_attention_brute(q, k, v, 0.4), rtol=0, atol=1e-13)


def test_attention_one_key_returns_its_value():
    rng = np.random.default_rng(11)
    v = rng.standard_normal((1, 8))
    empty = np.zeros((0, 1, 8))
    y = O.attention(rng.standard_normal((1, 8)), rng.standard_normal((1, 8)), v, empty, empty, 0, 5, 0, 1, 1, 8, 1.0)
    assert np.allclose(y, v, rtol=0, atol=1e-15)


def test_attention_gqa_maps_contiguous_heads():
    rows, hd, nh, kv = 2, 4, 4, 2
    q = np.zeros((rows, nh * hd))
    k = np.zeros((rows, kv * hd))
    v = np.concatenate([np.zeros((rows, hd)), np.ones((rows, hd))], axis=1)
    empty = np.zeros((0, kv, hd))
    y = O.attention(q, k, v, empty, empty, 0, 0, 0, nh, kv, hd, 1.0).reshape(rows, nh, hd)
    assert np.all(y[:, :2] == 0.0) and np.all(y[:, 2:] == 1.0)


def test_attention_window_mask_uniform_weights_closed_form():
    # zero queries: every visible key weighs the same, so y is the mean of the visible values
    hd, rows, n, lo, anchor, window = 2, 3, 10, 20, 30, 6
    ck = np.zeros((n, 1, hd))
    cv = np.zeros((n, 1, hd))
    for j in range(n):
        cv[j, 0, :] = lo + j                # value = its position
    blk_v = np.full((rows, hd), 100.0)
    y = O.attention(np.zeros((rows, hd)), np.zeros((rows, hd)), blk_v, ck, cv, lo, anchor, window, 1, 1, hd, 1.0)
    for r in range(rows):
        first = anchor + r + 1 - window     # the row sees context positions >= first
        vis = [p for p in range(lo, lo + n) if p >= first]
        want = (sum(vis) + 100.0 * rows) / (len(vis) + rows)
        assert np.allclose(y[r], want, rtol=1e-14)


def test_attention_window_zero_equals_a_covering_window():
    rng = np.random.default_rng(12)
    rows, hd, n, anchor = 3, 4, 7, 7
    args = [rng.standard_normal((rows, 2 * hd)), rng.standard_normal((rows, hd)), rng.standard_normal((rows, hd)),
            rng.standard_normal((n, 1, hd)), rng.standard_normal((n, 1, hd))]
    y0 = O.attention(*args, 0, anchor, 0, 2, 1, hd, 0.5)
    y1 = O.attention(*args, 0, anchor, anchor + rows, 2, 1, hd, 0.5)
    assert np.array_equal(y0, y1)


def test_attention_block_rows_permutation_equivariant():
    rng = np.random.default_rng(13)
    rows, hd, n = 6, 4, 5
    q, k, v = rng.standard_normal((rows, 2 * hd)), rng.standard_normal((rows, hd)), rng.standard_normal((rows, hd))
    ck, cv = rng.standard_normal((n, 1, hd)), rng.standard_normal((n, 1, hd))
    perm = np.concatenate([[0], 1 + rng.permutation(rows - 1)])
    y = O.attention(q, k, v, ck, cv, 0, n, 0, 2, 1, hd, 0.5)
    yp = O.attention(q[perm], k[perm], v[perm], ck, cv, 0, n, 0, 2, 1, hd, 0.5)
    assert np.allclose(yp, y[perm], rtol=0, atol=1e-14)


def test_context_range_cases():
    assert O.context_range(0, 100, 100, 0) == (0, 100)
    assert O.context_range(0, 100, 100, 10) == (91, 100)          # row 0 sees 91..99
    assert O.context_range(0, 100, 60, 0) == (0, 60)              # nothing at or after the anchor
    assert O.context_range(50, 10, 55, 100) == (50, 55)
    assert O.context_range(50, 10, 40, 0) == (50, 50)             # anchor before the context: empty
    assert O.context_range(0, 5, 5, 2) == (4, 5)


# ------------------------------------------------------------------ top-k and the selector

def _golden_top_k():
    lines = [l.split() for l in open(os.path.join(GOLDEN, "top_k_worked_example.txt")) if l.strip() and not l.startswith("#")]
    x = np.array([float(v) for v in lines[0][1:]])
    cases = []
    for l in lines[1:]:
        k = int(l[1])
        exp = [(float(p.split(":")[0]), int(p.split(":")[1])) for p in l[3:]]
        cases.append((k, exp))
    return x, cases


def test_top_k_worked_example_of_the_page():
    x, cases = _golden_top_k()
    for k, exp in cases:
        assert [(float(v), i) for v, i in O.top_k(x, k)] == exp


def _top_k_insertion(x, k):
    """Insertion into a sorted list, as the page's top_k describes it in words."""
    best = []
    for i, v in enumerate(x):
        if len(best) == k and v <= best[-1][0]:
            continue
        at = 0
        while at < len(best) and best[at][0] >= v:
            at += 1
        best.insert(at, (v, i))
        del best[k:]
    return best


def test_top_k_brute_force_with_ties():
    rng = np.random.default_rng(14)
    for trial in range(200):
        n = int(rng.integers(1, 40))
        x = rng.integers(-3, 4, size=n).astype(np.float64) * 0.5
        k = int(rng.integers(1, n + 1))
        got = [(float(v), i) for v, i in O.top_k(x, k)]
        assert got == [(float(v), i) for v, i in _top_k_insertion(list(x), k)]


def _books(V, rank, rng, zero=False):
    if zero:
        return np.zeros((V, rank), np.float16), np.zeros((V, rank), np.float16)
    return rng.standard_normal((V, rank)).astype(np.float16), rng.standard_normal((V, rank)).astype(np.float16)


def test_select_without_codebooks_picks_the_plain_token():
    rng = np.random.default_rng(15)
    logits = rng.standard_normal((5, 50))
    hp = rng.standard_normal((5, 8))
    P, C = _books(50, 8, rng, zero=True)
    chosen, plain = O.select_with(hp, logits, 3, P, C, 6)
    assert chosen == plain == [int(np.argmax(r)) for r in logits]
    P, C = _books(50, 8, rng)
    chosen, plain = O.select_with(hp, logits, 3, P, C, 1)
    assert chosen == plain


def test_select_brute_force_over_the_vocabulary():
    rng = np.random.default_rng(16)
    V, rank, top, n = 30, 4, 5, 6
    for trial in range(20):
        logits = rng.standard_normal((n, V))
        hp = rng.standard_normal((n, rank))
        P, C = _books(V, rank, rng)
        anchor = int(rng.integers(0, V))
        chosen, _ = O.select_with(hp, logits, anchor, P, C, top)
        prev = anchor
        for j in range(n):
            allscores = logits[j] + (P[prev].astype(np.float64) * hp[j]) @ C.astype(np.float64).T
            order = sorted(range(V), key=lambda t: (-logits[j][t], t))[:top]
            best = max(order, key=lambda t: (allscores[t], -order.index(t)))
            assert chosen[j] == best
            prev = best


# ------------------------------------------------------------------ whole-pass invariants (tiny shapes)

def _tiny(**over):
    g = dataclasses.replace(di.workload("tiny").geometry, **over)
    return g, di.make_weights(g, 0)


def test_block_mask_rows_enter_identical():
    g, w = _tiny()
    o = O.Oracle(g, w)
    o.settle(0, di.make_taps(g, 0, 20))
    tr = {}
    o.block(20, di.block_rows(g, 0, 5), tr)
    L0 = tr["layers"][0]
    assert np.array_equal(L0["x"][1], L0["x"][7]) and np.array_equal(L0["ad"][2], L0["ad"][15])
    assert not np.array_equal(L0["xc"][1], L0["xc"][7]) or g.conv_kernel == 1


def test_block_window_zero_equals_covering_window():
    g, w = _tiny(windows=(0,))
    g2 = dataclasses.replace(g, windows=(64,))
    taps = di.make_taps(g, 0, 40)
    h = di.block_rows(g, 0, 9)
    a, b = O.Oracle(g, w), O.Oracle(g2, w)
    a.settle(0, taps); b.settle(0, taps)
    assert np.array_equal(a.block(40, h), b.block(40, h))
    # a window shorter than the context changes the result
    c = O.Oracle(dataclasses.replace(g, windows=(8,)), w)
    c.settle(0, taps)
    assert not np.allclose(a.block(40, h), c.block(40, h))


def test_block_no_rope_layer_is_position_invariant():
    g, w = _tiny(no_rope=(0,))
    taps = di.make_taps(g, 0, 24)
    h = di.block_rows(g, 0, 11)
    a, b = O.Oracle(g, w), O.Oracle(g, w)
    a.settle(0, taps)
    b.reset(first=1000); b.settle(1000, taps)
    assert np.allclose(a.block(24, h), b.block(1024, h), rtol=0, atol=1e-12)
    # with rotation the positions matter
    g2, _ = _tiny()
    c, d = O.Oracle(g2, w), O.Oracle(g2, w)
    c.settle(0, taps); d.reset(first=1000); d.settle(1000, taps)
    assert not np.allclose(c.block(24, h), d.block(1024, h), rtol=0, atol=1e-6)


def test_block_with_zero_output_matrices_is_the_final_norm_of_its_input():
    """With every layer's o and down matrices zero, both sub-layers add nothing to the
    residual stream (the stage-1 convolution of a zero signal is zero), so the block
    returns rms(h, norm) of its input rows; a nonzero o changes that."""
    g, w = _tiny()
    zero = lambda m: dataclasses.replace(m, codes=np.full_like(m.codes, 0x88))
    wz = dict(w, layers=[dict(L, o=zero(L["o"]), down=zero(L["down"])) for L in w["layers"]])
    o = O.Oracle(g, wz)
    o.settle(0, di.make_taps(g, 0, 20))
    h = di.block_rows(g, 0, 5)
    want = [[hv * wv / math.sqrt(sum(t * t for t in row) / g.hidden + g.eps) for hv, wv in zip(row, w["norm"])]
            for row in np.asarray(h, dtype=np.float64)]
    assert np.allclose(o.block(20, h), want, rtol=1e-12, atol=0)
    full = O.Oracle(g, dict(wz, layers=[dict(L, o=w["layers"][i]["o"]) for i, L in enumerate(wz["layers"])]))
    full.settle(0, di.make_taps(g, 0, 20))
    assert not np.allclose(full.block(20, h), want, rtol=1e-6, atol=0)


def test_block_with_empty_context():
    g, w = _tiny()
    o = O.Oracle(g, w)
    hn = o.block(0, di.block_rows(g, 0, 3))
    assert hn.shape == (g.block, g.hidden) and np.all(np.isfinite(hn))


def test_settle_rows_are_independent_and_values_position_free():
    g, w = _tiny()
    taps = di.make_taps(g, 0, 12)
    a = O.Oracle(g, w)
    a.settle(0, taps)
    b = O.Oracle(g, w)
    b.settle(0, taps[:5]); b.settle(5, taps[5:])
    assert np.allclose(a.ctx_k[0], b.ctx_k[0], rtol=0, atol=1e-13)
    _, kv0 = a.settle_rows(0, taps[:3])
    _, kv9 = a.settle_rows(100, taps[:3])
    assert np.array_equal(kv0[0][1], kv9[0][1])                      # V has no position
    inv = O.inv_freq(g.head_dim, g.rope_theta)
    # row 0 sits at position 0, where the rotation is the identity
    k_at_100 = O.rotate(kv0[0][0][:1].reshape(1, -1), g.kv_heads, [100], inv)
    assert np.allclose(kv9[0][0][:1].reshape(1, -1), k_at_100, rtol=0, atol=1e-13)


def test_settle_replaces_rows_from_pos_on():
    g, w = _tiny()
    taps = di.make_taps(g, 0, 10)
    other = di.make_taps(g, 1, 4)
    a = O.Oracle(g, w)
    a.settle(0, taps)
    a.settle(6, other)
    b = O.Oracle(g, w)
    b.settle(0, np.concatenate([taps[:6], other]))
    assert a.len == 10 and np.allclose(a.ctx_k[0], b.ctx_k[0], rtol=0, atol=1e-13)


def test_inputs_are_seeded():
    g = di.workload("tiny").geometry
    assert np.array_equal(di.make_taps(g, 3, 70)[64:], di.make_taps(g, 3, 6, start=64))
    assert not np.array_equal(di.make_taps(g, 3, 4), di.make_taps(g, 4, 4))


# ------------------------------------------------------------------ composition of the pass
# The primitives above are pinned on their own; these pin how the pass wires
# them: which block rows reach the head, the order of the settle's steps and
# which convolution kernel each residual add uses.

def _one_hot_int4(rows: int, cols: int, group: int, col_of, scale: float) -> "di.Int4":
    """A four-bit matrix with the single code +1 at (r, col_of(r)) of every row, scale `scale`."""
    q = np.zeros((rows, cols), dtype=np.int64)
    for r in range(rows):
        q[r, col_of(r)] = 1
    scales = np.full((rows, cols // group), scale, dtype=np.float16)
    return di.Int4(codes=_pack(q), scales=scales, rows=rows, cols=cols, group=group)


def test_head_and_selector_read_block_rows_one_to_k():
    """gpu dflash.rs ``Dev::block``: the head and the selector's projection take the
    final-normed rows 1..=k of the block (the anchor row 0 gets no logits), the head
    over its first ``width`` rows. With a head whose row v is the unit vector e_v and
    distinct rows hn[r][c] = 100 r + c, logit[j][v] must be hn[j + 1][v]."""
    g, w = _tiny()
    hs = g.hidden
    hn = np.array([[100.0 * r + c for c in range(hs)] for r in range(g.block)])
    rows = 48
    head = _one_hot_int4(rows, hs, g.quant_group, lambda r: r, 1.0)
    sel = np.zeros((g.selector_rank, hs), dtype=np.float16)
    for i in range(g.selector_rank):
        sel[i, 3 * i] = 1.0                      # hp[j][i] = f16(hn[j + 1][3 i]): exact integers < 2048
    o = O.Oracle(g, dict(w, head=head, sel=sel))
    for k, width in ((g.block - 1, rows), (4, 17)):
        lg = o.head_logits(hn, k, width)
        assert lg.shape == (k, width)
        assert np.array_equal(lg, [[100.0 * (j + 1) + v for v in range(width)] for j in range(k)])
        hp = o.selector_projection(hn, k)
        assert np.array_equal(hp, [[100.0 * (j + 1) + 3 * i for i in range(g.selector_rank)] for j in range(k)])


def test_settle_rows_closed_form_norm_then_rotation():
    """dflash.rs ``Drafter::settle_rows`` / gpu dflash.rs ``Dev::settle`` on matrices with a
    closed form: fc the identity on the first tap, so t = rms(f16(tap0), hidden_norm) (the
    norm after the fc, over its hidden outputs); Wk and Wv single codes, so k = s_k t and
    v = s_v t on the first kv_heads*head_dim channels; K = the head's RMS norm times k_norm
    (non-uniform), THEN the half-split rotation to pos + r. Normalising after the rotation,
    or norming the raw taps, or leaving out hidden_norm, each breaks an equality here."""
    g, w = _tiny()
    hs, hd, kvd, tw = g.hidden, g.head_dim, g.kv_heads * g.head_dim, g.tap_width
    fc = np.zeros((hs, tw), dtype=np.float16)
    fc[np.arange(hs), np.arange(hs)] = 1.0
    hidden_norm = (1.0 + np.arange(hs) / 64.0).astype(np.float32)
    L = dict(w["layers"][0])
    L["k_norm"] = (0.5 + np.arange(hd) / 16.0).astype(np.float32)
    L["k"] = _one_hot_int4(kvd, hs, g.quant_group, lambda r: r, 0.5)
    L["v"] = _one_hot_int4(kvd, hs, g.quant_group, lambda r: (r + 7) % hs, 0.25)
    o = O.Oracle(g, dict(w, fc=fc, hidden_norm=hidden_norm, layers=[L]))
    n, pos = 5, 37
    taps = di.make_taps(g, 4, n)
    _, kv = o.settle_rows(pos, taps)
    K, V = kv[0]
    eps = g.eps
    inv = [np.float32(g.rope_theta ** (-(2.0 * i) / hd)) for i in range(hd // 2)]
    for r in range(n):
        t0 = [float(np.float16(x)) for x in taps[r, :hs]]
        s = 1.0 / math.sqrt(sum(x * x for x in t0) / hs + eps)
        t = [t0[i] * s * float(hidden_norm[i]) for i in range(hs)]
        for h in range(g.kv_heads):
            for i in range(hd):
                assert abs(V[r, h, i] - 0.25 * t[(h * hd + i + 7) % hs]) <= 1e-12 * abs(t[(h * hd + i + 7) % hs]) + 1e-15
            k = [0.5 * t[h * hd + i] for i in range(hd)]
            sk = 1.0 / math.sqrt(sum(x * x for x in k) / hd + eps)
            kn = [k[i] * sk * float(L["k_norm"][i]) for i in range(hd)]
            for i in range(hd // 2):
                ang = float(np.float32(np.float32(pos + r) * inv[i]))
                c, sn = math.cos(ang), math.sin(ang)
                a, b = kn[i], kn[i + hd // 2]
                assert abs(K[r, h, i] - (a * c - b * sn)) <= 1e-12
                assert abs(K[r, h, i + hd // 2] - (b * c + a * sn)) <= 1e-12


def _scaled(m, factor: float):
    """The same codes with every scale multiplied by a power of two (exact in f16)."""
    return dataclasses.replace(m, scales=(m.scales.astype(np.float32) * factor).astype(np.float16))


def _layer_delta(g, w, layers):
    """The residual stream's change over the (single) layer: h after the layer minus h before."""
    o = O.Oracle(g, dict(w, layers=layers))
    o.settle(0, di.make_taps(g, 0, 20))
    h = di.block_rows(g, 0, 5)
    tr = {}
    o.block(20, h, tr)
    return tr["layers"][0]["h"] - np.asarray(h, np.float64), tr["layers"][0]


def test_attention_conv_out_uses_the_stage0_kernel_and_is_linear_in_o():
    """dflash.rs ``Drafter::block``: the attention's stage-1 convolution (conv_out) applies the
    kernel d computed from the sub-layer's input x (conv_in's d), not one computed from its
    own signal o. So with the MLP silenced (down = 0), doubling Wo doubles the residual
    change exactly, and changing only the stage-1 rows of attn_proj leaves q, k, v, y and
    o untouched while the residual change moves."""
    g, w = _tiny()
    zero = lambda m: dataclasses.replace(m, codes=np.full_like(m.codes, 0x88))
    L = dict(w["layers"][0], down=zero(w["layers"][0]["down"]))
    d1, t1 = _layer_delta(g, w, [L])
    d2, _ = _layer_delta(g, w, [dict(L, o=_scaled(L["o"], 2.0))])
    assert np.abs(d1).max() > 1e-3
    assert np.allclose(d2, 2.0 * d1, rtol=1e-12, atol=1e-12)
    stage1 = g.conv_kernel * g.groups                      # rows [stage 1][offset][group] of the projection
    ap = L["attn_proj"].copy()
    ap[stage1:] = (ap[stage1:].astype(np.float32) * 2.0).astype(np.float16)
    d3, t3 = _layer_delta(g, w, [dict(L, attn_proj=ap)])
    for name in ("x", "xc", "q", "k", "v", "y", "o"):
        assert np.array_equal(t1[name], t3[name]), name
    assert not np.allclose(d3, d1, rtol=1e-6, atol=0)


def test_mlp_conv_out_uses_the_mlp_kernel_not_the_attention_one():
    """dflash.rs ``Drafter::block``: the MLP's stage-1 convolution reuses md, the kernel of the
    MLP's own stage-0 input, not the attention's ad. With the attention silenced (o = 0), the
    stage-1 rows of attn_proj reach nothing; those of mlp_proj do; and doubling down doubles
    the residual change."""
    g, w = _tiny()
    zero = lambda m: dataclasses.replace(m, codes=np.full_like(m.codes, 0x88))
    L = dict(w["layers"][0], o=zero(w["layers"][0]["o"]))
    stage1 = g.conv_kernel * g.groups
    d1, t1 = _layer_delta(g, w, [L])
    assert np.abs(d1).max() > 1e-3
    ap = L["attn_proj"].copy()
    ap[stage1:] = 0
    d2, _ = _layer_delta(g, w, [dict(L, attn_proj=ap)])
    assert np.array_equal(d2, d1)
    mp = L["mlp_proj"].copy()
    mp[stage1:] = 0
    d3, t3 = _layer_delta(g, w, [dict(L, mlp_proj=mp)])
    assert np.array_equal(t1["dn"], t3["dn"]) and not np.allclose(d3, d1, rtol=1e-6, atol=0)
    d4, _ = _layer_delta(g, w, [dict(L, down=_scaled(L["down"], 2.0))])
    assert np.allclose(d4, 2.0 * d1, rtol=1e-12, atol=1e-12)


def test_select_scores_agree_with_select_with():
    """The per-candidate scores the token checker uses (``select_scores``) give, row by row
    along select_with's own chain, the token select_with chose (first strictly greater
    score in candidate order), and each score is the brute-force sum
    logit + sum_i P[prev][i] hp[i] C[cand][i]."""
    rng = np.random.default_rng(11)
    V, rank, top, k = 50, 4, 6, 7
    for trial in range(20):
        logits = rng.standard_normal((k, V))
        if trial % 4 == 0:
            logits[:, 3] = logits[:, 9] = logits.max() + 1.0          # an exact tie at the top
        hp = rng.standard_normal((k, rank))
        P = rng.standard_normal((V, rank)).astype(np.float16)
        Cb = rng.standard_normal((V, rank)).astype(np.float16)
        anchor = int(rng.integers(0, V))
        chosen, plain = O.select_with(hp, logits, anchor, P, Cb, top)
        prevs = [anchor] + chosen[:-1]
        scores = O.select_scores(hp, logits, prevs, P, Cb, top)
        for j in range(k):
            best_t, best_s = None, -np.inf
            for tok, s in scores[j]:
                want = logits[j, tok] + sum(float(P[prevs[j], i]) * hp[j, i] * float(Cb[tok, i]) for i in range(rank))
                assert abs(s - want) <= 1e-12 * max(1.0, abs(want))
                if s > best_s:
                    best_t, best_s = tok, s
            assert best_t == chosen[j]
            assert scores[j][0][0] == plain[j]


# ------------------------------------------------------------------ context bookkeeping
# Sequences worked by hand from dflash.rs: `Drafter::queue_context` (a gap starts over, a
# held position truncates, past the pending limit the oldest rows settle in multiples of
# CONTEXT_CHUNK), `settle`, `truncate` and the window trim at the end of `settle_rows`
# (a layer holding more than twice its window keeps its last `window` rows).

def _kv_of(o, pos, taps):
    return o.settle_rows(pos, taps)[1]


def test_window_trim_and_truncate_worked_sequence():
    g, w = _tiny(windows=(8,))
    taps = di.make_taps(g, 2, 40)
    o = O.Oracle(g, w)
    o.settle(0, taps[:20])                 # held 20 > 16: keeps 8, dropped 12
    assert (o.len, o.dropped) == (20, [12])
    k, v = _kv_of(o, 12, taps[12:20])[0]
    assert np.allclose(o.ctx_k[0], k, rtol=0, atol=1e-13) and np.allclose(o.ctx_v[0], v, rtol=0, atol=1e-13)
    o.settle(20, taps[20:25])              # held 13: nothing let go
    assert (o.len, o.dropped, len(o.ctx_k[0])) == (25, [12], 13)
    o.settle(25, taps[25:29])              # held 17 > 16: keeps 8, dropped 21
    assert (o.len, o.dropped, len(o.ctx_k[0])) == (29, [21], 8)
    o.truncate(27)                         # keeps positions 21..26
    assert (o.len, o.dropped, len(o.ctx_k[0])) == (27, [21], 6)
    o.truncate(10)                         # below what the layer holds: it holds nothing from 10 on
    assert (o.len, o.dropped, len(o.ctx_k[0])) == (10, [10], 0)
    o.settle(10, taps[30:33])              # new rows at 10..12
    assert (o.len, o.dropped, len(o.ctx_k[0])) == (13, [10], 3)
    k, v = _kv_of(o, 10, taps[30:33])[0]
    assert np.allclose(o.ctx_k[0], k, rtol=0, atol=1e-13)
    assert O.context_range(o.first, o.len, 13, 8, o.dropped[0]) == (10, 13)


def test_queue_pending_limit_gap_and_truncate_worked_sequence():
    g, w = _tiny()                          # window 0: the pending limit is 512
    assert O.pending_limit(g) == 512
    assert O.pending_limit(dataclasses.replace(g, windows=(600,))) == 856
    assert O.pending_limit(dataclasses.replace(g, windows=(100,))) == 512
    taps = di.make_taps(g, 3, 620)
    o = O.Oracle(g, w)
    o.queue(0, taps[:600])                 # 600 > 512: the oldest 128 settle (88 rounded up to 64s)
    assert (o.len, len(o.pending), o.next_position()) == (128, 472, 600)
    o.queue(600, taps[600:610])
    assert (o.len, len(o.pending)) == (128, 482)
    o.queue(300, taps[610:615])            # a held position: waiting rows from 300 on go
    assert (o.len, len(o.pending), o.next_position()) == (128, 177, 305)
    o.truncate(100)
    assert (o.len, len(o.pending)) == (100, 0)
    ref = O.Oracle(g, w)
    ref.settle(0, taps[:100])
    assert np.allclose(o.ctx_k[0], ref.ctx_k[0], rtol=0, atol=1e-13)
    o.queue(2000, taps[:3])                # a gap: the context starts over at 2000
    assert (o.first, o.len, len(o.pending)) == (2000, 0, 3)
    o.settle_pending()
    assert (o.first, o.len) == (2000, 3)
    k, _ = _kv_of(o, 2000, taps[:3])[0]
    assert np.allclose(o.ctx_k[0], k, rtol=0, atol=1e-13)
    o.queue(1500, taps[3:4])               # before first: a gap as well
    assert (o.first, o.len, len(o.pending)) == (1500, 0, 1)


def test_queued_rows_equal_settled_rows_and_blocks_wait_for_them():
    g, w = _tiny()
    taps = di.make_taps(g, 4, 90)
    a, b = O.Oracle(g, w), O.Oracle(g, w)
    a.settle(0, taps)
    for i in range(0, 90, 30):
        b.queue(i, taps[i:i + 30])
    with pytest.raises(AssertionError):
        b.block(90, di.block_rows(g, 0, 1))
    b.settle_pending()
    assert b.len == 90 and np.allclose(a.ctx_k[0], b.ctx_k[0], rtol=0, atol=1e-13)
    assert np.array_equal(a.block(90, di.block_rows(g, 0, 1)), b.block(90, di.block_rows(g, 0, 1)))


def test_pushed_rows_equal_settled_rows():
    """Rows imported with their keys and values (`Dev::push_rows`) are the context a settle of
    the same taps makes, the bookkeeping (trim included) the same."""
    g, w = _tiny(windows=(8,))
    taps = di.make_taps(g, 5, 30)
    a, b = O.Oracle(g, w), O.Oracle(g, w)
    a.settle(0, taps[:20])
    a.settle(20, taps[20:30])
    b.push_rows(0, _kv_of(b, 0, taps[:20]))
    b.push_rows(20, _kv_of(b, 20, taps[20:30]))
    assert (a.len, a.dropped) == (b.len, b.dropped) == (30, [22])   # 20 held: 8 kept; then 18: 8 kept
    assert np.allclose(a.ctx_k[0], b.ctx_k[0], rtol=0, atol=1e-13)
    assert np.allclose(a.block(30, di.block_rows(g, 0, 3)), b.block(30, di.block_rows(g, 0, 3)), rtol=0, atol=1e-12)


# ------------------------------------------------------------------ router margin

def _orthonormal_rows(rng, rank, hidden):
    """`rank` distinct rows of the Sylvester-Hadamard matrix over sqrt(hidden) (hidden a power of
    4): entries +-1/8 at 64, exact in f16, so the rows are exactly orthonormal."""
    H = np.array([[1.0]])
    while H.shape[0] < hidden:
        H = np.block([[H, H], [H, -H]])
    rows = rng.choice(hidden, size=rank, replace=False)
    return (H[rows] / np.sqrt(hidden)).astype(np.float16)


def test_recon_error_closed_forms():
    rng = np.random.default_rng(21)
    hs, rank = 64, 5
    B = _orthonormal_rows(rng, rank, hs)
    m = (rng.standard_normal(hs) * 0.1).astype(np.float16)
    Bf, mf = B.astype(np.float64), m.astype(np.float64)
    # a row inside the affine subspace is held exactly
    inside = mf + Bf.T @ rng.standard_normal(rank)
    assert O.recon_error(inside, m, B) < 1e-20
    # rank 0: the whole offset from the mean
    x = rng.standard_normal(hs)
    assert O.recon_error(x, m, np.zeros((0, hs), np.float16)) == pytest.approx(float((x - mf) @ (x - mf)), rel=1e-12)
    # against least squares (the distance to the span, by another route)
    coef, *_ = np.linalg.lstsq(Bf.T, x - mf, rcond=None)
    res = (x - mf) - Bf.T @ coef
    assert O.recon_error(x, m, B) == pytest.approx(float(res @ res), rel=1e-9)


def test_route_margin_closed_forms():
    rng = np.random.default_rng(22)
    hs = 64
    Bb, Bc = _orthonormal_rows(rng, 4, hs), _orthonormal_rows(rng, 6, hs)
    mb, mc = np.zeros(hs, np.float16), np.zeros(hs, np.float16)
    # a row along the block's first basis row: the block holds it, the chain does not
    row = 3.0 * Bb[0].astype(np.float64)
    m = O.route_margin(row, mb, Bb, mc, Bc)
    u = Bb[0].astype(np.float64) / np.linalg.norm(Bb[0].astype(np.float64))
    assert m == pytest.approx(O.recon_error(u, mc, Bc), abs=1e-9) and m > 0
    # scale-free, antisymmetric in the two subspaces, zero row guarded
    x = rng.standard_normal(hs)
    assert O.route_margin(x, mb, Bb, mc, Bc) == pytest.approx(O.route_margin(7.5 * x, mb, Bb, mc, Bc), rel=1e-12)
    assert O.route_margin(x, mb, Bb, mc, Bc) == pytest.approx(-O.route_margin(x, mc, Bc, mb, Bb), rel=1e-12)
    zero = O.route_margin(np.zeros(hs), mb, Bb, mc, Bc)
    assert zero == pytest.approx(0.0, abs=1e-12)        # both errors are |0 - mean|^2 = 0

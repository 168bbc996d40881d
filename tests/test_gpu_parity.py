"""Parity of the CUDA path (through the C ABI) with the CPU oracle, on seeded synthetic inputs."""
import dataclasses

import numpy as np
import pytest

import dflash_inputs as di
from oracle import dflash_oracle as O
from parity import LOGIT_REL, check_close, check_tokens, rel_err

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_block_drafter_gb300 import build
    build.build()


@pytest.fixture(autouse=True)
def no_device_error():
    """No kernel of the library may give up a bounded wait."""
    from speculative_block_drafter_gb300 import _lib as L
    yield
    torch.cuda.synchronize()
    assert L.dflash_device_error(reset=True) == 0


def _drafter():
    from speculative_block_drafter_gb300 import drafter
    return drafter


def _rand_int4(rng, rows, cols, group, zero_groups=False):
    q = rng.integers(-7, 8, size=(rows, cols))
    scales = (rng.random((rows, cols // group)) * 0.05 + 1e-3).astype(np.float16)
    if zero_groups:
        scales[::3, ::2] = 0
        q.reshape(rows, cols // group, group)[::3, ::2, :] = 0
    u = (q + 8).astype(np.uint8)
    codes = (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)
    return di.Int4(codes=codes, scales=scales, rows=rows, cols=cols, group=group)


# ------------------------------------------------------------------ dequant and GEMMs

@pytest.mark.parametrize("rows,cols,group", [(16, 64, 32), (48, 256, 64), (32, 384, 128), (160, 1024, 64)])
def test_dequant_bit_exact(rows, cols, group):
    rng = np.random.default_rng(rows + cols)
    m = _rand_int4(rng, rows, cols, group, zero_groups=True)
    got = _drafter().dequant_int4(m)
    ref = O.dequant_int4(m.codes, m.scales, group).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_dequant_bit_exact_generated_head():
    g = di.workload("tiny").geometry
    w = di.make_weights(g, 0)
    m = w["head"]
    got = _drafter().dequant_int4(m)
    ref = O.dequant_int4(m.codes, m.scales, m.group).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def _bound(wabs: np.ndarray, x: np.ndarray) -> float:
    return float((np.abs(x) @ wabs.T).max())


@pytest.mark.parametrize("rows,cols,group,T", [(16, 64, 32, 1), (64, 256, 64, 5), (48, 512, 128, 16),
                                               (96, 1024, 64, 17), (32, 2048, 64, 40), (2048, 5120, 64, 16),
                                               # many tokens: the split-weight kernel, one and two token tiles
                                               (300, 1024, 64, 256), (130, 512, 32, 100), (256, 768, 64, 480),
                                               (1024, 5120, 64, 256),
                                               # 19 row tiles, each one CTA's over its whole k-range
                                               (2432, 1024, 64, 256)])
def test_gemm_int4_matches_oracle(rows, cols, group, T):
    rng = np.random.default_rng(rows * 7 + T)
    m = _rand_int4(rng, rows, cols, group)
    x = rng.standard_normal((T, cols)).astype(np.float32)
    pm = _drafter().PackedMatrix(m)
    y = pm.matmul(torch.from_numpy(x).cuda()).cpu().numpy()
    ref = O.int4_matmul(m, x)
    wabs = np.abs(O.dequant_int4(m.codes, m.scales, group))
    err = np.abs(y - ref).max()
    assert err <= 2e-6 * _bound(wabs, x), (err, _bound(wabs, x))


@pytest.mark.parametrize("kind,rows,cols,T", [(4, 4096, 1024, 16), (4, 151936, 1024, 15), (4, 256, 17408, 32),
                                               (16, 1280, 5120, 16), (16, 512, 1024, 3)])
def test_gemm_packed_repeats_gemm(kind, rows, cols, T):
    """dflash_gemm_packed reruns dflash_gemm's kernel on the tiles it packed (whole and split k-ranges)."""
    from speculative_block_drafter_gb300.drafter import PackedMatrix
    rng = np.random.default_rng(rows + cols + T)
    if kind == 4:
        m = _rand_int4(rng, rows, cols, 64)
    else:
        m = (rng.standard_normal((rows, cols)) * 0.02).astype(np.float16)
    pm = PackedMatrix(m)
    x = torch.from_numpy(rng.standard_normal((T, cols)).astype(np.float32)).cuda()
    y1 = pm.matmul(x).clone()
    y2 = pm.matmul_packed(torch.full_like(y1, float("nan")))
    torch.cuda.synchronize()
    assert torch.allclose(y1, y2, rtol=1e-6, atol=1e-6 * float(y1.abs().max()))


@pytest.mark.parametrize("rows,cols,T", [(16, 64, 1), (64, 512, 16), (1280, 5120, 16), (128, 3072, 256), (64, 256, 33),
                                         (1024, 3072, 256), (200, 1024, 300), (5120, 2560, 256)])
def test_gemm_f16_matches_oracle(rows, cols, T):
    rng = np.random.default_rng(rows + cols + T)
    w = (rng.standard_normal((rows, cols)) / np.sqrt(cols)).astype(np.float16)
    x = rng.standard_normal((T, cols)).astype(np.float32)
    pm = _drafter().PackedMatrix(w)
    y = pm.matmul(torch.from_numpy(x).cuda()).cpu().numpy()
    ref = O.f16_matmul(w, x)
    err = np.abs(y - ref).max()
    assert err <= 2e-6 * _bound(np.abs(w.astype(np.float64)), x.astype(np.float16).astype(np.float64)), err


# ------------------------------------------------------------------ the pass

class Pair:
    """The GPU drafter and the oracle on the same weights, driven through the same calls."""

    def __init__(self, g, seed=0, max_batch=1, ctx_cap=4096, cache_format="planes", rings=None):
        self.g = g
        self.w = di.make_weights(g, seed)
        self.gpu = _drafter().Drafter(g, self.w, max_batch=max_batch, ctx_cap=ctx_cap, cache_format=cache_format,
                                      rings=rings)
        self.orc = [O.Oracle(g, self.w) for _ in range(max_batch)]
        # one f16 per element: the cache rounds each K/V value to 11 bits
        self.cache_rel = 1e-3 if cache_format == "f16" else 1e-4

    def settle(self, seq, pos, taps, chunk=1024):
        # each library call is one `push_context`: the oracle takes the same calls
        self.gpu.settle(seq, pos, torch.from_numpy(taps).cuda(), chunk=chunk)
        for i in range(0, len(taps), chunk):
            self.orc[seq].settle(pos + i, taps[i:i + chunk])

    def queue(self, seq, pos, taps, chunk=1024):
        self.gpu.queue(seq, pos, torch.from_numpy(taps).cuda(), chunk=chunk)
        for i in range(0, len(taps), chunk):
            self.orc[seq].queue(pos + i, taps[i:i + chunk])

    def settle_pending(self, seq):
        self.gpu.settle_pending(seq)
        self.orc[seq].settle_pending()

    def truncate(self, seq, pos):
        self.gpu.truncate(seq, pos)
        self.orc[seq].truncate(pos)

    def push_rows(self, seq, pos, kv):
        """kv: per layer (k, v) f64 [n][kv][hd] (the oracle's own rows), sent as f32."""
        k = [torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda() for a, _ in kv]
        v = [torch.from_numpy(np.ascontiguousarray(b, dtype=np.float32)).cuda() for _, b in kv]
        self.gpu.push_rows(seq, pos, k, v)
        self.orc[seq].push_rows(pos, [(a.astype(np.float32).astype(np.float64), b.astype(np.float32).astype(np.float64))
                                      for a, b in kv])

    def reset(self, seq, first):
        self.gpu.reset(seq, first)
        self.orc[seq].reset(first)

    def check_cache(self, seq=0):
        """The context's state and every layer's held rows against the oracle's."""
        torch.cuda.synchronize()
        o = self.orc[seq]
        f, n, pend, dropped = self.gpu.context_ex(seq)
        assert (f, n, pend, dropped) == (o.first, o.len, len(o.pending), o.dropped)
        worst = 0.0
        for l in range(self.g.layers):
            k, v = (t.cpu().numpy() for t in self.gpu.held_kv(seq, l))
            assert k.shape[0] == o.ctx_k[l].shape[0], (l, k.shape, o.ctx_k[l].shape)
            if k.shape[0]:
                worst = max(worst, check_close(f"K layer {l}", k, o.ctx_k[l], self.cache_rel),
                            check_close(f"V layer {l}", v, o.ctx_v[l], self.cache_rel))
        return worst

    def draft(self, anchors, hs_rows, anchor_toks, k=None, width=None, fused=False):
        """block + select (or, fused, dflash_draft) against the oracle's draft."""
        g = self.g
        k = g.block - 1 if k is None else k
        width = g.vocab if width is None else width
        h = torch.from_numpy(np.stack(hs_rows).astype(np.float32)).cuda().contiguous()
        at = torch.tensor(anchor_toks, dtype=torch.int32, device="cuda")
        if fused:
            logits, hp, chosen, plain = self.gpu.draft(anchors, h, at, k, width)
        else:
            logits, hp = self.gpu.block(anchors, h, k, width)
            chosen, plain = self.gpu.select(logits, hp, at)
        torch.cuda.synchronize()
        res = []
        for b in range(len(anchors)):
            _, lo, hpo, ch, pl = self.orc[b].draft(anchors[b], hs_rows[b], anchor_toks[b], k, width)
            lg = logits[b].cpu().numpy()
            hg = hp[b].cpu().numpy()
            el = check_close(f"logits seq {b}", lg, lo)
            eh = check_close(f"hp seq {b}", hg, hpo)
            ties = check_tokens(chosen[b].cpu().numpy(), plain[b].cpu().numpy(), hpo, lo, anchor_toks[b],
                                self.w["pred_book"], self.w["succ_book"], g.selector_top)
            res.append(dict(logit_err=el, hp_err=eh, ties=ties, chosen=chosen[b].cpu().numpy(),
                            oracle_chosen=np.array(ch)))
        return res


def _tiny(**over):
    return dataclasses.replace(di.workload("tiny").geometry, **over)


def test_settle_tiny_matches_oracle_with_ragged_chunks():
    g = _tiny()
    p = Pair(g, ctx_cap=1536)
    taps = di.make_taps(g, 0, 1301)
    p.settle(0, 0, taps[:1])            # one row
    p.settle(0, 1, taps[1:1300])        # 1024 + 275 rows, two calls
    p.settle(0, 1300, taps[1300:1301])
    assert p.check_cache() < 1e-4
    # rows at held positions replace them and what follows
    other = di.make_taps(g, 5, 40)
    p.settle(0, 200, other)
    assert p.check_cache() < 1e-4


def test_block_tiny_matches_oracle():
    wl = di.workload("tiny")
    g = wl.geometry
    p = Pair(g)
    p.settle(0, 0, di.make_taps(g, 0, wl.context))
    a = di.anchor_token(g, 0)
    r = p.draft([wl.context], [di.block_rows(g, 0, a)], [a])[0]
    # hp multiplies f16-rounded rows (as the oracle does): a one-ulp rounding flip moves it by ~1e-4
    assert r["logit_err"] < 1e-4 and r["hp_err"] < 5e-4


def test_cache_value_out_of_range_sets_the_error_word():
    """A K/V value of magnitude 65,536 or more does not fit the cache's hi plane: the settle
    writes infinity there and sets bit 1 (value 2) of the device error word. An ordinary
    settle of the same rows leaves the word clear."""
    from speculative_block_drafter_gb300 import _lib as L
    g = _tiny()
    w = di.make_weights(g, 0)
    taps = torch.from_numpy(di.make_taps(g, 0, 8)).cuda()
    d = _drafter().Drafter(g, w, max_batch=1, ctx_cap=64)
    d.settle(0, 0, taps)
    torch.cuda.synchronize()
    assert L.dflash_device_error(reset=True) == 0
    d.close()
    L0 = w["layers"][0]
    big = dataclasses.replace(L0["v"], scales=np.full_like(L0["v"].scales, 60000.0))
    d = _drafter().Drafter(g, dict(w, layers=[dict(L0, v=big)]), max_batch=1, ctx_cap=64)
    d.settle(0, 0, taps)
    torch.cuda.synchronize()
    assert L.dflash_device_error(reset=True) == 2
    k, v = d.context_kv(0, 0, 8)
    assert torch.isinf(v).any() and torch.isfinite(k).all()
    d.close()


@pytest.mark.parametrize("vocab", [4096, 151936])
def test_select_alone_on_identical_inputs(vocab):
    """The selector on the oracle's own logits and hp (f32): isolates it from the block.
    Rows of equal logits take the exact fallback (more candidates than a CTA holds)."""
    g = _tiny(vocab=vocab)
    rng = np.random.default_rng(3)
    w = di.make_weights(g, 0)
    d = _drafter().Drafter(g, w, max_batch=2, ctx_cap=64)
    k, width = g.block - 1, g.vocab
    logits = rng.standard_normal((2, k, width)).astype(np.float32)
    logits[0, 3, 10] = logits[0, 3, 20] = 9.0         # an exact tie: the lower index comes first
    logits[1, 5, :] = 0.5                              # a row of equal logits
    logits[0, 7, 100:3100] = 20.0                      # 3000 equal maxima
    hp = rng.standard_normal((2, k, g.selector_rank)).astype(np.float32)
    anchors = [5, 4000]
    ch, pl = d.select(torch.from_numpy(logits).cuda(), torch.from_numpy(hp).cuda(),
                      torch.tensor(anchors, dtype=torch.int32, device="cuda"))
    ch, pl = ch.cpu().numpy(), pl.cpu().numpy()
    for b in range(2):
        och, opl = O.select_with(hp[b], logits[b], anchors[b], w["pred_book"], w["succ_book"], g.selector_top)
        assert list(pl[b]) == opl
        check_tokens(ch[b], pl[b], hp[b].astype(np.float64), logits[b].astype(np.float64), anchors[b],
                     w["pred_book"], w["succ_book"], g.selector_top)
    assert pl[0, 3] == 10 and pl[1, 5] == 0 and pl[0, 7] == 100
    d.close()


@pytest.mark.parametrize("case", ["empty_context", "windowed", "short_k_shortlist", "no_rope_first_1000",
                                  "batch3", "rep4_long"])
def test_block_edge_cases(case):
    g = _tiny()
    seeds = [0]
    if case == "windowed":
        g = _tiny(windows=(40,))
    if case == "rep4_long":              # 4 query heads per KV head (64 queries a CTA), a longer context
        g = _tiny(heads=8, kv_heads=2, windows=(300,))
    if case == "no_rope_first_1000":
        g = _tiny(no_rope=(0,))
    batch = 3 if case == "batch3" else 1
    p = Pair(g, max_batch=batch, ctx_cap=1024)
    anchors, rows, toks, k, width = [], [], [], None, None
    for b in range(batch):
        first, n = 0, (700 if case == "rep4_long" else 100 + 37 * b)
        if case == "no_rope_first_1000":
            first = 1000
        p.reset(b, first)
        if case != "empty_context":
            p.settle(b, first, di.make_taps(g, b, n))
        else:
            n = 0
        a = first + n
        if case == "windowed":
            a = 90                       # anchored inside the context: rows at and after it are excluded
        tok = di.anchor_token(g, b + 1)
        anchors.append(a)
        rows.append(di.block_rows(g, b, tok))
        toks.append(tok)
    if case == "short_k_shortlist":
        k, width = 3, 1024
    for r in p.draft(anchors, rows, toks, k, width):
        assert r["logit_err"] < 1e-4


def test_full_qwen3_0p6b_workload():
    """The qwen3-0.6b workload: 1024 positions settled in 256-row calls (as the bench settles),
    then one block and the selector."""
    wl = di.workload("qwen3-0.6b")
    g = wl.geometry
    p = Pair(g, ctx_cap=wl.context + 256)
    p.settle(0, 0, di.make_taps(g, 0, wl.context), chunk=256)
    assert p.check_cache() < 1e-4
    a = di.anchor_token(g, 0)
    r = p.draft([wl.context], [di.block_rows(g, 0, a)], [a])[0]
    # both sides round the kernel projections' inputs to f16, so a 1e-6 difference in the
    # cache can flip one of them by an ulp (~5e-4 of that element); the contract is LOGIT_REL
    assert r["logit_err"] < 5e-4, r


def test_full_27b_workload():
    """The 27b workload at full size: 4096 positions settled in 256-row calls (as the bench
    settles), windowed and no-rope layers, one block over the whole head and the selector."""
    wl = di.workload("27b")
    g = wl.geometry
    p = Pair(g, seed=wl.seed, ctx_cap=wl.context + 256)
    p.settle(0, 0, di.make_taps(g, wl.seed, wl.context), chunk=256)
    assert p.check_cache() < 1e-4
    a = di.anchor_token(g, wl.seed)
    r = p.draft([wl.context], [di.block_rows(g, wl.seed, a)], [a])[0]
    assert r["logit_err"] < LOGIT_REL, r
    # dflash_draft: the head's GEMM finds the selector's chunk maxima itself
    r = p.draft([wl.context], [di.block_rows(g, wl.seed, a)], [a], fused=True)[0]
    assert r["logit_err"] < LOGIT_REL, r


@pytest.mark.parametrize("name,k,width", [("qwen3-0.6b", 15, None), ("qwen3-0.6b", 7, 100000), ("tiny", 15, None)])
def test_draft_equals_block_then_select(name, k, width):
    """dflash_draft gives the logits, hp and tokens of dflash_block then dflash_select
    (the head's chunk maxima in the GEMM when it takes whole k-ranges, the selector's
    own first stage otherwise: tiny's 4096-row head); the tokens also against the oracle."""
    wl = di.workload(name)
    g = wl.geometry
    p = Pair(g, seed=wl.seed, ctx_cap=wl.context + 256)
    p.settle(0, 0, di.make_taps(g, wl.seed, wl.context), chunk=256)
    a = di.anchor_token(g, wl.seed)
    rows = di.block_rows(g, wl.seed, a)
    width = g.vocab if width is None else width
    h = torch.from_numpy(rows[None].astype(np.float32)).cuda().contiguous()
    at = torch.tensor([a], dtype=torch.int32, device="cuda")
    lb, hb = p.gpu.block([wl.context], h, k, width)
    cb, pb = p.gpu.select(lb, hb, at)
    lb, hb, cb, pb = lb.clone(), hb.clone(), cb.clone(), pb.clone()
    ld, hd, cd, pd = p.gpu.draft([wl.context], h, at, k, width)
    torch.cuda.synchronize()
    # the block pass is the same launch sequence, but split GEMMs add with atomics: two
    # passes agree to rounding, which an f16 rounding of a kernel projection's input can
    # turn into about 5e-4 of a logit (the bar of the 0.6B workload's logits)
    assert float((ld - lb).abs().max()) <= 5e-4 * float(lb.abs().max())
    assert float((hd - hb).abs().max()) <= 5e-4 * float(hb.abs().max())
    if torch.equal(ld, lb) and torch.equal(hd, hb):
        assert torch.equal(cd, cb) and torch.equal(pd, pb)
    r = p.draft([wl.context], [rows], [a], k, width, fused=True)[0]
    assert r["logit_err"] < LOGIT_REL, r


def test_full_batched_workload_sampled_sequences():
    """The batched workload at full size (32 sequences of 8192 settled positions, one block of
    512 rows through the wide GEMMs and the split attention); the oracle recomputes three of the
    sequences from their own taps."""
    wl = di.workload("batched")
    g, B = wl.geometry, wl.batch
    w = di.make_weights(g, wl.seed)
    d = _drafter().Drafter(g, w, max_batch=B, ctx_cap=wl.context + g.block)
    for s in range(B):
        d.reset(s, 0)
        d.settle(s, 0, torch.from_numpy(di.make_taps(g, wl.seed + s, wl.context)).cuda())
    toks = [di.anchor_token(g, wl.seed + s) for s in range(B)]
    rows = [di.block_rows(g, wl.seed + s, toks[s]) for s in range(B)]
    h = torch.from_numpy(np.stack(rows).astype(np.float32)).cuda().contiguous()
    k = g.block - 1
    logits, hp = d.block([wl.context] * B, h, k, g.vocab)
    chosen, plain = d.select(logits, hp, torch.tensor(toks, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    for s in (0, 17, B - 1):
        o = O.Oracle(g, w)
        o.settle(0, di.make_taps(g, wl.seed + s, wl.context))
        _, lo, hpo, _, _ = o.draft(wl.context, rows[s], toks[s], k, g.vocab)
        check_close(f"logits seq {s}", logits[s].cpu().numpy(), lo)
        check_close(f"hp seq {s}", hp[s].cpu().numpy(), hpo)
        check_tokens(chosen[s].cpu().numpy(), plain[s].cpu().numpy(), hpo, lo, toks[s], w["pred_book"],
                     w["succ_book"], g.selector_top)
    d.close()


def test_full_settle_heavy_workload():
    """The settle-heavy workload at full size, in the bench's launch configuration: 32,768
    positions settled in 256-row calls (the oracle in 4096-row slices of the same taps), every
    layer over the whole context, one block over the whole head and the selector."""
    wl = di.workload("settle-heavy")
    g = wl.geometry
    p = Pair(g, seed=wl.seed, ctx_cap=wl.context + g.block)
    for start in range(0, wl.context, 4096):
        p.settle(0, start, di.make_taps(g, wl.seed, 4096, start), chunk=256)
    assert p.check_cache() < 1e-4
    a = di.anchor_token(g, wl.seed)
    r = p.draft([wl.context], [di.block_rows(g, wl.seed, a)], [a])[0]
    assert r["logit_err"] < LOGIT_REL, r


# ------------------------------------------------------------------ context bookkeeping, rings, f16 caches

@pytest.mark.parametrize("fmt,rings", [("planes", None), ("planes", "window"), ("f16", None), ("f16", "window")])
def test_bookkeeping_against_oracle(fmt, rings):
    """dflash.rs `Drafter`: settles that trim a windowed layer, queued rows past the pending
    limit, truncation below the held rows, a gap, imported rows; the caches linear or rings
    of twice the window (the rows wrap many times), two planes or one f16; each state and
    the blocks (anchored at the end and inside the context) against the oracle."""
    g = _tiny(windows=(40,))
    p = Pair(g, ctx_cap=4096, cache_format=fmt, rings=rings)
    p.gpu.bind_pending(0)
    taps = di.make_taps(g, 7, 1600)
    a = di.anchor_token(g, 3)
    rows = di.block_rows(g, 3, a)

    def draft(anchor):
        # planes: an f16 rounding flip of a kernel-projection input (both sides round) moves an
        # element by about 5e-4 of its value; one f16 per cache element: the contract's bound
        r = p.draft([anchor], [rows], [a])[0]
        assert r["logit_err"] < (LOGIT_REL if fmt == "f16" else 5e-4), r

    p.settle(0, 0, taps[:100], chunk=37)            # trims after the third call
    assert p.check_cache() < p.cache_rel
    draft(100)
    p.queue(0, 100, taps[100:160])
    p.truncate(0, 130)                               # waiting rows past 130 go
    p.settle_pending(0)
    assert p.check_cache() < p.cache_rel
    p.truncate(0, 70)                                # below the rows the layer holds
    p.settle(0, 70, taps[160:170])
    assert p.check_cache() < p.cache_rel
    draft(80)
    p.queue(0, 80, taps[170:770], chunk=300)          # past the 512-row limit: the oldest 128 settle
    assert p.gpu.context_ex(0)[2] == p.orc[0].pending.__len__() == 472
    p.settle_pending(0)
    assert p.check_cache() < p.cache_rel
    draft(680)
    draft(650)                                       # anchored inside the context
    kv = p.orc[0].settle_rows(680, taps[800:830])[1]
    p.push_rows(0, 680, kv)
    assert p.check_cache() < p.cache_rel
    draft(710)
    p.settle(0, 5000, taps[900:1000], chunk=64)       # a gap: the context starts over at 5000
    assert p.check_cache() < p.cache_rel
    draft(5100)


def test_block_refuses_waiting_rows():
    from speculative_block_drafter_gb300 import _lib as L
    g = _tiny()
    p = Pair(g, ctx_cap=256)
    p.gpu.bind_pending(0)
    p.queue(0, 0, di.make_taps(g, 1, 20))
    with pytest.raises(L.DflashError) as e:
        p.gpu.block([20], torch.from_numpy(di.block_rows(g, 0, 1)[None]).cuda().contiguous())
    assert e.value.code == 2 and "wait" in str(e.value)
    p.settle_pending(0)
    assert p.check_cache() < 1e-4


def test_full_27b_windows_f16_rings():
    """The 27b geometry with one-f16 caches and rings of twice the window for its four
    windowed layers (the no-rope layer 2 keeps a linear cache): 6,144 positions settled in
    256-row calls, so that the rings wrap and the window trim lets rows go; then one block
    over the whole head and the selector, against the oracle."""
    wl = di.workload("27b")
    g = wl.geometry
    n = 6144
    p = Pair(g, seed=wl.seed, ctx_cap=n + 256, cache_format="f16", rings="window")
    taps = di.make_taps(g, wl.seed, n)
    p.settle(0, 0, taps, chunk=256)
    assert p.check_cache() < 1e-3
    a = di.anchor_token(g, wl.seed)
    r = p.draft([n], [di.block_rows(g, wl.seed, a)], [a])[0]
    assert r["logit_err"] < LOGIT_REL, r


# ------------------------------------------------------------------ router margin

def test_route_margin_matches_oracle():
    """`Route::margin` on the 27B hidden size: rank-64 block and rank-48 chain subspaces with
    near-orthonormal f16 bases and small means; random rows, a row inside the block subspace
    (margin well above zero), one inside the chain's (below zero) and a zero row."""
    from speculative_block_drafter_gb300.drafter import Router
    rng = np.random.default_rng(31)
    hs = 5120
    qb, _ = np.linalg.qr(rng.standard_normal((hs, 64)))
    qc, _ = np.linalg.qr(rng.standard_normal((hs, 48)))
    Bb, Bc = qb.T.astype(np.float16), qc.T.astype(np.float16)
    mb = (rng.standard_normal(hs) * 0.002).astype(np.float16)
    mc = (rng.standard_normal(hs) * 0.002).astype(np.float16)
    rows = rng.standard_normal((37, hs)).astype(np.float32)
    rows[3] = (Bb.astype(np.float64).T @ rng.standard_normal(64)).astype(np.float32)
    rows[4] = (Bc.astype(np.float64).T @ rng.standard_normal(48)).astype(np.float32)
    rows[5] = 0.0
    got = Router(mb, Bb, mc, Bc).margin(torch.from_numpy(rows).cuda()).cpu().numpy()
    ref = np.array([O.route_margin(r, mb, Bb, mc, Bc) for r in rows])
    assert np.abs(got - ref).max() <= 2e-5 * max(1.0, np.abs(ref).max()), np.abs(got - ref).max()
    assert ref[3] > 0.5 and ref[4] < -0.5 and got[3] > 0.5 and got[4] < -0.5

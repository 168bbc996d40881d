"""dflash_select_static: the selector for callers that cannot allocate device memory
(a framework's memory pool owning the device heap, decode loops that must not
synchronise the device through cudaMalloc, foreign-function callers without a
device allocator). Its candidate scratch is a fixed array inside the library,
so it takes no workspace. It must give exactly what dflash_select gives, and
what the oracle's selector gives on the same inputs, call after call, although
every call reuses the same array; and its calls must leave the device's memory
use as they found it."""
import dataclasses

import numpy as np
import pytest

import dflash_inputs as di
from oracle import dflash_oracle as O
from parity import check_tokens

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_block_drafter_gb300 import build
    build.build()


def _inputs(rng, batch, k, width, rank, tie=False):
    logits = rng.standard_normal((batch, k, width)).astype(np.float32)
    if tie:
        logits[0, 2, 7] = logits[0, 2, 1500 % width] = 10.0   # equal values: the lower index first
    hp = rng.standard_normal((batch, k, rank)).astype(np.float32)
    return logits, hp


@pytest.mark.parametrize("vocab,rank,top,batch", [(4096, 16, 8, 2), (151936, 64, 16, 3)])
def test_select_static_equals_select_on_consecutive_calls(vocab, rank, top, batch):
    from speculative_block_drafter_gb300 import _lib as L
    from speculative_block_drafter_gb300.drafter import Drafter

    g = dataclasses.replace(di.workload("tiny").geometry, vocab=vocab, selector_rank=rank, selector_top=top)
    w = di.make_weights(g, 0)
    d = Drafter(g, w, max_batch=batch, ctx_cap=32)
    k = g.block - 1
    rng = np.random.default_rng(vocab + batch)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):                                   # two calls in a row share the fixed scratch
        logits, hp = _inputs(rng, batch, k, vocab, rank, tie=(call == 0))
        lg = torch.from_numpy(logits).cuda()
        hq = torch.from_numpy(hp).cuda()
        anchors = torch.tensor(rng.integers(0, vocab, size=batch), dtype=torch.int32, device="cuda")
        ref_chosen, ref_plain = d.select(lg, hq, anchors)
        chosen = torch.full((batch, k), -1, dtype=torch.int32, device="cuda")
        plain = torch.full((batch, k), -1, dtype=torch.int32, device="cuda")
        L.dflash_select_static(lg.data_ptr(), hq.data_ptr(), anchors.data_ptr(), d._weights.pred_book,
                               d._weights.succ_book, batch, k, vocab, vocab, rank, top, chosen.data_ptr(),
                               plain.data_ptr(), stream)
        torch.cuda.synchronize()
        # token ids: the tolerance is exact equality
        assert torch.equal(chosen, ref_chosen), (call, chosen, ref_chosen)
        assert torch.equal(plain, ref_plain), (call, plain, ref_plain)
        # and the oracle's selector on the same f32 inputs: the same row tops, the same chosen
        # tokens except where the oracle's top-two score margin is below 1e-3
        ch, pl = chosen.cpu().numpy(), plain.cpu().numpy()
        at = anchors.cpu().numpy()
        for b in range(batch):
            _, opl = O.select_with(hp[b], logits[b], int(at[b]), w["pred_book"], w["succ_book"], top)
            assert list(pl[b]) == opl, (call, b)
            check_tokens(ch[b], pl[b], hp[b].astype(np.float64), logits[b].astype(np.float64), int(at[b]),
                         w["pred_book"], w["succ_book"], top)
    d.close()


def test_select_static_leaves_device_memory_as_it_found_it():
    """After a first call (which looks up the array's device address), further calls allocate
    nothing: neither the device's free memory nor torch's allocator moves."""
    from speculative_block_drafter_gb300 import _lib as L
    vocab, rank, top, batch = 151936, 64, 16, 2
    g = dataclasses.replace(di.workload("tiny").geometry, vocab=vocab, selector_rank=rank, selector_top=top)
    w = di.make_weights(g, 0)
    k = g.block - 1
    rng = np.random.default_rng(7)
    logits, hp = _inputs(rng, batch, k, vocab, rank)
    lg = torch.from_numpy(logits).cuda()
    hq = torch.from_numpy(hp).cuda()
    pb = torch.from_numpy(np.ascontiguousarray(w["pred_book"]).view(np.int16)).cuda()
    sb = torch.from_numpy(np.ascontiguousarray(w["succ_book"]).view(np.int16)).cuda()
    anchors = torch.tensor([1, 2], dtype=torch.int32, device="cuda")
    chosen = torch.empty(batch, k, dtype=torch.int32, device="cuda")
    plain = torch.empty(batch, k, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream

    def call():
        L.dflash_select_static(lg.data_ptr(), hq.data_ptr(), anchors.data_ptr(), pb.data_ptr(), sb.data_ptr(), batch,
                               k, vocab, vocab, rank, top, chosen.data_ptr(), plain.data_ptr(), stream)

    call()
    torch.cuda.synchronize()
    first = chosen.clone()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(5):
        call()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0 and torch.cuda.memory_allocated() == alloc0
    assert torch.equal(chosen, first)


def test_select_static_rejects_what_does_not_fit():
    from speculative_block_drafter_gb300 import _lib as L
    with pytest.raises(L.DflashError) as e:
        # 1024 sequences x 15 rows at a 151,936 vocabulary need more than the fixed scratch
        L.dflash_select_static(16, 16, 16, 16, 16, 1024, 15, 151936, 151936, 64, 16, 16, 16, None)
    assert e.value.code == 3 and "8 MiB" in str(e.value)

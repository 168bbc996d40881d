"""bench.py's output contract and the library's loud failures, on the CPU.

The reference arm (the oracle timed on the host cores) prints one JSON line
with the keys the GPU arm prints; the GPU arm and the binding fail with an
error, never a host fallback, where there is no GPU or no built library.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args, timeout=300):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                          text=True, timeout=timeout, env={**os.environ, "RANK": "0", "WORLD_SIZE": "1"})


def test_reference_arm_prints_one_contract_line():
    sys.path.insert(0, ROOT)
    import bench
    p = _run("--impl", "reference", "--steps", "2", "--warmup", "0", "--workload", "tiny")
    assert p.returncode == 0, p.stderr
    lines = [l for l in p.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "blocks/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 0
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["value"] == pytest.approx(1e3 / d["ms_per_step"], rel=1e-9)
    assert d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert isinstance(cb["cores"], int) and cb["cores"] >= 1 and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_is_silent_on_other_ranks():
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--workload", "tiny"], cwd=ROOT, capture_output=True, text=True,
                       timeout=300, env={**os.environ, "RANK": "1", "WORLD_SIZE": "2"})
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""


def test_gpu_arm_fails_loudly_without_a_gpu():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    p = _run("--steps", "1", "--warmup", "0", "--workload", "tiny")
    assert p.returncode != 0
    assert '"metric"' not in p.stdout


def test_binding_raises_when_the_library_is_missing(monkeypatch):
    sys.path.insert(0, ROOT)
    from speculative_block_drafter_gb300 import _lib as L
    monkeypatch.setattr(L, "_lib", None)
    monkeypatch.setattr(L, "LIB_PATH", os.path.join(ROOT, "no-such-dir", "libdflash.so"))
    with pytest.raises(RuntimeError, match="missing"):
        L.lib()


def test_algorithmic_bytes_of_each_workload():
    """The roofline's per-unit bytes: every weight once per block (or per settle call), the K/V
    rows the windows admit at 4 bytes an element, taps in and K/V out for the settle. The
    figures of the five workloads: 0.6B block 120.5 MB, 27b block 1,495 MB, settle-heavy block
    2,737 MB, batched step 4,399 MB, a 27B settle row 1.276 MB at 256-row calls."""
    sys.path.insert(0, ROOT)
    import bench
    import dflash_inputs as di
    want = {"qwen3-0.6b": 120.5e6, "27b": 1495e6, "settle-heavy": 2737e6, "batched": 4399e6}
    for name, mb in want.items():
        wl = di.workload(name)
        g = wl.geometry
        ctx = bench.context_rows(g, wl.context, wl.context)
        nbytes, flops, parts = bench.block_cost(g, wl.head_width, ctx, wl.batch)
        assert nbytes == pytest.approx(mb, rel=2e-3), (name, nbytes)
        assert sum(parts.values()) == nbytes and flops > 0
    g27 = di.workload("27b").geometry
    assert bench.context_rows(g27, 4096, 4096) == [2047, 2047, 4096, 2047, 2047]
    per_row, flops = bench.settle_cost_per_row(g27, 256)
    assert per_row == pytest.approx(326.7e6 / 256, rel=2e-3)
    assert flops * 256 == pytest.approx(94.0e9, rel=2e-3)

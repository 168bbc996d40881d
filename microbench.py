"""Time one of the drafter's kernels alone through the C ABI (for tuning and profiling).

    python microbench.py gemm --rows 151936 --cols 1024 --tokens 15 --kind 4
    python microbench.py gemm --rows 5120 --cols 25600 --tokens 256 --kind 16
    python microbench.py block --workload batched --batch 8
    python microbench.py settle --workload 27b --rows 256 --calls 4

gemm: random codes / values of the given shape; the L2 cache is flushed
between launches; prints the mean time and the algorithmic bandwidth of one
launch (weights, activations in, outputs out).

block: the block pass of a workload's geometry at a chosen batch over its
settled synthetic context (settled first, outside the timed and profiled
range); the timed block passes sit between cudaProfilerStart and
cudaProfilerStop, so `ncu --profile-from-start off` sees only them.
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import dflash_inputs as di  # noqa: E402
from speculative_block_drafter_gb300 import build  # noqa: E402
from speculative_block_drafter_gb300.drafter import Drafter, PackedMatrix  # noqa: E402


def _int4(rows, cols, group, seed=0):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
    scales = (rng.random((rows, cols // group)) * 0.01 + 1e-3).astype(np.float16)
    return di.Int4(codes=codes, scales=scales, rows=rows, cols=cols, group=group)


def gemm(args):
    build.build()
    if args.kind == 4:
        m = _int4(args.rows, args.cols, args.group)
        wbytes = args.rows * args.cols // 2 + args.rows * (args.cols // args.group) * 2
    else:
        m = (np.random.default_rng(0).standard_normal((args.rows, args.cols)) * 0.01).astype(np.float16)
        wbytes = args.rows * args.cols * 2
    pm = PackedMatrix(m)
    x = torch.randn(args.tokens, args.cols, device="cuda")
    flush = torch.empty(256 << 18, device="cuda")
    for _ in range(3):
        pm.matmul(x)
    torch.cuda.synchronize()
    ts = []
    for _ in range(args.iters):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        pm.matmul(x)
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    ms = float(np.mean(ts))
    nbytes = wbytes + x.numel() * 4 + args.tokens * args.rows * 4
    print(json.dumps({"kernel": f"gemm kind {args.kind}", "rows": args.rows, "cols": args.cols, "tokens": args.tokens,
                      "ms": round(ms, 5), "GB/s": round(nbytes / ms / 1e6, 1),
                      "TFLOP/s": round(2 * args.rows * args.cols * args.tokens / ms / 1e9, 1)}))


def block(args):
    import dataclasses
    build.build()
    wl = di.workload(args.workload)
    if args.batch:
        wl = dataclasses.replace(wl, batch=args.batch)
    g, B = wl.geometry, wl.batch
    dev = torch.device("cuda", 0)
    d = Drafter(g, di.make_weights(g, wl.seed), max_batch=B, ctx_cap=wl.context + g.block)
    for s in range(B):
        d.reset(s, 0)
        d.settle(s, 0, torch.from_numpy(di.make_taps(g, wl.seed + s, wl.context)).to(dev))
    h = torch.from_numpy(np.stack([di.block_rows(g, wl.seed + s, di.anchor_token(g, wl.seed + s))
                                   for s in range(B)]).astype(np.float32)).to(dev).contiguous()
    k = g.block - 1
    logits = torch.empty(B, k, wl.head_width, device=dev)
    hp = torch.empty(B, k, g.selector_rank, device=dev)
    anchors = [wl.context] * B
    for _ in range(3):
        d.block(anchors, h, k, wl.head_width, out=(logits, hp))
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.profiler.start()
    a.record()
    for _ in range(args.iters):
        d.block(anchors, h, k, wl.head_width, out=(logits, hp))
    b.record()
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    print(json.dumps({"block": wl.name, "batch": B, "context": wl.context,
                      "us_per_block": round(a.elapsed_time(b) / args.iters * 1e3, 1)}))


def settle(args):
    """`calls` settles of `rows` tap rows each (positions 0.., one sequence), between
    cudaProfilerStart and cudaProfilerStop after two untimed ones."""
    build.build()
    wl = di.workload(args.workload)
    g = wl.geometry
    dev = torch.device("cuda", 0)
    n = args.rows * args.calls
    d = Drafter(g, di.make_weights(g, wl.seed), max_batch=1, ctx_cap=n + g.block, cache_format=args.cache,
                rings="window" if args.rings else None)
    taps = torch.from_numpy(di.make_taps(g, wl.seed, n)).to(dev)
    for _ in range(2):
        d.reset(0, 0)
        d.settle(0, 0, taps, chunk=args.rows)
    torch.cuda.synchronize()
    d.reset(0, 0)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.profiler.start()
    a.record()
    d.settle(0, 0, taps, chunk=args.rows)
    b.record()
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    ms = a.elapsed_time(b)
    print(json.dumps({"settle": wl.name, "rows_per_call": args.rows, "calls": args.calls,
                      "us_per_call": round(ms / args.calls * 1e3, 1), "rows_per_s": round(n / ms * 1e3, 1)}))


def main():
    p = argparse.ArgumentParser()
    sub = p.add_subparsers(dest="cmd", required=True)
    g = sub.add_parser("gemm")
    g.add_argument("--rows", type=int, default=151936)
    g.add_argument("--cols", type=int, default=1024)
    g.add_argument("--tokens", type=int, default=15)
    g.add_argument("--kind", type=int, default=4, choices=[4, 16])
    g.add_argument("--group", type=int, default=64)
    g.add_argument("--iters", type=int, default=20)
    k = sub.add_parser("block")
    k.add_argument("--workload", default="batched", choices=sorted(di.WORKLOADS))
    k.add_argument("--batch", type=int, default=0, help="sequences (default: the workload's)")
    k.add_argument("--iters", type=int, default=5)
    s = sub.add_parser("settle")
    s.add_argument("--workload", default="27b", choices=sorted(di.WORKLOADS))
    s.add_argument("--rows", type=int, default=256)
    s.add_argument("--calls", type=int, default=4)
    s.add_argument("--cache", default="planes", choices=["planes", "f16"])
    s.add_argument("--rings", action="store_true")
    args = p.parse_args()
    if args.cmd == "gemm":
        gemm(args)
    elif args.cmd == "settle":
        settle(args)
    else:
        block(args)


if __name__ == "__main__":
    main()

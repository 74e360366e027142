"""Run one operation of the library on one synthetic problem, for profiling
and quick timing.

    python -m ggml_block_quantized_linear_b300.cases --op gemv --fmt q8_0 \
        --n 4096 --k 4096 --m 1 --iters 3 [--time]

--op: quantize | dequantize | matmul.  Inputs are the seeded synthetic
weights / activations of ``inputs``.  Without --time the op is launched
``--iters`` times after one warm-up launch (a fixed, small launch count for
ncu).  With --time every launch is preceded by a 256 MB write that flushes
L2, and the median CUDA-event time per launch is printed with the achieved
bandwidth or FLOP rate.
"""
from __future__ import annotations

import argparse
import json
import statistics
import sys

import torch

import ggml_block_quantized_linear_b300 as q
from ggml_block_quantized_linear_b300 import inputs


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--op", choices=["quantize", "dequantize", "matmul"], required=True)
    ap.add_argument("--fmt", choices=sorted(q.FORMATS), default="q8_0")
    ap.add_argument("--n", type=int, default=4096)
    ap.add_argument("--k", type=int, default=4096)
    ap.add_argument("--m", type=int, default=1)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--time", action="store_true")
    a = ap.parse_args(argv)
    fmt = q.FORMATS[a.fmt]
    dev = torch.device("cuda:0")
    w = inputs.weights(a.n, a.k, 7, device=dev)
    packed = q.qmm_quantize(fmt, w)
    x = inputs.activations(a.m, a.k, 7, device=dev)
    y = torch.empty((a.m, a.n), dtype=torch.float32, device=dev)
    deq = torch.empty((a.n, a.k), dtype=torch.float32, device=dev) if a.op == "dequantize" else None
    out = torch.empty_like(packed)
    ws_bytes = q.qmm_matmul_workspace_bytes(fmt, a.m, a.n, a.k)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)

    def run():
        if a.op == "quantize":
            q.qmm_quantize(fmt, w, out=out)
        elif a.op == "dequantize":
            q.qmm_dequantize(fmt, packed, a.n, a.k, out=deq)
        else:
            q.qmm_matmul(fmt, packed, x, a.n, out=y, workspace=ws)

    run()
    torch.cuda.synchronize()
    if not a.time:
        for _ in range(a.iters):
            run()
        torch.cuda.synchronize()
        print("ran %d x %s %s N=%d K=%d M=%d" % (a.iters, a.op, a.fmt, a.n, a.k, a.m))
        return 0

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ts = []
    for _ in range(max(a.iters, 5)):
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        run()
        e1.record()
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e-3)
    t = statistics.median(ts)
    nw = a.n * a.k
    bw = q.qmm_packed_bytes(fmt, a.n, a.k) / nw  # packed bytes per weight
    rec = {"op": a.op, "fmt": a.fmt, "N": a.n, "K": a.k, "M": a.m, "us": round(t * 1e6, 2)}
    if a.op == "quantize":
        rec["GBps"] = round(nw * (2 + bw) / t / 1e9, 1)
    elif a.op == "dequantize":
        rec["GBps"] = round(nw * (bw + 4) / t / 1e9, 1)
    else:
        rec["weight_GBps"] = round(nw * bw / t / 1e9, 1)
        rec["TFLOPs"] = round(2.0 * a.m * nw / t / 1e12, 2)
    print(json.dumps(rec))
    return 0


if __name__ == "__main__":
    sys.exit(main())

#!/usr/bin/env python3
"""Benchmark of the B300 GGML block-quantized linear layer (Q8_0, Q4_K and
the other block types).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  The headline metric is the packed-weight
bandwidth of the decode GEMV at M = 1 over the decode-shaped linears
(N x K = 4096x4096, 1024x4096, 14336x4096, 4096x14336) in both formats,
with the weights cold in L2.  One step runs every stage of the path once,
each stage captured as a CUDA graph and replayed back to back:

  isq       quantize the four bf16 decode weights to Q8_0 and Q4_K
  dequant   dequantize them to fp32
  head      output head of the 8B-shape decoder at M = 1 (128256 x 4096) in
            the types the pages' sensitive-tensor policy gives it: Q6_K (Q4_K
            model) and Q8_0 (Q8_0 model); it runs before the GEMV sweeps so
            that they start with L2 holding clean lines of other weights
  gemv_m1   decode GEMV, M = 1, all 8 linears          (-> value)
  gemv_m4   ... M = 4
  gemv_m16  ... M = 16
  gemm_mid  tiled matmul at mid-size batches, M = 32 and 128, the 4 decode
            shapes x 2 formats
  gemm      prefill GEMM, M = 512 and 2048, 3 shapes x 2 formats
  fp8       FP8 E4M3 (row scales, W8A16) ISQ of the four decode weights, the
            M = 1 decode sweep over them and prefill at M = 2048
  kq        Q5_K, Q3_K and Q2_K: ISQ of the four decode weights and the
            M = 1 decode sweep over them
  embed     token-embedding lookup of 2048 tokens from the 128256 x 4096
            table, Q6_K and Q8_0, bf16 rows
  model     synthetic 8B-shape decoder (32 layers x 7 linears): ISQ of all
            224 bf16 weights to Q4_K and to Q8_0, then one M = 1 decode
            step (224 GEMVs) in each format

Inputs are seeded synthetic tensors (ggml_block_quantized_linear_b300.inputs);
the packed weights rotate through more than 200 MB per GEMV sweep, so every
GEMV reads its weights from HBM, not L2.

Under torchrun (N > 1) every rank runs the same per-GPU workload on its own
GPU (independent problems, weak scaling); there is no data-path collective,
only a barrier and a max over ranks of the timings.

`--impl reference` times the plain CPU oracle (oracle/) on the host cores on
a bounded sample of the same workload and metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Q8_0/Q4_K qmatmul weight GB/s vs HBM peak (M=1); TFLOP/s at M=2048"
UNIT = "GB/s"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# --------------------------------------------------------------------- utils
def env_rank():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# Source files that define each kernel family: a DRAM-traffic figure measured by
# ncu stays valid while these files are unchanged.
FAMILY_SOURCES = {
    "quantize": ("common.cuh", "quantize.cu"),
    "dequantize": ("common.cuh", "quantize.cu"),
    "gemv": ("common.cuh", "gemv.cu", "gemv_rows.cu"),
    "gemv_fp8": ("common.cuh", "gemv_rows.cu"),
    "quantize_fp8": ("common.cuh", "fp8.cu"),
    "gemm": ("common.cuh", "gemm.cu"),
    "gemm_mid": ("common.cuh", "gemm.cu"),
    "head": ("common.cuh", "q6k.cu", "gemv_rows.cu", "sbrows.cu"),
    "embed": ("common.cuh", "q6k.cu"),
    "quantize_kq": ("common.cuh", "kquant.cu"),
    "gemv_kq": ("common.cuh", "kquant.cu", "gemv_rows.cu", "sbrows.cu"),
}


def kernel_source_hash(names=None):
    """sha256 prefix over the CUDA sources `names` (default: every .cu/.cuh)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "ggml_block_quantized_linear_b300", "csrc")
    if names is None:
        names = [n for n in os.listdir(csrc) if n.endswith((".cu", ".cuh"))]
    for name in sorted(names):
        h.update(name.encode())
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


def load_traffic(path=None):
    """DRAM bytes per weight measured by ncu for each kernel family
    (profiles/dram_traffic.txt, lines `family=bytes_per_weight source_hash`).
    A figure is used only while the family's sources hash to the value it was
    measured on."""
    p = path or os.path.join(ROOT, "profiles", "dram_traffic.txt")
    out = {}
    if not os.path.exists(p):
        return out
    for line in open(p):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        k, _, v = line.partition("=")
        k, parts = k.strip(), v.split()
        if k not in FAMILY_SOURCES or len(parts) != 2:
            continue
        try:
            bpw = float(parts[0])
        except ValueError:
            continue
        if parts[1] == kernel_source_hash(FAMILY_SOURCES[k]):
            out[k] = bpw
    return out


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        try:
            sm = [float(r[1]) for r in rows]
            smax = max(float(r[2]) for r in rows)
            power = [float(r[3]) for r in rows if r[3].replace(".", "", 1).isdigit()]
        except ValueError:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [s for s, r in zip(sm, rows)] if sm else []
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------- our workload
class Workload:
    def __init__(self, device, with_model=True):
        import torch
        import ggml_block_quantized_linear_b300 as q
        from ggml_block_quantized_linear_b300 import inputs
        self.torch, self.q, self.inputs = torch, q, inputs
        self.dev = device
        self.fmts = [q.QMM_Q8_0, q.QMM_Q4_K]
        # decode-shaped linears: bf16 sources, packed weights, activations
        self.w_bf16 = []
        for si, (n, k) in enumerate(inputs.DECODE_SHAPES):
            self.w_bf16.append(inputs.weights(n, k, inputs.seed_for(2, si), device=device))
        self.packed = {f: [q.qmm_quantize(f, w) for w in self.w_bf16] for f in self.fmts}
        self.isq_out = {f: [torch.empty_like(p) for p in self.packed[f]] for f in self.fmts}
        self.deq_out = [torch.empty((n, k), dtype=torch.float32, device=device)
                        for (n, k) in inputs.DECODE_SHAPES]
        self.x = {}
        self.y = {}
        for mi, m in enumerate(inputs.DECODE_MS + inputs.PREFILL_MS + inputs.MID_MS):
            self.x[m] = [inputs.activations(m, k, inputs.seed_for(2, si, mi), device=device)
                         for si, (n, k) in enumerate(inputs.DECODE_SHAPES)]
            self.y[m] = {f: [torch.empty((m, n), dtype=torch.float32, device=device)
                             for (n, k) in inputs.DECODE_SHAPES] for f in self.fmts}
        self.gemm_ok = self._probe_gemm()
        # FP8 E4M3 weights with row scales (W8A16) of the same decode weights
        self.fp8 = [q.qmm_quantize(q.QMM_FP8_E4M3, w) for w in self.w_bf16]
        self.fp8_isq_out = [torch.empty_like(p) for p in self.fp8]
        self.fp8_y = {m: [torch.empty((m, n), dtype=torch.float32, device=device)
                          for (n, k) in inputs.DECODE_SHAPES] for m in (1, 2048)}
        # Q5_K / Q3_K / Q2_K (the other K-quants) of the same decode weights
        self.kq_fmts = [q.QMM_Q5_K, q.QMM_Q3_K, q.QMM_Q2_K]
        self.kq = {f: [q.qmm_quantize(f, w) for w in self.w_bf16] for f in self.kq_fmts}
        self.kq_isq_out = {f: [torch.empty_like(p) for p in self.kq[f]] for f in self.kq_fmts}
        self.kq_y = [torch.empty((1, n), dtype=torch.float32, device=device) for (n, k) in inputs.DECODE_SHAPES]
        # output head / embedding table of the 8B-shape decoder, in the types
        # of the sensitive-tensor policy (Q4_K model -> Q6_K, Q8_0 -> Q8_0)
        vocab, hidden = inputs.VOCAB, 4096
        head_w = inputs.weights(vocab, hidden, 70000, device=device)
        self.head_fmts = sorted({q.qmm_embedding_format(f) for f in self.fmts})
        self.head = {f: q.qmm_quantize(f, head_w) for f in self.head_fmts}
        del head_w
        self.head_x = inputs.activations(1, hidden, 70001, device=device)
        self.head_y = torch.empty((1, vocab), dtype=torch.float32, device=device)
        g = torch.Generator(device="cpu")
        g.manual_seed(70002)
        self.embed_ids = torch.randint(0, vocab, (2048,), generator=g, dtype=torch.int64).to(device)
        self.embed_out = torch.empty((2048, hidden), dtype=torch.bfloat16, device=device)
        self.model = None
        if with_model:
            self._make_model()

    def _probe_gemm(self):
        q = self.q
        try:
            q.qmm_matmul(q.QMM_Q8_0, self.packed[q.QMM_Q8_0][0], self.x[512][0], 4096,
                         out=self.y[512][q.QMM_Q8_0][0])
            self.torch.cuda.synchronize(self.dev)
            return True
        except q.QmmError:
            return False

    def _make_model(self):
        torch, q, inputs = self.torch, self.q, self.inputs
        self.model = {"w": [], "packed": {f: [] for f in self.fmts}, "x": [], "y": []}
        for layer in range(inputs.MODEL_LAYERS):
            for li, (name, n, k) in enumerate(inputs.MODEL_LINEARS):
                w = inputs.weights(n, k, inputs.model_weight_seed(layer, li), device=self.dev)
                self.model["w"].append(w)
                for f in self.fmts:
                    self.model["packed"][f].append(q.qmm_quantize(f, w))
                self.model["x"].append(inputs.activations(1, k, inputs.model_activation_seed(layer, li),
                                                          device=self.dev))
                self.model["y"].append(torch.empty((1, n), dtype=torch.float32, device=self.dev))

    # each stage: (name, callable, launches, algorithmic bytes, flops, kernel family)
    def stages(self):
        q, inputs = self.q, self.inputs
        S = []
        shapes = inputs.DECODE_SHAPES
        bw = {q.QMM_Q8_0: 34 / 32, q.QMM_Q4_K: 144 / 256}

        def isq():
            for f in self.fmts:
                for w, o in zip(self.w_bf16, self.isq_out[f]):
                    q.qmm_quantize(f, w, out=o)
        nw = sum(n * k for n, k in shapes)
        S.append(("isq", isq, 8, sum(nw * (2 + bw[f]) for f in self.fmts), 0.0, "quantize", 2 * nw))

        def deq():
            for f in self.fmts:
                for (n, k), p, o in zip(shapes, self.packed[f], self.deq_out):
                    q.qmm_dequantize(f, p, n, k, out=o)
        S.append(("dequant", deq, 8, sum(nw * (bw[f] + 4) for f in self.fmts), 0.0, "dequantize",
                  2 * nw))

        # The output head streams ~1 GB of packed weights and writes almost
        # nothing: run just before the GEMV sweeps, it leaves L2 holding clean
        # lines of other data (a decode step's GEMVs follow other weight
        # streams, not the gigabyte of fp32 the dequantize stage writes).
        vocab, hidden = inputs.VOCAB, 4096
        hbw = {f: q.BLOCK[f][1] / q.BLOCK[f][0] for f in self.head_fmts}

        def head():
            for f in self.head_fmts:
                q.qmm_matmul(f, self.head[f], self.head_x, vocab, out=self.head_y)
        S.append(("head_m1", head, len(self.head_fmts), sum(vocab * hidden * hbw[f] for f in self.head_fmts),
                  2.0 * vocab * hidden * len(self.head_fmts), "head", vocab * hidden * len(self.head_fmts)))

        for m in inputs.DECODE_MS:
            def gemv(m=m):
                for f in self.fmts:
                    for (n, k), p, x, y in zip(shapes, self.packed[f], self.x[m], self.y[m][f]):
                        q.qmm_matmul(f, p, x, n, out=y)
            wbytes = sum(nw * bw[f] for f in self.fmts)
            io = 2 * sum((2 * m * k + 4 * m * n) for n, k in shapes)
            # a call that takes the tiled kernel (it needs a workspace: long rows
            # from 12 tokens for Q8_0) launches the activation conversion too
            nl = sum(2 if q.qmm_matmul_workspace_bytes(f, m, n, k) > 0 else 1
                     for f in self.fmts for (n, k) in shapes)
            S.append(("gemv_m%d" % m, gemv, nl, wbytes + io, 2.0 * 2 * m * nw, "gemv", 2 * nw))

        if self.gemm_ok:
            for m in inputs.MID_MS:
                def gemm_mid(m=m):
                    for f in self.fmts:
                        for (n, k), p, x, y in zip(shapes, self.packed[f], self.x[m], self.y[m][f]):
                            q.qmm_matmul(f, p, x, n, out=y)
                S.append(("gemm_m%d" % m, gemm_mid, 16, sum(nw * bw[f] for f in self.fmts),
                          2 * 2.0 * m * nw, "gemm_mid", 2 * nw))

        f8 = q.QMM_FP8_E4M3
        f8bytes = sum(p.numel() for p in self.fp8)

        def fp8_isq():
            for w, o in zip(self.w_bf16, self.fp8_isq_out):
                q.qmm_quantize(f8, w, out=o)
        S.append(("isq_fp8", fp8_isq, 4, 2 * nw + f8bytes, 0.0, "quantize_fp8", nw))

        def fp8_gemv():
            for (n, k), p, x, y in zip(shapes, self.fp8, self.x[1], self.fp8_y[1]):
                q.qmm_matmul(f8, p, x, n, out=y)
        S.append(("gemv_fp8_m1", fp8_gemv, 4, f8bytes, 2.0 * nw, "gemv_fp8", nw))
        if self.gemm_ok:
            pshapes = inputs.PREFILL_SHAPES

            def fp8_gemm():
                for si, (n, k) in enumerate(shapes):
                    if (n, k) in pshapes:
                        q.qmm_matmul(f8, self.fp8[si], self.x[2048][si], n, out=self.fp8_y[2048][si])
            S.append(("gemm_fp8_m2048", fp8_gemm, 6, 0, 2 * 2048.0 * sum(n * k for n, k in pshapes),
                      "gemm", sum(n * k for n, k in pshapes)))

        kqb = {f: q.BLOCK[f][1] / q.BLOCK[f][0] for f in self.kq_fmts}

        def kq_isq():
            for f in self.kq_fmts:
                for w, o in zip(self.w_bf16, self.kq_isq_out[f]):
                    q.qmm_quantize(f, w, out=o)
        S.append(("isq_kq", kq_isq, 12, sum(nw * (2 + kqb[f]) for f in self.kq_fmts), 0.0, "quantize_kq",
                  3 * nw))

        def kq_gemv():
            for f in self.kq_fmts:
                for (n, k), p, x, y in zip(shapes, self.kq[f], self.x[1], self.kq_y):
                    q.qmm_matmul(f, p, x, n, out=y)
        S.append(("gemv_kq_m1", kq_gemv, 12, sum(nw * kqb[f] for f in self.kq_fmts), 2.0 * 3 * nw, "gemv_kq",
                  3 * nw))

        def embed():
            for f in self.head_fmts:
                q.qmm_embedding(f, self.head[f], self.embed_ids, hidden, out=self.embed_out)
        T = self.embed_ids.numel()
        S.append(("embed_t2048", embed, len(self.head_fmts),
                  sum(T * hidden * (hbw[f] + 2) + 8 * T for f in self.head_fmts), 0.0, "embed",
                  T * hidden * len(self.head_fmts)))

        if self.gemm_ok:
            pshapes = inputs.PREFILL_SHAPES
            for m in inputs.PREFILL_MS:
                def gemm(m=m):
                    for f in self.fmts:
                        for si, (n, k) in enumerate(shapes):
                            if (n, k) in pshapes:
                                q.qmm_matmul(f, self.packed[f][si], self.x[m][si], n,
                                             out=self.y[m][f][si])
                fl = 2 * 2.0 * m * sum(n * k for n, k in pshapes)
                # each prefill call launches two kernels: X -> binary16, then the GEMM
                S.append(("gemm_m%d" % m, gemm, 12, 0, fl, "gemm",
                          2 * sum(n * k for n, k in pshapes)))

        if self.model is not None:
            mw = sum(n * k for _, n, k in inputs.MODEL_LINEARS) * inputs.MODEL_LAYERS
            nl = len(self.model["w"])

            def model_isq():
                for f in self.fmts:
                    for w, p in zip(self.model["w"], self.model["packed"][f]):
                        q.qmm_quantize(f, w, out=p)
            S.append(("model_isq", model_isq, 2 * nl, sum(mw * (2 + bw[f]) for f in self.fmts),
                      0.0, "quantize", 2 * mw))
            for f in self.fmts:
                def model_decode(f=f):
                    for (_, n, k), p, x, y in zip(inputs.MODEL_LINEARS * inputs.MODEL_LAYERS,
                                                  self.model["packed"][f], self.model["x"],
                                                  self.model["y"]):
                        q.qmm_matmul(f, p, x, n, out=y)
                name = "model_decode_" + ("q8_0" if f == q.QMM_Q8_0 else "q4_k")
                S.append((name, model_decode, nl, mw * bw[f], 2.0 * mw, "gemv", mw))
        return S


def time_graphs(torch, graphs, steps, warmup, dev):
    """Replay every stage graph once per step; per-stage CUDA-event times."""
    names = [g[0] for g in graphs]
    for _ in range(warmup):
        for _, g in graphs:
            g.replay()
    torch.cuda.synchronize(dev)
    per = {n: [] for n in names}
    step_ms = []
    stream = torch.cuda.current_stream(dev)
    # NVTX range around the timed steps (a profiler can capture exactly these)
    torch.cuda.nvtx.range_push("qmm_timed_steps")
    for _ in range(steps):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(graphs) + 1)]
        evs[0].record(stream)
        for i, (_, g) in enumerate(graphs):
            g.replay()
            evs[i + 1].record(stream)
        evs[-1].synchronize()
        for i, n in enumerate(names):
            per[n].append(evs[i].elapsed_time(evs[i + 1]))
        step_ms.append(evs[0].elapsed_time(evs[-1]))
    torch.cuda.nvtx.range_pop()
    return per, step_ms


def parity_check(wl):
    """Sampled parity of the benchmarked kernels against the CPU oracle: the
    decode-shaped linears (packed bytes of 64 rows; outputs of 4 rows at
    M = 1, 16, 32 and 2048; FP8 bytes of 64 rows and outputs of 3 rows at
    M = 1 and 2048), the Q5_K / Q3_K / Q2_K linears (bytes of 32 rows and
    M = 1 outputs of 3 rows), the output head (bytes and M = 1 outputs of 4
    rows) and 4 embedding rows in each head format, and the last layer of
    the model (packed bytes and M = 1 outputs of 6 rows of each of its 7
    linears, both formats)."""
    import numpy as np
    import oracle
    q, inputs = wl.q, wl.inputs
    worst = 0.0
    for f in wl.fmts:
        for si, (n, k) in enumerate(inputs.DECODE_SHAPES):
            packed = wl.packed[f][si].cpu().numpy()
            want = oracle.quantize(f, inputs.bf16_bits(wl.w_bf16[si][:64].cpu()))
            if not np.array_equal(packed[:64], want):
                return "FAIL: packed bytes differ (fmt %d shape %d)" % (f, si)
            # FP8: bytes of the same rows, outputs at M = 1 and 2048
            f8 = q.QMM_FP8_E4M3
            want8 = oracle.quantize(f8, inputs.bf16_bits(wl.w_bf16[si][:64].cpu()))
            if not np.array_equal(wl.fp8[si][:64].cpu().numpy(), want8):
                return "FAIL: FP8 packed bytes differ (shape %d)" % si
            if f == wl.fmts[0]:
                for m in (1,) + ((2048,) if wl.gemm_ok and (n, k) in inputs.PREFILL_SHAPES else ()):
                    ns = np.array([0, 1, 63], dtype=np.int64)
                    xb = inputs.bf16_bits(wl.x[m][si])
                    Y, A = oracle.matmul(f8, want8[ns], xb, ns.size, k)
                    y = wl.fp8_y[m][si][:, ns].double().cpu().numpy()
                    worst = max(worst, float((np.abs(y - Y) / (1e-3 * A + 1e-6)).max()))
            for m in (1, 16) + ((32,) if wl.gemm_ok else ()) + (
                    (2048,) if wl.gemm_ok and (n, k) in inputs.PREFILL_SHAPES else ()):
                ns = np.array([0, 1, n // 2, n - 1], dtype=np.int64)
                xb = inputs.bf16_bits(wl.x[m][si])
                Y, A = oracle.matmul_columns(f, packed, xb, k, ns)
                y = wl.y[m][f][si][:, ns].double().cpu().numpy()
                r = float((np.abs(y - Y) / (1e-3 * A + 1e-6)).max())
                worst = max(worst, r)
    # the other K-quants: bytes of 32 rows and M = 1 outputs of 3 rows
    for f in wl.kq_fmts:
        for si, (n, k) in enumerate(inputs.DECODE_SHAPES):
            want = oracle.quantize(f, inputs.bf16_bits(wl.w_bf16[si][:32].cpu()))
            if not np.array_equal(wl.kq[f][si][:32].cpu().numpy(), want):
                return "FAIL: packed bytes differ (fmt %d shape %d)" % (f, si)
            y = q.qmm_matmul(f, wl.kq[f][si], wl.x[1][si], n)
            ns = np.array([0, 1, 31], dtype=np.int64)
            Y, A = oracle.matmul(f, want[ns], inputs.bf16_bits(wl.x[1][si]), ns.size, k)
            worst = max(worst, float((np.abs(y[:, ns].double().cpu().numpy() - Y) / (1e-3 * A + 1e-6)).max()))
    # output head (sampled rows, bytes and M = 1 outputs) and embedding rows
    torch = wl.torch
    vocab, hidden = inputs.VOCAB, 4096
    head_w = inputs.weights(vocab, hidden, 70000, device=wl.dev)
    rows = np.array([0, 1, vocab // 2, vocab - 1], dtype=np.int64)
    ridx = torch.from_numpy(rows).to(wl.dev)
    eids = wl.embed_ids[:4].cpu().numpy()
    for f in wl.head_fmts:
        want = oracle.quantize(f, inputs.bf16_bits(head_w[ridx]))
        if not np.array_equal(wl.head[f][ridx].cpu().numpy(), want):
            return "FAIL: output head packed bytes differ (fmt %d)" % f
        y = q.qmm_matmul(f, wl.head[f], wl.head_x, vocab)[:, ridx].double().cpu().numpy()
        Y, A = oracle.matmul(f, want, inputs.bf16_bits(wl.head_x), rows.size, hidden)
        worst = max(worst, float((np.abs(y - Y) / (1e-3 * A + 1e-6)).max()))
        ew = oracle.quantize(f, inputs.bf16_bits(head_w[torch.from_numpy(eids).to(wl.dev)]))
        erow = oracle.dequantize(f, ew, eids.size, hidden)
        got = q.qmm_embedding(f, wl.head[f], wl.embed_ids[:4], hidden, dtype=torch.bfloat16).cpu()
        if not torch.equal(got, torch.from_numpy(erow).to(torch.bfloat16)):
            return "FAIL: embedding rows differ (fmt %d)" % f
    del head_w
    if wl.model is not None:
        # the last model layer: its 7 linears, packed bytes and M = 1 outputs
        # on a row sample, both formats
        torch = wl.torch
        layer = inputs.MODEL_LAYERS - 1
        for li, (_, n, k) in enumerate(inputs.MODEL_LINEARS):
            j = layer * len(inputs.MODEL_LINEARS) + li
            rows = np.array(sorted({0, 1, n // 3, n // 2, n - 2, n - 1}), dtype=np.int64)
            ridx = torch.from_numpy(rows).to(wl.dev)
            wb = inputs.bf16_bits(wl.model["w"][j][ridx])
            xb = inputs.bf16_bits(wl.model["x"][j])
            for f in wl.fmts:
                want = oracle.quantize(f, wb)
                packed = wl.model["packed"][f][j]
                if not np.array_equal(packed[ridx].cpu().numpy(), want):
                    return "FAIL: model packed bytes differ (fmt %d linear %d)" % (f, j)
                y = q.qmm_matmul(f, packed, wl.model["x"][j], n)[:, ridx].double().cpu().numpy()
                Y, A = oracle.matmul(f, want, xb, rows.size, k)
                worst = max(worst, float((np.abs(y - Y) / (1e-3 * A + 1e-6)).max()))
    return "ok (max err/bound %.3f)" % worst if worst <= 1.0 else "FAIL (max err/bound %.3f)" % worst


def e2e_decode(wl, steps, warmup):
    """M = 1 decode sweep through the public API with pinned host buffers, as
    a decode loop runs it: the eight activation vectors are copied host ->
    device in one transfer, the eight qmm_matmul calls run, and the eight
    results come back in one device -> host transfer, the whole step
    captured once as a CUDA graph and replayed every step (copies included
    in the timed region)."""
    torch, q, inputs = wl.torch, wl.q, wl.inputs
    jobs = [(f, si, n, k) for f in wl.fmts for si, (n, k) in enumerate(inputs.DECODE_SHAPES)]
    xoff, yoff = [0], [0]
    for (_, _, n, k) in jobs:
        xoff.append(xoff[-1] + k)  # bf16 elements; every K is a multiple of 256: 16-byte aligned slices
        yoff.append(yoff[-1] + n)  # fp32 elements; every N is a multiple of 4
    hx = torch.empty(xoff[-1], dtype=torch.bfloat16).pin_memory()
    hy = torch.empty(yoff[-1], dtype=torch.float32).pin_memory()
    for j, (f, si, n, k) in enumerate(jobs):
        hx[xoff[j]:xoff[j + 1]].copy_(wl.x[1][si].reshape(-1).cpu())
    dx = torch.empty(xoff[-1], dtype=torch.bfloat16, device=wl.dev)
    dy = torch.empty(yoff[-1], dtype=torch.float32, device=wl.dev)
    xs = [dx[xoff[j]:xoff[j + 1]].view(1, -1) for j in range(len(jobs))]
    ys = [dy[yoff[j]:yoff[j + 1]].view(1, -1) for j in range(len(jobs))]

    def step():
        dx.copy_(hx, non_blocking=True)
        for j, (f, si, n, k) in enumerate(jobs):
            q.qmm_matmul(f, wl.packed[f][si], xs[j], n, out=ys[j])
        hy.copy_(dy, non_blocking=True)

    s = torch.cuda.Stream(wl.dev)
    s.wait_stream(torch.cuda.current_stream(wl.dev))
    with torch.cuda.stream(s):
        step()  # warm-up outside the capture (plans, attributes)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    s.synchronize()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize(wl.dev)
    stream = torch.cuda.current_stream(wl.dev)
    t = []
    for _ in range(steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        e1.synchronize()
        t.append(e0.elapsed_time(e1))
    # the results that came back equal the device-side sweep's (same inputs,
    # deterministic kernels)
    same = all(torch.equal(hy[yoff[j]:yoff[j + 1]], wl.y[1][f][si].reshape(-1).cpu())
               for j, (f, si, n, k) in enumerate(jobs))
    wbytes = sum(p.numel() for f in wl.fmts for p in wl.packed[f])
    ms = statistics.median(t)
    return {"value": round(wbytes / (ms * 1e-3) / 1e9, 1), "unit": UNIT,
            "h2d_bytes_per_step": hx.numel() * 2, "d2h_bytes_per_step": hy.numel() * 4,
            "matches_device_sweep": same,
            "ms_per_step": round(ms, 4), "launches_per_step": len(jobs),
            "capture": "one CUDA graph per step: one H2D copy of the 8 activation vectors, "
                       "8 qmm_matmul calls, one D2H copy of the 8 results"}


# ------------------------------------------------------------ CPU oracle arm
def oracle_decode_sample(threads=None, min_seconds=10.0):
    """Time the oracle's M = 1 matmul over the eight decode-shaped linears
    (rows sampled evenly, so that the sample takes ~min_seconds)."""
    import numpy as np
    import torch
    import oracle
    from ggml_block_quantized_linear_b300 import inputs
    if threads:
        oracle.set_threads(threads)
    cores = oracle.max_threads()
    probs = []
    for f in (oracle.Q8_0, oracle.Q4_K):
        for si, (n, k) in enumerate(inputs.DECODE_SHAPES):
            rows = 256  # weight rows per linear in the sample
            w = inputs.weights(rows, k, inputs.seed_for(2, si))
            packed = oracle.quantize(f, inputs.bf16_bits(w))
            xb = inputs.bf16_bits(inputs.activations(1, k, inputs.seed_for(2, si, 0)))
            probs.append((f, packed, xb, rows, k))
    nbytes = sum(p[1].size for p in probs)
    reps, total = 0, 0.0
    while total < min_seconds:
        t0 = time.perf_counter()
        for f, packed, xb, rows, k in probs:
            oracle.matmul(f, packed, xb, rows, k)
        total += time.perf_counter() - t0
        reps += 1
    gbs = nbytes * reps / total / 1e9
    return {"value": round(gbs, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "oracle fp64 matmul at M=1 over 256 weight rows of each of the 8 decode "
                      "linears (4 shapes x Q8_0/Q4_K), %d repetitions, %.1f s" % (reps, total)}


def run_reference(args):
    rank, world, _ = env_rank()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    cores = oracle.max_threads()
    # each step: one pass of the oracle over the bounded decode sample
    import numpy as np
    from ggml_block_quantized_linear_b300 import inputs
    probs = []
    for f in (oracle.Q8_0, oracle.Q4_K):
        for si, (n, k) in enumerate(inputs.DECODE_SHAPES):
            rows = 256
            w = inputs.weights(rows, k, inputs.seed_for(2, si))
            packed = oracle.quantize(f, inputs.bf16_bits(w))
            xb = inputs.bf16_bits(inputs.activations(1, k, inputs.seed_for(2, si, 0)))
            probs.append((f, packed, xb, rows, k))
    nbytes = sum(p[1].size for p in probs)

    def step():
        for f, packed, xb, rows, k in probs:
            oracle.matmul(f, packed, xb, rows, k)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = nbytes * args.steps / dt / 1e9
    sample = ("oracle fp64 matmul at M=1 over 256 weight rows of each of the 8 decode linears "
              "(4 shapes x Q8_0/Q4_K) per step")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(),
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def workload_config():
    return {"workload": "decode-shaped Q8_0/Q4_K linears (N x K = 4096x4096, 1024x4096, "
                        "14336x4096, 4096x14336), GEMV at M=1 (headline) plus M=4/16, ISQ, "
                        "dequant, mid-batch matmul M=32/128, prefill GEMM M=512/2048, FP8 "
                        "E4M3 W8A16 ISQ + M=1 sweep + M=2048 prefill, Q5_K/Q3_K/Q2_K ISQ + M=1 "
                        "sweep, a 128256x4096 output head (Q6_K / Q8_0, M=1), a 2048-token embedding "
                        "lookup and a 32-layer 8B-shape model (ISQ + 224-GEMV decode step) in "
                        "each step",
            "weights": "bf16 ~N(0,0.02) with 0.1% x20 outliers, seeded",
            "activations": "bf16 ~N(0,1), seeded",
            "l2": "inputs larger than L2: each GEMV sweep reads > 200 MB of distinct packed "
                  "weights, the model step 11.3 GB",
            "accumulate": "f32", "graphs": "each stage captured as one CUDA graph"}


# ------------------------------------------------------------- ranks (N > 1)
def max_over_ranks(dist, ms_step, med, names, device):
    """The step time and each stage's median time, as the maximum over the
    ranks of the process group (every rank times the same per-GPU work)."""
    import torch
    vals = torch.tensor([ms_step] + [med[n] for n in names], device=device, dtype=torch.float64)
    dist.all_reduce(vals, op=dist.ReduceOp.MAX)
    return float(vals[0]), {**med, **{n: float(vals[i + 1]) for i, n in enumerate(names)}}


def whole_job_gbps(bytes_per_rank, world, ms):
    """Whole-job throughput: the bytes all ranks processed over the slowest
    rank's time (weak scaling: the per-rank work is fixed)."""
    return bytes_per_rank * world / (ms * 1e-3) / 1e9


# --------------------------------------------------------------------- main
def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-model", action="store_true", help="skip the 32-layer model stage")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist
    rank, world, local = env_rank()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import ggml_block_quantized_linear_b300 as q
    q.load()

    wl = Workload(dev, with_model=not args.no_model)
    stages = wl.stages()
    # capture each stage as one graph (first call of every kernel happens in
    # the workload set-up above, so capture sees no lazy initialisation)
    for _, fn, *_ in stages:
        fn()
    torch.cuda.synchronize(dev)
    graphs = []
    cap = torch.cuda.Stream(dev)
    with torch.cuda.stream(cap):
        for name, fn, *_ in stages:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                fn()
            graphs.append((name, g))
    torch.cuda.synchronize(dev)
    if q.qmm_device_error_take() != 0:
        raise RuntimeError("device error during set-up")

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local)
    clocks.start()
    per, step_ms = time_graphs(torch, graphs, args.steps, args.warmup, dev)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    if q.qmm_device_error_take() != 0:
        raise RuntimeError("device error during the timed region")

    # median over steps per stage; max over ranks
    med = {n: statistics.median(v) for n, v in per.items()}
    ms_step = statistics.median(step_ms)
    if world > 1:
        ms_step, med = max_over_ranks(dist, ms_step, med, [n for n, *_ in stages], dev)

    peaks, peak_kind = load_peaks()
    traffic = load_traffic()
    info = {s[0]: s for s in stages}
    wbytes_m1 = sum(p.numel() for f in wl.fmts for p in wl.packed[f])
    value = whole_job_gbps(wbytes_m1, world, med["gemv_m1"])

    rows = {}
    fam_time = {}
    for name, _, launches, nbytes, flops, fam, _nw in stages:
        t = med[name] * 1e-3
        r = {"ms": round(med[name], 4), "launches": launches}
        if nbytes:
            r["GBps"] = round(nbytes / t / 1e9, 1)
        if fam in ("gemm", "gemm_mid"):
            r["TFLOPs"] = round(flops / t / 1e12, 1)
        rows[name] = r
        fam_time[fam] = fam_time.get(fam, 0.0) + med[name]
    for f, nm in ((q.QMM_Q8_0, "q8_0"), (q.QMM_Q4_K, "q4_k")):
        key = "model_decode_" + nm
        if key in rows:
            rows[key]["weight_GBps"] = rows[key].pop("GBps")
    for key in ("gemm_m32", "gemm_m128", "head_m1", "gemv_fp8_m1", "gemv_kq_m1"):
        if key in rows:
            rows[key]["weight_GBps"] = rows[key].pop("GBps")

    def roofline_for(fam):
        sel = [s for s in stages if s[5] == fam]
        t = sum(med[s[0]] for s in sel) * 1e-3
        launches = sum(s[2] for s in sel)
        if fam == "gemm":
            fl = sum(s[4] for s in sel)
            peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
            ach = fl / t / 1e12
            sus = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
            return {"bound": "tensor", "achieved": round(ach, 1), "peak": peak, "unit": "TFLOP/s",
                    "frac": round(ach / peak, 4), "traffic": None,
                    "peak_source": peak_kind + " bf16 burst (f16 same nominal rate)",
                    # the GEMM stages run back to back for milliseconds, under the power cap
                    "peak_sustained": sus, "frac_sustained": round(ach / sus, 4),
                    "launches": launches}
        nb = sum(s[3] for s in sel)
        nw = sum(s[6] for s in sel)
        peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
        ach = nb / t / 1e9
        bpw = traffic.get(fam)  # measured DRAM bytes per weight (one ncu capture)
        tr = bpw * nw / launches if bpw else None  # scaled to the average launch here
        return {"bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                "frac": round(ach / peak, 4),
                "traffic": round(tr) if tr else None,
                "traffic_ratio": round(tr / (nb / launches), 3) if tr else None,
                "peak_source": peak_kind + " copy bandwidth (burst)", "launches": launches}

    dominant = max(fam_time, key=fam_time.get)
    rooflines = {fam: roofline_for(fam) for fam in fam_time}
    gemv_roof = rooflines["gemv"]
    # the headline kernel: M = 1 decode GEMV sweep alone
    m1 = info["gemv_m1"]
    m1_ach = m1[3] / (med["gemv_m1"] * 1e-3) / 1e9
    rooflines["gemv_m1"] = {"bound": "hbm", "achieved": round(m1_ach, 1),
                            "peak": peaks.get("hbm_gbs"), "unit": "GB/s",
                            "frac": round(m1_ach / peaks.get("hbm_gbs"), 4),
                            "weight_only_frac": round(value / world / peaks.get("hbm_gbs"), 4)}

    line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic", "config": workload_config(),
            "roofline": dict(rooflines[dominant], kernel=dominant),
            "rooflines": rooflines, "rows": rows,
            "gemm_tflops_m2048": rows.get("gemm_m2048", {}).get("TFLOPs"),
            "clocks": clk, "gpu_launches": sum(s[2] for s in stages) * args.steps,
            "parity": None, "kernel_source": kernel_source_hash()}
    if rank == 0:
        line["parity"] = parity_check(wl)
        line["e2e"] = e2e_decode(wl, max(3, args.steps), 3)
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = oracle_decode_sample()
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

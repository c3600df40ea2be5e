#!/usr/bin/env python
"""Benchmark of the exact int8 (W8A8) / W4A8 quantized linear layer on GB300.

One step = the whole hot path over one batch of the 27B-class prefill
workload: per-token int8 quantization of the activations, then the W8A8
(Q8_0) GEMM, for both projections of that workload (gate/up: M=8192, K=5120,
N=17408; down: M=8192, K=17408, N=5120). Inputs are seeded synthetic (bf16
N(0,1) activations with 1% outlier channels x20; weights N(0,0.02) encoded
as Q8_0), resident in HBM when the timed region starts; L2 is flushed (a
512 MiB write) between timed steps, outside the per-step CUDA events.

`value` = int8 GEMM tera-operations per second (2*M*N*K per GEMM, both
projections, quantization time included). The `rows` object adds the other
workloads of the layer, each timed per launch with an L2 flush in between:
decode (M = 1, 8, 64) as weight-streaming GB/s, the 4B-class prefill, the
W4A8 (Q4_K) shapes and the activation quantizer alone (HBM GB/s). `--impl reference` times the CPU oracle on a bounded
sample of the same step instead.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_quantized_gemm_gb300 import synth  # noqa: E402

METRIC = "int8 GEMM TOPS (large M) & weight HBM GB/s (M<=64), % of GB300 roofline"
WORKLOAD = "prefill_27b_w8a8"
STEP_SHAPES = [tuple(s) for s in synth.CONFIGS[WORKLOAD]["shapes"]]  # (M, K, N): gate/up, down
CPU_SAMPLE_ROWS = 4096  # rows of the step the CPU baseline runs (about 10 s on 16 cores)
REF_SAMPLE_ROWS = 64    # rows per step of --impl reference
L2_FLUSH_BYTES = 512 << 20


def env_rank():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), d.get(
            "bf16_tflops_sustained", 1700.0), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 25 ms, each sample
    timestamped so that the summary can keep those inside a window (the timed
    region); start it before the warm-up so it is already sampling then."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    @staticmethod
    def _when(stamp):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(stamp.strip(), fmt).timestamp()
            except ValueError:
                continue
        return None

    def summary(self, window=None):
        """Median SM clock, max clock and the throttle reasons seen; samples
        inside `window` = (t0, t1) (host time.time()) when at least 3 fall in
        it, else all samples (the warm-up runs the same work)."""
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            try:
                rows.append((self._when(f[0]), float(f[2]), float(f[3]), f[6:10]))
            except (ValueError, IndexError):
                continue
        if not rows:
            return None
        scope = "timed region"
        if window is not None:
            inside = [r for r in rows if r[0] is not None and window[0] <= r[0] <= window[1]]
            if len(inside) >= 3:
                rows = inside
            else:
                scope = "warm-up and timed region (%d samples inside the timed region)" % len(inside)
        reasons = set()
        for r in rows:
            for name, val in zip(names, r[3]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[1] for r in rows),
                "sm_max_mhz": max(r[2] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows), "window": scope}


def source_sha(path):
    """Hash of a kernel source's code: comments removed and whitespace
    collapsed, so that a capture stays attached to the code it was taken on
    (a comment edit keeps it, any code edit drops it)."""
    import hashlib
    import re
    text = open(path, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return hashlib.sha1(" ".join(text.split()).encode()).hexdigest()


def sources_sha(paths):
    """One id for several files (their git blob ids, hashed in order)."""
    import hashlib
    h = hashlib.sha1()
    for p in paths:
        h.update(source_sha(p).encode())
    return h.hexdigest()


def measured_traffic():
    """DRAM bytes per GEMM call (one or two launches) on this workload, mean
    over the two projections, from the committed ncu summary -- None when a
    kernel source it was taken on changed since."""
    p = os.path.join(ROOT, "profiles", "prefill_traffic_27b_step.json")
    try:
        with open(p) as f:
            d = json.load(f)
        srcs = [os.path.join(ROOT, s) for s in d.get("source_files", [])]
        if not srcs or d.get("source_sha") != sources_sha(srcs):
            return None
        return d.get("bytes_per_gemm_call")
    except (OSError, ValueError):
        return None


def reduce_max(value, world):
    """Max over ranks (the slowest replica sets the job time)."""
    if world <= 1:
        return float(value)
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" \
        else torch.device("cpu")
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(ops_per_rank, world, ms_max):
    """Whole-job throughput (TOPS): every rank's units over the slowest rank's time."""
    return world * ops_per_rank / (ms_max * 1e-3) / 1e12


def make_step_inputs(dev):
    """Seeded inputs of the 27B-class prefill step (x bf16, packed Q8_0 weights)."""
    import bit_quantized_gemm_gb300 as qg
    layers = []
    for i, (M, K, N) in enumerate(STEP_SHAPES):
        x, bits = synth.config_activations(WORKLOAD, M, K, seed_offset=i)
        blocks = synth.config_weights(WORKLOAD, N, K, seed_offset=i)
        xd = torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)
        packed = qg.pack_q8_0(torch.from_numpy(blocks).to(dev), N, K)
        # the prefill kernel (M > 16) reads the fp16 copy alone: no int8 copy is written
        q = torch.empty((M, K), dtype=torch.int8, device=dev) if M <= qg.small_m_max() else None
        s = torch.empty((M,), dtype=torch.float32, device=dev)
        h = torch.empty((M, K), dtype=torch.float16, device=dev)
        out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        layers.append(dict(M=M, K=K, N=N, x=xd, bits=bits, blocks=blocks, packed=packed, q=q,
                           s=s, h=h, out=out))
    torch.cuda.synchronize()
    return layers


def step_kernels(dev):
    """The kernels the step's GEMM calls launch (the wave plan on this GPU)."""
    from bit_quantized_gemm_gb300 import _lib
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    parts = []
    for (M, K, N) in STEP_SHAPES:
        rows, kind, tokens = _lib.prefill_plan(M, N, sms)
        d = "%dx%dx%d: prefill_gemm_kernel 256-token tiles (tcgen05 kind::f16 on integer-valued " \
            "operands) for weight rows [0, %d)" % (M, K, N, rows)
        if kind == "tensor":
            d += ", rows [%d, %d) as %d-token tiles" % (rows, N, tokens)
        elif kind == "16-row":
            d += ", rows [%d, %d) as skinny_gemm_kernel %d-token 16-row tiles" % (rows, N, tokens)
        parts.append(d)
    return "; ".join(parts)


def step_ops():
    return sum(2.0 * M * N * K for (M, K, N) in STEP_SHAPES)


def run_step(layers, ev=None):
    """quantize + GEMM for each layer; ev: optional list of (start, end) event pairs per GEMM."""
    import bit_quantized_gemm_gb300 as qg
    for i, L in enumerate(layers):
        qg.quantize_act(L["x"], q16=True, out=(L["q"], L["s"], None, L["h"]))
        if ev is not None:
            ev[i][0].record()
        qg.gemm_w8a8_q8_0(L["q"], L["h"], L["s"], L["packed"], L["N"], out=L["out"])
        if ev is not None:
            ev[i][1].record()


def timed_launches(fn, reps, flush):
    """Median/mean device time (ms) of fn() over reps, with an L2 flush before each."""
    times = []
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    return times


ROTATE_COPIES = 4  # weight copies a small-M timing cycles through (4 x >= 95 MB > L2)


def timed_rotating(fns, reps, batches=5):
    """Device time (ms) per launch of a batch of `reps` back-to-back launches
    cycling through fns (each reads its own copy of the weights, so no
    launch finds its weights in L2); median over `batches`. A single
    microsecond-scale launch is below the event clock's resolution."""
    for f in fns:
        f()
    times = []
    for _ in range(batches):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(reps):
            fns[i % len(fns)]()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b) / reps)
    return times


def timed_graph(fns, reps, batches=5):
    """As timed_rotating, with the `reps` calls captured once as a CUDA graph
    and replayed, so that the host's per-call cost (two library calls per
    step for a quantize + GEMM pair) stays out of the device time."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for f in fns:
            f()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(reps):
            fns[i % len(fns)]()
    g.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(batches):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b) / reps)
    return times


def graph_fields(fns, algo_bytes, hbm):
    """The same back-to-back launches replayed from a CUDA graph, as a decode
    loop would issue them: without the stream's per-launch gap (~2 us on
    this GPU between eagerly launched kernels)."""
    t = statistics.median(timed_graph(fns, 40))
    gbs = algo_bytes / t / 1e6
    return {"ms_graph": round(t, 5), "gbs_graph": round(gbs, 1), "frac_graph": round(gbs / hbm, 4)}


def bench_rows(dev, flush, hbm, tf_burst, quick):
    """The other workloads of the layer, per launch (GEMM kernel only)."""
    import bit_quantized_gemm_gb300 as qg
    rows = {}
    reps = 5 if quick else 10

    def w8a8_rows(name, shapes):
        by_kn = {}
        small = all(M <= 64 for (M, _, _) in shapes)
        for (M, K, N) in shapes:
            if (K, N) not in by_kn:
                blocks = torch.from_numpy(synth.config_weights(name, N, K)).to(dev)
                by_kn[(K, N)] = [qg.pack_q8_0(blocks, N, K)
                                 for _ in range(ROTATE_COPIES if small else 1)]
                del blocks
            packs = by_kn[(K, N)]
            x, bits = synth.config_activations(name, M, K)
            xd = torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)
            q, s, _, h = qg.quantize_act(xd, q16=True)
            out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            fns = [lambda p=p: qg.gemm_w8a8_q8_0(q, h, s, p, N, out=out) for p in packs]
            fns[0]()
            if M <= 64:
                t = statistics.median(timed_rotating(fns, 40))
            else:
                t = statistics.median(timed_launches(fns[0], reps, flush))
            ops = 2.0 * M * N * K
            key = "%s_M%d_K%d_N%d" % (name, M, K, N)
            r = {"ms": round(t, 5), "tops": round(ops / t / 1e9, 2)}
            if M <= 64:
                wbytes = N * K + N * (K // 32) * 2
                algo = wbytes + M * K + 4 * M + 2 * M * N
                gbs = algo / t / 1e6
                r.update({"gbs": round(gbs, 1), "bound": "hbm", "frac": round(gbs / hbm, 4)})
                r.update(graph_fields(fns, algo, hbm))
            else:
                r.update({"bound": "tensor", "frac": round(ops / t / 1e9 / tf_burst, 4)})
            rows[key] = r
        by_kn.clear()

    w8a8_rows("decode_w8a8", synth.CONFIGS["decode_w8a8"]["shapes"])
    torch.cuda.empty_cache()
    w8a8_rows("prefill_4b_w8a8", synth.CONFIGS["prefill_4b_w8a8"]["shapes"])
    torch.cuda.empty_cache()
    rows.update(quantize_rows(dev, flush, hbm, reps))
    torch.cuda.empty_cache()
    # W4A8
    name = "w4a8_q4k"
    shapes = synth.CONFIGS[name]["shapes"]
    M0, K, N = shapes[0]
    sblocks = torch.from_numpy(synth.config_weights(name, N, K)).to(dev)
    packs = [qg.pack_q4k(sblocks, N, K) for _ in range(ROTATE_COPIES)]
    del sblocks
    for (M, K, N) in shapes:
        x, bits = synth.config_activations(name, M, K)
        xd = torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)
        q, s, bs, h = qg.quantize_act(xd, block_sums=True, q16=True)
        out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        fns = [lambda p=p: qg.gemm_w4a8_q4k(q, h, s, bs, p, N, out=out) for p in packs]
        fns[0]()
        if M <= 64:
            t = statistics.median(timed_rotating(fns, 40))
        else:
            t = statistics.median(timed_launches(fns[0], reps, flush))
        ops = 2.0 * M * N * K
        r = {"ms": round(t, 5), "tops": round(ops / t / 1e9, 2)}
        if M <= 64:
            algo = N * K // 256 * 144 + M * K + 4 * M + 4 * M * (K // 32) + 2 * M * N
            gbs = algo / t / 1e6
            r.update({"gbs": round(gbs, 1), "bound": "hbm", "frac": round(gbs / hbm, 4)})
            r.update(graph_fields(fns, algo, hbm))
        else:
            r.update({"bound": "tensor", "frac": round(ops / t / 1e9 / tf_burst, 4)})
        rows["%s_M%d_K%d_N%d" % (name, M, K, N)] = r
    del packs
    torch.cuda.empty_cache()
    rows.update(layer_rows(dev, hbm))
    return rows


def quantize_rows(dev, flush, hbm, reps):
    """The activation quantizer alone on the prefill shapes, per launch after
    an L2 flush, as the benchmark step calls it (fp16 copy of q only, the
    prefill GEMM's operand). HBM bytes = bf16 x read + fp16 q16 written +
    the fp32 row scales; `frac_int8_contract` uses the 3 B per element of an
    int8 output instead (bf16 in, int8 out)."""
    import bit_quantized_gemm_gb300 as qg
    rows = {}
    shapes = [(8192, 5120), (8192, 17408), (2048, 2560), (2048, 9728)]
    for (M, K) in shapes:
        x, bits = synth.activations(11, M, K, dtype="bf16", outlier_frac=0.01)
        xd = torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)
        s = torch.empty((M,), dtype=torch.float32, device=dev)
        h = torch.empty((M, K), dtype=torch.float16, device=dev)
        fn = lambda: qg.quantize_act(xd, q16=True, out=(None, s, None, h))
        fn()
        t = statistics.median(timed_launches(fn, reps, flush))
        nbytes = M * K * 2 + M * K * 2 + M * 4
        gbs = nbytes / t / 1e6
        rows["quantize_M%d_K%d" % (M, K)] = {
            "ms": round(t, 5), "gbs": round(gbs, 1), "bound": "hbm", "frac": round(gbs / hbm, 4),
            "frac_int8_contract": round((3 * M * K + 4 * M) / t / 1e6 / hbm, 4)}
        del xd, h
    return rows


def layer_rows(dev, hbm):
    """The whole layer (x in, y out) at decode sizes (1 and 8 rows: the decode
    GEMM) and 64 rows (the prefill kernels) through qg_linear_* (the GEMM
    launched as a programmatic dependent of the quantize kernel)
    against qg_quantize_act and the GEMM called separately, per call, cycling
    through four weight copies like the decode rows. Each is timed as issued
    (one host call per layer against two) and replayed from a CUDA graph
    (device time only)."""
    import bit_quantized_gemm_gb300 as qg
    rows = {}
    K, N = 5120, 17408
    for kind, name in (("q8_0", "decode_w8a8"), ("q4k", "w4a8_q4k")):
        q4k = kind == "q4k"
        wts = torch.from_numpy(synth.config_weights(name, N, K)).to(dev)
        pack = qg.pack_q4k if q4k else qg.pack_q8_0
        packs = [pack(wts, N, K) for _ in range(ROTATE_COPIES)]
        del wts
        lin = qg.linear_w4a8_q4k if q4k else qg.linear_w8a8_q8_0
        for M in (1, 8, 64):
            x, bits = synth.config_activations(name, M, K)
            xd = torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)
            out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = torch.empty((qg.linear_workspace_bytes(kind, M, K),), dtype=torch.uint8,
                             device=dev)
            q = torch.empty((M, K), dtype=torch.int8, device=dev)
            s = torch.empty((M,), dtype=torch.float32, device=dev)
            bs = torch.empty((M, K // 32), dtype=torch.int32, device=dev) if q4k else None
            wide = M > qg.small_m_max()  # the prefill kernels read the fp16 copy
            h = torch.empty((M, K), dtype=torch.float16, device=dev) if wide else None

            def two(p):
                qg.quantize_act(xd, block_sums=q4k, q16=wide, out=(q, s, bs, h))
                if q4k:
                    qg.gemm_w4a8_q4k(q, h, s, bs, p, N, out=out)
                else:
                    qg.gemm_w8a8_q8_0(q, h, s, p, N, out=out)

            layer = [lambda p=p: lin(xd, p, N, out=out, workspace=ws) for p in packs]
            separate = [lambda p=p: two(p) for p in packs]
            layer[0]()
            separate[0]()
            r = {"ms": round(statistics.median(timed_rotating(layer, 40)), 5),
                 "ms_two_calls": round(statistics.median(timed_rotating(separate, 40)), 5)}
            try:
                r["ms_graph"] = round(statistics.median(timed_graph(layer, 40)), 5)
                r["ms_two_calls_graph"] = round(statistics.median(timed_graph(separate, 40)), 5)
            except RuntimeError as e:  # capture unavailable: keep the issued timings
                r["graph"] = "unavailable: %s" % str(e).splitlines()[0][:120]
            wbytes = N * K // 256 * 144 if q4k else N * K + N * (K // 32) * 2
            algo = wbytes + 2 * M * K + 2 * M * N  # weights, bf16 x, bf16 out
            gbs = algo / r["ms"] / 1e6
            r.update({"launches": 1 + qg.gemm_launch_count(kind, M, K, N), "gbs": round(gbs, 1),
                      "bound": "hbm",
                      "frac": round(gbs / hbm, 4)})
            rows["layer_%s_M%d_K%d_N%d" % (name, M, K, N)] = r
        del packs
        torch.cuda.empty_cache()
    return rows


def oracle_step_data(layers, rows_sample):
    """Host inputs of a `rows_sample`-row slice of the step (the seeded bf16
    activations and Q8_0 blocks the GPU arm uploaded; rows are independent,
    so a slice is a fair sample)."""
    return [(np.ascontiguousarray(L["bits"][:rows_sample]), L["blocks"], L["N"], L["K"])
            for L in layers]


def host_step_inputs():
    """The step's seeded host inputs, without a GPU (the --impl reference arm)."""
    layers = []
    for i, (M, K, N) in enumerate(STEP_SHAPES):
        _, bits = synth.config_activations(WORKLOAD, M, K, seed_offset=i)
        blocks = synth.config_weights(WORKLOAD, N, K, seed_offset=i)
        layers.append(dict(M=M, K=K, N=N, bits=bits, blocks=blocks))
    return layers


def oracle_step(data):
    import oracle
    for bits, blocks, N, K in data:
        q, s = oracle.quantize_act(bits)
        oracle.gemm_w8a8_q8_0(q, s, blocks)


def cpu_baseline(layers, rows_sample=CPU_SAMPLE_ROWS):
    """The oracle, as it stands, timed on a bounded sample of the step:
    `rows_sample` of the 8192 rows of both projections (quantize + GEMM), on
    all host cores (input generation excluded)."""
    import oracle
    oracle.build()
    data = oracle_step_data(layers, rows_sample)
    t0 = time.perf_counter()
    oracle_step(data)
    dt = time.perf_counter() - t0
    ops = sum(2.0 * rows_sample * N * K for (_, _, N, K) in data)
    return {"value": round(ops / dt / 1e12, 6), "unit": "TOPS", "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": "%d of %d rows of both projections (quantize + W8A8 GEMM)"
                      % (rows_sample, STEP_SHAPES[0][0])}


# Token-row chunks per projection in the end-to-end step: chunk i's input
# copy, compute and output copy overlap the neighbouring chunks' (rows are
# batch-invariant, so chunking changes no bit of the output). The step is
# bound by the host copies (~210 GB/s host to device, ~190 back, ~160 each
# when both run); only the first input copy and the last output copy stay
# outside the overlap. Measured on GB300 for the 8192-token step (ms):
# (1, 1) 4.42, (2, 1) 4.29, (1, 2) 4.34, (2, 2) 4.21, (4, 2) 4.23, (4, 4)
# 4.38 -- four chunks' smaller GEMMs cost more than the shorter copies save.
E2E_CHUNKS = (2, 2)


def make_e2e_step(layers, dev, chunks=None):
    """The step through the public API with pinned host buffers in and out.

    Input copies run on one stream, the library's launches on the current
    stream, output copies on a third (the two directions use separate copy
    engines). Each projection is split into token-row chunks: a chunk's
    quantize + GEMM waits only for its own input rows, and its output rows
    leave as soon as its GEMM is done. Returns (step, h2d_bytes, d2h_bytes,
    host_outputs)."""
    import bit_quantized_gemm_gb300 as qg
    chunks = tuple(chunks or E2E_CHUNKS)
    hx = [L["x"].cpu().pin_memory() for L in layers]
    hout = [torch.empty(L["out"].shape, dtype=torch.bfloat16).pin_memory() for L in layers]
    h2d = sum(t.numel() * t.element_size() for t in hx)
    d2h = sum(t.numel() * t.element_size() for t in hout)
    copy_stream = torch.cuda.Stream(device=dev)   # host -> device
    back_stream = torch.cuda.Stream(device=dev)   # device -> host
    plan = []  # per layer: row ranges
    for L, c in zip(layers, chunks):
        M = L["M"]
        step_rows = -(-M // c)
        plan.append([(r, min(M, r + step_rows)) for r in range(0, M, step_rows)])

    def step():
        comp = torch.cuda.current_stream(dev)  # (a capture stream while a graph records it)
        copy_stream.wait_stream(comp)  # the copies start after the timing event
        back_stream.wait_stream(comp)
        copied = []
        with torch.cuda.stream(copy_stream):
            for L, hxi, ranges in zip(layers, hx, plan):
                for (r0, r1) in ranges:
                    L["x"][r0:r1].copy_(hxi[r0:r1], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(copy_stream)
                    copied.append(ev)
        done = []
        k = 0
        for L, ranges in zip(layers, plan):
            for (r0, r1) in ranges:
                comp.wait_event(copied[k])
                k += 1
                q = L["q"][r0:r1] if L["q"] is not None else None
                qg.quantize_act(L["x"][r0:r1], q16=True,
                                out=(q, L["s"][r0:r1], None, L["h"][r0:r1]))
                qg.gemm_w8a8_q8_0(q, L["h"][r0:r1], L["s"][r0:r1], L["packed"], L["N"],
                                  out=L["out"][r0:r1])
                ev2 = torch.cuda.Event()
                ev2.record(comp)
                done.append(ev2)
        k = 0
        with torch.cuda.stream(back_stream):
            for L, ho, ranges in zip(layers, hout, plan):
                for (r0, r1) in ranges:
                    back_stream.wait_event(done[k])
                    k += 1
                    ho[r0:r1].copy_(L["out"][r0:r1], non_blocking=True)
        comp.wait_stream(copy_stream)
        comp.wait_stream(back_stream)

    return step, h2d, d2h, hout


def run_only(args):
    """One kernel of the layer on one shape: for profiling and quick timing."""
    import bit_quantized_gemm_gb300 as qg
    kind, dims = args.only.split(":")
    M, K, N = (int(v) for v in dims.split(","))
    dev = torch.device("cuda", 0)
    name = "w4a8_q4k" if kind == "w4a8" else "prefill_27b_w8a8"
    x, bits = synth.activations(7, M, K, dtype="bf16", outlier_frac=0.01)
    xd = torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)
    q, s, bs, h = qg.quantize_act(xd, block_sums=True, q16=True)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    copies = ROTATE_COPIES if M <= 64 else 1
    fns = None
    if kind == "w8a8":
        wb = torch.from_numpy(synth.q8_0_weights(107, N, K)).to(dev)
        packs = [qg.pack_q8_0(wb, N, K) for _ in range(copies)]
        fns = [lambda p=p: qg.gemm_w8a8_q8_0(q, h, s, p, N, out=out, path=args.path)
               for p in packs]
    elif kind == "w4a8":
        wb = torch.from_numpy(synth.q4k_weights(107, N, K)).to(dev)
        packs = [qg.pack_q4k(wb, N, K) for _ in range(copies)]
        fns = [lambda p=p: qg.gemm_w4a8_q4k(q, h, s, bs, p, N, out=out, path=args.path)
               for p in packs]
    elif kind == "quant":
        fn = lambda: qg.quantize_act(xd, q16=True, out=(q, s, None, h))
    else:
        raise SystemExit("unknown kind " + kind)
    if fns is not None:
        fn = fns[0]
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush = lambda: flush_buf.fill_(1)
    for _ in range(args.warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    if fns is not None and copies > 1:
        t = timed_rotating(fns, 40, batches=max(args.steps, 3))
    else:
        t = timed_launches(fn, args.steps, flush)
    qg.check_device_error()
    ms = statistics.median(t)
    print(json.dumps({"only": args.only, "path": args.path, "ms_median": round(ms, 5),
                      "ms_all": [round(v, 5) for v in t],
                      "tops": round(2.0 * M * N * K / ms / 1e9, 2)}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-rows", action="store_true", help="skip the per-workload rows")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--only", default=None,
                    help="KIND:M,K,N (KIND w8a8|w4a8|quant): time that one launch alone "
                         "(--warmup untimed + --steps timed launches, L2 flushed before each); "
                         "used for profiling")
    ap.add_argument("--path", default="auto", choices=["auto", "small", "large"])
    args = ap.parse_args()
    rank, world, local = env_rank()
    hbm, tf_burst, tf_sus, peak_src = measured_peaks()

    if args.impl == "reference":
        if rank != 0:
            return
        # The CPU oracle on a bounded sample of the same step (REF_SAMPLE_ROWS per step).
        import oracle
        oracle.build()
        rows_sample = REF_SAMPLE_ROWS
        data = oracle_step_data(host_step_inputs(), rows_sample)

        def ref_step():
            oracle_step(data)
        for _ in range(args.warmup):
            ref_step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            ref_step()
        dt = (time.perf_counter() - t0) / args.steps
        ops = sum(2.0 * rows_sample * N * K for (_, _, N, K) in data)
        v = ops / dt / 1e12
        line = {"metric": METRIC, "value": round(v, 6), "unit": "TOPS", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "int8", "data": "synthetic", "impl": "reference",
                "config": {"workload": WORKLOAD, "shapes": STEP_SHAPES, "sample_rows": rows_sample},
                "cpu_baseline": {"value": round(v, 6), "unit": "TOPS", "cores": oracle.num_threads(),
                                 "kind": "oracle",
                                 "sample": "%d of %d rows of both projections per step"
                                           % (rows_sample, STEP_SHAPES[0][0])},
                "e2e": {"value": round(v, 6), "unit": "TOPS", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}))
        sys.exit(1)
    if args.only:
        return run_only(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    import bit_quantized_gemm_gb300 as qg
    qg.load()

    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def flush():
        flush_buf.fill_(1)

    layers = make_step_inputs(dev)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    step_ms, gemm_ms = [], []
    with ClockSampler(local) as clk:
        for _ in range(max(args.warmup, 3)):
            run_step(layers)
        torch.cuda.synchronize()
        barrier()
        t_wall0 = time.perf_counter()
        t_unix0 = time.time()
        for _ in range(args.steps):
            flush()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in layers]
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            run_step(layers, ev)
            b.record()
            b.synchronize()
            step_ms.append(a.elapsed_time(b))
            gemm_ms.append([e0.elapsed_time(e1) for e0, e1 in ev])
        barrier()
        t_wall = time.perf_counter() - t_wall0
        t_unix1 = time.time()
    clocks = clk.summary((t_unix0, t_unix1))
    ms = reduce_max(sum(step_ms) / len(step_ms), world)
    ops = step_ops()
    value = job_value(ops, world, ms)

    # roofline of the dominant kernel (the prefill GEMM; both shapes of the step)
    gemm_tot = sum(sum(g) for g in gemm_ms) / len(gemm_ms)
    achieved = ops / (gemm_tot * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": tf_burst,
                "unit": "TFLOP/s", "frac": round(achieved / tf_burst, 4),
                "traffic": measured_traffic(),
                "peak_source": "%s bf16 dense burst (same rate as the fp16 kind the kernel uses)"
                               % peak_src,
                "kernel": step_kernels(dev),
                "algorithmic_bytes_per_call": int(sum(
                    N * K + N * (K // 32) * 2 + M * K + 2 * M * N for (M, K, N) in STEP_SHAPES)
                    / len(STEP_SHAPES)),
                "per": "GEMM call (one or two launches of the kernel): achieved = 2*M*N*K of "
                       "the step's two calls / their CUDA-event time; traffic = DRAM bytes "
                       "of one call, mean of the two",
                "gemm_ms_per_step": round(gemm_tot, 4),
                "gemm_ms": [round(sum(g[i] for g in gemm_ms) / len(gemm_ms), 4)
                            for i in range(len(STEP_SHAPES))]}

    # end to end through the public API with host buffers
    e2e = None
    if rank == 0 or world > 1:
        e2e_step, h2d, d2h, _ = make_e2e_step(layers, dev)
        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        et = []
        for _ in range(max(3, args.steps // 2)):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            e2e_step()
            b.record()
            b.synchronize()
            et.append(a.elapsed_time(b))
        e2e_ms = sum(et) / len(et)
        e2e = {"value": round(world * ops / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TOPS",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)}

    host = [dict(bits=L["bits"], blocks=L["blocks"], N=L["N"], K=L["K"]) for L in layers]
    rows = None
    del layers
    torch.cuda.empty_cache()
    if not args.no_rows:
        rows = bench_rows(dev, flush, hbm, tf_burst, quick=True)

    # one quantize launch per projection, plus the GEMM's own launches (the
    # prefill GEMM splits a ragged last wave into a second, narrow-tile launch)
    launches_per_step = sum(1 + qg.gemm_launch_count("q8_0", M, K, N) for (M, K, N) in STEP_SHAPES)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(host)

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 3), "unit": "TOPS", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "int8", "data": "synthetic",
                "config": {"workload": WORKLOAD, "shapes_MKN": STEP_SHAPES,
                           "parallelism": "replicas" if world > 1 else "single",
                           "l2": "flushed between timed steps (512 MiB write, outside events)",
                           "wall_s": round(t_wall, 3)},
                "gpu_launches": launches_per_step * args.steps,
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
                "rows": rows}
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

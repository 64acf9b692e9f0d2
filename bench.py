"""Benchmark of the int4g hot path on one GB300 (prints one JSON line).

Workload (the timed step): Llama-7B-shaped decode linears, int4g group 128:
fused QKV (K=4096, N=12288), gate and up (K=4096, N=11008 each) and down
(K=11008, N=4096), at M = 1, 8 and 32 tokens -- 12 calls per step, each on
its own weight matrix (3 layer copies x 4 matrices, 290 MB, more than twice
the 129 MB L2, read in the same order every step, so no call finds its
weights in L2).  value = int4g weight bytes streamed per step / step time.

Also reported in the same line: prefill GEMM TFLOP/s and MoE-layer tokens/s
sections when those paths are measured (see --sections), the roofline of the
dominant kernel from per-launch CUDA events, SM clocks sampled during the
timed region, an end-to-end number through the public API with host
buffers, and the CPU oracle timed on a bounded sample (cpu_baseline).

--impl reference times the CPU oracle itself on a bounded sample of the same
workload and metric.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "int4g GEMV weight GB/s (% HBM peak); MoE layer tokens/s; GEMM % bf16 peak"
BYTES_PER_WEIGHT = 0.51953125          # 0.5 B code + 2 B scale / 128 + 0.5 B zero / 128
LLAMA = [("qkv", 4096, 12288), ("gate", 4096, 11008), ("up", 4096, 11008), ("down", 11008, 4096)]
DECODE_M = [1, 8, 32]
# DRAM traffic / algorithmic bytes of k_linear_rows, from one ncu capture of
# the M=1 fused-QKV launch (summary kept under profiles/): 26,214,144 B
# read, 0 written, for 26,181,632 algorithmic bytes.  Traffic grows in
# proportion to the super-blocks a launch streams, so the per-launch traffic
# is scaled from it.  Reset to None whenever the kernel changes after that
# capture.
TRAFFIC_RATIO = 26214144 / 26181632
WORKLOAD = "llama7b-decode-linears int4g g128: (K,N) in {(4096,12288),(4096,11008)x2,(11008,4096)} x M in {1,8,32}"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# --------------------------------------------------------------- clocks
class ClockSampler:
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
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
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
        self.f.close()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = max(mx, float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- GPU arm
def build_weights(torch, fl, inputs, n_layers, dev):
    """Per layer copy: the 4 Llama matrices quantized on the device (W ~ N(0, .02)
    with 0.1% outliers x20, drawn by the device generator) and repacked."""
    mats = []
    for layer in range(n_layers):
        row = []
        for name, K, N in LLAMA:
            W = inputs.device_normal((N, K), 1, layer, K, N, device=dev)
            n_out = int(round(inputs.OUTLIER_FRAC * N * K))
            g = torch.Generator(device=dev)
            g.manual_seed(inputs._seed64(4, layer, K, N))
            pos = torch.unique(torch.randint(0, N * K, (n_out + n_out // 8,), generator=g, device=dev))[:n_out]
            W.view(-1)[pos] *= inputs.OUTLIER_MUL
            q, s, z = fl.fl_int4g_quantize(W)
            del W
            w = fl.fl_int4g_repack(q, s, z, N, K)
            del q, s, z
            row.append((name, K, N, w))
        mats.append(row)
    torch.cuda.synchronize()
    return mats


QWEN = dict(name="qwen3-moe", E=128, H=2048, I=768, k=8, scoring=0, shared=False, hot=0, Ms=(1, 64, 256))
DSV3 = dict(name="deepseek-v3-moe", E=256, H=7168, I=2048, k=8, scoring=1, shared=True, hot=51, Ms=(1, 16, 128, 1024))
PREFILL = [(512, 4096, 11008), (512, 11008, 4096), (2048, 4096, 11008), (2048, 11008, 4096)]


def _flush_l2(torch, buf):
    buf.add_(1)          # 256 MB read+write: evicts the 129 MB L2


def _median_time(torch, fn, flush, reps, stream):
    """Median CUDA-event time of fn() over reps calls, L2 flushed before each."""
    ts = []
    for _ in range(reps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def run_moe_section(torch, np, fl, inputs, dev, pk, reps, cfgs=(QWEN, DSV3)):
    """MoE layer tokens/s for the Qwen3- and DeepSeek-V3-shaped configs."""
    out = {}
    stream = torch.cuda.current_stream()
    flushbuf = torch.zeros(64 << 20, dtype=torch.float32, device=dev)
    for cfg in cfgs:
        E, H, I, k = cfg["E"], cfg["H"], cfg["I"], cfg["k"]

        def packed(e, which, layer=1000):
            N, K = (2 * I, H) if which == 0 else (H, I)
            W = inputs.device_normal((N, K), 1, layer, e, which, device=dev)
            q, s, z = fl.fl_int4g_quantize(W)
            del W
            return fl.fl_int4g_repack(q, s, z, N, K)

        w13 = torch.cat([packed(e, 0) for e in range(E)])
        w2 = torch.cat([packed(e, 1) for e in range(E)])
        sw13 = packed(E, 0) if cfg["shared"] else None
        sw2 = packed(E, 1) if cfg["shared"] else None
        eb = (w13.numel() + w2.numel()) / E
        sb = (sw13.numel() + sw2.numel()) if cfg["shared"] else 0
        res = {}
        for M in cfg["Ms"]:
            x = torch.from_numpy(inputs.activations(M, H, stream=M).view(np.int16)).to(dev).view(torch.bfloat16)
            lg = torch.from_numpy(inputs.router_logits(M, E, stream=M, hot=cfg["hot"])).to(dev)
            y = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
            ids = torch.empty((M, k), dtype=torch.int32, device=dev)
            ws = torch.zeros(fl.fl_moe_int4g_workspace(M, E, k, H, I, cfg["shared"]), dtype=torch.uint8, device=dev)

            def call():
                fl.fl_moe_int4g(x, lg, k, I, w13, w2, scoring=cfg["scoring"], renorm=True, shared_w13=sw13,
                                shared_w2=sw2, y=y, topk_ids=ids, ws=ws)
            call()
            torch.cuda.synchronize()
            assert fl.fl_int4g_status(ws) == 0
            ms = _median_time(torch, call, lambda: _flush_l2(torch, flushbuf), reps, stream)
            touched = int(torch.unique(ids).numel())
            nbytes = touched * eb + sb + 2 * M * H * 2
            flops = 2.0 * (M * k + (M if cfg["shared"] else 0)) * 3 * H * I
            t_roof = max(nbytes / (pk["hbm_gbs"] * 1e9), flops / (pk["bf16_tflops"] * 1e12))
            res[str(M)] = {"ms": round(ms, 4), "tokens_per_s": round(M / (ms * 1e-3), 1),
                           "experts_touched": touched, "weight_GB": round(nbytes / 1e9, 4),
                           "GBps": round(nbytes / (ms * 1e-3) / 1e9, 1),
                           "roofline_frac_of_measured": round(t_roof / (ms * 1e-3), 4)}
        out[cfg["name"]] = res
        del w13, w2, sw13, sw2
        torch.cuda.empty_cache()
    return out


def _graph_time_per_launch(torch, launches, stream, replays):
    """Mean time per launch (ms) of `launches` (callables) captured in one
    CUDA graph, over `replays` replays after one warm-up replay; CUDA events
    on the launching stream."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        launches[0]()
        stream.synchronize()
    with torch.cuda.graph(g, stream=stream):
        for f in launches:
            f()
    with torch.cuda.stream(stream):
        g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(replays):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (replays * len(launches))


def _weight_copies(torch, fl, inputs, dev, K, N, copies, layer0):
    out = []
    for i in range(copies):
        W = inputs.device_normal((N, K), 1, layer0 + i, K, N, device=dev)
        q, s, z = fl.fl_int4g_quantize(W)
        del W
        out.append(fl.fl_int4g_repack(q, s, z, N, K))
        del q, s, z
    return out


def run_gemv_config1(torch, np, fl, inputs, dev, pk):
    """The single int4g GEMV, M=1, K=1024, N=3072 (Qwen3-0.6B up_proj shape):
    192 weight copies (313 MB, more than twice the L2) in one CUDA graph of
    192 launches, replayed 3 times (576 timed launches)."""
    M, K, N, copies = 1, 1024, 3072, 192
    ws_list = _weight_copies(torch, fl, inputs, dev, K, N, copies, 3000)
    x = torch.from_numpy(inputs.activations(M, K, stream=0).view(np.int16)).to(dev).view(torch.bfloat16)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(fl.fl_int4g_linear_workspace(M, N, K), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    ms = _graph_time_per_launch(torch, [lambda w=w: fl.fl_int4g_linear(x, w, N, y=y, ws=ws) for w in ws_list],
                                stream, 3)
    assert fl.fl_int4g_status(ws) == 0
    wb = BYTES_PER_WEIGHT * N * K
    algo = wb + 2 * M * K + 2 * M * N
    del ws_list
    torch.cuda.empty_cache()
    return {"shape": "M=1 K=1024 N=3072", "us_per_launch": round(ms * 1e3, 3),
            "weight_GBps": round(wb / (ms * 1e-3) / 1e9, 1), "algo_GBps": round(algo / (ms * 1e-3) / 1e9, 1),
            "hbm_frac_of_measured": round(algo / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
            "timing": "graph of 192 launches over 192 weight copies (313 MB), 3 replays"}


def run_gemm_section(torch, np, fl, inputs, dev, pk):
    """Prefill int4g GEMM TFLOP/s (M in {512, 2048}): per shape, 12 weight
    copies (281 MB) in one CUDA graph of 24 launches, replayed 3 times."""
    out = {}
    stream = torch.cuda.Stream(device=dev)
    for K, N in sorted(set((K, N) for (_m, K, N) in PREFILL)):
        ws_list = _weight_copies(torch, fl, inputs, dev, K, N, 12, 77)
        for M in sorted(set(m for (m, k, n) in PREFILL if (k, n) == (K, N))):
            x = torch.from_numpy(inputs.activations(M, K, stream=M).view(np.int16)).to(dev).view(torch.bfloat16)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = torch.zeros(fl.fl_int4g_linear_workspace(M, N, K), dtype=torch.uint8, device=dev)
            launches = [lambda w=w: fl.fl_int4g_linear(x, w, N, y=y, ws=ws) for w in ws_list * 2]
            ms = _graph_time_per_launch(torch, launches, stream, 3)
            assert fl.fl_int4g_status(ws) == 0
            tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
            out[f"M{M}_K{K}_N{N}"] = {"ms": round(ms, 4), "TFLOPs": round(tf, 2),
                                     "frac_of_measured_bf16": round(tf / pk["bf16_tflops"], 4),
                                     "timing": "graph of 24 launches over 12 weight copies, 3 replays"}
        del ws_list
        torch.cuda.empty_cache()
    return out


def _mlp_copies(torch, fl, inputs, dev, H, I, copies, layer0):
    out = []
    for i in range(copies):
        out.append(tuple(_weight_copies(torch, fl, inputs, dev, K, N, 1, layer0 + 10 * i + j)[0]
                         for j, (K, N) in enumerate([(H, I), (H, I), (I, H)])))
    return out


def run_mlp_section(torch, np, fl, inputs, dev, pk, Ms=(1, 8)):
    """Llama-7B MLP block (H=4096, I=11008: gate, up, down; 70.3 MB of int4g
    weights) at M in {1, 8}: fl_int4g_mlp (gate/up + SwiGLU launch, then the
    down launch), the one-launch cooperative form (fl_int4g_mlp_fused) and,
    for comparison, the same three matrices as three fl_int4g_linear calls
    (SwiGLU not applied there).  4 weight copies (281 MB) in one CUDA graph,
    replayed 30 times."""
    H, I = 4096, 11008
    copies = _mlp_copies(torch, fl, inputs, dev, H, I, 4, 5000)
    wb = BYTES_PER_WEIGHT * 3 * H * I
    stream = torch.cuda.Stream(device=dev)
    out = {}
    for M in Ms:
        x = torch.from_numpy(inputs.activations(M, H, stream=M).view(np.int16)).to(dev).view(torch.bfloat16)
        y = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
        ws = torch.zeros(fl.fl_int4g_mlp_workspace(M, H, I), dtype=torch.uint8, device=dev)
        ms = _graph_time_per_launch(torch, [lambda c=c: fl.fl_int4g_mlp(x, c[0], c[1], c[2], I, y=y, ws=ws)
                                            for c in copies], stream, 30)
        ms1 = _graph_time_per_launch(torch, [lambda c=c: fl.fl_int4g_mlp(x, c[0], c[1], c[2], I, y=y, ws=ws,
                                                                         one_launch=True)
                                             for c in copies], stream, 30)
        assert fl.fl_int4g_status(ws) == 0
        hx = torch.from_numpy(inputs.activations(M, I, stream=M).view(np.int16)).to(dev).view(torch.bfloat16)
        gu = torch.empty((M, I), dtype=torch.bfloat16, device=dev)
        lw = torch.zeros(max(fl.fl_int4g_linear_workspace(M, I, H), fl.fl_int4g_linear_workspace(M, H, I)),
                         dtype=torch.uint8, device=dev)
        launches = []
        for c in copies:
            launches += [lambda c=c: fl.fl_int4g_linear(x, c[0], I, y=gu, ws=lw),
                         lambda c=c: fl.fl_int4g_linear(x, c[1], I, y=gu, ws=lw),
                         lambda c=c: fl.fl_int4g_linear(hx, c[2], H, y=y, ws=lw)]
        ms3 = _graph_time_per_launch(torch, launches, stream, 30) * 3
        out[str(M)] = {"us_per_block": round(ms * 1e3, 3), "weight_GBps": round(wb / (ms * 1e-3) / 1e9, 1),
                       "hbm_frac_of_measured": round(wb / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
                       "one_launch_us": round(ms1 * 1e3, 3), "one_launch_GBps": round(wb / (ms1 * 1e-3) / 1e9, 1),
                       "three_linear_calls_us": round(ms3 * 1e3, 3),
                       "three_linear_calls_GBps": round(wb / (ms3 * 1e-3) / 1e9, 1)}
    del copies
    torch.cuda.empty_cache()
    out["timing"] = "graph of 4 blocks over 4 weight copies (281 MB), 30 replays; weight bytes 70.3 MB per block"
    return out


def input_digests(np, calls):
    """numpy / torch versions and SHA-256 (first 16 hex digits) of each decode
    call's inputs: x (bf16 bits) and the interleaved weights."""
    import hashlib
    import torch
    d = {}
    for (M, K, N, x, w, y, ws) in calls:
        h = hashlib.sha256()
        h.update(x.view(torch.int16).cpu().numpy().tobytes())
        h.update(w.cpu().numpy().tobytes())
        d[f"M{M}_K{K}_N{N}"] = h.hexdigest()[:16]
    return {"numpy": np.__version__, "torch": torch.__version__, "sha256_x_and_w": d}


def run_gpu(args, barrier=None):
    """One GPU's run.  barrier: called just before and just after the timed
    region (after a device synchronize), so that replicas start and stop
    their timed steps together."""
    import numpy as np
    import torch

    import int4_group_quantized_int4g_gb300 as fl
    from int4_group_quantized_int4g_gb300 import _build, inputs

    _build.build()
    fl.lib()
    dev = torch.device("cuda", torch.cuda.current_device())
    torch.cuda.set_device(dev)
    pk = peaks()

    mats = build_weights(torch, fl, inputs, len(DECODE_M), dev)
    calls = []          # (M, K, N, x, w, y, ws)
    for li, M in enumerate(DECODE_M):
        for name, K, N, w in mats[li]:
            x = torch.from_numpy(inputs.activations(M, K, stream=M).view(np.int16)).to(dev).view(torch.bfloat16)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = torch.zeros(fl.fl_int4g_linear_workspace(M, N, K), dtype=torch.uint8, device=dev)
            calls.append((M, K, N, x, w, y, ws))
    wbytes = sum(BYTES_PER_WEIGHT * N * K for (M, K, N, *_r) in calls)

    stream = torch.cuda.Stream(device=dev)

    def launch_all(subset=None):
        for (M, K, N, x, w, y, ws) in (subset or calls):
            fl.fl_int4g_linear(x, w, N, y=y, ws=ws)

    # warm the launch path (sets kernel attributes) outside capture
    with torch.cuda.stream(stream):
        launch_all()
    stream.synchronize()

    # The step is one CUDA graph of the 12 launches; consecutive launches are
    # linked by programmatic dependent launch, so no timing node may sit between
    # them.  The per-launch duration of the (only) kernel is the timed region
    # divided by the number of launches in it.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        launch_all()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    stream.synchronize()

    uuid = str(torch.cuda.get_device_properties(dev).uuid)
    clk = ClockSampler(uuid if uuid.startswith("GPU-") else "GPU-" + uuid)
    clk.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    with torch.cuda.stream(stream):
        t0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        t1.record(stream)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    clocks = clk.stop()
    ms_total = t0.elapsed_time(t1)
    ms_step = ms_total / args.steps
    value = wbytes / (ms_step * 1e-3) / 1e9

    # per-M breakdown (outside the timed region): a graph of each M's calls
    # over all 3 layer copies (12 launches, 290 MB of distinct weights, more
    # than twice the L2), replayed 20 times after a warm-up replay
    per_m = {}
    for M in DECODE_M:
        sub = []
        for li in range(len(mats)):
            for name, K, N, w in mats[li]:
                c = next(c for c in calls if c[0] == M and c[1] == K and c[2] == N)
                sub.append((M, K, N, c[3], w, c[5], c[6]))
        gm = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gm, stream=stream):
            launch_all(sub)
        with torch.cuda.stream(stream):
            gm.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(20):
                gm.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        b = 20 * sum(BYTES_PER_WEIGHT * N * K for (_m, K, N, *_r) in sub)
        per_m[M] = round(b / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)

    # roofline of the dominant kernel, k_linear_rows (the M <= 8 calls): a
    # graph of its launches at M = 1 and 8 over all 3 layer copies (24
    # launches; 290 MB of distinct weights between two reads of one matrix,
    # so every launch streams from HBM), timed with CUDA events on the
    # launching stream
    rows_calls = []
    for M in (1, 8):
        for li in range(len(mats)):
            for name, K, N, w in mats[li]:
                c = next(c for c in calls if c[0] == M and c[1] == K and c[2] == N)
                rows_calls.append((M, K, N, c[3], w, c[5], c[6]))
    g_rows = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_rows, stream=stream):
        launch_all(rows_calls)
    reps_rows = 100
    with torch.cuda.stream(stream):
        for _ in range(3):
            g_rows.replay()
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        r0.record(stream)
        for _ in range(reps_rows):
            g_rows.replay()
        r1.record(stream)
    torch.cuda.synchronize()
    rows_launch_s = r0.elapsed_time(r1) * 1e-3 / (reps_rows * len(rows_calls))
    rows_algo = sum(BYTES_PER_WEIGHT * N * K + 2 * M * K + 2 * M * N for (M, K, N, *_r) in rows_calls) / len(rows_calls)
    achieved = rows_algo / rows_launch_s / 1e9

    for (M, K, N, x, w, y, ws) in calls:
        assert torch.isfinite(y.float()).all(), "non-finite output"
    st = [fl.fl_int4g_status(ws) for (*_r, ws) in calls]
    assert all(v == 0 for v in st), f"device status {st}"

    # ---- end to end through the public API with pinned host buffers: every
    # step copies its 12 inputs host -> device in one transfer, makes the 12
    # library calls, and reads the 12 outputs back in one transfer.  Measured
    # two ways:
    #  - pipelined (the reported value): double-buffered device inputs and
    #    outputs; step i+1's inputs go in and step i-1's outputs come out on
    #    two copy streams while step i computes, as a serving loop would;
    #  - serial: copy in, compute, copy out, one after the other.
    # Every step's transfers are inside the timed region in both.
    xs = [2 * M * K for (M, K, N, *_r) in calls]
    ys = [2 * M * N for (M, K, N, *_r) in calls]
    h2d, d2h = sum(xs), sum(ys)
    NBUF = 2
    host_xb = [torch.empty(h2d, dtype=torch.uint8).pin_memory() for _ in range(NBUF)]
    host_yb = [torch.empty(d2h, dtype=torch.uint8).pin_memory() for _ in range(NBUF)]
    dev_xb = [torch.empty(h2d, dtype=torch.uint8, device=dev) for _ in range(NBUF)]
    dev_yb = [torch.empty(d2h, dtype=torch.uint8, device=dev) for _ in range(NBUF)]
    e2e_calls = [[] for _ in range(NBUF)]
    for b in range(NBUF):
        ox = oy = 0
        for (M, K, N, x, w, y, ws), nx, ny in zip(calls, xs, ys):
            host_xb[b][ox:ox + nx].copy_(x.view(torch.uint8).reshape(-1).cpu())
            xv = dev_xb[b][ox:ox + nx].view(torch.bfloat16).view(M, K)
            yv = dev_yb[b][oy:oy + ny].view(torch.bfloat16).view(M, N)
            e2e_calls[b].append((N, xv, w, yv, ws))
            ox += nx
            oy += ny
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)

    def e2e_serial_step():
        dev_xb[0].copy_(host_xb[0], non_blocking=True)
        for (N, xv, w, yv, ws) in e2e_calls[0]:
            fl.fl_int4g_linear(xv, w, N, y=yv, ws=ws)
        host_yb[0].copy_(dev_yb[0], non_blocking=True)

    def e2e_pipelined(nsteps):
        ev_in = [torch.cuda.Event() for _ in range(NBUF)]
        ev_done = [torch.cuda.Event() for _ in range(NBUF)]
        ev_out = [torch.cuda.Event() for _ in range(NBUF)]
        s_in.wait_stream(stream)
        for i in range(nsteps):
            b = i % NBUF
            with torch.cuda.stream(s_in):
                if i >= NBUF:
                    s_in.wait_event(ev_done[b])   # step i-2 has consumed dev_xb[b]
                dev_xb[b].copy_(host_xb[b], non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if i >= NBUF:
                stream.wait_event(ev_out[b])      # step i-2's outputs have left dev_yb[b]
            for (N, xv, w, yv, ws) in e2e_calls[b]:
                fl.fl_int4g_linear(xv, w, N, y=yv, ws=ws)
            ev_done[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[b])
                host_yb[b].copy_(dev_yb[b], non_blocking=True)
                ev_out[b].record(s_out)
        stream.wait_stream(s_out)
        stream.wait_stream(s_in)

    def timed(fn):
        with torch.cuda.stream(stream):
            fn(args.warmup)
        torch.cuda.synchronize()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a0.record(stream)
            fn(args.steps)
            a1.record(stream)
        torch.cuda.synchronize()
        return a0.elapsed_time(a1) / args.steps

    e2e_serial_ms = timed(lambda n: [e2e_serial_step() for _ in range(n)])
    e2e_ms = timed(e2e_pipelined)
    e2e_value = wbytes / (e2e_ms * 1e-3) / 1e9
    e2e_serial_value = wbytes / (e2e_serial_ms * 1e-3) / 1e9
    # the e2e outputs are those of the same calls on the device-resident inputs
    for b in range(NBUF):
        oy = 0
        for (M, K, N, x, w, y, ws), ny in zip(calls, ys):
            got = host_yb[b][oy:oy + ny].view(torch.bfloat16).view(M, N)
            ref = fl.fl_int4g_linear(x, w, N, ws=ws)
            assert torch.equal(got.view(torch.int16), ref.cpu().view(torch.int16)), "e2e output differs"
            oy += ny

    inputs_digest = input_digests(np, calls)
    sections = {"gemv_qwen3_up": run_gemv_config1(torch, np, fl, inputs, dev, pk),
                "mlp_block": run_mlp_section(torch, np, fl, inputs, dev, pk)}
    if not args.no_sections:
        sections["moe"] = run_moe_section(torch, np, fl, inputs, dev, pk, reps=5)
        sections["gemm"] = run_gemm_section(torch, np, fl, inputs, dev, pk)

    out = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": WORKLOAD,
            "calls_per_step": len(calls),
            "weight_bytes_per_step": int(wbytes),
            "l2": "3 layer copies (290 MB) rotated, > 2x L2 (129 MB): every call reads its weights from HBM",
            "graph": "one CUDA graph per step; launches chained by programmatic dependent launch",
            "e2e_transfers": "per step: one pinned host -> device copy of the 12 inputs, the 12 fl_int4g_linear "
                             "calls (public API, no graph), one device -> pinned host copy of the 12 outputs; "
                             "e2e.value pipelines them (double buffers: step i+1's inputs in and step i-1's "
                             "outputs out on two copy streams while step i computes); e2e.serial_value runs "
                             "copy in, compute, copy out one after the other",
            "hbm_frac_of_measured": round(value / pk["hbm_gbs"], 4),
            "per_M_weight_GBps_untimed": {str(M): v for M, v in per_m.items()},
            "inputs": inputs_digest,
        },
        "roofline": {
            "kernel": "k_linear_rows (decode int4g linear, M <= 8): the step's launches at M in {1, 8}",
            "duration": "events around 100 replays of a graph of its 24 launches (M = 1, 8 x 4 matrices x 3 layer "
                        "copies, 290 MB of distinct weights) / launches (PDL-chained)",
            "launch_us": round(rows_launch_s * 1e6, 3),
            "bytes_per_launch": round(rows_algo),
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": pk["hbm_gbs"],
            "peak_source": pk["source"] + " burst copy",
            "unit": "GB/s",
            "frac": round(achieved / pk["hbm_gbs"], 4),
            "traffic": (round(rows_algo * TRAFFIC_RATIO / 1e6, 3) if TRAFFIC_RATIO else None),
            "traffic_unit": "MB per launch (DRAM read + write of the ncu capture of the M=1 fused-QKV launch, "
                            "scaled by algorithmic bytes)",
        },
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "serial_value": round(e2e_serial_value, 1)},
        "gpu_launches": len(calls) * args.steps,
        "clocks": clocks,
        "sections": sections,
    }
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline()
    return out


# --------------------------------------------------------------- CPU oracle
# The oracle is timed in a child interpreter that never touches the GPU
# (BLAS pinned to one thread).  Per configuration a bounded sample runs on
# one core; then `cores` forked copies of the same sample run at once, and
# the all-core figure is their total work over the wall time.
_ORACLE_SAMPLE = r"""
import json, multiprocessing as mp, os, sys, time
sys.path.insert(0, {root!r})
import numpy as np
from oracle import int4g_oracle as O
from int4_group_quantized_int4g_gb300 import inputs
SECONDS, CORES, ONLY = {seconds}, {cores}, {only!r}
rows = 2048
llama = [(K, O.quantize(inputs.dense_weight(rows, K, layer=K + N))) for (_n, K, N) in {mats!r}]
def decode():
    b = 0.0
    for M in (1, 8, 32):
        for K, (Q, S, Z) in llama:
            O.linear(O.bf16_value(inputs.activations(M, K, stream=M)), Q, S, Z)
            b += 0.51953125 * rows * K
    return b
jobs = {{"decode": (decode, "GB/s", 1e-9)}}
if ONLY is None:
    c1 = O.quantize(inputs.dense_weight(3072, 1024, layer=0, outliers=False))
    x1 = O.bf16_value(inputs.activations(1, 1024, stream=0))
    def gemv():
        O.linear(x1, *c1)
        return 0.51953125 * 3072 * 1024
    pr = O.quantize(inputs.dense_weight(256, 4096, layer=77))
    xp = O.bf16_value(inputs.activations(512, 4096, stream=512))
    def prefill():
        O.linear(xp, *pr)
        return 2.0 * 512 * 256 * 4096
    def moe_case(E, H, I, k, scoring, shared, hot, layer):
        logits = inputs.router_logits(1, E, stream=1, hot=hot)
        ids, _ = O.route(logits, k, scoring, True)
        w13, w2 = {{}}, {{}}
        for e in list(ids[0]) + ([E] if shared else []):
            w13[int(e)] = O.quantize(inputs.expert_weight(2 * I, H, layer, int(e), 0))
            w2[int(e)] = O.quantize(inputs.expert_weight(H, I, layer, int(e), 1))
        x = O.bf16_value(inputs.activations(1, H, stream=1))
        def run():
            O.moe(x, logits, k, w13, w2, scoring, True, w13.get(E), w2.get(E))
            return 1.0
        return run
    jobs["gemv_qwen3_up"] = (gemv, "GB/s", 1e-9)
    jobs["prefill_M512_K4096"] = (prefill, "TFLOP/s", 1e-12)
    jobs["qwen3_moe_M1"] = (moe_case(128, 2048, 768, 8, O.SOFTMAX, False, 0, 1000), "tokens/s", 1.0)
    jobs["deepseek_moe_M1"] = (moe_case(256, 7168, 2048, 8, O.SIGMOID, True, 51, 1000), "tokens/s", 1.0)
def timed(fn):
    work, t0 = 0.0, time.perf_counter()
    while True:
        work += fn()
        t = time.perf_counter() - t0
        if t >= SECONDS:
            return work, t
def one_copy(args):
    return timed(jobs[args][0])
out = {{}}
for name, (fn, unit, scale) in jobs.items():
    w1, t1 = timed(fn)
    res = {{"unit": unit, "cores_1": w1 / t1 * scale, "seconds_1": round(t1, 2)}}
    if CORES > 1:
        t0 = time.perf_counter()
        with mp.get_context("fork").Pool(CORES) as pool:
            parts = pool.map(one_copy, [name] * CORES)
        wall = time.perf_counter() - t0
        res["cores_n"] = sum(w for w, _t in parts) / wall * scale
        res["seconds_n"] = round(wall, 2)
    out[name] = res
print(json.dumps({{"cores": CORES, "numpy": np.__version__, "results": out}}))
"""


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def _oracle_sample(seconds, cores=1, only=None, timeout=900):
    """Runs the oracle samples in a child interpreter: {"cores", "numpy",
    "results": {config: {"unit", "cores_1", "cores_n", ...}}}, or None and
    the error text.  only="decode" runs just the decode-linear sample."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = _ORACLE_SAMPLE.format(root=ROOT, mats=LLAMA, seconds=seconds, cores=cores, only=only)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=timeout)
    if r.returncode != 0:
        return None, r.stderr[-300:]
    return json.loads(r.stdout.strip().splitlines()[-1]), ""


def cpu_baseline(seconds=6.0):
    """The oracle on the host cores, per configuration: the decode-linear
    sample (the headline metric: the 4 Llama matrices cut to 2048 output
    rows, at M = 1, 8, 32), the single GEMV (M=1, K=1024, N=3072), a prefill
    slice (M=512, K=4096, 256 output rows), and one token of the Qwen3- and
    DeepSeek-V3-shaped MoE layers; each repeated for about `seconds` on one
    core, then as one copy per host core at once."""
    cores = host_cores()
    d, err = _oracle_sample(seconds, cores)
    if d is None:
        return {"value": None, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": "failed: " + err}
    res = {k: {kk: (round(v, 6) if isinstance(v, float) else v) for kk, v in r.items()} for k, r in d["results"].items()}
    dec = res["decode"]
    value = dec.get("cores_n", dec["cores_1"])
    return {"value": round(value, 4), "unit": "GB/s", "cores": d["cores"], "kind": "oracle",
            "sample": f"float64 numpy oracle, BLAS 1 thread per process; value: the decode-linear sample (the 4 "
                      f"Llama matrices cut to 2048 output rows, M = 1, 8, 32) as {d['cores']} concurrent copies "
                      f"for about {seconds:.0f} s; per_config: 1 core and all {d['cores']} cores",
            "numpy": d["numpy"], "per_config": res}


def run_reference(args):
    """The CPU oracle as the reference arm: each step is the bounded sample;
    value = its int4g weight bytes / its oracle time over the timed steps."""
    vals, secs = [], 0.0
    for i in range(args.warmup + args.steps):
        d, err = _oracle_sample(1.0, 1, only="decode")
        if d is None:
            last = err.strip().splitlines()[-1] if err.strip() else "no error text"
            return {"impl": "reference", "unavailable": "the CPU oracle sample failed: " + last}
        if i >= args.warmup:
            r = d["results"]["decode"]
            vals.append(r["cores_1"])
            secs += r["seconds_1"]
    value = round(sum(vals) / len(vals), 4)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs * 1e3 / args.steps, 1),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "per step: dequantized linear at M=1,8,32 on 2048 output rows of each Llama "
                                   "matrix, repeated to about 1 s of oracle time, one core"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_case(args):
    """One shape on its own (profiling): --case linear --M --K --N, or --case
    mlp --M (the Llama-7B MLP block).  Enough weight copies to exceed 2x L2
    are launched back to back in one CUDA graph; reports the mean time per
    launch."""
    import numpy as np
    import torch

    import int4_group_quantized_int4g_gb300 as fl
    from int4_group_quantized_int4g_gb300 import _build, inputs

    _build.build()
    fl.lib()
    dev = torch.device("cuda:0")
    if args.case == "mlp":
        print(json.dumps({"case": f"mlp M={args.M}", **run_mlp_section(torch, np, fl, inputs, dev, peaks(),
                                                                        Ms=(args.M,))}))
        return
    if args.case == "moe":
        cfg = dict(QWEN if args.model == "qwen3" else DSV3, Ms=(args.M,))
        print(json.dumps({"case": f"moe {cfg['name']} M={args.M}",
                          **run_moe_section(torch, np, fl, inputs, dev, peaks(), reps=args.iters, cfgs=(cfg,))}))
        return
    M, K, N = args.M, args.K, args.N
    nb = BYTES_PER_WEIGHT * N * K
    copies = max(1, min(64, int(np.ceil(300e6 / nb))))
    ws_list = []
    for i in range(copies):
        W = inputs.device_normal((N, K), 1, i, K, N, device=dev)
        q, s, z = fl.fl_int4g_quantize(W)
        del W
        ws_list.append(fl.fl_int4g_repack(q, s, z, N, K))
        del q, s, z
    x = torch.from_numpy(inputs.activations(M, K).view(np.int16)).to(dev).view(torch.bfloat16)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(fl.fl_int4g_linear_workspace(M, N, K), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        fl.fl_int4g_linear(x, ws_list[0], N, y=y, ws=ws)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for w in ws_list:
                fl.fl_int4g_linear(x, w, N, y=y, ws=ws)
        times = []
        for _ in range(args.iters):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            stream.synchronize()
            times.append(e0.elapsed_time(e1) / copies)
    assert fl.fl_int4g_status(ws) == 0
    t = statistics.median(times)
    print(json.dumps({"case": f"linear M={M} K={K} N={N}", "copies": copies, "median_ms_per_launch": round(t, 5),
                      "weight_GBps": round(nb / (t * 1e-3) / 1e9, 1), "iters": args.iters}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # defaults: ~0.7 s of timed decode steps, long enough to sample SM clocks
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sections", action="store_true", help="skip the MoE and prefill GEMM sections")
    ap.add_argument("--case", choices=["linear", "mlp", "moe"], help="time one shape on its own (profiling)")
    ap.add_argument("--model", choices=["qwen3", "deepseek"], default="qwen3", help="--case moe: the layer shape")
    ap.add_argument("--M", type=int, default=1)
    ap.add_argument("--K", type=int, default=4096)
    ap.add_argument("--N", type=int, default=12288)
    ap.add_argument("--iters", type=int, default=5)
    args = ap.parse_args()
    if args.case:
        run_case(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)))
        return
    if world > 1:
        out = run_replicas(args, rank, world)
        if rank == 0:
            print(json.dumps(out))
        return
    print(json.dumps(run_gpu(args)))


def aggregate_replicas(out, world, max_over_ranks):
    """Job-wide line of `world` independent replicas from one rank's line:
    the step time is the maximum over ranks, value = the weight bytes all
    ranks streamed per step / that time, and the end-to-end figure likewise
    (world x the slowest rank's).  max_over_ranks(v) returns the maximum of v
    over the ranks (a collective: every rank calls it, in the same order)."""
    ms = max_over_ranks(out["ms_per_step"])
    agg = dict(out)
    agg["config"] = dict(out["config"])
    agg["n_gpus"] = world
    agg["ms_per_step"] = round(ms, 4)
    agg["value"] = round(out["config"]["weight_bytes_per_step"] * world / (ms * 1e-3) / 1e9, 1)
    agg["config"]["parallelism"] = f"replicas{world}"
    if isinstance(out.get("e2e"), dict) and out["e2e"].get("value") is not None:
        slowest = -max_over_ranks(-out["e2e"]["value"])
        agg["e2e"] = dict(out["e2e"])
        agg["e2e"]["value"] = round(world * slowest, 1)
        if out["e2e"].get("serial_value") is not None:
            agg["e2e"]["serial_value"] = round(world * -max_over_ranks(-out["e2e"]["serial_value"]), 1)
    return agg


def run_replicas(args, rank, world):
    """N independent replicas (the path needs no exchange): each rank runs the
    same step on its own GPU, starting and stopping its timed region at a
    barrier; value = sum over ranks, time = max over ranks."""
    import torch
    import torch.distributed as dist
    local = int(os.environ.get("LOCAL_RANK", rank))
    torch.cuda.set_device(local)
    dist.init_process_group("nccl")
    args.no_cpu_baseline = args.no_cpu_baseline or rank != 0
    dist.barrier()
    out = run_gpu(args, barrier=dist.barrier)

    def max_over_ranks(v):
        t = torch.tensor([float(v)], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    agg = aggregate_replicas(out, world, max_over_ranks)
    dist.destroy_process_group()
    return agg


if __name__ == "__main__":
    main()

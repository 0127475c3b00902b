"""Benchmark of the BitNet b1.58 BitLinear hot path on B300.

Default workload (one "step"): a batch-1 decode step over 2B-class layer
shapes, 30 layers with distinct weight sets (521 MB of packed ternary weights,
4x the 126 MB L2, so every step streams its weights from HBM).  Per layer,
four dependent BitLinear phases with the data flow of a decoder layer:
  QKV   : the layer input (bf16) -> Q (bf16), K, V (binary32);
  O     : subln(Q) -> O (bf16)   (Q stands in for the attention output,
          which is not BitLinear);
  up/gate: subln(O) -> h = relu(gate)^2 * up (binary32);
  down  : h -> the next layer's input (bf16).
Every phase quantises its input per token to int8.  The step is one
bitnet_decode_chain_run (one persistent kernel; each phase reads the previous
phase's output as it is produced), captured once in a CUDA graph and replayed.

Metric: GB/s of algorithmic bytes (packed weights + scales + norm gains +
activations read and written in their stated precision) per second; the
roofline block reports the dominant kernel (the chain) against the measured
HBM copy bandwidth.  `--impl reference` times the CPU oracle on a bounded
sample of the same workload instead.  Under torchrun every rank runs an
independent replica (the path needs no exchange between GPUs) and rank 0
prints one JSON line.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

EPS = 1e-5
# Model dimensions: (hidden, FFN, K/V width, layers).  2B: the BitNet b1.58
# 2B4T shapes the pages describe; 8B: the Llama3-8B-1.58 model the pages list
# (hidden 4096, FFN 14336, 8 K/V heads of 128 -- the reading of that
# architecture's dimensions).
DIMS_2B = (2560, 6912, 640, 30)
DIMS_8B = (4096, 14336, 1024, 32)
HIDDEN, FFN = DIMS_2B[0], DIMS_2B[1]


def layer_shapes(dims=DIMS_2B):
    """(name, N, K, phase) of one decoder layer's BitLinear products."""
    H, F, KV = dims[0], dims[1], dims[2]
    return [("q", H, H, "qkv"), ("k", KV, H, "qkv"), ("v", KV, H, "qkv"), ("o", H, H, "o"),
            ("up", F, H, "ffn"), ("gate", F, H, "ffn"), ("down", H, F, "down")]


LAYER_SHAPES = layer_shapes(DIMS_2B)
METRIC = "BitLinear decode GB/s & % HBM roofline; prefill int8 TOPS & % tensor peak"
WORKLOAD = ("decode step, batch 1, 2B-class shapes (hidden 2560, FFN 6912), 30 layers of "
            "distinct ternary weights, dependent phases QKV -> subln O -> subln up/gate "
            "ReLU^2 -> down")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--layers", type=int, default=30)
    ap.add_argument("--impl", default="b300", choices=["b300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--case", default=None,
                    choices=["prefill", "gemv100b", "fused_small_m", "ffn", "gemv2560", "8b",
                             "lut"],
                    help="run only this secondary measurement and print it (for profiling "
                         "one kernel under ncu)")
    return ap.parse_args()


def layer_bytes(dims=DIMS_2B):
    """Algorithmic bytes of one layer: packed weights and their scales, the
    two norm gains, each phase's input read once in its precision (QKV, O,
    up/gate: bf16 [hidden]; down: binary32 h [FFN]) and every output written
    once (Q, O, down: bf16; K, V, h: binary32)."""
    H, F, KV = dims[0], dims[1], dims[2]
    w = sum(N * K // 4 + 4 for _, N, K, _ in layer_shapes(dims))
    gains = 2 * 4 * H
    inputs = 3 * 2 * H + 4 * F
    outputs = 2 * H + 2 * 4 * KV + 2 * H + 4 * F + 2 * H
    return w + gains + inputs + outputs


def weight_bytes(dims=DIMS_2B):
    return sum(N * K // 4 for _, N, K, _ in layer_shapes(dims))


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------- GPU arm
class DecodeStep:
    """Resident weights, norm gains, activations and the chain of the decode
    step.  weights: optional per-layer {name: (Wq, w_scale)} device tensors
    (default: synthetic N(0, 0.02) weights quantised on the GPU); x0: the
    step input (bf16 [1, HIDDEN]); gains: optional (attention-side, FFN-side)
    lists of binary32 [HIDDEN] gains per layer."""

    def __init__(self, layers, weights=None, x0=None, gains=None, seed=0, dims=DIMS_2B):
        import torch
        import bitlinear_bitnet_linear_03_b300 as bn
        from bitlinear_bitnet_linear_03_b300 import synth
        self.torch, self.bn = torch, bn
        dev = torch.device("cuda")
        self.layers = layers
        self.dims = dims
        H, F, KV = dims[0], dims[1], dims[2]
        if weights is None:
            ws_q = torch.empty(bn.bitnet_quantize_weights_workspace(F, H) * 2,
                               dtype=torch.uint8, device=dev)
            weights = []
            for li in range(layers):
                L = {}
                for j, (name, N, K, _) in enumerate(layer_shapes(dims)):
                    W = synth.weights_f32(N, K, seed=seed * 100000 + li * 16 + j, device="cuda")
                    L[name] = bn.bitnet_quantize_weights(W, ws=ws_q)
                    del W
                weights.append(L)
        self.W = weights
        if gains is None:
            gains = ([torch.from_numpy(synth.gain_random(H, 300 + li)).to(dev)
                      for li in range(layers)],
                     [torch.from_numpy(synth.gain_random(H, 600 + li)).to(dev)
                      for li in range(layers)])
        self.g_attn, self.g_ffn = gains
        if x0 is None:
            x0 = synth.tokens_bf16(1, H, seed=seed * 100000 + 77, device="cuda")
        self.x0 = x0.contiguous()
        bf, f32 = torch.bfloat16, torch.float32
        self.out = []
        # every layer's K and V outputs are views of one block, so that the
        # step's results leave the device in two copies, not one per array
        self.kv = torch.empty((layers, 2, 1, KV), dtype=f32, device=dev)
        for li in range(layers):
            self.out.append(dict(q=torch.empty((1, H), dtype=bf, device=dev),
                                 k=self.kv[li, 0],
                                 v=self.kv[li, 1],
                                 o=torch.empty((1, H), dtype=bf, device=dev),
                                 h=torch.empty((1, F), dtype=f32, device=dev),
                                 y=torch.empty((1, H), dtype=bf, device=dev)))
        torch.cuda.synchronize()

    def phases(self):
        """The 4 phases per layer, as bitnet_decode_chain_build takes them."""
        ph = []
        for li in range(self.layers):
            W, o = self.W[li], self.out[li]
            x = self.x0 if li == 0 else self.out[li - 1]["y"]
            ph.append({"x": x, "targets": [(*W["q"], None, None, o["q"]), (*W["k"], o["k"]),
                                           (*W["v"], o["v"])]})
            ph.append({"x": o["q"], "norm_gain": self.g_attn[li], "norm_eps": EPS,
                       "targets": [(*W["o"], None, None, o["o"])]})
            ph.append({"x": o["o"], "norm_gain": self.g_ffn[li], "norm_eps": EPS, "gated": True,
                       "h": o["h"], "targets": [(*W["up"], None), (*W["gate"], None)]})
            ph.append({"x_f32": o["h"], "targets": [(*W["down"], None, None, o["y"])]})
        return ph

    def build_chain(self):
        self.chain = self.bn.bitnet_decode_chain_build(self.phases())

    def step(self):
        self.bn.bitnet_decode_chain_run(self.chain)

    def launches_per_step(self):
        return 1

    def layer_outputs(self, li):
        return self.out[li]

    def input_tensors(self):
        return [self.x0]

    def output_tensors(self):
        return [t for o in self.out for t in o.values()]

    def result_tensors(self):
        """What a decode step hands back: the last layer's output and every
        layer's K and V (the cache entries of this token, one block)."""
        return [self.out[-1]["y"], self.kv]


def capture(torch, fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm the library (first-call set-up) outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_graph(torch, g, steps, warmup, barrier):
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3


def read_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return None


def profiled_traffic(kernel_file, profile_file):
    """Per-launch DRAM bytes from a committed ncu summary, or None when the
    kernel source changed since the capture (the summary records its hash)."""
    try:
        src = open(os.path.join(ROOT, kernel_file), "rb").read()
        text = open(os.path.join(ROOT, profile_file)).read()
    except OSError:
        return None
    digest = hashlib.sha256(src).hexdigest()[:16]
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith(("source_sha256_16", "dram_bytes_per_launch")):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha256_16") != digest:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def _time_calls(torch, fn, reps, warm=3, graph=False):
    """Seconds per call of fn(i), CUDA events after warm-up.  With graph=True
    the reps calls are captured once in a CUDA graph (short calls: keeps the
    host's launch cost out of the device time)."""
    for i in range(warm):
        fn(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if graph:
        g = capture(torch, lambda: [fn(i) for i in range(reps)])
        g.replay()
        torch.cuda.synchronize()
        e0.record()
        g.replay()
        e1.record()
    else:
        e0.record()
        for i in range(reps):
            fn(i)
        e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3 / reps


def _weight_sets(torch, bn, synth, N, K, count, seed):
    sets = []
    for r in range(count):
        W = synth.weights_f32(N, K, seed=seed + r, device="cuda")
        sets.append(bn.bitnet_quantize_weights(W))
        del W
    return sets


def _cpu_rate(fn, units, budget_s, threads):
    """Units per second of fn(threads) over about budget_s (at least once)."""
    fn(threads)
    n, t0 = 0, time.perf_counter()
    while n == 0 or time.perf_counter() - t0 < budget_s:
        fn(threads)
        n += 1
    return units * n / (time.perf_counter() - t0)


def oracle_secondary_baselines(budget_s=1.5):
    """The CPU oracle on bounded samples of the secondary workloads (weights as
    ternary codes drawn directly: the oracle's time does not depend on their
    values), on all host cores and, for the decode shapes, on one."""
    import oracle
    from bitlinear_bitnet_linear_03_b300 import synth
    allc = oracle.default_threads()
    out = {}

    def linear_case(key, N, K, M, rows, unit, single=True):
        q = synth.ternary_codes(rows, K, seed=17)
        Wq, ws = oracle.pack(q), synth.weight_scale(17)
        qx, sx = oracle.quantize_act_bf16(synth.tokens_bf16(M, K, seed=18, outlier_frac=0.01))
        run = lambda th: oracle.linear(Wq, ws, qx, sx, K, threads=th)
        if unit == "GB/s":
            units = rows * K / 4 + M * K + 4 * M * rows
        else:
            units = 2.0 * M * rows * K / 1e3  # TOPS after the 1e9 below
        rec = {"value": round(_cpu_rate(run, units, budget_s, allc) / 1e9, 5), "unit": unit,
               "cores": allc, "kind": "oracle",
               "sample": f"{rows} of the {N} output rows, M = {M}" + (
                   " (rate of the slice; the full shape scales with rows)" if rows < N else "")}
        if single:
            rec["single_thread"] = round(_cpu_rate(run, units, budget_s, 1) / 1e9, 5)
        out[key] = rec

    linear_case("gemv_2560x2560_M1", 2560, 2560, 1, 2560, "GB/s")
    linear_case("100b_M1_K8192_N28672", 28672, 8192, 1, 2048, "GB/s")
    linear_case("100b_M4_K8192_N28672", 28672, 8192, 4, 2048, "GB/s")
    linear_case("prefill_M4096_K2560_N6912", 6912, 2560, 256, 6912, "TFLOP/s", single=False)
    out["prefill_M4096_K2560_N6912"]["sample"] = ("256 of the 4096 tokens, all 6912 rows (rate of "
                                                 "the slice)")
    H, F = HIDDEN, FFN
    ws = [(oracle.pack(synth.ternary_codes(n, k, seed=30 + i)), synth.weight_scale(30 + i))
          for i, (n, k) in enumerate([(F, H), (F, H), (H, F)])]
    g = synth.gain_random(H, 3)
    for M, key, unit in ((1, "ffn_seq1", "GB/s"), (64, "ffn_seq4096", "TFLOP/s")):
        x = synth.tokens_bf16(M, H, seed=31)
        run = lambda th, x=x: oracle.ffn(x, g, EPS, ws[0][0], ws[0][1], ws[1][0], ws[1][1],
                                         ws[2][0], ws[2][1], threads=th)
        units = (3 * H * F / 4 + 2 * H + 4 * H) if unit == "GB/s" else 2.0 * M * 3 * H * F / 1e3
        rec = {"value": round(_cpu_rate(run, units, budget_s, allc) / 1e9, 5), "unit": unit,
               "cores": allc, "kind": "oracle",
               "sample": "one token" if M == 1 else f"{M} of the 4096 tokens (rate of the slice)"}
        if M == 1:
            rec["single_thread"] = round(_cpu_rate(run, units, budget_s, 1) / 1e9, 5)
        out[key] = rec
    return out


def secondary_measurements(torch, bn, peaks, only=None, cpu=True):
    """The other workloads, each timed with CUDA events after warm-up, weights
    rotated over enough distinct sets that every timed call streams from HBM
    (more than the 126 MB L2 between reuses), inputs resident:
      * single GEMV 2560x2560, batch 1 (80 weight sets);
      * 100B-class shapes 8192->28672 and 28672->8192: M = 1 (and M = 4 at
        K = 8192) through bitnet_linear_bf16 (bf16 tokens with 1% outliers
        quantised in the launch, static weights), the rest (M = 4 at
        K = 28672, M = 8, 16, 32, 64) through bitnet_linear on int8 codes;
      * 2B-class shapes at M = 16 and 64 through bitnet_linear;
      * prefill M = 4096 on the 2B FFN shapes, binary32 and bf16 outputs
        (tensor-core roofline against the measured bf16 dense peak: sm_103a has
        no integer tensor-core MMA, so the exact integer products run as e4m3
        digit MMAs, whose tensor time equals bf16's);
      * the fused FFN (hidden 2560, FFN 6912) at seq 1 and seq 4096;
      * 8B-class shapes (hidden 4096, FFN 14336, K/V 1024): the 32-layer
        decode step as one chain, and prefill M = 4096;
    and, with cpu=True, the oracle on bounded samples of the same workloads."""
    from bitlinear_bitnet_linear_03_b300 import synth
    out = {}
    dev = torch.device("cuda")
    hbm = float(peaks["hbm_gbs"]) if peaks and peaks.get("hbm_gbs") else 6400.0
    tpk = float(peaks["bf16_tflops"]) if peaks and peaks.get("bf16_tflops") else 1800.0

    def hbm_roof(gbs):
        return {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(gbs / hbm, 4)}

    def tc_roof(tops):
        return {"bound": "tensor", "achieved": round(tops, 1), "peak": tpk, "unit": "TFLOP/s",
                "frac": round(tops / tpk, 4),
                "peak_source": "measured bf16 dense (no int8 tensor MMA on sm_103a)"}

    def want(case):
        return only is None or only == case

    # single GEMV 2560x2560, M = 1
    if want("gemv2560"):
        N = K = 2560
        sets = _weight_sets(torch, bn, synth, N, K, 80, 100)
        x = synth.tokens_bf16(1, K, seed=0, device="cuda")
        y = torch.empty((1, N), dtype=torch.float32, device=dev)
        t = _time_calls(torch, lambda i: bn.bitnet_linear_bf16(
            x, [(sets[i % 80][0], sets[i % 80][1], y)], weights_static=True), 400, graph=True)
        byts = N * K // 4 + 2 * K + 4 + 4 * N
        out["gemv_2560x2560_M1"] = {"us": round(t * 1e6, 2), "GBps": round(byts / t / 1e9, 1),
                                    "roofline": hbm_roof(byts / t / 1e9)}
        del sets

    # 100B-class shapes (each timed as a CUDA graph of calls)
    ms_100b = [m for m, c in ((1, "gemv100b"), (4, "gemv100b"), (8, "fused_small_m"),
                              (16, "fused_small_m"), (32, "fused_small_m"),
                              (64, "fused_small_m")) if want(c)]
    for (N, K) in ([(28672, 8192), (8192, 28672)] if ms_100b else []):
        sets = _weight_sets(torch, bn, synth, N, K, 3, 200)
        for M in ms_100b:
            x = synth.tokens_bf16(M, K, seed=1, outlier_frac=0.01, device="cuda")
            y = torch.empty((M, N), dtype=torch.float32, device=dev)
            if M == 1 or (M <= 4 and K <= 16384):  # bitnet_linear_bf16's K range
                call = lambda i: bn.bitnet_linear_bf16(x, [(sets[i % 3][0], sets[i % 3][1], y)],
                                                       weights_static=True)
                byts = N * K // 4 + 2 * M * K + 4 * M * N + 4 * M + 4
                entry = "bitnet_linear_bf16 (static weights)"
            else:
                entry = "bitnet_linear"
                xq, sx = bn.bitnet_quantize_act(x)
                ws = torch.empty(max(bn.bitnet_linear_workspace(M, N, K), 16), dtype=torch.uint8,
                                 device=dev)
                call = lambda i: bn.bitnet_linear(sets[i % 3][0], sets[i % 3][1], xq, sx, y=y, ws=ws)
                byts = N * K // 4 + M * K + 4 * M * N + 4 * M + 4
            t = _time_calls(torch, call, 12, graph=True)
            out[f"100b_M{M}_K{K}_N{N}"] = {
                "us": round(t * 1e6, 1), "GBps": round(byts / t / 1e9, 1),
                "tops": round(2 * M * N * K / t / 1e12, 2), "roofline": hbm_roof(byts / t / 1e9),
                "entry": entry}
        del sets

    # 2B-class shapes at small M (the tensor-core path: the e4m3 digit form
    # for 16 <= M <= 64), each timed as a graph of calls over weight sets
    # that exceed L2.
    for (N, K) in ([(2560, 2560), (6912, 2560), (2560, 6912)] if want("fused_small_m") else []):
        nset = min(80, max(3, int(3 * 126e6 / (N * K / 4)) + 1))
        sets = _weight_sets(torch, bn, synth, N, K, nset, 700)
        for M in (16, 64):
            xq, sx = bn.bitnet_quantize_act(synth.tokens_bf16(M, K, seed=701, outlier_frac=0.01,
                                                              device="cuda"))
            y = torch.empty((M, N), dtype=torch.float32, device=dev)
            ws = torch.empty(max(bn.bitnet_linear_workspace(M, N, K), 16), dtype=torch.uint8,
                             device=dev)
            t = _time_calls(torch, lambda i: bn.bitnet_linear(sets[i % nset][0], sets[i % nset][1],
                                                              xq, sx, y=y, ws=ws), 4 * nset,
                            graph=True)
            byts = N * K // 4 + M * K + 4 * M * N + 4 * M + 4
            out[f"2b_M{M}_K{K}_N{N}"] = {
                "us": round(t * 1e6, 1), "GBps": round(byts / t / 1e9, 1),
                "tops": round(2 * M * N * K / t / 1e12, 2), "roofline": hbm_roof(byts / t / 1e9),
                "entry": "bitnet_linear"}
        del sets

    # 100B-class layers through the decode chain: 16 independent phases per
    # launch (each its own bf16 input and output), cycling over 4 weight sets
    # (235 MB, so every phase streams its weights from HBM); the weight stream
    # runs on across phase boundaries instead of ramping up per launch.
    for (N, K, M) in ([(28672, 8192, 1), (8192, 28672, 1), (28672, 8192, 4)]
                      if want("gemv100b") else []):
        nset, nph = 4, 16
        sets = _weight_sets(torch, bn, synth, N, K, nset, 300)
        xs = [synth.tokens_bf16(M, K, seed=310 + i, outlier_frac=0.01, device="cuda")
              for i in range(nph)]
        ys = [torch.empty((M, N), dtype=torch.float32, device=dev) for _ in range(nph)]
        chain = bn.bitnet_decode_chain_build(
            [{"x": xs[i], "targets": [(sets[i % nset][0], sets[i % nset][1], ys[i])]}
             for i in range(nph)])
        g = capture(torch, lambda: bn.bitnet_decode_chain_run(chain))
        t = time_graph(torch, g, 20, 3, lambda: None) / 20 / nph
        byts = N * K // 4 + 2 * M * K + 4 * M * N + 4 + 4
        out[f"100b_chain_M{M}_K{K}_N{N}"] = {
            "us_per_layer": round(t * 1e6, 2), "GBps": round(byts / t / 1e9, 1),
            "roofline": hbm_roof(byts / t / 1e9),
            "entry": f"bitnet_decode_chain_run, {nph} independent phases per launch"}
        del chain, g, sets, xs, ys

    # Lookup-table ablation: one token, the table-lookup inner product, the
    # dp4a control on the same kernel skeleton, and the production decode path
    # (bitnet_linear, int8 input), each timed as a graph of calls over weight
    # sets that exceed L2.
    for (N, K) in ([(2560, 2560), (6912, 2560), (2560, 6912), (28672, 8192)]
                   if want("lut") else []):
        nset = max(2, int(math.ceil(3 * 126e6 / (N * K / 4))))
        sets = _weight_sets(torch, bn, synth, N, K, nset, 900)
        xq, sx = bn.bitnet_quantize_act(synth.tokens_bf16(1, K, seed=901, device="cuda"))
        y = torch.empty((1, N), dtype=torch.float32, device=dev)
        byts = N * K // 4 + K + 4 * N + 8
        rec = {}
        for name, call in (
                ("lut", lambda i: bn.bitnet_linear_lut(sets[i % nset][0], sets[i % nset][1], xq,
                                                       sx, variant=0, y=y)),
                ("dp4a_same_skeleton", lambda i: bn.bitnet_linear_lut(
                    sets[i % nset][0], sets[i % nset][1], xq, sx, variant=1, y=y)),
                ("production", lambda i: bn.bitnet_linear(sets[i % nset][0], sets[i % nset][1],
                                                          xq, sx, y=y))):
            t = _time_calls(torch, call, 4 * nset, graph=True)
            rec[name] = {"us": round(t * 1e6, 2), "GBps": round(byts / t / 1e9, 1),
                         "roofline": hbm_roof(byts / t / 1e9)}
        out[f"lut_ablation_M1_K{K}_N{N}"] = rec
        del sets

    # prefill (2B FFN shapes; binary32 output, and bf16 output for K = 2560)
    def prefill(N, K, key, sets_seed, out_bf16=False):
        M = 4096
        sets = _weight_sets(torch, bn, synth, N, K, 4, sets_seed)
        x = synth.tokens_bf16(M, K, seed=600, device="cuda")
        xq, sx = bn.bitnet_quantize_act(x)
        y = torch.empty((M, N), dtype=torch.bfloat16 if out_bf16 else torch.float32, device=dev)
        ws = torch.empty(max(bn.bitnet_linear_workspace(M, N, K), 16), dtype=torch.uint8,
                         device=dev)
        if out_bf16:
            call = lambda i: bn.bitnet_linear(sets[i % 4][0], sets[i % 4][1], xq, sx, y=None,
                                              y_bf16=y, ws=ws)
        else:
            call = lambda i: bn.bitnet_linear(sets[i % 4][0], sets[i % 4][1], xq, sx, y=y, ws=ws)
        t = _time_calls(torch, call, 20)
        tops = 2 * M * N * K / t / 1e12
        out[key] = {"ms": round(t * 1e3, 4), "tops": round(tops, 1), "roofline": tc_roof(tops)}

    if want("prefill"):
        prefill(6912, 2560, "prefill_M4096_K2560_N6912", 500)
        prefill(2560, 6912, "prefill_M4096_K6912_N2560", 510)
        prefill(6912, 2560, "prefill_M4096_K2560_N6912_bf16out", 520, out_bf16=True)

    # fused FFN
    H, F = HIDDEN, FFN
    for M, nsets, reps in ([(1, 10, 200), (4096, 2, 6)] if want("ffn") else []):
        ffn_sets = []
        for r in range(nsets):
            ffn_sets.append([bn.bitnet_quantize_weights(synth.weights_f32(n_, k_, seed=700 + 3 * r + j,
                                                                           device="cuda"))
                             for j, (n_, k_) in enumerate([(F, H), (F, H), (H, F)])])
        x = synth.tokens_bf16(M, H, seed=0, device="cuda")
        g = torch.ones(H, dtype=torch.float32, device=dev)
        y = torch.empty((M, H), dtype=torch.float32, device=dev)
        ws = torch.empty(bn.bitnet_ffn_workspace(M, H, F), dtype=torch.uint8, device=dev)

        def ffn_call(i):
            (wu, su), (wg, sg), (wd, sd) = ffn_sets[i % nsets]
            bn.bitnet_ffn(x, g, 1e-5, wu, su, wg, sg, wd, sd, y=y, ws=ws)
        t = _time_calls(torch, ffn_call, reps, graph=(M == 1))
        packed = 3 * H * F // 4
        key = f"ffn_seq{M}"
        if M == 1:
            byts = packed + 2 * H + 4 * H + 3 * 4
            out[key] = {"us": round(t * 1e6, 2), "GBps": round(byts / t / 1e9, 1),
                        "roofline": hbm_roof(byts / t / 1e9)}
        else:
            tops = 2 * M * 3 * H * F / t / 1e12
            out[key] = {"ms": round(t * 1e3, 3), "tops": round(tops, 1), "roofline": tc_roof(tops)}
        del ffn_sets, ws, y

    # 8B-class shapes
    if want("8b"):
        step = DecodeStep(DIMS_8B[3], dims=DIMS_8B)
        step.build_chain()
        g8 = capture(torch, step.step)
        t = time_graph(torch, g8, 50, 5, lambda: None) / 50
        byts = layer_bytes(DIMS_8B) * DIMS_8B[3]
        out["decode_8b_32layers"] = {"us": round(t * 1e6, 1), "GBps": round(byts / t / 1e9, 1),
                                     "roofline": hbm_roof(byts / t / 1e9),
                                     "packed_weight_bytes": weight_bytes(DIMS_8B) * DIMS_8B[3]}
        del step, g8
        prefill(14336, 4096, "prefill_8b_M4096_K4096_N14336", 800)
        prefill(4096, 14336, "prefill_8b_M4096_K14336_N4096", 810)
    if cpu and only is None:
        for k, rec in oracle_secondary_baselines().items():
            if k in out:
                out[k]["cpu_baseline"] = rec
    return out


def run_gpu_arm(args, rank, world, barrier, max_over_ranks):
    import torch
    import bitlinear_bitnet_linear_03_b300 as bn
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    bn.lib()
    step = DecodeStep(args.layers)
    step.build_chain()
    graph = capture(torch, step.step)

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    dt = time_graph(torch, graph, args.steps, args.warmup, barrier)
    clk = clocks.stop()
    dt = max_over_ranks(dt)

    bytes_step = layer_bytes() * args.layers
    value = aggregate_rate(bytes_step, args.steps, world, dt) / 1e9

    # e2e: the step input copied in from pinned host memory and the step's
    # results (last layer output, every layer's K and V) copied out, every step.
    ins = step.input_tensors()
    outs = step.result_tensors()
    h_in = [t.cpu().pin_memory() for t in ins]
    h_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in ins)
    d2h = sum(t.numel() * t.element_size() for t in outs)

    def e2e_step():
        for d, h in zip(ins, h_in):
            d.copy_(h, non_blocking=True)
        graph.replay()
        for h, d in zip(h_out, outs):
            h.copy_(d, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    # (a short run is dominated by one-off costs of the first host copies:
    # warm up at least 20 steps and time at least 100)
    for _ in range(max(20, args.warmup)):
        e2e_step()
    e2e_steps = max(100, min(args.steps, 500))
    barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    t_e2e = max_over_ranks(time.perf_counter() - t0)
    e2e_value = aggregate_rate(bytes_step, e2e_steps, world, t_e2e) / 1e9

    # Dominant kernel: the chain is the step's only kernel; its average launch
    # duration is the graph replay time (CUDA events on the replaying stream).
    reps = max(20, min(args.steps, 400))
    t_lin = time_graph(torch, graph, reps, 5, lambda: None)
    per_launch_s = t_lin / reps
    achieved = bytes_step / per_launch_s / 1e9
    peaks = read_peaks()
    if peaks and peaks.get("hbm_gbs"):
        peak, peak_src = float(peaks["hbm_gbs"]), "measured"
    else:
        peak, peak_src = 6400.0, "fallback"
    traffic = profiled_traffic("bitlinear_bitnet_linear_03_b300/csrc/decode_chain.cu",
                               "profiles/decode_chain_2b_30layers.md")

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 x ternary (int32 acc; f32 / bf16 out)",
        "data": "synthetic: weights N(0,0.02) ternarized, activations bf16 N(0,1), seeded",
        "config": {"workload": WORKLOAD, "layers": args.layers, "batch_tokens": 1,
                   "packed_weight_bytes_per_step": weight_bytes() * args.layers,
                   "algorithmic_bytes_per_step": bytes_step,
                   "l2": "inputs larger than L2 (521 MB of weights per step vs 126 MB L2)",
                   "graph": "whole step captured in one CUDA graph",
                   "parallelism": f"replicas x{world}"},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": step.launches_per_step() * args.steps,
        "roofline": {"bound": "hbm", "kernel": "k_decode_chain (bitnet_decode_chain_run)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_src,
                     "traffic": traffic, "launch_us": round(per_launch_s * 1e6, 3),
                     "bytes_per_launch": bytes_step},
        "clocks": clk,
    }
    if not args.no_secondary:
        result["secondary"] = secondary_measurements(torch, bn, peaks)
    return result


# ----------------------------------------------------------------- oracle arm
class OracleSample:
    """One decode layer built on the host for the oracle (never touched by
    the GPU path): packed weights, norm gains, the layer input."""

    def __init__(self, seed=0, dims=DIMS_2B):
        import oracle
        from bitlinear_bitnet_linear_03_b300 import synth
        self.oracle = oracle
        self.dims = dims
        self.W = {}
        for j, (name, N, K, _) in enumerate(layer_shapes(dims)):
            Wq, s, _ = oracle.quantize_weights(synth.weights_f32(N, K, seed=7000 + j))
            self.W[name] = (Wq, s)
        self.x = synth.tokens_bf16(1, dims[0], seed=7100)
        self.g_attn = synth.gain_random(dims[0], 7200)
        self.g_ffn = synth.gain_random(dims[0], 7201)

    def phase_bytes(self):
        """Algorithmic bytes of the layer's four phases (their sum is
        layer_bytes): weights and scales, gain, input read, outputs written."""
        H, F, KV = self.dims[0], self.dims[1], self.dims[2]
        wb = {name: N * K // 4 + 4 for name, N, K, _ in layer_shapes(self.dims)}
        return [wb["q"] + wb["k"] + wb["v"] + 2 * H + 2 * H + 2 * 4 * KV,
                wb["o"] + 4 * H + 2 * H + 2 * H,
                wb["up"] + wb["gate"] + 4 * H + 2 * H + 4 * F,
                wb["down"] + 4 * F + 2 * H]

    def run_phase(self, k, threads):
        """Phase k of the layer (0 QKV, 1 subln O, 2 subln up/gate ReLU^2,
        3 down) on the previous phase's output; returns its bytes."""
        o, W = self.oracle, self.W
        H, F = self.dims[0], self.dims[1]
        if k == 0:
            q, s = o.quantize_act_bf16(self.x)
            self._Q = o.f32_to_bf16(o.linear(*W["q"], q, s, H, threads=threads)[0])
            o.linear(*W["k"], q, s, H, threads=threads)
            o.linear(*W["v"], q, s, H, threads=threads)
        elif k == 1:
            n, _ = o.rmsnorm_bf16(self._Q, self.g_attn, EPS)
            q, s = o.quantize_act_f32(n)
            self._O = o.f32_to_bf16(o.linear(*W["o"], q, s, H, threads=threads)[0])
        elif k == 2:
            n, _ = o.rmsnorm_bf16(self._O, self.g_ffn, EPS)
            q, s = o.quantize_act_f32(n)
            u = o.linear(*W["up"], q, s, H, threads=threads)[0]
            v = o.linear(*W["gate"], q, s, H, threads=threads)[0]
            self._h = o.relu2_mul(u, v)
        else:
            q, s = o.quantize_act_f32(self._h)
            o.f32_to_bf16(o.linear(*W["down"], q, s, F, threads=threads)[0])
        return self.phase_bytes()[k]

    def run(self, threads):
        """The layer's four phases, in order; returns its algorithmic bytes."""
        return sum(self.run_phase(k, threads) for k in range(4))


def _oracle_rate(sample, threads, budget_s):
    """GB/s of the oracle over whole decode layers for about budget_s."""
    sample.run(threads)  # warm-up
    nbytes, t0, layers = 0, time.perf_counter(), 0
    while time.perf_counter() - t0 < budget_s or layers == 0:
        nbytes += sample.run(threads)
        layers += 1
    dt = time.perf_counter() - t0
    return nbytes / dt / 1e9, layers, dt


def cpu_baseline(budget_s=12.0, single_budget_s=6.0):
    """The oracle on the host: all cores (the reported value) and one thread."""
    import oracle
    threads = oracle.default_threads()
    sample = OracleSample()
    value, layers, dt = _oracle_rate(sample, threads, budget_s)
    one, layers1, dt1 = _oracle_rate(sample, 1, single_budget_s)
    return {"value": round(value, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "single_thread": {"value": round(one, 4), "unit": "GB/s", "cores": 1,
                              "sample": f"{layers1} layers, {dt1:.1f} s"},
            "sample": f"{layers} repetitions of one decode layer (its 4 dependent phases, "
                      f"{layer_bytes()} algorithmic bytes each) of the 30-layer step, "
                      f"{dt:.1f} s"}


def run_reference_arm(args, rank):
    if rank != 0:
        return None
    import oracle
    threads = oracle.default_threads()
    sample = OracleSample()
    # A step is one whole decode layer while the run stays within about two
    # minutes, else one phase of the layer (cycling through the four).
    t0 = time.perf_counter()
    sample.run(threads)
    per_layer = time.perf_counter() - t0
    by_phase = per_layer * (args.steps + args.warmup) > 120.0
    step = ((lambda i: sample.run_phase(i % 4, threads)) if by_phase
            else (lambda i: sample.run(threads)))
    for i in range(args.warmup):
        step(i)
    nbytes, t0 = 0, time.perf_counter()
    for i in range(args.steps):
        nbytes += step(i)
    dt = time.perf_counter() - t0
    what = ("one phase of a decode layer, the four phases in turn (QKV, subln O, subln "
            "up/gate ReLU^2, down), each on the previous phase's output" if by_phase else
            "one decode layer of the step (its 4 dependent phases: QKV, subln O, subln "
            "up/gate ReLU^2, down)")
    value = nbytes / dt / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 x ternary (int32 acc; f32 / bf16 out)",
        "data": "synthetic: weights N(0,0.02) ternarized, activations bf16 N(0,1), seeded",
        "config": {"workload": WORKLOAD, "layers": args.layers, "batch_tokens": 1,
                   "parallelism": "replicas x1"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle",
                         "sample": "each step: " + what},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def rank_tools(torch, dist, device):
    """Barrier and max-over-ranks of the timed region: no-ops with one rank,
    else collectives of the process group (NCCL on GPUs; gloo in the CPU
    tests)."""
    def barrier():
        if dist is not None:
            dist.barrier()

    def max_over_ranks(v):
        if dist is None:
            return v
        t = torch.tensor([v], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return barrier, max_over_ranks


def aggregate_rate(units_per_step, steps, world, seconds):
    """Whole-job rate with replicas: every rank runs `steps` steps of
    `units_per_step`, and the job takes the slowest rank's time."""
    return units_per_step * steps * world / seconds


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        res = run_reference_arm(args, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    import torch
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")

    barrier, max_over_ranks = rank_tools(torch, dist, "cuda")

    if args.case is not None:
        import bitlinear_bitnet_linear_03_b300 as bn
        bn.lib()
        print(json.dumps(secondary_measurements(torch, bn, read_peaks(), only=args.case)),
              flush=True)
        return
    res = run_gpu_arm(args, rank, world, barrier, max_over_ranks)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline()
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

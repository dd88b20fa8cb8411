#!/usr/bin/env python3
"""Benchmark: Qwen3-8B-shaped layer prefill through the fused Q4_K GEMM.

One step = one pass of the hot path over one batch: the four Q4_K projections
of one Qwen3-8B-shaped layer (qkv K4096->N6144, o K4096->N4096, gate+up
K4096->N24576, down K12288->N4096) for M=105 prompt tokens, bf16 activations,
fp32 outputs.  Inputs are synthetic (seeded Q4_K blocks with d, dmin uniform in
[1e-3, 4e-3], N(0,1) bf16 activations).  Weights rotate over enough copies that
every step reads them from HBM (working set > 2x the 126 MB L2).

Each timed step replays CUDA graphs of the library calls (one graph for qkv and o,
one for gate+up, one for down, per weight copy), so the host's per-call launch
cost is not in the GPU timeline; CUDA events between the graphs time the
dominant kernel inside the timed region.  The end-to-end figure calls the API
eagerly with pinned host buffers and the copies in the timed region.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle
(fp64 dequant + naive GEMM) on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Fused Q4_K GEMM TFLOP/s (% bf16 TC peak); Qwen3-8B-shape layer prefill tok/s"
LAYER = (("qkv", 4096, 6144), ("o", 4096, 4096), ("gate_up", 4096, 24576), ("down", 12288, 4096))
M_TOKENS = 105
DOMINANT = "gate_up"
REF_BUDGET_S = 100.0  # reference arm: host seconds for warm-up + steps
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def layer_flops(M):
    return sum(2.0 * M * N * K for _, K, N in LAYER)


def layer_bytes(M):
    return sum(0.5625 * N * K + 2.0 * M * K + 4.0 * M * N for _, K, N in LAYER)


def kernel_source_files() -> list:
    """The sources the prefill kernel is compiled from: qwp_gemm.cu and the local
    headers it includes, followed transitively (paths relative to the repo)."""
    csrc = os.path.join(ROOT, "quantized_weight_prefill_gb300", "csrc")
    todo, seen = [os.path.join(csrc, "qwp_gemm.cu")], []
    while todo:
        path = os.path.normpath(todo.pop(0))
        if path in seen:
            continue
        seen.append(path)
        with open(path, "rb") as fh:
            for inc in re.findall(rb'#include "([^"]+)"', fh.read()):
                todo.append(os.path.join(os.path.dirname(path), inc.decode()))
    return [os.path.relpath(p, ROOT) for p in seen]


def strip_c_comments(text: str) -> str:
    """C/C++ source without its comments and with whitespace runs collapsed (string
    and character literals kept as they are)."""
    out = re.sub(r'"(?:\\.|[^"\\\n])*"|\'(?:\\.|[^\'\\\n])*\'|//[^\n]*|/\*.*?\*/',
                 lambda m: m.group(0) if m.group(0)[0] in "\"'" else " ", text, flags=re.S)
    return re.sub(r"\s+", " ", out).strip()


def kernel_source_hash() -> str:
    """Hash of kernel_source_files() with comments and layout ignored: a DRAM-traffic
    record stays valid while the code it was captured from is unchanged."""
    h = hashlib.sha256()
    for rel in kernel_source_files():
        with open(os.path.join(ROOT, rel), encoding="utf-8") as fh:
            h.update(rel.encode())
            h.update(strip_c_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = self.samples
        if self.window:
            inside = [r for r in rows if self.window[0] - 0.2 <= r[0] <= self.window[1] + 0.2]
            rows = inside or rows
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for _, p in rows if num(p[1]) is not None]
        smax = [num(p[2]) for _, p in rows if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, p in rows for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def dist_setup(n_gpus):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, local, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------- oracle leg

def layer_workload():
    return (f"Qwen3-8B-shape layer prefill: qkv K4096->N6144, o K4096->N4096, "
            f"gate+up K4096->N24576, down K12288->N4096; Q4_K weights, bf16 x, fp32 y")


def oracle_layer_sample(frac: float, seed: int = 7, min_rows: int = 1):
    """Inputs of one oracle step over all M_TOKENS tokens and the first
    max(min_rows, round(frac * N)) weight rows of every projection (at most N);
    returns the inputs and
    the fraction of the layer's weights they cover.  x is decoded to fp64 here,
    once: a step's time is then linear in the rows (every row is dequantized and
    multiplied once per step), so a row slice times its share of the layer."""
    import oracle
    import synth

    inputs, rows_k = [], 0
    for i, (_, K, N) in enumerate(LAYER):
        n = min(N, max(min_rows, int(round(frac * N))))
        blocks = synth.q4k_weights(N, K, seed=seed + i).reshape(N, -1)[:n]
        x = oracle.bf16_to_f64(synth.activations_bf16(M_TOKENS, K, seed=seed + 10 + i))
        inputs.append((blocks, x, n, K))
        rows_k += n * K
    return inputs, rows_k / sum(N * K for _, K, N in LAYER)


def oracle_layer_step(inputs):
    """One step of the CPU oracle (exact fp64 dequant of the rows + naive fp64 GEMM)."""
    import oracle

    for blocks, x, n, K in inputs:
        for n0 in range(0, n, 2048):
            n1 = min(n, n0 + 2048)
            oracle.gemm(x, oracle.q4k_dequant(blocks[n0:n1], n1 - n0, K), with_abs=False)


def oracle_layer_tokens_per_s(min_seconds: float):
    """The CPU oracle over the whole layer and all M_TOKENS tokens, repeated for at
    least `min_seconds`; returns (tok/s, seconds, steps, threads)."""
    import oracle

    inputs, _ = oracle_layer_sample(1.0)
    steps, t0 = 0, time.perf_counter()
    while True:
        oracle_layer_step(inputs)
        steps += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            return M_TOKENS * steps / dt, dt, steps, oracle.num_threads()


def run_reference(args):
    """The oracle as the reference arm: each step is the whole layer's M_TOKENS tokens
    over a row slice of every projection, sized (from a timed 1% slice) so that
    warm-up and steps together take about --ref-seconds on the host cores, but
    with at least two rows per oracle thread (at very many steps the run then
    takes longer); tok/s counts the slice's share of the layer."""
    import oracle

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    # The oracle parallelises over weight rows: a slice keeps at least two rows per
    # thread in every projection, so that it runs at the whole layer's rate.
    min_rows = 2 * oracle.num_threads()
    # calibrate: time a 1% slice, extrapolate to the whole layer
    probe, probe_share = oracle_layer_sample(0.01, min_rows=min_rows)
    oracle_layer_step(probe)
    c0 = time.perf_counter()
    oracle_layer_step(probe)
    full_step_s = (time.perf_counter() - c0) / probe_share
    frac = min(1.0, args.ref_seconds / (full_step_s * max(1, args.steps + args.warmup)))
    inputs, share = oracle_layer_sample(frac, min_rows=min_rows)
    for _ in range(args.warmup):
        oracle_layer_step(inputs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_layer_step(inputs)
    total = time.perf_counter() - t0
    value = M_TOKENS * share * args.steps / total
    threads = oracle.num_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": layer_workload(), "global_batch": M_TOKENS, "seq_len": M_TOKENS,
                   "parallelism": "none (host cores)"},
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": threads, "kind": "oracle",
                         "sample": f"per step all {M_TOKENS} tokens over {share:.4%} of the layer's weight rows "
                                   "(every weight dequantized exactly in fp64, then naive fp64 GEMM), "
                                   f"{args.steps} steps in {total:.1f} s"},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------------- single GEMMs

# Every GEMM shape of the workloads: Q4_K M=32 2048x2048; the Qwen3-8B-shaped
# layer at M = 105, 658, 2048; W4A16 (group 128) at M=2048; the stress sweep.
SWEEP = (["q4k:32:2048:2048"]
         + [f"q4k:{m}:{n}:{k}" for m in (105, 658, 2048) for _, k, n in LAYER]
         + ["w4a16:2048:12288:4096:128", "w4a16:2048:4096:12288:128",
            "w4a16:2048:12288:4096:128:sym", "w4a16:2048:12288:4096:128:bf16",
            "q6k:105:1024:4096", "q6k:105:4096:12288", "q6k:2048:4096:12288",
            "q4k:1:6144:4096", "q4k:1:4096:4096", "q4k:1:24576:4096", "q4k:1:4096:12288",
            "q4k:8:6144:4096", "q4k:8:4096:4096", "q4k:8:24576:4096", "q4k:8:4096:12288",
            "q6k:1:4096:12288", "w4a16:8:12288:4096:128:sym",
            "q4k:4096:32:4096", "q4k:8192:12288:4096"])


def parse_gemm(spec):
    parts = spec.split(":")
    kind = parts[0]
    if kind in ("q4k", "q6k", "q4kq8") and len(parts) == 4:
        M, N, K = map(int, parts[1:])
        return kind, M, N, K, 0, set()
    if kind == "q4kb" and len(parts) == 5:  # a strided batch: q4kb:B:M:N:K (B in the group slot)
        B, M, N, K = map(int, parts[1:])
        return kind, M, N, K, B, set()
    if kind == "w4a16" and len(parts) >= 5 and set(parts[5:]) <= {"sym", "bf16"}:
        M, N, K, g = map(int, parts[1:5])
        return kind, M, N, K, g, set(parts[5:])
    raise ValueError(f"bad --gemm spec {spec!r}: q4k:M:N:K, q6k:M:N:K, q4kq8:M:N:K, q4kb:B:M:N:K or "
                     "w4a16:M:N:K:group[:sym][:bf16]")


def time_gemm(spec, steps, warmup, dev):
    """Time one GEMM shape: graph replays of the library call (Q4_K, Q6_K: bf16 x;
    W4A16: fp16 x, or bf16 x with ':bf16', no zero points with ':sym'; q4kq8: the
    activation quantization of bf16 x and the Q4_K product with it; q4kb: a strided
    batch of B Q4_K products in one call, all counted), one call per
    input copy in the graph (weights and x both rotate; the copies together are
    larger than 2.5x L2, so every call streams its inputs from HBM), CUDA events on
    the launching stream around the timed replays.  Returns the JSON record."""
    import torch

    import quantized_weight_prefill_gb300 as qwp
    import synth

    stream = torch.cuda.current_stream(dev)
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2 ** 20)
    hbm, tc_burst, _, peak_kind = measured_peaks()
    kind, M, N, K, g, flags = parse_gemm(spec)
    nb = g if kind == "q4kb" else 1  # problems per call
    if kind in ("q4k", "q6k", "q4kq8", "q4kb"):
        wbytes = nb * N * K // 256 * (210 if kind == "q6k" else 144)
    else:
        wbytes = N * K // 2 + (N * K // g) * (2 if "sym" in flags else 3)
    xbytes = 2 * M * K * nb
    copies = max(2, min(64, int(np.ceil(2.5 * l2 / (wbytes + xbytes)))))
    ws, xs = [], []
    bf16_x = kind in ("q4k", "q6k", "q4kq8", "q4kb") or "bf16" in flags
    xqs = []
    for c in range(copies):
        if kind in ("q4k", "q4kq8"):
            blocks = synth.q4k_weights(N, K, seed=100 + c)
            ws.append((qwp.q4k_repack(torch.from_numpy(blocks.reshape(-1)).to(dev), N, K),))
        elif kind == "q4kb":
            ws.append((torch.cat([qwp.q4k_repack(torch.from_numpy(synth.q4k_weights(N, K, seed=100 + c * nb + p)
                                                                  .reshape(-1)).to(dev), N, K) for p in range(nb)]),))
        elif kind == "q6k":
            blocks = synth.q6k_weights(N, K, seed=100 + c)
            ws.append((qwp.q6k_repack(torch.from_numpy(blocks.reshape(-1)).to(dev), N, K),))
        else:
            wq, sc, z = synth.w4a16_weights(N, K, g, seed=100 + c)
            ws.append((qwp.w4a16_repack(torch.from_numpy(wq.view(np.int32)).to(dev)),
                       torch.from_numpy(sc).to(dev), None if "sym" in flags else torch.from_numpy(z).to(dev)))
        if kind == "q4kb":
            xs.append(torch.from_numpy(np.ascontiguousarray(np.stack([synth.activations_bf16(M, K, seed=7 + c * nb + p)
                                                                      for p in range(nb)])).view(np.int16))
                      .to(dev).view(torch.bfloat16))
        elif bf16_x:
            xs.append(torch.from_numpy(synth.activations_bf16(M, K, seed=7 + c).view(np.int16)).to(dev)
                      .view(torch.bfloat16))
        else:
            xs.append(torch.from_numpy(synth.activations_f16(M, K, seed=7 + c)).to(dev))
        if kind == "q4kq8":
            xqs.append(torch.empty(qwp.q8_activation_bytes(M, K), dtype=torch.uint8, device=dev))
    y = torch.empty(nb, M, N, dtype=torch.float32, device=dev) if kind == "q4kb" else \
        torch.empty(M, N, dtype=torch.float32, device=dev)

    def call(c):
        if kind == "q4k":
            qwp.q4k_gemm(ws[c][0], xs[c], N, out=y)
        elif kind == "q4kq8":
            qwp.q8_quantize(xs[c], out=xqs[c])
            qwp.q4k_q8_gemm(ws[c][0], xqs[c], M, N, K, out=y)
        elif kind == "q4kb":
            qwp.q4k_gemm_batched(ws[c][0], xs[c], N, out=y)
        elif kind == "q6k":
            qwp.q6k_gemm(ws[c][0], xs[c], N, out=y)
        else:
            gemm = qwp.w4a16_gemm_bf16 if "bf16" in flags else qwp.w4a16_gemm
            gemm(ws[c][0], ws[c][1], ws[c][2], xs[c], N, g, out=y)

    for s in range(warmup):
        call(s % copies)
    torch.cuda.synchronize()
    # One graph holds a call per input copy, back to back, so that the host's
    # graph-launch rate does not pace short GEMMs; it is replayed until at least
    # `steps` calls have run.
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        for c in range(copies):
            call(c)
    gr.replay()
    torch.cuda.synchronize()
    reps = max(1, -(-steps // copies))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        gr.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    if qwp.device_status() != 0:
        raise RuntimeError(f"kernel timeout in {spec}")
    t = e0.elapsed_time(e1) * 1e-3 / (reps * copies)
    flops = 2.0 * M * N * K * nb
    byts = wbytes + xbytes + 4.0 * M * N * nb
    t_tc, t_hbm = flops / (tc_burst * 1e12), byts / (hbm * 1e9)
    plan = ({"kernel": "decode (8-bit activations)"} if kind == "q4kq8"
            else {"kernel": "prefill (batch of %d)" % nb} if kind == "q4kb" else qwp.gemm_plan(kind, M, N, K))
    rec = {
        "gemm": spec, "us": t * 1e6, "tflops": flops / t / 1e12,
        "pct_bf16_peak": 100.0 * flops / t / 1e12 / tc_burst,
        "gbs": byts / t / 1e9, "bound": "tensor" if t_tc >= t_hbm else "hbm",
        "roofline_us": max(t_tc, t_hbm) * 1e6, "roofline_frac": max(t_tc, t_hbm) / t,
        "peak_source": peak_kind, "calls_timed": reps * copies, "input_copies": copies,
        "launches_per_call": 2 if kind in ("q4kq8", "q4kb") or (bf16_x and plan.get("kernel") == "prefill") else 1,
        "plan": plan,
    }
    del ws, xs, xqs, gr
    torch.cuda.empty_cache()
    return rec


def run_gemms(args, specs):
    """One JSON line per GEMM shape (see time_gemm)."""
    import torch

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    for spec in specs:
        print(json.dumps(time_gemm(spec, args.steps, args.warmup, dev)), flush=True)
    return 0


# The benchmark spec's targets, timed inside the default run: the M>=2048 tensor-core
# target on the largest projection, and the two HBM-bound targets (M<=32, skinny N).
TARGETS = (("gate_up_m2048", "q4k:2048:24576:4096", "tensor >= 0.60 of bf16 dense peak"),
           ("q4k_m32_n2048_k2048", "q4k:32:2048:2048", "HBM roofline >= 0.70"),
           ("q4k_m32_n2048_k2048_batch32", "q4kb:32:32:2048:2048",
            "HBM roofline >= 0.70 (32 independent products of that shape in one launch)"),
           ("skinny_n32_m4096_k4096", "q4k:4096:32:4096", "HBM roofline >= 0.70"),
           ("decode_m1_n152064_k4096", "q4k:1:152064:4096", "HBM roofline >= 0.70"),
           ("decode_q8_m1_n152064_k4096", "q4kq8:1:152064:4096", "HBM roofline >= 0.70 (8-bit activations)"))

# Load-time repacks timed on their own: the layer's four Q4_K projections and the
# two W4A16 shapes.
REPACKS = (("q4k", "qkv", 4096, 6144), ("q4k", "o", 4096, 4096), ("q4k", "gate_up", 4096, 24576),
           ("q4k", "down", 12288, 4096), ("w4a16", "w4a16_4096x12288", 4096, 12288),
           ("w4a16", "w4a16_12288x4096", 12288, 4096))


def time_repacks(dev, reps=20):
    """Each load-time repack alone: CUDA events around `reps` back-to-back repacks of
    one matrix (inputs of tens of MB: the first repack reads from HBM, later ones may
    partly hit L2; the figure is the mean).  Bytes = packed bytes read + written."""
    import torch

    import quantized_weight_prefill_gb300 as qwp
    import synth

    stream = torch.cuda.current_stream(dev)
    out = {}
    for fmt, name, K, N in REPACKS:
        if fmt == "q4k":
            src = torch.from_numpy(synth.q4k_weights(N, K, seed=300).reshape(-1)).to(dev)
            nbytes = src.numel()
            fn = lambda: qwp.q4k_repack(src, N, K)  # noqa: E731
        else:
            wq, _, _ = synth.w4a16_weights(N, K, 128, seed=300)
            src = torch.from_numpy(wq.view(np.int32)).to(dev)
            nbytes = src.numel() * 4
            fn = lambda: qwp.w4a16_repack(src)  # noqa: E731
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        out[name] = {"format": fmt, "N": N, "K": K, "bytes": nbytes, "ms": ms,
                     "gbs": 2.0 * nbytes / (ms * 1e-3) / 1e9}
        del src
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------------- GPU leg

def run_gpu(args):
    import torch

    import quantized_weight_prefill_gb300 as qwp
    import synth

    rank, local, world = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)

    M = M_TOKENS
    layer_w_bytes = sum(N * K // 256 * 144 for _, K, N in LAYER)
    copies = max(3, int(np.ceil(2.5 * l2 / layer_w_bytes)))
    weights = []  # [copy][proj] repacked Q4_K on the device
    for c in range(copies):
        per = []
        for i, (_, K, N) in enumerate(LAYER):
            blocks = synth.q4k_weights(N, K, seed=1000 * c + 10 * rank + i)
            g = torch.from_numpy(blocks.reshape(-1)).to(dev)
            per.append(qwp.q4k_repack(g, N, K))
            del g
        weights.append(per)
    xs = []
    for i, (_, K, N) in enumerate(LAYER):
        xb = synth.activations_bf16(M, K, seed=50 + 10 * rank + i)
        xs.append(torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16))
    ys = [torch.empty(M, N, dtype=torch.float32, device=dev) for _, _, N in LAYER]
    torch.cuda.synchronize()

    dom = [n for n, _, _ in LAYER].index(DOMINANT)
    dom_events = []

    def calls(c, which):
        w = weights[c]
        for i in which:
            _, K, N = LAYER[i]
            qwp.q4k_gemm(w[i], xs[i], N, out=ys[i])

    # warm up eagerly (library set-up happens outside any capture), then capture
    # one graph per weight copy holding the whole layer, and one graph holding
    # 4 x copies consecutive layers (the weight copies in turn), as a model's
    # layers run back to back.  The timed steps replay the multi-layer graph (each
    # replay is 4 x copies steps) and single-layer graphs for any remainder.  A
    # second set, with timing-event nodes around the dominant
    # GEMM, serves its per-launch time in a second timed pass: event nodes inside a
    # graph cost ~4 us each (they end the overlap of one launch with the next), so
    # they stay out of the steps that give the tok/s figure, and the per-launch time
    # they give is a slight overestimate.
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for s in range(args.warmup):
            calls(s % copies, range(len(LAYER)))
    stream.wait_stream(side)
    torch.cuda.synchronize()
    if qwp.device_status() != 0:
        raise RuntimeError("kernel timeout during warm-up")
    graphs, ev_graphs = [], []
    for c in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            calls(c, range(len(LAYER)))
        graphs.append(g)
        g = torch.cuda.CUDAGraph()
        e0 = torch.cuda.Event(enable_timing=True, external=True)
        e1 = torch.cuda.Event(enable_timing=True, external=True)
        with torch.cuda.graph(g):
            calls(c, range(dom))
            e0.record()
            calls(c, [dom])
            e1.record()
            calls(c, range(dom + 1, len(LAYER)))
        ev_graphs.append(g)
        dom_events.append((e0, e1))
    span_layers = 4 * copies  # layers per multi-layer graph (the end-to-end graph holds as many steps)
    multi = torch.cuda.CUDAGraph()
    with torch.cuda.graph(multi):
        for j in range(span_layers):
            calls(j % copies, range(len(LAYER)))
    for g in graphs + ev_graphs + [multi]:
        g.replay()
    torch.cuda.synchronize()

    def run_steps(n):
        # n steps: whole multi-layer replays, then single layers (weight copies keep
        # rotating in order either way)
        for _ in range(n // span_layers):
            multi.replay()
        for s in range(n % span_layers):
            graphs[s % copies].replay()

    run_steps(max(args.warmup, span_layers))
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    start.record(stream)
    run_steps(args.steps)
    end.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier(world)
    sampler.mark(wall0, wall1)
    ms_total = start.elapsed_time(end)
    ms_total = max_over_ranks(ms_total, world)
    if qwp.device_status() != 0:
        raise RuntimeError("kernel timeout during the timed region")
    # Second timed pass: the dominant GEMM's time per launch, from the event nodes of
    # the layer graphs (each replay re-records its copy's pair; read them per round).
    dom_samples = []
    for _ in range(max(1, min(25, args.steps // copies))):
        for g in ev_graphs:
            g.replay()
        torch.cuda.synchronize()
        dom_samples += [a.elapsed_time(b) for a, b in dom_events]
    if qwp.device_status() != 0:
        raise RuntimeError("kernel timeout during the per-launch timing pass")
    dom_ms = float(np.mean(dom_samples))

    # ---- end to end: host buffers, copies inside the timed region.  Steps run as
    # a serving loop would: every step copies its four x from pinned host memory
    # (side stream h2d_s, one copy: the four x sit back to back in one buffer), runs
    # the four library calls on the main stream once they have arrived, and copies
    # the four y back to pinned host memory (side stream d2h_s, one copy) once the
    # step's GEMMs are done.  Device x/y and host y are double-buffered, so step
    # s+1's copies and GEMMs overlap step s's read-back; a buffer is reused only
    # after the step two back has finished with it.  One CUDA graph holds E2E_SPAN
    # steps (every weight copy at least once).
    def packed(tensors, make):
        """One buffer holding the tensors' shapes back to back, and views of it."""
        total = sum(t.numel() for t in tensors)
        buf = make(total, tensors[0].dtype)
        views, off = [], 0
        for t in tensors:
            views.append(buf[off:off + t.numel()].view(t.shape))
            off += t.numel()
        return buf, views

    pinned = lambda n, dt: torch.empty(n, dtype=dt).pin_memory()  # noqa: E731
    on_dev = lambda n, dt: torch.empty(n, dtype=dt, device=dev)  # noqa: E731
    x_host_buf, x_host = packed(xs, pinned)
    for i, x in enumerate(xs):
        x_host[i].copy_(x.cpu())
    x_dev = [packed(xs, on_dev) for _ in range(2)]
    y_dev = [packed(ys, on_dev) for _ in range(2)]
    y_host = [packed(ys, pinned) for _ in range(2)]
    h2d = x_host_buf.numel() * x_host_buf.element_size()
    d2h = y_host[0][0].numel() * y_host[0][0].element_size()
    h2d_s = torch.cuda.Stream(dev)
    d2h_s = torch.cuda.Stream(dev)
    span = 4 * copies

    def e2e_graph():
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cap = torch.cuda.current_stream(dev)
            h2d_s.wait_stream(cap)
            d2h_s.wait_stream(cap)
            gemm_done, y_read = [], []
            for j in range(span):
                b, w = j % 2, weights[j % copies]
                with torch.cuda.stream(h2d_s):
                    if j >= 2:
                        h2d_s.wait_event(gemm_done[j - 2])  # x_dev[b] read by then
                    x_dev[b][0].copy_(x_host_buf, non_blocking=True)
                    x_in = torch.cuda.Event()
                    x_in.record(h2d_s)
                cap.wait_event(x_in)
                if j >= 2:
                    cap.wait_event(y_read[j - 2])  # y_dev[b] copied out by then
                for i, (_, K, N) in enumerate(LAYER):
                    qwp.q4k_gemm(w[i], x_dev[b][1][i], N, out=y_dev[b][1][i])
                done = torch.cuda.Event()
                done.record(cap)
                d2h_s.wait_event(done)
                with torch.cuda.stream(d2h_s):
                    y_host[b][0].copy_(y_dev[b][0], non_blocking=True)
                    read = torch.cuda.Event()
                    read.record(d2h_s)
                gemm_done.append(done)
                y_read.append(read)
            cap.wait_stream(h2d_s)
            cap.wait_stream(d2h_s)
        return g

    e2e_g = e2e_graph()
    e2e_g.replay()
    torch.cuda.synchronize()
    replays = max(1, min(args.steps, 2000) // span)
    e2e_steps = replays * span
    for _ in range(max(1, args.warmup // span)):
        e2e_g.replay()
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(replays):
        e2e_g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    if qwp.device_status() != 0:
        raise RuntimeError("kernel timeout during the end-to-end pass")
    # the last two steps' results reached the host: spot-check them against the device
    for b in range(2):
        if not torch.equal(y_host[b][0], y_dev[b][0].cpu()):
            raise RuntimeError("end-to-end copy of y does not match the device result")
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    sampler.stop()

    if rank != 0:
        return 0

    # The benchmark spec's target shapes and the load-time repacks, each timed on its own
    # after the layer (rank 0).
    targets = {}
    if not args.no_targets:
        for name, spec, goal in TARGETS:
            rec = time_gemm(spec, 200, args.warmup, dev)
            rec["target"] = goal
            targets[name] = rec
    repack = time_repacks(dev)

    hbm, tc_burst, tc_sust, peak_kind = measured_peaks()
    ms_step = ms_total / args.steps
    value = world * M * args.steps / (ms_total * 1e-3)
    tflops_layer = layer_flops(M) / (ms_step * 1e-3) / 1e12
    _, Kd, Nd = LAYER[dom]
    dom_flops = 2.0 * M * Nd * Kd
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    traffic = None
    if os.path.exists(TRAFFIC_FILE):
        with open(TRAFFIC_FILE) as f:
            tr = json.load(f)
        if tr.get("kernel_hash") == kernel_source_hash() and tr.get("workload") == f"M{M} N{Nd} K{Kd}":
            traffic = tr.get("bytes_per_launch")

    cpu = None
    if not args.no_cpu_baseline:
        tok_s, dt, nsteps, threads = oracle_layer_tokens_per_s(args.cpu_seconds)
        cpu = {"value": tok_s, "unit": "tok/s", "cores": threads, "kind": "oracle",
               "sample": f"{nsteps} whole-layer steps of all {M} tokens (every weight dequantized exactly "
                         f"in fp64, naive fp64 GEMM), {dt:.1f} s"}

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tok/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp16 operands (bf16 input), fp32 accumulate",
        "data": "synthetic",
        "config": {
            "workload": layer_workload(),
            "global_batch": M * world, "seq_len": M, "parallelism": f"replicas x{world}",
            "l2": f"weights rotate over {copies} copies ({copies * layer_w_bytes / 1e6:.0f} MB > 2x L2)",
            "launch": f"CUDA graphs of {4 * copies} consecutive layers (the four library calls each, the "
                      f"{copies} weight copies in turn), as a model's layers run back to back; each replay is "
                      f"{4 * copies} steps",
        },
        "layer_tflops": tflops_layer,
        "layer_pct_bf16_peak": 100.0 * tflops_layer / tc_burst,
        "layer_roofline_frac": (max(layer_flops(M) / (tc_burst * 1e12), layer_bytes(M) / (hbm * 1e9))
                                / (ms_step * 1e-3)),
        "roofline": {
            "kernel": f"qwp_gemm_kernel<Q4_K> {DOMINANT} M{M} N{Nd} K{Kd}",
            "bound": "tensor", "achieved": achieved, "peak": tc_burst, "unit": "TFLOP/s",
            "frac": achieved / tc_burst, "traffic": traffic,
            "peak_source": f"{peak_kind} bf16 dense (burst)",
            "hbm_gbs": (0.5625 * Nd * Kd + 2.0 * M * Kd + 4.0 * M * Nd) / (dom_ms * 1e-3) / 1e9,
            "ms_per_launch": dom_ms,
            "launch_timing": "CUDA events recorded inside the layer graphs around the dominant GEMM (conversion included), second timed pass after the steps",
        },
        "targets": targets,
        "repack": repack,
        "cpu_baseline": cpu,
        "e2e": {"value": world * M * e2e_steps / (e2e_ms * 1e-3), "unit": "tok/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "every step copies its four x from pinned host memory (one copy) and its four y back to "
                       "pinned host memory (one copy) around the four public API calls (copies on side streams, "
                       "double-buffered so a step's read-back overlaps the next step's GEMMs); "
                       f"{span} steps per CUDA graph replay"},
        # per call: the bf16 -> fp16 activation conversion and the GEMM
        "gpu_launches": 2 * len(LAYER) * args.steps,
        "clocks": sampler.summary(),
    }
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=REF_BUDGET_S,
                    help="reference arm: host seconds that warm-up and steps together aim at")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-targets", action="store_true", help="skip the per-GEMM target shapes after the layer")
    ap.add_argument("--gemm", action="append", default=[],
                    help="time single GEMMs instead of the layer: q4k:M:N:K, q6k:M:N:K or w4a16:M:N:K:group[:sym][:bf16]")
    ap.add_argument("--sweep", action="store_true", help="time every GEMM shape of the workloads")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.gemm or args.sweep:
        if args.steps == ap.get_default("steps"):
            args.steps = 200
        return run_gemms(args, args.gemm + (SWEEP if args.sweep else []))
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())

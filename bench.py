#!/usr/bin/env python3
"""Benchmark of the chunked GDN/KDA prefill hot path on GB300.

One step = one pass of the whole hot path over one packed batch that is already resident in
HBM: conv1d + SiLU (carried conv state) -> L2 over the q|k heads -> chunked gated delta rule,
all through the C ABI. Default workload: the largest one, KDA varlen, 64 streams with
log-uniform lengths in [16, 16384] summing to 262144 tokens, 32 heads, head dim 128, bf16
activations, fp32 states, with the conv1d + SiLU + L2 front end.

Prints ONE JSON line (rank 0). `--impl reference` times the fp64 CPU oracle instead (the
reference arm of this path), on bounded samples of the same workload.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
                       [--streams S]   (profiling slices: the first S streams of the workload)
Multi-GPU (replicas, weak scaling): torchrun --nproc-per-node N bench.py --gpus N ...
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from linear_attention_chunked_conv1d_gb300.inputs import (  # noqa: E402
    DECODE_WORKLOADS, PROJ_WORKLOADS, WORKLOADS, make_inputs)

DEFAULT_WORKLOAD = "kda_varlen_64_h32_d128"
METRIC = "prefill tokens/s per GDN/KDA layer"
DECODE_METRIC = "decode tokens/s per GDN/KDA layer"
PROJ_METRIC = "phase-1 projection tokens/s (QKVZ GEMM)"
ALL_WORKLOADS = {**WORKLOADS, **DECODE_WORKLOADS, **PROJ_WORKLOADS}
CHUNK = 64
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------------------ accounting
def act_bytes(wl) -> int:
    return 2 if wl.dtype == "bf16" else 4


def path_algorithmic(wl, lengths):
    """Algorithmic bytes and FLOPs of one pass of the (fused) path: x read once, gates, output,
    states read + written, conv weights. FLOPs per token and v-head: 2C dk (K K^T, Q K^T lower
    triangles) + C (dk + dv) (forward substitution) + C dv (P U') + 6 dk dv (w H, Q H, K^T U')."""
    s = act_bytes(wl)
    T = sum(lengths)
    d, K = wl.d, wl.conv_kernel
    gate = 4 * wl.Hv * (d if wl.variant == "kda" else 1)
    per_tok = wl.cd * s + gate + 4 * wl.Hv + wl.Hv * d * s
    per_stream = 2 * 4 * wl.Hv * d * d + 2 * s * (K - 1) * wl.cd
    B = per_tok * T + per_stream * len(lengths) + wl.cd * K * s
    F = T * wl.Hv * (2 * CHUNK * d + CHUNK * 2 * d + CHUNK * d + 6 * d * d)
    return B, F


def decode_algorithmic_bytes(wl):
    """Algorithmic bytes of one decode step (B streams, one token each): x row, gates, output,
    h state read + written, conv state read + written, per stream; conv weights once."""
    s = act_bytes(wl)
    d, K = wl.d, wl.conv_kernel
    gate = 4 * wl.Hv * (d if wl.variant == "kda" else 1)
    per_stream = (wl.cd * s + gate + 4 * wl.Hv + wl.Hv * d * s + 2 * 4 * wl.Hv * d * d
                  + 2 * s * (K - 1) * wl.cd)
    return per_stream * wl.B + wl.cd * K * s


def kernel_algorithmic_bytes(wl, lengths):
    """Algorithmic bytes per launch of each kernel of the (unfused) path."""
    s = act_bytes(wl)
    T, d, K = sum(lengths), wl.d, wl.conv_kernel
    B = len(lengths)
    conv = 2 * T * wl.cd * s + wl.cd * K * s + 2 * B * (K - 1) * wl.cd * s
    l2 = 2 * T * 2 * wl.Hk * d * s
    gate = 4 * wl.Hv * (d if wl.variant == "kda" else 1)
    rec = (T * (2 * wl.Hk * d * s + wl.Hv * d * s + gate + 4 * wl.Hv + wl.Hv * d * s)
           + 2 * B * wl.Hv * d * d * 4)
    return {"conv1d_silu": conv, "l2norm_heads": l2, "recurrence": rec}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_sha(name: str) -> str:
    src = os.path.join(ROOT, "linear_attention_chunked_conv1d_gb300", "csrc", name)
    with open(src, "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()[:12]


def profiled_traffic(kernel_file: str, workload: str, kind: str):
    """DRAM bytes (read + write) per launch from profiles/traffic.txt, only if the kernel source
    is unchanged since the counters were taken (lines: file workload sha12 bytes kind, kind
    'fused' for the one-launch layer kernel, 'split' for the recurrence of the two-launch path)."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    sha = kernel_source_sha(kernel_file)
    for line in open(p):
        parts = line.split()
        if (len(parts) == 5 and parts[0] == kernel_file and parts[1] == workload
                and parts[2] == sha and parts[4] == kind):
            return int(parts[3])
    return None


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        # let nvidia-smi finish starting up (it loads NVML and competes for the host cores)
        # before the timed steps begin; its samples continue through them
        t0 = time.time()
        while not self.lines and time.time() - t0 < 3.0 and self.proc.poll() is None:
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------ CPU oracle
def oracle_sample(wl, inputs_cpu_stream, threads):
    """The oracle (as it stands) over one stream: front end + recurrence, all heads."""
    import oracle
    x, conv_state, h, g, beta, L, conv_w = inputs_cpu_stream
    cu = np.array([0, L])
    q, k, v, _ = oracle.front_end(x, conv_w, conv_state[None], cu, Hk=wl.Hk,
                                  Hv=wl.Hv, dk=wl.d, dv=wl.d, eps=1e-6, act_dtype=wl.dtype)
    oracle.gated_delta(h[None], q, k, v, g, beta, cu.astype(np.int32),
                       scale=1.0 / math.sqrt(wl.d), per_channel=wl.variant == "kda",
                       threads=threads)


def stream_cpu(inp, s, conv_w):
    cu = np.concatenate([[0], np.cumsum(inp["lengths"])])
    a, b = int(cu[s]), int(cu[s + 1])
    f = lambda t: t.detach().to("cpu", torch.float64).numpy()  # noqa: E731
    return (f(inp["x"][a:b]), f(inp["conv_state"][s]), f(inp["h"][s]), f(inp["g"][a:b]),
            f(inp["beta"][a:b]), b - a, conv_w)


# Workloads whose oracle time is also reported on one host thread (the two small GDN ones).
SINGLE_THREAD_BASELINE = ("gdn_t100_h4_d64_f32", "gdn_batched_8x2048_h16_d128")


def _oracle_over_streams(wl, inp, conv_w, threads, budget_s):
    done_tokens, elapsed, streams = 0, 0.0, 0
    for s in range(wl.B):
        data = stream_cpu(inp, s, conv_w)
        t0 = time.perf_counter()
        oracle_sample(wl, data, threads)
        elapsed += time.perf_counter() - t0
        done_tokens += data[5]
        streams += 1
        if elapsed >= budget_s:
            break
    return done_tokens, elapsed, streams


def cpu_baseline(wl, inp, budget_s=12.0):
    """Time the oracle on whole streams of the workload until about budget_s of CPU work, on
    every host core; for the two small GDN workloads also on one thread."""
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    conv_w = inp["conv_w"].detach().to("cpu", torch.float64).numpy()
    done_tokens, elapsed, streams = _oracle_over_streams(wl, inp, conv_w, threads, budget_s)
    res = {"value": done_tokens / elapsed, "unit": "tokens/s", "cores": threads,
           "kind": "oracle",
           "sample": f"{streams} of {wl.B} streams ({done_tokens} tokens, all {wl.Hv} v-heads): "
                     f"fp64 conv1d+SiLU -> L2 -> token-by-token recurrence, {elapsed:.1f} s"}
    if wl.name in SINGLE_THREAD_BASELINE:
        t1, e1, s1 = _oracle_over_streams(wl, inp, conv_w, 1, budget_s / 2)
        res["single_thread"] = {
            "value": t1 / e1, "unit": "tokens/s", "cores": 1,
            "sample": f"{s1} of {wl.B} streams ({t1} tokens, all {wl.Hv} v-heads) on one "
                      f"host thread, {e1:.1f} s"}
    return res


def run_reference_proj(args, wl):
    """Reference arm of the projection workload: the oracle's fp64 product over a sample of the
    stacked rows (256 per step) against the full weight, timed on the host cores."""
    import oracle
    Kd, N = wl.hidden, 4 * wl.Hv * wl.d
    gen = torch.Generator("cpu")
    gen.manual_seed(0)
    rows = 256
    a = torch.randn(rows, Kd, generator=gen).to(torch.bfloat16)
    w = (torch.randn(N, Kd, generator=gen) / math.sqrt(Kd)).to(torch.bfloat16)
    af, wf = a.to(torch.float64).numpy(), w.to(torch.float64).numpy()
    for _ in range(args.warmup):
        oracle.linear(af, wf)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.linear(af, wf)
    total = time.perf_counter() - t0
    value = rows * args.steps / total
    threads = os.cpu_count() or 1
    line = {
        "impl": "reference", "metric": PROJ_METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; hidden rows ~N(0,1), weights ~N(0,1/hidden))",
        "config": {"workload": wl.name, "hidden": Kd, "outputs": N},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"each step: {rows} of the stacked rows against the full "
                                   f"{N} x {Kd} weight, fp64 matrix product"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference(args, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    if wl.mode == "proj":
        run_reference_proj(args, wl)
        return
    import oracle
    oracle.build()
    # each step: the oracle over one whole stream (all v-heads), cycling through the workload's
    # first two streams (drawn as in the whole workload; only those are generated on the host)
    sample_wl = stream_slice(wl, min(wl.B, 2)) if wl.mode == "prefill" and wl.B > 2 else wl
    inp = make_inputs(sample_wl, device="cpu", seed=0)
    conv_w = inp["conv_w"].to(torch.float64).numpy()
    threads = os.cpu_count() or 1
    data = [stream_cpu(inp, s, conv_w) for s in range(min(sample_wl.B, 2))]
    for i in range(args.warmup):
        oracle_sample(wl, data[i % len(data)], threads)
    times, toks = [], 0
    for i in range(args.steps):
        d = data[i % len(data)]
        t0 = time.perf_counter()
        oracle_sample(wl, d, threads)
        times.append(time.perf_counter() - t0)
        toks += d[5]
    total = sum(times)
    value = toks / total
    line = {
        "impl": "reference", "metric": DECODE_METRIC if wl.mode == "decode" else METRIC,
        "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; x~N(0,1), conv w~N(0,0.25), h~N(0,0.02), g=-softplus(N(0,1)), beta=sigmoid(N(0,1)))",
        "config": {"workload": wl.name, "streams": wl.B, "Hk": wl.Hk, "Hv": wl.Hv,
                   "head_dim": wl.d, "variant": wl.variant, "activations": wl.dtype},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"each step: one whole stream ({data[0][5]} tokens, all "
                                   f"{wl.Hv} v-heads) of the workload, fp64 front end + "
                                   "token-by-token recurrence"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------ replicas
def aggregate(tokens_local: int, ms_local: float, pg=None, device=None):
    """Whole-job throughput of weak-scaled replicas: every rank processes its own batch; the
    job takes as long as the slowest rank. Returns (tokens/s over all ranks, max ms, ranks)."""
    if pg is None:
        return tokens_local / (ms_local * 1e-3), ms_local, 1
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    n = torch.tensor([float(tokens_local)], dtype=torch.float64, device=device)
    pg.all_reduce(n, op=pg.ReduceOp.SUM)
    ms = float(t.item())
    return float(n.item()) / (ms * 1e-3), ms, pg.get_world_size()


def stream_slice(wl, n):
    """The workload restricted to its first n streams: lengths drawn as for the whole workload
    (same seed), the other inputs drawn afresh for these streams only (same distributions)."""
    from linear_attention_chunked_conv1d_gb300.inputs import draw_lengths
    gen = torch.Generator("cpu")
    gen.manual_seed(0)
    lengths = draw_lengths(wl, gen)[:n]
    return wl.replace(name=f"{wl.name}[streams 0..{n - 1}]", B=n,
                      lengths="list:" + ",".join(str(v) for v in lengths))


def uses_tensor_cores(wl) -> bool:
    return wl.dtype == "bf16" and wl.d == 128


# ------------------------------------------------------------------------------ GPU arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(ALL_WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--streams", type=int, default=0,
                    help="profiling slice: keep only the first S streams of the workload (their "
                         "lengths as drawn for the whole workload)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    wl = ALL_WORKLOADS[args.workload]
    if args.streams and wl.mode == "prefill" and args.streams < wl.B:
        wl = stream_slice(wl, args.streams)
    if args.impl == "reference":
        run_reference(args, wl)
        return

    import linear_attention_chunked_conv1d_gb300 as la
    from linear_attention_chunked_conv1d_gb300.path import PrefillPass

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    la._load()
    if wl.mode == "proj":
        run_proj(args, wl, dev, local, rank, world, pg)
        return
    inp = make_inputs(wl, device=dev, seed=rank)  # each replica its own batch (weak scaling)
    if wl.mode == "decode":
        run_decode(args, wl, inp, dev, local, rank, world, pg)
        return
    lengths = inp["lengths"]
    T = sum(lengths)
    p = PrefillPass(wl, inp)
    flush = torch.zeros(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)

    def flush_l2():
        """Evict L2 by reading a buffer twice its size: the lines it leaves are clean, so the
        timed step that follows pays no write-back for them."""
        torch.max(flush)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        p.run()
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    torch.cuda.synchronize()

    fused = p.can_fuse  # one launch (conv + L2 + recurrence) where the tensor-core path runs

    # a single stream with too few (stream, head) units to fill the GPU: the chunk-parallel scan
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    seg_s = min(8, max(1, (n_sm // wl.Hv + 1) // 2)) if (fused and wl.B == 1) else 1

    def timed_steps(mode):
        """Per-step CUDA events on the launching stream, L2 flushed before each step (outside
        the events). mode: "split" (front end, then the recurrence), "fused" (one launch),
        "seg" (front end, then the segmented recurrence)."""
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush_l2()
            ev[i][0].record(stream)
            if mode == "fused":
                p.fused()
            else:
                p.front_end()
            ev[i][1].record(stream)
            if mode == "split":
                p.recurrence()
            elif mode == "seg":
                p.recurrence_segmented(seg_s)
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        return ([e[0].elapsed_time(e[2]) for e in ev], [e[0].elapsed_time(e[1]) for e in ev],
                [e[1].elapsed_time(e[2]) for e in ev])

    # Every public path that applies (two launches; one fused launch; for a single stream the
    # segmented scan); the step is the fastest, decided on this run's own timings.
    clocks = ClockSampler(local)
    clocks.start()
    # every path is warmed up on its own before its timed steps (the warm-up above ran p.run(),
    # which is the fused launch where it applies: the split path's kernels would otherwise pay
    # their first-launch costs inside the timed region)
    for _ in range(args.warmup):
        p.front_end()
        p.recurrence()
    torch.cuda.synchronize()
    split_ms, front_ms, rec_ms = timed_steps("split")
    fused_ms = seg_ms = seg_rec_ms = None
    if fused:
        for _ in range(args.warmup):
            p.fused()
        torch.cuda.synchronize()
        fused_ms, _, _ = timed_steps("fused")
    if seg_s > 1:
        for _ in range(args.warmup):
            p.front_end()
            p.recurrence_segmented(seg_s)
        torch.cuda.synchronize()
        seg_ms, _, seg_rec_ms = timed_steps("seg")
    # The same steps replayed from a CUDA graph of the path's public calls: the kernels and
    # their arguments are those above, but the host launches (and the gaps between the kernels
    # of a multi-launch step) are paid once at capture. Paced launches remain the fallback.
    def graph_of(mode):
        def body():
            if mode == "fused":
                p.fused()
            else:
                p.front_end()
                if mode == "split":
                    p.recurrence()
                else:
                    p.recurrence_segmented(seg_s)
        try:
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                body()
            torch.cuda.synchronize()
            for _ in range(args.warmup):
                g.replay()
            torch.cuda.synchronize()
            return g
        except Exception:  # capture unsupported here: keep the paced timings
            torch.cuda.synchronize()
            return None

    def timed_graph(g):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush_l2()
            ev[i][0].record(stream)
            g.replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        return [e[0].elapsed_time(e[1]) for e in ev]

    paced = {"split": split_ms, "fused": fused_ms, "seg": seg_ms}
    graphed = {}
    for mode in [m for m in ("split", "fused", "seg") if paced[m]]:
        g = graph_of(mode)
        if g is not None:
            graphed[mode] = timed_graph(g)
            del g
    clk = clocks.stop()
    cands = {}
    for mode, ms_list in paced.items():
        if ms_list:
            cands[(mode, "paced")] = sum(ms_list)
    for mode, ms_list in graphed.items():
        cands[(mode, "graph")] = sum(ms_list)
    best, best_launch = min(cands, key=cands.get)
    use_fused = best == "fused"
    step_ms = (graphed if best_launch == "graph" else paced)[best]
    value, ms, _ = aggregate(T, sum(step_ms) / len(step_ms), pg, dev)

    # ---- end to end through the public API: pinned host inputs in, result out, every step
    x_h = inp["x"].cpu().pin_memory()
    g_h = inp["g"].cpu().pin_memory()
    b_h = inp["beta"].cpu().pin_memory()
    out_h = torch.empty(p.out.shape, dtype=p.out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (x_h, g_h, b_h))
    d2h = out_h.numel() * out_h.element_size()
    # pipelined: the copies of neighbouring steps overlap each step's compute (path.StreamedPrefill)
    from linear_attention_chunked_conv1d_gb300.path import StreamedPrefill
    sp = StreamedPrefill(wl, inp, mode=best, segments=seg_s, compute_stream=stream)
    for i in range(2 + 2):
        sp.step(i, x_h, g_h, b_h, out_h)
    sp.finish()
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    sp.start(e0)
    for i in range(args.steps):
        sp.step(i, x_h, g_h, b_h, out_h)
    sp.finish()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_value, e2e_ms, _ = aggregate(T, e0.elapsed_time(e1) / args.steps, pg, dev)

    if rank != 0:
        if pg:
            pg.barrier()
            pg.destroy_process_group()
        return

    peaks, peak_src = load_peaks()
    kb = kernel_algorithmic_bytes(wl, lengths)
    rec_avg = sum(rec_ms) / len(rec_ms)
    front_avg = sum(front_ms) / len(front_ms)
    step_avg = sum(step_ms) / len(step_ms)
    split_avg = sum(split_ms) / len(split_ms)
    fused_avg = sum(fused_ms) / len(fused_ms) if fused else None
    hbm = float(peaks["hbm_gbs"])
    B_alg, F_alg = path_algorithmic(wl, lengths)
    # dominant kernel: the fused layer kernel (its events also bracket the one-block stream
    # order kernel launched before it), else the recurrence of the two-launch path
    seg_rec_avg = sum(seg_rec_ms) / len(seg_rec_ms) if seg_rec_ms else None
    dom_bytes, dom_ms = ((B_alg, fused_avg) if use_fused else
                         (kb["recurrence"], seg_rec_avg if best == "seg" else rec_avg))
    dom_achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    t_roof = max(F_alg / (float(peaks["bf16_tflops"]) * 1e12), B_alg / (hbm * 1e9))
    tc = uses_tensor_cores(wl)
    kernel_file = "chunk_tc.cu" if tc else "chunk_simt.cu"
    kernel_name = "chunk_tc_kernel" if tc else "chunk_simt_kernel"
    traffic = profiled_traffic(kernel_file, wl.name, best)
    # fused: stream order + layer kernel; else conv(+L2), (stream order), recurrence
    launches_per_step = 2 if use_fused else (6 if best == "seg" else (3 if tc else 2))
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.dtype,
        "data": "synthetic (seeded; x~N(0,1), conv w~N(0,0.25), h~N(0,0.02), "
                "g=-softplus(N(0,1)), beta=sigmoid(N(0,1)))",
        "config": {"workload": wl.name, "streams": wl.B, "tokens_per_step": T,
                   "path": ("one fused launch (la_prefill_front)" if use_fused else
                            f"fused conv1d+SiLU+L2, then the segmented recurrence ({seg_s} "
                            "segments, la_prefill_segmented)" if best == "seg" else
                            "two launches (fused conv1d+SiLU+L2, then the recurrence)"),
                   "Hk": wl.Hk, "Hv": wl.Hv, "head_dim": wl.d, "variant": wl.variant,
                   "activations": wl.dtype, "states": "f32", "chunk": CHUNK,
                   "compute": ("tensor cores: bf16 (raw inputs) and tf32 (state-derived) MMAs, "
                               "fp32 accumulate; CUDA cores fp32" if tc else "CUDA cores fp32"),
                   "l2": "flushed between timed steps (read of a 258 MiB buffer, outside the events)",
                   "launch": ("one CUDA graph replay per step (the path's public calls, "
                              "captured once)" if best_launch == "graph" else
                              "host launches per step"),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipeline": "host->device copy of step i+1 and device->host copy of step i-1 "
                            "overlap step i's compute (two buffer sets, three streams)"},
        "roofline": {"bound": "hbm",
                     "kernel": kernel_name + (" (conv1d+SiLU+L2+recurrence, one launch)"
                                              if use_fused else
                                              f" (segmented recurrence, {seg_s} segments: setup, "
                                              "recurrence, join, correction launches)"
                                              if best == "seg" else " (recurrence)"),
                     "achieved": dom_achieved, "peak": hbm, "unit": "GB/s",
                     "frac": dom_achieved / hbm, "traffic": traffic,
                     "peak_source": f"{peak_src} hbm_gbs",
                     "algorithmic_bytes_per_launch": dom_bytes,
                     "avg_launch_ms": dom_ms},
        "phases_ms": {"two launches": split_avg, "front_end(conv1d+silu, l2)": front_avg,
                      "recurrence": rec_avg,
                      **({"one fused launch (la_prefill_front)": fused_avg} if fused else {}),
                      **({f"front end + segmented recurrence ({seg_s} segments)":
                          sum(seg_ms) / len(seg_ms),
                          "segmented recurrence": seg_rec_avg} if seg_ms else {}),
                      **{f"graph replay, {m}": sum(v) / len(v) for m, v in graphed.items()}},
        "step_roofline": {"t_roof_ms": t_roof * 1e3, "frac": t_roof / (ms * 1e-3),
                          "bytes_alg": B_alg, "flops_alg": F_alg,
                          "peaks": f"{peak_src}: {hbm} GB/s, {peaks['bf16_tflops']} TFLOP/s bf16"},
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, inp)
    print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


def run_proj(args, wl, dev, local, rank, world, pg):
    """One step = the QKVZ projection GEMM of the stacked tokens (la_gemm_bf16), operands in
    HBM; tensor-bound. torch.matmul (cuBLAS) on the same operands is timed beside it."""
    import linear_attention_chunked_conv1d_gb300 as la
    T = wl.B * int(wl.lengths.split(":")[1])
    Kd, N = wl.hidden, 4 * wl.Hv * wl.d
    gen = torch.Generator(dev)
    gen.manual_seed(rank)
    a = torch.randn(T, Kd, generator=gen, device=dev).to(torch.bfloat16)
    w = (torch.randn(N, Kd, generator=gen, device=dev) / math.sqrt(Kd)).to(torch.bfloat16)
    c = torch.empty(T, N, dtype=torch.bfloat16, device=dev)
    flush = torch.zeros(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)

    def flush_l2():
        """Evict L2 by reading a buffer twice its size: the lines it leaves are clean, so the
        timed step that follows pays no write-back for them."""
        torch.max(flush)
    stream = torch.cuda.current_stream()

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush_l2()
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        return sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps

    if pg:
        pg.barrier()
    clocks = ClockSampler(local)
    clocks.start()
    ms_ours = timed(lambda: la.gemm_bf16(a, w, c))
    clk = clocks.stop()
    ms_cublas = timed(lambda: torch.matmul(a, w.t(), out=c))
    value, ms, _ = aggregate(T, ms_ours, pg, dev)
    # end to end: the hidden rows in from pinned host memory, the projection out
    a_h = a.cpu().pin_memory()
    c_h = torch.empty(c.shape, dtype=c.dtype).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(2):
        a.copy_(a_h, non_blocking=True)
        la.gemm_bf16(a, w, c)
        c_h.copy_(c, non_blocking=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        a.copy_(a_h, non_blocking=True)
        la.gemm_bf16(a, w, c)
        c_h.copy_(c, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_value, _, _ = aggregate(T, e0.elapsed_time(e1) / args.steps, pg, dev)
    if rank != 0:
        if pg:
            pg.barrier()
            pg.destroy_process_group()
        return
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    flops = 2.0 * T * N * Kd
    achieved = flops / (ms_ours * 1e-3) / 1e12
    line = {
        "metric": PROJ_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; hidden rows ~N(0,1), weights ~N(0,1/hidden))",
        "config": {"workload": wl.name, "tokens_per_step": T, "hidden": Kd, "outputs": N,
                   "path": "la_gemm_bf16 (tcgen05 + TMA, 128x256 tiles, fp32 accumulation)",
                   "l2": "flushed between timed steps (read of a 258 MiB buffer, outside the events)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "gpu_launches": args.steps,
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": a_h.numel() * 2,
                "d2h_bytes_per_step": c_h.numel() * 2},
        "roofline": {"bound": "tensor", "kernel": "gemm_bf16_kernel", "achieved": achieved,
                     "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak, "traffic": None,
                     "peak_source": f"{peak_src} bf16_tflops (burst: the kernel is timed alone)",
                     "flops_per_launch": flops, "avg_launch_ms": ms_ours},
        "cublas_same_shape": {"ms": ms_cublas,
                              "tflops": flops / (ms_cublas * 1e-3) / 1e12,
                              "note": "torch.matmul on the same operands, context only"},
    }
    print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


def capture_step(body, stream, warmup):
    """A CUDA graph of one step's public calls (captured on a side stream, then replayed
    `warmup` times), or None where capture is not possible; the caller keeps its paced timings
    then."""
    try:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            body()
        torch.cuda.synchronize()
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        return g
    except Exception:
        torch.cuda.synchronize()
        return None


def run_decode(args, wl, inp, dev, local, rank, world, pg):
    """One step = one decode step of the layer for B streams (one new token each), states in
    HBM: la_decode_step (conv + SiLU + L2 launch, then the recurrence launch)."""
    from linear_attention_chunked_conv1d_gb300.path import DecodeStep

    p = DecodeStep(wl, inp)
    flush = torch.zeros(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)

    def flush_l2():
        """Evict L2 by reading a buffer twice its size: the lines it leaves are clean, so the
        timed step that follows pays no write-back for them."""
        torch.max(flush)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        p.run()
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    def timed(step):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush_l2()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        return [e[0].elapsed_time(e[1]) for e in ev]

    paced_ms = timed(p.run)
    # the same two launches replayed from a CUDA graph of the public call
    g = capture_step(p.run, stream, args.warmup)
    graph_ms = timed(g.replay) if g is not None else None
    clk = clocks.stop()
    use_graph = graph_ms is not None and sum(graph_ms) < sum(paced_ms)
    step_ms = graph_ms if use_graph else paced_ms
    T = wl.B
    value, ms, _ = aggregate(T, sum(step_ms) / len(step_ms), pg, dev)

    # end to end through the public API: this step's token rows, gates in; outputs out
    x_h = inp["x"].cpu().pin_memory()
    g_h = inp["g"].cpu().pin_memory()
    b_h = inp["beta"].cpu().pin_memory()
    out_h = torch.empty(p.out.shape, dtype=p.out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (x_h, g_h, b_h))
    d2h = out_h.numel() * out_h.element_size()
    for _ in range(2):
        inp["x"].copy_(x_h, non_blocking=True)
        p.run()
        out_h.copy_(p.out, non_blocking=True)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        inp["x"].copy_(x_h, non_blocking=True)
        inp["g"].copy_(g_h, non_blocking=True)
        inp["beta"].copy_(b_h, non_blocking=True)
        p.run()
        out_h.copy_(p.out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_value, _, _ = aggregate(T, e0.elapsed_time(e1) / args.steps, pg, dev)
    if rank != 0:
        if pg:
            pg.barrier()
            pg.destroy_process_group()
        return
    peaks, peak_src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    step_avg = sum(step_ms) / len(step_ms)
    B_alg = decode_algorithmic_bytes(wl)
    achieved = B_alg / (step_avg * 1e-3) / 1e9
    line = {
        "metric": DECODE_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic (seeded; x~N(0,1), conv w~N(0,0.25), conv state~N(0,1), "
                "h~N(0,0.02), g=-softplus(N(0,1)), beta=sigmoid(N(0,1)))",
        "config": {"workload": wl.name, "streams": wl.B, "tokens_per_step": T, "Hk": wl.Hk,
                   "Hv": wl.Hv, "head_dim": wl.d, "variant": wl.variant,
                   "activations": wl.dtype, "states": "f32",
                   "path": "la_decode_step (conv1d+SiLU+L2 launch, recurrence launch)",
                   "compute": "CUDA cores fp32 (matrix-vector work per state)",
                   "l2": "flushed between timed steps (read of a 258 MiB buffer, outside the events); the h states "
                         f"({wl.B * wl.Hv * wl.d * wl.d * 4 >> 20} MiB) exceed L2 as well",
                   "launch": ("one CUDA graph replay per step (the public call, captured once)"
                              if use_graph else "host launches per step"),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "roofline": {"bound": "hbm",
                     "kernel": "decode step (conv1d_silu_step_kernel + decode_rec_kernel; the "
                               "events bracket both launches)",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": None, "peak_source": f"{peak_src} hbm_gbs",
                     "algorithmic_bytes_per_launch": B_alg, "avg_launch_ms": step_avg},
        "phases_ms": {"host launches": sum(paced_ms) / len(paced_ms),
                      **({"graph replay": sum(graph_ms) / len(graph_ms)} if graph_ms else {})},
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, inp)
    print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()

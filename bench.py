"""Benchmark of the KDA core library on one GB300 (or N independent replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 2|4|5] [--no-decode] [--no-cpu-baseline]

A step is one chunked prefill (sequence table, K1 preparation, K2 recurrence,
checkpoint writer) over the chosen prefill workload, default the largest one
that fits one GPU, "varlen prefill 16 seqs U[1024,32768] H32 D128 bf16"
(274,076 tokens).  The other prefill workloads ("prefill B1 H32 T8192 D128
bf16" and the 131,072-token prefill with four 32K-token snapshots) are timed
in the same run with fewer steps and reported under "prefill_other".  Decode
(state GB/s) is timed over the decode workload "decode N256 H32 D128 bf16",
64 consecutive steps, and reported under "decode".  Inputs are seeded synthetic draws (see
linear_attention_serving_k1_gb300/workloads.py) made on the device; every
timed prefill step starts from an idle device and L2 is flushed (a 512 MiB
write) before it.  (Back to back, without the synchronisation between steps,
a workload-2 call measures about 5% longer.)  "graph_replay" reports the same
call captured once in a CUDA graph and replayed, timed the same way.

Rank 0 prints one JSON line.  With --impl reference the float64 CPU oracle is
timed instead, on the same workload (or its first heads when it is large).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from linear_attention_serving_k1_gb300 import kda, workloads  # noqa: E402

METRIC = "KDA chunked-prefill tokens/s and decode state GB/s, % of roofline, 1×GB300"
L2_FLUSH_BYTES = 512 << 20


# ------------------------------------------------------------------ accounting
def prefill_algorithmic_bytes(w) -> int:
    """Bytes a prefill must move at minimum: q, k, v (dtype), g (fp32), beta
    (fp32), out (dtype) per token-head, plus the initial and final state and
    every checkpoint (fp32)."""
    es = 2 if w.dtype == "bf16" else 4
    D, H = w.D, w.H
    per_th = 3 * D * es + D * 4 + 4 + D * es
    n_ck = kda.num_checkpoints(w.lens, w.ckpt_stride)
    states = (2 if w.init != "zeros" else 1) * w.num_seqs * H * D * D * 4
    return w.total_tokens * H * per_th + states + n_ck * H * D * D * 4


def prefill_flops(w) -> int:
    """Triangle-aware FLOPs of the chunked form per token-head: 5CD + 6D^2 + C^2/3."""
    C, D = 64, w.D
    return int(w.total_tokens * w.H * (5 * C * D + 6 * D * D + C * C / 3))


def decode_cost_per_head(D: int, es: int = 2):
    """(FLOPs, bytes) of one decode step of one head.  The state part is the
    KDA pages' estimate, 7*D^2 FLOPs and 8*D^2 bytes (fp32 read + write); the
    per-token vectors q, k, v, out (dtype) and g (fp32), beta add 4*D*es+4*D+4."""
    return 7 * D * D, 8 * D * D + 4 * D * es + 4 * D + 4


def load_traffic(key):
    """DRAM bytes per launch that an ncu capture of the current kernels
    recorded (profiles/traffic.json, written with the summary that names the
    command); None if absent."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            return json.load(f).get(key)
    except Exception:
        return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, flag in zip(names, parts[5:9]):
                if flag.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ helpers
def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of x over the ranks (the job's time is the slowest rank's)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = device if device is not None else ("cuda" if torch.cuda.is_available() else "cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, rank_ms_per_step: float, world: int, device=None) -> float:
    """Units per second of the whole job: every rank processes units_per_rank
    per step (replicas of independent work, weak scaling); the step takes as
    long as the slowest rank."""
    ms = max_over_ranks(rank_ms_per_step, world, device)
    return units_per_rank * world / (ms / 1e3)


def time_steps(fn, steps, warmup, flush_buf, stream):
    """Runs fn() warmup + steps times; returns per-step ms (CUDA events on stream)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        # each timed step starts from an idle device: the previous step has
        # finished (synchronize) and L2 holds only the flush buffer's lines
        torch.cuda.synchronize()
        flush_buf.fill_(1.0)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in times]


# ------------------------------------------------------------------ our arm
def bench_prefill(w, steps, warmup, dev, flush_buf, world, e2e=True, graph=True):
    inp = workloads.make_prefill(w, device=dev)
    q, k, v, g, beta = (inp[n] for n in ("q", "k", "v", "g", "beta"))
    s0, cu = inp["init_state"], inp["cu_seqlens"]
    T, H, D, N = w.total_tokens, w.H, w.D, w.num_seqs
    n_ck = kda.num_checkpoints(w.lens, w.ckpt_stride)
    L = max(w.lens)   # the longest sequence: bounds the segment plan and the workspace
    desc = kda.make_desc(T, H, D, N, kda.DTYPE_BF16 if w.dtype == "bf16" else kda.DTYPE_FP32, 64,
                         w.ckpt_stride, n_ck, max_seq_len=L)
    ws = kda.alloc_workspace(desc, dev)
    launches = kda.launch_count(desc)
    out = torch.empty_like(v)
    fin = torch.empty(N, H, D, D, dtype=torch.float32, device=dev)
    ck = torch.empty(max(n_ck, 1), H, D, D, dtype=torch.float32, device=dev) if n_ck else None
    stream = torch.cuda.current_stream()

    def step():
        kda.prefill(q, k, v, g, beta, s0, cu, num_seqs=N, ckpt_stride=w.ckpt_stride, ckpts=ck,
                    ckpt_capacity=n_ck, out=out, final_state=fin, workspace=ws, stream=stream, max_seq_len=L)

    barrier(world)
    torch.cuda.synchronize()
    ms = time_steps(step, steps, warmup, flush_buf, stream)
    barrier(world)
    torch.cuda.synchronize()
    assert kda.prefill_status(ws) == 0

    # the same call captured once in a CUDA graph and replayed every step: the
    # same kernels on the same inputs, without the host-side launches and with
    # shorter gaps between kernels; reported beside the eager number
    graph_ms = None
    try:
        if not graph:
            raise RuntimeError("not requested")
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            kda.prefill(q, k, v, g, beta, s0, cu, num_seqs=N, ckpt_stride=w.ckpt_stride, ckpts=ck,
                        ckpt_capacity=n_ck, out=out, final_state=fin, workspace=ws, stream=cap, max_seq_len=L)
        torch.cuda.synchronize()
        graph_ms = time_steps(graph.replay, steps, warmup, flush_buf, stream)
        assert kda.prefill_status(ws) == 0
    except RuntimeError as e:   # capture unsupported here: report the eager number only
        if graph:
            print(f"graph replay skipped: {e}", file=sys.stderr)
    barrier(world)

    if not e2e:
        return ms, None, 0, 0, launches, graph_ms
    # end to end: every step copies its inputs from pinned host memory to the
    # device, runs the prefill and copies o and the final states back.  Two
    # buffer slots let step i + 1's inputs travel (two copy streams) while step
    # i computes and step i - 1's outputs travel back (a third stream); the
    # time per step is the whole run's time over the steps (inputs exceed L2).
    names = ("q", "k", "v", "g", "beta")
    host_in = {n: inp[n].cpu().pin_memory() for n in names}
    host_s0 = s0.cpu().pin_memory() if s0 is not None else None
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    h2d += host_s0.numel() * 4 if host_s0 is not None else 0
    d2h = out.numel() * out.element_size() + fin.numel() * 4
    slots = []
    for _ in range(2):
        slots.append({
            "in": {n: torch.empty_like(inp[n]) for n in names},
            "s0": torch.empty_like(s0) if s0 is not None else None,
            "out": torch.empty_like(out), "fin": torch.empty_like(fin),
            "host_out": torch.empty(out.shape, dtype=out.dtype).pin_memory(),
            "host_fin": torch.empty(fin.shape, dtype=fin.dtype).pin_memory(),
            "in_ready": [torch.cuda.Event(), torch.cuda.Event()],
            "comp_done": torch.cuda.Event(), "out_done": torch.cuda.Event(), "used": False})
    h2d_streams = [torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)]
    d2h_stream = torch.cuda.Stream(device=dev)
    split = [["q", "v", "beta"], ["k", "g"]]   # about half of the input bytes each

    def run(n_steps):
        for i in range(n_steps):
            sl = slots[i % 2]
            for j, hs in enumerate(h2d_streams):
                if sl["used"]:
                    hs.wait_event(sl["comp_done"])
                with torch.cuda.stream(hs):
                    for n in split[j]:
                        sl["in"][n].copy_(host_in[n], non_blocking=True)
                    if j == 0 and sl["s0"] is not None:
                        sl["s0"].copy_(host_s0, non_blocking=True)
                sl["in_ready"][j].record(hs)
            for ev in sl["in_ready"]:
                stream.wait_event(ev)
            if sl["used"]:
                stream.wait_event(sl["out_done"])
            d = sl["in"]
            kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], sl["s0"], cu, num_seqs=N,
                        ckpt_stride=w.ckpt_stride, ckpts=ck, ckpt_capacity=n_ck, out=sl["out"],
                        final_state=sl["fin"], workspace=ws, stream=stream, max_seq_len=L)
            sl["comp_done"].record(stream)
            d2h_stream.wait_event(sl["comp_done"])
            with torch.cuda.stream(d2h_stream):
                sl["host_out"].copy_(sl["out"], non_blocking=True)
                sl["host_fin"].copy_(sl["fin"], non_blocking=True)
            sl["out_done"].record(d2h_stream)
            sl["used"] = True
        for sl in slots:
            stream.wait_event(sl["out_done"])

    run(max(3, warmup))
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    run(steps)
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = [a.elapsed_time(b) / steps] * steps
    del slots, host_in
    return ms, e2e_ms, h2d, d2h, launches, graph_ms


def bench_decode(steps_total, dev, flush_buf, warmup=3):
    w = workloads.workload(3)
    st = workloads.make_decode_state(w, device=dev)
    xs = [workloads.make_decode_step(w, s, device=dev) for s in range(steps_total)]
    out = torch.empty(w.N, w.H, w.D, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    for s in range(warmup):
        x = xs[s % len(xs)]
        kda.decode(x["q"], x["k"], x["v"], x["g"], x["beta"], st, out=out, stream=stream)
    torch.cuda.synchronize()
    evs = []
    for s in range(steps_total):
        x = xs[s]
        flush_buf.fill_(1.0)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        kda.decode(x["q"], x["k"], x["v"], x["g"], x["beta"], st, out=out, stream=stream)
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in evs]
    return w, ms


def cpu_baseline_prefill(w, max_token_heads=4_000_000):
    """Times the float64 oracle (OpenMP over sequence x head) on the prefill
    workload: the whole workload when it has at most max_token_heads
    token-heads, else its first heads.  Returns the dict of the JSON line."""
    from oracle import oracle
    inp = workloads.make_prefill(w)
    heads = list(range(w.H))
    while len(heads) > 1 and w.total_tokens * len(heads) > max_token_heads:
        heads = heads[: len(heads) // 2]
    args = [inp[n] for n in ("q", "k", "v", "g", "beta")]
    t0 = time.perf_counter()
    oracle.prefill_heads(*args, inp["init_state"], inp["cu_host"].numpy(), w.ckpt_stride, heads=heads)
    elapsed = time.perf_counter() - t0
    value = w.total_tokens * len(heads) / w.H / elapsed
    what = "the whole workload" if len(heads) == w.H else f"{len(heads)} of {w.H} heads"
    return {"value": round(value, 1), "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{what} ({w.total_tokens} tokens), float64 token recurrence, {elapsed:.2f} s; "
                      f"tokens/s counts all H heads of a token"}


def shrink(w, factor: int):
    """The workload with every sequence length divided by ``factor`` (at least
    one token), named accordingly; ``factor`` 1 returns it unchanged."""
    if factor <= 1:
        return w
    import dataclasses
    lens = tuple(max(1, L // factor) for L in w.lens)
    stride = w.ckpt_stride // factor // 64 * 64 if w.ckpt_stride else 0
    return dataclasses.replace(w, lens=lens, ckpt_stride=stride, name=f"{w.name}, lengths / {factor}")


def run_ours(args):
    world, rank, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local if world > 1 else 0)
    kda.load_library()
    peaks = load_peaks()
    w = shrink(workloads.workload(args.workload), args.shrink)
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    clk = ClockSampler(dev.index if dev.index is not None else 0)
    clk.start()
    ms, e2e_ms, h2d, d2h, launches, graph_ms = bench_prefill(w, args.steps, args.warmup, dev, flush_buf,
                                                             world, not args.no_e2e)
    others = []
    if not args.no_other:
        for wi in (2, 4, 5):
            if wi == args.workload:
                continue
            wo = workloads.workload(wi)
            o_ms, _, _, _, o_launch, _ = bench_prefill(wo, max(3, args.steps // 2), args.warmup, dev, flush_buf,
                                                        world, e2e=False, graph=False)
            others.append((wo, wi, o_ms, o_launch))
            torch.cuda.empty_cache()
    dec = None
    if not args.no_decode:
        dec_w, dec_ms = bench_decode(64, dev, flush_buf)
    clocks = clk.stop()

    ms_per_step = max_over_ranks(sum(ms) / len(ms), world)
    value = job_throughput(w.total_tokens, sum(ms) / len(ms), world)
    e2e_val = job_throughput(w.total_tokens, sum(e2e_ms) / len(e2e_ms), world) if e2e_ms else None
    graph = None
    if graph_ms:
        g_ms = max_over_ranks(sum(graph_ms) / len(graph_ms), world)
        graph = {"value": round(job_throughput(w.total_tokens, sum(graph_ms) / len(graph_ms), world), 1),
                 "unit": "tokens/s", "ms_per_step": round(g_ms, 4),
                 "frac": round(prefill_algorithmic_bytes(w) / (g_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                 "note": "the same call captured once in a CUDA graph and replayed each step "
                         "(same kernels and inputs, same flush and timing)"}

    alg_bytes = prefill_algorithmic_bytes(w)
    achieved = alg_bytes / (ms_per_step / 1e3) / 1e9
    roof = {"kernel": f"kda_prefill: one call = {launches} launches (sequence table, then K1 and K2 per "
                      "segment, overlapped on two streams), timed as a unit",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": load_traffic(f"prefill_w{args.workload}"),
            "algorithmic_bytes_per_launch": alg_bytes,
            "tensor_tflops": round(prefill_flops(w) / (ms_per_step / 1e3) / 1e12, 2),
            "peak_source": peaks["source"]}
    if not args.no_decode:
        f_h, b_h = decode_cost_per_head(dec_w.D)
        heads = dec_w.N * dec_w.H
        dec_ms_med = statistics.median(dec_ms)
        dec_mean = sum(dec_ms) / len(dec_ms)
        dec_gbs = b_h * heads / (dec_mean / 1e3) / 1e9
        dec = {"workload": dec_w.name, "metric": "decode state GB/s", "unit": "GB/s",
               "value": round(dec_gbs, 1), "us_per_step": round(dec_mean * 1e3, 2),
               "us_per_step_median": round(dec_ms_med * 1e3, 2), "steps": len(dec_ms),
               "roofline": {"bound": "hbm", "achieved": round(dec_gbs, 1), "peak": peaks["hbm_gbs"],
                            "unit": "GB/s", "frac": round(dec_gbs / peaks["hbm_gbs"], 4),
                            "traffic": load_traffic("decode_w3"),
                            "algorithmic_bytes_per_launch": b_h * heads}}
    line = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": len(ms), "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic (seeded, on device)",
            "config": {"workload": w.name, "tokens_per_step": w.total_tokens, "heads": w.H,
                       "head_dim": w.D, "chunk": 64, "ckpt_stride": w.ckpt_stride,
                       "l2": "flushed (512 MiB write) before every timed step, each step started from an idle device; inputs also exceed L2",
                       "parallelism": f"replicas x{world}"},
            "roofline": roof,
            "e2e": ({"value": round(e2e_val, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                     "d2h_bytes_per_step": d2h,
                     "pipeline": "two buffer slots: step i+1's pinned-host inputs copied (two streams) "
                                 "while step i computes and step i-1's o and final states copy back"}
                    if e2e_val else None),
            "gpu_launches": launches * len(ms),
            "graph_replay": graph,
            "clocks": clocks,
            "decode": dec}
    if others:
        line["prefill_other"] = []
        for wo, wi, o_ms, o_launch in others:
            o_mean = max_over_ranks(sum(o_ms) / len(o_ms), world)
            o_bytes = prefill_algorithmic_bytes(wo)
            o_gbs = o_bytes / (o_mean / 1e3) / 1e9
            line["prefill_other"].append({
                "workload": wo.name, "ms_per_step": round(o_mean, 4), "steps": len(o_ms),
                "value": round(job_throughput(wo.total_tokens, sum(o_ms) / len(o_ms), world), 1),
                "unit": "tokens/s", "gpu_launches": o_launch * len(o_ms),
                "roofline": {"bound": "hbm", "achieved": round(o_gbs, 1), "peak": peaks["hbm_gbs"],
                             "unit": "GB/s", "frac": round(o_gbs / peaks["hbm_gbs"], 4),
                             "traffic": load_traffic(f"prefill_w{wi}"), "algorithmic_bytes_per_launch": o_bytes}})
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_prefill(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------ reference arm
def run_reference(args):
    """The float64 CPU oracle on the same workload, metric and unit (the
    pages publish no implementation to run): every step is the whole prefill
    workload (about a second on 16 cores for the default workload), or its
    first heads when the workload is larger."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    from oracle import oracle
    w = workloads.workload(args.workload)
    inp = workloads.make_prefill(w)
    heads = list(range(w.H))
    while len(heads) > 1 and w.total_tokens * len(heads) > 1_000_000:
        heads = heads[: len(heads) // 2]
    args_ = [inp[n] for n in ("q", "k", "v", "g", "beta")]
    cu = inp["cu_host"].numpy()

    def step():
        oracle.prefill_heads(*args_, inp["init_state"], cu, w.ckpt_stride, heads=heads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    ms_per_step = el / args.steps * 1e3
    value = w.total_tokens * len(heads) / w.H / (ms_per_step / 1e3)
    what = "the whole workload" if len(heads) == w.H else f"{len(heads)} of {w.H} heads of the workload"
    sample = f"{what} per step ({w.total_tokens} tokens), float64 token recurrence; tokens/s counts all H heads"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": w.name, "sample": sample},
            "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=5, choices=[1, 2, 4, 5])
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-other", action="store_true", help="skip the other prefill workloads")
    ap.add_argument("--shrink", type=int, default=1,
                    help="divide every sequence length of the workload by this factor (a smaller case of the "
                         "same shape for profiler captures; the JSON line then names the shrunk workload)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end timing")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

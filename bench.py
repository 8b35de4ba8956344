#!/usr/bin/env python
"""Benchmark of the SSD chunked-scan forward on the Mamba-2 2.7B shape.

Workload: batch 8, seqlen 4096, 80 heads, headdim 64 (d_inner 5120), dstate
128, 1 group, chunk 256, bf16 inputs, fp32 states, z gate and D skip on;
synthetic seeded inputs (ssd_inputs.py).  One step = one ssd_scan_fwd call
over the whole batch (all four stages).

Prints ONE JSON line (rank 0).  `value` is whole-job tokens/s with inputs
resident in HBM (one event pair per call: mean, median and p90 per call; a
second, seconds-long block of back-to-back calls gives ms_per_step_long);
`e2e` is the same metric with the host->device copy of the inputs and the
device->host copy of the output inside the timed region.  `roofline` rates
the kernel that takes most of the step against the measured peaks in
MEASURED_PEAKS.json.  `cpu_baseline` times the fp64 CPU oracle on a bounded
sample of the same workload, and `parity` compares that sample with the GPU
output (max and mean relative error, mean signed error, 99.9th percentile).
`other_configs` times the chained-prefill and packed-documents workloads the
same way (inputs drawn on the device), the decode step, the forward in fp32,
a bf16 shape outside the fused kernel (headdim 128 at the same width), the
backward (ssd_scan_bwd, fp32) and the block's conv1d and grouped RMSNorm
passes at the same shape.

`--impl reference` times the oracle alone (the only reference this workload
has) and prints its own line.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SSD chunked-scan fwd tokens/s at 2.7B shape, bf16; % of roofline"
# the 2.7B shape's inner width (5120) with headdim 128: a bf16 shape the fused
# kernel does not take
HD128 = (40, 128)
UNIT = "tokens/s"
WORKLOAD = "mamba2_2p7b"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0, "source": "fallback"}
FP32_LANES_PER_SM = 128


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD,
                    help="mamba2_2p7b (default), or one other workload alone: chained, packed, "
                         "backward, forward_fp32, forward_bf16_hd128")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle sample")
    ap.add_argument("--long-seconds", type=float, default=3.0,
                    help="length of the back-to-back block (0: skip)")
    ap.add_argument("--no-other", action="store_true", help="skip the other workloads")
    ap.add_argument("--batch", type=int, default=None,
                    help="batch of --workload backward / forward_fp32 (default: the 2.7B "
                         "shape's 8; smaller for profiler captures)")
    return ap.parse_args()


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    return dict(FALLBACK_PEAKS)


# ---------------------------------------------------------------------------
# algorithmic work per call (counts the method needs, not what a kernel does)
# ---------------------------------------------------------------------------

def algorithmic(cfg, seqlen=None, init=False, final=False, seq=False) -> dict:
    """Counts of one call over `seqlen` tokens (default the workload's):
    read x, z, dt, B, C, A, D, dt_bias (and initial states, seq_idx) once,
    write out (and final states) once."""
    e = 2 if cfg.dtype == "bf16" else 4
    Bz, L, H, P, N, G, Q = (cfg.batch, seqlen or cfg.seqlen, cfg.nheads, cfg.headdim,
                            cfg.dstate, cfg.ngroups, cfg.chunk_size)
    nc = -(-L // Q)
    x = Bz * L * H * P * e
    bc = Bz * L * G * N * e
    dt = Bz * L * H * e
    state = Bz * nc * H * P * N * 4
    chunk_f32 = Bz * H * nc * Q * 4
    hstate = Bz * H * P * N * 4
    io = ((3 if cfg.has_z else 2) * x + 2 * bc + dt + 3 * H * 4
          + (hstate if init else 0) + (hstate if final else 0) + (Bz * L * 4 if seq else 0))
    tri = Q * (Q + 1) // 2
    # causal flops: C B^T once per group, masked (CB) x and C h per head, B^T x per head
    flops = Bz * nc * (G * tri * N * 2 + H * (tri * P * 2 + 2 * Q * N * P * 2))
    return dict(io_bytes=io, flops=flops, x=x, bc=bc, dt=dt, state=state, chunk_f32=chunk_f32,
                tri=tri, nc=nc)


def kernel_models(cfg, peaks, num_sms, **kw) -> dict:
    """Per-kernel algorithmic bytes / flops and the roofline that bounds it."""
    a = algorithmic(cfg, **kw)
    Bz, H, P, N, G, Q, nc = (cfg.batch, cfg.nheads, cfg.headdim, cfg.dstate, cfg.ngroups,
                             cfg.chunk_size, a["nc"])
    hbm = peaks["hbm_gbs"] * 1e9
    alu = num_sms * FP32_LANES_PER_SM * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6
    m = {}
    m["dt_cumsum"] = dict(bytes=a["dt"] + 2 * a["chunk_f32"], flops=0, bound="hbm", peak=hbm)
    m["chunk_state"] = dict(bytes=a["x"] + a["bc"] + 2 * a["chunk_f32"] + a["state"],
                            flops=Bz * nc * H * 2 * Q * N * P, bound="alu", peak=alu)
    m["state_passing"] = dict(bytes=2 * a["state"], flops=0, bound="hbm", peak=hbm)
    # the fused kernel runs all four stages: its algorithmic bytes are the
    # scan's own I/O, its flops all the causal flops
    m["scan_fused"] = dict(bytes=a["io_bytes"], flops=a["flops"], bound="hbm", peak=hbm,
                           tensor_peak=peaks["bf16_tflops"] * 1e12)
    m["chunk_scan"] = dict(bytes=3 * a["x"] + 2 * a["bc"] + 2 * a["chunk_f32"] + a["state"],
                           flops=Bz * nc * (G * a["tri"] * N * 2 + H * (a["tri"] * P * 2 +
                                                                       Q * N * P * 2)),
                           bound="alu", peak=alu)
    return m


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch recorded from an ncu capture (profiles/
    dram_traffic.txt), or None when none was taken or the kernel's source
    has changed since."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        f = line.split()
        if len(f) != 5 or line.startswith("#") or f[0] != kernel or f[4] != workload:
            continue
        src = os.path.join(ROOT, f[2])
        if not os.path.exists(src):
            return None
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:12]
        return int(f[1]) if sha == f[3] else None
    return None


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        self.proc.wait(timeout=10)
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows),
                "power_w_max": max((float(r[3]) for r in rows
                                    if r[3].replace(".", "").isdigit()), default=None)}


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample
# ---------------------------------------------------------------------------

def oracle_sample(cfg, inputs, target_s: float, seed_heads=0):
    """Times the fp64 oracle on a sample of (batch row, head) recurrences sized
    to about target_s seconds.  Returns a dict: rate (tokens/s equivalent; a
    token-equivalent is one token through all heads), cores, description,
    seconds, and the sample's outputs with the batch rows and heads it covers."""
    from oracle import ssd_oracle as so
    cores = so.default_threads()
    H, L, Bz = cfg.nheads, cfg.seqlen, cfg.batch
    t = time.perf_counter()   # calibration: one (row, head) on one thread
    so.scan_sequential(inputs, heads=[seed_heads % H], batches=[0], nthreads=1)
    one = max(time.perf_counter() - t, 1e-3)
    pairs = int(max(min(cores, H), min(Bz * H, round(target_s * cores / one))))
    if pairs <= H:
        batches, heads = [0], [(seed_heads + i) % H for i in range(pairs)]
    else:
        batches, heads = list(range(min(Bz, -(-pairs // H)))), None
    t = time.perf_counter()
    y, fin = so.scan_sequential(inputs, heads=heads, batches=batches, nthreads=cores)
    dt = time.perf_counter() - t
    nh = H if heads is None else len(heads)
    tokens_equiv = L * len(batches) * nh / H
    desc = (f"fp64 sequential oracle on {len(batches)} batch row(s) x {nh} of {H} "
            f"heads, seqlen {L}: {tokens_equiv:.0f} token-equivalents (one token through "
            f"all heads) in {dt:.2f} s")
    return dict(rate=tokens_equiv / dt, cores=cores, desc=desc, seconds=dt, y=y, fin=fin,
                batches=batches, heads=list(range(H)) if heads is None else heads)


def error_metrics(pairs) -> dict:
    """max |err| / max |ref|, mean |err| / mean |ref|, mean signed error and
    the 99.9th percentile of |err| / max |ref| (the largest over the pieces,
    which are batch rows of equal size) over (got, ref) array pairs."""
    import numpy as np
    mx = mref = sabs = sref = sdiff = 0.0
    n = 0
    qs = []
    for got, ref in pairs:
        d = np.asarray(got, dtype=np.float64) - ref
        ad = np.abs(d)
        mx, mref = max(mx, float(ad.max())), max(mref, float(np.abs(ref).max()))
        sabs += float(ad.sum())
        sref += float(np.abs(ref).sum())
        sdiff += float(d.sum())
        n += ad.size
        qs.append(np.quantile(ad, 0.999))   # per piece; the pieces are equal-sized rows
    return {"max_rel": mx / max(mref, 1e-300), "mean_rel": sabs / max(sref, 1e-300),
            "mean_diff": sdiff / max(n, 1), "p999_rel": float(max(qs)) / max(mref, 1e-300),
            "elements": n}


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


# ---------------------------------------------------------------------------

def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest value of a per-rank float over all ranks of the job (a
    replicated job's step time is its slowest rank's); x itself for one rank.
    Uses the default process group (nccl on GPUs, gloo in the CPU tests)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_string(cfg) -> str:
    return (f"{cfg.name}: batch {cfg.batch}, seqlen {cfg.seqlen}, nheads {cfg.nheads}, "
            f"headdim {cfg.headdim}, dstate {cfg.dstate}, ngroups {cfg.ngroups}, chunk "
            f"{cfg.chunk_size}, z gate + D skip, fp32 state")


def bench_line(cfg, world: int, steps: int, warmup: int, ms: float, extra: dict) -> dict:
    """The JSON line of the device-timed arm: every rank runs the whole
    workload (replicas, weak scaling), so the job's throughput counts all
    ranks' tokens over the slowest rank's step time ms.  extra carries the
    measured sections (roofline, whole_call, cpu_baseline, e2e, gpu_launches,
    clocks)."""
    line = {
        "metric": METRIC, "value": cfg.tokens * world / (ms / 1e3), "unit": UNIT,
        "n_gpus": world, "steps": steps, "warmup": warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if cfg.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": workload_string(cfg),
                   "global_batch": cfg.batch * world, "seq_len": cfg.seqlen,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (x, z, out are 335 MB each; L2 129 MB)"},
    }
    line.update(extra)
    return line


def run_reference(args, cfg):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import ssd_inputs as si
    inputs = si.make_inputs(cfg, 1002)
    per_step = max(1.0, 90.0 / max(1, args.steps + args.warmup))
    rates = []
    desc = cores = None
    for i in range(args.warmup + args.steps):
        s = oracle_sample(cfg, inputs, per_step, seed_heads=i)
        cores, desc = s["cores"], s["desc"]
        del s["y"], s["fin"]
        if i >= args.warmup:
            rates.append(s["rate"])
    value = statistics.median(rates)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * cfg.tokens / value, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_string(cfg), "sample": desc},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc, "cpu": cpu_model()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def time_calls(torch, step, n, stream):
    """n calls of step() with one CUDA event between consecutive calls, on the
    launching stream; returns (mean ms per call, per-call ms list)."""
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    evs[0].record(stream)
    for i in range(n):
        step()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(n)]
    return evs[0].elapsed_time(evs[n]) / n, per


def spread(per) -> dict:
    s = sorted(per)
    return {"median": statistics.median(s), "p90": s[min(len(s) - 1, int(0.9 * len(s)))],
            "min": s[0], "max": s[-1]}


def other_workload(torch, ssd, si, name, dev, stream, peaks, steps, warmup, num_sms):
    """Times one more workload through ssd_scan_fwd with inputs drawn on the
    device: the chained prefill (segments with the final states fed back as
    the next initial states; all tokens counted) or the packed documents (one
    call with seq_idx)."""
    cfg = si.CONFIGS[name]
    g = si.make_inputs(cfg, 2000 + len(name), device=dev)
    Q = cfg.chunk_size
    S = cfg.segments
    seg_len = cfg.seqlen // S
    Bz, H, P, N = cfg.batch, cfg.nheads, cfg.headdim, cfg.dstate
    parts = [{k: g[k][:, s * seg_len:(s + 1) * seg_len].contiguous()
              for k in ("x", "dt", "B", "C", "z")} for s in range(S)] if S > 1 else [g]
    outs = [torch.empty_like(p["x"]) for p in parts]
    fins = [torch.empty(Bz, H, P, N, dtype=torch.float32, device=dev) for _ in range(2)]
    ws = torch.empty(ssd.workspace_bytes(Bz, seg_len, H, P, N, cfg.ngroups, Q, g["x"].dtype),
                     dtype=torch.uint8, device=dev)
    chained = S > 1

    def step():
        init = g["initial_states"]
        for s, p in enumerate(parts):
            ssd.ssd_scan_fwd(p["x"], p["dt"], g["A"], p["B"], p["C"], chunk_size=Q,
                             dt_bias=g["dt_bias"], D=g["D"], z=p["z"], initial_states=init,
                             seq_idx=g["seq_idx"], out=outs[s],
                             final_states=fins[s % 2] if chained else None,
                             return_final_states=chained, workspace=ws, stream=stream)
            init = fins[s % 2]

    for _ in range(max(warmup, 2)):
        step()
    torch.cuda.synchronize()
    ms, per = time_calls(torch, step, steps, stream)
    ssd.scan_status(reset=True, stream=stream)
    a = algorithmic(cfg, seqlen=seg_len, init=g["initial_states"] is not None or chained,
                    final=chained, seq=g["seq_idx"] is not None)
    ms_call = ms / S
    achieved = a["io_bytes"] / (ms_call / 1e3) / 1e9
    del g, parts, outs, fins, ws
    torch.cuda.empty_cache()
    return {"workload": workload_string(cfg) + (f", {S} chained calls of {seg_len} tokens"
                                                if chained else ", seq_idx documents"),
            "tokens_per_step": cfg.tokens, "calls_per_step": S, "ms_per_step": ms,
            "ms_per_call": ms_call, "value": cfg.tokens / (ms / 1e3), "unit": UNIT,
            "per_step_ms": spread(per), "steps": steps,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         "alg_bytes_per_call": a["io_bytes"], "alg_flops_per_call": a["flops"],
                         "tensor_frac": a["flops"] / (ms_call / 1e3) / (peaks["bf16_tflops"]
                                                                        * 1e12)},
            "gpu_launches": steps * S, "data": "synthetic, drawn on the device"}


def decode_workload(torch, ssd, si, dev, stream, peaks, steps):
    """Decode steps (ssd_decode_step) at the 2.7B shape: one token per batch
    row from a state in HBM, advanced in place; HBM-bound on the fp32 state
    (read and written once per step)."""
    cfg = si.CONFIGS["mamba2_2p7b"]
    Bz, H, P, N, G = cfg.batch, cfg.nheads, cfg.headdim, cfg.dstate, cfg.ngroups
    gen = torch.Generator(device=dev).manual_seed(77)
    bf = torch.bfloat16
    x = torch.randn(Bz, H, P, generator=gen, device=dev).to(bf)
    z = torch.randn(Bz, H, P, generator=gen, device=dev).to(bf)
    dt = torch.randn(Bz, H, generator=gen, device=dev).to(bf)
    Bm = torch.randn(Bz, G, N, generator=gen, device=dev).to(bf)
    Cm = torch.randn(Bz, G, N, generator=gen, device=dev).to(bf)
    A = -torch.exp(torch.rand(H, generator=gen, device=dev) * 2.77)
    bias = torch.full((H,), -3.0, device=dev)
    D = torch.randn(H, generator=gen, device=dev)
    state = torch.randn(Bz, H, P, N, generator=gen, device=dev) * 0.1
    out = torch.empty_like(x)
    n = max(steps, 200)

    def step():
        ssd.ssd_decode_step(x, dt, A, Bm, Cm, state, dt_bias=bias, D=D, z=z, out=out,
                            stream=stream)

    for _ in range(20):
        step()
    torch.cuda.synchronize()
    ms_host, per = time_calls(torch, step, n, stream)   # one host call per step
    # a decoding loop replays captured steps: 64 steps per CUDA graph
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for _ in range(3):
            ssd.ssd_decode_step(x, dt, A, Bm, Cm, state, dt_bias=bias, D=D, z=z, out=out,
                                stream=side)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cap = torch.cuda.current_stream(dev)
        for _ in range(64):
            ssd.ssd_decode_step(x, dt, A, Bm, Cm, state, dt_bias=bias, D=D, z=z, out=out,
                                stream=cap)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    reps = max(1, n // 64)
    ms_graph, _ = time_calls(torch, graph.replay, reps, torch.cuda.current_stream(dev))
    ms = ms_graph / 64
    alg = 2 * state.numel() * 4 + 3 * x.numel() * 2 + dt.numel() * 2 + 2 * Bm.numel() * 2 + 3 * H * 4
    achieved = alg / (ms / 1e3) / 1e9
    return {"workload": f"decode step: batch {Bz}, nheads {H}, headdim {P}, dstate {N}, ngroups "
                        f"{G}, bf16, fp32 state", "ms_per_call": ms, "us_per_call": ms * 1e3,
            "us_per_call_host_launched": ms_host * 1e3,
            "value": Bz / (ms / 1e3), "unit": "tokens/s", "per_call_ms_host_launched": spread(per),
            "calls": reps * 64, "timing": "CUDA graph of 64 steps, replayed",
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         "alg_bytes_per_call": alg},
            "gpu_launches": reps * 64 + n, "data": "synthetic, drawn on the device"}


def backward_workload(torch, ssd, si, dev, stream, peaks, steps, batch=None):
    """The backward (ssd_scan_bwd, fp32) at the 2.7B shape: gradients of
    sum(out * dout) for every input, inputs drawn on the device.  Its
    contractions run on the tensor cores as 3xTF32 (three tf32 MMAs per fp32
    product), so the binding roofline is the tf32 tensor peak (the measured
    bf16 burst x 1/2, the nominal tf32 : bf16 ratio); the HBM view of the
    same call is reported beside it."""
    cfg = si.CONFIGS["mamba2_2p7b"].with_(dtype="f32", init_std=0.1)
    if batch:
        cfg = cfg.with_(batch=batch)
    d = si.make_inputs(cfg, 91, device=dev)
    Bz, L, H, P, N, G = cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim, cfg.dstate, cfg.ngroups
    gen = torch.Generator(device=dev).manual_seed(92)
    dout = torch.randn(Bz, L, H, P, generator=gen, device=dev)
    ws = torch.empty(ssd.bwd_workspace_bytes(Bz, L, H, P, N, G, cfg.chunk_size),
                     dtype=torch.uint8, device=dev)

    def step():
        ssd.ssd_scan_bwd(dout, d["x"], d["dt"], d["A"], d["B"], d["C"],
                         chunk_size=cfg.chunk_size, dt_bias=d["dt_bias"], D=d["D"], z=d["z"],
                         initial_states=d["initial_states"], workspace=ws, stream=stream)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    n = max(3, min(steps, 10))
    ms, per = time_calls(torch, step, n, stream)
    ssd.scan_status(stream=stream)
    f4 = 4
    alg = f4 * (5 * Bz * L * H * P + 2 * Bz * L * H + 4 * Bz * L * G * N + 2 * Bz * H * P * N
                + 6 * H)
    # MMA work per (batch row, 128-token chunk, head): two scans in each
    # orientation (headdim x dstate and dstate x headdim), each the
    # inter-chunk term, M x and the chunk state, and C B^T -- once per group
    # for the headdim x dstate scans (one product serves both), per head for
    # the swapped ones; 3 tf32 products per fp32 one
    Q = 128
    nc = (L + Q - 1) // Q
    tiles = Bz * nc * H

    def scan_macs(p, n_):
        return Q * p * n_ + Q * p * Q + p * n_ * Q
    macs = (2 * scan_macs(P, N) + 2 * scan_macs(N, P) + 2 * Q * Q * P) * tiles \
        + Bz * nc * G * Q * Q * N
    fl_alg = 2 * macs
    fl_exec = 3 * fl_alg
    peak_tf32 = peaks["bf16_tflops"] / 2
    ach = fl_exec / (ms / 1e3) / 1e12
    hbm = alg / (ms / 1e3) / 1e9
    return {"workload": f"backward: batch {Bz}, seqlen {L}, nheads {H}, headdim {P}, dstate {N}, "
                        f"ngroups {G}, chunk {cfg.chunk_size} (run at 128), fp32, z gate, D, "
                        "initial states; gradients of every input",
            "ms_per_call": ms, "per_call_ms": spread(per), "calls": n,
            "value": Bz * L / (ms / 1e3), "unit": "tokens/s",
            "roofline": {"bound": "tensor", "achieved": ach, "peak": peak_tf32,
                         "unit": "TFLOP/s", "frac": ach / peak_tf32,
                         "peak_source": "measured bf16 burst x 1/2 (nominal tf32 : bf16)",
                         "flop_per_call_executed": fl_exec, "flop_per_call_fp32": fl_alg,
                         "note": "executed = 3 tf32 MMAs per fp32 product (3xTF32)"},
            "hbm_view": {"alg_bytes_per_call": alg, "achieved_gbs": hbm,
                         "frac": hbm / peaks["hbm_gbs"]},
            "data": "synthetic, drawn on the device"}


def fp32_forward_workload(torch, ssd, si, dev, stream, peaks, steps, batch=None, dtype="f32",
                          heads_dim=None):
    """The forward in fp32 at the 2.7B shape: the four stage kernels, with
    chunk_state and chunk_scan on the tensor cores (3xTF32, run at 128-token
    chunks); HBM roofline on the call's algorithmic bytes.  With dtype
    "bf16" and heads_dim (nheads, headdim) a bf16 shape the fused kernel does
    not take, which runs the same stages on fp32 copies of its inputs."""
    cfg = si.CONFIGS["mamba2_2p7b"].with_(dtype=dtype)
    if heads_dim:
        cfg = cfg.with_(nheads=heads_dim[0], headdim=heads_dim[1])
    if batch:
        cfg = cfg.with_(batch=batch)
    d = si.make_inputs(cfg, 93, device=dev)
    Bz, L, H, P, N, G = cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim, cfg.dstate, cfg.ngroups
    out = torch.empty_like(d["x"])
    fin = torch.empty(Bz, H, P, N, device=dev)
    ws = torch.empty(ssd.workspace_bytes(Bz, L, H, P, N, G, cfg.chunk_size, d["x"].dtype),
                     dtype=torch.uint8, device=dev)

    def step():
        ssd.ssd_scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], chunk_size=cfg.chunk_size,
                         dt_bias=d["dt_bias"], D=d["D"], z=d["z"], out=out, final_states=fin,
                         return_final_states=True, workspace=ws, stream=stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    n = max(5, min(steps, 20))
    ms, per = time_calls(torch, step, n, stream)
    e = 2 if dtype == "bf16" else 4
    alg = (e * (3 * Bz * L * H * P + Bz * L * H + 2 * Bz * L * G * N)
           + 4 * (Bz * H * P * N + 3 * H))
    ach = alg / (ms / 1e3) / 1e9
    route = "(stages at 128)" if dtype == "f32" else "(fp32 stages at 128 on fp32 copies)"
    return {"workload": f"forward {dtype}: batch {Bz}, seqlen {L}, nheads {H}, headdim {P}, dstate "
                        f"{N}, ngroups {G}, chunk {cfg.chunk_size} {route}, z gate, D, "
                        "final states",
            "ms_per_call": ms, "per_call_ms": spread(per), "calls": n,
            "value": Bz * L / (ms / 1e3), "unit": "tokens/s",
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": ach / peaks["hbm_gbs"], "alg_bytes_per_call": alg},
            "data": "synthetic, drawn on the device"}


def block_workload(torch, ssd, dev, stream, peaks, steps):
    """The block around the scan on the 2.7B shape (d_inner 5120, 1 group,
    dstate 128): the causal depthwise conv1d (width 4, bias, SiLU) over the
    xBC slice of the input projection zxbcdt (a strided view), and the grouped
    RMSNorm of the gated out (in place); HBM roofline on each pass's bytes."""
    Bz, L, H, P, G, N, W = 8, 4096, 80, 64, 1, 128, 4
    di, cbc = H * P, H * P + 2 * G * N
    g = torch.Generator(device=dev).manual_seed(95)
    zxbcdt = torch.randn(Bz, L, 2 * di + 2 * G * N + H, generator=g, device=dev).bfloat16()
    xbc = zxbcdt[:, :, di:di + cbc]
    wconv = torch.randn(cbc, W, generator=g, device=dev) * 0.5
    bconv = torch.randn(cbc, generator=g, device=dev) * 0.1
    conv_out = torch.empty(Bz, L, cbc, dtype=torch.bfloat16, device=dev)
    y = torch.randn(Bz, L, di, generator=g, device=dev).bfloat16()
    wnorm = torch.rand(di, generator=g, device=dev) + 0.5
    n = max(5, min(steps, 20))
    res = {}
    for name, step, nbytes in (
            ("conv1d", lambda: ssd.causal_conv1d(xbc, wconv, bconv, out=conv_out, stream=stream),
             2 * Bz * L * cbc * 2 + cbc * (W + 1) * 4),
            ("group_rmsnorm", lambda: ssd.group_rmsnorm_(y, wnorm, group_size=di // G,
                                                         stream=stream),
             2 * Bz * L * di * 2 + di * 4)):
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        ms, per = time_calls(torch, step, n, stream)
        ach = nbytes / (ms / 1e3) / 1e9
        res[name] = {"ms_per_call": ms, "per_call_ms": spread(per), "calls": n,
                     "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"],
                                  "unit": "GB/s", "frac": ach / peaks["hbm_gbs"],
                                  "alg_bytes_per_call": nbytes}}
    res["workload"] = (f"block around the scan: batch {Bz}, seqlen {L}, d_inner {di}, ngroups {G}, "
                       f"dstate {N}; conv1d width {W} + SiLU over the xBC slice of zxbcdt, "
                       "grouped RMSNorm of out in place")
    res["data"] = "synthetic, drawn on the device"
    return res


def main():
    args = parse_args()
    import ssd_inputs as si
    if args.workload in ("backward", "forward_fp32", "forward_bf16_hd128"):
        # the backward or a stage-kernel forward alone (for profiling it): its own line
        import torch
        import selective_state_space_05_gb300 as ssd
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        st0, pk = torch.cuda.current_stream(), load_peaks()
        if args.workload == "backward":
            res = backward_workload(torch, ssd, si, dev, st0, pk, args.steps, batch=args.batch)
            metric, dtype = "SSD scan backward (all gradients) tokens/s at 2.7B shape, fp32", "f32"
        elif args.workload == "forward_fp32":
            res = fp32_forward_workload(torch, ssd, si, dev, st0, pk, args.steps, batch=args.batch)
            metric, dtype = "SSD chunked-scan fwd tokens/s at 2.7B shape, fp32", "f32"
        else:
            res = fp32_forward_workload(torch, ssd, si, dev, st0, pk, args.steps, batch=args.batch,
                                        dtype="bf16", heads_dim=HD128)
            metric = "SSD chunked-scan fwd tokens/s at 2.7B width, headdim 128, bf16"
            dtype = "bf16"
        print(json.dumps({"metric": metric, **res, "n_gpus": 1, "higher_is_better": True,
                          "dtype": dtype}), flush=True)
        return
    cfg = si.CONFIGS[args.workload]
    if args.impl == "reference":
        run_reference(args, cfg)
        return

    import torch
    import torch.distributed as dist
    import selective_state_space_05_gb300 as ssd

    if args.workload in ("chained", "packed"):
        # one of the other workloads alone (for profiling it): its own line
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        res = other_workload(torch, ssd, si, args.workload, dev, torch.cuda.current_stream(),
                             load_peaks(), args.steps, args.warmup,
                             torch.cuda.get_device_properties(dev).multi_processor_count)
        print(json.dumps({"metric": METRIC, **res, "n_gpus": 1, "warmup": args.warmup,
                          "higher_is_better": True, "dtype": "bf16"}), flush=True)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = load_peaks()
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count

    host = si.make_inputs(cfg, 1002 + rank)
    g = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in host.items()}
    Q = cfg.chunk_size
    out = torch.empty_like(g["x"])
    fin = torch.empty(cfg.batch, cfg.nheads, cfg.headdim, cfg.dstate, dtype=torch.float32,
                      device=dev)
    ws = torch.empty(ssd.workspace_bytes(cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim,
                                         cfg.dstate, cfg.ngroups, Q, g["x"].dtype),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        ssd.ssd_scan_fwd(g["x"], g["dt"], g["A"], g["B"], g["C"], chunk_size=Q,
                         dt_bias=g["dt_bias"], D=g["D"], z=g["z"],
                         initial_states=g["initial_states"], seq_idx=g["seq_idx"],
                         out=out, final_states=fin, return_final_states=True, workspace=ws,
                         stream=stream)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(3):   # the sampler's start left the GPU idle: bring the clocks back up
        step()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    ms_local, per_call = time_calls(torch, step, args.steps, stream)
    barrier()
    # a second, seconds-long block of back-to-back calls (steadier clocks)
    long = None
    if args.long_seconds > 0:
        n_long = max(args.steps, int(args.long_seconds / (ms_local / 1e3)))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_long):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        long = {"calls": n_long, "ms_per_step": e0.elapsed_time(e1) / n_long}
    barrier()
    clk = clocks.stop()
    ssd.scan_status(reset=True, stream=stream)   # no launch gave up a bounded wait
    ms = max_over_ranks(ms_local, world, dev)
    tokens = cfg.tokens * world

    # per-kernel durations: the fused path is one kernel (all four stages),
    # timed by the per-call events above; the SIMT path is the four stage
    # kernels, timed with events between them
    fused = (cfg.dtype == "bf16" and cfg.headdim == 64 and cfg.dstate == 128
             and Q in (128, 256) and (cfg.nheads // cfg.ngroups) % 2 == 0)
    if fused:
        per = {"scan_fused": statistics.mean(per_call)}
    else:
        names = ["dt_cumsum", "chunk_state", "state_passing", "chunk_scan"]
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)]
               for _ in range(args.steps)]
        for k in range(args.steps):
            e = evs[k]
            e[0].record(stream)
            dto, cso, sego = ssd.ssd_dt_cumsum(g["dt"], g["A"], chunk_size=Q,
                                               dt_bias=g["dt_bias"], seq_idx=g["seq_idx"],
                                               stream=stream)
            e[1].record(stream)
            st2 = ssd.ssd_chunk_state(g["x"], g["B"], dto, cso, sego, chunk_size=Q,
                                      stream=stream)
            e[2].record(stream)
            ssd.ssd_state_passing(st2, cso, sego, seqlen=cfg.seqlen, chunk_size=Q,
                                  initial_states=g["initial_states"], stream=stream)
            e[3].record(stream)
            ssd.ssd_chunk_scan(g["x"], g["B"], g["C"], dto, cso, sego, st2, chunk_size=Q,
                               D=g["D"], z=g["z"], out=out, stream=stream)
            e[4].record(stream)
            del st2, dto, cso, sego
        torch.cuda.synchronize()
        per = {n: statistics.mean(evs[k][i].elapsed_time(evs[k][i + 1])
                                  for k in range(args.steps))
               for i, n in enumerate(names)}
    has_init = g["initial_states"] is not None
    has_seq = g["seq_idx"] is not None
    models = kernel_models(cfg, peaks, num_sms, init=has_init, final=True, seq=has_seq)
    top = max(per, key=per.get)
    mdl = models[top]
    dur_s = per[top] / 1e3
    if mdl["bound"] == "hbm":
        achieved, peak, unit = mdl["bytes"] / dur_s / 1e9, peaks["hbm_gbs"], "GB/s"
    else:
        achieved, peak, unit = mdl["flops"] / dur_s / 1e12, mdl["peak"] / 1e12, "TFLOP/s"
    extra = {}
    if "tensor_peak" in mdl:
        extra["tensor_tflops"] = mdl["flops"] / dur_s / 1e12
        extra["tensor_frac"] = mdl["flops"] / dur_s / mdl["tensor_peak"]
    a = algorithmic(cfg, init=has_init, final=True, seq=has_seq)
    a_io = algorithmic(cfg, init=has_init, final=False, seq=has_seq)
    roofline = {"kernel": top, "bound": mdl["bound"], "achieved": achieved, "peak": peak,
                **extra,
                "unit": unit, "frac": achieved / peak,
                "frac_without_final_states": (a_io["io_bytes"] / dur_s / 1e9 / peak
                                              if mdl["bound"] == "hbm" else None),
                "traffic": measured_traffic(top, cfg.name),
                "alg_bytes": mdl["bytes"], "alg_flops": mdl["flops"],
                "alg_bytes_note": "x, z, out, B, C, dt, A, D, dt_bias and the final states "
                                  "the step writes",
                "peak_source": peaks.get("source"),
                "kernel_ms": {n: round(v, 4) for n, v in per.items()},
                "share": {n: round(v / sum(per.values()), 4) for n, v in per.items()}}
    whole = {"alg_bytes": a["io_bytes"], "alg_flops": a["flops"],
             "hbm_time_us": a["io_bytes"] / (peaks["hbm_gbs"] * 1e9) * 1e6,
             "frac_of_hbm_roofline": (a["io_bytes"] / (peaks["hbm_gbs"] * 1e9)) / (ms / 1e3)}
    timing = {"per_call_ms": spread(per_call)}
    if long is not None:
        timing["ms_per_step_long"] = long["ms_per_step"]
        timing["calls_long"] = long["calls"]
    if clk.get("sm_mhz"):
        timing["kcycles_per_call_at_median_sm_clock"] = ms * clk["sm_mhz"]   # ms x MHz = kcycles
        if long is not None:
            timing["kcycles_per_call_long"] = long["ms_per_step"] * clk["sm_mhz"]

    # end to end through ssd_scan_fwd_host: the inputs live in pinned host
    # memory and the output goes back to it, every step (the library pipelines
    # the copies with the scan over batch slices)
    e2e = None
    if not args.no_e2e:
        hin = {k: host[k].contiguous().pin_memory() for k in ("x", "dt", "B", "C", "z")}
        hsmall = {k: (host[k].contiguous() if torch.is_tensor(host[k]) else None)
                  for k in ("A", "dt_bias", "D", "initial_states", "seq_idx")}
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in list(hin.values()) + list(hsmall.values())
                  if v is not None)
        d2h = hout.numel() * hout.element_size()
        hws = torch.empty(ssd.host_workspace_bytes(cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim,
                                                   cfg.dstate, cfg.ngroups, Q, g["x"].dtype),
                          dtype=torch.uint8, device=dev)

        def e2e_step():
            ssd.ssd_scan_fwd_host(hin["x"], hin["dt"], hsmall["A"], hin["B"], hin["C"],
                                  chunk_size=Q, dt_bias=hsmall["dt_bias"], D=hsmall["D"],
                                  z=hin["z"], initial_states=hsmall["initial_states"],
                                  seq_idx=hsmall["seq_idx"], out=hout, workspace=hws,
                                  stream=stream, synchronize=False)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier()
        ems_local, eper = time_calls(torch, e2e_step, args.steps, stream)
        barrier()
        ems = max_over_ranks(ems_local, world, dev)
        e2e = {"value": tokens / (ems / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ems, "per_call_ms": spread(eper)}
        del hws, hin, hout

    others = None
    if not args.no_other and world == 1 and args.workload == WORKLOAD:
        others = {}
        for name in ("chained", "packed"):
            others[name] = other_workload(torch, ssd, si, name, dev, stream, peaks, args.steps,
                                          args.warmup, num_sms)
        others["decode"] = decode_workload(torch, ssd, si, dev, stream, peaks, args.steps)
        others["forward_fp32"] = fp32_forward_workload(torch, ssd, si, dev, stream, peaks,
                                                       args.steps)
        others["forward_bf16_hd128"] = fp32_forward_workload(
            torch, ssd, si, dev, stream, peaks, args.steps, dtype="bf16", heads_dim=HD128)
        others["backward"] = backward_workload(torch, ssd, si, dev, stream, peaks, args.steps)
        others["block"] = block_workload(torch, ssd, dev, stream, peaks, args.steps)

    cpu = parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        s = oracle_sample(cfg, host, args.cpu_seconds)
        cpu = {"value": s["rate"], "unit": UNIT, "cores": s["cores"], "kind": "oracle",
               "sample": s["desc"], "cpu": cpu_model()}
        # the GPU output of the timed calls (same inputs) against the sample
        yg, fg = out.cpu(), fin.cpu()
        hs = s["heads"]
        pieces_y = [(yg[b:b + 1][:, :, hs].double().numpy(), s["y"][i:i + 1])
                    for i, b in enumerate(s["batches"])]
        pieces_f = [(fg[b:b + 1][:, hs].double().numpy(), s["fin"][i:i + 1])
                    for i, b in enumerate(s["batches"])]
        parity = {"out": error_metrics(pieces_y), "final_states": error_metrics(pieces_f),
                  "tol": 2e-2 if cfg.dtype == "bf16" else 1e-4,
                  "pairs": len(s["batches"]) * len(hs),
                  "against": "fp64 oracle on the cpu_baseline sample"}
        parity["pass"] = (parity["out"]["max_rel"] <= parity["tol"]
                          and parity["final_states"]["max_rel"] <= parity["tol"])

    if rank == 0:
        line = bench_line(cfg, world, args.steps, args.warmup, ms,
                          {"roofline": roofline, "whole_call": whole, "timing": timing,
                           "cpu_baseline": cpu, "parity": parity, "e2e": e2e,
                           "other_configs": others,
                           "gpu_launches": (1 if fused else 4) * args.steps,
                           "clocks": clk})
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

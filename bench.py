#!/usr/bin/env python
"""Benchmark of the SSD chunked-scan forward on the Mamba-2 2.7B shape.

Workload: batch 8, seqlen 4096, 80 heads, headdim 64 (d_inner 5120), dstate
128, 1 group, chunk 256, bf16 inputs, fp32 states, z gate and D skip on;
synthetic seeded inputs (ssd_inputs.py).  One step = one ssd_scan_fwd call
over the whole batch (all four stages).

Prints ONE JSON line (rank 0).  `value` is whole-job tokens/s with inputs
resident in HBM; `e2e` is the same metric with the host->device copy of the
inputs and the device->host copy of the output inside the timed region.
`roofline` rates the kernel that takes most of the step against the measured
peaks in MEASURED_PEAKS.json.  `cpu_baseline` times the fp64 CPU oracle on a
bounded sample of the same workload.

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
UNIT = "tokens/s"
WORKLOAD = "mamba2_2p7b"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0, "source": "fallback"}
NUM_SMS = 152
FP32_LANES_PER_SM = 128


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle sample")
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

def algorithmic(cfg) -> dict:
    e = 2 if cfg.dtype == "bf16" else 4
    Bz, L, H, P, N, G, Q = (cfg.batch, cfg.seqlen, cfg.nheads, cfg.headdim, cfg.dstate,
                            cfg.ngroups, cfg.chunk_size)
    nc = -(-L // Q)
    x = Bz * L * H * P * e
    bc = Bz * L * G * N * e
    dt = Bz * L * H * e
    state = Bz * nc * H * P * N * 4
    chunk_f32 = Bz * H * nc * Q * 4
    io = 3 * x + 2 * bc + dt + 3 * H * 4          # x, z, out, B, C, dt, (A, D, dt_bias)
    tri = Q * (Q + 1) // 2
    # causal flops: C B^T once per group, masked (CB) x and C h per head, B^T x per head
    flops = Bz * nc * (G * tri * N * 2 + H * (tri * P * 2 + 2 * Q * N * P * 2))
    return dict(io_bytes=io, flops=flops, x=x, bc=bc, dt=dt, state=state, chunk_f32=chunk_f32,
                tri=tri, nc=nc)


def kernel_models(cfg, peaks) -> dict:
    """Per-kernel algorithmic bytes / flops and the roofline that bounds it."""
    a = algorithmic(cfg)
    Bz, H, P, N, G, Q, nc = (cfg.batch, cfg.nheads, cfg.headdim, cfg.dstate, cfg.ngroups,
                             cfg.chunk_size, a["nc"])
    hbm = peaks["hbm_gbs"] * 1e9
    alu = NUM_SMS * FP32_LANES_PER_SM * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6
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

def oracle_sample_rate(cfg, inputs, target_s: float, seed_heads=0):
    """Times the fp64 oracle on a sample of (batch row, head) recurrences sized
    to about target_s seconds; returns (tokens/s equivalent, cores,
    description, seconds).  A token-equivalent is one token through all heads."""
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
    so.scan_sequential(inputs, heads=heads, batches=batches, nthreads=cores)
    dt = time.perf_counter() - t
    nh = H if heads is None else len(heads)
    tokens_equiv = L * len(batches) * nh / H
    desc = (f"fp64 sequential oracle on {len(batches)} batch row(s) x {nh} of {H} "
            f"heads, seqlen {L}: {tokens_equiv:.0f} token-equivalents (one token through "
            f"all heads) in {dt:.2f} s")
    return tokens_equiv / dt, cores, desc, dt


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
        "config": {"workload": f"{cfg.name}: batch {cfg.batch}, seqlen {cfg.seqlen}, "
                               f"nheads {cfg.nheads}, headdim {cfg.headdim}, dstate "
                               f"{cfg.dstate}, ngroups {cfg.ngroups}, chunk "
                               f"{cfg.chunk_size}, z gate + D skip, fp32 state",
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
        r, cores, desc, _ = oracle_sample_rate(cfg, inputs, per_step, seed_heads=i)
        if i >= args.warmup:
            rates.append(r)
    value = statistics.median(rates)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * cfg.tokens / value, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{cfg.name}: batch {cfg.batch}, seqlen {cfg.seqlen}, "
                               f"nheads {cfg.nheads}, headdim {cfg.headdim}, dstate "
                               f"{cfg.dstate}, ngroups {cfg.ngroups}, chunk {cfg.chunk_size}",
                   "sample": desc},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc, "cpu": cpu_model()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    import ssd_inputs as si
    cfg = si.CONFIGS[args.workload]
    if args.impl == "reference":
        run_reference(args, cfg)
        return

    import torch
    import torch.distributed as dist
    import selective_state_space_05_gb300 as ssd

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = load_peaks()

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
    barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = max_over_ranks(t0.elapsed_time(t1) / args.steps, world, dev)
    tokens = cfg.tokens * world

    # per-kernel durations, with events between the launches: the fused path
    # is one kernel (all four stages); the SIMT path is the four stage kernels
    fused = (cfg.dtype == "bf16" and cfg.headdim == 64 and cfg.dstate == 128
             and Q in (128, 256) and (cfg.nheads // cfg.ngroups) % 2 == 0)
    names = (["scan_fused"] if fused else
             ["dt_cumsum", "chunk_state", "state_passing", "chunk_scan"])
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
           for _ in range(args.steps)]
    for k in range(args.steps):
        e = evs[k]
        e[0].record(stream)
        if fused:
            step()
            e[1].record(stream)
            continue
        dto, cso, sego = ssd.ssd_dt_cumsum(g["dt"], g["A"], chunk_size=Q, dt_bias=g["dt_bias"],
                                           seq_idx=g["seq_idx"], stream=stream)
        e[1].record(stream)
        st2 = ssd.ssd_chunk_state(g["x"], g["B"], dto, cso, sego, chunk_size=Q, stream=stream)
        e[2].record(stream)
        ssd.ssd_state_passing(st2, cso, sego, seqlen=cfg.seqlen, chunk_size=Q,
                              initial_states=g["initial_states"], stream=stream)
        e[3].record(stream)
        ssd.ssd_chunk_scan(g["x"], g["B"], g["C"], dto, cso, sego, st2, chunk_size=Q,
                           D=g["D"], z=g["z"], out=out, stream=stream)
        e[4].record(stream)
        del st2, dto, cso, sego
    torch.cuda.synchronize()
    per = {n: statistics.mean(evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(args.steps))
           for i, n in enumerate(names)}
    models = kernel_models(cfg, peaks)
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
    roofline = {"kernel": top, "bound": mdl["bound"], "achieved": achieved, "peak": peak,
                **extra,
                "unit": unit, "frac": achieved / peak,
                "traffic": measured_traffic(top, cfg.name),
                "alg_bytes": mdl["bytes"], "alg_flops": mdl["flops"],
                "peak_source": peaks.get("source"),
                "kernel_ms": {n: round(v, 4) for n, v in per.items()},
                "share": {n: round(v / sum(per.values()), 4) for n, v in per.items()}}
    a = algorithmic(cfg)
    whole = {"alg_bytes": a["io_bytes"], "alg_flops": a["flops"],
             "hbm_time_us": a["io_bytes"] / (peaks["hbm_gbs"] * 1e9) * 1e6,
             "frac_of_hbm_roofline": (a["io_bytes"] / (peaks["hbm_gbs"] * 1e9)) / (ms / 1e3)}

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
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        s1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ems = max_over_ranks(s0.elapsed_time(s1) / args.steps, world, dev)
        e2e = {"value": tokens / (ems / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ems}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r, cores, desc, _ = oracle_sample_rate(cfg, host, args.cpu_seconds)
        cpu = {"value": r, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc,
               "cpu": cpu_model()}

    if rank == 0:
        line = bench_line(cfg, world, args.steps, args.warmup, ms,
                          {"roofline": roofline, "whole_call": whole, "cpu_baseline": cpu,
                           "e2e": e2e, "gpu_launches": (1 if fused else 4) * args.steps,
                           "clocks": clk})
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""SSM-layer decode benchmark of librs on GB300.

A step is one standard decode step of the whole batch through the C ABI:
append the step's record, replay the buffer against the checkpoint for the
output, and (every L steps) fold the window into the checkpoint.  Workload:
Mamba-2 layer, B=256 sequences, 128 heads, headdim 64, dstate 128, 8 B/C
groups, window L=16, fp32 checkpoint (4 MiB per sequence), seeded synthetic
inputs.  The timed region covers whole windows, so flushes are amortised.

Prints one JSON line: decode tokens/s (whole job), achieved HBM GB/s of the
replay kernel against the measured peak, the eager load-update-store kernel
on the same workload, an end-to-end number through host buffers, the fp64
CPU oracle on a bounded sample, and the SM clocks seen while timing.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]
Under torchrun every rank runs its own B sequences (weak scaling, no
collective on the data path); rank 0 prints the max-over-ranks timing.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SSM-layer decode tokens/s at B=256, L=16 (1 GB300); achieved HBM GB/s vs peak"
WORKLOAD = "mamba2"
INPUT_POOL = 256  # distinct seeded input steps, cycled through the timed region


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2048)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", default="librs", choices=["librs", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-eager", action="store_true")
    ap.add_argument("--batch", type=int, default=0,
                    help="sequences per GPU (default: the workload's 256; smaller only for profiling)")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), ws, int(os.environ.get("LOCAL_RANK", "0"))


def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in ("rs_replay.cu", "rs_common.cuh"):
        with open(os.path.join(ROOT, "rs_decode_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic() -> float | None:
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (its source hash matches)."""
    path = os.path.join(ROOT, "profiles", "replay_mamba2_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except OSError:
        return None
    if rec.get("source_hash") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_launch_full_size")


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.seek(0)
        rows = [r.split(", ") for r in self.tmp.read().strip().splitlines() if r.count(",") >= 9]
        os.unlink(self.tmp.name)
        return rows

    @staticmethod
    def summarise(rows, t0: float, t1: float) -> dict | None:
        if not rows:
            return None
        import datetime
        sel = []
        for r in rows:
            try:
                ts = datetime.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            if t0 - 0.06 <= ts <= t1 + 0.06:
                sel.append(r)
        sel = sel or rows[-3:]
        sm = [float(r[2]) for r in sel if r[2].strip().replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in sel:
            for n, v in zip(names, r[6:10]):
                if v.strip() == "Active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(sel[0][3]) if sel[0][3].strip().replace(".", "").isdigit() else None,
                "reasons": sorted(reasons), "samples": len(sel),
                "power_w_max": max(float(r[4]) for r in sel if r[4].strip().replace(".", "").isdigit())}


# ----------------------------------------------------------------------------- ranks
def max_over_ranks(x: float, device=None) -> float:
    """Largest value over all ranks (the job's time is its slowest rank's).
    Without an initialised process group this is x itself."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    if device is None or dist.get_backend() == "gloo":
        device = torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(rank: int) -> int:
    """Each rank decodes its own, independently seeded sequences (weak scaling)."""
    return rank


# ----------------------------------------------------------------------------- CPU oracle
def time_oracle(w, seconds: float, batch: int = 16):
    """fp64 oracle on the host cores: batch sequences of the workload, as many
    steps as fit in ``seconds`` (at least one).  Returns tokens/s and details."""
    import oracle
    from rs_decode_gb300 import synth
    ws = w.with_(B=batch)
    params = synth.layer_params(ws)
    model = oracle.Model(ws.kind, synth.initial_state(ws), params)
    inputs = [synth.step_inputs(ws, s, params=params) for s in range(4)]
    steps, t0 = 0, time.perf_counter()
    while True:
        model.step(inputs[steps % len(inputs)])
        steps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": batch * steps / el, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{batch} sequences x {steps} decode steps of the {w.name} workload "
                      f"(H={w.H}, P={w.P}, N={w.N}), fp64 eager recurrence, {el:.1f} s"}


# ----------------------------------------------------------------------------- main arm
def run_librs(args, rank: int, world: int, local_rank: int) -> dict | None:
    import torch
    import torch.distributed as dist

    from rs_decode_gb300 import binding as rb
    from rs_decode_gb300 import synth, traffic
    from rs_decode_gb300.layer import Layer, to_device

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = synth.WORKLOADS[WORKLOAD]
    if args.batch:
        w = w.with_(B=args.batch)
    K, W = args.steps, args.warmup
    params = synth.layer_params(w)
    gp = {"A": torch.from_numpy(params["A"]).to(dev), "D": torch.from_numpy(params["D"]).to(dev)}
    npool = min(INPUT_POOL, K + W)
    host_steps = [synth.step_inputs(w, s, seed=rank_seed(rank), params=params) for s in range(npool)]
    dev_steps = [to_device(d, dev) for d in host_steps]

    layer = Layer("mamba2", w.B, w.H, w.G, w.P, w.N, w.L)
    g = torch.Generator(device=dev).manual_seed(1000 + rank)
    S0 = torch.randn(layer.shape, generator=g, device=dev, dtype=torch.float32).mul_(w.init_std)
    layer.init(S0)
    y = torch.empty(w.B, w.H, w.P, device=dev)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()

    # ---- replay path, device-resident inputs
    for s in range(W):
        layer.decode(dev_steps[s % npool], gp, y)
    torch.cuda.synchronize()
    h0 = int(layer.h[0].item())
    clocks = ClockSampler(local_rank)
    clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start.record(stream)
    for s in range(K):
        ev[s][0].record(stream)
        layer.decode(dev_steps[(W + s) % npool], gp, y)
        ev[s][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier()
    rows = clocks.stop()
    ms_total = start.elapsed_time(end)
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    if layer.status() != 0:
        raise RuntimeError("device status bits set during the benchmark")

    # algorithmic bytes of the timed launches (pointer schedule is lockstep)
    shape = traffic.Shape("mamba2", w.B, w.H, w.G, w.P, w.N)
    total_bytes, h = 0, h0
    for _ in range(K):
        flush = h + 1 >= w.L
        total_bytes += traffic.replay_step_bytes(shape, h, flush)
        h = 0 if flush else h + 1

    # ---- eager baseline on the same workload
    ms_eager = None
    if not args.no_eager:
        S_eager = S0.clone()
        desc = layer.desc
        Ke = min(K, 512)
        def eager(s):
            d = dev_steps[s % npool]
            rb.rs_eager_step_mamba2(desc, S_eager, d["x"], d["dt"], gp["A"], d["Bm"], d["Cm"], gp["D"], y)
        for s in range(W):
            eager(s)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for s in range(Ke):
            eager(W + s)
        e1.record(stream)
        torch.cuda.synchronize()
        ms_eager = e0.elapsed_time(e1) / Ke
        del S_eager

    # ---- end to end through host buffers (pinned), copies inside the timed region
    e2e = None
    if not args.no_e2e:
        pinned = [{k: v.pin_memory() for k, v in to_device(d, "cpu").items()} for d in host_steps[:64]]
        stage = {k: torch.empty_like(v, device=dev) for k, v in pinned[0].items()}
        y_host = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
        bi = sum(v.numel() * v.element_size() for v in pinned[0].values())
        bo = y.numel() * y.element_size()
        Kx = min(K, 512)
        def e2e_step(s):
            for k, v in pinned[s % len(pinned)].items():
                stage[k].copy_(v, non_blocking=True)
            layer.decode(stage, gp, y)
            y_host.copy_(y, non_blocking=True)
        for s in range(W):
            e2e_step(s)
        torch.cuda.synchronize()
        x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        x0.record(stream)
        for s in range(Kx):
            e2e_step(s)
        x1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ms_x = x0.elapsed_time(x1) / Kx
        e2e = {"value": w.B * world / (ms_x * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": bi,
               "d2h_bytes_per_step": bo, "ms_per_step": ms_x}

    # ---- max over ranks
    ms_total = max_over_ranks(ms_total, dev)
    if rank != 0:
        return None

    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = peak or 6800.0
    avg_launch_s = statistics.fmean(launch_ms) * 1e-3
    achieved = total_bytes / K / avg_launch_s / 1e9
    eager_bytes = traffic.eager_step_bytes(shape)
    clk = ClockSampler.summarise(rows, t_wall0, t_wall1)
    out = {
        "metric": METRIC,
        "value": w.B * K * world / (ms_total * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": ms_total / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": f"mamba2 decode B={w.B} H={w.H} P={w.P} N={w.N} G={w.G} L={w.L} fp32 checkpoint",
                   "B_per_gpu": w.B, "window_L": w.L, "state_mib_per_seq": w.H * w.N * w.P * 4 / 2**20,
                   "parallelism": f"dp{world}" if world > 1 else "single",
                   "l2": "inputs larger than L2 (1 GiB checkpoint per step)",
                   "inputs": f"{npool} distinct seeded steps cycled"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": profiled_traffic(),
                     "peak_source": f"{peak_src} (copy bandwidth)",
                     "algorithmic_bytes_per_launch": total_bytes / K,
                     "kernel": "replay_kernel<mamba2,64,128,HPC=2,TMAX=1,256>"},
        "hbm_gbs": achieved,
        "eager": None if ms_eager is None else {
            "ms_per_step": ms_eager, "value": w.B / (ms_eager * 1e-3), "unit": "tokens/s",
            "achieved_gbs": eager_bytes / (ms_eager * 1e-3) / 1e9,
            "bytes_per_step": eager_bytes, "speedup_of_replay": ms_eager / (ms_total / K)},
        "gpu_launches": K,
        "clocks": clk,
        "e2e": e2e,
    }
    return out


def main():
    args = parse()
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return 0
        from rs_decode_gb300 import synth
        w = synth.WORKLOADS[WORKLOAD]
        ref = time_oracle(w, max(2.0, args.cpu_seconds))
        line = {"impl": "reference", "metric": METRIC, "value": ref["value"], "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": f"mamba2 decode B={w.B} H={w.H} P={w.P} N={w.N} G={w.G} L={w.L}"},
                "cpu_baseline": ref,
                "e2e": {"value": ref["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    out = run_librs(args, rank, world, local_rank)
    if out is not None:
        if not args.no_cpu_baseline and world == 1:
            from rs_decode_gb300 import synth
            out["cpu_baseline"] = time_oracle(synth.WORKLOADS[WORKLOAD], args.cpu_seconds)
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

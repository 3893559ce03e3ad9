#!/usr/bin/env python
"""SSM-layer decode benchmark of librs on GB300.

A step is one standard decode step of the whole batch through the C ABI:
append the step's record, replay the buffer against the checkpoint for the
output, and (every L steps) fold the window into the checkpoint.  Headline
workload: Mamba-2 layer, B=256 sequences, 128 heads, headdim 64, dstate 128,
8 B/C groups, window L=16, fp32 checkpoint (4 MiB per sequence), seeded
synthetic inputs.  The timed region starts at a window boundary (h = 0); with
K a multiple of L (the default, 2048) it covers whole windows, and the line
also gives the window-weighted step (one folding launch and L - 1 streaming
ones), so that flushes are amortised either way.

Prints one JSON line: decode tokens/s (whole job), achieved HBM GB/s of the
replay kernel against the measured peak, the eager load-update-store kernel
on the same workload, an end-to-end number through host buffers, the fp64
CPU oracle on a bounded sample, the SM clocks seen while timing, and (unless
--headline-only) the other workloads: GDN decode, decode with one decay per
key channel, Mamba-2 speculative verification, two-precision GDN speculative
verification, each against its baseline kernel.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]
Under torchrun every rank runs its own B sequences (weak scaling, no
collective on the data path); rank 0 prints the max-over-ranks timing.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SSM-layer decode tokens/s at B=256, L=16 (1 GB300); achieved HBM GB/s vs peak"
INPUT_POOL = 256  # distinct seeded input steps, cycled through the timed region


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2048)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", default="librs", choices=["librs", "reference"])
    ap.add_argument("--workload", default="mamba2", choices=["mamba2", "gdn", "kda"],
                    help="decode workload of the headline line")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-eager", action="store_true")
    ap.add_argument("--headline-only", action="store_true", help="skip the other workloads")
    ap.add_argument("--spec", default="", choices=["", "mamba2_spec", "gdn_spec"],
                    help="time only this speculative workload (verify + commit rounds) and print its line")
    ap.add_argument("--rounds", type=int, default=64)
    ap.add_argument("--sweep", action="store_true",
                    help="print one JSON line per point of the window / batch / draft-count sweeps instead")
    ap.add_argument("--batch", type=int, default=0,
                    help="sequences per GPU (default: the workload's 256; smaller only for profiling)")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), ws, int(os.environ.get("LOCAL_RANK", "0"))


NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal


def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {}


def _code_only(text: str) -> str:
    """The source with comments and blank lines removed: what the compiler sees
    (a comment edit does not change the kernel the traffic was measured on)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln.strip())


# The sources each workload's replay kernel is built from (the launch entry,
# the planning and device helpers, the pipeline, the family's translation unit).
KERNEL_SOURCES = {
    "mamba2": ("rs_internal.h", "rs_common.cuh", "rs_plan.cuh", "rs_replay_rows.cuh", "rs_replay.cu", "rs_replay_m2.cu"),
    "gdn": ("rs_internal.h", "rs_common.cuh", "rs_plan.cuh", "rs_replay_cols.cuh", "rs_replay.cu", "rs_replay_gdn.cu"),
    "kda": ("rs_internal.h", "rs_common.cuh", "rs_plan.cuh", "rs_replay_cols.cuh", "rs_replay.cu", "rs_replay_kda.cu"),
}


def kernel_source_hash(workload: str) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[workload]:
        with open(os.path.join(ROOT, "rs_decode_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str) -> float | None:
    """DRAM bytes per launch (window average, full size) from the committed
    ncu summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", f"replay_{workload}_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except OSError:
        return None
    if rec.get("source_hash") != kernel_source_hash(workload):
        return None
    return rec.get("dram_bytes_per_launch")


def recorded_output_error() -> dict | None:
    """The two-precision and shared-bf16 output errors of the gdn_spec workload
    against the fp64 oracle, as the full-length parity test recorded them
    (profiles/gdn_spec_output_error.json), if taken on the current kernel
    source; else None.  The benchmark itself never runs the oracle on the GPU
    workloads."""
    path = os.path.join(ROOT, "profiles", "gdn_spec_output_error.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except OSError:
        return None
    if rec.get("source_hash") != kernel_source_hash("gdn"):
        return None
    return {k: rec[k] for k in ("workload", "two_precision", "shared_bf16", "slow_decay_variant", "metric", "sample",
                                "test") if k in rec}


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

    def stop(self):
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
        num = lambda v: v.strip().replace(".", "").isdigit()
        sm = [float(r[2]) for r in sel if num(r[2])]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in sel:
            for n, v in zip(names, r[6:10]):
                if v.strip() == "Active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(sel[0][3]) if num(sel[0][3]) else None,
                "reasons": sorted(reasons), "samples": len(sel),
                "power_w_max": max([float(r[4]) for r in sel if num(r[4])] or [0.0])}


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


def run_reference(w, K: int, W: int, budget_s: float = 120.0) -> dict:
    """The oracle as a benchmark arm: W untimed and K timed decode steps, each
    step one eager fp64 step of a bounded sample of the workload's sequences.
    The sample (16 sequences, halved while the whole run would exceed
    budget_s by a probe step's time) keeps the run within a few minutes."""
    import oracle
    from rs_decode_gb300 import synth

    def setup(batch):
        ws = w.with_(B=batch)
        params = synth.layer_params(ws)
        model = oracle.Model(ws.kind, synth.initial_state(ws), params)
        return model, [synth.step_inputs(ws, s, params=params) for s in range(4)]

    batch = 16
    model, inputs = setup(batch)
    t0 = time.perf_counter()
    model.step(inputs[0])
    probe = time.perf_counter() - t0
    while batch > 1 and probe * (K + W) > budget_s:
        batch //= 2
        probe /= 2
    model, inputs = setup(batch)
    for s in range(W):
        model.step(inputs[s % len(inputs)])
    t0 = time.perf_counter()
    for s in range(K):
        model.step(inputs[(W + s) % len(inputs)])
    el = time.perf_counter() - t0
    return {"value": batch * K / el, "unit": "tokens/s", "ms_per_step": el * 1e3 / K,
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{batch} sequences per step, {K} timed decode steps after {W} warm-up steps, of the "
                      f"{w.name} workload (H={w.H}, P={w.P}, N={w.N}), fp64 eager recurrence, {el:.1f} s"}


# ----------------------------------------------------------------------------- GPU helpers
def _events(n):
    import torch
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def _params(w, dev):
    import torch
    from rs_decode_gb300 import synth
    params = synth.layer_params(w)
    if w.kind == "mamba2":
        return params, {"A": torch.from_numpy(params["A"]).to(dev), "D": torch.from_numpy(params["D"]).to(dev)}
    return params, {}


def _init_state(layer, w, dev, seed):
    import torch
    g = torch.Generator(device=dev).manual_seed(1000 + seed)
    S0 = torch.randn(layer.shape, generator=g, device=dev, dtype=torch.float32).mul_(w.init_std)
    layer.init(S0)
    return S0


def measure_decode(w, K, W, dev, rank, world, want_eager=True, want_e2e=True, want_clocks=True):
    """Standard decode of workload w: K timed steps after W warm-up steps."""
    import torch
    import torch.distributed as dist

    from rs_decode_gb300 import binding as rb
    from rs_decode_gb300 import synth, traffic
    from rs_decode_gb300.layer import Layer, to_device

    params, gp = _params(w, dev)
    npool = min(INPUT_POOL, K + W)
    host_steps = [synth.step_inputs(w, s, seed=rank_seed(rank), params=params) for s in range(npool)]
    dev_steps = [to_device(d, dev) for d in host_steps]
    prec = rb.PRECISIONS[w.precision]
    layer = Layer(w.kind, w.B, w.H, w.G, w.P, w.N, w.L, capacity=w.cap, precision=prec)
    S0 = _init_state(layer, w, dev, rank)
    y = torch.empty(w.B, w.H, w.P, device=dev)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()

    # W warm-up steps, then more until the window restarts (h = 0), so that the
    # timed region begins with a whole window (the pointers move in lockstep)
    for s in range(W):
        layer.decode(dev_steps[s % npool], gp, y)
    torch.cuda.synchronize()
    extra = (w.L - int(layer.h[0].item())) % w.L
    for s in range(W, W + extra):
        layer.decode(dev_steps[s % npool], gp, y)
    torch.cuda.synchronize()
    W += extra
    h0 = int(layer.h[0].item())
    assert h0 == 0
    clocks = ClockSampler(dev.index or 0) if want_clocks else None
    if clocks:
        clocks.start()
    start, end = _events(2)
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start.record(stream)
    for s in range(K):
        layer.decode(dev_steps[(W + s) % npool], gp, y)
    end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier()
    rows = clocks.stop() if clocks else None
    ms_total = start.elapsed_time(end)

    # The folding / streaming split: K more launches after the timed region,
    # each between its own pair of events (recording them costs host time,
    # which would slow a host-bound small-batch loop if taken inside it).
    hs = int(layer.h[0].item())
    ev = list(zip(_events(K), _events(K)))
    for s in range(K):
        ev[s][0].record(stream)
        layer.decode(dev_steps[(W + K + s) % npool], gp, y)
        ev[s][1].record(stream)
    torch.cuda.synchronize()
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    if layer.status() != 0:
        raise RuntimeError("device status bits set during the benchmark")

    # algorithmic bytes of the launches (the pointer schedule is lockstep)
    shape = traffic.Shape(w.kind, w.B, w.H, w.G, w.P, w.N, u_bytes=2 if "u16" in w.precision else 4)
    two = w.precision.startswith("two")

    def launch_bytes(h):
        flush = h + 1 >= w.L
        rd = 4 if (flush or not two) else 2          # two-precision: bf16 copy off the flush steps
        wr = 6 if two else 4                          # a fold writes both copies
        return flush, traffic.replay_step_bytes(shape, h, flush, rd, wr)

    total_bytes, folds_timed, h = 0, 0, h0
    for s in range(K):  # the timed launches
        flush, nb = launch_bytes(h)
        total_bytes += nb
        folds_timed += flush
        h = 0 if flush else h + 1
    per_launch, h = [], hs  # (folds, bytes, ms) of every launch of the split pass
    for s in range(K):
        flush, nb = launch_bytes(h)
        per_launch.append((flush, nb, launch_ms[s]))
        h = 0 if flush else h + 1

    def split(fold):
        sel = [(b, t) for f, b, t in per_launch if f == fold]
        if not sel:
            return None
        ms = statistics.fmean(t for _, t in sel)
        nb = statistics.fmean(b for b, _ in sel)
        return {"launches": len(sel), "ms": ms, "bytes": nb, "achieved_gbs": nb / (ms * 1e-3) / 1e9}

    # the window-weighted step: one folding launch and L - 1 streaming ones
    fl, sl = split(True), split(False)
    ww = None
    if fl and sl:
        ww_ms = (fl["ms"] + (w.L - 1) * sl["ms"]) / w.L
        ww = {"ms_per_step": ww_ms, "value": w.B * world / (ww_ms * 1e-3), "unit": "tokens/s",
              "how": f"(1 folding + {w.L - 1} streaming launches) / {w.L}, from the per-launch events"}
    out = {"ms_total": ms_total, "ms_per_step": ms_total / K, "launch_ms": statistics.fmean(launch_ms),
           "bytes_per_launch": total_bytes / K, "clock_rows": rows, "t_wall": (t_wall0, t_wall1),
           "fold_launch": fl, "stream_launch": sl, "window_weighted": ww, "folds_timed": folds_timed,
           "eager": None, "e2e": None}

    if want_eager:
        S_e = S0.clone()
        desc = layer.desc
        Ke = min(K, 512)

        def eager(s):
            d = dev_steps[s % npool]
            if w.kind == "mamba2":
                rb.rs_eager_step_mamba2(desc, S_e, d["x"], d["dt"], gp["A"], d["Bm"], d["Cm"], gp["D"], y)
            else:
                fn = rb.rs_eager_step_gdn if w.kind == "gdn" else rb.rs_eager_step_kda
                fn(desc, S_e, d["q"], d["k"], d["v"], d["alpha"], d["beta"], y)
        for s in range(W):
            eager(s)
        torch.cuda.synchronize()
        e0, e1 = _events(2)
        e0.record(stream)
        for s in range(Ke):
            eager(W + s)
        e1.record(stream)
        torch.cuda.synchronize()
        ms_e = e0.elapsed_time(e1) / Ke
        eb = traffic.eager_step_bytes(shape)
        out["eager"] = {"ms_per_step": ms_e, "value": w.B / (ms_e * 1e-3), "unit": "tokens/s",
                        "achieved_gbs": eb / (ms_e * 1e-3) / 1e9, "bytes_per_step": eb,
                        "speedup_of_replay": ms_e / (ms_total / K)}
        del S_e

    if want_e2e:
        # End to end through the public API: every step uploads its inputs from
        # pinned host memory and reads its output back.  The uploads run on one
        # copy stream and the read-backs on another, double-buffered, so that
        # step s+1's upload and step s-1's read-back overlap step s's kernel.
        pinned = [{k: v.pin_memory() for k, v in to_device(d, "cpu").items()} for d in host_steps[:64]]
        stage = [{k: torch.empty_like(v, device=dev) for k, v in pinned[0].items()} for _ in range(2)]
        ybuf = [torch.empty_like(y) for _ in range(2)]
        y_host = [torch.empty(y.shape, dtype=y.dtype, pin_memory=True) for _ in range(4)]
        bi = sum(v.numel() * v.element_size() for v in pinned[0].values())
        bo = y.numel() * y.element_size()
        Kx = min(K, 512)
        up_s, dn_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

        def run_e2e(n):
            up = [torch.cuda.Event() for _ in range(n)]
            done = [torch.cuda.Event() for _ in range(n)]
            dn = [torch.cuda.Event() for _ in range(n)]
            for s in range(n):
                k = s % 2
                with torch.cuda.stream(up_s):
                    if s >= 2:
                        up_s.wait_event(done[s - 2])          # stage[k] no longer read
                    for key, v in pinned[s % len(pinned)].items():
                        stage[k][key].copy_(v, non_blocking=True)
                    up[s].record(up_s)
                stream.wait_event(up[s])
                if s >= 2:
                    stream.wait_event(dn[s - 2])              # ybuf[k] read back
                layer.decode(stage[k], gp, ybuf[k])
                done[s].record(stream)
                with torch.cuda.stream(dn_s):
                    dn_s.wait_event(done[s])
                    y_host[s % 4].copy_(ybuf[k], non_blocking=True)
                    dn[s].record(dn_s)
            stream.wait_stream(up_s)
            stream.wait_stream(dn_s)

        run_e2e(max(W, 4))
        torch.cuda.synchronize()
        x0, x1 = _events(2)
        barrier()
        x0.record(stream)
        up_s.wait_stream(stream)
        dn_s.wait_stream(stream)
        run_e2e(Kx)
        x1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ms_x = max_over_ranks(x0.elapsed_time(x1) / Kx, dev)
        out["e2e"] = {"value": w.B * world / (ms_x * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": bi,
                      "d2h_bytes_per_step": bo, "ms_per_step": ms_x,
                      "copies": "inputs uploaded and outputs read back on two copy streams, overlapped with the kernels"}
    del layer
    torch.cuda.empty_cache()
    return out


def measure_spec(w, rounds, W, dev, rank):
    """Speculative rounds of workload w (verify T drafts + commit) against the
    per-draft snapshot baseline; committed and verified tokens/s and GB/s."""
    import torch

    from rs_decode_gb300 import binding as rb
    from rs_decode_gb300 import synth, traffic
    from rs_decode_gb300.layer import Layer, to_device

    params, gp = _params(w, dev)
    npool = 32
    host = [synth.round_inputs(w, r, seed=rank_seed(rank), params=params) for r in range(npool)]
    dev_rounds = [to_device(d, dev) for d in host]
    prec = rb.PRECISIONS[w.precision]
    layer = Layer(w.kind, w.B, w.H, w.G, w.P, w.N, w.L, T_max=w.T, capacity=w.cap, precision=prec)
    y = torch.empty(w.B, w.T, w.H, w.P, device=dev)
    stream = torch.cuda.current_stream()

    def round_(r):
        d = dev_rounds[r % npool]
        layer.verify(w.T, d, gp, y)
        layer.commit(d["accepted"])

    # accounting pass: the committed counts before every round (the trajectory
    # is deterministic, so the timed pass repeats it exactly)
    S0 = _init_state(layer, w, dev, rank)
    h_before = []
    for r in range(W + rounds):
        h_before.append(layer.h.cpu().numpy().copy())
        round_(r)
    layer.init(S0)
    for r in range(W):
        round_(r)
    torch.cuda.synchronize()
    e0, e1 = _events(2)
    e0.record(stream)
    for r in range(W, W + rounds):
        round_(r)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / rounds
    if layer.status() != 0:
        raise RuntimeError("device status bits set during the speculative benchmark")
    shape = traffic.Shape(w.kind, w.B, w.H, w.G, w.P, w.N, u_bytes=2 if "u16" in w.precision else 4)
    two = w.precision.startswith("two")
    tot_bytes, folds, committed = 0, 0, 0
    for r in range(W, W + rounds):
        for hb in h_before[r]:
            fold = traffic.spec_folds(int(hb), w.T, w.L)
            folds += fold
            rd = 4 if (fold or not two) else 2
            wr = (6 if two else 4) if fold else 0
            tot_bytes += traffic.verify_round_bytes(shape, w.T, int(hb), fold, rd, wr)
        committed += int(host[r % npool]["accepted"].sum())
    # baseline: per-draft snapshots (one state read + T state writes per round)
    desc = layer.desc
    del layer
    torch.cuda.empty_cache()
    pool = torch.empty(w.B, w.T + 1, w.H, w.N, w.P, device=dev)
    pool[:, 0].copy_(S0)
    del S0
    cur = torch.zeros(w.B, dtype=torch.int32, device=dev)

    def snap(r):
        d = dev_rounds[r % npool]
        ins = (rb.make_inputs(x=d["x"], dt=d["dt"], A=gp["A"], Bm=d["Bm"], Cm=d["Cm"], D=gp["D"])
               if w.kind == "mamba2" else
               rb.make_inputs(q=d["q"], k=d["k"], v=d["v"], alpha=d["alpha"], beta=d["beta"]))
        rb.rs_eager_verify_snapshots(desc, pool, cur, w.T, ins, y)
        rb.rs_eager_select(desc, cur, d["accepted"])
    for r in range(W):
        snap(r)
    torch.cuda.synchronize()
    b0, b1 = _events(2)
    b0.record(stream)
    for r in range(W, W + rounds):
        snap(r)
    b1.record(stream)
    torch.cuda.synchronize()
    ms_b = b0.elapsed_time(b1) / rounds
    base_bytes = w.B * traffic.snapshot_round_bytes(shape, w.T)
    del pool
    torch.cuda.empty_cache()
    per_round_committed = committed / rounds
    return {"workload": f"{w.name}: {w.kind} B={w.B} H={w.H} G={w.G} P={w.P} N={w.N} L={w.L} T={w.T} "
                        f"capacity={w.cap} accept={w.accept} precision={w.precision}",
            "ms_per_round": ms, "committed_tokens_per_s": per_round_committed / (ms * 1e-3),
            "verified_tokens_per_s": w.B * w.T / (ms * 1e-3),
            "achieved_gbs": tot_bytes / rounds / (ms * 1e-3) / 1e9,
            "bytes_per_round": tot_bytes / rounds, "fold_fraction": folds / (rounds * w.B),
            "baseline": {"kind": "per-draft snapshots", "ms_per_round": ms_b,
                         "committed_tokens_per_s": per_round_committed / (ms_b * 1e-3),
                         "achieved_gbs": base_bytes / (ms_b * 1e-3) / 1e9, "bytes_per_round": base_bytes},
            "speedup": ms_b / ms, "rounds": rounds, "launches_per_round": 2}


# ----------------------------------------------------------------------------- sweeps
def measure_decode_graph(w, dev, reps: int = 50) -> dict:
    """GPU time per standard decode step of workload w, replay and eager alike:
    two windows of steps (2L launches, each with its own inputs) captured in
    one CUDA graph and replayed, so that the host's per-call cost, which bounds
    a small batch launched step by step, drops out of both arms."""
    import torch

    from rs_decode_gb300 import binding as rb
    from rs_decode_gb300 import synth, traffic
    from rs_decode_gb300.layer import Layer, to_device

    params, gp = _params(w, dev)
    steps = [to_device(synth.step_inputs(w, s, seed=0, params=params), dev) for s in range(2 * w.L)]
    layer = Layer(w.kind, w.B, w.H, w.G, w.P, w.N, w.L, capacity=w.cap, precision=rb.PRECISIONS[w.precision])
    S0 = _init_state(layer, w, dev, 0)
    S_e = S0.clone()
    y = torch.empty(w.B, w.H, w.P, device=dev)

    def replay():
        for d in steps:
            layer.decode(d, gp, y)

    def eager():
        for d in steps:
            if w.kind == "mamba2":
                rb.rs_eager_step_mamba2(layer.desc, S_e, d["x"], d["dt"], gp["A"], d["Bm"], d["Cm"], gp["D"], y)
            else:
                fn = rb.rs_eager_step_gdn if w.kind == "gdn" else rb.rs_eager_step_kda
                fn(layer.desc, S_e, d["q"], d["k"], d["v"], d["alpha"], d["beta"], y)

    def per_step_ms(fn):
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):  # warm-up (one-time set-up happens outside the capture)
            fn()
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            fn()
        for _ in range(3):
            g.replay()
        a, b = _events(2)
        torch.cuda.synchronize(dev)
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / (reps * len(steps))

    ms_r, ms_e = per_step_ms(replay), per_step_ms(eager)
    if layer.status() != 0:
        raise RuntimeError("device status bits set during the benchmark")
    shape = traffic.Shape(w.kind, w.B, w.H, w.G, w.P, w.N)
    nb = sum(traffic.replay_step_bytes(shape, h, h + 1 >= w.L) for h in range(w.L)) / w.L
    return {"ms_per_step": ms_r, "eager_ms_per_step": ms_e, "bytes_per_step": nb, "speedup_vs_eager": ms_e / ms_r}


def run_sweeps(dev):
    """Window size L, batch B, draft count T and two-precision sweeps of the
    Mamba-2 serving layer (the pages' window trade-off and small-batch remark,
    "ReplaySSM: Cache SSM Inputs, Not State", sections "How it works" and
    "Limits"), each point against its baseline kernel."""
    from rs_decode_gb300 import synth
    peak = measured_peaks().get("hbm_gbs") or 6800.0
    base = synth.WORKLOADS["mamba2"]

    def dec(w, K=256):
        m = measure_decode(w, K, 2 * w.L, dev, 0, 1, want_e2e=False, want_clocks=False)
        gbs = m["bytes_per_launch"] / (m["ms_per_step"] * 1e-3) / 1e9
        return {"tokens_per_s": w.B / (m["ms_per_step"] * 1e-3), "achieved_gbs": gbs, "frac": gbs / peak,
                "eager_tokens_per_s": m["eager"]["value"], "speedup_vs_eager": m["eager"]["speedup_of_replay"]}

    for L in (8, 16, 32):
        print(json.dumps({"sweep": "window", "L": L, "B": 256, **dec(base.with_(L=L), K=16 * L)}), flush=True)
    for B in (1, 8, 32, 128, 512):
        print(json.dumps({"sweep": "batch", "L": 16, "B": B, **dec(base.with_(B=B))}), flush=True)
    for B in (1, 4, 8, 16, 32):  # small batches, GPU time (CUDA-graph replay, both arms)
        m = measure_decode_graph(base.with_(B=B), dev)
        gbs = m["bytes_per_step"] / (m["ms_per_step"] * 1e-3) / 1e9
        print(json.dumps({"sweep": "batch (graph replay)", "L": 16, "B": B,
                          "tokens_per_s": B / (m["ms_per_step"] * 1e-3), "achieved_gbs": gbs, "frac": gbs / peak,
                          "eager_tokens_per_s": B / (m["eager_ms_per_step"] * 1e-3),
                          "speedup_vs_eager": m["speedup_vs_eager"]}), flush=True)
    print(json.dumps({"sweep": "precision", "precision": "two", "B": 256, "L": 16,
                      **dec(base.with_(precision="two"))}), flush=True)
    gdn = synth.WORKLOADS["gdn"]
    for prec in ("fp32", "fp32+u16"):  # GDN records with u in fp32 or bf16
        m = measure_decode(gdn.with_(precision=prec), 256, 2 * gdn.L, dev, 0, 1, want_e2e=False, want_clocks=False)
        gbs = m["bytes_per_launch"] / (m["ms_per_step"] * 1e-3) / 1e9
        print(json.dumps({"sweep": "gdn records", "precision": prec, "B": 256, "L": 16,
                          "tokens_per_s": gdn.B / (m["ms_per_step"] * 1e-3), "bytes_per_step": m["bytes_per_launch"],
                          "achieved_gbs": gbs, "frac": gbs / peak}), flush=True)
    spec = synth.WORKLOADS["mamba2_spec"]
    for T in (1, 2, 4, 5, 8):
        o = measure_spec(spec.with_(T=T, capacity=16 + T), 64, 8, dev, 0)
        print(json.dumps({"sweep": "drafts", "T": T, "B": 256, "L": 16,
                          "verified_tokens_per_s": o["verified_tokens_per_s"],
                          "committed_tokens_per_s": o["committed_tokens_per_s"],
                          "achieved_gbs": o["achieved_gbs"], "frac": o["achieved_gbs"] / peak,
                          "snapshot_committed_tokens_per_s": o["baseline"]["committed_tokens_per_s"],
                          "speedup_vs_snapshots": o["speedup"]}), flush=True)


# ----------------------------------------------------------------------------- main arm
def frac_of(d: dict | None, peak: float) -> dict | None:
    if d is None:
        return None
    return dict(d, frac=d["achieved_gbs"] / peak)


def run_librs(args, rank: int, world: int, local_rank: int) -> dict | None:
    import torch

    from rs_decode_gb300 import synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = synth.WORKLOADS[args.workload]
    if args.batch:
        w = w.with_(B=args.batch)
    K, W = args.steps, args.warmup
    m = measure_decode(w, K, W, dev, rank, world, want_eager=not args.no_eager, want_e2e=not args.no_e2e)
    ms_total = max_over_ranks(m["ms_total"], dev)

    peak = measured_peaks().get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = peak or 6800.0
    others = {}
    if not args.headline_only and world == 1 and not args.batch:
        for other in [k for k in ("mamba2", "gdn", "kda") if k != w.kind]:
            ow = synth.WORKLOADS[other]
            g = measure_decode(ow, 512, W, dev, rank, world, want_e2e=False, want_clocks=False)
            gbs = g["bytes_per_launch"] / (g["ms_per_step"] * 1e-3) / 1e9
            others[other] = {"workload": f"{other} decode B={ow.B} H={ow.H} G={ow.G} P={ow.P} N={ow.N} L={ow.L}, "
                                         f"fp32 checkpoint" + (", one decay per key channel" if other == "kda" else ""),
                             "value": ow.B / (g["ms_per_step"] * 1e-3), "unit": "tokens/s",
                             "ms_per_step": g["ms_per_step"], "achieved_gbs": gbs,
                             "bytes_per_step": g["bytes_per_launch"], "frac_of_measured_peak": gbs / peak,
                             "window_weighted": g["window_weighted"], "eager": g["eager"]}
        for name in ("mamba2_spec", "gdn_spec"):
            o = measure_spec(synth.WORKLOADS[name], 64, 8, dev, rank)
            o["frac_of_measured_peak"] = o["achieved_gbs"] / peak
            others[name] = o
        others["gdn_spec"]["output_error_vs_oracle"] = recorded_output_error()
    if rank != 0:
        return None

    # algorithmic bytes per launch / the timed region's time per launch
    achieved = m["bytes_per_launch"] / (m["ms_per_step"] * 1e-3) / 1e9
    clk = ClockSampler.summarise(m["clock_rows"], *m["t_wall"]) if m["clock_rows"] else None
    kernel = {"mamba2": "rows::replay_pipe_kernel<mamba2, P=64, N=128, HU=8, TMAX=1, NC=256, NS=2, SPLIT=1>",
              "gdn": "cols::replay_pipe_kernel<gdn, P=128, N=128, TMAX=1, TC=0> (launch: HU=2, NS=5, 2 CTAs/SM)",
              "kda": "cols::replay_pipe_kernel<kda, P=128, N=128, TMAX=1, TC=0>"}[w.kind]
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
        "config": {"workload": f"{w.kind} decode B={w.B} H={w.H} P={w.P} N={w.N} G={w.G} L={w.L} fp32 checkpoint",
                   "B_per_gpu": w.B, "window_L": w.L, "state_mib_per_seq": w.H * w.N * w.P * 4 / 2**20,
                   "parallelism": f"dp{world}" if world > 1 else "single",
                   "l2": "inputs larger than L2 (1 GiB checkpoint per step)",
                   "inputs": f"{min(INPUT_POOL, K + W)} distinct seeded steps cycled"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": profiled_traffic(w.kind),
                     "peak_source": f"{peak_src} (copy bandwidth, MEASURED_PEAKS.json hbm_gbs)",
                     "algorithmic_bytes_per_launch": m["bytes_per_launch"], "kernel": kernel,
                     "duration": "timed region / K (CUDA events on the launching stream)",
                     # the launches that fold the window (checkpoint read + write, the flush route) and
                     # the others (checkpoint read only), each against the same peak
                     "fold_launch": frac_of(m["fold_launch"], peak), "stream_launch": frac_of(m["stream_launch"], peak),
                     "split": "K more launches after the timed region, each between its own events",
                     # the nominal HBM3e figure, for context (the fraction above is against the measured copy)
                     "frac_of_nominal": achieved / NOMINAL_HBM_GBS, "nominal_peak": NOMINAL_HBM_GBS},
        "hbm_gbs": achieved,
        "timed_region": {"starts_at_window_position": 0, "folds": m["folds_timed"], "window_L": w.L,
                         "whole_windows": K % w.L == 0},
        "window_weighted": m["window_weighted"],
        "eager": m["eager"],
        "gpu_launches": K,
        "clocks": clk,
        "e2e": m["e2e"],
    }
    if others:
        out["workloads"] = others
    return out


def main():
    args = parse()
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return 0
        from rs_decode_gb300 import synth
        w = synth.WORKLOADS[args.workload]
        ref = run_reference(w, args.steps, args.warmup)
        line = {"impl": "reference", "metric": METRIC, "value": ref["value"], "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ref["ms_per_step"],
                "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": f"{w.kind} decode B={w.B} H={w.H} P={w.P} N={w.N} G={w.G} L={w.L}"},
                "cpu_baseline": ref,
                "e2e": {"value": ref["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    import torch
    if args.sweep:
        torch.cuda.set_device(local_rank)
        run_sweeps(torch.device("cuda", local_rank))
        return 0
    if args.spec:
        from rs_decode_gb300 import synth
        torch.cuda.set_device(local_rank)
        w = synth.WORKLOADS[args.spec]
        if args.batch:
            w = w.with_(B=args.batch)
        o = measure_spec(w, args.rounds, args.warmup, torch.device("cuda", local_rank), rank)
        o["frac_of_measured_peak"] = o["achieved_gbs"] / (measured_peaks().get("hbm_gbs") or 6800.0)
        print(json.dumps(o))
        return 0
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    out = run_librs(args, rank, world, local_rank)
    if out is not None:
        if not args.no_cpu_baseline and world == 1:
            from rs_decode_gb300 import synth
            out["cpu_baseline"] = time_oracle(synth.WORKLOADS[args.workload], args.cpu_seconds)
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

"""Shared test harness: run the CUDA library and the fp64 oracle on the same
seeded inputs and compare.

Error metric (a reading of "max relative error"): per (step, sequence) the
normwise relative error max|gpu - ref| / max|ref| over all heads and
elements of that sequence's output (or state); the worst case is checked.
Tolerances: 2e-3 for results computed from the fp32 checkpoint with bf16
inputs, 3e-2 for outputs read from the bf16 checkpoint.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from oracle.pointers import Pointers
from rs_decode_gb300 import binding as rb
from rs_decode_gb300 import synth
from rs_decode_gb300.layer import Layer, to_device

TOL_HP = 2e-3
TOL_LP = 3e-2

PREC = rb.PRECISIONS


def rel_err(got, ref) -> np.ndarray:
    """Per-sequence normwise relative error; arrays with the batch first."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    B = ref.shape[0]
    g, r = got.reshape(B, -1), ref.reshape(B, -1)
    return np.max(np.abs(g - r), axis=1) / np.maximum(np.max(np.abs(r), axis=1), 1e-300)


def _head_view(a, H: int) -> np.ndarray:
    a = np.asarray(a, np.float64)
    n, P = a.shape[0], a.shape[-1]
    return np.moveaxis(a.reshape(n, -1, H, P), 2, 1).reshape(n, H, -1)


def rel_err_heads(got, ref, H: int) -> np.ndarray:
    """Per-(sequence, head) normwise relative error [n, H] of outputs shaped
    [n, H, P] or [n, T, H, P]: the same metric as ``rel_err`` taken over one
    head's elements of one call.  Ill-conditioned where a head's outputs
    cancel to almost nothing in that call; ``HeadErr`` takes it over a run."""
    g, r = _head_view(got, H), _head_view(ref, H)
    return np.max(np.abs(g - r), axis=2) / np.maximum(np.max(np.abs(r), axis=2), 1e-300)


class HeadErr:
    """Per-(sequence, head) normwise relative error over a whole run: the
    largest error of a head's outputs over all calls, divided by the largest
    magnitude of its outputs over all calls.

    So a head whose outputs are small throughout cannot hide its error behind
    the sequence's largest head, while a call in which one head's outputs
    cancel to almost nothing (a query nearly orthogonal to that head's state:
    the fp32 replay form itself then misses the fp64 value by order one, as at
    step 100 of the gdn workload, sequence 175, head 26, whose outputs were
    1e-7 of their usual size) is judged against the head's usual size."""

    def __init__(self, H: int):
        self.H = H
        self.err = self.mag = None

    def add(self, got, ref) -> None:
        g, r = _head_view(got, self.H), _head_view(ref, self.H)
        e, m = np.max(np.abs(g - r), axis=2), np.max(np.abs(r), axis=2)
        self.err = e if self.err is None else np.maximum(self.err, e)
        self.mag = m if self.mag is None else np.maximum(self.mag, m)

    def worst(self) -> float:
        return float(np.max(self.err / np.maximum(self.mag, 1e-300)))


def state_errs(t: torch.Tensor, ref: np.ndarray, idx) -> tuple[np.ndarray, np.ndarray]:
    """Normwise relative errors of device states t fp32 [B,H,N,P] (key-major)
    at sequences idx against the oracle's ref f64 [n,H,P,N], computed on the
    device (full-size states): per sequence [n] and per (sequence, head) [n,H]."""
    dev = t.device
    g = t[torch.as_tensor(np.asarray(idx), device=dev)].to(torch.float64)
    r = torch.from_numpy(np.ascontiguousarray(ref, dtype=np.float64)).to(dev).transpose(-1, -2)
    d = (g - r).abs().flatten(2).amax(-1)
    m = r.abs().flatten(2).amax(-1)
    per_head = (d / m.clamp_min(1e-300)).cpu().numpy()
    per_seq = (d.amax(-1) / m.amax(-1).clamp_min(1e-300)).cpu().numpy()
    del g, r
    return per_seq, per_head


def parity_sample(B: int, n: int = 64, seed: int = 0) -> np.ndarray:
    """n sequences of a batch of B for the oracle to recompute: the first, the
    last and n - 2 others drawn without replacement (all of them if B <= n)."""
    if B <= n:
        return np.arange(B)
    rng = np.random.Generator(np.random.PCG64(seed))
    mid = rng.choice(np.arange(1, B - 1), n - 2, replace=False)
    return np.sort(np.concatenate([[0, B - 1], mid]))


def state_np_to_gpu(S: np.ndarray) -> torch.Tensor:
    """[B,H,P,N] (math layout) -> device fp32 [B,H,N,P] (key-major slabs)."""
    return torch.from_numpy(np.ascontiguousarray(np.swapaxes(np.asarray(S, np.float32), -1, -2))).cuda()


def state_gpu_to_np(t: torch.Tensor) -> np.ndarray:
    """device [B,H,N,P] -> numpy [B,H,P,N] float64."""
    return np.swapaxes(t.detach().cpu().numpy().astype(np.float64), -1, -2)


def make_layer(w: synth.Workload, precision: str | None = None, T_max: int | None = None) -> Layer:
    prec = PREC[precision or w.precision]
    tmax = w.T if T_max is None and w.spec else (T_max or 0)
    return Layer(w.kind, w.B, w.H, w.G, w.P, w.N, w.L, T_max=tmax,
                 capacity=w.capacity or None, precision=prec)


def gpu_params(w, params) -> dict:
    if w.kind == "mamba2":
        return {"A": torch.from_numpy(params["A"]).cuda(), "D": torch.from_numpy(params["D"]).cuda()}
    return {}


class StandardRun:
    """Runs standard decode steps on the GPU and on the oracle side by side.

    ``sample`` restricts the oracle to a subset of sequences (full-size runs);
    the GPU always runs all w.B sequences.
    """

    def __init__(self, w: synth.Workload, seed: int = 0, precision: str | None = None,
                 sample=None, S0: np.ndarray | None = None):
        self.w, self.seed = w, seed
        self.params = synth.layer_params(w, seed)
        self.gp = gpu_params(w, self.params)
        S0 = synth.initial_state(w, seed) if S0 is None else S0
        self.idx = np.arange(w.B) if sample is None else np.asarray(sample)
        self.layer = make_layer(w, precision)
        self.layer.init(state_np_to_gpu(S0))
        self.model = oracle.Model(w.kind, S0[self.idx], self.params)
        self.ptr = Pointers(w.L, w.cap)
        del S0
        self.t = 0

    def step(self):
        d = synth.step_inputs(self.w, self.t, self.seed, self.params)
        y = self.layer.decode(to_device(d), self.gp).cpu().numpy()
        y_ref = self.model.step(synth.slice_batch(d, self.idx))
        folded = self.ptr.standard_step()
        self.t += 1
        return y[self.idx], y_ref, folded

    def checkpoint(self) -> np.ndarray:
        hp = self.layer.checkpoint_hp()
        t = hp if hp is not None else self.layer.checkpoint_lp_f32()
        return state_gpu_to_np(t[torch.from_numpy(self.idx).cuda()])

    def materialized(self) -> np.ndarray:
        return state_gpu_to_np(self.layer.materialize()[torch.from_numpy(self.idx).cuda()])


class SpecRun:
    """Speculative rounds (verify T drafts, then commit) on GPU and oracle.

    ``alpha_pow`` raises every drawn decay to that power before both sides
    see it (a slower-decaying variant of the input recipe)."""

    def __init__(self, w: synth.Workload, seed: int = 0, precision: str | None = None, sample=None,
                 alpha_pow: float | None = None):
        self.w, self.seed, self.alpha_pow = w, seed, alpha_pow
        self.params = synth.layer_params(w, seed)
        self.gp = gpu_params(w, self.params)
        S0 = synth.initial_state(w, seed)
        self.idx = np.arange(w.B) if sample is None else np.asarray(sample)
        self.layer = make_layer(w, precision)
        self.layer.init(state_np_to_gpu(S0))
        self.model = oracle.Model(w.kind, S0[self.idx], self.params)
        self.ptrs = [Pointers(w.L, w.cap) for _ in range(w.B)]
        del S0
        self.r = 0

    def round(self, accepted: np.ndarray | None = None):
        """Returns (y_gpu, y_ref, folded[B] bool, S_before (oracle committed state))."""
        d = synth.round_inputs(self.w, self.r, self.seed, self.params)
        if self.alpha_pow is not None:
            d["alpha"] = np.power(d["alpha"], np.float32(self.alpha_pow)).astype(np.float32)
        if accepted is not None:
            d["accepted"] = np.asarray(accepted, np.int32)
        dev = to_device(d)
        y = self.layer.verify(self.w.T, dev, self.gp).cpu().numpy()
        folded = np.array([p.verify(self.w.T) > 0 for p in self.ptrs])
        S_before = self.model.S.copy()
        y_ref = self.model.spec_round(synth.slice_batch(d, self.idx))
        self.layer.commit(dev["accepted"])
        for p, a in zip(self.ptrs, d["accepted"]):
            p.commit(int(a))
        self.r += 1
        return y[self.idx], y_ref, folded[self.idx], S_before, d["accepted"][self.idx]

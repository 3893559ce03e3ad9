"""Seeded synthetic inputs for the ReplaySSM decode workloads.

This module only draws random numbers and rounds them to the storage types
(bf16 as raw uint16 bits, fp32, int32). It holds none of the method's
arithmetic: no decay, no recurrence, no replay. Both the fp64 oracle and the
CUDA path consume exactly the arrays produced here.

Every tensor is drawn from its own stream,
``PCG64(SeedSequence([seed, step, tensor_id]))``, so any step can be
regenerated on its own and the two sides never depend on draw order.

Workloads (shapes and distributions follow the serving-scale settings the
ReplaySSM pages describe: batch 256, window L = 16, 4 MiB fp32 state per
sequence per layer; "ReplaySSM: Cache SSM Inputs, Not State", sections
"What it claims" and "Evidence"):

* ``tiny``      Mamba-2, B=4, H=8, P=64, N=128, G=1, L=16, 48 steps, S0 = 0.
* ``mamba2``    Mamba-2, B=256, H=128, P=64, N=128, G=8, L=16, 256 steps,
                S0 ~ N(0, 0.1^2).
* ``gdn``       Gated DeltaNet, B=256, H_k=16, H_v=32, d_k=d_v=128, L=16,
                256 steps, S0 ~ N(0, 0.1^2).
* ``mamba2_spec`` Mamba-2 shapes of ``mamba2``, T=4 drafts, capacity 20,
                128 rounds, accepted length ~ U{0..4}.
* ``gdn_spec``  GDN shapes of ``gdn`` at B=512, T=3, capacity 19, 128 rounds,
                accepted length ~ Binomial(3, 0.7), two-precision checkpoint.
* ``kda``       the shapes of ``gdn`` with one decay per key channel (a reading
                of Kimi Delta Attention, named as compatible in section
                "Limits" of the same page), 256 steps.

Mamba-2 per step: x ~ N(0,1) bf16 [B,H,P]; B, C ~ N(0,1)/sqrt(N) bf16
[B,G,N]; dt = softplus(N(-2, 0.5)) fp32 [B,H]; per head A = -exp(U(0, log 16))
and D ~ N(0,1).
GDN per step: q, k ~ N(0,1) rounded to bf16, L2-normalised per head in fp32
and rounded to bf16 again [B,H_k,d]; v ~ N(0,1) bf16 [B,H_v,d];
alpha = exp(-softplus(N(0,1)) * s_h) with s_h = exp(U(log 1, log 16)) drawn
once per head; beta = sigmoid(N(0,1)); alpha and beta fp32 [B,H_v].
Per-channel decay: as GDN, but alpha = exp(-softplus(N(0,1)) * s_h / 16) is
drawn for every key channel, fp32 [B,H_v,d_k], so that over a 16-record window
the channels of one head range from nearly forgotten to nearly kept.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

# Stream identifiers (one per tensor kind).
_ID = {
    "x": 1, "dt": 2, "Bm": 3, "Cm": 4, "A": 5, "D": 6, "S0": 7,
    "q": 11, "k": 12, "v": 13, "alpha_n": 14, "alpha_s": 15, "beta": 16, "alpha_c": 17,
    "accept": 21,
}
_PARAM_STEP = 0xFFFFFFF  # "step" slot used for per-layer parameters


def _rng(seed: int, step: int, name: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, step, _ID[name]])))


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (round to nearest, ties to even) as raw uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _softplus(z: np.ndarray) -> np.ndarray:
    return np.logaddexp(0.0, z)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "mamba2", "gdn" or "kda" (per-channel decay)
    B: int
    H: int               # value heads (Mamba-2 heads, GDN v-heads)
    G: int               # Mamba-2 B/C groups, GDN k-heads
    P: int               # headdim (Mamba-2) / d_v (GDN)
    N: int               # dstate (Mamba-2) / d_k (GDN)
    L: int
    steps: int           # standard steps, or verify rounds for spec workloads
    T: int = 1           # drafts per verify round (1 = standard decode)
    capacity: int = 0    # circular buffer capacity (0 -> L)
    init_std: float = 0.0
    accept: str = ""     # "uniform" or "binomial0.7" for spec workloads
    precision: str = "fp32"   # "fp32", "two", "shared_bf16"; GDN "+u16": records keep u in bf16

    @property
    def cap(self) -> int:
        return self.capacity or self.L

    @property
    def spec(self) -> bool:
        return self.T > 1 or bool(self.accept)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", "mamba2", B=4, H=8, G=1, P=64, N=128, L=16, steps=48),
    "mamba2": Workload("mamba2", "mamba2", B=256, H=128, G=8, P=64, N=128, L=16, steps=256,
                       init_std=0.1),
    "gdn": Workload("gdn", "gdn", B=256, H=32, G=16, P=128, N=128, L=16, steps=256, init_std=0.1),
    "mamba2_spec": Workload("mamba2_spec", "mamba2", B=256, H=128, G=8, P=64, N=128, L=16,
                            steps=128, T=4, capacity=20, init_std=0.1, accept="uniform"),
    "gdn_spec": Workload("gdn_spec", "gdn", B=512, H=32, G=16, P=128, N=128, L=16, steps=128,
                         T=3, capacity=19, init_std=0.1, accept="binomial0.7", precision="two"),
    "kda": Workload("kda", "kda", B=256, H=32, G=16, P=128, N=128, L=16, steps=256, init_std=0.1),
}


# ----------------------------------------------------------------------------- parameters
def layer_params(w: Workload, seed: int = 0) -> dict:
    """Per-layer constants: Mamba-2 A, D per head; GDN decay scale per head."""
    if w.kind == "mamba2":
        A = -np.exp(_rng(seed, _PARAM_STEP, "A").uniform(0.0, math.log(16.0), w.H))
        D = _rng(seed, _PARAM_STEP, "D").standard_normal(w.H)
        return {"A": A.astype(np.float32), "D": D.astype(np.float32)}
    s = np.exp(_rng(seed, _PARAM_STEP, "alpha_s").uniform(math.log(1.0), math.log(16.0), w.H))
    return {"alpha_scale": s.astype(np.float32)}


def initial_state(w: Workload, seed: int = 0, batch: slice | None = None) -> np.ndarray:
    """Initial state S0, fp32 [B, H, P, N] (value index p, key index n)."""
    shape = (w.B, w.H, w.P, w.N)
    if w.init_std == 0.0:
        s = np.zeros(shape, np.float32)
    else:
        s = (_rng(seed, _PARAM_STEP, "S0").standard_normal(shape, dtype=np.float32)
             * np.float32(w.init_std))
    return s if batch is None else np.ascontiguousarray(s[batch])


# ----------------------------------------------------------------------------- per step
def _l2norm_bf16(a_bits: np.ndarray) -> np.ndarray:
    a = bf16_bits_to_f32(a_bits)
    n = np.sqrt(np.sum(a * a, axis=-1, keepdims=True, dtype=np.float32))
    return to_bf16_bits(a / np.maximum(n, np.float32(1e-6)))


def _mamba2_draw(w: Workload, seed: int, step: int, lead: tuple) -> dict:
    x = to_bf16_bits(_rng(seed, step, "x").standard_normal(lead + (w.H, w.P), dtype=np.float32))
    dt = _softplus(_rng(seed, step, "dt").normal(-2.0, 0.5, lead + (w.H,))).astype(np.float32)
    sc = np.float32(1.0 / math.sqrt(w.N))
    Bm = to_bf16_bits(_rng(seed, step, "Bm").standard_normal(lead + (w.G, w.N), dtype=np.float32) * sc)
    Cm = to_bf16_bits(_rng(seed, step, "Cm").standard_normal(lead + (w.G, w.N), dtype=np.float32) * sc)
    return {"x": x, "dt": dt, "Bm": Bm, "Cm": Cm}


def _gdn_draw(w: Workload, seed: int, step: int, lead: tuple, params: dict) -> dict:
    q = _l2norm_bf16(to_bf16_bits(_rng(seed, step, "q").standard_normal(lead + (w.G, w.N), dtype=np.float32)))
    k = _l2norm_bf16(to_bf16_bits(_rng(seed, step, "k").standard_normal(lead + (w.G, w.N), dtype=np.float32)))
    v = to_bf16_bits(_rng(seed, step, "v").standard_normal(lead + (w.H, w.P), dtype=np.float32))
    if w.kind == "kda":  # one decay per key channel
        g = _softplus(_rng(seed, step, "alpha_c").standard_normal(lead + (w.H, w.N)))
        alpha = np.exp(-g * params["alpha_scale"].astype(np.float64)[:, None] / 16.0).astype(np.float32)
    else:
        g = _softplus(_rng(seed, step, "alpha_n").standard_normal(lead + (w.H,)))
        alpha = np.exp(-g * params["alpha_scale"].astype(np.float64)).astype(np.float32)
    beta = (1.0 / (1.0 + np.exp(-_rng(seed, step, "beta").standard_normal(lead + (w.H,))))).astype(np.float32)
    return {"q": q, "k": k, "v": v, "alpha": alpha, "beta": beta}


def step_inputs(w: Workload, step: int, seed: int = 0, params: dict | None = None) -> dict:
    """Inputs of standard decode step ``step`` (0-based) for all B sequences.

    Mamba-2: x u16[B,H,P], dt f32[B,H], Bm u16[B,G,N], Cm u16[B,G,N].
    GDN:     q,k u16[B,G,N], v u16[B,H,P], alpha f32[B,H], beta f32[B,H].
    kda:     as GDN with alpha f32[B,H,N].
    """
    if w.kind == "mamba2":
        return _mamba2_draw(w, seed, step, (w.B,))
    return _gdn_draw(w, seed, step, (w.B,), params if params is not None else layer_params(w, seed))


def round_inputs(w: Workload, rnd: int, seed: int = 0, params: dict | None = None) -> dict:
    """Draft inputs of verify round ``rnd``: as :func:`step_inputs` with a
    draft axis after the batch axis ([B, T, ...]), plus ``accepted`` i32[B]."""
    lead = (w.B, w.T)
    if w.kind == "mamba2":
        d = _mamba2_draw(w, seed, rnd, lead)
    else:
        d = _gdn_draw(w, seed, rnd, lead, params if params is not None else layer_params(w, seed))
    r = _rng(seed, rnd, "accept")
    if w.accept == "binomial0.7":
        a = r.binomial(w.T, 0.7, w.B)
    else:
        a = r.integers(0, w.T + 1, w.B)
    d["accepted"] = a.astype(np.int32)
    return d


def slice_batch(d: dict, idx) -> dict:
    """Restrict every per-sequence array of an input dict to sequences ``idx``."""
    return {k: np.ascontiguousarray(v[idx]) for k, v in d.items()}

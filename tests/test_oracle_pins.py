"""Pins for the fp64 oracle: checks against what the mathematics fixes.

None of these re-type the oracle's own loop.  They use

* the unrolled (checkpoint + input buffer) form of the recurrence evaluated in
  exact rational arithmetic (the representation the method is built on:
  "ReplaySSM: Cache SSM Inputs, Not State", section "How it works");
* closed forms of special cases (alpha = 1, alpha = 0, one step from zero,
  the GDN delta-rule overwrite, beta = 0; for the per-channel decay, a decay
  equal on every channel is GDN, and a zero decay clears its key channel);
* hand-worked examples stored in ``tests/golden/hand_worked.json``;
* the speculative-round semantics (flowchart on the same page): outputs of a
  round equal the outputs of standard steps over the drafts, a = 0 leaves the
  committed state unchanged, commit a equals recomputation over the prefix.

``test_pins_reject_planted_mistakes`` compiles copies of the oracle with a
plausible mistake planted in each and checks that some pin fails for each.
"""
from __future__ import annotations

import json
import math
import os
import shutil
import subprocess
from fractions import Fraction

import numpy as np
import pytest

import oracle
from rs_decode_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))

TINY_M2 = synth.Workload("pin_m2", "mamba2", B=2, H=4, G=2, P=2, N=3, L=4, steps=6, init_std=0.5)
TINY_GDN = synth.Workload("pin_gdn", "gdn", B=2, H=4, G=2, P=2, N=3, L=4, steps=6, init_std=0.5)
TINY_KDA = TINY_GDN.with_(name="pin_kda", kind="kda")


def _fr(a) -> np.ndarray:
    """Exact rational copy of a float array (object dtype)."""
    flat = [Fraction(float(v)) for v in np.asarray(a, dtype=np.float64).ravel()]
    return np.array(flat, dtype=object).reshape(np.shape(a))


def _bf(bits) -> np.ndarray:
    return _fr(synth.bf16_bits_to_f32(bits))


def _close(got, ref, tol=1e-12):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, dtype=object).astype(np.float64)
    scale = max(1.0, float(np.max(np.abs(ref))))
    err = float(np.max(np.abs(got - ref)))
    assert err <= tol * scale, f"max abs err {err:.3e} (scale {scale:.3e})"


# ----------------------------------------------------------------------------- unrolled brute force
def _unrolled_mamba2(w, S0, params, steps):
    """y_t = gamma(t) S0 q_t + sum_j w_j(t) v_j (k_j . q_t) + D x_t, exactly."""
    A, D = params["A"], params["D"]
    hpg = w.H // w.G
    ys = []
    rec = []  # per step: (alpha[B,H], v[B,H,P], k[B,H,N])
    for d in steps:
        alpha = np.empty((w.B, w.H), dtype=object)
        v = np.empty((w.B, w.H, w.P), dtype=object)
        k = np.empty((w.B, w.H, w.N), dtype=object)
        q = np.empty((w.B, w.H, w.N), dtype=object)
        x = _bf(d["x"])
        Bm, Cm = _bf(d["Bm"]), _bf(d["Cm"])
        for b in range(w.B):
            for h in range(w.H):
                dt = float(d["dt"][b, h])
                alpha[b, h] = Fraction(math.exp(dt * float(A[h])))
                v[b, h] = Fraction(dt) * x[b, h]
                k[b, h] = Bm[b, h // hpg]
                q[b, h] = Cm[b, h // hpg]
        rec.append((alpha, v, k))
        t = len(rec)
        y = np.empty((w.B, w.H, w.P), dtype=object)
        S0f = _fr(S0)
        for b in range(w.B):
            for h in range(w.H):
                gamma = Fraction(1)
                for j in range(t):
                    gamma *= rec[j][0][b, h]
                acc = gamma * S0f[b, h].dot(q[b, h])
                for j in range(t):
                    wj = Fraction(1)
                    for i in range(j + 1, t):
                        wj *= rec[i][0][b, h]
                    acc = acc + wj * rec[j][1][b, h] * rec[j][2][b, h].dot(q[b, h])
                y[b, h] = acc + Fraction(float(D[h])) * x[b, h]
        ys.append(y)
    return ys


def _unrolled_gdn(w, S0, steps):
    """Replay form: S_{t-1} k_t and y_t from S0 and the buffered u_j, exactly."""
    ratio = w.H // w.G
    S0f = _fr(S0)
    rec = []  # (alpha[B,H], u[B,H,P], k[B,H,N])
    ys, us = [], []
    for d in steps:
        q_all, k_all, v_all = _bf(d["q"]), _bf(d["k"]), _bf(d["v"])
        alpha = _fr(d["alpha"])
        beta = _fr(d["beta"])
        t = len(rec)  # records before this step
        u = np.empty((w.B, w.H, w.P), dtype=object)
        y = np.empty((w.B, w.H, w.P), dtype=object)
        kk = np.empty((w.B, w.H, w.N), dtype=object)
        for b in range(w.B):
            for h in range(w.H):
                kt, qt = k_all[b, h // ratio], q_all[b, h // ratio]
                kk[b, h] = kt

                def decay(lo, hi):  # prod_{i=lo}^{hi-1} alpha_i over recorded steps
                    r = Fraction(1)
                    for i in range(lo, hi):
                        r *= rec[i][0][b, h] if i < t else alpha[b, h]
                    return r

                sk = decay(0, t) * S0f[b, h].dot(kt)
                for j in range(t):
                    sk = sk + decay(j + 1, t) * rec[j][1][b, h] * rec[j][2][b, h].dot(kt)
                u[b, h] = beta[b, h] * (v_all[b, h] - alpha[b, h] * sk)
                acc = decay(0, t + 1) * S0f[b, h].dot(qt)
                for j in range(t):
                    acc = acc + decay(j + 1, t + 1) * rec[j][1][b, h] * rec[j][2][b, h].dot(qt)
                acc = acc + u[b, h] * kt.dot(qt)
                y[b, h] = acc
        rec.append((alpha, u, kk))
        ys.append(y)
        us.append(u)
    return ys, us


def _unrolled_kda(w, S0, steps):
    """Replay form with one decay per key channel, exactly.  With
    w_j(t) = alpha_{j+1} * ... * alpha_t (elementwise over channels) and
    gamma(t) = alpha_1 * ... * alpha_t:
      D_t k_t = S0 (gamma(t) * k_t) + sum_{j<t} u_j ((w_j(t) * k_j) . k_t)
      u_t = beta_t (v_t - D_t k_t)
      y_t = S0 (gamma(t) * q_t) + sum_{j<t} u_j ((w_j(t) * k_j) . q_t) + u_t (k_t . q_t)"""
    ratio = w.H // w.G
    S0f = _fr(S0)
    rec = []  # (alpha[B,H,N], u[B,H,P], k[B,H,N])
    ys, us = [], []
    for d in steps:
        q_all, k_all, v_all = _bf(d["q"]), _bf(d["k"]), _bf(d["v"])
        alpha, beta = _fr(d["alpha"]), _fr(d["beta"])
        t = len(rec)
        u = np.empty((w.B, w.H, w.P), dtype=object)
        y = np.empty((w.B, w.H, w.P), dtype=object)
        kk = np.empty((w.B, w.H, w.N), dtype=object)
        for b in range(w.B):
            for h in range(w.H):
                kt, qt = k_all[b, h // ratio], q_all[b, h // ratio]
                kk[b, h] = kt

                def decay(lo):  # elementwise product of alpha_i for records lo..t (this step included)
                    r = np.array([Fraction(1)] * w.N, dtype=object)
                    for i in range(lo, t):
                        r = r * rec[i][0][b, h]
                    return r * alpha[b, h]

                dk = S0f[b, h].dot(decay(0) * kt)
                acc = S0f[b, h].dot(decay(0) * qt)
                for j in range(t):
                    wk = decay(j + 1) * rec[j][2][b, h]
                    dk = dk + rec[j][1][b, h] * wk.dot(kt)
                    acc = acc + rec[j][1][b, h] * wk.dot(qt)
                u[b, h] = beta[b, h] * (v_all[b, h] - dk)
                y[b, h] = acc + u[b, h] * kt.dot(qt)
        rec.append((alpha, u, kk))
        ys.append(y)
        us.append(u)
    return ys, us


def pin_unrolled_mamba2():
    w = TINY_M2
    params = synth.layer_params(w, seed=3)
    S0 = synth.initial_state(w, seed=3)
    steps = [synth.step_inputs(w, s, seed=3) for s in range(w.steps)]
    ref = _unrolled_mamba2(w, S0, params, steps)
    m = oracle.Model("mamba2", S0, params)
    for s, d in enumerate(steps):
        _close(m.step(d), ref[s])


def pin_unrolled_gdn():
    w = TINY_GDN
    params = synth.layer_params(w, seed=4)
    S0 = synth.initial_state(w, seed=4)
    steps = [synth.step_inputs(w, s, seed=4, params=params) for s in range(w.steps)]
    ref_y, ref_u = _unrolled_gdn(w, S0, steps)
    S = np.array(S0, np.float64)
    for s, d in enumerate(steps):
        y, u = oracle.gdn_step(S, d["q"], d["k"], d["v"], d["alpha"], d["beta"], want_u=True)
        _close(y, ref_y[s])
        _close(u, ref_u[s])


def pin_unrolled_kda():
    w = TINY_KDA
    params = synth.layer_params(w, seed=12)
    S0 = synth.initial_state(w, seed=12)
    steps = [synth.step_inputs(w, s, seed=12, params=params) for s in range(w.steps)]
    assert steps[0]["alpha"].shape == (w.B, w.H, w.N)
    ref_y, ref_u = _unrolled_kda(w, S0, steps)
    S = np.array(S0, np.float64)
    for s, d in enumerate(steps):
        y, u = oracle.kda_step(S, d["q"], d["k"], d["v"], d["alpha"], d["beta"], want_u=True)
        _close(y, ref_y[s])
        _close(u, ref_u[s])


# ----------------------------------------------------------------------------- closed forms
def _m2_inputs(w, seed, A, D):
    params = {"A": np.full(w.H, A, np.float32), "D": np.full(w.H, D, np.float32)}
    steps = [synth.step_inputs(w, s, seed=seed) for s in range(w.steps)]
    return params, steps


def pin_mamba2_alpha_one_is_matmul():
    """alpha = 1 (A = 0), S0 = 0, D = 0: S_t = V_t K_t^T, a plain matrix product."""
    w = TINY_M2.with_(init_std=0.0)
    params, steps = _m2_inputs(w, 5, 0.0, 0.0)
    m = oracle.Model("mamba2", synth.initial_state(w), params)
    hpg = w.H // w.G
    for t, d in enumerate(steps, 1):
        y = m.step(d)
        for b in range(w.B):
            for h in range(w.H):
                V = np.stack([s["dt"][b, h].astype(np.float64)
                              * synth.bf16_bits_to_f32(s["x"][b, h]).astype(np.float64)
                              for s in steps[:t]], axis=1)              # P x t
                K = np.stack([synth.bf16_bits_to_f32(s["Bm"][b, h // hpg]).astype(np.float64)
                              for s in steps[:t]], axis=1)              # N x t
                q = synth.bf16_bits_to_f32(d["Cm"][b, h // hpg]).astype(np.float64)
                np.testing.assert_allclose(m.S[b, h], V @ K.T, rtol=1e-12, atol=1e-14)
                np.testing.assert_allclose(y[b, h], (V @ K.T) @ q, rtol=1e-12, atol=1e-14)


def pin_mamba2_alpha_zero_forgets():
    """alpha = 0 (A = -inf): S_t = v_t k_t^T, y_t = v_t (k_t . q_t) + D x_t."""
    w = TINY_M2
    params, steps = _m2_inputs(w, 6, -np.inf, 0.75)
    m = oracle.Model("mamba2", synth.initial_state(w, seed=6), params)
    hpg = w.H // w.G
    for d in steps:
        y = m.step(d)
        for b in range(w.B):
            for h in range(w.H):
                x = synth.bf16_bits_to_f32(d["x"][b, h]).astype(np.float64)
                v = float(d["dt"][b, h]) * x
                k = synth.bf16_bits_to_f32(d["Bm"][b, h // hpg]).astype(np.float64)
                q = synth.bf16_bits_to_f32(d["Cm"][b, h // hpg]).astype(np.float64)
                np.testing.assert_allclose(m.S[b, h], np.outer(v, k), rtol=1e-14, atol=0)
                np.testing.assert_allclose(y[b, h], v * (k @ q) + 0.75 * x, rtol=1e-12, atol=1e-14)


def pin_mamba2_single_step_from_zero():
    """One step from S0 = 0: y = dt x (B . C) + D x."""
    w = TINY_M2.with_(init_std=0.0)
    params = synth.layer_params(w, seed=7)
    d = synth.step_inputs(w, 0, seed=7)
    y = oracle.Model("mamba2", synth.initial_state(w), params).step(d)
    hpg = w.H // w.G
    for b in range(w.B):
        for h in range(w.H):
            x = synth.bf16_bits_to_f32(d["x"][b, h]).astype(np.float64)
            k = synth.bf16_bits_to_f32(d["Bm"][b, h // hpg]).astype(np.float64)
            q = synth.bf16_bits_to_f32(d["Cm"][b, h // hpg]).astype(np.float64)
            ref = float(d["dt"][b, h]) * x * (k @ q) + float(params["D"][h]) * x
            np.testing.assert_allclose(y[b, h], ref, rtol=1e-13, atol=1e-15)


def pin_gdn_delta_rule_overwrite():
    """alpha = beta = 1 and a unit key: S_t k_t = v_t exactly (delta rule)."""
    w = TINY_GDN
    rng = np.random.default_rng(8)
    S = np.array(synth.initial_state(w, seed=8), np.float64)
    for _ in range(w.steps):
        kidx = rng.integers(0, w.N, (w.B, w.G))
        k = np.zeros((w.B, w.G, w.N), np.float32)
        for b in range(w.B):
            for g in range(w.G):
                k[b, g, kidx[b, g]] = 1.0
        kb = synth.to_bf16_bits(k)
        v = synth.to_bf16_bits(rng.standard_normal((w.B, w.H, w.P)).astype(np.float32))
        one = np.ones((w.B, w.H), np.float32)
        y = oracle.gdn_step(S, kb, kb, v, one, one)   # q = k, so y_t = S_t k_t
        np.testing.assert_array_equal(y, synth.bf16_bits_to_f32(v).astype(np.float64))


def pin_gdn_beta_zero_decays():
    """beta = 0: u = 0, S_t = gamma(t) S0, y_t = gamma(t) S0 q_t."""
    w = TINY_GDN
    params = synth.layer_params(w, seed=9)
    S0 = np.array(synth.initial_state(w, seed=9), np.float64)
    S = S0.copy()
    gamma = np.ones((w.B, w.H))
    ratio = w.H // w.G
    for s in range(w.steps):
        d = synth.step_inputs(w, s, seed=9, params=params)
        d["beta"] = np.zeros_like(d["beta"])
        y = oracle.gdn_step(S, d["q"], d["k"], d["v"], d["alpha"], d["beta"])
        gamma = gamma * d["alpha"].astype(np.float64)
        np.testing.assert_allclose(S, gamma[:, :, None, None] * S0, rtol=1e-13, atol=0)
        for b in range(w.B):
            for h in range(w.H):
                q = synth.bf16_bits_to_f32(d["q"][b, h // ratio]).astype(np.float64)
                np.testing.assert_allclose(y[b, h], gamma[b, h] * (S0[b, h] @ q), rtol=1e-12,
                                           atol=1e-15)


def pin_kda_uniform_decay_is_gdn():
    """A decay equal on every key channel is the scalar GDN decay: the
    per-channel recurrence then matches the (separately pinned) GDN one."""
    w = TINY_GDN
    params = synth.layer_params(w, seed=13)
    S0 = np.array(synth.initial_state(w, seed=13), np.float64)
    Sg, Sk = S0.copy(), S0.copy()
    for s in range(w.steps):
        d = synth.step_inputs(w, s, seed=13, params=params)
        a = np.ascontiguousarray(np.repeat(d["alpha"][:, :, None], w.N, axis=2))
        yg, ug = oracle.gdn_step(Sg, d["q"], d["k"], d["v"], d["alpha"], d["beta"], want_u=True)
        yk, uk = oracle.kda_step(Sk, d["q"], d["k"], d["v"], a, d["beta"], want_u=True)
        np.testing.assert_allclose(yk, yg, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(uk, ug, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(Sk, Sg, rtol=1e-12, atol=1e-15)


def pin_kda_beta_zero_decays_channels():
    """beta = 0: u = 0 and S_t = S0 diag(gamma(t)), gamma(t) the elementwise
    product of the decays; y_t = S0 (gamma(t) * q_t)."""
    w = TINY_KDA
    params = synth.layer_params(w, seed=14)
    S0 = np.array(synth.initial_state(w, seed=14), np.float64)
    S = S0.copy()
    gamma = np.ones((w.B, w.H, w.N))
    ratio = w.H // w.G
    for s in range(w.steps):
        d = synth.step_inputs(w, s, seed=14, params=params)
        y = oracle.kda_step(S, d["q"], d["k"], d["v"], d["alpha"], np.zeros_like(d["beta"]))
        gamma = gamma * d["alpha"].astype(np.float64)
        np.testing.assert_allclose(S, S0 * gamma[:, :, None, :], rtol=1e-13, atol=0)
        for b in range(w.B):
            for h in range(w.H):
                q = synth.bf16_bits_to_f32(d["q"][b, h // ratio]).astype(np.float64)
                np.testing.assert_allclose(y[b, h], S0[b, h] @ (gamma[b, h] * q), rtol=1e-12, atol=1e-15)


def pin_kda_zero_decay_clears_its_channel():
    """alpha_t = 0 on key channel m: column m of S_t is exactly u_t k_t[m]
    (the old column is forgotten before the rank-one update); with alpha = 1
    elsewhere and k_t[m'] = 0 on another channel m', column m' is unchanged."""
    w = TINY_KDA
    params = synth.layer_params(w, seed=15)
    S = np.array(synth.initial_state(w, seed=15), np.float64)
    ratio = w.H // w.G
    for s in range(w.steps):
        d = synth.step_inputs(w, s, seed=15, params=params)
        m, m2 = s % w.N, (s + 1) % w.N
        d["alpha"][:] = 1.0
        d["alpha"][:, :, m] = 0.0
        k = synth.bf16_bits_to_f32(d["k"]).copy()
        k[:, :, m2] = 0.0
        d["k"] = synth.to_bf16_bits(k)
        before = S.copy()
        _, u = oracle.kda_step(S, d["q"], d["k"], d["v"], d["alpha"], d["beta"], want_u=True)
        for b in range(w.B):
            for h in range(w.H):
                km = float(synth.bf16_bits_to_f32(d["k"][b, h // ratio])[m])
                np.testing.assert_array_equal(S[b, h, :, m], u[b, h] * km)
                np.testing.assert_array_equal(S[b, h, :, m2], before[b, h, :, m2])


def pin_hand_worked():
    with open(os.path.join(HERE, "golden", "hand_worked.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        S = np.array(c["S0"], np.float64)[None, None]
        for st in c["steps"]:
            if c["kind"] == "mamba2":
                y = oracle.mamba2_step(
                    S, synth.to_bf16_bits(np.array([[st["x"]]], np.float32)),
                    np.array([[st["dt"]]], np.float32), np.array([c["A"]], np.float32),
                    synth.to_bf16_bits(np.array([[st["B"]]], np.float32)),
                    synth.to_bf16_bits(np.array([[st["C"]]], np.float32)),
                    np.array([c["D"]], np.float32))
            else:
                bits = lambda a: synth.to_bf16_bits(np.array([[a]], np.float32))
                step = oracle.gdn_step if c["kind"] == "gdn" else oracle.kda_step
                y, u = step(S, bits(st["q"]), bits(st["k"]), bits(st["v"]),
                            np.array([[st["alpha"]]], np.float32),
                            np.array([[st["beta"]]], np.float32), want_u=True)
                np.testing.assert_array_equal(u[0, 0], st["u"])
            np.testing.assert_array_equal(S[0, 0], np.array(st["S"], np.float64))
            np.testing.assert_array_equal(y[0, 0], st["y"])


# ----------------------------------------------------------------------------- speculative rounds
def _spec_check(kind):
    w = {"mamba2": TINY_M2, "gdn": TINY_GDN, "kda": TINY_KDA}[kind].with_(T=3, capacity=7, accept="uniform")
    params = synth.layer_params(w, seed=10)
    S0 = synth.initial_state(w, seed=10)
    spec = oracle.Model(kind, S0, params)
    ref = oracle.Model(kind, S0, params)
    for r in range(4):
        d = synth.round_inputs(w, r, seed=10, params=params)
        if r == 1:
            d["accepted"][:] = 0
        before = spec.S.copy()
        y = spec.spec_round(d)
        # outputs equal standard steps over all T drafts from the committed state
        for b in range(w.B):
            run = oracle.Model(kind, before[b:b + 1], params)
            for i in range(w.T):
                di = {k: np.ascontiguousarray(v[b:b + 1, i]) for k, v in d.items()
                      if k != "accepted"}
                np.testing.assert_array_equal(run.step(di)[0], y[b, i])
                if i + 1 == d["accepted"][b]:
                    committed = run.S.copy()
            if d["accepted"][b] == 0:
                committed = before[b:b + 1]
                np.testing.assert_array_equal(spec.S[b], before[b])   # a = 0: unchanged
            np.testing.assert_array_equal(spec.S[b:b + 1], committed)
        # committing a drafts equals recomputing standard steps over the prefix
        for b in range(w.B):
            for i in range(d["accepted"][b]):
                di = {k: np.ascontiguousarray(v[b:b + 1, i]) for k, v in d.items()
                      if k != "accepted"}
                sub = oracle.Model(kind, ref.S[b:b + 1], params)
                sub.step(di)
                ref.S[b] = sub.S[0]
        np.testing.assert_array_equal(spec.S, ref.S)


def pin_spec_mamba2():
    _spec_check("mamba2")


def pin_spec_gdn():
    _spec_check("gdn")


def pin_spec_kda():
    _spec_check("kda")


def pin_spec_t1_all_accepted_is_standard():
    w = TINY_M2.with_(T=1, capacity=5, accept="uniform")
    params = synth.layer_params(w, seed=11)
    S0 = synth.initial_state(w, seed=11)
    spec, std = oracle.Model("mamba2", S0, params), oracle.Model("mamba2", S0, params)
    for r in range(5):
        d = synth.round_inputs(w, r, seed=11)
        d["accepted"][:] = 1
        y = spec.spec_round(d)
        ys = std.step({k: np.ascontiguousarray(v[:, 0]) for k, v in d.items() if k != "accepted"})
        np.testing.assert_array_equal(y[:, 0], ys)
        np.testing.assert_array_equal(spec.S, std.S)


PINS = [pin_unrolled_mamba2, pin_unrolled_gdn, pin_mamba2_alpha_one_is_matmul,
        pin_mamba2_alpha_zero_forgets, pin_mamba2_single_step_from_zero,
        pin_gdn_delta_rule_overwrite, pin_gdn_beta_zero_decays, pin_hand_worked,
        pin_spec_mamba2, pin_spec_gdn, pin_spec_t1_all_accepted_is_standard,
        pin_unrolled_kda, pin_kda_uniform_decay_is_gdn, pin_kda_beta_zero_decays_channels,
        pin_kda_zero_decay_clears_its_channel, pin_spec_kda]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


# ----------------------------------------------------------------------------- planted mistakes
MUTATIONS = {
    "mamba2_no_decay": ("row[n] = alpha * row[n] + v * bf16(kb[n]);",
                        "row[n] = row[n] + v * bf16(kb[n]);"),
    "mamba2_no_skip_term": ("y[p] = acc + D * bf16(x[p]);", "y[p] = acc;"),
    "mamba2_wrong_group": ("const int g = h / hpg;\n            const size_t bh",
                           "const int g = h % G;\n            const size_t bh"),
    "mamba2_dt_not_in_v": ("const double v = dt * bf16(x[p]);", "const double v = bf16(x[p]);"),
    "gdn_sign": ("const double u = beta * (bf16(vb[p]) - alpha * sk);",
                 "const double u = beta * (bf16(vb[p]) + alpha * sk);"),
    "gdn_q_k_swapped": ("for (int n = 0; n < N; ++n) sk += row[n] * bf16(kb[n]);",
                        "for (int n = 0; n < N; ++n) sk += row[n] * bf16(qb[n]);"),
    "gdn_no_beta": ("const double u = beta * (bf16(vb[p]) - alpha * sk);",
                    "const double u = (bf16(vb[p]) - alpha * sk);"),
    "gdn_old_state_in_output": ("row[n] = alpha * row[n] + u * bf16(kb[n]);\n            acc += row[n] * bf16(qb[n]);",
                                "acc += row[n] * bf16(qb[n]);\n            row[n] = alpha * row[n] + u * bf16(kb[n]);"),
    "spec_off_by_one": ("if (i + 1 == accepted[b]) memcpy(s, work",
                        "if (i == accepted[b]) memcpy(s, work"),
    "kda_no_decay": ("row[n] *= (double)alpha[n];\n            dk += row[n] * bf16(kb[n]);",
                     "dk += row[n] * bf16(kb[n]);"),
    "kda_u_from_undecayed": ("row[n] *= (double)alpha[n];\n            dk += row[n] * bf16(kb[n]);",
                             "dk += row[n] * bf16(kb[n]);\n            row[n] *= (double)alpha[n];"),
    "kda_channel_reversed": ("row[n] *= (double)alpha[n];", "row[n] *= (double)alpha[N - 1 - n];"),
    "kda_decay_by_value_index": ("row[n] *= (double)alpha[n];", "row[n] *= (double)alpha[p];"),
    "kda_no_beta": ("const double u = beta * (bf16(vb[p]) - dk);", "const double u = (bf16(vb[p]) - dk);"),
    "kda_q_for_k": ("dk += row[n] * bf16(kb[n]);", "dk += row[n] * bf16(qb[n]);"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_planted_mistakes(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = MUTATIONS[name]
    assert old in src, f"mutation anchor not found: {name}"
    (tmp_path / "oracle.c").write_text(src.replace(old, new))
    lib = str(tmp_path / "libmut.so")
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11",
                           str(tmp_path / "oracle.c"), "-o", lib, "-lm"])
    failed = []
    oracle.use_library(lib)
    try:
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                failed.append(pin.__name__)
    finally:
        oracle.use_library(None)
    assert failed, f"no pin caught the planted mistake {name}"

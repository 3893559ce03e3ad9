"""The replay form in fp32 meets the parity tolerance against the fp64 oracle.

A plain numpy model of what the method computes ("ReplaySSM: Cache SSM
Inputs, Not State", section "How it works"): each output comes from the
checkpoint and the buffered records, S_c is only rewritten when L records
have been buffered, and everything is held in fp32 (records, decays,
checkpoint), as a GPU kernel would.  Over several windows it must stay within
the 2e-3 normwise tolerance of the fp64 eager oracle, for the two families
and for the per-channel decay whose kernel comes next; this checks that the
tolerance is reachable in fp32 on these input recipes, independently of any
kernel.  (Not the oracle: a second, fp32 computation used only here.)
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from rs_decode_gb300 import synth

TOL = 2e-3


def _bf(bits) -> np.ndarray:
    return synth.bf16_bits_to_f32(bits).astype(np.float32)


class ReplayFp32:
    """Checkpoint + record buffer of one layer, fp32 throughout.  Decays are
    (B, H, 1) for a scalar per head, (B, H, N) for one per key channel."""

    def __init__(self, kind: str, S0: np.ndarray, L: int, params: dict):
        self.kind, self.L, self.params = kind, L, params
        self.Sc = S0.astype(np.float32).copy()          # [B, H, P, N]
        self.recs = []                                   # (alpha, v or u, k), fp32

    def _decays(self, alpha_t):
        """gamma and w_j for the records so far plus this step's decay."""
        alphas = [a for a, _, _ in self.recs] + [alpha_t]
        suffix = [np.ones_like(alpha_t)]
        for a in reversed(alphas[1:]):
            suffix.append(suffix[-1] * a)
        suffix.reverse()                                 # suffix[j] = prod of alphas after j
        gamma = suffix[0] * alphas[0]
        return gamma, suffix[:-1]                        # w_j for the buffered records

    def _dot_state(self, gamma, ws, vec):
        """(gamma S_c + sum_j w_j v_j k_j^T) vec with per-channel or scalar decays."""
        out = np.einsum("bhpn,bhn->bhp", self.Sc, gamma * vec)
        for (_, v, k), w in zip(self.recs, ws):
            out += v * np.sum(w * k * vec, axis=-1, keepdims=True)
        return out

    def step(self, d: dict) -> np.ndarray:
        B, H = self.Sc.shape[:2]
        if self.kind == "mamba2":
            hpg = H // d["Bm"].shape[1]
            k = np.repeat(_bf(d["Bm"]), hpg, axis=1)
            q = np.repeat(_bf(d["Cm"]), hpg, axis=1)
            dt = d["dt"].astype(np.float32)[:, :, None]
            alpha = np.exp(dt * self.params["A"].astype(np.float32)[None, :, None])
            v = dt * _bf(d["x"])
            self.recs.append((alpha, v, k))
            gamma, ws = self._decays_all()
            y = self._dot_state(gamma, ws, q) + self.params["D"].astype(np.float32)[None, :, None] * _bf(d["x"])
        else:
            ratio = H // d["k"].shape[1]
            k = np.repeat(_bf(d["k"]), ratio, axis=1)
            q = np.repeat(_bf(d["q"]), ratio, axis=1)
            a = d["alpha"].astype(np.float32)
            alpha = a if a.ndim == 3 else a[:, :, None]
            gamma, ws = self._decays(alpha)
            dk = self._dot_state(gamma, ws, k)           # (S_{t-1} diag(alpha_t)) k_t
            u = d["beta"].astype(np.float32)[:, :, None] * (_bf(d["v"]) - dk)
            self.recs.append((alpha, u, k))
            gamma, ws = self._decays_all()
            y = self._dot_state(gamma, ws, q)
        if len(self.recs) >= self.L:                     # the window is full: fold
            gamma, ws = self._decays_all()
            S = self.Sc * self._fold_gamma(gamma)[:, :, None, :]
            for (_, v, kk), w in zip(self.recs, ws):
                S += v[..., None] * (w * kk)[:, :, None, :]
            self.Sc, self.recs = S.astype(np.float32), []
        return y

    def _fold_gamma(self, gamma):
        return gamma

    def _decays_all(self):
        """gamma and w_j when every decay is already a record."""
        alphas = [a for a, _, _ in self.recs]
        ws = [np.ones_like(alphas[-1])]
        for a in reversed(alphas[1:]):
            ws.append(ws[-1] * a)
        ws.reverse()
        return ws[0] * alphas[0], ws


class FoldWithoutDecay(ReplayFp32):
    """Negative control: a fold that forgets to decay the old checkpoint."""

    def _fold_gamma(self, gamma):
        return np.ones_like(gamma)


def _worst(kind: str, model) -> float:
    base = {"mamba2": synth.WORKLOADS["mamba2"], "gdn": synth.WORKLOADS["gdn"], "kda": synth.WORKLOADS["kda"]}[kind]
    w = base.with_(B=2, H=8, G=2, P=32, N=64, L=16)
    params = synth.layer_params(w, seed=21)
    S0 = synth.initial_state(w, seed=21)
    ref = oracle.Model(kind, S0, params)
    rep = model(kind, S0, w.L, params)
    worst = 0.0
    for s in range(3 * w.L + 5):                        # three folds and a partial window
        d = synth.step_inputs(w, s, seed=21, params=params)
        y_ref, y = ref.step(d), rep.step(d)
        err = np.max(np.abs(y - y_ref).reshape(w.B, -1), axis=1) / np.max(np.abs(y_ref).reshape(w.B, -1), axis=1)
        worst = max(worst, float(err.max()))
    return worst


@pytest.mark.parametrize("kind", ["mamba2", "gdn", "kda"])
def test_fp32_replay_form_within_tolerance(kind):
    worst = _worst(kind, ReplayFp32)
    assert 0.0 < worst <= TOL, worst                     # fp32 differs from fp64, within the tolerance
    assert _worst(kind, FoldWithoutDecay) > 10 * TOL     # and the check can fail

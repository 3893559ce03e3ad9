"""GPU parity of the per-channel decay (RS_KDA) against the fp64 oracle.

The layer is Gated DeltaNet with one decay per key channel, the reading of
Kimi Delta Attention that "ReplaySSM: Cache SSM Inputs, Not State", section
"Limits", names as compatible without defining: D_t = S_{t-1} diag(alpha_t),
u_t = beta_t (v_t - D_t k_t), S_t = D_t + u_t k_t^T, y_t = S_t q_t.  Standard
decode (with the fused fold), speculative rounds in every draft bucket,
forced flush and materialise, the eager baseline, and the full-size workload
in the benchmark's launch configuration.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from harness import (TOL_HP, HeadErr, StandardRun, gpu_params, parity_sample, rel_err, state_errs,
                     state_gpu_to_np, state_np_to_gpu)
from rs_decode_gb300 import binding as rb
from rs_decode_gb300 import synth
from rs_decode_gb300.layer import to_device
from test_gpu_decode import _run_standard
from test_gpu_spec import _run_spec

pytestmark = pytest.mark.gpu

KDA = synth.WORKLOADS["kda"]


def test_kda_small_batch():
    _, _, flushes = _run_standard(KDA.with_(B=4), 36, seed=31)
    assert flushes == 2


def test_kda_small_slabs():
    w = synth.Workload("kda64", "kda", B=5, H=4, G=2, P=64, N=64, L=4, steps=11, init_std=0.3)
    _run_standard(w, 11, seed=32)


def test_kda_long_window():
    """A 32-record window: the fold gathers its coefficients in several
    chunks and keeps the partial sums in the staged blocks between them."""
    _run_standard(KDA.with_(B=3, L=32), 40, seed=33)


def test_kda_forced_flush_and_materialize():
    run = StandardRun(KDA.with_(B=2), seed=34)
    for s in range(21):
        y, y_ref, _ = run.step()
        assert rel_err(y, y_ref).max() <= TOL_HP
        if s in (3, 11, 12):
            run.layer.flush()
            run.ptr.flush()
            assert (run.layer.pointers()["h"] == 0).all()
            assert rel_err(run.checkpoint(), run.model.S).max() <= TOL_HP
    assert rel_err(run.materialized(), run.model.S).max() <= TOL_HP
    assert run.layer.status() == 0


def test_kda_full_batch_full_length():
    """B = 256 in the benchmark's launch configuration, all 256 steps; the
    oracle recomputes 64 sampled sequences: outputs every step (per sequence,
    and per head over the run), the checkpoint at every fold, the committed
    state at every fifth step."""
    idx = parity_sample(KDA.B)
    run = StandardRun(KDA, seed=0, sample=idx)
    heads = HeadErr(KDA.H)
    folds = 0
    for s in range(KDA.steps):
        y, y_ref, folded = run.step()
        e = rel_err(y, y_ref).max()
        assert e <= TOL_HP, f"step {s}: outputs rel err {e:.3e}"
        heads.add(y, y_ref)
        if folded:
            folds += 1
            per_seq, per_head = state_errs(run.layer.checkpoint_hp(), run.model.S, idx)
            assert max(per_seq.max(), per_head.max()) <= TOL_HP, f"step {s}: flushed checkpoint"
        if s % 5 == 4:
            per_seq, per_head = state_errs(run.layer.materialize(), run.model.S, idx)
            assert max(per_seq.max(), per_head.max()) <= TOL_HP, f"step {s}: committed state"
    assert folds == KDA.steps // KDA.L
    assert heads.worst() <= TOL_HP, f"outputs per head: rel err {heads.worst():.3e}"
    assert run.layer.status() == 0


@pytest.mark.parametrize("T", [1, 2, 3, 4, 8])
def test_kda_spec_rounds(T):
    """Verify T drafts + commit (draft buckets 1, 3, 4 and 8), folds of the
    committed records before acceptance, against the oracle's round."""
    w = KDA.with_(B=4, T=T, capacity=16 + T, steps=12, accept="binomial0.7")
    _, nfold, _ = _run_spec(w, 30 if T <= 2 else 12, seed=40 + T)
    assert nfold > 0


def test_kda_eager_step():
    w = KDA.with_(B=3)
    params = synth.layer_params(w, 35)
    S0 = synth.initial_state(w, 35)
    S = state_np_to_gpu(S0)
    model = oracle.Model("kda", S0, params)
    desc = rb.make_desc(rb.KDA, w.B, w.H, w.G, w.P, w.N, w.L)
    y = torch.empty(w.B, w.H, w.P, device="cuda")
    for s in range(20):
        d = synth.step_inputs(w, s, 35, params)
        dd = to_device(d)
        rb.rs_eager_step_kda(desc, S, dd["q"], dd["k"], dd["v"], dd["alpha"], dd["beta"], y)
        y_ref = model.step(d)
        assert rel_err(y.cpu().numpy(), y_ref).max() <= TOL_HP
        assert rel_err(state_gpu_to_np(S), model.S).max() <= TOL_HP

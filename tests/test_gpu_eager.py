"""GPU parity of the eager baselines (load-update-store decode and per-draft
snapshots) against the fp64 oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from harness import TOL_HP, gpu_params, rel_err, state_gpu_to_np, state_np_to_gpu
from rs_decode_gb300 import binding as rb
from rs_decode_gb300 import synth
from rs_decode_gb300.layer import to_device

pytestmark = pytest.mark.gpu


def _desc(w, T_max=0):
    k = rb.MAMBA2 if w.kind == "mamba2" else rb.GDN
    return rb.make_desc(k, w.B, w.H, w.G, w.P, w.N, w.L, T_max, w.L + T_max)


@pytest.mark.parametrize("name", ["tiny", "mamba2", "gdn"])
def test_eager_step(name):
    w = synth.WORKLOADS[name].with_(B=min(synth.WORKLOADS[name].B, 3))
    params = synth.layer_params(w, 11)
    S0 = synth.initial_state(w, 11)
    S = state_np_to_gpu(S0)
    model = oracle.Model(w.kind, S0, params)
    gp = gpu_params(w, params)
    desc = _desc(w)
    y = torch.empty(w.B, w.H, w.P, device="cuda")
    for s in range(20):
        d = synth.step_inputs(w, s, 11, params)
        dd = to_device(d)
        if w.kind == "mamba2":
            rb.rs_eager_step_mamba2(desc, S, dd["x"], dd["dt"], gp["A"], dd["Bm"], dd["Cm"], gp["D"], y)
        else:
            rb.rs_eager_step_gdn(desc, S, dd["q"], dd["k"], dd["v"], dd["alpha"], dd["beta"], y)
        y_ref = model.step(d)
        assert rel_err(y.cpu().numpy(), y_ref).max() <= TOL_HP
        assert rel_err(state_gpu_to_np(S), model.S).max() <= TOL_HP


@pytest.mark.parametrize("name", ["mamba2_spec", "gdn_spec"])
def test_eager_snapshots(name):
    w = synth.WORKLOADS[name].with_(B=4)
    params = synth.layer_params(w, 12)
    S0 = synth.initial_state(w, 12)
    model = oracle.Model(w.kind, S0, params)
    gp = gpu_params(w, params)
    desc = _desc(w, w.T)
    slots = w.T + 1
    pool = torch.zeros(w.B, slots, w.H, w.N, w.P, device="cuda")
    pool[:, 0] = state_np_to_gpu(S0)
    cur = torch.zeros(w.B, dtype=torch.int32, device="cuda")
    y = torch.empty(w.B, w.T, w.H, w.P, device="cuda")
    for r in range(8):
        d = synth.round_inputs(w, r, 12, params)
        dd = to_device(d)
        ins = (rb.make_inputs(x=dd["x"], dt=dd["dt"], A=gp["A"], Bm=dd["Bm"], Cm=dd["Cm"], D=gp["D"])
               if w.kind == "mamba2" else
               rb.make_inputs(q=dd["q"], k=dd["k"], v=dd["v"], alpha=dd["alpha"], beta=dd["beta"]))
        rb.rs_eager_verify_snapshots(desc, pool, cur, w.T, ins, y)
        rb.rs_eager_select(desc, cur, dd["accepted"])
        y_ref = model.spec_round(d)
        assert rel_err(y.cpu().numpy().reshape(w.B, -1), y_ref.reshape(w.B, -1)).max() <= TOL_HP
        c = cur.cpu().numpy()
        got = np.stack([state_gpu_to_np(pool[b, c[b]][None])[0] for b in range(w.B)])
        assert rel_err(got, model.S).max() <= TOL_HP

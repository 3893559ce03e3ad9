"""rs_decode_mamba2_noalloc: Mamba-2 decode for callers that cannot allocate.

Some callers can give the library nothing beyond inputs, outputs and the layer
state: an engine plugin that only receives pre-planned tensors, or a server
that forbids device allocation after start-up.  This entry point keeps the
kernel's per-sequence arrival counters in a static device array of the
library.  These tests check that it gives the same outputs as
rs_decode_mamba2 on two consecutive calls and that it rejects a batch above
its static limit.  The file is named so that pytest collects it last.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from harness import TOL_HP, gpu_params, rel_err, state_np_to_gpu
from rs_decode_gb300 import binding as rb
from rs_decode_gb300 import synth
from rs_decode_gb300.layer import Layer, to_device


def test_batch_above_static_limit_is_rejected():
    lib = rb.load()
    d = rb.make_desc(rb.MAMBA2, rb.STATIC_MAX_SEQS + 1, 8, 1, 64, 128, 16)
    st = rb.State()
    status = lib.rs_decode_mamba2_noalloc(ctypes.byref(d), ctypes.byref(st), *([None] * 8))
    assert rb.STATUS[status] == "RS_ERR_STATIC_LIMIT"
    assert "static" in rb.rs_status_string(status)


@pytest.mark.gpu
def test_noalloc_matches_rs_decode_mamba2_on_two_calls():
    w = synth.WORKLOADS["mamba2"].with_(B=8)
    params = synth.layer_params(w, 21)
    S0 = state_np_to_gpu(synth.initial_state(w, 21))
    gp = gpu_params(w, params)
    ref = Layer("mamba2", w.B, w.H, w.G, w.P, w.N, w.L)
    new = Layer("mamba2", w.B, w.H, w.G, w.P, w.N, w.L)
    ref.init(S0)
    new.init(S0)
    st = rb.State.from_buffer_copy(new.state)
    st.arrive = None  # the entry point brings its own counters
    for step in range(2):
        d = to_device(synth.step_inputs(w, step, 21))
        y_ref = ref.decode(d, gp)
        y_new = torch.empty_like(y_ref)
        rb.rs_decode_mamba2_noalloc(new.desc, st, d["x"], d["dt"], gp["A"], d["Bm"], d["Cm"], gp["D"], y_new)
        torch.cuda.synchronize()
        err = rel_err(y_new.cpu().numpy(), y_ref.cpu().numpy()).max()
        assert err <= TOL_HP, f"call {step}: rel err {err:.3e}"
        pr, pn = ref.pointers(), new.pointers()
        assert all(np.array_equal(pr[k], pn[k]) for k in pr)
    assert new.status() == 0 and ref.status() == 0

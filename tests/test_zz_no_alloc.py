"""rs_decode_mamba2_noalloc: Mamba-2 decode for callers that cannot allocate.

Some callers can give the library nothing beyond inputs, outputs and the layer
state: an engine plugin that only receives pre-planned tensors, or a server
that forbids device allocation after start-up.  This entry point keeps the
kernel's per-sequence arrival counters in a static device array of the
library.  These tests check that, over more calls than a window holds (so
that the window's last call folds the records into the checkpoint), its
outputs and checkpoint match both the fp64 oracle and rs_decode_mamba2, also
when a second, smaller layer's calls share the static array in between; and
that it rejects a batch above its static limit.  The file is named so that
pytest collects it last.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
from harness import TOL_HP, HeadErr, gpu_params, rel_err, state_errs, state_np_to_gpu
from oracle.pointers import Pointers
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


class _Pair:
    """One workload decoded three ways on the same inputs: rs_decode_mamba2,
    rs_decode_mamba2_noalloc (the state's arrival counters unset) and the
    oracle."""

    def __init__(self, w, seed):
        self.w, self.seed, self.t = w, seed, 0
        self.params = synth.layer_params(w, seed)
        S0 = synth.initial_state(w, seed)
        self.gp = gpu_params(w, self.params)
        self.ref = Layer("mamba2", w.B, w.H, w.G, w.P, w.N, w.L)
        self.new = Layer("mamba2", w.B, w.H, w.G, w.P, w.N, w.L)
        self.ref.init(state_np_to_gpu(S0))
        self.new.init(state_np_to_gpu(S0))
        self.st = rb.State.from_buffer_copy(self.new.state)
        self.st.arrive = None  # the entry point brings its own counters
        self.model = oracle.Model("mamba2", S0, self.params)
        self.ptr = Pointers(w.L, w.cap)
        self.heads = {k: HeadErr(w.H) for k in ("rs_decode_mamba2", "noalloc", "noalloc vs rs_decode_mamba2")}

    def call(self):
        w, gp = self.w, self.gp
        d = synth.step_inputs(w, self.t, self.seed)
        dd = to_device(d)
        y_ref = self.ref.decode(dd, gp)
        y_new = torch.empty_like(y_ref)
        rb.rs_decode_mamba2_noalloc(self.new.desc, self.st, dd["x"], dd["dt"], gp["A"], dd["Bm"], dd["Cm"],
                                    gp["D"], y_new)
        y_or = self.model.step(d)
        folded = self.ptr.standard_step()
        torch.cuda.synchronize()
        y_new, y_ref = y_new.cpu().numpy(), y_ref.cpu().numpy()
        tag = f"B={w.B} call {self.t}"
        for got, what in ((y_ref, "rs_decode_mamba2"), (y_new, "noalloc")):
            e = rel_err(got, y_or).max()
            assert e <= TOL_HP, f"{tag}: {what} vs oracle rel err {e:.3e}"
            self.heads[what].add(got, y_or)
        e = rel_err(y_new, y_ref).max()
        assert e <= TOL_HP, f"{tag}: noalloc vs rs_decode_mamba2 rel err {e:.3e}"
        self.heads["noalloc vs rs_decode_mamba2"].add(y_new, y_ref)
        pr, pn = self.ref.pointers(), self.new.pointers()
        assert all(np.array_equal(pr[k], pn[k]) for k in pr), tag
        assert (pn["h"] == self.ptr.h).all() and (pn["base"] == self.ptr.base).all(), tag
        if folded:
            idx = np.arange(w.B)
            for lay, what in ((self.new, "noalloc"), (self.ref, "rs_decode_mamba2")):
                per_seq, per_head = state_errs(lay.checkpoint_hp(), self.model.S, idx)
                assert max(per_seq.max(), per_head.max()) <= TOL_HP, f"{tag}: {what} flushed checkpoint"
            ck = rel_err(self.new.checkpoint_hp().cpu().numpy(), self.ref.checkpoint_hp().cpu().numpy()).max()
            assert ck <= TOL_HP, f"{tag}: noalloc checkpoint vs rs_decode_mamba2 {ck:.3e}"
        self.t += 1
        return folded


@pytest.mark.gpu
def test_noalloc_matches_oracle_and_rs_decode_mamba2_across_a_fold():
    """L + 3 calls on an 8-sequence layer (a fold on call L), with a
    3-sequence layer's calls interleaved from call 5 on: both layers use the
    one static counter array, one after the other on the same stream."""
    big = _Pair(synth.WORKLOADS["mamba2"].with_(B=8), 21)
    small = _Pair(synth.WORKLOADS["mamba2"].with_(B=3, L=4), 22)
    folds = {"big": 0, "small": 0}
    for c in range(big.w.L + 3):
        folds["big"] += bool(big.call())
        if c >= 5:
            folds["small"] += bool(small.call())
    assert folds["big"] == 1 and folds["small"] >= 3
    for p in (big, small):
        assert p.new.status() == 0 and p.ref.status() == 0
        for what, acc in p.heads.items():
            assert acc.worst() <= TOL_HP, f"B={p.w.B}: {what} per head rel err {acc.worst():.3e}"

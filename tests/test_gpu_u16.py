"""GPU parity of Gated DeltaNet records that keep the correction term u in
bf16 (RS_U_BF16), against the fp64 oracle, and its error next to the fp32-u
buffer on the same inputs.

"ReplaySSM: Cache SSM Inputs, Not State", section "How it works", Gated
DeltaNet bullet: each record stores u_j in place of v_j; the pages do not say
in which precision.  With u in bf16, outputs and folds read rounded u, so their
bound is the one for values read from bf16 (3e-2); the fp32 buffer keeps 2e-3.
With RS_REPORT_DIR set, the full-size comparison is written there as JSON.
"""
from __future__ import annotations

import json
import os

import numpy as np
import pytest

from harness import (TOL_HP, TOL_LP, HeadErr, SpecRun, StandardRun, parity_sample, rel_err, state_errs)
from rs_decode_gb300 import synth, traffic

pytestmark = pytest.mark.gpu


def _decode(w, precision, steps, seed, idx=None):
    """Per-(step, sequence) output errors and the flushed checkpoints' errors."""
    run = StandardRun(w, seed=seed, precision=precision, sample=idx)
    heads = HeadErr(w.H)
    e, ck = [], []
    for _ in range(steps):
        y, y_ref, folded = run.step()
        e.append(rel_err(y, y_ref))
        heads.add(y, y_ref)
        if folded:
            ck.append(state_errs(run.layer.checkpoint_hp(), run.model.S, run.idx)[0])
    assert run.layer.status() == 0
    return np.array(e), np.array(ck), heads.worst()


def test_gdn_u16_decode_small_batch():
    w = synth.WORKLOADS["gdn"].with_(B=4)
    e16, ck16, h16 = _decode(w, "fp32+u16", 36, 51)
    e32, ck32, h32 = _decode(w, "fp32", 36, 51)
    assert e16.max() <= TOL_LP and ck16.max() <= TOL_LP and h16 <= TOL_LP
    assert e32.max() <= TOL_HP and ck32.max() <= TOL_HP and h32 <= TOL_HP
    assert e16.mean() > e32.mean()  # rounding u costs accuracy, as it must


def test_gdn_u16_spec_two_precision():
    """Two-precision speculative rounds with bf16 u: outputs, folded
    checkpoints and committed states within the bf16-read bound."""
    w = synth.WORKLOADS["gdn_spec"].with_(B=6, precision="two+u16")
    run = SpecRun(w, seed=52)
    nfold = 0
    for r in range(16):
        y, y_ref, folded, S_before, _ = run.round()
        e = rel_err(y.reshape(w.B, -1), y_ref.reshape(w.B, -1))
        assert e.max() <= TOL_LP, f"round {r}: {e.max():.3e}"
        if folded.any():
            nfold += int(folded.sum())
            per_seq, _ = state_errs(run.layer.checkpoint_hp(), S_before, run.idx)
            assert per_seq[folded].max() <= TOL_LP
        per_seq, _ = state_errs(run.layer.materialize(), run.model.S, run.idx)
        assert per_seq.max() <= TOL_LP
    assert nfold > 0 and run.layer.status() == 0


def test_gdn_u16_full_batch_report():
    """The gdn workload at full batch (B = 256), 64 steps (four folds), 64
    sampled sequences, with u in fp32 and in bf16: both errors and the bytes
    each moves per step."""
    w = synth.WORKLOADS["gdn"]
    idx = parity_sample(w.B)
    e32, ck32, h32 = _decode(w, "fp32", 64, 0, idx)
    e16, ck16, h16 = _decode(w.with_(precision="fp32+u16"), "fp32+u16", 64, 0, idx)
    assert e32.max() <= TOL_HP and e16.max() <= TOL_LP and h16 <= TOL_LP
    stats = lambda e: {"mean": float(e.mean()), "max": float(e.max())}
    byts = {}
    for name, ub in (("fp32", 4), ("bf16", 2)):
        s = traffic.Shape("gdn", w.B, w.H, w.G, w.P, w.N, u_bytes=ub)
        byts[name] = sum(traffic.replay_step_bytes(s, h, h + 1 >= w.L) for h in range(w.L)) / w.L
    report = {"workload": f"gdn decode: B={w.B} H={w.H} G={w.G} P={w.P} N={w.N} L={w.L}, 64 steps, fp32 checkpoint",
              "sample": f"{len(idx)} sequences incl. 0 and {w.B - 1}",
              "metric": "per (step, sequence) normwise relative output error vs the fp64 oracle; checkpoints at folds",
              "test": "tests/test_gpu_u16.py::test_gdn_u16_full_batch_report",
              "u_fp32": {"outputs": stats(e32), "checkpoints": stats(ck32), "per_head_run": h32,
                         "bytes_per_step": byts["fp32"]},
              "u_bf16": {"outputs": stats(e16), "checkpoints": stats(ck16), "per_head_run": h16,
                         "bytes_per_step": byts["bf16"]}}
    print(json.dumps(report))
    out = os.environ.get("RS_REPORT_DIR")
    if out:
        os.makedirs(out, exist_ok=True)
        with open(os.path.join(out, "gdn_u16_output_error.json"), "w") as f:
            json.dump(report, f, indent=1)

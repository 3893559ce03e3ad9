"""GPU parity of speculative verification, commit and rollback against the
fp64 oracle (eager recurrence over the drafts, commit of the accepted prefix).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from harness import TOL_HP, TOL_LP, HeadErr, SpecRun, rel_err, state_gpu_to_np
from rs_decode_gb300 import synth

pytestmark = pytest.mark.gpu


def _run_spec(w, rounds, seed=0, precision=None, sample=None, accept=None, alpha_pow=None):
    run = SpecRun(w, seed=seed, precision=precision, sample=sample, alpha_pow=alpha_pow)
    prec = precision or w.precision
    errs, folds = [], []
    nfold = 0
    heads = HeadErr(w.H)
    for r in range(rounds):
        a = None if accept is None else accept(r, w.B)
        y, y_ref, folded, S_before, acc = run.round(a)
        e = rel_err(y.reshape(len(run.idx), -1), y_ref.reshape(len(run.idx), -1))
        tol = np.where(folded | (prec == "fp32"), TOL_HP, TOL_LP) if prec != "shared_bf16" else TOL_LP
        assert (e <= tol).all(), f"round {r}: verify rel err {e.max():.3e}"
        heads.add(y, y_ref)
        errs.append(e)
        folds.append(folded)
        if folded.any():
            nfold += int(folded.sum())
            ck = run.layer.checkpoint_hp()
            ck = ck if ck is not None else run.layer.checkpoint_lp_f32()
            got = state_gpu_to_np(ck[torch.from_numpy(run.idx).cuda()])
            ce = rel_err(got[folded], S_before[folded])
            assert ce.max() <= (TOL_HP if prec != "shared_bf16" else TOL_LP), f"round {r}: fold {ce.max():.3e}"
        if prec != "shared_bf16":
            m = rel_err(state_gpu_to_np(run.layer.materialize()[torch.from_numpy(run.idx).cuda()]), run.model.S)
            assert m.max() <= TOL_HP, f"round {r}: committed state rel err {m.max():.3e}"
    assert heads.worst() <= (TOL_HP if prec == "fp32" else TOL_LP), f"per-head rel err {heads.worst():.3e}"
    ptr = run.layer.pointers()
    assert (ptr["h"][run.idx] == [run.ptrs[b].h for b in run.idx]).all()
    assert (ptr["base"][run.idx] == [run.ptrs[b].base for b in run.idx]).all()
    assert run.layer.status() == 0
    return np.stack(errs), nfold, np.stack(folds)


def test_mamba2_spec_small_batch():
    w = synth.WORKLOADS["mamba2_spec"].with_(B=8)
    _, nfold, _ = _run_spec(w, 14, seed=1)
    assert nfold > 0


def test_gdn_spec_two_precision_small_batch():
    w = synth.WORKLOADS["gdn_spec"].with_(B=8)
    _, nfold, _ = _run_spec(w, 14, seed=2)
    assert nfold > 0


@pytest.mark.parametrize("kind", ["mamba2", "gdn"])
def test_two_precision_beats_shared_bf16(kind):
    """Separate precisions keep bf16 rounding out of the recurrence, so their
    output error does not exceed that of a shared bf16 checkpoint.  Until a
    sequence first folds, both arms read the same bf16 values (summed in a
    different order: tensor cores for the two-precision bf16 reads of GDN), so
    the comparison takes the rounds after each sequence's first fold, where
    the two-precision copy is a rounding of the fp32 fold and the shared one
    has carried bf16 rounding through it.  The GDN recipe's decays shrink a
    checkpoint to about 1e-5 of itself within one window, so that no rounding
    of it survives a window and the arms tie (to 1e-12 relative at B = 6);
    its decays are slowed here to alpha^(1/50), so that the checkpoint carries
    over windows as a slowly forgetting layer's does."""
    base = synth.WORKLOADS["gdn_spec" if kind == "gdn" else "mamba2_spec"].with_(B=6)
    ap = 0.02 if kind == "gdn" else None
    e_two, _, folds = _run_spec(base, 24, seed=3, precision="two", alpha_pow=ap)
    e_shared, _, folds_sh = _run_spec(base, 24, seed=3, precision="shared_bf16", alpha_pow=ap)
    assert np.array_equal(folds, folds_sh)
    first = np.where(folds.any(0), folds.argmax(0), len(folds))
    after = np.arange(len(folds))[:, None] > first[None, :]
    assert after.sum() >= len(folds) * base.B // 2
    assert np.mean(e_two[after]) <= np.mean(e_shared[after])


@pytest.mark.parametrize("kind", ["mamba2", "gdn"])
def test_spec_full_batch_sampled(kind):
    w = synth.WORKLOADS["gdn_spec" if kind == "gdn" else "mamba2_spec"]
    _run_spec(w, 6, seed=0, sample=[0, 3, 255, w.B - 1])


@pytest.mark.parametrize("T", [1, 2, 8])
def test_draft_counts(T):
    w = synth.WORKLOADS["tiny"].with_(B=3, T=T, capacity=16 + T, accept="uniform")
    _run_spec(w, 12, seed=4 + T)


def test_reject_everything_keeps_checkpoint():
    """a = 0 every round: nothing is committed, the checkpoint never changes."""
    w = synth.WORKLOADS["mamba2_spec"].with_(B=3)
    run = SpecRun(w, seed=5)
    ck0 = run.layer.checkpoint_hp().clone()
    for r in range(6):
        y, y_ref, folded, _, _ = run.round(np.zeros(w.B, np.int32))
        assert rel_err(y.reshape(w.B, -1), y_ref.reshape(w.B, -1)).max() <= TOL_HP
        assert not folded.any()
    assert torch.equal(run.layer.checkpoint_hp(), ck0)
    assert (run.layer.pointers()["h"] == 0).all()


def test_accept_all_equals_standard_decode():
    """T = 1 with every draft accepted reproduces standard decode outputs."""
    w = synth.WORKLOADS["tiny"].with_(B=2, T=1, capacity=17, accept="uniform")
    run = SpecRun(w, seed=6)
    for r in range(40):
        y, y_ref, _, _, _ = run.round(np.ones(w.B, np.int32))
        assert rel_err(y.reshape(w.B, -1), y_ref.reshape(w.B, -1)).max() <= TOL_HP


def test_rollback_then_verify_again():
    """rs_rollback discards drafts: re-verifying from the same committed state
    gives the same outputs."""
    from rs_decode_gb300.layer import to_device
    w = synth.WORKLOADS["mamba2_spec"].with_(B=2)
    run = SpecRun(w, seed=7)
    run.round()
    d = to_device(synth.round_inputs(w, 99, 7, run.params))
    y1 = run.layer.verify(w.T, d, run.gp).clone()
    run.layer.rollback()
    assert (run.layer.pointers()["nd"] == 0).all()
    y2 = run.layer.verify(w.T, d, run.gp)
    run.layer.rollback()
    assert torch.equal(y1, y2)
    assert run.layer.status() == 0


def test_bad_accept_sets_status_bit():
    from rs_decode_gb300 import binding as rb
    w = synth.WORKLOADS["mamba2_spec"].with_(B=2)
    run = SpecRun(w, seed=8)
    d = synth.round_inputs(w, 0, 8, run.params)
    from rs_decode_gb300.layer import to_device
    run.layer.verify(w.T, to_device(d), run.gp)
    run.layer.commit(torch.tensor([w.T + 3, -1], dtype=torch.int32, device="cuda"))
    assert run.layer.status() & rb.DEV_ACCEPT
    ptr = run.layer.pointers()
    assert list(ptr["h"]) == [w.T, 0] and (ptr["nd"] == 0).all()


@pytest.mark.parametrize("T", [2, 4, 8])
def test_gdn_draft_counts(T):
    """GDN rounds in every draft bucket (3, 4 and 8), fp32 checkpoint."""
    w = synth.WORKLOADS["gdn_spec"].with_(B=3, T=T, capacity=16 + T, precision="fp32", accept="uniform")
    _run_spec(w, 10, seed=13)


@pytest.mark.parametrize("T", [1, 3, 4, 8])
@pytest.mark.parametrize("precision", ["two", "shared_bf16"])
def test_gdn_draft_counts_bf16(T, precision):
    """GDN rounds in every draft bucket whose bf16 row blocks are dotted on the
    tensor cores (1, 3, 4 and 8 drafts: 2 to 16 vectors, one or two groups of
    the B operand), with folds of the fp32 or the bf16 copy."""
    w = synth.WORKLOADS["gdn_spec"].with_(B=4, T=T, capacity=16 + T, precision=precision, accept="uniform")
    _, nfold, _ = _run_spec(w, 40 if T == 1 else 12, seed=17 + T)
    assert nfold > 0

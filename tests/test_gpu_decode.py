"""GPU parity of standard decode (Mamba-2 and GDN) against the fp64 oracle.

Every check goes through the C ABI (librs.so via the ctypes binding).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from harness import TOL_HP, TOL_LP, HeadErr, StandardRun, rel_err, state_gpu_to_np, make_layer
from rs_decode_gb300 import synth

pytestmark = pytest.mark.gpu


def _run_standard(w, steps, seed=0, precision="fp32", sample=None, check_materialize=True):
    run = StandardRun(w, seed=seed, precision=precision, sample=sample)
    tol_y = TOL_HP if precision == "fp32" else TOL_LP
    worst_y = worst_ck = 0.0
    flushes = 0
    heads = HeadErr(w.H)
    for s in range(steps):
        y, y_ref, folded = run.step()
        e = rel_err(y, y_ref).max()
        # two-precision: flush steps read the fp32 copy
        tol = TOL_HP if (precision == "two" and folded) else tol_y
        assert e <= tol, f"step {s}: output rel err {e:.3e} > {tol}"
        heads.add(y, y_ref)
        worst_y = max(worst_y, e)
        if folded:
            flushes += 1
            ck = rel_err(run.checkpoint(), run.model.S).max()
            tol_ck = TOL_LP if precision == "shared_bf16" else TOL_HP  # a bf16 checkpoint
            assert ck <= tol_ck, f"step {s}: flushed checkpoint rel err {ck:.3e}"
            worst_ck = max(worst_ck, ck)
        if check_materialize:
            m = rel_err(run.materialized(), run.model.S).max()
            assert m <= TOL_HP, f"step {s}: materialised state rel err {m:.3e}"
    assert heads.worst() <= tol_y, f"outputs per head: rel err {heads.worst():.3e}"
    ptr = run.layer.pointers()
    assert (ptr["h"][run.idx] == run.ptr.h).all() and (ptr["base"][run.idx] == run.ptr.base).all()
    assert run.layer.status() == 0
    return worst_y, worst_ck, flushes


def test_tiny_mamba2_all_steps():
    """The tiny Mamba-2 workload: 48 steps, flushes at 16, 32, 48."""
    w = synth.WORKLOADS["tiny"]
    _, _, flushes = _run_standard(w, w.steps)
    assert flushes == 3


def test_mamba2_serving_shapes_small_batch():
    """Serving-scale head shapes (128 heads, 8 groups) at B=6, 40 steps."""
    w = synth.WORKLOADS["mamba2"].with_(B=6)
    _run_standard(w, 40, seed=1)


def test_gdn_small_batch():
    w = synth.WORKLOADS["gdn"].with_(B=4)
    _run_standard(w, 36, seed=2)


@pytest.mark.parametrize("kind", ["mamba2", "gdn"])
@pytest.mark.parametrize("precision", ["two", "shared_bf16"])
def test_low_precision_modes(kind, precision):
    w = synth.WORKLOADS[kind].with_(B=3)
    _run_standard(w, 34, seed=3, precision=precision, check_materialize=(precision == "two"))


@pytest.mark.parametrize("L", [1, 3, 32])
def test_window_sizes(L):
    w = synth.WORKLOADS["tiny"].with_(L=L, B=3)
    _run_standard(w, 2 * L + 3 if L < 32 else 40, seed=4)


def test_ragged_heads_single_head_ctas():
    """H/G odd: one head per CTA; B=1; N=64 slabs."""
    w = synth.Workload("odd", "mamba2", B=1, H=6, G=2, P=64, N=64, L=5, steps=12, init_std=0.3)
    _run_standard(w, 12, seed=5)


def test_gdn_small_slabs():
    w = synth.Workload("gdn64", "gdn", B=5, H=4, G=2, P=64, N=64, L=4, steps=11, init_std=0.3)
    _run_standard(w, 11, seed=6)


@pytest.mark.parametrize("kind", ["mamba2", "gdn"])
def test_full_batch_sampled(kind):
    """Full serving batch (B=256) in the benchmark's launch configuration;
    the oracle recomputes a sample of sequences one by one."""
    w = synth.WORKLOADS[kind]
    sample = [0, 1, 127, 200, 255]
    _run_standard(w, 20, seed=0, sample=sample, check_materialize=False)


def test_determinism():
    """Two runs on the same inputs give identical output bytes."""
    w = synth.WORKLOADS["mamba2"].with_(B=4)
    ys = []
    for _ in range(2):
        run = StandardRun(w, seed=7)
        ys.append(np.stack([run.step()[0] for _ in range(18)]))
    assert np.array_equal(ys[0], ys[1])


def test_forced_flush_and_materialize():
    """rs_flush at an arbitrary point folds the committed records; outputs
    and states stay equal to the eager recurrence."""
    w = synth.WORKLOADS["tiny"].with_(B=2)
    run = StandardRun(w, seed=8)
    for s in range(23):
        y, y_ref, _ = run.step()
        assert rel_err(y, y_ref).max() <= TOL_HP
        if s in (4, 9, 10):
            run.layer.flush()
            run.ptr.flush()
            assert (run.layer.pointers()["h"] == 0).all()
            assert rel_err(run.checkpoint(), run.model.S).max() <= TOL_HP
    assert rel_err(run.materialized(), run.model.S).max() <= TOL_HP


def test_append_then_decode():
    """rs_append records committed without outputs, then decode continues."""
    import oracle
    from rs_decode_gb300.layer import to_device
    from harness import gpu_params, state_np_to_gpu
    w = synth.WORKLOADS["tiny"].with_(B=3, init_std=0.2)
    params = synth.layer_params(w, 9)
    S0 = synth.initial_state(w, 9)
    layer = make_layer(w)
    layer.init(state_np_to_gpu(S0))
    model = oracle.Model("mamba2", S0, params)
    gp = gpu_params(w, params)
    n = 5
    recs = [synth.step_inputs(w, s, 9) for s in range(n)]
    stacked = {k: np.stack([r[k] for r in recs], axis=1) for k in ("x", "dt", "Bm")}
    layer.append(n, to_device(stacked), gp)
    for r in recs:
        model.step(r)
    assert (layer.pointers()["h"] == n).all()
    assert rel_err(state_gpu_to_np(layer.materialize()), model.S).max() <= TOL_HP
    for s in range(n, n + 14):
        d = synth.step_inputs(w, s, 9)
        y = layer.decode(to_device(d), gp).cpu().numpy()
        assert rel_err(y, model.step(d)).max() <= TOL_HP
    assert layer.status() == 0


@pytest.mark.parametrize("precision", ["fp32", "shared_bf16", "two"])
def test_gdn_long_window(precision):
    """GDN with a 32-record window: a fold takes the coefficients of its 32
    records in several gathers (fp32 checkpoints keep the partial sums in the
    staged blocks between gathers, bf16 ones in registers).  Two-precision
    runs the tensor-core kernel: bf16 steps on the tensor cores, the flush step
    on the fp32 copy with the several-gather fold."""
    w = synth.WORKLOADS["gdn"].with_(B=3, L=32)
    _run_standard(w, 40, seed=11, precision=precision, check_materialize=(precision != "shared_bf16"))


def test_gdn_forced_flush_and_materialize():
    """rs_flush and rs_materialize on GDN layers (fold-only launches)."""
    w = synth.WORKLOADS["gdn"].with_(B=2)
    run = StandardRun(w, seed=12)
    for s in range(21):
        y, y_ref, _ = run.step()
        assert rel_err(y, y_ref).max() <= TOL_HP
        if s in (3, 11, 12):
            run.layer.flush()
            run.ptr.flush()
            assert (run.layer.pointers()["h"] == 0).all()
            assert rel_err(run.checkpoint(), run.model.S).max() <= TOL_HP
    assert rel_err(run.materialized(), run.model.S).max() <= TOL_HP


def test_small_batch_kernel_and_pipeline_share_the_state():
    """At B = 8, standard steps of the fp32 Mamba-2 layer run on the
    small-batch kernel and verify rounds on the streaming pipeline, so each
    reads records, pointers and checkpoints that the other wrote: standard
    steps, rounds of 4 drafts with commits, and standard steps again across
    folds, all against the oracle."""
    import oracle
    from harness import gpu_params, state_np_to_gpu
    from oracle.pointers import Pointers
    from rs_decode_gb300.layer import to_device

    w = synth.WORKLOADS["mamba2_spec"].with_(B=8)
    seed = 9
    params = synth.layer_params(w, seed)
    gp = gpu_params(w, params)
    S0 = synth.initial_state(w, seed)
    layer = make_layer(w)
    layer.init(state_np_to_gpu(S0))
    model = oracle.Model(w.kind, S0, params)
    ptrs = [Pointers(w.L, w.cap) for _ in range(w.B)]
    heads = HeadErr(w.H)
    t = r = folds = 0
    for phase, n in (("std", 11), ("spec", 5), ("std", 13), ("spec", 6), ("std", 17)):
        for _ in range(n):
            if phase == "std":
                d = synth.step_inputs(w, t, seed, params)
                y = layer.decode(to_device(d), gp).cpu().numpy()
                y_ref = model.step(d)
                folds += sum(p.standard_step() > 0 for p in ptrs)
                t += 1
            else:
                d = synth.round_inputs(w, r, seed, params)
                dev = to_device(d)
                y = layer.verify(w.T, dev, gp).cpu().numpy()
                folds += sum(p.verify(w.T) > 0 for p in ptrs)
                y_ref = model.spec_round(d)
                layer.commit(dev["accepted"])
                for p, a in zip(ptrs, d["accepted"]):
                    p.commit(int(a))
                r += 1
            e = rel_err(y, y_ref).max()
            assert e <= TOL_HP, f"{phase} call {t + r}: output rel err {e:.3e}"
            heads.add(y, y_ref)
            ptr = layer.pointers()
            assert (ptr["h"] == [p.h for p in ptrs]).all() and (ptr["base"] == [p.base for p in ptrs]).all()
    assert folds >= 2 * w.B
    assert heads.worst() <= TOL_HP
    assert rel_err(state_gpu_to_np(layer.materialize()), model.S).max() <= TOL_HP
    assert layer.status() == 0


@pytest.mark.parametrize("precision", ["fp32", "two", "shared_bf16"])
def test_mamba2_step_shape_at_b64(precision):
    """B = 64 is the smallest batch whose standard steps take the four-warp,
    three-stage row-split shape (half-slab stages): every checkpoint precision
    across two folds, a forced flush between them and materialised states,
    on sampled sequences against the oracle."""
    w = synth.WORKLOADS["mamba2"].with_(B=64)
    sample = [0, 17, 42, 63]
    run = StandardRun(w, seed=12, precision=precision, sample=sample)
    heads = HeadErr(w.H)
    tol_y = TOL_HP if precision == "fp32" else TOL_LP
    for s in range(37):
        y, y_ref, folded = run.step()
        tol = TOL_HP if (precision == "two" and folded) else tol_y
        e = rel_err(y, y_ref).max()
        assert e <= tol, f"step {s}: output rel err {e:.3e} > {tol}"
        heads.add(y, y_ref)
        if folded or s == 20:
            if s == 20:
                run.layer.flush()
                run.ptr.flush()
            ck = rel_err(run.checkpoint(), run.model.S).max()
            assert ck <= (TOL_LP if precision == "shared_bf16" else TOL_HP), f"step {s}: checkpoint rel err {ck:.3e}"
        if s % 9 == 4:
            m = rel_err(run.materialized(), run.model.S).max()
            assert m <= TOL_HP if precision != "shared_bf16" else m <= TOL_LP, f"step {s}: materialised rel err {m:.3e}"
    assert heads.worst() <= tol_y
    ptr = run.layer.pointers()
    assert (ptr["h"][run.idx] == run.ptr.h).all() and (ptr["base"][run.idx] == run.ptr.base).all()
    assert run.layer.status() == 0

"""Host-side logic of the benchmark that needs no GPU: the key under which a
measured DRAM traffic record is kept, and the algorithmic bytes (the roofline
numerator)."""
from __future__ import annotations

import bench


def test_code_only_ignores_comments_and_blank_lines():
    a = "int x = 1;  // one\n\n/* a\n   block */\nint y = 2;\n"
    b = "// header\nint x = 1;\n   \nint y = 2;  /* trailing */\n"
    assert bench._code_only(a) == bench._code_only(b) == "int x = 1;\nint y = 2;"


def test_code_only_sees_code_changes():
    assert bench._code_only("int x = 1;\n") != bench._code_only("int x = 2;\n")


def test_algorithmic_bytes_of_the_mamba2_workload():
    """The roofline numerator at the headline shape (B=256, H=128, G=8, P=64,
    N=128, window 16), averaged over one window (h = 0..15, the 16th step
    folds), against a count by hand: a 4 MiB fp32 checkpoint read per step, a
    4 MiB write once per window, 7.5 records of 19 KiB read on average, one
    record appended on 15 of 16 steps, 20.5 KiB of inputs and 32 KiB of
    outputs per sequence; the eager step reads and writes the checkpoint."""
    from rs_decode_gb300 import traffic
    s = traffic.Shape("mamba2", 256, 128, 8, 64, 128)
    avg = sum(traffic.replay_step_bytes(s, h, flush=(h == 15)) for h in range(16)) / 16
    rec, inp, out, ck = 19 * 1024, 20.5 * 1024, 32 * 1024, 4 * 2**20
    hand = 256 * (ck + ck / 16 + 7.5 * rec + 15 / 16 * rec + inp + out)
    assert avg == hand == 1196638208
    assert traffic.eager_step_bytes(s) == 256 * (2 * ck + inp + out)
    assert abs(avg / traffic.eager_step_bytes(s) - 0.5537) < 1e-3


def _row(clock: str, sm: str, power: str, *active: str) -> list[str]:
    reasons = ["Active" if n in active else "Not Active"
               for n in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")]
    return [f"2026/12/03 10:00:{clock}", "0", sm, "2070", power, "0x0", *reasons]


def test_clock_summary_keeps_the_timed_window():
    """Samples outside the timed region (with a slowdown) are left out; the
    median SM clock, the active reasons and the peak power are of the rest."""
    import datetime
    rows = [_row("00.000", "1200", "300.0"),
            _row("01.000", "2070", "1200.5", "sw_power_cap"),
            _row("01.500", "2040", "1310.0"),
            _row("02.000", "2060", "1250.0"),
            _row("05.000", "900", "200.0", "hw_slowdown")]
    t = lambda s: datetime.datetime(2026, 12, 3, 10, 0, int(s), int(round((s % 1) * 1e6))).timestamp()
    c = bench.ClockSampler.summarise(rows, t(0.9), t(2.0))
    assert c["samples"] == 3 and c["sm_mhz"] == 2060 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"] and c["power_w_max"] == 1310.0


def test_clock_summary_without_samples_in_the_window():
    """A run shorter than the sampling period keeps the last samples taken."""
    rows = [_row("00.000", "2070", "800.0"), _row("00.050", "2055", "900.0", "hw_thermal_slowdown")]
    c = bench.ClockSampler.summarise(rows, 0.0, 1.0)
    assert c["samples"] == 2 and c["reasons"] == ["hw_thermal_slowdown"]
    assert bench.ClockSampler.summarise([], 0.0, 1.0) is None


def test_algorithmic_bytes_of_the_gdn_workload():
    """Same count for GDN decode (B=256, H_v=32, H_k=16, d=128, window 16): a
    2 MiB checkpoint, records of u fp32 (16 KiB) + alpha (128 B) + k bf16
    (4 KiB), inputs q, k (4 KiB each), v (8 KiB), alpha, beta (128 B each),
    16 KiB of outputs."""
    from rs_decode_gb300 import traffic
    s = traffic.Shape("gdn", 256, 32, 16, 128, 128)
    avg = sum(traffic.replay_step_bytes(s, h, flush=(h == 15)) for h in range(16)) / 16
    rec, inp, out, ck = 16 * 1024 + 128 + 4096, 16 * 1024 + 256, 16 * 1024, 2 * 2**20
    assert avg == 256 * (ck + ck / 16 + 7.5 * rec + 15 / 16 * rec + inp + out) == 623392768
    assert traffic.eager_step_bytes(s) == 256 * (2 * ck + inp + out)


def test_algorithmic_bytes_of_a_folding_verify_round():
    """A Mamba-2 round of 4 drafts with 13 committed records (13 + 4 > 16, so
    it folds): checkpoint read and written, 13 records read, and per draft its
    inputs read, its record appended and its output written; the snapshot
    baseline reads the state once and writes 4 snapshots."""
    from rs_decode_gb300 import traffic
    s = traffic.Shape("mamba2", 256, 128, 8, 64, 128)
    KiB, ck = 1024, 4 * 2**20
    assert traffic.verify_round_bytes(s, 4, 13, True, 4, 4) == ck + 13 * 19 * KiB + 4 * (20.5 + 19 + 32) * KiB + ck
    assert traffic.snapshot_round_bytes(s, 4) == 5 * ck + 4 * (20.5 + 32) * KiB


def test_fold_rule_of_the_byte_model_matches_the_pointer_model():
    """The byte model's fold decision for a round is the pointer model's."""
    from oracle.pointers import Pointers
    from rs_decode_gb300 import traffic
    for L in range(1, 9):
        for T in range(1, 9):
            for h in range(0, max(L, T) + 1):
                p = Pointers(L, max(L, T) + T, h=h)
                assert traffic.spec_folds(h, T, L) == (p.verify(T) > 0), (L, T, h)


def test_reference_arm_prints_one_line_on_rank_zero_only():
    """`--impl reference` times the oracle for W + K steps on rank 0 and prints
    the benchmark's JSON line; other ranks exit 0 without work."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "4", "--warmup", "3"]
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
    env.update(RANK="0", LOCAL_RANK="0")
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["steps"] == 4 and out["warmup"] == 3 and out["value"] > 0
    assert out["unit"] == "tokens/s" and out["higher_is_better"] is True
    assert out["cpu_baseline"]["kind"] == "oracle" and out["cpu_baseline"]["value"] == out["value"]
    assert out["e2e"] == {"value": out["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}
    assert "4 timed decode steps after 3 warm-up steps" in out["cpu_baseline"]["sample"]


def test_algorithmic_bytes_with_per_channel_decay():
    """With one decay per key channel (gdn shapes), a record carries 32 x 128
    fp32 decays (16 KiB) instead of 32, and so does a step's input: a window's
    average step moves about 6% more than the scalar-decay GDN step."""
    from rs_decode_gb300 import traffic
    g = traffic.Shape("gdn", 256, 32, 16, 128, 128)
    k = traffic.Shape("kda", 256, 32, 16, 128, 128)
    assert k.record_bytes - g.record_bytes == k.input_bytes - g.input_bytes == 32 * 127 * 4
    avg = lambda s: sum(traffic.replay_step_bytes(s, h, flush=(h == 15)) for h in range(16)) / 16
    rec, inp, out, ck = 16 * 1024 + 16 * 1024 + 4096, 16 * 1024 + 16 * 1024 + 128, 16 * 1024, 2 * 2**20
    assert avg(k) == 256 * (ck + ck / 16 + 7.5 * rec + 15 / 16 * rec + inp + out)
    assert 1.05 < avg(k) / avg(g) < 1.08


def test_traffic_records_are_keyed_by_their_kernels_sources():
    """A workload's recorded DRAM traffic stays valid while the sources its
    replay kernel is built from are unchanged: the row-split pipeline for
    Mamba-2, the column-split one for GDN and the per-channel decay."""
    assert "rs_replay_rows.cuh" in bench.KERNEL_SOURCES["mamba2"]
    assert "rs_replay_cols.cuh" not in bench.KERNEL_SOURCES["mamba2"]
    for wl in ("gdn", "kda"):
        assert "rs_replay_cols.cuh" in bench.KERNEL_SOURCES[wl]
        assert "rs_replay_rows.cuh" not in bench.KERNEL_SOURCES[wl]
    assert len({bench.kernel_source_hash(w) for w in ("mamba2", "gdn", "kda")}) == 3


def test_algorithmic_bytes_with_bf16_u_records():
    """GDN records that keep u in bf16: a record's u costs 2 bytes per value
    instead of 4 (H_v x d_v = 32 x 128 values, 8 KiB instead of 16 KiB), and
    nothing else changes: the gdn workload's count with the smaller record."""
    from rs_decode_gb300 import traffic
    g32 = traffic.Shape("gdn", 256, 32, 16, 128, 128)
    g16 = traffic.Shape("gdn", 256, 32, 16, 128, 128, u_bytes=2)
    assert g32.record_bytes - g16.record_bytes == 32 * 128 * 2
    assert g32.input_bytes == g16.input_bytes and g32.state_elems == g16.state_elems
    avg = sum(traffic.replay_step_bytes(g16, h, flush=(h == 15)) for h in range(16)) / 16
    rec, inp, out, ck = 8 * 1024 + 128 + 4096, 16 * 1024 + 256, 16 * 1024, 2 * 2**20
    assert avg == 256 * (ck + ck / 16 + 7.5 * rec + 15 / 16 * rec + inp + out) == 605698048

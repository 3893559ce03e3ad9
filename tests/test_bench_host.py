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

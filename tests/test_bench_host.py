"""Host-side logic of bench.py that needs no GPU: the key under which a
measured DRAM traffic record is kept."""
from __future__ import annotations

import bench


def test_code_only_ignores_comments_and_blank_lines():
    a = "int x = 1;  // one\n\n/* a\n   block */\nint y = 2;\n"
    b = "// header\nint x = 1;\n   \nint y = 2;  /* trailing */\n"
    assert bench._code_only(a) == bench._code_only(b) == "int x = 1;\nint y = 2;"


def test_code_only_sees_code_changes():
    assert bench._code_only("int x = 1;\n") != bench._code_only("int x = 2;\n")


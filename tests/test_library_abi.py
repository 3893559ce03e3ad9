"""CPU-only checks of the C ABI: the library builds, loads without a GPU,
exports every entry point that include/rs.h declares, and its host-side
argument validation rejects bad calls before anything is launched."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from rs_decode_gb300 import build, binding
    build.build()
    return binding.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "rs.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(rs_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ["rs_init", "rs_decode_mamba2", "rs_decode_gdn", "rs_verify", "rs_commit",
                     "rs_rollback", "rs_append", "rs_flush", "rs_materialize", "rs_get_status",
                     "rs_eager_step_mamba2", "rs_eager_step_gdn", "rs_eager_verify_snapshots",
                     "rs_eager_select", "rs_state_bytes_for"]:
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_every_symbol():
    from rs_decode_gb300 import binding
    for name in declared_functions():
        assert name in binding._SIGS, name


def test_version_and_status_strings(lib):
    from rs_decode_gb300 import binding as rb
    assert "sm_103a" in rb.rs_version()
    assert rb.rs_status_string(0) == "ok"
    assert rb.rs_status_string(1) == "invalid argument"


def _desc(**kw):
    from rs_decode_gb300 import binding as rb
    base = dict(kind=rb.MAMBA2, B=256, H=128, G=8, P=64, N=128, L=16, T_max=0, capacity=16,
                precision=rb.PREC_FP32)
    base.update(kw)
    return rb.LayerDesc(**base)


def test_state_sizes(lib):
    from rs_decode_gb300 import binding as rb
    s = rb.rs_state_bytes_for(_desc())
    assert s.ckpt_hp == 256 * 128 * 64 * 128 * 4 == 1 << 30   # 4 MiB per sequence
    assert s.ckpt_lp == 0
    assert s.buf_v == 256 * 16 * 128 * 64 * 2
    assert s.buf_k == 256 * 16 * 8 * 128 * 2
    assert s.buf_a == s.buf_s == 256 * 16 * 128 * 4
    g = rb.rs_state_bytes_for(_desc(kind=rb.GDN, H=32, G=16, P=128, N=128, precision=rb.PREC_TWO,
                                    T_max=3, capacity=19, B=512))
    assert g.ckpt_hp == 512 * 32 * 128 * 128 * 4 and g.ckpt_lp == g.ckpt_hp // 2
    assert g.buf_v == 512 * 19 * 32 * 128 * 4 and g.buf_s == 0
    k = rb.rs_state_bytes_for(_desc(kind=rb.KDA, H=32, G=16, P=128, N=128))
    assert k.buf_a == 256 * 16 * 32 * 128 * 4 and k.buf_v == 256 * 16 * 32 * 128 * 4 and k.buf_s == 0


@pytest.mark.parametrize("kw,status", [
    (dict(H=7, G=2), 1),            # H % G != 0
    (dict(P=48), 2),                # no kernel for this shape
    (dict(capacity=15), 3),         # below L
    (dict(T_max=4, capacity=19), 3),
    (dict(L=2, T_max=4, capacity=6), 3),   # L + T_max, but T_max > L needs 2 T_max
    (dict(L=2, T_max=4, capacity=8), 0),
    (dict(L=16, T_max=4, capacity=20), 0),
    (dict(capacity=40), 1),         # above 32 slots
    (dict(T_max=9, capacity=25), 1),
    (dict(precision=7), 1),
    (dict(kind=5), 1),
    (dict(B=0), 1),
    (dict(B=65535, H=2048, G=8), 1),  # 2^27 slabs: beyond 32-bit-safe slab indexing
    (dict(B=65535, H=1024, G=8), 0),  # 2^26 - 2^10 slabs
    (dict(kind=2, H=32, G=16, P=128, N=128), 0),                  # per-channel decay, fp32 checkpoint
    (dict(kind=2, H=32, G=16, P=128, N=128, precision=1), 2),     # ... has no bf16-copy kernels
    (dict(kind=2, H=32, G=16, P=128, N=64), 2),
    (dict(kind=3), 1),
])
def test_descriptor_validation(lib, kw, status):
    from rs_decode_gb300 import binding as rb
    out = rb.StateBytes()
    assert lib.rs_state_bytes_for(ctypes.byref(_desc(**kw)), ctypes.byref(out)) == status


def test_calls_with_missing_pointers_fail_on_the_host(lib):
    from rs_decode_gb300 import binding as rb
    d = _desc()
    st = rb.State()  # all null
    assert lib.rs_decode_mamba2(ctypes.byref(d), ctypes.byref(st), *([None] * 8)) == 1
    assert lib.rs_init(ctypes.byref(d), ctypes.byref(st), None, None) == 1
    assert lib.rs_verify(ctypes.byref(d), ctypes.byref(st), 1, None, None, None) == 1
    assert lib.rs_commit(ctypes.byref(d), ctypes.byref(st), None, None) == 1
    assert lib.rs_flush(ctypes.byref(d), None, None) == 1
    assert lib.rs_get_status(None, None, 0, None) == 1
    # misaligned (but non-null) state pointers are rejected too
    st2 = rb.State(*([0x1001] * 11))
    st2.ckpt_lp = None
    st2.buf_s = 0x1000
    assert lib.rs_materialize(ctypes.byref(d), ctypes.byref(st2), 0x2000, None) == 1
    # GDN append is not defined (its records depend on the state)
    g = _desc(kind=rb.GDN, H=32, G=16, P=128)
    assert lib.rs_append(ctypes.byref(g), ctypes.byref(st), 1, None, None) == 2


def test_verify_rejects_draft_count_above_t_max(lib):
    from rs_decode_gb300 import binding as rb
    d = _desc(T_max=4, capacity=20)
    aligned = [0x100000 * (i + 1) for i in range(11)]
    st = rb.State(*aligned)
    st.ckpt_lp = None
    ins = rb.Inputs(x=0x200000, dt=0x300000, A=0x400000, Bm=0x500000, Cm=0x600000)
    assert lib.rs_verify(ctypes.byref(d), ctypes.byref(st), 5, ctypes.byref(ins), 0x700000, None) == 1
    assert lib.rs_verify(ctypes.byref(d), ctypes.byref(st), 0, ctypes.byref(ins), 0x700000, None) == 1
    # inputs of the other family are rejected
    bad = rb.Inputs(x=0x200000, dt=0x300000, A=0x400000, Bm=0x500000, Cm=0x600000, q=0x800000)
    assert lib.rs_verify(ctypes.byref(d), ctypes.byref(st), 2, ctypes.byref(bad), 0x700000, None) == 1


def test_missing_library_fails_loudly(tmp_path):
    """Without the compiled library the binding raises; there is no other
    code path to fall back to."""
    from rs_decode_gb300 import binding as rb
    with pytest.raises(RuntimeError, match="librs.so not found"):
        rb.load(str(tmp_path / "librs.so"))


def test_product_package_does_not_reach_the_oracle():
    """The package and the benchmark's timed path never import the oracle:
    only tests, the smoke check and the benchmark's CPU legs may."""
    pkg = os.path.join(ROOT, "rs_decode_gb300")
    for name in sorted(os.listdir(pkg)):
        if name.endswith(".py"):
            src = open(os.path.join(pkg, name), encoding="utf-8").read()
            assert not re.search(r"^\s*(import oracle|from oracle)", src, re.M), name
    bench_src = open(os.path.join(ROOT, "bench.py"), encoding="utf-8").read()
    for m in re.finditer(r"^\s*(import oracle|from oracle)", bench_src, re.M):
        fn = [d for d in re.finditer(r"^def (\w+)", bench_src[:m.start()], re.M)][-1].group(1)
        assert fn in ("time_oracle", "run_reference"), fn


def test_oracle_does_not_reach_the_product():
    """The oracle shares no code with the CUDA path: it neither imports the
    package nor includes or loads anything of librs."""
    odir = os.path.join(ROOT, "oracle")
    for name in sorted(os.listdir(odir)):
        if name.endswith((".py", ".c", ".h")):
            src = open(os.path.join(odir, name), encoding="utf-8").read()
            assert not re.search(r"^\s*(import|from)\s+rs_decode_gb300", src, re.M), name
            assert not re.search(r'#\s*include\s*[<"]rs', src), name
            assert "librs" not in src, name


def test_every_declaration_cites_its_source():
    """Each function of include/rs.h carries a "Source:" line in the comment
    just above it (two consecutive declarations may share one): a passage of
    the pages by its key, or "none" for plumbing with no counterpart there.
    The keys are defined at the top of the header with the pages' titles."""
    src = open(os.path.join(ROOT, "include", "rs.h")).read()
    keys = {"[CSI]": "ReplaySSM: Cache SSM Inputs, Not State", "[THR]": "Songlin Yang releases ReplaySSM",
            "[TLDR]": "ReplaySSM speeds up SSM decoding", "[ABS]": "paper abstract"}
    head = src[:src.index("#ifndef RS_H")]
    for key, title in keys.items():
        assert re.search(re.escape(key) + r"\s+[\"(]?[^\n]*" + re.escape(title.split()[0]), head), key
        assert title in re.sub(r"\s*\n\s*\*\s*", " ", head), title
    # tokens: comments and function declarations, in order
    toks = [(m.start(), "c", m.group(0)) for m in re.finditer(r"/\*.*?\*/", src, re.S)]
    code = re.sub(r"/\*.*?\*/", lambda m: " " * len(m.group(0)), src, flags=re.S)
    toks += [(m.start(), "f", m.group(1)) for m in re.finditer(r"^[a-z][\w ]*?\**\b(rs_[a-z0-9_]+)\s*\(", code, re.M)]
    toks.sort()
    last_comment = None
    for _, kind, text in toks:
        if kind == "c":
            last_comment = text
            continue
        assert last_comment is not None, text
        m = re.search(r"Source:\s*(.*)", last_comment, re.S)
        assert m, f"{text}: no Source: line"
        cited = m.group(1)
        assert cited.lstrip().startswith("none") or any(k in cited for k in keys), f"{text}: {cited[:60]!r}"
    assert sum(1 for t in toks if t[1] == "f") == len(declared_functions())

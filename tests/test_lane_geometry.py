"""Shared-memory geometry of the column-split consumer warps, checked on the CPU.

This restates the lane-to-address arithmetic of ``WGeo`` and of the fp32 fold
in ``rs_decode_gb300/csrc/rs_replay_cols.cuh`` (it is a check of that design,
not a run of the kernel) and checks, for every slab shape and element type
the column split instantiates:

* coverage: the consumer warps' lanes, over their rows of every row block,
  read each 16-byte chunk of a staged slab exactly once;
* no bank conflicts: the 8 lanes of each shared-memory phase (one 16-byte
  load each) fall in 8 different 16-byte bank groups under the 128-byte swizzle;
* one swizzle phase per lane: a lane's later rows are a multiple of 8 lines
  on, so its swizzled chunk offset is fixed (one base address per lane).

A stage is one row block of N lines of 128 bytes: whole key rows of the slab,
each row NCB lines, chunk c of line l stored at l * 128 + ((c ^ (l & 7)) << 4).
"""
from __future__ import annotations

import math

import pytest

NCW = 4  # consumer warps

# (P, N, element bytes): GDN and the per-channel decay, 128x128 and 64x64
# slabs, and Mamba-2 rounds of 5..8 drafts on 64x64 slabs (fp32 and bf16)
SHAPES = [(128, 128, 4), (128, 128, 2), (64, 64, 4), (64, 64, 2)]


def geometry(P: int, N: int, esz: int) -> dict:
    ncb = P * esz // 128
    wpc = NCW // ncb
    cpw = 8 // wpc
    rgw = 32 // cpw
    g = dict(NCB=ncb, WPC=wpc, CPW=cpw, LCG=int(math.log2(cpw)), RGW=rgw,
             LPH=int(math.log2(8 // cpw)), SH=int(math.log2(cpw // ncb)) if cpw >= ncb else -1,
             RB=N // ncb)
    g["RK"] = g["RB"] // rgw
    g["LSTRIDE"] = rgw * ncb
    return g


def row_of(g: dict, rg: int) -> int:
    if g["SH"] == 0:
        return rg
    msk = (2 << g["LPH"]) - 1
    low = rg & msk
    return (rg & ~msk) | (((low << 1) | (low >> g["LPH"])) & msk)


def swizzled(line: int, chunk: int) -> int:
    return line * 128 + ((chunk ^ (line & 7)) << 4)


@pytest.mark.parametrize("P,N,esz", SHAPES)
def test_static_conditions(P, N, esz):
    """The kernel's static_asserts hold for every instantiated shape."""
    g = geometry(P, N, esz)
    assert g["NCB"] >= 1 and NCW % g["NCB"] == 0 and g["CPW"] * g["WPC"] == 8 and g["CPW"] * NCW == 8 * g["NCB"]
    assert 0 <= g["SH"] <= 1 and g["LSTRIDE"] % 8 == 0 and g["RGW"] >= (1 << (g["LPH"] + g["SH"]))
    assert g["RB"] * g["NCB"] * 128 == N * 128 and g["RB"] % g["RGW"] == 0   # a stage is N lines


@pytest.mark.parametrize("P,N,esz", SHAPES)
def test_streaming_reads_cover_the_stage_without_conflicts(P, N, esz):
    g = geometry(P, N, esz)
    seen = {}
    for warp in range(NCW):
        cb = warp // g["WPC"]
        for k in range(g["RK"]):
            addrs = []
            for lane in range(32):
                cg, rg = lane & (g["CPW"] - 1), lane >> g["LCG"]
                ch = (warp % g["WPC"]) * g["CPW"] + cg
                row0 = row_of(g, rg)
                line0 = row0 * g["NCB"] + cb
                base = swizzled(line0, ch)                        # the lane's one base address
                addr = base + k * g["LSTRIDE"] * 128
                line = (row0 + k * g["RGW"]) * g["NCB"] + cb
                assert addr == swizzled(line, ch)                 # same swizzle phase on every row
                assert (line, ch) not in seen
                seen[(line, ch)] = (warp, lane, k)
                addrs.append(addr)
            for ph in range(4):
                groups = {(a // 16) % 8 for a in addrs[8 * ph:8 * ph + 8]}
                assert len(groups) == 8, (warp, k, ph)
    assert len(seen) == g["RB"] * g["NCB"] * 8                     # every chunk of the stage once


@pytest.mark.parametrize("P,N,esz", [s for s in SHAPES
                                     if s[2] == 4 and geometry(*s)["CPW"] == 8 and geometry(*s)["RK"] == 8])
def test_fp32_fold_rows(P, N, esz):
    """The fp32 fold with 8 chunks per warp and 8 rows per lane (the 128 x 128
    GDN slab; other shapes fold with the streaming geometry) takes rows
    8 rg .. 8 rg + 7 instead: still every chunk once, still conflict-free."""
    g = geometry(P, N, esz)
    seen = set()
    for warp in range(NCW):
        cb = warp // g["WPC"]
        for k in range(8):
            addrs = []
            for lane in range(32):
                cg, rg = lane & 7, lane >> 3
                line = (8 * rg + k) * g["NCB"] + cb
                assert (line, cg) not in seen
                seen.add((line, cg))
                addrs.append(swizzled(line, cg))
            for ph in range(4):
                assert len({(a // 16) % 8 for a in addrs[8 * ph:8 * ph + 8]}) == 8
    assert len(seen) == g["RB"] * g["NCB"] * 8


@pytest.mark.parametrize("P,N,esz", [s for s in SHAPES if geometry(*s)["CPW"] < 8])
def test_rows_unrotated_would_conflict(P, N, esz):
    """Negative control: where a phase spans several rows (fewer than 8 chunks
    per warp), row(rg) = rg would put lanes of one phase in the same bank
    groups, which is why the kernel rotates the low row-group bits."""
    g = geometry(P, N, esz)
    worst = 8
    for warp in range(NCW):
        cb = warp // g["WPC"]
        addrs = []
        for lane in range(32):
            cg, rg = lane & (g["CPW"] - 1), lane >> g["LCG"]
            ch = (warp % g["WPC"]) * g["CPW"] + cg
            addrs.append(swizzled(rg * g["NCB"] + cb, ch))
        for ph in range(4):
            worst = min(worst, len({(a // 16) % 8 for a in addrs[8 * ph:8 * ph + 8]}))
    assert worst < 8

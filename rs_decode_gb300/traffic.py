"""Algorithmic HBM bytes of the decode path (the roofline numerator).

Counts the bytes each operation must move at least once: checkpoint read,
buffered records read, step inputs read, appended record written, outputs
written, and the checkpoint written on a flush.  Shared per-group data (keys,
queries) is counted once per group, not once per reading CTA.  These are the
"bytes moved = checkpoint read + buffer read + inputs + flush write" of the
ReplaySSM traffic argument ("ReplaySSM: Cache SSM Inputs, Not State", section
"How it works": reads stay at one full-state read per step, writes drop to one
per window).
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Shape:
    kind: str
    B: int
    H: int
    G: int
    P: int
    N: int
    u_bytes: int = 4                       # GDN records' u: 4 (fp32) or 2 (bf16)

    @property
    def state_elems(self) -> int:          # per sequence
        return self.H * self.N * self.P

    @property
    def record_bytes(self) -> int:         # one buffered record, per sequence
        if self.kind == "mamba2":          # x bf16, dt f32, alpha f32, B bf16
            return self.H * self.P * 2 + self.H * 4 + self.H * 4 + self.G * self.N * 2
        # u (fp32, or bf16), alpha f32 (one per head, or one per key channel with a per-channel decay), k bf16
        return self.H * self.P * self.u_bytes + self.H * self.decays * 4 + self.G * self.N * 2

    @property
    def input_bytes(self) -> int:          # one step's inputs, per sequence
        if self.kind == "mamba2":          # x, dt, B, C
            return self.H * self.P * 2 + self.H * 4 + 2 * self.G * self.N * 2
        # q, k, v, alpha, beta
        return 2 * self.G * self.N * 2 + self.H * self.P * 2 + self.H * self.decays * 4 + self.H * 4

    @property
    def decays(self) -> int:               # decays per head and record: N for a per-channel decay
        return self.N if self.kind == "kda" else 1

    @property
    def y_bytes(self) -> int:
        return self.H * self.P * 4


def replay_step_bytes(s: Shape, h_before: int, flush: bool, ckpt_read_bytes: int = 4,
                      ckpt_write_bytes: int = 4) -> int:
    """One standard decode step of all B sequences with h_before committed
    records each.  ckpt_*_bytes per state element: 4 (fp32), 2 (bf16), 6 (both)."""
    per_seq = (s.state_elems * ckpt_read_bytes + h_before * s.record_bytes + s.input_bytes + s.y_bytes
               + (s.state_elems * ckpt_write_bytes if flush else s.record_bytes))
    return s.B * per_seq


def eager_step_bytes(s: Shape) -> int:
    """Conventional decode: load and store the fp32 state every step."""
    return s.B * (s.state_elems * 8 + s.input_bytes + s.y_bytes)


def verify_round_bytes(s: Shape, T: int, h_before: int, flush: bool, read_bytes: int,
                       write_bytes: int) -> int:
    """One speculative round of one sequence: checkpoint read, committed records
    read, T drafts' inputs read and records appended, T outputs written, and
    the checkpoint written when the committed records are folded."""
    return (s.state_elems * read_bytes + h_before * s.record_bytes
            + T * (s.input_bytes + s.record_bytes + s.y_bytes)
            + (s.state_elems * write_bytes if flush else 0))


def snapshot_round_bytes(s: Shape, T: int) -> int:
    """Per-draft snapshot baseline, one sequence: read the state, write T states."""
    return s.state_elems * 4 * (1 + T) + T * (s.input_bytes + s.y_bytes)


def spec_folds(h_before: int, T: int, L: int) -> bool:
    """Whether a verify round starting with h_before committed records folds
    them into the checkpoint (the library's rule: h + T > L and h > 0)."""
    return h_before + T > L and h_before > 0

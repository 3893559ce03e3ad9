"""Model check of the stage-ring protocol of the replay kernels (the column
split, and with per-head hold flags the row split).

The kernel streams checkpoint row blocks through a ring of NS shared-memory
stages.  Each stage has a "full" mbarrier (one producer arrival plus the
copy's transaction bytes) and an "empty" mbarrier (one arrival per consumer
warp).  Waits are by phase parity, which cannot tell a phase from the one two
phases later, so the protocol must never let a waiter fall a whole ring
behind.  The rule the kernel follows: the producer fills positions in order,
and every consumer warp waits on every stage in ring order and arrives once
on each.  A warp waits on all the blocks of a head before it releases any
(a streamed head after its dots, a folding head block by block as each one
reaches registers), so the ring must be at least as deep as the largest head.

This is a randomised discrete-event model of that protocol (copies complete
out of order, warps advance at random), not a run of the kernel.  It checks
that every read sees the position it expects, that no barrier gets more
arrivals than it counts, and that the pipeline drains; a ring shallower than
a head stalls (on the GPU the bounded waits turn this into a status bit, and
the launch shape never picks such a ring).  A negative control
replays the first design, in which each warp waited only on the stages of its
own column block, and must fail.
"""
from __future__ import annotations

import random

import pytest


class MBarrier:
    """Arrival count + transaction count; the phase flips when both reach zero."""

    def __init__(self, count: int):
        self.count = self.pending = count
        self.tx = 0
        self.phase = 0

    def arrive(self) -> None:
        if self.pending == 0:
            raise AssertionError("more arrivals than the barrier counts")
        self.pending -= 1
        self._flip()

    def expect_tx(self, n: int) -> None:
        self.tx += n

    def complete_tx(self, n: int) -> None:
        self.tx -= n
        self._flip()

    def _flip(self) -> None:
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def parity_done(self, parity: int) -> bool:
        """try_wait.parity: the phase with this parity has completed (at
        initialisation the phase before phase 0, parity 1, counts as done)."""
        return (self.phase & 1) != parity


def simulate(NS: int, heads: list[int], NCW: int, seed: int, own_blocks_only: bool = False,
             max_events: int = 400_000, held: list[bool] | None = None):
    """heads: blocks per head in stream order (2 for a bf16 head, 4 for an
    fp32 head).  held (the row split): per head, whether its blocks are held
    until all are read (a folding head) or each is released right after its
    read (a streamed head); None: every head is held (the column split).
    Returns (errors, drained)."""
    rnd = random.Random(seed)
    if own_blocks_only:  # the first design: as many arrivals as warps per column block
        assert len(set(heads)) == 1 and NCW % heads[0] == 0
    full = [MBarrier(1) for _ in range(NS)]
    empty = [MBarrier(NCW // heads[0] if own_blocks_only else NCW) for _ in range(NS)]
    data = [None] * NS                       # which stream position a stage holds
    positions = [(hd, blk) for hd, nb in enumerate(heads) for blk in range(nb)]
    total = len(positions)
    produced, inflight, errors = 0, [], []

    class Warp:
        def __init__(self):
            self.q = 0            # next position to wait on
            self.held = []        # positions waited on and read, not yet released

    warps = [Warp() for _ in range(NCW)]

    def mine(w: int, q: int) -> bool:
        if not own_blocks_only:
            return True
        hd, blk = positions[q]
        return blk == w * heads[hd] // NCW   # the warp's own column block

    for _ in range(max_events):
        if produced == total and not inflight and all(w.q == total and not w.held for w in warps):
            return errors, True
        actor = rnd.randrange(NCW + 2)
        if actor == NCW:                     # producer: next position, if its stage is free
            if produced < total:
                s, ph = produced % NS, (produced // NS) & 1
                if empty[s].parity_done(ph ^ 1):
                    full[s].expect_tx(1)
                    full[s].arrive()
                    inflight.append((s, produced))
                    produced += 1
        elif actor == NCW + 1:               # one copy lands, in any order
            if inflight:
                s, q = inflight.pop(rnd.randrange(len(inflight)))
                data[s] = q
                full[s].complete_tx(1)
        else:
            w = warps[actor]
            # release what is held once the head's blocks are all in registers
            if w.held and (w.q == total or positions[w.q][0] != positions[w.held[0]][0]):
                q = w.held.pop(0)
                s = q % NS
                if data[s] != q:
                    errors.append(("overwritten before release", actor, q, data[s]))
                empty[s].arrive()
                continue
            if w.q == total:
                continue
            if not mine(actor, w.q):
                w.q += 1
                continue
            s, ph = w.q % NS, (w.q // NS) & 1
            if not full[s].parity_done(ph):
                continue
            if data[s] != w.q:
                errors.append(("stale read", actor, w.q, data[s]))
            if own_blocks_only:
                empty[s].arrive()            # the first design: its one block, at once
            elif held is not None and not held[positions[w.q][0]]:
                empty[s].arrive()            # a streamed row-split head: each block after its read
            else:
                w.held.append(w.q)           # the head's blocks are all waited on first
            w.q += 1
    return errors, False


def _heads(rnd: random.Random, n: int) -> list[int]:
    return [rnd.choice((2, 4)) for _ in range(n)]


@pytest.mark.parametrize("NS", [4, 5, 6, 8])
def test_every_warp_waits_on_every_stage(NS):
    for seed in range(40):
        heads = _heads(random.Random(seed), 12)
        errors, drained = simulate(NS, heads, NCW=4, seed=seed)
        assert not errors, errors[:3]
        assert drained, f"NS={NS} seed={seed}: did not drain"


def test_ring_shallower_than_a_head_stalls():
    """Three stages cannot hold a four-block fp32 head, nor one stage a
    two-block bf16 head: no progress (the kernel's bounded waits report this
    as a time-out instead of hanging)."""
    assert simulate(3, [4, 2, 4], NCW=4, seed=1) == ([], False)
    assert simulate(1, [2, 2], NCW=4, seed=2) == ([], False)


def test_bf16_heads_drain_in_two_stages():
    for NS in (2, 3):
        assert simulate(NS, [2] * 10, NCW=4, seed=NS) == ([], True)


def test_first_design_fails():
    """Negative control: with fp32 heads of 4 blocks and one warp per block,
    warps that wait only on their own block's stages read stale data or
    over-arrive when the ring depth is not a multiple of 4, and are safe
    when it is."""
    for NS in (5, 6, 7):
        failed = 0
        for seed in range(20):
            try:
                errors, drained = simulate(NS, [4] * 10, NCW=4, seed=seed, own_blocks_only=True)
            except AssertionError:
                failed += 1
                continue
            assert drained or errors
            failed += bool(errors)
        assert failed > 0, NS
    for NS in (4, 8):
        for seed in range(10):
            assert simulate(NS, [4] * 10, NCW=4, seed=seed, own_blocks_only=True) == ([], True)


def test_tensor_core_heads_occupy_adjacent_stages():
    """With an even ring depth and heads of 2 or 4 blocks, every head starts
    at an even position, so the two column blocks of a bf16 head sit in
    stages s and s + 1 of the same ring pass (the MMA operand spans both)."""
    rnd = random.Random(7)
    for NS in (2, 4, 6, 8):
        q = 0
        for nb in _heads(rnd, 200):
            if nb == 2:
                assert q % 2 == 0 and (q % NS) + 1 == (q + 1) % NS
            q += nb


@pytest.mark.parametrize("NS,SPLIT,NCW", [(2, 1, 8), (2, 2, 4), (3, 2, 4), (4, 1, 8), (4, 2, 4), (3, 1, 8)])
def test_row_split_rings(NS, SPLIT, NCW):
    """The row split's shapes: SPLIT row blocks per head (1: whole slabs, 2:
    half slabs), rings of NS >= SPLIT stages, 8 or 4 consumer warps; streamed
    heads release each block after its read, folding heads (about one in six
    here, at random) hold all of theirs until the fold has read them."""
    for seed in range(30):
        rnd = random.Random(1000 + seed)
        n = 16
        held = [rnd.random() < 0.17 for _ in range(n)]
        errors, drained = simulate(NS, [SPLIT] * n, NCW=NCW, seed=seed, held=held)
        assert not errors, errors[:3]
        assert drained, f"NS={NS} SPLIT={SPLIT} seed={seed}: did not drain"


def test_row_split_fold_needs_a_ring_as_deep_as_a_head():
    """A folding head of two row blocks cannot be held in a one-stage ring
    (the launch shapes never pick one); streamed heads alone drain."""
    assert simulate(1, [2, 2, 2], NCW=4, seed=3, held=[False, True, False]) == ([], False)
    assert simulate(1, [2, 2, 2], NCW=4, seed=3, held=[False, False, False]) == ([], True)

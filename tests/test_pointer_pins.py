"""Pins of the pointer model (oracle/pointers.py) against what the pages fix.

The model keeps per sequence a base slot, h committed records and nd drafts
in a circular buffer ("ReplaySSM: Cache SSM Inputs, Not State", section "How
it works": the checkpoint, the record buffer and the flush at the window
size; the speculative flowchart: fold the committed records when h + T > L,
commit advances the pointer by the accepted length, rollback is free).  These
pins check it with arithmetic it does not use:

* a record ledger that follows record identities (which record sits in which
  slot of a ring of `cap` cells) instead of modular pointers: the slots the
  model names must hold exactly the ledger's records, no record the
  checkpoint does not yet hold may be overwritten, and every fold must take
  exactly the records the ledger folds;
* closed forms for pure decode (a flush every L steps, base = L * flushes);
* the smallest safe capacity, found by exhaustive search over the reachable
  pointer states, equals max(L, T) + T (L + T when T <= L, the capacity the
  pages give), which is the bound the library's descriptor check enforces.

Planted mistakes in a copy of the model must each fail one pin.
"""
from __future__ import annotations

import importlib.util
import random
import sys

import pytest

import oracle.pointers as pointers_mod

SMALL = [(L, T) for L in (1, 2, 3, 5) for T in (0, 1, 2, 3, 4)]


def safe_capacity(L: int, T: int) -> int:
    return max(L, T) + T


class Ledger:
    """Record-level bookkeeping: the checkpoint holds a prefix of the
    committed records, the records since then follow in order, and drafts
    are appended after them.  A ring of cells shows where each record sits."""

    def __init__(self, L: int, cap: int):
        self.L, self.cap = L, cap
        self.ring = [None] * cap
        self.ckpt = 0          # committed records folded into the checkpoint
        self.live = []         # committed records since the checkpoint, in order
        self.drafts = []
        self.next_id = 0

    def _write(self, slot: int, rid: int) -> None:
        assert self.ring[slot] not in self.live, "a record since the checkpoint was overwritten"
        self.ring[slot] = rid

    def _new(self) -> int:
        self.next_id += 1
        return self.next_id

    def standard(self, slot_of) -> int:
        self.drafts = []
        rid = self._new()
        self._write(slot_of(0), rid)
        self.live.append(rid)
        if len(self.live) >= self.L:
            return self.fold()
        return 0

    def verify(self, T: int, slot_of) -> int:
        rids = [self._new() for _ in range(T)]
        slots = [slot_of(i) for i in range(T)]
        assert len(set(slots)) == T, "two drafts share a slot"
        for s, r in zip(slots, rids):
            self._write(s, r)
        folded = self.fold() if len(self.live) + T > self.L else 0
        self.drafts = rids
        return folded

    def commit(self, a: int) -> None:
        self.live += self.drafts[:a]
        self.drafts = []

    def rollback(self) -> None:
        self.drafts = []

    def fold(self) -> int:
        n = len(self.live)
        self.ckpt += n
        self.live = []
        return n


def _agree(p, led: Ledger) -> None:
    assert [led.ring[(p.base + i) % p.cap] for i in range(p.h)] == led.live
    assert [led.ring[(p.base + p.h + i) % p.cap] for i in range(p.nd)] == led.drafts
    assert p.h + p.nd <= p.cap


def _walk(cls, L: int, T: int, cap: int, rng: random.Random, ops: int) -> None:
    p, led = cls(L, cap), Ledger(L, cap)
    for _ in range(ops):
        choice = rng.randrange(4 if T else 2)
        if p.nd:  # a round is open: it ends by commit or rollback
            if choice == 3:
                p.rollback()
                led.rollback()
            else:
                a = rng.randrange(p.nd + 1)
                p.commit(a)
                led.commit(a)
        elif choice == 0:
            base, h = p.base, p.h
            assert p.standard_step() == led.standard(lambda i: (base + h + i) % cap)
        elif choice == 1:
            base, h = p.base, p.h
            assert p.flush() == led.fold()
            assert p.base == (base + h) % cap
        else:
            t = rng.randint(1, T)
            base, h = p.base, p.h
            assert p.verify(t) == led.verify(t, lambda i: (base + h + i) % cap)
        _agree(p, led)


def pin_ledger_random_walks(cls=pointers_mod.Pointers):
    """Random mixes of standard steps, forced flushes and speculative rounds
    (commit of any prefix, or rollback) at the safe capacity."""
    rng = random.Random(20240611)
    for L, T in SMALL:
        for _ in range(60):
            _walk(cls, L, T, safe_capacity(L, T), rng, 80)


def pin_decode_closed_form(cls=pointers_mod.Pointers):
    """Standard steps only: step k (from 1) folds L records iff L divides k;
    afterwards h = k mod L and base = L * floor(k / L) mod cap."""
    for L in (1, 2, 3, 16):
        for cap in (L, L + 4):
            p = cls(L, cap)
            for k in range(1, 5 * L + 3):
                folded = p.standard_step()
                assert folded == (L if k % L == 0 else 0)
                assert p.h == k % L and p.nd == 0
                assert p.base == (L * (k // L)) % cap


def _max_slots(cls, L: int, T: int) -> int:
    """Largest number of cells one call needs at once (the records since the
    checkpoint plus the ones it appends), over every pointer state reachable
    from a fresh sequence; a search over (h, nd), which is finite."""
    big = 4 * (L + T) + 8  # room, so that the search sees what the rules need
    seen, todo, need = set(), [(0, 0)], 0

    def fresh(h, nd):
        p = cls(L, big)
        p.h, p.nd = h, nd
        return p

    while todo:
        h, nd = todo.pop()
        if (h, nd) in seen or h > big:
            continue
        seen.add((h, nd))
        nxt = []
        if nd:
            for a in range(nd + 1):
                p = fresh(h, nd)
                p.commit(a)
                nxt.append((p.h, p.nd))
            p = fresh(h, nd)
            p.rollback()
            nxt.append((p.h, p.nd))
        else:
            need = max(need, h + 1)
            p = fresh(h, nd)
            p.standard_step()
            nxt.append((p.h, p.nd))
            p = fresh(h, nd)
            p.flush()
            nxt.append((p.h, p.nd))
            for t in range(1, T + 1):
                need = max(need, h + t)
                p = fresh(h, nd)
                p.verify(t)
                nxt.append((p.h, p.nd))
        todo += nxt
    return need


def pin_capacity_is_tight(cls=pointers_mod.Pointers):
    """The cells needed at once never exceed max(L, T) + T, and some state
    needs exactly that many; with T <= L it is the pages' L + T."""
    for L, T in SMALL:
        assert _max_slots(cls, L, T) == safe_capacity(L, T), (L, T)
    assert safe_capacity(16, 4) == 20 and safe_capacity(16, 3) == 19 and safe_capacity(16, 0) == 16


def pin_below_safe_capacity_overwrites(cls=pointers_mod.Pointers):
    """One cell fewer and a live record gets overwritten (or the drafts no
    longer fit): the walk that reaches the worst state, run on the ledger."""
    for L, T in SMALL:
        if T == 0:
            continue
        cap = safe_capacity(L, T) - 1
        p, led = cls(L, cap), Ledger(L, cap)
        with pytest.raises(AssertionError):
            # reach h = max(L, T): fully accepted rounds (and standard steps
            # up to L - T when T < L), then open one more round of T drafts
            for _ in range(max(L - T, 0)):
                base, h = p.base, p.h
                p.standard_step()
                led.standard(lambda i: (base + h + i) % cap)
            for _ in range(2):
                base, h = p.base, p.h
                p.verify(T)
                led.verify(T, lambda i: (base + h + i) % cap)
                _agree(p, led)
                p.commit(T)
                led.commit(T)
                _agree(p, led)


PINS = [pin_ledger_random_walks, pin_decode_closed_form, pin_capacity_is_tight,
        pin_below_safe_capacity_overwrites]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


# ----------------------------------------------------------------------------- planted mistakes
MUTATIONS = {
    "standard_fold_late": ("if t >= self.L:", "if t > self.L:"),
    "standard_base_short": ("self.base = (self.base + t) % self.cap",
                            "self.base = (self.base + t - 1) % self.cap"),
    "verify_fold_at_equal": ("if self.h + T > self.L:", "if self.h + T >= self.L:"),
    "verify_folds_drafts": ("folded = self.h\n            self.base = (self.base + self.h) % self.cap",
                            "folded = self.h\n            self.base = (self.base + self.h + T) % self.cap"),
    "commit_takes_all": ("self.h += a", "self.h += self.nd"),
    "rollback_commits": ("    def rollback(self) -> None:\n        self.nd = 0",
                         "    def rollback(self) -> None:\n        self.h += self.nd\n        self.nd = 0"),
    "flush_keeps_h": ("self.h = 0\n        return folded", "return folded"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_planted_mistakes(name, tmp_path):
    src = open(pointers_mod.__file__, encoding="utf-8").read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation anchor not found once: {name}"
    path = tmp_path / "pointers_mut.py"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"pointers_mut_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    sys.modules[spec.name] = mod  # the dataclass decorator looks its module up
    try:
        spec.loader.exec_module(mod)
    finally:
        del sys.modules[spec.name]
    failed = []
    for pin in PINS:
        try:
            pin(mod.Pointers)
        except (AssertionError, pytest.fail.Exception):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name}"

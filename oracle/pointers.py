"""Reference model of the checkpoint / circular-buffer pointer rules.

TEST INFRASTRUCTURE ONLY (part of the oracle).  Per sequence the method keeps
a checkpoint, a circular buffer of the SSM inputs recorded since that
checkpoint, and pointers into it ("ReplaySSM: Cache SSM Inputs, Not State",
section "How it works"; the thread's post [4/N]):

* ``base``: buffer slot of the first record after the checkpoint;
* ``h``:    number of committed records after the checkpoint;
* ``nd``:   number of appended, not yet accepted draft records.

Rules as read from the pages:

* Standard step: append one record (t = h + 1 records).  A new checkpoint is
  stored once per window of L records: if t >= L the step folds all t
  records into the checkpoint (base += t, h = 0), else h = t.
* Speculative round with T drafts (flowchart on the same page): append T
  draft records; if h + T > L, fold the h committed records (drafts
  excluded) into the checkpoint, base += h, h = 0; nd = T.  The ring holds
  the committed records and the drafts: L + T slots when T <= L.
* Commit a accepted drafts: h += a, nd = 0 (the flowchart's commit moves the
  pointer by the accepted count).  Rollback: nd = 0 (a pointer move;
  rejected records are overwritten later).
* Forced flush: fold the h committed records, base += h, h = 0.
"""
from __future__ import annotations

import dataclasses


@dataclasses.dataclass
class Pointers:
    L: int
    cap: int
    base: int = 0
    h: int = 0
    nd: int = 0

    def standard_step(self) -> int:
        """Returns the number of records folded (0 if no flush)."""
        t = self.h + 1
        self.nd = 0
        if t >= self.L:
            self.base = (self.base + t) % self.cap
            self.h = 0
            return t
        self.h = t
        return 0

    def verify(self, T: int) -> int:
        """Returns the number of committed records folded (0 if no flush)."""
        folded = 0
        if self.h + T > self.L:
            folded = self.h
            self.base = (self.base + self.h) % self.cap
            self.h = 0
        self.nd = T
        return folded

    def commit(self, a: int) -> None:
        assert 0 <= a <= self.nd
        self.h += a
        self.nd = 0

    def rollback(self) -> None:
        self.nd = 0

    def flush(self) -> int:
        folded = self.h
        self.base = (self.base + self.h) % self.cap
        self.h = 0
        return folded

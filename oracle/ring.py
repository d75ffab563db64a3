"""Ring-buffer cursor of one sequence as plain integers (test infrastructure only).

The ring holds the input records appended since the last flush.  Record j
(0-based, counted from the last flush) lives in slot (head + j) mod C, where
C = L + T_max is the ring capacity.  The transitions follow:

* decode: the current record is appended; when that append makes the ring
  hold L records, the step is a flush step: the L records are folded into the
  checkpoint, which is written once, and the buffer is cleared
  ([richland] What shipped: "When the 16-record buffer fills ... a flush step
  folds the records into the checkpoint, writes it to HBM once, and clears
  the buffer"; [ai-jitan] ReplaySSMは何をする手法か, third bullet).
* verify: T draft records are appended after the committed ones; the cursor
  does not move ([richland] What shipped: "drafts are just appended to the
  input buffer, verification runs").
* commit n: the accepted prefix is committed by advancing the pointer; later
  draft slots are ignored and overwritten ([richland] What shipped: "the
  accepted prefix is committed by advancing a pointer; records past the
  pointer are ignored and overwritten"; [warp-studio] 推測デコーディングの強化).
  When the committed records reach L, all of them are folded (the same flush).
* flush: fold whatever is buffered now (used to export or re-quantise).

Flushing moves head past the folded records; head is never reset.
"""

from __future__ import annotations


class RingModel:
    def __init__(self, ring_len: int, capacity: int):
        if ring_len < 1 or capacity < ring_len:
            raise ValueError("need 1 <= L <= C")
        self.L = ring_len
        self.C = capacity
        self.head = 0
        self.count = 0
        self.pending = 0          # draft records appended by the last verify
        self.last_flush = 0       # 1 if the last call flushed this sequence
        self.folded = 0           # records folded by that flush

    def slot(self, j: int) -> int:
        """Ring slot of record j (0-based since the last flush)."""
        return (self.head + j) % self.C

    def _fold(self) -> None:
        self.folded = self.count
        self.head = (self.head + self.count) % self.C
        self.count = 0
        self.last_flush = 1

    def decode(self) -> int:
        """Standard decode step; returns 1 if the step is a flush step."""
        if self.pending:
            raise RuntimeError("decode with drafts pending: commit first")
        self.last_flush = 0
        self.folded = 0
        if self.count + 1 == self.L:
            self.count += 1
            self._fold()
        else:
            self.count += 1
        return self.last_flush

    def verify(self, T: int) -> list[int]:
        """Append T drafts after the committed records; returns their slots."""
        if self.pending:
            raise RuntimeError("verify with drafts pending: commit first")
        if self.count + T > self.C:
            raise ValueError("ring overflow")
        self.last_flush = 0
        self.folded = 0
        self.pending = T
        return [self.slot(self.count + i) for i in range(T)]

    def commit(self, n: int) -> int:
        """Commit the first n drafts; returns 1 if the commit flushed."""
        if not 0 <= n <= self.pending:
            raise ValueError("accepted count out of range")
        self.pending = 0
        self.last_flush = 0
        self.folded = 0
        self.count += n
        if self.count >= self.L:
            self._fold()
        return self.last_flush

    def flush(self) -> None:
        """Fold all buffered records (possibly none)."""
        if self.pending:
            raise RuntimeError("flush with drafts pending: commit first")
        self._fold()

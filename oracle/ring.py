"""The sliding-window ring and its rollback rule, at the level of positions. TEST INFRASTRUCTURE.

[TS] "sliding-window caches and rollback": a local layer keeps exactly one
window of positions in a circular cache, slot = position % W. A verify writes
every row's K/V at its true position, so once the context has wrapped, row
p + i lands on the slot that held position p + i - W. The trunk therefore keeps
what a verify is about to evict and, after the acceptance, puts the rejected
rows back; on a full acceptance it restores nothing (restoring there left the
committed rows holding the evicted positions, the bug the page reports).

WindowRing tracks which position every slot holds. It pins that rule: after
any sequence of verifies and acceptances, the ring holds every position the
next token's window needs, and during a verify every row finds each position of
its own window either in the ring or among the saved rows. `restore` selects
the rule ("rejected", the page's) or one of two wrong ones for negative checks
("never", "always").
"""
from __future__ import annotations


class WindowRing:
    def __init__(self, window: int, restore: str = "rejected"):
        assert restore in ("rejected", "never", "always")
        self.W = window
        self.slot = [None] * window
        self.length = 0
        self.saved = {}        # span row i -> the position its slot held before the verify
        self.span = (0, 0)
        self.restore = restore

    def verify(self, S: int):
        """Rows at positions p..p+S-1 (p = the cache length) write their slots; returns, for each
        row, whether every position of its window [p+i-W+1, p+i] was found (ring or saved)."""
        assert 1 <= S <= self.W
        p = self.length
        self.saved, self.span = {}, (p, S)
        for i in range(S):
            s = (p + i) % self.W
            self.saved[i] = self.slot[s]
            self.slot[s] = p + i
        saved = set(v for v in self.saved.values() if v is not None)
        ok = []
        for i in range(S):
            q = p + i
            ok.append(all(self.slot[u % self.W] == u or u in saved for u in range(max(0, q - self.W + 1), q + 1)))
        return ok

    def accept(self, m: int) -> None:
        """m drafts accepted (rows 0..m kept): the cache length becomes p + m + 1."""
        p, S = self.span
        assert 0 <= m < S
        if self.restore == "always" or (self.restore == "rejected" and m < S - 1):
            first = 0 if self.restore == "always" else m + 1
            for j in range(first, S):
                if self.restore == "always" and j <= m:
                    # the rows kept in a full acceptance are put back as well (the page's first version)
                    self.slot[(p + j) % self.W] = self.saved[j]
                elif j > m:
                    self.slot[(p + j) % self.W] = self.saved[j]
        self.length = p + m + 1

    def window_intact(self) -> bool:
        """The next token (position q = length) finds every earlier position of its window."""
        q = self.length
        return all(self.slot[u % self.W] == u for u in range(max(0, q - self.W + 1), q))

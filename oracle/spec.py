"""Acceptance, n-gram prompt lookup and the adaptive draft length. TEST INFRASTRUCTURE."""
from __future__ import annotations

import numpy as np


def accept_greedy(drafts, argmax):
    """Greedy acceptance of one verify span.

    [PI] "the transaction", Accept: keep the longest prefix where each draft
    matches the target argmax, then append the target's own token at the first
    mismatch (the bonus), so a step commits 1..K+1 tokens.
    [TS] "the protocol", Verify: row m's drawn token is the corrected (or bonus)
    token.

    drafts = d_1..d_k, argmax = a_0..a_k (a_i is row i's argmax; row 0 is the
    current token). m = the largest j <= k with d_i == a_{i-1} for every i <= j.
    Returns (m, [a_0..a_m]).
    """
    k = len(drafts)
    assert len(argmax) == k + 1
    m = 0
    while m < k and int(drafts[m]) == int(argmax[m]):
        m += 1
    return m, [int(a) for a in argmax[:m + 1]]


def ngram_propose(history, k: int, n: int = 2):
    """Prompt lookup: propose what followed the most recent earlier occurrence
    of the last n tokens.

    [TS] "n-gram": drafts by finding where the last few tokens occurred earlier
    in the context and proposing what followed; the corpus is the emitted token
    history. [CA] "--ngram-min 2": draft only off a match of at least two
    tokens.

    Reading: the match is the most recent j (the follower position) with
    n <= j <= len-1 and history[j-n:j] == history[len-n:len]; the drafts are
    history[j : min(j+k, len)], fewer than k when the history ends first; no
    match (or k <= 0) gives no drafts.
    """
    L = len(history)
    if k <= 0 or L < n + 1:
        return []
    key = [int(t) for t in history[L - n:]]
    for j in range(L - 1, n - 1, -1):
        if [int(t) for t in history[j - n:j]] == key:
            return [int(t) for t in history[j:min(j + k, L)]]
    return []


def adapt_k(K: int, n_drafted: int, m: int, k_max: int) -> int:
    """[CA] "adaptive K": start at 1; after a fully accepted round K += 2; after
    any rejection K -= 1; clamp to [1, K_max].

    Reading for the cases the page leaves open: a round that proposed nothing
    leaves K unchanged; "fully accepted" means every proposed draft was
    accepted (m == n_drafted >= 1), even when fewer than K were proposed.
    """
    if n_drafted == 0:
        return K
    if m == n_drafted:
        return min(K + 2, k_max)
    return max(K - 1, 1)


def required_order(n_min: int, n_max: int, pmin: float) -> int:
    """[TS] "--spec-pmin": for the n-gram drafter pmin does not gate a probability, it scales the
    required match length ("a 2-token context matches somewhere ... almost always ... a 6-token
    context never matches at all"). [CA] "--ngram-min 2": draft only off a match of at least n_min
    tokens.

    Reading: pmin in [0, 1] moves the required length linearly from n_min (pmin = 0) to n_max
    (pmin = 1), rounded half up: n_req = n_min + floor(pmin * (n_max - n_min) + 1/2).
    """
    assert 1 <= n_min <= n_max and 0.0 <= pmin <= 1.0
    return n_min + int(np.floor(pmin * (n_max - n_min) + 0.5))


def ngram_propose_multi(history, k: int, n_min: int = 2, n_max: int = 2, pmin: float = 0.0):
    """Prompt lookup over several n-gram orders ([TS] "n-gram": one incrementally maintained hash
    index per n-gram order): the longest order n in [n_req, n_max] whose last-n-token context
    occurred earlier with a follower wins, and within it the most recent occurrence (as
    ngram_propose); fewer than n_req matching tokens give no drafts."""
    n_req = required_order(n_min, n_max, pmin)
    for n in range(n_max, n_req - 1, -1):
        d = ngram_propose(history, k, n)
        if d:
            return d
    return []


class NgramIndex:
    """The incremental form of ngram_propose_multi: per order n a map from an n-token context to
    the position of its most recent follower, updated as tokens are appended (exact keys)."""

    def __init__(self, n_max: int):
        self.n_max = n_max
        self.hist = []
        self.maps = {n: {} for n in range(1, n_max + 1)}

    def append(self, tok: int) -> None:
        L = len(self.hist)
        for n in range(1, min(self.n_max, L) + 1):
            self.maps[n][tuple(self.hist[L - n:L])] = L      # context ending at L-1 -> follower L
        self.hist.append(int(tok))

    def propose(self, k: int, n_min: int, pmin: float):
        n_req = required_order(n_min, self.n_max, pmin)
        L = len(self.hist)
        if k <= 0:
            return []
        for n in range(self.n_max, n_req - 1, -1):
            if L < n + 1:
                continue
            j = self.maps[n].get(tuple(self.hist[L - n:L]))
            if j is not None:
                return self.hist[j:min(j + k, L)]
        return []

"""Pins for acceptance, prompt lookup, adaptive K, the page pool and the loop.

Hand-worked fixtures under tests/golden/ cite the passage each follows;
brute force and independent formulations cover the rest.
"""
import itertools
import os

import numpy as np
import pytest

import oracle
import synth
from oracle import CapacityError, DenseDecoder, PagePool, accept_greedy, adapt_k, generate, ngram_propose
from synth import workloads

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    for line in open(os.path.join(GOLD, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            yield [c.strip() for c in line.split("|")]


def _ints(s):
    return [] if s.strip() in ("-", "") else [int(t) for t in s.split()]


def test_accept_golden():
    for drafts, argmax, m, committed in _rows("accept_examples.txt"):
        got_m, got_c = accept_greedy(_ints(drafts), _ints(argmax))
        assert got_m == int(m) and got_c == _ints(committed)


def test_accept_brute_force_is_longest_common_prefix():
    # Every (drafts, argmax) over a 3-letter alphabet with k <= 4.
    for k in range(0, 5):
        for d in itertools.product(range(3), repeat=k):
            for a in itertools.product(range(3), repeat=k + 1):
                m, c = accept_greedy(list(d), list(a))
                lcp = len(os.path.commonprefix([list(d), list(a[:k])]))
                assert m == lcp
                assert 1 <= len(c) <= k + 1 and len(c) == m + 1
                assert c[:m] == list(d[:m]) and c[-1] == a[m]


def test_ngram_golden():
    for hist, k, drafts in _rows("ngram_examples.txt"):
        assert ngram_propose(_ints(hist), int(k), 2) == _ints(drafts), (hist, k)


def _ngram_by_index(hist, k, n=2):
    # Independent formulation: an incrementally built dict from each n-gram to the
    # position of its follower, later insertions overwriting earlier ones.
    idx = {}
    for p in range(n, len(hist)):
        idx[tuple(hist[p - n:p])] = p
    if k <= 0 or len(hist) < n + 1:
        return []
    j = idx.get(tuple(hist[-n:]))
    return [] if j is None else list(hist[j:min(j + k, len(hist))])


@pytest.mark.parametrize("vocab", [3, 5, 50])
def test_ngram_matches_hash_index_and_properties(vocab):
    for s in range(200):
        L = 2 + s % 60
        hist = [int(t) for t in synth.tokens(11, f"ng{vocab}", L, vocab, offset=1000 * s)]
        for k in (0, 1, 4, 7):
            d = ngram_propose(hist, k)
            assert d == _ngram_by_index(hist, k)
            if d:
                # the drafts follow an occurrence of the last two tokens, and no later one exists
                starts = [j for j in range(2, L) if hist[j - 2:j] == hist[-2:] and hist[j:j + len(d)] == d]
                assert starts and max(starts) == max(j for j in range(2, L) if hist[j - 2:j] == hist[-2:])
                assert len(d) == min(k, L - max(starts))


def test_adaptive_k_golden():
    for kmax, rounds, expect in _rows("adaptive_k_trace.txt"):
        K, got = 1, []
        for r in rounds.split():
            nd, m = (int(x) for x in r.split(","))
            K = adapt_k(K, nd, m, int(kmax))
            got.append(K)
        assert got == _ints(expect)


def test_adaptive_k_stays_in_range():
    K = 1
    for i in range(1000):
        nd = int(synth.ints(2, "nd", 1, 0, 7, offset=i)[0])
        m = int(synth.ints(2, "m", 1, 0, nd, offset=i)[0]) if nd else 0
        K = adapt_k(K, nd, m, 7)
        assert 1 <= K <= 7


def _state(pool):
    return [list(t) for t in pool.table], list(pool.free)


def test_page_pool_golden():
    pool = PagePool(7, 4, 2, 4)
    for op, t0, t1, free in _rows("page_pool_trace.txt"):
        name, *args = op.split()
        args = [int(a) for a in args]
        before = _state(pool)
        if t0 == "error":
            with pytest.raises((CapacityError, ValueError)):
                getattr(pool, {"ensure": "ensure_capacity", "rewind": "rewind"}[name])(args)
            assert _state(pool) == before
            continue
        if name == "ensure":
            pool.ensure_capacity(args)
        elif name == "advance":
            for b, a in enumerate(args):
                assert a <= len(pool.table[b]) * 4
                pool.set_length(b, a)
        else:
            pool.rewind(args)
        tables, fr = _state(pool)
        assert tables[0] == _ints(t0) and tables[1] == _ints(t1) and fr == _ints(free), op


def test_page_pool_conservation_and_undo():
    pool = PagePool(64, 16, 4, 8)
    for step in range(300):
        req = [int(x) for x in synth.ints(3, "req", 4, -1, 128, offset=4 * step)]
        pool.rewind(list(pool.length))          # tight: each table holds exactly ceil(length / 16) pages
        before = _state(pool)
        try:
            pool.ensure_capacity(req)
        except CapacityError:
            assert _state(pool) == before
            continue
        if step % 3 == 0:
            # a rewind to the lengths held before the reservation undoes it exactly
            pool.rewind(list(pool.length))
            assert _state(pool) == before
            continue
        for b, r in enumerate(req):
            if r >= 0:
                pool.set_length(b, r)
        if step % 5 == 0:
            pool.rewind([l // 2 for l in pool.length])
        used = sorted(p for t in pool.table for p in t)
        assert sorted(used + pool.free) == list(range(64)) and len(set(used)) == len(used)


@pytest.fixture(scope="module")
def tiny_model():
    W = synth.weights(synth.TINY, 1)
    return DenseDecoder(synth.TINY, lambda n: W[n])


def test_spec_on_equals_spec_off(tiny_model):
    # [PI] losslessness: spec-on equals spec-off token for token (exact in float64).
    prompt = workloads.motif_prompt()
    on, rec_on, _ = generate(tiny_model, [prompt], 32, drafter="ngram", k=4)
    off, rec_off, _ = generate(tiny_model, [prompt], 32, drafter="none")
    assert on == off and len(on[0]) == 32
    for r in rec_on:
        assert 1 <= len(r.committed[0]) <= len(r.spans[0])    # 1..K+1 per step
    assert all(len(r.spans[0]) == 1 for r in rec_off)


def test_spec_on_equals_spec_off_adaptive_table_and_batch(tiny_model):
    prompts = [workloads.motif_prompt(), synth.tokens(8, "p2", 41, synth.TINY.vocab),
               synth.tokens(8, "p3", 17, synth.TINY.vocab)]
    off, _, pool_off = generate(tiny_model, prompts, 24, drafter="none", prefill_chunk=16)
    on, rec, pool_on = generate(tiny_model, prompts, 24, drafter="ngram", adaptive=True, k_max=7,
                                prefill_chunk=16)
    assert on == off
    assert all(1 <= r.k_used[b] <= 7 for r in rec for b in range(3))
    # a table drafter that proposes the true continuation is accepted in full
    tables = [np.array(s + [0] * 8) for s in off]          # table[j] = generated token j
    tab, rec_t, _ = generate(tiny_model, prompts, 24, drafter="table", k=5, tables=tables, prefill_chunk=16)
    assert tab == off
    assert all(r.m[b] == len(r.spans[b]) - 1 for r in rec_t for b in range(3) if r.m[b] >= 0)


def test_rewind_leaves_later_forwards_as_if_never_drafted(tiny_model):
    # [CA] rollback == do not advance; [PI] LIFO drop of the reservation. With one
    # sequence, the page table after each spec step equals the plain loop's table
    # at the same length, and the cached K/V rows below the length agree.
    prompt = workloads.motif_prompt()
    sh = synth.TINY
    from oracle import SeqCache
    _, rec, pool = generate(tiny_model, [prompt], 32, drafter="table", k=4,
                            tables=[synth.tokens(3, "junk", 64, sh.vocab)])
    _, rec_off, pool_off = generate(tiny_model, [prompt], 32, drafter="none")
    off_tables = {r.new_len[0]: r.page_table[0] for r in rec_off}
    for r in rec:
        assert r.page_table[0] == off_tables[r.new_len[0]]


def test_truncation_at_output_budget(tiny_model):
    # [PI] capture-shape gotcha: a span is cut to max_tokens - generated.
    prompt = workloads.motif_prompt()
    s, rec, _ = generate(tiny_model, [prompt], 9, drafter="table", k=7, tables=[np.arange(100)])
    gen = 1
    for r in rec:
        assert len(r.spans[0]) - 1 == min(7, 9 - gen - 1)
        gen += len(r.committed[0])
    assert len(s[0]) == 9


def test_oracle_reproduces_its_recorded_ngram_k4_run(tiny_model):
    # Regression pin: the stored run was written by tests/golden/make_golden.py (oracle only).
    rows = list(_rows("tiny_ngram_k4_oracle.txt"))
    stream = _ints(rows[0][1])
    s, rec, _ = generate(tiny_model, [workloads.motif_prompt(1)], 32, drafter="ngram", k=4)
    assert s[0] == stream
    for r, row in zip(rec, rows[1:]):
        assert r.spans[0] == _ints(row[1]) and r.argmax[0] == _ints(row[2])
        assert r.m[0] == int(row[3]) and r.new_len[0] == int(row[4])


# ----------------------------------------------------------------------------- multi-order n-gram

def test_required_order_reading():
    """[TS] "--spec-pmin" scales the n-gram drafter's required match length; [CA] "--ngram-min 2".
    Reading: linear from n_min (pmin 0) to n_max (pmin 1), rounded half up."""
    assert [oracle.required_order(2, 6, p) for p in (0.0, 0.25, 0.5, 0.75, 1.0)] == [2, 3, 4, 5, 6]
    assert [oracle.required_order(1, 4, p) for p in (0.0, 0.1, 0.2, 0.5, 0.9, 1.0)] == [1, 1, 2, 3, 4, 4]
    assert oracle.required_order(3, 3, 0.7) == 3


def test_multi_order_prefers_the_longest_match():
    h = [5, 3, 4, 8, 2, 3, 4, 9, 6, 5, 3, 4]
    assert oracle.ngram_propose(h, 2, 2) == [9, 6]                    # most recent 2-gram [3, 4]
    assert oracle.ngram_propose_multi(h, 2, 2, 3) == [8, 2]          # the 3-gram [5, 3, 4] wins
    assert oracle.ngram_propose_multi(h, 2, 2, 3, pmin=1.0) == [8, 2]
    assert oracle.ngram_propose_multi(h, 2, 2, 4, pmin=1.0) == []    # no 4-token context repeats
    assert oracle.ngram_propose_multi(h, 2, 3, 3) == [8, 2]
    assert oracle.ngram_propose_multi(h, 0, 2, 3) == []


@pytest.mark.parametrize("vocab", [3, 6, 40])
def test_multi_order_index_matches_brute_force(vocab):
    """The incremental per-order index against the backward scan at every prefix of random and
    repeat-heavy histories, for several (n_min, n_max, pmin); with n_min = n_max = 2 both reduce to
    the 2-gram proposer."""
    rng = np.random.default_rng(vocab)
    hists = [rng.integers(0, vocab, 160).tolist(),
             list(map(int, workloads.span_repeat_prompt(vocab, n_spans=20, span=8, vocab=vocab)))]
    for h in hists:
        for n_min, n_max, pmin in ((2, 2, 0.0), (1, 4, 0.0), (2, 6, 0.5), (2, 5, 1.0), (3, 6, 0.3)):
            idx = oracle.NgramIndex(n_max)
            for L, t in enumerate(h):
                idx.append(t)
                k = 1 + (L % 7)
                brute = oracle.ngram_propose_multi(h[:L + 1], k, n_min, n_max, pmin)
                assert idx.propose(k, n_min, pmin) == brute, (L, n_min, n_max, pmin)
                if (n_min, n_max) == (2, 2):
                    assert brute == oracle.ngram_propose(h[:L + 1], k, 2)
                if brute:   # the drafts follow an earlier occurrence of at least n_req context tokens
                    n_req = oracle.required_order(n_min, n_max, pmin)
                    ctx = h[L + 1 - n_req:L + 1]
                    assert any(h[j - n_req:j] == ctx and h[j:j + len(brute)] == brute
                               for j in range(n_req, L + 1))


# ----------------------------------------------------------------------------- sliding-window ring

def _ring_trace(rule, W, seed, steps=400, max_span=None):
    from oracle.ring import WindowRing
    rng = np.random.default_rng(seed)
    ring = WindowRing(W, rule)
    ok = True
    for _ in range(steps):
        S = int(rng.integers(1, (max_span or W) + 1))
        seen = ring.verify(S)
        ok &= all(seen)
        m = int(rng.integers(0, S)) if rng.random() < 0.7 else S - 1      # partial or full acceptance
        ring.accept(m)
        ok &= ring.window_intact()
    return ok


@pytest.mark.parametrize("W,max_span", [(8, 8), (16, 5), (32, 17)])
def test_window_ring_rule_keeps_every_window(W, max_span):
    """[TS] sliding-window caches and rollback: saving what a verify evicts and putting back the
    rejected rows (nothing on a full acceptance) keeps every row's window and the next token's
    window in the one-window ring, over random spans and acceptances well past the wrap."""
    for seed in range(10):
        assert _ring_trace("rejected", W, seed, max_span=max_span)


def test_window_ring_wrong_rules_fail():
    """The two rules the page rules out: never restoring loses evicted positions once two or more
    rows are rejected; restoring on a full acceptance puts evicted positions over committed rows."""
    assert not all(_ring_trace("never", 16, s) for s in range(5))
    assert not all(_ring_trace("always", 16, s) for s in range(5))
    from oracle.ring import WindowRing
    r = WindowRing(8, "never")                 # the page's example: two rows rejected past the wrap
    r.verify(8); r.accept(7)
    r.verify(5); r.accept(1)                   # rows 2..4 rejected; the next token needs position 3+...
    assert not r.window_intact()
    r = WindowRing(8, "rejected")
    r.verify(8); r.accept(7)
    r.verify(5); r.accept(1)
    assert r.window_intact()


def test_window_attention_pins():
    """The oracle's sliding-window attention: a window as long as the context is full causal
    attention; a window of one returns the row's own value; otherwise it equals full attention over
    the window's keys alone."""
    from oracle import attention_rows
    rng = np.random.default_rng(9)
    T, S, nq, nkv, D = 40, 6, 4, 2, 16
    q = rng.standard_normal((S, nq, D))
    K, V = rng.standard_normal((T, nkv, D)), rng.standard_normal((T, nkv, D))
    pos = np.arange(T - S, T)
    full = attention_rows(q, K, V, pos, 0.25)
    np.testing.assert_array_equal(attention_rows(q, K, V, pos, 0.25, window=T), full)
    one = attention_rows(q, K, V, pos, 0.25, window=1)
    np.testing.assert_allclose(one, np.repeat(V[pos], nq // nkv, axis=1), rtol=0, atol=1e-15)
    W = 9
    win = attention_rows(q, K, V, pos, 0.25, window=W)
    for i, t in enumerate(pos):
        lo = t - W + 1
        ref = attention_rows(q[i:i + 1], K[lo:t + 1], V[lo:t + 1], np.array([W - 1]), 0.25)
        np.testing.assert_allclose(win[i], ref[0], rtol=1e-13, atol=1e-13)

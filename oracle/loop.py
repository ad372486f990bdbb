"""The speculative step loop (propose, verify, accept, commit/rewind) over a
batch of sequences. TEST INFRASTRUCTURE.

  [PI] "the transaction": propose K tokens, verify [current, d1..dK] in one
       forward, accept the longest matching prefix plus the bonus token,
       commit the accepted KV and drop the rest of the reservation.
  [PI] "draft-seed alignment": after m accepted drafts, the m+1 rows
       [current, d1..dm] are committed and the KV position advances by m+1;
       the next current token (argmax of row m) has not been forwarded.
  [PI] "capture-shape gotcha": a span is truncated to the output budget
       (max_tokens - generated).
  [PI] losslessness / [CA] "off is the identical loop with drafting disabled":
       the plain loop is this loop with no drafts (one-row steps).
  [CA] "adaptive K".
  [TS] "the protocol", Verify: the caller's sampler draws each row and drafts
       are accepted while the drawn token matches (oracle.sampling).

Conventions (readings): the prompt is prefilled sequence by sequence in
chunks of at most ``prefill_chunk`` tokens, each chunk preceded by a capacity
reservation for that sequence alone; the first generated token is the argmax
of the prompt's last row; ``n_tokens`` counts that first token; no stop token
is honoured (every sequence generates exactly n_tokens).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .model import SeqCache, argmax_lowest
from .pages import PagePool
from .sampling import draw_rows
from .spec import accept_greedy, adapt_k, ngram_propose


@dataclass
class StepRecord:
    spans: list                      # per sequence [current, d1..dk]; [] once the sequence is done
    argmax: list                     # per sequence, argmax of every row
    m: list                          # accepted drafts per sequence (-1 when inactive)
    committed: list                  # per sequence a_0..a_m
    len_before: list
    new_len: list
    k_used: list                     # the draft length K in force at this step
    page_table: list                 # per sequence, after the rewind
    logits: list = field(default=None)


def generate(model, prompts, n_tokens: int, drafter: str = "ngram", k: int = 4, adaptive: bool = False,
             k_max: int = 7, ngram_n: int = 2, tables=None, page_size: int = 16, n_pages: int = None,
             max_pages_per_seq: int = None, prefill_chunk: int = 128, keep_logits: bool = False,
             kv_dtype: str = "f64", temperature: float = 0.0, seed: int = 0):
    """Run the loop for every sequence until each has n_tokens generated tokens.

    drafter: "ngram" (prompt lookup over the sequence's history), "table"
    (drafts = tables[b][g : g+k] where g tokens are generated so far), or
    "none" (the plain loop: one-row steps). temperature > 0 draws every row
    with the sampler of oracle.sampling (key `seed`, sequence slot b, the row's
    position) instead of taking its argmax. Returns (streams, records, pool).
    """
    sh = model.shape
    B = len(prompts)
    cap = max(len(p) for p in prompts) + n_tokens + k_max + 2
    if max_pages_per_seq is None:
        max_pages_per_seq = -(-cap // page_size)
    if n_pages is None:
        n_pages = B * max_pages_per_seq
    caches = [SeqCache(sh, cap, kv_dtype) for _ in range(B)]
    pool = PagePool(n_pages, page_size, B, max_pages_per_seq)

    def draw(b, logits, positions):
        if temperature > 0:
            return [int(x) for x in draw_rows(logits, temperature, seed, b, positions)]
        return [int(x) for x in argmax_lowest(logits)]

    last_logits = []
    for b in range(B):                                        # prefill, sequence by sequence
        p = np.asarray(prompts[b], dtype=np.int64)
        lg = None
        for c0 in range(0, len(p), prefill_chunk):
            chunk = p[c0:c0 + prefill_chunk]
            req = [-1] * B
            req[b] = caches[b].length + len(chunk)
            pool.ensure_capacity(req)
            spans = [[] for _ in range(B)]
            spans[b] = chunk
            lg = model.forward(caches, spans, last_row_logits=True)[b]
            pool.set_length(b, caches[b].length)
        last_logits.append(lg[-1])
    first = [draw(b, last_logits[b][None], [len(prompts[b]) - 1])[0] for b in range(B)]
    streams = [[f] for f in first]
    hists = [list(map(int, prompts[b])) + [first[b]] for b in range(B)]
    K = [1 if adaptive else k for _ in range(B)]
    records = []

    while any(len(s) < n_tokens for s in streams):
        active = [len(streams[b]) < n_tokens for b in range(B)]
        drafts, spans = [], []
        for b in range(B):
            if not active[b]:
                drafts.append([])
                spans.append([])
                continue
            g = len(streams[b])
            k_eff = min(K[b], n_tokens - g - 1)
            if drafter == "ngram":
                d = ngram_propose(hists[b], k_eff, ngram_n)
            elif drafter == "table":
                d = [int(t) for t in tables[b][g:g + k_eff]] if k_eff > 0 else []
            elif drafter == "none":
                d = []
            else:
                raise ValueError(drafter)
            drafts.append(d)
            spans.append([hists[b][-1]] + d)
        len_before = [caches[b].length for b in range(B)]
        pool.ensure_capacity([len_before[b] + len(spans[b]) if active[b] else -1 for b in range(B)])
        lg = model.forward(caches, spans)
        for b in range(B):
            if active[b]:
                pool.set_length(b, caches[b].length)
        am, ms, com, new_len = [], [], [], []
        for b in range(B):
            if not active[b]:
                am.append([]); ms.append(-1); com.append([]); new_len.append(-1)
                continue
            a = draw(b, lg[b], [len_before[b] + i for i in range(len(spans[b]))])
            m, c = accept_greedy(drafts[b], a)
            am.append(a); ms.append(m); com.append(c)
            new_len.append(len_before[b] + m + 1)
            caches[b].length = len_before[b] + m + 1          # rollback == do not advance
        pool.rewind(new_len)
        k_used = list(K)
        for b in range(B):
            if active[b]:
                streams[b] += com[b]
                hists[b] += com[b]
                if adaptive:
                    K[b] = adapt_k(K[b], len(drafts[b]), ms[b], k_max)
        records.append(StepRecord(spans=[list(map(int, s)) for s in spans], argmax=am, m=ms, committed=com,
                                  len_before=len_before, new_len=new_len, k_used=k_used,
                                  page_table=[list(t) for t in pool.table],
                                  logits=[np.array(x) for x in lg] if keep_logits else None))
    return streams, records, pool

"""Seeded workload recipes: prompts, contexts, drafts and context lengths.

Every array here is an input. The recipes follow the synthetic workloads the
speculative-decoding pages measure on (random-context verify, an 848-token
cost sweep, repeat-heavy prompts for prompt lookup); no public dataset is used
or reproduced.
"""
from __future__ import annotations

import numpy as np

from . import TINY, QWEN3_4B, ints, tokens, unit


def motif_prompt(seed: int = 1, motif_len: int = 16, repeats: int = 8, vocab: int = TINY.vocab) -> np.ndarray:
    """A uniform-random motif repeated back to back (tiny-decoder workload: 16 x 8 = 128 tokens)."""
    motif = tokens(seed, "prompt.motif", motif_len, vocab)
    return np.tile(motif, repeats).astype(np.int32)


def uniform_context(seed: int, n: int, vocab: int = QWEN3_4B.vocab, name: str = "context") -> np.ndarray:
    """Uniform-random context tokens (already-in-cache context for the verify-cost workloads)."""
    return tokens(seed, name, n, vocab)


def uniform_drafts(seed: int, step: int, k: int, vocab: int, name: str = "drafts") -> np.ndarray:
    """k uniform-random draft tokens for one verify step (draws [step*32, step*32+k) of one stream)."""
    assert k <= 32
    return tokens(seed, name, k, vocab, offset=step * 32)


def context_lengths(seed: int, batch: int, lo: int = 512, hi: int = 4096) -> np.ndarray:
    """Per-sequence context lengths, integers uniform in [lo, hi] inclusive."""
    return ints(seed, "context_len", batch, lo, hi)


def corrupt(seed: int, b: int, continuation: np.ndarray, p: float, vocab: int) -> np.ndarray:
    """Replace each position with a uniform token with probability p (the replacement may coincide)."""
    n = len(continuation)
    u = unit(seed, f"corrupt.{b}", n)
    r = tokens(seed, f"corrupt_tok.{b}", n, vocab)
    return np.where(u < p, r, np.asarray(continuation, dtype=np.int32)).astype(np.int32)


def span_repeat_prompt(seed: int, n_spans: int = 32, span: int = 32, p_repeat: float = 0.5,
                       vocab: int = QWEN3_4B.vocab) -> np.ndarray:
    """Prompt of n_spans spans of `span` tokens. Span 0 is fresh; each later span,
    with probability p_repeat, copies a uniformly chosen earlier span, else it is
    fresh uniform tokens."""
    coin = unit(seed, "span.repeat", n_spans)
    out = []
    for s in range(n_spans):
        if s > 0 and coin[s] < p_repeat:
            src = int(ints(seed, "span.source", 1, 0, s - 1, offset=s)[0])
            out.append(out[src].copy())
        else:
            out.append(tokens(seed, "span.fresh", span, vocab, offset=s * span))
    return np.concatenate(out).astype(np.int32)

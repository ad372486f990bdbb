"""Sampled (temperature) verify: the caller's sampler draws each row. TEST INFRASTRUCTURE.

[TS] "the protocol", Verify: the trunk forwards [lastToken, d1..dK] as one
batch with per-row logits; the caller's sampler draws each row, and drafts are
accepted while the drawn token matches; row m's drawn token is the corrected
(or bonus) token. Greedy verification is the special case of a sampler that
returns the argmax.

Reading (the page names no sampler): row r of sequence b, at absolute
position p, draws from softmax(logits / T_b) by the Gumbel-max construction
(Gumbel 1954; the "Gumbel-max trick" of Maddison, Tarlow and Minka, 2014):

    drawn = argmax_v ( logits_v / T_b + g(seed, b, p, v) ),   g = -log(-log(u))

with u uniform on (0, 1) taken from a counter-based stream keyed by the
sequence slot b, the row's position p and the vocabulary index v, so the noise
a position receives does not depend on how many rows share its forward, on the
step or on earlier rejections: speculation on and off draw the same token at
every position, and the accept rule of greedy verification (longest prefix of
drafts equal to the drawn tokens, plus the drawn token after it) is unchanged.
T_b <= 0 means greedy (the argmax, lowest index on an exact tie).

The stream is SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014, output function with the constants Vigna
publishes): mix64(z) = z3 with z1 = (z ^ z >> 30) * 0xBF58476D1CE4E5B9,
z2 = (z1 ^ z1 >> 27) * 0x94D049BB133111EB, z3 = z2 ^ z2 >> 31 (mod 2^64), and
the i-th output of the stream keyed k is mix64(k + (i + 1) * 0x9E3779B97F4A7C15).
Keys chain as
    k_b = stream(seed)[b],   k_bp = stream(k_b)[p],   x = stream(k_bp)[v]
and u = ((x >> 41) + 1/2) * 2^-23, a 23-bit uniform that float32 holds
exactly, strictly inside (0, 1).
"""
from __future__ import annotations

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
MASK = (1 << 64) - 1


def mix64_int(z: int) -> int:
    """SplitMix64 output function on a Python integer (exact 64-bit arithmetic by masking)."""
    z &= MASK
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
    return z ^ (z >> 31)


def stream_int(key: int, i: int) -> int:
    """Output i of the SplitMix64 stream keyed `key`."""
    return mix64_int(key + (i + 1) * GOLDEN)


def _mix64_u64(z: np.ndarray) -> np.ndarray:
    """The same output function over a numpy uint64 array (arithmetic wraps mod 2^64)."""
    z = z ^ (z >> np.uint64(30))
    z = z * np.uint64(0xBF58476D1CE4E5B9)
    z = z ^ (z >> np.uint64(27))
    z = z * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def row_key(seed: int, b: int, pos: int) -> int:
    """The key of the stream that covers the vocabulary of sequence b's row at position pos."""
    return stream_int(stream_int(seed, b), pos)


def uniforms(seed: int, b: int, pos: int, vocab: int) -> np.ndarray:
    """u(seed, b, pos, v) for v = 0..vocab-1, float64 values in (0, 1) on a 2^-23 grid."""
    k = np.uint64(row_key(seed, b, pos))
    with np.errstate(over="ignore"):
        z = k + (np.arange(vocab, dtype=np.uint64) + np.uint64(1)) * np.uint64(GOLDEN)
        x = _mix64_u64(z)
    return ((x >> np.uint64(41)).astype(np.float64) + 0.5) * 2.0 ** -23


def gumbel(seed: int, b: int, pos: int, vocab: int) -> np.ndarray:
    """Standard Gumbel noise g = -log(-log(u)) for every vocabulary index."""
    return -np.log(-np.log(uniforms(seed, b, pos, vocab)))


def perturbed(logits: np.ndarray, temperature: float, seed: int, b: int, positions) -> np.ndarray:
    """logits / T + g for every row (logits [S, V], positions [S]); the score whose argmax is drawn."""
    V = logits.shape[-1]
    g = np.stack([gumbel(seed, b, int(p), V) for p in positions]) if len(positions) else np.zeros((0, V))
    return logits / temperature + g


def draw_rows(logits: np.ndarray, temperature: float, seed: int, b: int, positions) -> np.ndarray:
    """The token each row draws: the argmax of the perturbed scores (lowest index on an exact tie),
    or the plain argmax when temperature <= 0."""
    if temperature <= 0:
        return np.argmax(logits, axis=-1).astype(np.int64)
    return np.argmax(perturbed(logits, temperature, seed, b, positions), axis=-1).astype(np.int64)

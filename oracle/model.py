"""Dense decoder forward over a multi-row span, in float64. TEST INFRASTRUCTURE.

What it computes follows the verify step of the pages:
  [PI] "the transaction", Verify: one prefill-style forward over the K+1 span
       [current_token, d1..dK] that reports the argmax at every position.
  [TS] "the shared loop" (SpecForward): a multi-row forward with per-row
       logits, so a whole draft window costs about one decode step.
  [CA] "dense rollback": the forward writes K/V at offset = (positions) -
       (inputs) and each row attends [0, offset + q); rows past the accepted
       prefix are stale but never read.
  [TS] "sliding-window caches and rollback": a verify writes every row's K/V
       at its true position.

The pages do not spell out the decoder's layer internals. The reading used
here: pre-norm RMSNorm (Zhang and Sennrich, 2019) with gains; grouped-query
attention (Ainslie et al., 2023) with per-head RMSNorm on q and k and
rotate-half RoPE (Su et al., RoFormer; the "neox" pairing (j, j + D/2)) --
the same q/k treatment the TensorSharp page gives for its DFlash drafter's
pass B (K = rope_neox(headnorm(...))); SwiGLU FFN (Shazeer, 2020); no biases;
softmax scale 1/sqrt(D); separate (untied) embedding and LM head.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) to float64; bf16 is the top half of an IEEE float32."""
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even), returned as float64.

    The value is first rounded to float32 (nearest even), then its low 16 bits
    are rounded away: add 0x7FFF plus the lowest kept bit, truncate.
    """
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16 << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g over the last axis."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


def silu(z: np.ndarray) -> np.ndarray:
    """z * sigmoid(z) = z / (1 + e^-z)."""
    return z / (1.0 + np.exp(-z))


def rope_neox(u: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half RoPE over the last axis (length D).

    For j < D/2 the pair (u_j, u_{j+D/2}) is rotated by the angle
    pos * theta^(-2j/D):  (a, b) -> (a cos - b sin, b cos + a sin).
    ``pos`` broadcasts against u.shape[:-1].
    """
    D = u.shape[-1]
    half = D // 2
    j = np.arange(half, dtype=np.float64)
    inv_freq = theta ** (-2.0 * j / D)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    a, b = u[..., :half], u[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def attention_rows(q: np.ndarray, K: np.ndarray, V: np.ndarray, q_pos: np.ndarray, scale: float,
                   window: int = 0) -> np.ndarray:
    """Causal grouped-query attention of query rows against one sequence's cache.

    q: [S, nq, D]; K, V: [T, nkv, D] (positions 0..T-1); q_pos[i] is row i's
    absolute position, and row i attends keys 0..q_pos[i] (the cache prefix
    plus the span rows up to and including itself). q head h reads kv head
    h // (nq / nkv). With window > 0 (a sliding-window layer, [TS] sliding-window
    caches: a local layer keeps exactly one window of positions) row i attends
    only the last `window` positions, max(0, q_pos[i] - window + 1)..q_pos[i].
    """
    S, nq, D = q.shape
    nkv = K.shape[1]
    grp = nq // nkv
    out = np.empty((S, nq, D), dtype=np.float64)
    for i in range(S):
        n = int(q_pos[i]) + 1
        lo = max(0, n - window) if window > 0 else 0
        qi = q[i].reshape(nkv, grp, D)                       # [g, r, D]
        s = np.einsum("grd,tgd->grt", qi, K[lo:n]) * scale   # [g, r, n - lo]
        s = s - s.max(axis=-1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=-1, keepdims=True)
        out[i] = np.einsum("grt,tgd->grd", p, V[lo:n]).reshape(nq, D)
    return out


def argmax_lowest(logits: np.ndarray) -> np.ndarray:
    """Per-row argmax over the last axis; the lowest index wins an exact tie."""
    return np.argmax(logits, axis=-1).astype(np.int64)


class SeqCache:
    """One sequence's K/V for every layer at positions 0..capacity-1 and its length.

    Positions at or beyond ``length`` may hold stale rows from a rejected
    verify; nothing reads them before the next forward overwrites them.

    kv_dtype is the storage precision of the cache: "f64" keeps K/V exactly;
    "bf16" stores them rounded to bf16, as the bf16 KV cache of the bf16
    target models on the pages does (pegainfer's Qwen3-4B runs in bf16).
    """

    def __init__(self, shape, capacity: int, kv_dtype: str = "f64"):
        assert kv_dtype in ("f64", "bf16")
        self.K = [np.zeros((capacity, shape.n_kv_heads, shape.head_dim)) for _ in range(shape.n_layers)]
        self.V = [np.zeros((capacity, shape.n_kv_heads, shape.head_dim)) for _ in range(shape.n_layers)]
        self.length = 0
        self.capacity = capacity
        self.kv_dtype = kv_dtype

    def store(self, l: int, at: int, k: np.ndarray, v: np.ndarray) -> None:
        if self.kv_dtype == "bf16":
            k, v = round_bf16(k), round_bf16(v)
        self.K[l][at:at + len(k)] = k
        self.V[l][at:at + len(v)] = v


class DenseDecoder:
    """Weights come from ``tensor_fn(name)`` as bf16 bit patterns; they are held
    (or converted on use) as float64 values, so the oracle computes on exactly
    the values the GPU holds, in float64 arithmetic."""

    def __init__(self, shape, tensor_fn, cache_weights: bool = True):
        self.shape = shape
        self._fn = tensor_fn
        self._cache = {} if cache_weights else None

    def w(self, name: str) -> np.ndarray:
        if self._cache is not None and name in self._cache:
            return self._cache[name]
        t = bf16_to_f64(self._fn(name))
        if self._cache is not None:
            self._cache[name] = t
        return t

    def embed(self, toks: np.ndarray) -> np.ndarray:
        # only the gathered rows are converted
        return bf16_to_f64(self._fn("embed")[toks])

    def forward(self, caches: list, spans: list, keep_hidden: bool = False, last_row_logits: bool = False):
        """One forward over span b of every sequence b (spans may be empty).

        Rows of sequence b sit at positions caches[b].length + i. Every row's
        K/V is written before any row attends; afterwards each cache length
        grows by its span length. Returns per-sequence logits [S_b, V]; with
        last_row_logits only the last row of each span gets logits ([1, V]),
        the others are not computed.
        """
        sh = self.shape
        eps, D, nq, nkv = sh.rms_eps, sh.head_dim, sh.n_q_heads, sh.n_kv_heads
        toks = np.concatenate([np.asarray(s, dtype=np.int64) for s in spans]) if spans else np.zeros(0, np.int64)
        counts = [len(s) for s in spans]
        starts = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
        R = int(starts[-1])
        pos = np.concatenate([np.arange(c) + caches[b].length for b, c in enumerate(counts)]).astype(np.int64) \
            if R else np.zeros(0, np.int64)
        for b, c in enumerate(counts):
            if caches[b].length + c > caches[b].capacity:
                raise ValueError("span exceeds the oracle cache capacity")

        x = self.embed(toks)                                          # [R, H]
        scale = 1.0 / np.sqrt(D)
        for l in range(sh.n_layers):
            p = f"layers.{l}."
            a = rmsnorm(x, self.w(p + "attn_norm"), eps)
            q = (a @ self.w(p + "wq").T).reshape(R, nq, D)
            k = (a @ self.w(p + "wk").T).reshape(R, nkv, D)
            v = (a @ self.w(p + "wv").T).reshape(R, nkv, D)
            if sh.qk_norm:
                q = rmsnorm(q, self.w(p + "q_norm"), eps)
                k = rmsnorm(k, self.w(p + "k_norm"), eps)
            q = rope_neox(q, pos[:, None], sh.rope_theta)
            k = rope_neox(k, pos[:, None], sh.rope_theta)
            for b, c in enumerate(counts):                            # K/V of every row first
                L0, r0 = caches[b].length, starts[b]
                caches[b].store(l, L0, k[r0:r0 + c], v[r0:r0 + c])
            o = np.empty((R, nq, D))
            for b, c in enumerate(counts):
                if c == 0:
                    continue
                L0, r0 = caches[b].length, starts[b]
                o[r0:r0 + c] = attention_rows(q[r0:r0 + c], caches[b].K[l][:L0 + c], caches[b].V[l][:L0 + c],
                                              pos[r0:r0 + c], scale, sh.swa_window if sh.is_local(l) else 0)
            x = x + o.reshape(R, nq * D) @ self.w(p + "wo").T
            hb = rmsnorm(x, self.w(p + "ffn_norm"), eps)
            f = silu(hb @ self.w(p + "w_gate").T) * (hb @ self.w(p + "w_up").T)
            x = x + f @ self.w(p + "w_down").T
        y = rmsnorm(x, self.w("final_norm"), eps)
        for b, c in enumerate(counts):
            caches[b].length += c
        if last_row_logits:
            last = [starts[b + 1] - 1 for b in range(len(spans)) if counts[b] > 0]
            lg = y[last] @ self.w("lm_head").T
            out, k = [], 0
            for b in range(len(spans)):
                if counts[b] > 0:
                    out.append(lg[k:k + 1])
                    k += 1
                else:
                    out.append(np.zeros((0, sh.vocab)))
            return (out, y) if keep_hidden else out
        logits = y @ self.w("lm_head").T                               # [R, V]
        out = [logits[starts[b]:starts[b + 1]] for b in range(len(spans))]
        if keep_hidden:
            return out, y
        return out

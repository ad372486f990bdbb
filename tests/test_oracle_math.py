"""Pins for the oracle's numeric building blocks and its decoder forward.

Each check compares against something other than the oracle's own formula:
torch float64 library routines, a complex-number formulation of RoPE, closed
forms, special cases and invariants of the forward.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synth
from oracle import DenseDecoder, SeqCache, attention_rows, rmsnorm, rope_neox, silu
from oracle.model import bf16_to_f64

rng = np.random.default_rng(1234)


def test_bf16_conversion_matches_torch():
    bits = synth.normal_bf16(3, "conv", 4096)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(bf16_to_f64(bits), ref)


def test_rmsnorm_matches_torch():
    x = rng.standard_normal((7, 256)) * 3.0
    g = rng.standard_normal(256)
    ref = F.rms_norm(torch.from_numpy(x), (256,), torch.from_numpy(g), eps=1e-6).numpy()
    np.testing.assert_allclose(rmsnorm(x, g, 1e-6), ref, rtol=1e-13, atol=1e-13)


def test_silu_matches_torch():
    z = rng.standard_normal(1000) * 8
    np.testing.assert_allclose(silu(z), F.silu(torch.from_numpy(z)).numpy(), rtol=1e-13, atol=1e-15)


def test_rope_matches_complex_rotation():
    D, theta = 64, 1e6
    u = rng.standard_normal((5, 3, D))
    pos = np.array([0, 1, 17, 848, 32767])
    half = D // 2
    z = u[..., :half] + 1j * u[..., half:]
    ang = pos[:, None, None] * theta ** (-2.0 * np.arange(half) / D)
    w = z * np.exp(1j * ang)
    ref = np.concatenate([w.real, w.imag], axis=-1)
    np.testing.assert_allclose(rope_neox(u, pos[:, None], theta), ref, rtol=1e-12, atol=1e-12)


def test_rope_position_zero_is_identity_and_norm_preserved():
    u = rng.standard_normal((4, 128))
    np.testing.assert_array_equal(rope_neox(u, np.zeros((4,)), 1e6), u)
    r = rope_neox(u, np.array([3, 100, 5000, 9]), 1e6)
    np.testing.assert_allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(u, axis=-1), rtol=1e-13)


def test_rope_scores_depend_only_on_relative_position():
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    for p, u, s in [(10, 3, 7), (500, 499, 1000), (0, 0, 123)]:
        a = rope_neox(q, np.array(p), 1e6) @ rope_neox(k, np.array(u), 1e6)
        b = rope_neox(q, np.array(p + s), 1e6) @ rope_neox(k, np.array(u + s), 1e6)
        assert abs(a - b) < 1e-10


def test_rope_two_dims_is_plane_rotation():
    # D = 2: one pair rotated by angle pos * theta^0 = pos radians.
    u = np.array([0.3, -1.2])
    for pos in [0.0, 1.0, 2.5]:
        R = np.array([[np.cos(pos), -np.sin(pos)], [np.sin(pos), np.cos(pos)]])
        np.testing.assert_allclose(rope_neox(u, np.array(pos), 10.0), R @ u, rtol=1e-14, atol=1e-15)


def _sdpa_ref(q, K, V, q_pos, scale):
    S, nq, D = q.shape
    T = K.shape[0]
    mask = np.arange(T)[None, :] <= q_pos[:, None]                      # [S, T]
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]                     # [1, nq, S, D]
    kt = torch.from_numpy(K).permute(1, 0, 2)[None]
    vt = torch.from_numpy(V).permute(1, 0, 2)[None]
    o = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.from_numpy(mask)[None, None],
                                       scale=scale, enable_gqa=True)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("S,T,nq,nkv", [(1, 1, 4, 2), (5, 40, 4, 2), (17, 865, 32, 8), (8, 8, 8, 8)])
def test_attention_matches_torch_sdpa(S, T, nq, nkv):
    D = 64
    q = rng.standard_normal((S, nq, D))
    K = rng.standard_normal((T, nkv, D))
    V = rng.standard_normal((T, nkv, D))
    q_pos = np.arange(T - S, T)
    out = attention_rows(q, K, V, q_pos, 1 / np.sqrt(D))
    np.testing.assert_allclose(out, _sdpa_ref(q, K, V, q_pos, 1 / np.sqrt(D)), rtol=1e-11, atol=1e-12)


def test_attention_special_cases():
    D = 16
    q = rng.standard_normal((1, 2, D))
    K = rng.standard_normal((1, 1, D))
    V = rng.standard_normal((1, 1, D))
    # One key: the output is that key's value exactly.
    np.testing.assert_array_equal(attention_rows(q, K, V, np.array([0]), 0.25)[0, 0], V[0, 0])
    # Identical keys: uniform weights, the output is the mean of the values.
    K6 = np.repeat(rng.standard_normal((1, 1, D)), 6, axis=0)
    V6 = rng.standard_normal((6, 1, D))
    np.testing.assert_allclose(attention_rows(q, K6, V6, np.array([5]), 0.25)[0, 1], V6[:, 0].mean(0), rtol=1e-13)
    # Causal: a row never sees keys past its position, whatever they hold.
    K2 = rng.standard_normal((9, 1, D))
    V2 = rng.standard_normal((9, 1, D))
    q2 = rng.standard_normal((3, 2, D))
    a = attention_rows(q2, K2, V2, np.array([4, 5, 6]), 0.25)
    K2[7:] = 1e3
    V2[7:] = -1e3
    b = attention_rows(q2, K2, V2, np.array([4, 5, 6]), 0.25)
    np.testing.assert_array_equal(a, b)


# ----------------------------------------------------------------------------- decoder forward

@pytest.fixture(scope="module")
def tiny():
    W = synth.weights(synth.TINY, 1)
    return W, DenseDecoder(synth.TINY, lambda n: W[n])


def _torch_forward(W, sh, toks):
    """The decoder composed from torch float64 library ops (F.linear, F.rms_norm,
    F.scaled_dot_product_attention with GQA, F.silu), positions 0..S-1, no cache."""
    T = lambda n: torch.from_numpy(bf16_to_f64(W[n]))
    D, nq, nkv, eps = sh.head_dim, sh.n_q_heads, sh.n_kv_heads, sh.rms_eps
    S = len(toks)
    x = T("embed")[torch.as_tensor(toks)]
    half = D // 2
    inv = sh.rope_theta ** (-2.0 * torch.arange(half, dtype=torch.float64) / D)
    ang = torch.arange(S, dtype=torch.float64)[:, None] * inv
    cos = torch.cat([torch.cos(ang), torch.cos(ang)], -1)[None]
    sin = torch.cat([torch.sin(ang), torch.sin(ang)], -1)[None]

    def rot(t):  # [H, S, D]; the usual "rotate_half" formulation
        r = torch.cat([-t[..., half:], t[..., :half]], -1)
        return t * cos + r * sin

    for l in range(sh.n_layers):
        p = f"layers.{l}."
        a = F.rms_norm(x, (sh.hidden,), T(p + "attn_norm"), eps)
        q = F.linear(a, T(p + "wq")).view(S, nq, D)
        k = F.linear(a, T(p + "wk")).view(S, nkv, D)
        v = F.linear(a, T(p + "wv")).view(S, nkv, D)
        q = F.rms_norm(q, (D,), T(p + "q_norm"), eps).transpose(0, 1)
        k = F.rms_norm(k, (D,), T(p + "k_norm"), eps).transpose(0, 1)
        o = F.scaled_dot_product_attention(rot(q)[None], rot(k)[None], v.transpose(0, 1)[None],
                                           is_causal=True, enable_gqa=True)[0]
        x = x + F.linear(o.transpose(0, 1).reshape(S, nq * D), T(p + "wo"))
        b = F.rms_norm(x, (sh.hidden,), T(p + "ffn_norm"), eps)
        x = x + F.linear(F.silu(F.linear(b, T(p + "w_gate"))) * F.linear(b, T(p + "w_up")), T(p + "w_down"))
    y = F.rms_norm(x, (sh.hidden,), T("final_norm"), eps)
    return F.linear(y, T("lm_head")).numpy()


def test_forward_matches_torch_library_composition(tiny):
    W, m = tiny
    toks = synth.tokens(9, "fwd", 37, synth.TINY.vocab)
    c = SeqCache(synth.TINY, 64)
    got = m.forward([c], [toks])[0]
    np.testing.assert_allclose(got, _torch_forward(W, synth.TINY, toks), rtol=1e-10, atol=1e-10)
    assert c.length == 37


def test_forward_with_random_gains_matches_torch(tiny):
    # Norm gains are 1.0 in the synthetic models; random gains pin that each
    # gain multiplies the right normalised tensor.
    W, _ = tiny
    W2 = dict(W)
    for name in W2:
        if name.split(".")[-1] in synth.NORM_NAMES:
            W2[name] = synth.normal_bf16(5, name, W2[name].size, 1.0).reshape(W2[name].shape)
    m2 = DenseDecoder(synth.TINY, lambda n: W2[n])
    toks = synth.tokens(9, "fwd2", 20, synth.TINY.vocab)
    got = m2.forward([SeqCache(synth.TINY, 32)], [toks])[0]
    np.testing.assert_allclose(got, _torch_forward(W2, synth.TINY, toks), rtol=1e-10, atol=1e-10)


def test_rows_gate_sequential_vs_one_span(tiny):
    # [CA] rows gate: q sequential one-row decodes against one q-row forward.
    _, m = tiny
    toks = synth.tokens(4, "gate", 48, synth.TINY.vocab)
    c1, c2 = SeqCache(synth.TINY, 64), SeqCache(synth.TINY, 64)
    m.forward([c1], [toks[:40]])
    m.forward([c2], [toks[:40]])
    one = m.forward([c1], [toks[40:]])[0]
    seq = np.concatenate([m.forward([c2], [toks[i:i + 1]])[0] for i in range(40, 48)])
    np.testing.assert_allclose(one, seq, rtol=1e-11, atol=1e-11)
    np.testing.assert_array_equal(one.argmax(-1), seq.argmax(-1))
    for l in range(synth.TINY.n_layers):
        np.testing.assert_allclose(c1.K[l][:48], c2.K[l][:48], rtol=1e-12, atol=1e-12)


def test_causality_later_tokens_do_not_change_earlier_rows(tiny):
    _, m = tiny
    toks = synth.tokens(4, "causal", 30, synth.TINY.vocab)
    t2 = toks.copy()
    t2[20:] = (t2[20:] + 7) % synth.TINY.vocab
    a = m.forward([SeqCache(synth.TINY, 32)], [toks])[0]
    b = m.forward([SeqCache(synth.TINY, 32)], [t2])[0]
    np.testing.assert_array_equal(a[:20], b[:20])
    assert np.abs(a[20:] - b[20:]).max() > 1e-3


def test_stale_rows_past_length_are_never_read(tiny):
    # [CA] dense rollback: rows past the cache length are stale but never read.
    _, m = tiny
    toks = synth.tokens(6, "stale", 24, synth.TINY.vocab)
    c1, c2 = SeqCache(synth.TINY, 40), SeqCache(synth.TINY, 40)
    m.forward([c1], [toks[:16]])
    m.forward([c2], [toks[:16]])
    m.forward([c2], [synth.tokens(6, "junk", 7, synth.TINY.vocab)])   # a rejected verify of 7 rows
    c2.length = 16                                                       # rewind: do not advance
    a = m.forward([c1], [toks[16:]])[0]
    b = m.forward([c2], [toks[16:]])[0]
    np.testing.assert_array_equal(a, b)


def test_batch_rows_are_independent(tiny):
    _, m = tiny
    p1 = synth.tokens(7, "b1", 19, synth.TINY.vocab)
    p2 = synth.tokens(7, "b2", 33, synth.TINY.vocab)
    ca, cb, c1, c2 = (SeqCache(synth.TINY, 40) for _ in range(4))
    la, lb = m.forward([ca, cb], [p1, p2])
    np.testing.assert_allclose(la, m.forward([c1], [p1])[0], rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(lb, m.forward([c2], [p2])[0], rtol=1e-11, atol=1e-11)
    # An empty span leaves that sequence untouched.
    out = m.forward([ca, cb], [[], p1[:3]])
    assert out[0].shape == (0, synth.TINY.vocab) and ca.length == 19 and cb.length == 36


def test_last_row_logits_equal_full_logits(tiny):
    _, m = tiny
    toks = synth.tokens(4, "lastrow", 21, synth.TINY.vocab)
    full = m.forward([SeqCache(synth.TINY, 32)], [toks])[0]
    last = m.forward([SeqCache(synth.TINY, 32)], [toks], last_row_logits=True)[0]
    np.testing.assert_allclose(last[0], full[-1], rtol=1e-12, atol=1e-12)


def test_round_bf16_matches_torch_conversion():
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 6, 20000), [0.0, -0.0, 1.0, 3.0]])
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).double().numpy()
    from oracle import round_bf16
    np.testing.assert_array_equal(round_bf16(x), ref)


def test_bf16_kv_cache_stores_rounded_values(tiny):
    _, m = tiny
    toks = synth.tokens(4, "kvdt", 12, synth.TINY.vocab)
    a, b = SeqCache(synth.TINY, 16), SeqCache(synth.TINY, 16, kv_dtype="bf16")
    m.forward([a], [toks])
    m.forward([b], [toks])
    from oracle import round_bf16
    # layer 0 sees identical inputs: its stored K/V are exactly the rounded exact ones
    np.testing.assert_array_equal(b.K[0][:12], round_bf16(a.K[0][:12]))
    np.testing.assert_array_equal(b.V[0][:12], round_bf16(a.V[0][:12]))
    assert np.abs(b.K[0][:12] - a.K[0][:12]).max() > 0
    for l in range(synth.TINY.n_layers):                       # every stored value is a bf16 value
        np.testing.assert_array_equal(b.K[l][:12], round_bf16(b.K[l][:12]))
        np.testing.assert_array_equal(b.V[l][:12], round_bf16(b.V[l][:12]))


def test_argmax_lowest_index_wins_exact_ties():
    """The tie rule of the per-row argmax: among exactly equal maxima the lowest
    vocabulary index is reported. Hand-made rows put the tie at the front, the
    back, far apart and across the whole row; random rows over a three-value
    alphabet (ties everywhere) are checked against the first index holding the
    row maximum, found by a plain scan."""
    from oracle import argmax_lowest
    rows = np.array([
        [5.0, 3.0, 5.0, 1.0, 5.0],      # tie at 0, 2, 4 -> 0
        [1.0, 7.0, 2.0, 7.0, 0.0],      # tie at 1, 3 -> 1
        [0.0, 0.0, 0.0, 0.0, 9.0],      # unique maximum at the end -> 4
        [-1.0, -2.0, -3.0, 4.0, 4.0],   # tie at the last two -> 3
        [2.5, 2.5, 2.5, 2.5, 2.5],      # all equal -> 0
        [-np.inf, -7.0, -np.inf, -7.0, -8.0],
    ])
    np.testing.assert_array_equal(argmax_lowest(rows), [0, 1, 4, 3, 0, 1])
    r = np.random.default_rng(7).integers(0, 3, size=(400, 37)).astype(np.float64)
    expect = [next(i for i in range(r.shape[1]) if r[k, i] == r[k].max()) for k in range(r.shape[0])]
    np.testing.assert_array_equal(argmax_lowest(r), expect)
    # a batch of logits [B, S, V] reduces over the last axis only
    np.testing.assert_array_equal(argmax_lowest(rows.reshape(2, 3, 5)), [[0, 1, 4], [3, 0, 1]])

"""Pins for the oracle's sampled verify (oracle/sampling.py).

The stream is pinned to SplitMix64's published outputs and to a second,
independent implementation (numpy uint64 arithmetic against Python integers);
the Gumbel-max draw to the softmax distribution it must sample (a frequency
test) and to greedy argmax at vanishing temperature; the loop to losslessness
([TS] the protocol: every emitted token is drawn from a trunk row, so
speculation on and off emit the same stream at a fixed seed).
"""
import numpy as np
import pytest

import oracle
import synth
from oracle import sampling
from synth import workloads

# SplitMix64 seeded with 0: the first outputs as published with the generator (Vigna's reference
# implementation; also the stream Java's SplittableRandom produces from seed 0 with its gamma).
SPLITMIX64_SEED0 = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F, 0xF88BB8A8724C81EC,
                    0x1B39896A51A8749B]


def test_stream_matches_published_splitmix64_outputs():
    assert [sampling.stream_int(0, i) for i in range(5)] == SPLITMIX64_SEED0


def test_vectorised_stream_matches_integer_arithmetic():
    rng = np.random.default_rng(3)
    for _ in range(20):
        seed, b, pos = int(rng.integers(0, 2**63)), int(rng.integers(0, 256)), int(rng.integers(0, 40000))
        u = sampling.uniforms(seed, b, pos, 300)
        k = sampling.stream_int(sampling.stream_int(seed, b), pos)
        expect = [((sampling.stream_int(k, v) >> 41) + 0.5) * 2.0 ** -23 for v in range(300)]
        np.testing.assert_array_equal(u, expect)
    assert u.min() > 0 and u.max() < 1
    # every u is a float32 value (23 bits after the point), so a float32 sampler sees the same u
    np.testing.assert_array_equal(u.astype(np.float32).astype(np.float64), u)


def test_gumbel_max_draws_follow_the_softmax():
    """Draws over 40,000 positions of one fixed row of logits: every token's frequency within four
    standard errors of softmax(logits / T), at two temperatures."""
    logits = np.array([1.5, 0.2, -0.7, 1.1, 0.0, -2.0])
    n = 40000
    for T in (1.0, 0.6):
        p = np.exp(logits / T) / np.exp(logits / T).sum()
        g = np.stack([sampling.gumbel(11, 0, pos, len(logits)) for pos in range(n)])
        draws = np.argmax(logits / T + g, axis=-1)
        freq = np.bincount(draws, minlength=len(logits)) / n
        se = np.sqrt(p * (1 - p) / n)
        assert np.all(np.abs(freq - p) < 4 * se), (T, freq, p)


def test_vanishing_temperature_is_greedy():
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((50, 400)) * 3
    greedy = oracle.argmax_lowest(logits)
    np.testing.assert_array_equal(sampling.draw_rows(logits, 0.0, 9, 2, range(50)), greedy)
    # margins here exceed 1e-3 while the noise spans [-2.8, 16.6]: at T = 1e-5 the logits dominate
    top2 = np.sort(logits, -1)[:, -2:]
    assert (top2[:, 1] - top2[:, 0]).min() > 1e-3
    np.testing.assert_array_equal(sampling.draw_rows(logits, 1e-5, 9, 2, range(50)), greedy)


def test_draws_depend_on_seed_sequence_and_position_only():
    rng = np.random.default_rng(6)
    logits = rng.standard_normal((4, 1000))
    a = sampling.draw_rows(logits, 1.0, 1, 0, [10, 11, 12, 13])
    np.testing.assert_array_equal(a, [sampling.draw_rows(logits[i:i + 1], 1.0, 1, 0, [10 + i])[0] for i in range(4)])
    assert (sampling.draw_rows(logits, 1.0, 1, 0, [10, 11, 12, 13]) == a).all()
    b = [sampling.draw_rows(logits, 1.0, s, q, [10, 11, 12, 13]) for s, q in ((2, 0), (1, 1))]
    assert not (b[0] == a).all() and not (b[1] == a).all()


@pytest.fixture(scope="module")
def tiny_model():
    shape = synth.TINY
    host = {n: synth.tensor(shape, 1, n) for n in shape.tensor_shapes()}
    return oracle.DenseDecoder(shape, lambda n: host[n])


@pytest.mark.parametrize("T", [0.05, 0.1])
def test_sampled_spec_on_equals_spec_off(tiny_model, T):
    """[TS] the protocol: drafts are accepted while the drawn token matches, so the sampled stream
    with n-gram drafts (fixed and adaptive K) is the plain sampled stream, token for token. The
    random-init tiny model's logits are small, so the temperatures are low enough for drafts to
    be accepted and still high enough for the stream to leave the greedy one."""
    prompt = workloads.motif_prompt(1)
    off, _, _ = oracle.generate(tiny_model, [prompt], 40, drafter="none", temperature=T, seed=21)
    on, recs, _ = oracle.generate(tiny_model, [prompt], 40, drafter="ngram", k=4, temperature=T, seed=21)
    ad, _, _ = oracle.generate(tiny_model, [prompt], 40, drafter="ngram", adaptive=True, temperature=T, seed=21)
    assert on == off and ad == off
    assert sum(r.m[0] for r in recs) > 0                    # some drafts were accepted
    greedy, _, _ = oracle.generate(tiny_model, [prompt], 40, drafter="none")
    assert off != greedy                                      # the sampler did draw
    for r in recs:                                            # 1..k+1 tokens per step
        assert 1 <= len(r.committed[0]) <= len(r.spans[0])


def test_sampled_batch_rows_use_their_own_slot(tiny_model):
    """Two sequences with the same prompt draw different streams (the noise is keyed by the
    sequence slot), and each equals its own single-sequence run in that slot."""
    prompt = workloads.motif_prompt(1)
    both, _, _ = oracle.generate(tiny_model, [prompt, prompt], 24, drafter="ngram", k=3, temperature=1.0, seed=4)
    assert both[0] != both[1]
    solo, _, _ = oracle.generate(tiny_model, [prompt], 24, drafter="none", temperature=1.0, seed=4)
    assert both[0] == solo[0]

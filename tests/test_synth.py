"""The seeded input generator against its published definition (pure Python)."""
import math
import struct

import numpy as np

import synth

M64 = (1 << 64) - 1


def _mix64(z):
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def _fnv1a64(s):
    h = 0xcbf29ce484222325
    for ch in s.encode():
        h = ((h ^ ch) * 0x100000001b3) & M64
    return h


def _u64(seed, name, i):
    key = _mix64(seed ^ _fnv1a64(name))
    return _mix64((key + (i + 1) * 0x9E3779B97F4A7C15) & M64)


def _bf16_rne(x):
    u = struct.unpack("<I", struct.pack("<f", x))[0]
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) & 0xFFFF


def test_raw_stream_matches_splitmix64_definition():
    for seed, name in [(1, "embed"), (2, "layers.0.wq"), (12345678901, "x")]:
        assert synth.key(seed, name) == _mix64(seed ^ _fnv1a64(name))
        for i in (0, 1, 2, 1000, 2**40):
            assert synth.u64(seed, name, i) == _u64(seed, name, i)


def test_normal_bf16_matches_box_muller_definition():
    bits = synth.normal_bf16(7, "w", 64, 0.02, offset=10)
    for j in range(64):
        i = 10 + j
        p = i // 2
        u1 = ((_u64(7, "w", 2 * p) >> 11) + 1) * 2.0 ** -53
        u2 = (_u64(7, "w", 2 * p + 1) >> 11) * 2.0 ** -53
        r = math.sqrt(-2 * math.log(u1))
        z = r * (math.cos(2 * math.pi * u2) if i % 2 == 0 else math.sin(2 * math.pi * u2))
        f = struct.unpack("<f", struct.pack("<f", 0.02 * z))[0]
        assert bits[j] == _bf16_rne(f)


def test_tokens_units_ints_match_definition():
    t = synth.tokens(3, "tok", 50, 151936, offset=5)
    assert all(t[j] == (_u64(3, "tok", 5 + j) * 151936) >> 64 for j in range(50))
    u = synth.unit(3, "u", 20)
    assert all(u[j] == (_u64(3, "u", j) >> 11) * 2.0 ** -53 for j in range(20))
    v = synth.ints(3, "i", 20, 512, 4096)
    assert all(v[j] == 512 + ((_u64(3, "i", j) * 3585) >> 64) for j in range(20))
    assert v.min() >= 512 and v.max() <= 4096


def test_offsets_are_consistent_and_statistics_sane():
    a = synth.normal_bf16(1, "big", 200001)
    b = synth.normal_bf16(1, "big", 1001, offset=99999)
    np.testing.assert_array_equal(a[99999:101000], b)
    f = synth.bf16_bits_to_f64(a)
    assert abs(f.mean()) < 2e-4 and abs(f.std() - 0.02) < 2e-4
    assert synth.TINY.weight_bytes() > 0 and synth.QWEN3_4B.kv_bytes_per_token() == 147456

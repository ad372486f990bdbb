"""Seeded synthetic inputs shared by the oracle and the GPU path.

Only input generation lives here (weights, token streams, uniform draws and
the workload recipes built from them). Nothing in this package computes any
step of speculative decoding; both the CPU oracle and the CUDA path consume
what it produces. The generator definition is in ``synth.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "_synth.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile synth.c into _synth.so beside it (gcc, OpenMP)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, i64, u32, d = ctypes.c_uint64, ctypes.c_int64, ctypes.c_uint32, ctypes.c_double
        p = ctypes.c_void_p
        lib.synth_key.restype = u64
        lib.synth_key.argtypes = [u64, ctypes.c_char_p]
        lib.synth_u64.restype = u64
        lib.synth_u64.argtypes = [u64, u64]
        lib.synth_normal_at.restype = d
        lib.synth_normal_at.argtypes = [u64, u64]
        lib.synth_normal_bf16.argtypes = [u64, ctypes.c_char_p, d, u64, u64, p]
        lib.synth_tokens.argtypes = [u64, ctypes.c_char_p, u64, u64, u32, p]
        lib.synth_unit.argtypes = [u64, ctypes.c_char_p, u64, u64, p]
        lib.synth_ints.argtypes = [u64, ctypes.c_char_p, u64, u64, i64, i64, p]
        _lib = lib
    return _lib


# ----------------------------------------------------------------------------- raw streams

def key(seed: int, name: str) -> int:
    return _load().synth_key(seed, name.encode())


def u64(seed: int, name: str, i: int) -> int:
    return _load().synth_u64(key(seed, name), i)


def normal_bf16(seed: int, name: str, n: int, std: float = 0.02, offset: int = 0) -> np.ndarray:
    """bf16 bit patterns (uint16) of std * N(0,1)."""
    out = np.empty(n, dtype=np.uint16)
    if n:
        _load().synth_normal_bf16(seed, name.encode(), std, offset, n, out.ctypes.data)
    return out


def tokens(seed: int, name: str, n: int, vocab: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    if n:
        _load().synth_tokens(seed, name.encode(), offset, n, vocab, out.ctypes.data)
    return out


def unit(seed: int, name: str, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    if n:
        _load().synth_unit(seed, name.encode(), offset, n, out.ctypes.data)
    return out


def ints(seed: int, name: str, n: int, lo: int, hi: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.int64)
    if n:
        _load().synth_ints(seed, name.encode(), offset, n, lo, hi, out.ctypes.data)
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------- model shapes

@dataclass(frozen=True)
class Shape:
    """Dense decoder shape (pre-norm, GQA attention, SwiGLU FFN)."""
    name: str
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    qk_norm: bool = True
    swa_window: int = 0        # > 0: local (sliding-window) layers attend the last swa_window positions
    swa_global_every: int = 0  # with a window: layer l is global iff (l + 1) % swa_global_every == 0 (0: none)

    def with_layers(self, n: int) -> "Shape":
        return Shape(f"{self.name}-L{n}", n, self.hidden, self.n_q_heads, self.n_kv_heads, self.head_dim,
                     self.ffn, self.vocab, self.rms_eps, self.rope_theta, self.qk_norm, self.swa_window,
                     self.swa_global_every)

    def with_window(self, window: int, global_every: int = 0) -> "Shape":
        return Shape(f"{self.name}-W{window}", self.n_layers, self.hidden, self.n_q_heads, self.n_kv_heads,
                     self.head_dim, self.ffn, self.vocab, self.rms_eps, self.rope_theta, self.qk_norm, window,
                     global_every)

    def is_local(self, layer: int) -> bool:
        """Whether `layer` is a sliding-window layer."""
        if self.swa_window <= 0:
            return False
        return self.swa_global_every <= 0 or (layer + 1) % self.swa_global_every != 0

    def tensor_shapes(self) -> dict:
        H, D, F, V = self.hidden, self.head_dim, self.ffn, self.vocab
        s = {"embed": (V, H), "lm_head": (V, H), "final_norm": (H,)}
        for l in range(self.n_layers):
            p = f"layers.{l}."
            s[p + "attn_norm"] = (H,)
            s[p + "wq"] = (self.n_q_heads * D, H)
            s[p + "wk"] = (self.n_kv_heads * D, H)
            s[p + "wv"] = (self.n_kv_heads * D, H)
            s[p + "q_norm"] = (D,)
            s[p + "k_norm"] = (D,)
            s[p + "wo"] = (H, self.n_q_heads * D)
            s[p + "ffn_norm"] = (H,)
            s[p + "w_gate"] = (F, H)
            s[p + "w_up"] = (F, H)
            s[p + "w_down"] = (H, F)
        return s

    def weight_bytes(self) -> int:
        return 2 * sum(int(np.prod(v)) for v in self.tensor_shapes().values())

    def kv_bytes_per_token(self) -> int:
        return 2 * self.n_kv_heads * self.head_dim * 2 * self.n_layers


# Tiny decoder: 2 layers, hidden 256, 4 q heads / 2 KV heads of dim 64, FFN 688, vocab 2048.
TINY = Shape("tiny", 2, 256, 4, 2, 64, 688, 2048)
# Qwen3-4B-shaped decoder: 36 layers, hidden 2560, 32 q / 8 KV heads of dim 128, FFN 9728, vocab 151936.
QWEN3_4B = Shape("qwen3-4b", 36, 2560, 32, 8, 128, 9728, 151936)

NORM_NAMES = ("attn_norm", "ffn_norm", "q_norm", "k_norm", "final_norm")
BF16_ONE = np.uint16(0x3F80)


def tensor(shape: Shape, seed: int, name: str) -> np.ndarray:
    """One weight tensor as bf16 bit patterns. Matrices and the embedding are
    N(0, 0.02); every norm gain is 1.0."""
    dims = shape.tensor_shapes()[name]
    n = int(np.prod(dims))
    if name.split(".")[-1] in NORM_NAMES:
        return np.full(dims, BF16_ONE, dtype=np.uint16)
    return normal_bf16(seed, name, n, 0.02).reshape(dims)


def weights(shape: Shape, seed: int) -> dict:
    return {name: tensor(shape, seed, name) for name in shape.tensor_shapes()}

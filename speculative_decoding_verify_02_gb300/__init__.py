"""Python binding for libsdv (include/sdv.h): the speculative-decoding verify
path on one GB300.

Argument marshalling only: every step of the path runs in the CUDA kernels
behind the C ABI. PyTorch supplies device memory and streams. If the CUDA
library is missing or cannot be loaded, importing the binding's entry points
raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsdv.so")

SDV_OK = 0
SDV_ERR_ARG = -1
SDV_ERR_CAPACITY = -2
SDV_ERR_CUDA = -3
SDV_ERR_DEVICE = -4
SDV_ERR_DEVICE_TIMEOUT = -5
SDV_ERR_UNSUPPORTED = -6
SDV_DRAFT_NONE, SDV_DRAFT_NGRAM, SDV_DRAFT_TABLE = 0, 1, 2

# Every entry point include/sdv.h declares.
EXPORTS = (
    "sdv_workspace_bytes", "sdv_kv_pool_bytes", "sdv_create", "sdv_destroy", "sdv_ensure_capacity",
    "sdv_spec_forward", "sdv_spec_forward_sampled", "sdv_accept_greedy", "sdv_rewind_cache", "sdv_cache_seq_len", "sdv_page_table",
    "sdv_ngram_commit", "sdv_gen_init", "sdv_propose", "sdv_reset_seq", "sdv_get_status", "sdv_status_str",
    "sdv_op_attention", "sdv_profile_enable", "sdv_profile_read", "sdv_paged_attention_noalloc",
    "sdv_fwd_trace", "sdv_noalloc_status", "sdv_ngram_params", "sdv_governor_create", "sdv_governor_destroy",
    "sdv_governor_decide", "sdv_governor_record", "sdv_governor_new_request", "sdv_governor_stats",
)
PHASES = ("prepare", "qkv_gemm", "attention", "o_gemm", "gateup_gemm", "down_gemm", "lmhead_gemm")
# sdv_fwd_trace: stamps per CTA, CTAs per region (one region per launch of a forward)
TRACE_STAMPS, TRACE_REGION_CTAS = 16, 8192


class SdvError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_str(code)} ({code})")
        self.code = code


class ModelCfg(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("hidden", ctypes.c_int), ("n_q_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("vocab", ctypes.c_int), ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
                ("qk_norm", ctypes.c_int), ("swa_window", ctypes.c_int), ("swa_global_every", ctypes.c_int)]


class CacheCfg(ctypes.Structure):
    _fields_ = [("page_size", ctypes.c_int), ("n_pages", ctypes.c_int), ("max_batch", ctypes.c_int),
                ("max_rows", ctypes.c_int), ("max_span", ctypes.c_int), ("max_context", ctypes.c_int),
                ("ngram_capacity", ctypes.c_int), ("ngram_max_order", ctypes.c_int)]


class GovernorCfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("probe_steps", "reprobe_steps", "first_park", "max_park", "hold_window",
                                              "remeasure_every", "remeasure_steps", "zero_accept_end",
                                              "baseline_samples")]


class GovernorStats(ctypes.Structure):
    _fields_ = [("plain_ms_per_tok", ctypes.c_float), ("spec_ms_per_tok", ctypes.c_float), ("wins", ctypes.c_int),
                ("losses", ctypes.c_int), ("parked_steps", ctypes.c_int), ("state", ctypes.c_int)]


LAYER_FIELDS = ("attn_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo", "ffn_norm", "w_gate", "w_up", "w_down")


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in LAYER_FIELDS]


class Weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("lm_head", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
                ("layers", ctypes.POINTER(LayerWeights))]


_lib = None


def lib():
    """Load libsdv.so (built by __graft_entry__.build() or build.py); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing (run the build step)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    P = ctypes.POINTER
    L.sdv_workspace_bytes.argtypes = [P(ModelCfg), P(CacheCfg), P(sz)]
    L.sdv_kv_pool_bytes.argtypes = [P(ModelCfg), P(CacheCfg), P(sz)]
    L.sdv_create.argtypes = [P(ModelCfg), P(CacheCfg), P(Weights), vp, vp, vp, P(vp)]
    L.sdv_destroy.argtypes = [vp]
    L.sdv_ensure_capacity.argtypes = [vp, vp, i32, vp]
    L.sdv_spec_forward.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, vp]
    L.sdv_spec_forward_sampled.argtypes = [vp, vp, vp, i32, i32, i32, vp, ctypes.c_uint64, vp, vp, vp]
    L.sdv_accept_greedy.argtypes = [vp, vp, vp, vp, i32, i32, vp, vp, vp, vp, vp]
    L.sdv_rewind_cache.argtypes = [vp, vp, i32, vp]
    L.sdv_cache_seq_len.argtypes = [vp, vp, vp]
    L.sdv_page_table.argtypes = [vp, vp, vp, vp, vp]
    L.sdv_ngram_commit.argtypes = [vp, vp, vp, i32, i32, vp]
    L.sdv_gen_init.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp]
    L.sdv_ngram_params.argtypes = [vp, i32, ctypes.c_float]
    L.sdv_governor_create.argtypes = [P(GovernorCfg), P(vp)]
    L.sdv_governor_destroy.argtypes = [vp]
    L.sdv_governor_decide.argtypes = [vp, P(ctypes.c_int32)]
    L.sdv_governor_record.argtypes = [vp, i32, ctypes.c_float, i32, i32, i32]
    L.sdv_governor_new_request.argtypes = [vp]
    L.sdv_governor_stats.argtypes = [vp, P(GovernorStats)]
    L.sdv_propose.argtypes = [vp, i32, vp, i32, i32, i32, vp, vp, vp, vp]
    L.sdv_reset_seq.argtypes = [vp, i32, vp]
    L.sdv_get_status.argtypes = [vp, P(ctypes.c_int32)]
    L.sdv_status_str.argtypes = [i32]
    L.sdv_status_str.restype = ctypes.c_char_p
    L.sdv_op_attention.argtypes = [vp, i32, vp, vp, vp, i32, i32, vp, vp]
    L.sdv_profile_enable.argtypes = [vp, i32]
    L.sdv_profile_read.argtypes = [vp, P(ctypes.c_float), P(ctypes.c_int32)]
    L.sdv_fwd_trace.argtypes = [vp, vp, ctypes.c_size_t]
    L.sdv_paged_attention_noalloc.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp]
    L.sdv_noalloc_status.argtypes = [P(ctypes.c_int32)]
    for name in EXPORTS:
        if name != "sdv_status_str":
            getattr(L, name).restype = i32
    _lib = L
    return L


def status_str(code: int) -> str:
    return lib().sdv_status_str(code).decode()


def _check(code: int, what: str):
    if code != SDV_OK:
        raise SdvError(code, what)


def model_cfg(shape) -> ModelCfg:
    return ModelCfg(shape.n_layers, shape.hidden, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, shape.ffn,
                    shape.vocab, shape.rms_eps, shape.rope_theta, 1 if shape.qk_norm else 0,
                    getattr(shape, "swa_window", 0), getattr(shape, "swa_global_every", 0))


def workspace_bytes(mcfg: ModelCfg, ccfg: CacheCfg) -> int:
    n = ctypes.c_size_t()
    _check(lib().sdv_workspace_bytes(ctypes.byref(mcfg), ctypes.byref(ccfg), ctypes.byref(n)), "workspace_bytes")
    return n.value


def kv_pool_bytes(mcfg: ModelCfg, ccfg: CacheCfg) -> int:
    n = ctypes.c_size_t()
    _check(lib().sdv_kv_pool_bytes(ctypes.byref(mcfg), ctypes.byref(ccfg), ctypes.byref(n)), "kv_pool_bytes")
    return n.value


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _stream(stream) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def paged_attention_noalloc(q, kv_layer, page_table, pages_per_seq, page_size, n_pages, row_off, base, B,
                            n_q_heads, n_kv_heads, head_dim, max_span, max_context, out, stream=None):
    """Paged attention with no device allocation (scratch in a static device array)."""
    _check(lib().sdv_paged_attention_noalloc(_ptr(q), _ptr(kv_layer), _ptr(page_table), pages_per_seq, page_size,
                                             n_pages, _ptr(row_off), _ptr(base), B, n_q_heads, n_kv_heads, head_dim,
                                             max_span, max_context, _ptr(out), _stream(stream)),
           "paged_attention_noalloc")


def noalloc_status() -> int:
    """Status word of the last paged_attention_noalloc call on the current device (synchronises,
    then clears it)."""
    v = ctypes.c_int32()
    _check(lib().sdv_noalloc_status(ctypes.byref(v)), "noalloc_status")
    return v.value


def upload_bf16(bits: np.ndarray, device="cuda"):
    """bf16 bit patterns (uint16 numpy) -> a torch bfloat16 device tensor."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


class Governor:
    """The speculation cost governor (host policy in the library): decide() before a step,
    record() after it."""
    STATES = ("calibrate", "probe", "hold", "remeasure", "parked")

    def __init__(self, cfg: GovernorCfg = None):
        g = ctypes.c_void_p()
        _check(lib().sdv_governor_create(ctypes.byref(cfg) if cfg is not None else None, ctypes.byref(g)),
               "governor_create")
        self.g = g

    def decide(self) -> bool:
        v = ctypes.c_int32()
        _check(lib().sdv_governor_decide(self.g, ctypes.byref(v)), "governor_decide")
        return bool(v.value)

    def record(self, speculative: bool, ms: float, committed: int, drafted: int, accepted: int):
        _check(lib().sdv_governor_record(self.g, int(speculative), float(ms), int(committed), int(drafted),
                                         int(accepted)), "governor_record")

    def new_request(self):
        _check(lib().sdv_governor_new_request(self.g), "governor_new_request")

    def stats(self) -> dict:
        s = GovernorStats()
        _check(lib().sdv_governor_stats(self.g, ctypes.byref(s)), "governor_stats")
        return {"plain_ms_per_tok": None if s.plain_ms_per_tok < 0 else s.plain_ms_per_tok,
                "spec_ms_per_tok": None if s.spec_ms_per_tok < 0 else s.spec_ms_per_tok,
                "wins": s.wins, "losses": s.losses, "parked": s.parked_steps, "state": self.STATES[s.state]}

    def close(self):
        if self.g:
            lib().sdv_governor_destroy(self.g)
            self.g = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Verifier:
    """One context: borrowed weights, a KV pool and a workspace, all torch-owned."""

    def __init__(self, shape, weights: dict, page_size=16, n_pages=1024, max_batch=1, max_rows=32, max_span=17,
                 max_context=4096, ngram_capacity=0, ngram_max_order=0, stream=None):
        import torch
        self.shape = shape
        self.mcfg = model_cfg(shape)
        self.ccfg = CacheCfg(page_size, n_pages, max_batch, max_rows, max_span, max_context, ngram_capacity,
                             ngram_max_order)
        self.weights = weights                       # name -> torch bf16 device tensor (kept alive)
        self.pool = torch.empty(kv_pool_bytes(self.mcfg, self.ccfg), dtype=torch.uint8, device="cuda")
        self.workspace = torch.empty(workspace_bytes(self.mcfg, self.ccfg) + 256, dtype=torch.uint8, device="cuda")
        base = _ptr(self.workspace)
        self._ws_ptr = (base + 255) // 256 * 256
        layers = (LayerWeights * shape.n_layers)()
        for l in range(shape.n_layers):
            for f in LAYER_FIELDS:
                setattr(layers[l], f, _ptr(weights[f"layers.{l}.{f}"]))
        self._layers = layers
        self._w = Weights(_ptr(weights["embed"]), _ptr(weights["lm_head"]), _ptr(weights["final_norm"]),
                          ctypes.cast(layers, ctypes.POINTER(LayerWeights)))
        ctx = ctypes.c_void_p()
        _check(lib().sdv_create(ctypes.byref(self.mcfg), ctypes.byref(self.ccfg), ctypes.byref(self._w),
                                _ptr(self.pool), self._ws_ptr, _stream(stream), ctypes.byref(ctx)), "sdv_create")
        self.ctx = ctx
        self.pages_per_seq = -(-max_context // page_size)

    def close(self):
        if self.ctx:
            lib().sdv_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # --- the ABI, one method per call (device tensors in, device tensors out)
    def ensure_capacity(self, required, B, stream=None):
        _check(lib().sdv_ensure_capacity(self.ctx, _ptr(required), B, _stream(stream)), "ensure_capacity")

    def spec_forward(self, tokens, row_off, B, max_rows, max_span, argmax, logits=None, stream=None):
        _check(lib().sdv_spec_forward(self.ctx, _ptr(tokens), _ptr(row_off), B, max_rows, max_span, _ptr(argmax),
                                      _ptr(logits), _stream(stream)), "spec_forward")

    def spec_forward_sampled(self, tokens, row_off, B, max_rows, max_span, temperature, seed, drawn, logits=None,
                             stream=None):
        """The verify forward with each row drawn at its sequence's temperature (float32 device
        tensor [B]; <= 0 = greedy) from the noise keyed by `seed`, the sequence slot and the row's
        position."""
        _check(lib().sdv_spec_forward_sampled(self.ctx, _ptr(tokens), _ptr(row_off), B, max_rows, max_span,
                                              _ptr(temperature), int(seed) & (2**64 - 1), _ptr(drawn),
                                              _ptr(logits), _stream(stream)), "spec_forward_sampled")

    def accept_greedy(self, tokens, row_off, argmax, B, max_commit, n_accept, committed, n_commit, new_len,
                      stream=None):
        _check(lib().sdv_accept_greedy(self.ctx, _ptr(tokens), _ptr(row_off), _ptr(argmax), B, max_commit,
                                       _ptr(n_accept), _ptr(committed), _ptr(n_commit), _ptr(new_len),
                                       _stream(stream)), "accept_greedy")

    def rewind_cache(self, length, B, stream=None):
        _check(lib().sdv_rewind_cache(self.ctx, _ptr(length), B, _stream(stream)), "rewind_cache")

    def cache_seq_len(self, out, stream=None):
        _check(lib().sdv_cache_seq_len(self.ctx, _ptr(out), _stream(stream)), "cache_seq_len")

    def page_table(self, table, n_pages, free_top, stream=None):
        _check(lib().sdv_page_table(self.ctx, _ptr(table), _ptr(n_pages), _ptr(free_top), _stream(stream)),
               "page_table")

    def ngram_commit(self, tokens, counts, B, stride, stream=None):
        _check(lib().sdv_ngram_commit(self.ctx, _ptr(tokens), _ptr(counts), B, stride, _stream(stream)),
               "ngram_commit")

    def gen_init(self, first, budget, B, k_init, adaptive, k_max, stream=None):
        _check(lib().sdv_gen_init(self.ctx, _ptr(first), _ptr(budget), B, k_init, int(adaptive), k_max,
                                  _stream(stream)), "gen_init")

    def ngram_params(self, min_order, pmin=0.0):
        _check(lib().sdv_ngram_params(self.ctx, min_order, float(pmin)), "ngram_params")

    def propose(self, drafter, table, table_stride, B, max_span, tokens, row_off, required, stream=None):
        _check(lib().sdv_propose(self.ctx, drafter, _ptr(table), table_stride, B, max_span, _ptr(tokens),
                                 _ptr(row_off), _ptr(required), _stream(stream)), "propose")

    def reset_seq(self, b, stream=None):
        _check(lib().sdv_reset_seq(self.ctx, b, _stream(stream)), "reset_seq")

    def get_status(self) -> int:
        v = ctypes.c_int32()
        _check(lib().sdv_get_status(self.ctx, ctypes.byref(v)), "get_status")
        return v.value

    def profile_enable(self, on: bool):
        _check(lib().sdv_profile_enable(self.ctx, int(on)), "profile_enable")

    def profile_read(self):
        """{phase: (total ms, launches)} since the last read (synchronises)."""
        ms = (ctypes.c_float * len(PHASES))()
        cnt = (ctypes.c_int32 * len(PHASES))()
        _check(lib().sdv_profile_read(self.ctx, ms, cnt), "profile_read")
        return {PHASES[i]: (ms[i], cnt[i]) for i in range(len(PHASES))}

    def fwd_trace(self, buf):
        """Record the per-launch, per-CTA device timeline of later forwards into
        `buf` (an int64 device tensor of regions x 2048 x 16), or stop with None."""
        n = buf.numel() * buf.element_size() if buf is not None else 0
        _check(lib().sdv_fwd_trace(self.ctx, _ptr(buf) if buf is not None else None, n), "fwd_trace")

    def op_attention(self, layer, q, row_off, base, B, max_span, out, stream=None):
        _check(lib().sdv_op_attention(self.ctx, layer, _ptr(q), _ptr(row_off), _ptr(base), B, max_span, _ptr(out),
                                      _stream(stream)), "op_attention")

"""Host-side sequencing of the C ABI for whole generations.

Nothing here computes a step of the method: it only orders the library calls
(prefill chunks, then per step propose -> ensure_capacity -> spec_forward ->
accept_greedy -> rewind_cache -> ngram_commit), owns the device buffers those
calls read and write, can capture one step as a CUDA graph so that a step
costs one launch, and can let the library's speculation cost governor decide
each step. Every length the kernels need stays in device memory, so a
captured step replays correctly whatever the spans and cache lengths are.
"""
from __future__ import annotations

import numpy as np

from . import SDV_DRAFT_NGRAM, SDV_DRAFT_NONE, SDV_DRAFT_TABLE, Verifier  # noqa: F401


def _i32(n, device="cuda"):
    import torch
    return torch.zeros(max(1, n), dtype=torch.int32, device=device)


class SpecLoop:
    """Buffers and call order for B sequences with verify spans of at most max_span rows."""

    def __init__(self, v: Verifier, B: int, max_span: int):
        import torch
        self.v, self.B, self.max_span = v, B, max_span
        self.max_rows = B * max_span
        assert self.max_rows <= v.ccfg.max_rows and max_span <= v.ccfg.max_span
        self.tokens = _i32(self.max_rows)
        self.row_off = _i32(B + 1)
        self.required = _i32(B)
        self.argmax = _i32(self.max_rows)
        self.n_accept = _i32(B)
        self.committed = _i32(B * max_span)
        self.n_commit = _i32(B)
        self.new_len = _i32(B)
        self.first = _i32(B)
        self.budget = _i32(B)
        self.logits = None
        self.graph = None
        self.stream = torch.cuda.current_stream()

    # ------------------------------------------------------------------ prefill
    def prefill(self, prompts, chunk: int = 128, ngram: bool = False, temperature=None, seed: int = 0):
        """Forward each prompt in chunks (sequence by sequence, a capacity
        reservation before each chunk); returns the first generated token of
        each sequence (host numpy) and leaves it in self.first. With
        `temperature` (a float32 device tensor [B]) the first token is drawn
        by the sampled verify's sampler instead of taken as the argmax."""
        import torch
        B, v = self.B, self.v
        assert chunk <= v.ccfg.max_span and chunk <= v.ccfg.max_rows
        tok = _i32(chunk)
        ro = _i32(B + 1)
        req = _i32(B)
        am = _i32(chunk)
        first = np.zeros(B, dtype=np.int32)
        lens = np.zeros(B, dtype=np.int64)
        for b in range(B):
            p = np.asarray(prompts[b], dtype=np.int32)
            for c0 in range(0, len(p), chunk):
                piece = p[c0:c0 + chunk]
                n = len(piece)
                offs = np.zeros(B + 1, dtype=np.int32)
                offs[b + 1:] = n
                r = np.full(B, -1, dtype=np.int32)
                lens[b] += n
                r[b] = lens[b]
                tok[:n].copy_(torch.from_numpy(piece))
                ro.copy_(torch.from_numpy(offs))
                req.copy_(torch.from_numpy(r))
                v.ensure_capacity(req, B)
                if temperature is None:
                    v.spec_forward(tok, ro, B, max(n, 1), max(n, 1), am)
                else:
                    v.spec_forward_sampled(tok, ro, B, max(n, 1), max(n, 1), temperature, seed, am)
            first[b] = int(am[len(p) - 1 - (len(p) - 1) // chunk * chunk].item())
        self.first.copy_(torch.from_numpy(first))
        if ngram:
            # the n-gram history starts as prompt + first token
            for b in range(B):
                p = np.concatenate([np.asarray(prompts[b], dtype=np.int32), first[b:b + 1]])
                buf = torch.from_numpy(np.ascontiguousarray(p)).cuda()
                counts = torch.zeros(B, dtype=torch.int32, device="cuda")
                counts[b] = len(p)
                stride = len(p)
                allbuf = torch.zeros(B * stride, dtype=torch.int32, device="cuda")
                allbuf[b * stride:(b + 1) * stride] = buf
                v.ngram_commit(allbuf, counts, B, stride)
        return first

    def start(self, budget, k_init: int, adaptive: bool = False, k_max: int = 7):
        import torch
        self.budget.copy_(torch.as_tensor(np.asarray(budget, dtype=np.int32)))
        self.v.gen_init(self.first, self.budget, self.B, k_init, adaptive, k_max)

    # ------------------------------------------------------------------ one step
    def step(self, drafter=SDV_DRAFT_NGRAM, table=None, table_stride=0, logits=None, ngram=True, temperature=None,
             seed: int = 0):
        """One transaction: propose, reserve, verify (greedy, or sampled at `temperature`, a float32
        device tensor [B]), accept, rewind, and commit to the n-gram index."""
        v, B = self.v, self.B
        v.propose(drafter, table, table_stride, B, self.max_span, self.tokens, self.row_off, self.required)
        v.ensure_capacity(self.required, B)
        if temperature is None:
            v.spec_forward(self.tokens, self.row_off, B, self.max_rows, self.max_span, self.argmax, logits)
        else:
            v.spec_forward_sampled(self.tokens, self.row_off, B, self.max_rows, self.max_span, temperature, seed,
                                   self.argmax, logits)
        v.accept_greedy(self.tokens, self.row_off, self.argmax, B, self.max_span, self.n_accept, self.committed,
                        self.n_commit, self.new_len)
        v.rewind_cache(self.new_len, B)
        if ngram:
            v.ngram_commit(self.committed, self.n_commit, B, self.max_span)

    def governed_step(self, governor, drafter=SDV_DRAFT_NGRAM, **kw):
        """One step under the speculation cost governor: it decides whether this step drafts (else
        a plain one-row step through the same calls), the step's device time is measured with CUDA
        events, and the governor records it with the tokens committed, drafted and accepted over
        the batch. Returns (speculated, committed tokens, ms). Synchronises once per step."""
        import torch
        spec = governor.decide()
        s = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        self.step(drafter=drafter if spec else SDV_DRAFT_NONE, **kw)
        e1.record(s)
        e1.synchronize()
        ms = e0.elapsed_time(e1)
        n_commit = self.n_commit.cpu().numpy()
        n_accept = self.n_accept.cpu().numpy()
        spans = np.diff(self.row_off.cpu().numpy())
        committed = int(n_commit.sum())
        drafted = int(np.clip(spans - 1, 0, None).sum())
        accepted = int(np.clip(n_accept, 0, None).sum())
        if committed > 0:  # a step after every budget is met is not a sample
            governor.record(spec, ms, committed, drafted, accepted)
        return spec, committed, ms

    def capture(self, **kw):
        """Capture one step as a CUDA graph (replayed by replay())."""
        import torch
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                self.step(**kw)
        torch.cuda.current_stream().wait_stream(s)
        self.graph = g
        return g

    def replay(self):
        self.graph.replay()

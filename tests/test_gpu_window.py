"""Sliding-window (ring) KV layers on the GPU against the oracle.

[TS] sliding-window caches and rollback: a local layer keeps exactly one window
of positions in a ring (slot = position % W). A verify writes every row's K/V at
its true position and so evicts the positions W back; the device keeps what a
span evicts, reads it for the span's own earlier rows, and after acceptance puts
the rejected rows back (nothing on a full acceptance). The oracle keeps the
whole history and masks to the window, the plain definition; the device must
reproduce it through every wrap, partial acceptance and rewind.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import workloads
from tests.helpers import check_rows, upload_weights

pytestmark = pytest.mark.gpu


def _t(a):
    import torch
    return torch.as_tensor(np.asarray(a, dtype=np.int32)).cuda()


@pytest.fixture(scope="module")
def tiny_weights():
    import torch
    torch.cuda.init()
    return upload_weights(synth.TINY, 1)


def _verifier(shape, dev, **kw):
    from speculative_decoding_verify_02_gb300 import Verifier
    cfg = dict(page_size=16, n_pages=256, max_batch=2, max_rows=128, max_span=32, max_context=1024,
               ngram_capacity=2048)
    cfg.update(kw)
    return Verifier(shape, dev, **cfg)


@pytest.mark.parametrize("window,global_every,k", [(32, 2, 4), (48, 0, 7), (16, 0, 7)])
def test_window_spec_loop_teacher_forced(tiny_weights, window, global_every, k):
    """Tiny decoder with local layers (window 32 next to a global layer; every layer local with
    windows 48 and 16): the oracle's n-gram loop over the 128-token motif prompt (the rings wrap
    several times, drafts are partly accepted) drives the GPU step by step; per-row logits,
    argmax, acceptance, new lengths, then the oracle's rewind with the ring restore."""
    import torch
    host, dev = tiny_weights
    shape = synth.TINY.with_window(window, global_every)
    om = oracle.DenseDecoder(shape, lambda n: host[n])
    prompt = workloads.motif_prompt(1)
    chunk = min(32, window)
    streams, recs, _ = oracle.generate(om, [prompt], 40, drafter="ngram", k=k, keep_logits=True, kv_dtype="bf16",
                                       prefill_chunk=chunk)
    v = _verifier(shape, dev, max_batch=1, max_span=min(window, 32))
    from speculative_decoding_verify_02_gb300.runner import SpecLoop
    first = SpecLoop(v, 1, 8).prefill([prompt], chunk=chunk)
    ref_first = streams[0][0]
    n_acc, com, n_com, new_len = _t([0]), _t(np.zeros(8)), _t([0]), _t([0])
    flips_all, exact, partial = [], 0, 0
    for step, r in enumerate(recs):
        span = r.spans[0]
        S = len(span)
        v.ensure_capacity(_t([r.len_before[0] + S]), 1)
        lg = torch.zeros(S, shape.vocab, dtype=torch.float32, device="cuda")
        am = _t(np.zeros(S))
        tok, ro = _t(span), _t([0, S])
        v.spec_forward(tok, ro, 1, S, S, am, lg)
        v.accept_greedy(tok, ro, am, 1, 8, n_acc, com, n_com, new_len)
        torch.cuda.synchronize()
        assert v.get_status() == 0, step
        flips, _ = check_rows(lg.cpu().numpy(), am.cpu().numpy(), r.logits[0], f"W{window} step {step}")
        flips_all += [(step, f) for f in flips]
        if not flips:
            exact += 1
            assert n_acc[0].item() == r.m[0] and new_len[0].item() == r.new_len[0], step
        partial += 0 < r.m[0] + 1 < S
        v.rewind_cache(_t([r.new_len[0]]), 1)                  # teacher forcing; restores rejected slots
    torch.cuda.synchronize()
    assert v.get_status() == 0
    assert partial >= 1, "a partial acceptance past the wrap was exercised"
    print(f"window {window}/{global_every}: {exact}/{len(recs)} steps exact, {partial} partial, flips {flips_all}, "
          f"first token {int(first[0])} vs {ref_first}")
    v.close()


def test_window_spec_on_equals_spec_off(tiny_weights):
    """Rollback over the rings is exact on the device: the n-gram loop (K = 7, eager and captured
    as a CUDA graph) gives the plain loop's stream, with every layer local (window 16)."""
    import torch
    from speculative_decoding_verify_02_gb300 import SDV_DRAFT_NGRAM, SDV_DRAFT_NONE
    from speculative_decoding_verify_02_gb300.runner import SpecLoop
    host, dev = tiny_weights
    shape = synth.TINY.with_window(16, 0)
    prompts = [workloads.motif_prompt(1), synth.tokens(8, "win.p2", 70, shape.vocab)]

    def run(drafter, graph):
        v = _verifier(shape, dev, max_span=16)
        loop = SpecLoop(v, 2, 8)
        first = loop.prefill(prompts, chunk=16, ngram=True)
        loop.start([48, 48], k_init=7 if drafter else 0)
        kw = dict(drafter=drafter, ngram=True)
        if graph:
            loop.capture(**kw)
        streams = [[int(f)] for f in first]
        acc = 0
        for _ in range(60):
            loop.replay() if graph else loop.step(**kw)
            torch.cuda.synchronize()
            nc, cm = loop.n_commit.cpu().numpy(), loop.committed.cpu().numpy().reshape(2, 8)
            acc += int(np.clip(loop.n_accept.cpu().numpy(), 0, None).sum())
            for b in range(2):
                streams[b] += cm[b, :nc[b]].tolist()
            if all(len(s) >= 48 for s in streams):
                break
        assert v.get_status() == 0
        v.close()
        return streams, acc

    off, _ = run(SDV_DRAFT_NONE, False)
    on, acc = run(SDV_DRAFT_NGRAM, False)
    ong, _ = run(SDV_DRAFT_NGRAM, True)
    assert on == off and ong == off and acc > 0


def test_window_4b_shape_verify():
    """The 4B shape (2 layers: a local layer with a 512-position window, then a global one) at an
    848-token context, so the ring has wrapped: one verify of 8 rows against the oracle."""
    import torch
    from speculative_decoding_verify_02_gb300 import Verifier
    from speculative_decoding_verify_02_gb300.runner import SpecLoop
    shape = synth.QWEN3_4B.with_layers(2).with_window(512, 2)
    host, dev = upload_weights(shape, 2)
    om = oracle.DenseDecoder(shape, lambda n: host[n])
    ctx = workloads.uniform_context(2, 848, shape.vocab, name="window.ctx")
    cache = oracle.SeqCache(shape, 900, kv_dtype="bf16")
    om.forward([cache], [ctx], last_row_logits=True)
    v = Verifier(shape, dev, page_size=16, n_pages=128, max_batch=1, max_rows=128, max_span=128, max_context=1024)
    SpecLoop(v, 1, 8).prefill([ctx], chunk=128)
    span = [int(t) for t in synth.tokens(2, "window.span", 8, shape.vocab)]
    ref = om.forward([cache], [span])[0]
    v.ensure_capacity(_t([856]), 1)
    am = _t(np.zeros(8))
    lg = torch.zeros(8, shape.vocab, dtype=torch.float32, device="cuda")
    v.spec_forward(_t(span), _t([0, 8]), 1, 8, 8, am, lg)
    torch.cuda.synchronize()
    assert v.get_status() == 0
    flips, d = check_rows(lg.cpu().numpy(), am.cpu().numpy(), ref, "4B window verify")
    print(f"4B window 512: max |dlogit| {d:.3e}, flips {flips}")
    v.close()

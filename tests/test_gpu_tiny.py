"""Tiny decoder (2 layers, hidden 256, 4/2 heads of 64, FFN 688, vocab 2048):
the full verify path on the GPU against the float64 oracle, teacher-forced.

The oracle's spec loop (128-token motif prompt, 2-gram lookup, K=4, 32 tokens)
drives both sides: each step the GPU verifies the oracle's span, and per-row
logits, argmax (outside near-ties), acceptance, committed tokens, new lengths
and page tables are compared.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import workloads
from tests.helpers import check_rows, upload_weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny():
    import torch
    from speculative_decoding_verify_02_gb300 import Verifier
    torch.cuda.init()
    host, dev = upload_weights(synth.TINY, 1)
    model = oracle.DenseDecoder(synth.TINY, lambda n: host[n])
    return host, dev, model


def _verifier(dev, **kw):
    from speculative_decoding_verify_02_gb300 import Verifier
    cfg = dict(page_size=16, n_pages=64, max_batch=1, max_rows=128, max_span=128, max_context=512,
               ngram_capacity=1024)
    cfg.update(kw)
    return Verifier(synth.TINY, dev, **cfg)


def _t(a):
    import torch
    return torch.as_tensor(np.asarray(a, dtype=np.int32)).cuda()


def test_tiny_prefill_logits(tiny):
    import torch
    host, dev, model = tiny
    v = _verifier(dev)
    prompt = workloads.motif_prompt(1)
    ref = model.forward([oracle.SeqCache(synth.TINY, 256, kv_dtype="bf16")], [prompt])[0]
    v.ensure_capacity(_t([128]), 1)
    am = _t(np.zeros(128))
    lg = torch.zeros(128, synth.TINY.vocab, dtype=torch.float32, device="cuda")
    v.spec_forward(_t(prompt), _t([0, 128]), 1, 128, 128, am, lg)
    torch.cuda.synchronize()
    assert v.get_status() == 0
    flips, d = check_rows(lg.cpu().numpy(), am.cpu().numpy(), ref, "prefill")
    print(f"prefill: max |dlogit| {d:.3e}, near-tie flips {flips}")


def test_tiny_spec_loop_teacher_forced(tiny):
    import torch
    host, dev, model = tiny
    prompt = workloads.motif_prompt(1)
    streams, recs, pool = oracle.generate(model, [prompt], 32, drafter="ngram", k=4, keep_logits=True,
                                          kv_dtype="bf16")
    v = _verifier(dev)
    # prefill in one chunk, as the oracle does (prefill_chunk 128)
    v.ensure_capacity(_t([128]), 1)
    am = _t(np.zeros(128))
    v.spec_forward(_t(prompt), _t([0, 128]), 1, 128, 128, am)
    out = {k: _t(np.zeros(8)) for k in ("n_accept", "n_commit", "new_len")}
    committed = _t(np.zeros(8 * 5))
    table = _t(np.zeros(1 * 32))
    npages = _t(np.zeros(1))
    ftop = _t(np.zeros(1))
    all_flips = []
    for step, r in enumerate(recs):
        span = r.spans[0]
        S = len(span)
        v.ensure_capacity(_t([r.len_before[0] + S]), 1)
        lg = torch.zeros(S, synth.TINY.vocab, dtype=torch.float32, device="cuda")
        amS = _t(np.zeros(S))
        tok, ro = _t(span), _t([0, S])
        v.spec_forward(tok, ro, 1, S, S, amS, lg)
        v.accept_greedy(tok, ro, amS, 1, 5, out["n_accept"], committed, out["n_commit"], out["new_len"])
        torch.cuda.synchronize()
        assert v.get_status() == 0, f"step {step}"
        g_am = amS.cpu().numpy()
        flips, _ = check_rows(lg.cpu().numpy(), g_am, r.logits[0], f"step {step}")
        all_flips += [(step, f) for f in flips]
        if not flips:
            assert out["n_accept"][0].item() == r.m[0]
            assert out["new_len"][0].item() == r.new_len[0]
            assert committed[:r.m[0] + 1].cpu().tolist() == r.committed[0]
        # teacher forcing: follow the oracle's acceptance
        v.rewind_cache(_t([r.new_len[0]]), 1)
        v.page_table(table, npages, ftop)
        torch.cuda.synchronize()
        n = npages[0].item()
        assert table[:n].cpu().tolist() == r.page_table[0]
    print("near-tie flips:", all_flips)

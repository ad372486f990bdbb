"""Sampled (temperature) verify on the GPU against the oracle's sampler.

[TS] the protocol, Verify: the caller's sampler draws each row and drafts are
accepted while the drawn token matches. The LM-head kernel draws each row by the
Gumbel-max construction from its own SplitMix64 streams; the oracle implements
the same definition independently (oracle/sampling.py). A drawn token is an
argmax over perturbed scores logit / T + g, so, as for greedy rows, the two
sides must agree wherever the oracle's top-2 margin of those scores exceeds the
logit tolerance scaled by 1 / T (MARGIN / T); closer rows are near-ties,
reported, not failed.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import workloads
from tests.helpers import LOGIT_TOL, MARGIN, margins, upload_weights

pytestmark = pytest.mark.gpu


def _t(a):
    import torch
    return torch.as_tensor(np.asarray(a, dtype=np.int32)).cuda()


def _f(a):
    import torch
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).cuda()


@pytest.fixture(scope="module")
def tiny():
    import torch
    torch.cuda.init()
    host, dev = upload_weights(synth.TINY, 1)
    return host, dev, oracle.DenseDecoder(synth.TINY, lambda n: host[n])


def _verifier(dev, shape=synth.TINY, **kw):
    from speculative_decoding_verify_02_gb300 import Verifier
    cfg = dict(page_size=16, n_pages=256, max_batch=2, max_rows=128, max_span=128, max_context=1024,
               ngram_capacity=2048)
    cfg.update(kw)
    return Verifier(shape, dev, **cfg)


def _check_draws(gpu_drawn, gpu_logits, ref_logits, T, seed, b, positions, what):
    """Logits within tolerance; drawn tokens equal to the oracle's draws wherever the perturbed
    top-2 margin exceeds MARGIN / T. Returns the near-tie rows."""
    d = np.abs(gpu_logits.astype(np.float64) - ref_logits).max()
    assert d <= LOGIT_TOL, f"{what}: max |dlogit| {d:.4g}"
    score = oracle.perturbed(ref_logits, T, seed, b, positions)
    ref = score.argmax(-1)
    mg = margins(score)
    near = []
    for i in range(len(ref)):
        if gpu_drawn[i] != ref[i]:
            assert mg[i] <= MARGIN / T, f"{what}: row {i} drew {gpu_drawn[i]} != {ref[i]} at margin {mg[i]:.4f}"
            near.append((i, float(mg[i])))
    return near


def test_sampled_rows_match_oracle_teacher_forced(tiny):
    """The tiny decoder's sampled loop (T = 0.5, 2-gram drafts, K = 4) in the oracle drives the
    GPU step by step: every row's logits and drawn token, acceptance, committed tokens and new
    lengths, teacher-forced."""
    import torch
    host, dev, om = tiny
    T, seed = 0.5, 77
    prompt = workloads.motif_prompt(1)
    streams, recs, _ = oracle.generate(om, [prompt], 24, drafter="ngram", k=4, keep_logits=True, kv_dtype="bf16",
                                       temperature=T, seed=seed)
    v = _verifier(dev, max_batch=1)
    temp = _f([T])
    v.ensure_capacity(_t([128]), 1)
    drawn = _t(np.zeros(128))
    lg = torch.zeros(128, synth.TINY.vocab, dtype=torch.float32, device="cuda")
    v.spec_forward_sampled(_t(prompt), _t([0, 128]), 1, 128, 128, temp, seed, drawn, lg)
    torch.cuda.synchronize()
    ref_pre = om.forward([oracle.SeqCache(synth.TINY, 256, kv_dtype="bf16")], [prompt])[0]
    near = _check_draws(drawn.cpu().numpy(), lg.cpu().numpy(), ref_pre, T, seed, 0, range(128), "prefill")
    n_acc, com, n_com, new_len = _t([0]), _t(np.zeros(8)), _t([0]), _t([0])
    checked = 0
    for step, r in enumerate(recs):
        span = r.spans[0]
        S = len(span)
        v.ensure_capacity(_t([r.len_before[0] + S]), 1)
        lgS = torch.zeros(S, synth.TINY.vocab, dtype=torch.float32, device="cuda")
        dS = _t(np.zeros(S))
        tok, ro = _t(span), _t([0, S])
        v.spec_forward_sampled(tok, ro, 1, S, S, temp, seed, dS, lgS)
        v.accept_greedy(tok, ro, dS, 1, 8, n_acc, com, n_com, new_len)
        torch.cuda.synchronize()
        assert v.get_status() == 0
        pos = range(r.len_before[0], r.len_before[0] + S)
        flips = _check_draws(dS.cpu().numpy(), lgS.cpu().numpy(), r.logits[0], T, seed, 0, pos, f"step {step}")
        near += flips
        if not flips:
            checked += 1
            np.testing.assert_array_equal(dS.cpu().numpy(), r.argmax[0])
            assert n_acc[0].item() == r.m[0] and new_len[0].item() == r.new_len[0]
            assert com[:r.m[0] + 1].cpu().tolist() == r.committed[0]
        v.rewind_cache(_t([r.new_len[0]]), 1)
    assert checked >= len(recs) - 2
    print(f"sampled tiny: {checked}/{len(recs)} steps exact, near ties {near}")


def test_temperature_zero_is_the_greedy_forward(tiny):
    """Per-sequence temperatures: a sequence at T = 0 draws exactly the argmax of the greedy
    forward, bit for bit, next to a sampled sequence in the same launch."""
    import torch
    host, dev, om = tiny
    v = _verifier(dev)
    toks = [int(t) for t in synth.tokens(1, "t0.span", 20, synth.TINY.vocab)]
    v.ensure_capacity(_t([10, 10]), 2)
    am = _t(np.zeros(20))
    lg = torch.zeros(20, synth.TINY.vocab, dtype=torch.float32, device="cuda")
    v.spec_forward(_t(toks), _t([0, 10, 20]), 2, 20, 10, am, lg)
    v.rewind_cache(_t([0, 0]), 2)
    v.ensure_capacity(_t([10, 10]), 2)
    dr = _t(np.zeros(20))
    lg2 = torch.zeros(20, synth.TINY.vocab, dtype=torch.float32, device="cuda")
    v.spec_forward_sampled(_t(toks), _t([0, 10, 20]), 2, 20, 10, _f([0.0, 0.8]), 5, dr, lg2)
    torch.cuda.synchronize()
    assert v.get_status() == 0
    assert (lg.cpu().numpy() == lg2.cpu().numpy()).all()          # sampling leaves the logits alone
    np.testing.assert_array_equal(dr[:10].cpu().numpy(), am[:10].cpu().numpy())
    near = _check_draws(dr[10:].cpu().numpy(), lg2[10:].cpu().numpy(), lg2[10:].cpu().numpy().astype(np.float64),
                        0.8, 5, 1, range(10), "T=0.8")
    assert not near


def _sampled_loop(v, prompt, budget, k, drafter, T, seed, graph):
    import torch
    from speculative_decoding_verify_02_gb300.runner import SpecLoop
    loop = SpecLoop(v, 1, 8)
    temp = _f([T])
    first = loop.prefill([prompt], ngram=(drafter == 1), temperature=temp, seed=seed)
    loop.start([budget], k_init=max(k, 1) if drafter else 0, adaptive=False)
    stream = [int(first[0])]
    kw = dict(drafter=drafter, ngram=(drafter == 1), temperature=temp, seed=seed)
    if graph:
        loop.capture(**kw)
    steps = accepted = 0
    for _ in range(budget + 2):
        loop.replay() if graph else loop.step(**kw)
        torch.cuda.synchronize()
        n = int(loop.n_commit[0].item())
        stream += loop.committed[:n].cpu().tolist()
        accepted += max(0, int(loop.n_accept[0].item()))
        steps += 1
        if len(stream) >= budget:
            break
    assert v.get_status() == 0
    return stream, accepted


@pytest.mark.parametrize("T", [0.05, 0.1])
def test_sampled_spec_on_equals_spec_off_on_gpu(tiny, T):
    """Lossless sampled speculation on the device: the 2-gram loop (K = 4, eager and captured as a
    CUDA graph) emits the plain sampled loop's stream token for token at a fixed seed, with drafts
    accepted along the way, and the stream is not the greedy one."""
    host, dev, om = tiny
    prompt = workloads.motif_prompt(1)
    off, _ = _sampled_loop(_verifier(dev, max_batch=1), prompt, 40, 0, 0, T, 21, False)
    on, acc = _sampled_loop(_verifier(dev, max_batch=1), prompt, 40, 4, 1, T, 21, False)
    ong, _ = _sampled_loop(_verifier(dev, max_batch=1), prompt, 40, 4, 1, T, 21, True)
    assert on[:40] == off[:40] and ong[:40] == off[:40]
    assert acc > 0
    greedy, _ = _sampled_loop(_verifier(dev, max_batch=1), prompt, 40, 0, 0, 0.0, 21, False)
    assert greedy[:40] != off[:40]


def test_sampled_verify_4b_shape(tiny):
    """The 4B shape (2 layers): one sampled verify of 8 rows at an 848-token context, T = 0.8,
    against the oracle's draws on the same context."""
    import torch
    from speculative_decoding_verify_02_gb300 import Verifier
    from speculative_decoding_verify_02_gb300.runner import SpecLoop
    from tests.helpers import oracle_cache_from_pool
    shape = synth.QWEN3_4B.with_layers(2)
    host, dev = upload_weights(shape, 2)
    om = oracle.DenseDecoder(shape, lambda n: host[n])
    v = Verifier(shape, dev, page_size=16, n_pages=128, max_batch=1, max_rows=128, max_span=128, max_context=1024)
    ctx = workloads.uniform_context(2, 848, shape.vocab, name="sampled.ctx")
    SpecLoop(v, 1, 8).prefill([ctx])
    cache = oracle_cache_from_pool(v, shape, 0, 848, 900)
    span = [int(t) for t in synth.tokens(2, "sampled.span", 8, shape.vocab)]
    T, seed = 0.8, 2024
    v.ensure_capacity(_t([856]), 1)
    dr = _t(np.zeros(8))
    lg = torch.zeros(8, shape.vocab, dtype=torch.float32, device="cuda")
    v.spec_forward_sampled(_t(span), _t([0, 8]), 1, 8, 8, _f([T]), seed, dr, lg)
    torch.cuda.synchronize()
    assert v.get_status() == 0
    ref = om.forward([cache], [span])[0]
    near = _check_draws(dr.cpu().numpy(), lg.cpu().numpy(), ref, T, seed, 0, range(848, 856), "4B sampled")
    greedy = ref.argmax(-1)
    print(f"4B sampled verify: near ties {near}; rows differing from greedy "
          f"{int((dr.cpu().numpy() != greedy).sum())}/8")
    v.close()

"""Device-side transaction pieces on the GPU: the n-gram index and proposer,
adaptive K, the whole loop captured as a CUDA graph with ragged and
truncated spans, spec-on against spec-off, and the error paths.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import workloads
from tests.helpers import MARGIN, margins, upload_weights

pytestmark = pytest.mark.gpu


def _t(a):
    import torch
    return torch.as_tensor(np.asarray(a, dtype=np.int32)).cuda()


@pytest.fixture(scope="module")
def tiny():
    import torch
    torch.cuda.init()
    host, dev = upload_weights(synth.TINY, 1)
    return host, dev, oracle.DenseDecoder(synth.TINY, lambda n: host[n])


def _verifier(dev, shape=synth.TINY, **kw):
    from speculative_decoding_verify_02_gb300 import Verifier
    cfg = dict(page_size=16, n_pages=256, max_batch=4, max_rows=128, max_span=128, max_context=1024,
               ngram_capacity=2048)
    cfg.update(kw)
    return Verifier(shape, dev, **cfg)


def test_ngram_proposer_matches_oracle(tiny):
    """[TS] n-gram lookup: the device hash index + proposer against the oracle's
    backward scan, on repeat-heavy histories, at every prefix length."""
    import torch
    from speculative_decoding_verify_02_gb300 import SDV_DRAFT_NGRAM
    _, dev, _ = tiny
    B, V = 4, 12                                               # a small alphabet: many matches
    hists = [list(map(int, workloads.span_repeat_prompt(40 + b, n_spans=12, span=8, vocab=V))) for b in range(B)]
    v = _verifier(dev, max_batch=B)
    max_span = 8
    toks, ro, req = _t(np.zeros(B * max_span)), _t(np.zeros(B + 1)), _t(np.zeros(B))
    stride = 1
    for n in range(3, len(hists[0]) + 1):
        if n == 3:                                              # first commit: three tokens each
            buf = np.array([h[:3] for h in hists], dtype=np.int32).reshape(-1)
            v.ngram_commit(_t(buf), _t([3] * B), B, 3)
        else:
            v.ngram_commit(_t([h[n - 1] for h in hists]), _t([1] * B), B, stride)
        k = 1 + n % 7
        v.gen_init(_t([h[n - 1] for h in hists]), _t([10_000] * B), B, k, False, 7)
        v.propose(SDV_DRAFT_NGRAM, None, 0, B, max_span, toks, ro, req)
        torch.cuda.synchronize()
        t, o = toks.cpu().numpy(), ro.cpu().numpy()
        for b in range(B):
            d = oracle.ngram_propose(hists[b][:n], k)
            span = t[o[b]:o[b + 1]].tolist()
            assert span == [hists[b][n - 1]] + d, (n, b, span, d)
    assert v.get_status() == 0


@pytest.mark.parametrize("n_max,n_min,pmin", [(6, 2, 0.0), (6, 2, 0.5), (4, 1, 0.0), (3, 3, 0.0), (5, 2, 1.0)])
def test_multi_order_ngram_proposer_matches_oracle(tiny, n_max, n_min, pmin):
    """[TS] one index per n-gram order and --spec-pmin scaling the required match length; [CA]
    --ngram-min: the device's longest-match lookup against the oracle's backward scan, at every
    prefix of repeat-heavy histories over a small alphabet."""
    import torch
    from speculative_decoding_verify_02_gb300 import SDV_DRAFT_NGRAM
    _, dev, _ = tiny
    B, V = 4, 6
    hists = [list(map(int, workloads.span_repeat_prompt(60 + b, n_spans=14, span=6, vocab=V))) for b in range(B)]
    v = _verifier(dev, max_batch=B, ngram_max_order=n_max)
    v.ngram_params(n_min, pmin)
    max_span = 8
    toks, ro, req = _t(np.zeros(B * max_span)), _t(np.zeros(B + 1)), _t(np.zeros(B))
    hit = 0
    for n in range(1, len(hists[0]) + 1):
        v.ngram_commit(_t([h[n - 1] for h in hists]), _t([1] * B), B, 1)
        k = 1 + n % 7
        v.gen_init(_t([h[n - 1] for h in hists]), _t([10_000] * B), B, k, False, 7)
        v.propose(SDV_DRAFT_NGRAM, None, 0, B, max_span, toks, ro, req)
        torch.cuda.synchronize()
        t, o = toks.cpu().numpy(), ro.cpu().numpy()
        for b in range(B):
            d = oracle.ngram_propose_multi(hists[b][:n], k, n_min, n_max, pmin)
            hit += bool(d)
            assert t[o[b]:o[b + 1]].tolist() == [hists[b][n - 1]] + d, (n, b)
    assert v.get_status() == 0
    assert hit > 0
    v.close()


def test_adaptive_k_trajectory(tiny):
    """[CA] adaptive K inside accept_greedy, read back through the proposer's
    span lengths (table drafter), against the oracle's rule on scripted rounds."""
    import torch
    from speculative_decoding_verify_02_gb300 import SDV_DRAFT_TABLE
    _, dev, _ = tiny
    B, max_span = 1, 8
    v = _verifier(dev, max_batch=B)
    table = _t(np.arange(1000) % synth.TINY.vocab)
    v.gen_init(_t([5]), _t([10_000]), B, 1, True, 7)
    toks, ro, req = _t(np.zeros(max_span)), _t([0, 0]), _t([0])
    n_acc, com, n_com, nl = _t([0]), _t(np.zeros(max_span)), _t([0]), _t([0])
    K = 1
    rng = np.random.default_rng(0)
    for step in range(40):
        v.propose(SDV_DRAFT_TABLE, table, 1000, B, max_span, toks, ro, req)
        torch.cuda.synchronize()
        S = int(ro[1].item())
        assert S - 1 == K, (step, S, K)
        span = toks[:S].cpu().numpy()
        m = int(rng.integers(0, S))                            # accept m drafts
        am = np.array([span[i + 1] if i < m else (span[i + 1] + 1) % 100 if i + 1 < S else 3 for i in range(S)])
        v.ensure_capacity(_t([1 + step * 8 + S]), B)
        v.accept_greedy(toks, ro, _t(am), B, max_span, n_acc, com, n_com, nl)
        torch.cuda.synchronize()
        assert int(n_acc[0].item()) == m
        K = oracle.adapt_k(K, S - 1, m, 7)
    assert v.get_status() == 0


def _run_loop(v, B, prompts, budget, k, drafter, table=None, graph=False, max_span=8):
    """The device loop until every sequence meets its budget; returns the streams."""
    import torch
    from speculative_decoding_verify_02_gb300.runner import SpecLoop
    loop = SpecLoop(v, B, max_span)
    first = loop.prefill(prompts, ngram=(drafter == 1))
    loop.start(budget, k_init=max(k, 1) if drafter else 0, adaptive=False)
    streams = [[int(f)] for f in first]
    kw = dict(drafter=drafter, table=table, table_stride=(table.numel() // B if table is not None else 0),
              ngram=(drafter == 1))
    if graph:
        loop.capture(**kw)
    for _ in range(max(budget) + 2):
        loop.replay() if graph else loop.step(**kw)
        torch.cuda.synchronize()
        nc, cm = loop.n_commit.cpu().numpy(), loop.committed.cpu().numpy().reshape(B, max_span)
        for b in range(B):
            streams[b] += cm[b, :nc[b]].tolist()
        if all(len(s) >= bb for s, bb in zip(streams, budget)):
            break
    assert v.get_status() == 0
    return streams


def test_graph_replay_ragged_and_truncated_spans_match_eager(tiny):
    """[PI] capture-shape gotcha: one captured step replays correctly while spans
    are ragged and get truncated near the output budget (lengths live in device
    memory, so capture shape and replay shape never disagree). The captured
    loop, the eager loop and the oracle's loop give the same streams."""
    _, dev, om = tiny
    B = 3
    prompts = [workloads.motif_prompt(1), synth.tokens(8, "cap.p2", 41, synth.TINY.vocab),
               synth.tokens(8, "cap.p3", 17, synth.TINY.vocab)]
    budget = [5, 23, 14]
    ref, _, _ = oracle.generate(om, prompts, max(budget), drafter="none", kv_dtype="bf16")
    tables = np.stack([np.array((ref[b] + [0] * 64)[:64]) for b in range(B)])
    tables[:, 1::3] = 7                                         # corrupt a third: partial acceptance
    import torch
    table = torch.as_tensor(tables.astype(np.int32).reshape(-1)).cuda()
    eager = _run_loop(_verifier(dev, max_batch=B), B, prompts, budget, 6, 2, table)
    graph = _run_loop(_verifier(dev, max_batch=B), B, prompts, budget, 6, 2, table, graph=True)
    assert eager == graph
    plain = _run_loop(_verifier(dev, max_batch=B), B, prompts, budget, 0, 0)
    assert eager == plain                                       # spec-on equals spec-off on the device
    for b in range(B):
        assert len(eager[b]) == budget[b]
        # against the oracle: equal up to the first near-tie flip
        for i, (g, o) in enumerate(zip(eager[b], ref[b][:budget[b]])):
            if g != o:
                cache = oracle.SeqCache(synth.TINY, 256, kv_dtype="bf16")
                lg = om.forward([cache], [list(prompts[b]) + ref[b][:i]])[0][-1]
                assert margins(lg[None])[0] <= MARGIN, (b, i)
                break


def test_ngram_loop_spec_on_equals_spec_off(tiny):
    """The tiny-model loop on the device (2-gram lookup, K=4, 32 tokens) gives the same
    stream as the device's plain loop, and commits 1..K+1 tokens per step."""
    _, dev, om = tiny
    prompt = workloads.motif_prompt(1)
    on = _run_loop(_verifier(dev, max_batch=1), 1, [prompt], [32], 4, 1)
    off = _run_loop(_verifier(dev, max_batch=1), 1, [prompt], [32], 0, 0)
    assert on == off and len(on[0]) == 32


def test_governed_loop_is_lossless(tiny):
    """[TS] the cost governor parks and re-probes drafting by measured step time; whatever it
    decides, every emitted token is drawn from a trunk row, so the governed n-gram loop emits the
    plain loop's stream. The governor sees real step times and samples."""
    import speculative_decoding_verify_02_gb300 as sdv
    from speculative_decoding_verify_02_gb300.runner import SpecLoop
    _, dev, _ = tiny
    prompts = [workloads.motif_prompt(1), synth.tokens(8, "gov.p2", 57, synth.TINY.vocab)]
    B, budget = 2, [40, 40]
    plain = _run_loop(_verifier(dev, max_batch=B), B, prompts, budget, 0, 0)
    v = _verifier(dev, max_batch=B)
    loop = SpecLoop(v, B, 8)
    first = loop.prefill(prompts, ngram=True)
    loop.start(budget, k_init=1, adaptive=True, k_max=7)
    gov = sdv.Governor(sdv.GovernorCfg(4, 2, 4, 16, 4, 8, 2, 3, 16))      # short intervals: every state
    streams = [[int(f)] for f in first]
    decisions = []
    for _ in range(200):
        spec, committed, ms = loop.governed_step(gov, drafter=sdv.SDV_DRAFT_NGRAM, ngram=True)
        nc, cm = loop.n_commit.cpu().numpy(), loop.committed.cpu().numpy().reshape(B, 8)
        for b in range(B):
            streams[b] += cm[b, :nc[b]].tolist()
        decisions.append(spec)
        if all(len(s) >= bb for s, bb in zip(streams, budget)):
            break
    assert v.get_status() == 0
    assert streams == plain
    st = gov.stats()
    assert st["plain_ms_per_tok"] and st["spec_ms_per_tok"] and st["wins"] + st["losses"] >= 1
    assert any(decisions) and not all(decisions)
    print("governor:", st)
    gov.close()
    v.close()


def test_error_paths_report_and_leave_state(tiny):
    """Failures are reported through the status word and leave the state as it was:
    the pool running dry, a request past the page table, a rewind past the written
    length, a forward without capacity, a token id past the vocabulary, a span
    longer than declared; host-side argument errors raise at once."""
    import torch
    import speculative_decoding_verify_02_gb300 as sdv
    _, dev, _ = tiny
    v = _verifier(dev, n_pages=6, max_batch=2, max_context=64)   # 6 pages; 4 per sequence at most
    tab, npg, top = _t(np.zeros(2 * 4)), _t([0, 0]), _t([0])

    def state():
        v.page_table(tab, npg, top)
        torch.cuda.synchronize()
        return tab.cpu().tolist(), npg.cpu().tolist(), top.cpu().tolist()

    v.ensure_capacity(_t([48, 16]), 2)
    assert v.get_status() == 0
    s0 = state()
    v.ensure_capacity(_t([64, 64]), 2)                         # needs 4 more pages, 2 free
    assert v.get_status() == sdv.SDV_ERR_CAPACITY and state() == s0
    v.ensure_capacity(_t([65, -1]), 2)                         # past the page table
    assert v.get_status() == sdv.SDV_ERR_CAPACITY and state() == s0
    v.rewind_cache(_t([1, -1]), 2)                             # nothing written yet
    assert v.get_status() == sdv.SDV_ERR_ARG and state() == s0
    am = _t(np.zeros(17))
    v.spec_forward(_t([1] * 17), _t([0, 17, 17]), 2, 17, 17, am)   # 17 rows into sequence 0's 48 slots
    assert v.get_status() == 0
    lens = _t([0, 0])
    v.cache_seq_len(lens)
    torch.cuda.synchronize()
    assert lens.cpu().tolist() == [17, 0]
    v.spec_forward(_t([1] * 17), _t([0, 0, 17]), 2, 17, 17, am)    # sequence 1 holds 16 slots only
    assert v.get_status() == sdv.SDV_ERR_CAPACITY
    v.spec_forward(_t([synth.TINY.vocab]), _t([0, 1, 1]), 2, 1, 1, am)   # token id past the vocabulary
    assert v.get_status() == sdv.SDV_ERR_DEVICE
    v.spec_forward(_t([1] * 5), _t([0, 5, 5]), 2, 5, 4, am)        # span of 5 declared as at most 4
    assert v.get_status() == sdv.SDV_ERR_ARG
    with pytest.raises(sdv.SdvError):
        v.spec_forward(_t([1]), _t([0, 1, 1, 1]), 3, 1, 1, am)     # B past max_batch
    with pytest.raises(sdv.SdvError):
        v.spec_forward(_t([1]), _t([0, 1, 1]), 2, 200, 1, am)      # max_rows past the context's
    assert v.get_status() == 0

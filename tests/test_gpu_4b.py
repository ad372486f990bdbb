"""The Qwen3-4B-shaped verify path on the GPU against the float64 oracle.

Two decoder layers of the 4B shape (hidden 2560, 32/8 heads of 128, FFN 9728,
vocab 151936) exercise every GEMM and attention tile shape of the 36-layer
model at a fraction of the oracle's cost; the full model is covered in
test_gpu_full.py. Parity rules are those of tests/helpers.py.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import workloads
from tests.helpers import MARGIN, check_rows, margins, oracle_cache_from_pool, upload_weights

pytestmark = pytest.mark.gpu

SHAPE = synth.QWEN3_4B.with_layers(2)
SEED = 2


@pytest.fixture(scope="module")
def model():
    import torch
    torch.cuda.init()
    host, dev = upload_weights(SHAPE, SEED)
    return host, dev, oracle.DenseDecoder(SHAPE, lambda n: host[n])


def _t(a):
    import torch
    return torch.as_tensor(np.asarray(a, dtype=np.int32)).cuda()


def _verifier(dev, **kw):
    from speculative_decoding_verify_02_gb300 import Verifier
    cfg = dict(page_size=16, n_pages=512, max_batch=1, max_rows=128, max_span=128, max_context=2048)
    cfg.update(kw)
    return Verifier(SHAPE, dev, **cfg)


def _forward(v, tokens, row_off, B, max_span, logits=True):
    import torch
    R = len(tokens)
    am = _t(np.zeros(max(R, max_span)))
    lg = torch.zeros(max(R, max_span), SHAPE.vocab, dtype=torch.float32, device="cuda") if logits else None
    v.spec_forward(_t(tokens), _t(row_off), B, max(R, max_span), max_span, am, lg)
    torch.cuda.synchronize()
    return (lg[:R].cpu().numpy() if logits else None), am[:R].cpu().numpy()


def test_verify_step_parity_848_context(model):
    """4B shape, batch 1, 848-token context: prefill, then an S=8 verify with uniform drafts."""
    import torch
    from speculative_decoding_verify_02_gb300.runner import SpecLoop
    host, dev, om = model
    ctx = workloads.uniform_context(SEED, 848, SHAPE.vocab)
    cache = oracle.SeqCache(SHAPE, 900, kv_dtype="bf16")
    ref_pre = om.forward([cache], [ctx], last_row_logits=True)[0]
    v = _verifier(dev)
    loop = SpecLoop(v, 1, 17)
    first = int(loop.prefill([ctx], chunk=128)[0])
    if margins(ref_pre)[0] > MARGIN:
        assert first == int(ref_pre.argmax())
    first = int(ref_pre.argmax())                              # teacher-forced from here
    span = [first] + [int(t) for t in workloads.uniform_drafts(SEED, 0, 7, SHAPE.vocab)]
    ref = om.forward([cache], [span])[0]
    v.ensure_capacity(_t([848 + 8]), 1)
    lg, am = _forward(v, span, [0, 8], 1, 8)
    assert v.get_status() == 0
    flips, d = check_rows(lg, am, ref, "verify S=8")
    print(f"4B-L2 verify: max |dlogit| {d:.3e}, near-tie flips {flips}")
    # the paged K/V the GEMM epilogue wrote, at sampled positions, against the oracle's cache
    tab = _t(np.zeros(v.pages_per_seq))
    npg, top = _t([0]), _t([0])
    v.page_table(tab, npg, top)
    torch.cuda.synchronize()
    tab = tab.cpu().numpy()
    P, nkv, D = 16, SHAPE.n_kv_heads, SHAPE.head_dim
    pool = v.pool.view(torch.bfloat16).view(SHAPE.n_layers, v.ccfg.n_pages, 2, nkv, P, D)
    for l in range(SHAPE.n_layers):
        for pos in (0, 1, 15, 16, 500, 847, 848, 855):
            k = pool[l, tab[pos // P], 0, :, pos % P].float().cpu().numpy()
            val = pool[l, tab[pos // P], 1, :, pos % P].float().cpu().numpy()
            np.testing.assert_allclose(k, cache.K[l][pos], atol=3e-2, rtol=2e-2)
            np.testing.assert_allclose(val, cache.V[l][pos], atol=3e-2, rtol=2e-2)


def test_rows_gate_and_width_invariance(model):
    """[CA] rows gate on the GPU: q one-row forwards equal one q-row forward, and
    the same rows inside a wider span (a wider MMA) are unchanged, bit for bit."""
    host, dev, om = model
    ctx = workloads.uniform_context(SEED, 300, SHAPE.vocab, name="gate.ctx")
    toks = [int(t) for t in synth.tokens(SEED, "gate.span", 17, SHAPE.vocab)]
    from speculative_decoding_verify_02_gb300.runner import SpecLoop
    v = _verifier(dev)
    SpecLoop(v, 1, 17).prefill([ctx])
    v.ensure_capacity(_t([300 + 17]), 1)
    one, am_one = _forward(v, toks[:8], [0, 8], 1, 8)
    v.rewind_cache(_t([300]), 1)
    v.ensure_capacity(_t([300 + 17]), 1)                   # the rewind released the span's pages
    seq = []
    for i in range(8):
        lg, _ = _forward(v, toks[i:i + 1], [0, 1], 1, 1)
        seq.append(lg[0])
    seq = np.stack(seq)
    v.rewind_cache(_t([300]), 1)
    v.ensure_capacity(_t([300 + 17]), 1)
    wide, _ = _forward(v, toks, [0, 17], 1, 17)              # 17 rows: MMA width 32 instead of 16
    assert v.get_status() == 0
    assert np.abs(one - seq).max() == 0.0, np.abs(one - seq).max()
    assert np.abs(one - wide[:8]).max() == 0.0, np.abs(one - wide[:8]).max()
    np.testing.assert_array_equal(am_one, one.argmax(-1))


def test_batch16_ragged_teacher_forced(model):
    """Batch of 16 sequences with ragged contexts and corrupted-greedy drafts
    (mixed acceptance): per-row logits, acceptance, committed tokens, new
    lengths and page tables against the oracle, step by step."""
    import torch
    host, dev, om = model
    B, N, K = 16, 12, 7
    lens = synth.ints(3, "b16.len", B, 20, 100)
    prompts = [workloads.uniform_context(3, int(n), SHAPE.vocab, name=f"b16.ctx.{b}") for b, n in enumerate(lens)]
    plain, _, _ = oracle.generate(om, prompts, N, drafter="none", prefill_chunk=128, kv_dtype="bf16")
    tables = [workloads.corrupt(3, b, np.array(plain[b] + [0] * 16), 0.3, SHAPE.vocab) for b in range(B)]
    streams, recs, pool = oracle.generate(om, prompts, N, drafter="table", k=K, tables=tables,
                                          prefill_chunk=128, keep_logits=True, n_pages=B * 16, max_pages_per_seq=16,
                                          kv_dtype="bf16")
    v = _verifier(dev, n_pages=B * 16, max_batch=B, max_context=256)
    from speculative_decoding_verify_02_gb300.runner import SpecLoop
    SpecLoop(v, B, 8).prefill(prompts, chunk=128)
    n_acc, com, n_com, new_len = _t(np.zeros(B)), _t(np.zeros(B * 8)), _t(np.zeros(B)), _t(np.zeros(B))
    tab, npg, top = _t(np.zeros(B * v.pages_per_seq)), _t(np.zeros(B)), _t([0])
    flips_all, checked = [], 0
    for step, r in enumerate(recs):
        spans = r.spans
        offs = np.concatenate([[0], np.cumsum([len(s) for s in spans])]).astype(np.int32)
        flat = [t for s in spans for t in s]
        v.ensure_capacity(_t([r.len_before[b] + len(spans[b]) if spans[b] else -1 for b in range(B)]), B)
        tok_t, off_t = _t(flat), _t(offs)
        lg, am = _forward(v, flat, offs, B, 8)
        v.accept_greedy(tok_t, off_t, _t(am), B, 8, n_acc, com, n_com, new_len)
        torch.cuda.synchronize()
        assert v.get_status() == 0
        g_m, g_new = n_acc.cpu().numpy(), new_len.cpu().numpy()
        for b in range(B):
            if not spans[b]:
                assert g_m[b] == -1
                continue
            flips, _ = check_rows(lg[offs[b]:offs[b + 1]], am[offs[b]:offs[b + 1]], r.logits[b], f"s{step} b{b}")
            flips_all += [(step, b, f) for f in flips]
            if not flips:
                checked += 1
                assert g_m[b] == r.m[b] and g_new[b] == r.new_len[b], (step, b)
                assert com[b * 8:b * 8 + r.m[b] + 1].cpu().tolist() == r.committed[b]
        v.rewind_cache(_t([nl for nl in r.new_len]), B)      # teacher forcing: the oracle's lengths
        v.page_table(tab, npg, top)
        torch.cuda.synchronize()
        t, n = tab.cpu().numpy().reshape(B, -1), npg.cpu().numpy()
        for b in range(B):
            assert t[b, :n[b]].tolist() == r.page_table[b], (step, b)
    ms = [r.m[b] for r in recs for b in range(B) if r.m[b] >= 0]
    assert len(set(ms)) >= 3, ms                               # mixed acceptance lengths were exercised
    print(f"batch16: {checked} sequence-steps compared exactly, near-tie flips {flips_all}, m histogram "
          f"{np.bincount(ms).tolist()}")


def test_verify_every_span_length_1_to_17(model):
    """[CA] verify cost against S: the config-2 sweep S = 1..17 at an 848-token context. Every
    span is checked against the oracle's verify over the same (GPU-written) context, and its rows
    must equal the first rows of the 17-row span bit for bit (one-row to 17-row forwards, GEMM
    widths 16 and 32, one to three attention launches)."""
    host, dev, om = model
    ctx = workloads.uniform_context(SEED, 848, SHAPE.vocab, name="sweep.ctx")
    toks = [int(t) for t in synth.tokens(SEED, "sweep.span", 17, SHAPE.vocab)]
    from speculative_decoding_verify_02_gb300.runner import SpecLoop
    v = _verifier(dev)
    SpecLoop(v, 1, 17).prefill([ctx])
    base = oracle_cache_from_pool(v, SHAPE, 0, 848, 900)
    wide, worst, flips_all = None, 0.0, []
    for S in [17] + list(range(1, 17)):
        v.ensure_capacity(_t([848 + 17]), 1)
        lg, am = _forward(v, toks[:S], [0, S], 1, S)
        v.rewind_cache(_t([848]), 1)
        assert v.get_status() == 0
        cache = oracle.SeqCache(SHAPE, 900, kv_dtype="bf16")
        for l in range(SHAPE.n_layers):
            cache.K[l][:848], cache.V[l][:848] = base.K[l][:848], base.V[l][:848]
        cache.length = 848
        ref = om.forward([cache], [toks[:S]])[0]
        flips, d = check_rows(lg, am, ref, f"sweep S={S}")
        worst = max(worst, d)
        flips_all += [(S, f) for f in flips]
        if wide is None:
            wide = lg
        else:
            assert np.abs(lg - wide[:S]).max() == 0.0, (S, np.abs(lg - wide[:S]).max())
    print(f"sweep S=1..17: max |dlogit| {worst:.3e}, near-tie flips {flips_all}")


def test_rows_independent_of_batch_width(model):
    """Batch invariance across GEMM widths: the same verify rows computed for 16 sequences at once
    (128 rows: MMA width N = 128, whose stages take 32-wide k-blocks), for the first 6 (48 rows:
    N = 64), for the first 3 (24 rows: N = 32) and for each sequence alone (8 rows: N = 16) are
    bit-identical; the first six sequences also match the oracle's verify."""
    import torch
    from speculative_decoding_verify_02_gb300.runner import SpecLoop
    host, dev, om = model
    B, S = 16, 8
    lens = [int(n) for n in synth.ints(SEED, "width.len", B, 200, 700)]
    prompts = [workloads.uniform_context(SEED, L, SHAPE.vocab, name=f"width.ctx.{b}") for b, L in enumerate(lens)]
    v = _verifier(dev, max_batch=B, n_pages=sum(-(-(L + S) // 16) for L in lens) + 8)
    SpecLoop(v, B, S).prefill(prompts, chunk=128)
    caches = [oracle_cache_from_pool(v, SHAPE, b, L, L + S + 1) for b, L in enumerate(lens[:6])]
    spans = [[int(t) for t in synth.tokens(SEED, f"width.span.{b}", S, SHAPE.vocab)] for b in range(B)]

    def run(seqs):
        """Verify the spans of sequences `seqs` (the others get no rows), then rewind them."""
        v.ensure_capacity(_t([lens[b] + S if b in seqs else -1 for b in range(B)]), B)
        sp = [spans[b] if b in seqs else [] for b in range(B)]
        offs = np.concatenate([[0], np.cumsum([len(s) for s in sp])]).astype(np.int32)
        lg, am = _forward(v, [t for s in sp for t in s], offs, B, S)
        assert v.get_status() == 0
        v.rewind_cache(_t([lens[b] if b in seqs else -1 for b in range(B)]), B)
        torch.cuda.synchronize()
        return {b: lg[offs[b]:offs[b + 1]] for b in seqs}

    all16 = run(list(range(B)))
    first6 = run(list(range(6)))
    first3 = run([0, 1, 2])
    alone = {b: run([b])[b] for b in range(B)}
    for b in range(B):
        assert np.array_equal(all16[b], alone[b]), (b, float(np.abs(all16[b] - alone[b]).max()))
        if b < 6:
            assert np.array_equal(first6[b], alone[b]), (b, float(np.abs(first6[b] - alone[b]).max()))
        if b < 3:
            assert np.array_equal(first3[b], alone[b]), (b, float(np.abs(first3[b] - alone[b]).max()))
    ref = om.forward(caches[:6], spans[:6])
    worst = 0.0
    for b in range(6):
        _, d = check_rows(all16[b], all16[b].argmax(-1), ref[b], f"width b{b}")
        worst = max(worst, d)
    print(f"rows at N = 16, 32, 64 and 128 bit-identical; 128-row step max |dlogit| {worst:.3e} (first 6)")

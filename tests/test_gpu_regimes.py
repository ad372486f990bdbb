"""The verify path in the batch-16 and long-context regimes, against the oracle.

[PI] measures the verify step at batch 1, 8 and 16 and serves up to 16
concurrent sequences; the workloads here follow that: 16 sequences with
contexts drawn uniformly from [512, 4096] (1 to 5 key groups of 1024 positions
each, so one attention launch merges several groups of several sequences), and
one sequence over a 32768-token cache. The oracle runs its verify step on the
K/V the GPU wrote during the prefill (read back through the page table), which
keeps the oracle's cost to the verify itself; the GPU-written K/V is checked
against an oracle prefill here for the first 512 tokens of two of the batch-16
sequences, and in tests/test_gpu_4b.py at 848 tokens.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import workloads
from tests.helpers import check_rows, oracle_cache_from_pool, page_tables, upload_weights

pytestmark = pytest.mark.gpu

SHAPE = synth.QWEN3_4B.with_layers(2)
SEED = 2
P = 16


def _t(a):
    import torch
    return torch.as_tensor(np.asarray(a, dtype=np.int32)).cuda()


def _f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.fixture(scope="module")
def model():
    import torch
    torch.cuda.init()
    host, dev = upload_weights(SHAPE, SEED)
    return host, dev, oracle.DenseDecoder(SHAPE, lambda n: host[n])


# ----------------------------------------------------------------------------- attention alone

@pytest.mark.parametrize("spans", ["uniform8", "ragged1to17"])
def test_attention_batch16_multigroup_against_oracle(spans):
    """Paged attention of 16 sequences in one call, contexts U[512, 4096] (seed 3), synthetic
    bf16 K/V and queries: every output row of every sequence against the oracle's attention on
    the same values. The ragged case mixes spans of 1..17 rows (up to three launches of 8 span
    rows at 4 q heads per kv head)."""
    lens = [int(n) for n in workloads.context_lengths(3, 16)]
    S = [8] * 16 if spans == "uniform8" else [1, 17, 8, 3, 12, 5, 9, 2, 16, 7, 4, 11, 6, 10, 13, 1]
    assert max(lens) > 3 * 1024
    _attention_batch(lens, S, max(lens) + 32, spans)


def test_attention_mixed_group_counts():
    """One launch holding sequences of 1, 3, 9 and 20 key groups under a 24K-token configuration
    (one CTA per group: every multi-group sequence is merged by the separate merge kernel)."""
    _attention_batch([700, 2500, 9000, 20000], [8, 3, 17, 8], 24576, "mixed")


@pytest.mark.parametrize("L", [5000, 12000])
def test_attention_merge_in_kernel_and_by_merge_kernel(L):
    """Batch 1 under a 16K-token configuration (four CTAs per key group): 5 groups are merged
    inside the attention kernel, 12 groups by the merge kernel."""
    _attention_batch([L], [8], 16384, f"merge{L}")


@pytest.mark.parametrize("page", [8, 32, 64, 128])
def test_attention_page_sizes(page):
    """The K/V copies at other page sizes: one box per page below 64 slots, one per 64-slot half of a
    128-slot page; ragged contexts so chunks end mid-page and mid-box, one multi-group sequence."""
    _attention_batch([37, 700, 1500, 2100], [8, 3, 17, 5], 2200, f"page{page}", page=page)


def _attention_batch(lens, S, max_context, tag, page=P):
    import torch
    import speculative_decoding_verify_02_gb300 as sdv
    shape = synth.Shape("attn-4b-heads", 1, 256, 32, 8, 128, 256, 256)     # the 4B model's heads
    weights = {n: torch.zeros(d, dtype=torch.bfloat16, device="cuda") for n, d in shape.tensor_shapes().items()}
    B = len(lens)
    spans = tag
    R = sum(S)
    assert R <= 128
    P = page
    need = sum(-(-(L + s) // P) for L, s in zip(lens, S))
    v = sdv.Verifier(shape, weights, page_size=P, n_pages=need + 8, max_batch=B, max_rows=128, max_span=17,
                     max_context=max_context)
    v.ensure_capacity(_t([L + s for L, s in zip(lens, S)]), B)
    tab, _, _ = page_tables(v)
    nkv, nq, D = 8, 32, 128
    pool = v.pool.view(torch.bfloat16).view(v.ccfg.n_pages, 2, nkv, P, D)
    kvs = []
    for b in range(B):
        T = lens[b] + S[b]
        kv = synth.normal_bf16(3, f"b16attn.kv.{b}", 2 * T * nkv * D, 1.0).reshape(2, T, nkv, D)
        kvs.append(kv)
        npg = -(-T // P)
        padded = torch.zeros(2, npg * P, nkv, D, dtype=torch.bfloat16, device="cuda")
        padded[:, :T] = sdv.upload_bf16(kv)
        idx = torch.as_tensor(tab[b, :npg].astype(np.int64), device="cuda")
        pool[idx] = padded.view(2, npg, P, nkv, D).permute(1, 0, 3, 2, 4)
    q = synth.normal_bf16(3, f"b16attn.q.{spans}", R * nq * D, 1.0).reshape(R, nq, D)
    out = torch.zeros(R, nq * D, dtype=torch.bfloat16, device="cuda")
    row_off = np.concatenate([[0], np.cumsum(S)])
    v.op_attention(0, sdv.upload_bf16(q), _t(row_off), _t(lens), B, max(S), out)
    torch.cuda.synchronize()
    assert v.get_status() == 0
    got = out.float().cpu().numpy().reshape(R, nq, D)
    worst = 0.0
    for b in range(B):
        r0, r1 = row_off[b], row_off[b + 1]
        ref = oracle.attention_rows(_f64(q[r0:r1]), _f64(kvs[b][0]), _f64(kvs[b][1]),
                                    np.arange(lens[b], lens[b] + S[b]), 1 / np.sqrt(D))
        err = float(np.abs(got[r0:r1] - ref).max())
        assert err <= 2e-2, (b, lens[b], S[b], err)
        worst = max(worst, err)
    print(f"b16 attention ({spans}): max |d| {worst:.3e} over {R} rows, contexts {min(lens)}..{max(lens)}")


# ----------------------------------------------------------------------------- whole verify steps

def _oracle_pool_after_prefill(v, lens, chunk=128):
    """The oracle page pool after the same per-chunk reservations as SpecLoop.prefill."""
    B = len(lens)
    pool = oracle.PagePool(v.ccfg.n_pages, P, B, v.pages_per_seq)
    for b, L in enumerate(lens):
        for c0 in range(0, L, chunk):
            req = [-1] * B
            req[b] = min(c0 + chunk, L)
            pool.ensure_capacity(req)
            pool.set_length(b, req[b])
    return pool


def _verify_over_gpu_kv(model, lens, S, name):
    """Prefill `lens` uniform contexts on the GPU, then one verify step of S rows per sequence
    (current token = the GPU's first token, uniform drafts), compared with the oracle's verify on
    the GPU-written K/V: per-row logits and argmax, the K/V the span wrote, acceptance, new
    lengths and the page tables after the rewind."""
    import torch
    from speculative_decoding_verify_02_gb300 import Verifier
    from speculative_decoding_verify_02_gb300.runner import SpecLoop
    host, dev, om = model
    B = len(lens)
    prompts = [workloads.uniform_context(3, L, SHAPE.vocab, name=f"{name}.ctx.{b}") for b, L in enumerate(lens)]
    n_pages = sum(-(-(L + S) // P) for L in lens) + 8
    v = Verifier(SHAPE, dev, page_size=P, n_pages=n_pages, max_batch=B, max_rows=128, max_span=128,
                 max_context=max(lens) + 64)
    first = SpecLoop(v, B, S).prefill(prompts, chunk=128)
    caches = [oracle_cache_from_pool(v, SHAPE, b, L, L + S + 1) for b, L in enumerate(lens)]
    spans = [[int(first[b])] + [int(t) for t in synth.tokens(SEED, f"{name}.drafts.{b}", S - 1, SHAPE.vocab)]
             for b in range(B)]
    offs = np.concatenate([[0], np.cumsum([len(s) for s in spans])]).astype(np.int32)
    flat = [t for s in spans for t in s]
    R = len(flat)
    v.ensure_capacity(_t([L + S for L in lens]), B)
    am = _t(np.zeros(R))
    lg = torch.zeros(R, SHAPE.vocab, dtype=torch.float32, device="cuda")
    tok_t, off_t = _t(flat), _t(offs)
    v.spec_forward(tok_t, off_t, B, R, S, am, lg)
    n_acc, com, n_com, new_len = _t(np.zeros(B)), _t(np.zeros(B * S)), _t(np.zeros(B)), _t(np.zeros(B))
    v.accept_greedy(tok_t, off_t, am, B, S, n_acc, com, n_com, new_len)
    torch.cuda.synchronize()
    assert v.get_status() == 0
    lg, am = lg.cpu().numpy(), am.cpu().numpy()
    tab_before, _, _ = page_tables(v)
    pool_dev = v.pool.view(torch.bfloat16).view(SHAPE.n_layers, v.ccfg.n_pages, 2, SHAPE.n_kv_heads, P,
                                                 SHAPE.head_dim)
    ref = om.forward(caches, spans)
    g_m, g_new = n_acc.cpu().numpy(), new_len.cpu().numpy()
    opool = _oracle_pool_after_prefill(v, lens)
    opool.ensure_capacity([L + S for L in lens])
    flips_all, worst, checked = [], 0.0, 0
    new_lens = []
    for b in range(B):
        r0, r1 = offs[b], offs[b + 1]
        flips, d = check_rows(lg[r0:r1], am[r0:r1], ref[b], f"{name} b{b}")
        worst = max(worst, d)
        flips_all += [(b, f) for f in flips]
        m, committed = oracle.accept_greedy(spans[b][1:], [int(x) for x in ref[b].argmax(-1)])
        nl = lens[b] + m + 1
        new_lens.append(nl)
        if not flips:
            checked += 1
            assert g_m[b] == m and g_new[b] == nl, (b, g_m[b], m)
            assert com[b * S:b * S + m + 1].cpu().tolist() == committed
        # the span's K/V as the GPU wrote it, against the oracle's (bf16-rounded) rows
        for pos in (lens[b], lens[b] + S - 1):
            page = tab_before[b, pos // P]
            for l in range(SHAPE.n_layers):
                k = pool_dev[l, page, 0, :, pos % P].double().cpu().numpy()
                np.testing.assert_allclose(k, caches[b].K[l][pos], atol=3e-2, rtol=2e-2)
        opool.set_length(b, lens[b] + S)
    v.rewind_cache(_t(new_lens), B)                                  # teacher forcing: the oracle's lengths
    opool.rewind(new_lens)
    tab, npg, top = page_tables(v)
    for b in range(B):
        assert tab[b, :npg[b]].tolist() == opool.table[b], b
    assert top == len(opool.free)
    print(f"{name}: max |dlogit| {worst:.3e}, {checked}/{B} sequences exact, near-tie flips {flips_all}")
    v.close()


def test_prefill_kv_of_two_batch16_sequences(model):
    """The paged K/V the GPU prefill writes, every position of both layers, against the oracle's
    prefill (its cache rounded to bf16 like the pool): the first 512 tokens of two of config 3's
    sequences, prefilled together in 128-row chunks."""
    import torch
    from speculative_decoding_verify_02_gb300 import Verifier
    from speculative_decoding_verify_02_gb300.runner import SpecLoop
    host, dev, om = model
    n = 512
    prompts = [workloads.uniform_context(3, n, SHAPE.vocab, name=f"b16.ctx.{b}") for b in (0, 1)]
    caches = [oracle.SeqCache(SHAPE, n + 8, kv_dtype="bf16") for _ in prompts]
    for c, p in zip(caches, prompts):
        om.forward([c], [p], last_row_logits=True)
    v = Verifier(SHAPE, dev, page_size=P, n_pages=2 * n // P + 8, max_batch=2, max_rows=128, max_span=128,
                 max_context=n + 64)
    SpecLoop(v, 2, 8).prefill(prompts, chunk=128)
    assert v.get_status() == 0
    tab, _, _ = page_tables(v)
    nkv, D = SHAPE.n_kv_heads, SHAPE.head_dim
    pool = v.pool.view(torch.bfloat16).view(SHAPE.n_layers, v.ccfg.n_pages, 2, nkv, P, D)
    same = total = 0
    worst = 0.0
    for b in range(2):
        pages = torch.as_tensor(tab[b, :n // P].astype(np.int64), device="cuda")
        for l in range(SHAPE.n_layers):
            kv = pool[l].index_select(0, pages).permute(1, 0, 3, 2, 4).reshape(2, n, nkv, D).double().cpu().numpy()
            for which, ref in ((0, caches[b].K[l][:n]), (1, caches[b].V[l][:n])):
                np.testing.assert_allclose(kv[which], ref, atol=3e-2, rtol=2e-2)
                worst = max(worst, float(np.abs(kv[which] - ref).max()))
                same += int((kv[which] == ref).sum())
                total += kv[which].size
    print(f"prefill K/V of two batch-16 sequences: {same / total:.4f} of the values bit-identical, "
          f"max |d| {worst:.3e}")
    v.close()


def test_verify_step_batch16_contexts_512_to_4096(model):
    """Config 3's regime: 16 sequences, contexts U[512, 4096], K = 7."""
    lens = [int(n) for n in workloads.context_lengths(3, 16)]
    _verify_over_gpu_kv(model, lens, 8, "b16")


def test_verify_step_32k_context(model):
    """Config 4's regime: one sequence over a 32768-token cache, K = 7 (33 key groups)."""
    _verify_over_gpu_kv(model, [32768], 8, "ctx32k")

"""The scratch-free paged-attention entry point, sdv_paged_attention_noalloc.

It serves callers that cannot allocate device memory (code running under CUDA
graph capture, plug-ins handed only their buffers, fixed-memory deployments):
its scratch is a static device array inside the library. These tests call it
through the C ABI and check it against the context-based sdv_op_attention and
the oracle's attention on the same inputs, on two calls in a row (the second
reuses the scratch the first left behind), and check the status word that
sdv_noalloc_status reads back. The file is named to run last; it also passes
alone.
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

TOL = 3e-2
P = 16


def _t(a):
    import torch
    return torch.as_tensor(np.asarray(a, dtype=np.int32)).cuda()


def _f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _setup(shape, bases, spans, max_context, seed_name):
    """A context with one layer of synthetic K/V and queries; returns what the calls need."""
    import torch
    import speculative_decoding_verify_02_gb300 as sdv
    from tests.helpers import page_tables
    weights = {n: torch.zeros(d, dtype=torch.bfloat16, device="cuda") for n, d in shape.tensor_shapes().items()}
    B = len(bases)
    v = sdv.Verifier(shape, weights, page_size=P, n_pages=B * (max_context // P) + 8, max_batch=B, max_rows=128,
                     max_span=max(spans), max_context=max_context)
    v.ensure_capacity(_t([min(b + s, max_context) for b, s in zip(bases, spans)]), B)
    tab, _, _ = page_tables(v)
    assert v.get_status() == 0
    nkv, nq, D = shape.n_kv_heads, shape.n_q_heads, shape.head_dim
    layer_elems = v.ccfg.n_pages * 2 * nkv * P * D
    bits = synth.normal_bf16(11, f"{seed_name}.kv", layer_elems, 1.0)
    pool = v.pool.view(torch.bfloat16)[:layer_elems]                    # layer 0
    pool.copy_(sdv.upload_bf16(bits))
    R = sum(spans)
    qbits = synth.normal_bf16(11, f"{seed_name}.q", R * nq * D, 1.0)
    return v, tab, bits.reshape(v.ccfg.n_pages, 2, nkv, P, D), pool, qbits.reshape(R, nq, D)


def _oracle_rows(shape, tab, kv_pages, qbits, bases, spans):
    """The oracle's attention of every accepted sequence, reading K/V through the page table."""
    D = shape.head_dim
    out, r0 = [], 0
    for b, (L, S) in enumerate(zip(bases, spans)):
        T = L + S
        pages = tab[b, :-(-T // P)]
        kv = kv_pages[pages].transpose(1, 0, 3, 2, 4).reshape(2, -1, shape.n_kv_heads, D)[:, :T]
        out.append(oracle.attention_rows(_f64(qbits[r0:r0 + S]), _f64(kv[0]), _f64(kv[1]), np.arange(L, T),
                                         1 / np.sqrt(D)))
        r0 += S
    return out


def test_noalloc_attention_matches_op_attention_twice():
    """head_dim 128, 4 q heads per kv head (the 4B model's grouping); one single-group and one
    multi-group sequence: two calls in a row against sdv_op_attention and the oracle."""
    import torch
    import speculative_decoding_verify_02_gb300 as sdv
    shape = synth.Shape("attn-probe", 1, 256, 8, 2, 128, 256, 256)
    bases, spans, max_context = [700, 2500], [5, 8], 3072
    v, tab, kv_pages, pool, q = _setup(shape, bases, spans, max_context, "noalloc")
    nq, nkv, D = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    R = sum(spans)
    q_dev = sdv.upload_bf16(q)
    row_off, base = _t([0, spans[0], R]), _t(bases)
    ref = torch.zeros(R, nq * D, dtype=torch.bfloat16, device="cuda")
    v.op_attention(0, q_dev, row_off, base, 2, max(spans), ref)
    table = _t(tab.reshape(-1))
    outs = []
    for _ in range(2):
        out = torch.full((R, nq * D), float("nan"), dtype=torch.bfloat16, device="cuda")
        sdv.paged_attention_noalloc(q_dev, pool, table, v.pages_per_seq, P, v.ccfg.n_pages, row_off, base, 2, nq,
                                    nkv, D, max(spans), max_context, out)
        outs.append(out)
    assert sdv.noalloc_status() == 0
    torch.cuda.synchronize()
    assert v.get_status() == 0
    r = ref.float().cpu().numpy()
    assert np.isfinite(r).all()
    expect = np.concatenate([x.reshape(-1, nq * D) for x in _oracle_rows(shape, tab, kv_pages, q, bases, spans)])
    for o in outs:
        got = o.float().cpu().numpy()
        np.testing.assert_allclose(got, r, atol=TOL, rtol=0)
        np.testing.assert_allclose(got, expect, atol=TOL, rtol=0)

    # sizes beyond the scratch are refused on the host with a clear error, and nothing runs
    with pytest.raises(sdv.SdvError) as e:
        sdv.paged_attention_noalloc(q_dev, pool, table, v.pages_per_seq, P, v.ccfg.n_pages, row_off, base, 64, nq,
                                    nkv, D, 128, max_context, ref)
    assert e.value.code == sdv.SDV_ERR_CAPACITY
    v.close()


def test_noalloc_head_dim_64_multi_launch_and_rejected_rows():
    """head_dim 64, spans of 20 and 24 rows (more than 64 / 4 = 16 span rows per launch, so the
    launch loop runs twice over the shared, self-resetting group counters), and a third sequence
    whose span passes max_context: its rows come back NaN and the status reads SDV_ERR_CAPACITY;
    the accepted sequences match the oracle."""
    import torch
    import speculative_decoding_verify_02_gb300 as sdv
    shape = synth.Shape("attn-probe-64", 1, 256, 8, 2, 64, 256, 256)
    max_context = 2048
    bases, spans = [100, 1500, 2040], [20, 24, 16]                 # the third passes max_context
    v, tab, kv_pages, pool, q = _setup(shape, bases, spans, max_context, "noalloc64")
    nq, nkv, D = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    R = sum(spans)
    q_dev = sdv.upload_bf16(q)
    offs = np.concatenate([[0], np.cumsum(spans)])
    table = _t(tab.reshape(-1))
    expect = _oracle_rows(shape, tab, kv_pages, q, bases[:2], spans[:2])
    for _ in range(2):
        out = torch.zeros(R, nq * D, dtype=torch.bfloat16, device="cuda")
        sdv.paged_attention_noalloc(q_dev, pool, table, v.pages_per_seq, P, v.ccfg.n_pages, _t(offs), _t(bases), 3,
                                    nq, nkv, D, max(spans), max_context, out)
        assert sdv.noalloc_status() == sdv.SDV_ERR_CAPACITY
        got = out.float().cpu().numpy()
        for b in range(2):
            np.testing.assert_allclose(got[offs[b]:offs[b + 1]], expect[b].reshape(spans[b], nq * D), atol=TOL,
                                       rtol=0)
        assert np.isnan(got[offs[2]:offs[3]]).all()
    # a span longer than max_span: rejected the same way, with SDV_ERR_ARG
    out = torch.zeros(R, nq * D, dtype=torch.bfloat16, device="cuda")
    sdv.paged_attention_noalloc(q_dev, pool, table, v.pages_per_seq, P, v.ccfg.n_pages, _t(offs[:3]),
                                _t(bases[:2]), 2, nq, nkv, D, 20, max_context, out)
    assert sdv.noalloc_status() == sdv.SDV_ERR_ARG
    got = out.float().cpu().numpy()
    np.testing.assert_allclose(got[:20], expect[0].reshape(20, nq * D), atol=TOL, rtol=0)
    assert np.isnan(got[20:44]).all()
    assert sdv.noalloc_status() == 0                              # reading cleared it
    v.close()


def test_noalloc_page_id_out_of_range_sets_status():
    """A page table entry outside [0, n_pages): the kernel skips those loads (zero K/V rows) and
    the status word reports SDV_ERR_CAPACITY; the next good call reports 0 again."""
    import torch
    import speculative_decoding_verify_02_gb300 as sdv
    shape = synth.Shape("attn-probe", 1, 256, 8, 2, 128, 256, 256)
    bases, spans, max_context = [300], [4], 512
    v, tab, kv_pages, pool, q = _setup(shape, bases, spans, max_context, "noalloc.bad")
    nq, nkv, D = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    q_dev = sdv.upload_bf16(q)
    bad = tab.copy()
    bad[0, 3] = v.ccfg.n_pages + 5
    out = torch.zeros(4, nq * D, dtype=torch.bfloat16, device="cuda")
    args = (v.pages_per_seq, P, v.ccfg.n_pages, _t([0, 4]), _t(bases), 1, nq, nkv, D, 4, max_context, out)
    sdv.paged_attention_noalloc(q_dev, pool, _t(bad.reshape(-1)), *args)
    assert sdv.noalloc_status() == sdv.SDV_ERR_CAPACITY
    sdv.paged_attention_noalloc(q_dev, pool, _t(tab.reshape(-1)), *args)
    assert sdv.noalloc_status() == 0
    expect = _oracle_rows(shape, tab, kv_pages, q, bases, spans)[0].reshape(4, nq * D)
    np.testing.assert_allclose(out.float().cpu().numpy(), expect, atol=TOL, rtol=0)
    v.close()

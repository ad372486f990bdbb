"""The scratch-free paged-attention entry point, sdv_paged_attention_noalloc.

It serves callers that cannot allocate device memory (code running under CUDA
graph capture, plug-ins handed only their buffers, fixed-memory deployments):
its scratch is a static device array inside the library. This checks it,
through the C ABI, against the context-based sdv_op_attention on the same
inputs, on two calls in a row (the second reuses the scratch the first left
behind). The file is named to run last; it also passes alone.
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

# Attention-only shape: head_dim 128 with 4 q heads per kv head, as in the 4B model.
SHAPE = synth.Shape("attn-probe", 1, 256, 8, 2, 128, 256, 256)
TOL = 3e-2


def test_noalloc_attention_matches_op_attention_twice():
    import torch
    import speculative_decoding_verify_02_gb300 as sdv

    weights = {n: torch.zeros(dims, dtype=torch.bfloat16, device="cuda") for n, dims in SHAPE.tensor_shapes().items()}
    P, max_context = 16, 3072
    v = sdv.Verifier(SHAPE, weights, page_size=P, n_pages=max_context // P * 2 + 8, max_batch=2, max_rows=128,
                     max_span=16, max_context=max_context)
    bases, spans = [700, 2500], [5, 8]                 # one single-group and one multi-group sequence
    t = lambda a: torch.as_tensor(np.asarray(a, dtype=np.int32)).cuda()
    v.ensure_capacity(t([b + s for b, s in zip(bases, spans)]), 2)
    table = t(np.zeros(2 * v.pages_per_seq))
    n_pages, free_top = t([0, 0]), t([0])
    v.page_table(table, n_pages, free_top)
    torch.cuda.synchronize()
    assert v.get_status() == 0

    nkv, nq, D = SHAPE.n_kv_heads, SHAPE.n_q_heads, SHAPE.head_dim
    layer_elems = v.ccfg.n_pages * 2 * nkv * P * D
    pool = v.pool.view(torch.bfloat16)[:layer_elems]  # layer 0
    pool.copy_(sdv.upload_bf16(synth.normal_bf16(11, "noalloc.kv", layer_elems, 1.0)))
    R = sum(spans)
    q = sdv.upload_bf16(synth.normal_bf16(11, "noalloc.q", R * nq * D, 1.0))
    row_off, base = t([0, spans[0], R]), t(bases)

    ref = torch.zeros(R, nq * D, dtype=torch.bfloat16, device="cuda")
    v.op_attention(0, q, row_off, base, 2, max(spans), ref)
    outs = []
    for _ in range(2):
        out = torch.full((R, nq * D), float("nan"), dtype=torch.bfloat16, device="cuda")
        sdv.paged_attention_noalloc(q, pool, table, v.pages_per_seq, P, v.ccfg.n_pages, row_off, base, 2, nq, nkv, D,
                                    max(spans), max_context, out)
        outs.append(out)
    torch.cuda.synchronize()
    assert v.get_status() == 0
    r = ref.float().cpu().numpy()
    assert np.isfinite(r).all()
    for o in outs:
        np.testing.assert_allclose(o.float().cpu().numpy(), r, atol=TOL, rtol=0)

    # sizes beyond the scratch are refused on the host with a clear error, and nothing runs
    with pytest.raises(sdv.SdvError) as e:
        sdv.paged_attention_noalloc(q, pool, table, v.pages_per_seq, P, v.ccfg.n_pages, row_off, base, 64, nq, nkv,
                                    D, 128, max_context, ref)
    assert e.value.code == sdv.SDV_ERR_CAPACITY
    v.close()

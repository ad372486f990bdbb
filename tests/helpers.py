"""Shared test plumbing: weight upload, context construction and the parity rules.

Parity rules (the tolerance the verify path is held to):
  * logits: max |GPU - oracle| <= LOGIT_TOL (bf16 weights and activations with
    fp32 accumulation against the float64 oracle);
  * argmax: identical wherever the oracle's top-2 margin exceeds MARGIN;
    rows at or under that margin are near-ties, reported, not failed.
"""
import numpy as np

LOGIT_TOL = 3e-2
MARGIN = 0.05


def upload_weights(shape, seed):
    import synth
    from speculative_decoding_verify_02_gb300 import upload_bf16
    host = {}
    dev = {}
    for name in shape.tensor_shapes():
        host[name] = synth.tensor(shape, seed, name)
        dev[name] = upload_bf16(host[name])
    return host, dev


def margins(logits):
    top2 = np.sort(logits, axis=-1)[..., -2:]
    return top2[..., 1] - top2[..., 0]


def check_rows(gpu_logits, gpu_argmax, ref_logits, what=""):
    """Compare per-row logits and argmax; returns the near-tie flips (row, margin)."""
    d = np.abs(gpu_logits.astype(np.float64) - ref_logits).max() if ref_logits.size else 0.0
    assert d <= LOGIT_TOL, f"{what}: max |dlogit| {d:.4g} > {LOGIT_TOL}"
    ref_am = ref_logits.argmax(-1)
    mg = margins(ref_logits)
    flips = []
    for r in range(len(ref_am)):
        if gpu_argmax[r] != ref_am[r]:
            assert mg[r] <= MARGIN, f"{what}: row {r} argmax {gpu_argmax[r]} != {ref_am[r]} at margin {mg[r]:.4f}"
            flips.append((r, float(mg[r])))
    # the reported argmax must be the argmax of the reported logits (lowest index on a tie)
    np.testing.assert_array_equal(gpu_argmax, gpu_logits.argmax(-1))
    return flips, d


def page_tables(v):
    """(page table [max_batch][pages_per_seq], pages held [max_batch], free-stack depth) on the host."""
    import torch
    B = v.ccfg.max_batch
    tab = torch.zeros(B * v.pages_per_seq, dtype=torch.int32, device="cuda")
    npg = torch.zeros(B, dtype=torch.int32, device="cuda")
    top = torch.zeros(1, dtype=torch.int32, device="cuda")
    v.page_table(tab, npg, top)
    torch.cuda.synchronize()
    return tab.cpu().numpy().reshape(B, -1), npg.cpu().numpy(), int(top.item())


def oracle_cache_from_pool(v, shape, b, length, capacity):
    """An oracle cache of sequence b whose positions 0..length-1 hold the K/V the GPU wrote into
    the paged pool (bf16 values, read through the page table), so that an oracle verify step can
    run on the GPU-written KV."""
    import oracle
    import torch
    P, nkv, D = v.ccfg.page_size, shape.n_kv_heads, shape.head_dim
    tab, _, _ = page_tables(v)
    pages = torch.as_tensor(tab[b, :-(-length // P)].astype(np.int64), device="cuda")
    pool = v.pool.view(torch.bfloat16).view(shape.n_layers, v.ccfg.n_pages, 2, nkv, P, D)
    cache = oracle.SeqCache(shape, capacity, kv_dtype="bf16")
    for l in range(shape.n_layers):
        kv = pool[l].index_select(0, pages)                      # [pages][2][nkv][P][D]
        kv = kv.permute(1, 0, 3, 2, 4).reshape(2, -1, nkv, D)[:, :length]
        kv = kv.double().cpu().numpy()
        cache.K[l][:length] = kv[0]
        cache.V[l][:length] = kv[1]
    cache.length = length
    return cache

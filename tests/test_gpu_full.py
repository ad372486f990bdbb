"""Full-size checks: the 36-layer Qwen3-4B-shaped verify step at the benchmark's
configuration (848-token context, S = 8), and paged attention at a
32768-token context (the long-context configuration), against the oracle.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import workloads
from tests.helpers import MARGIN, check_rows, margins

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

# Bound on max |dlogit| of the 36-layer verify against the oracle whose cache keeps K/V in float64
# instead of bf16: the K/V rounding alone moves logits by about 0.02 per 2 layers of emulation and
# measured 0.054 at 36 layers; the bar is set at 0.1.
EXACT_KV_BOUND = 0.1


def _t(a):
    import torch
    return torch.as_tensor(np.asarray(a, dtype=np.int32)).cuda()


def test_full_model_verify_step_848():
    """All 36 layers, bench configuration: every logit of the 8 verify rows within
    tolerance of the float64 oracle, argmax equal outside near-ties."""
    import torch
    from speculative_decoding_verify_02_gb300 import Verifier, upload_bf16
    from speculative_decoding_verify_02_gb300.runner import SpecLoop
    shape, seed = synth.QWEN3_4B, 2
    host = {n: synth.tensor(shape, seed, n) for n in shape.tensor_shapes()}
    dev = {n: upload_bf16(a) for n, a in host.items()}
    v = Verifier(shape, dev, page_size=16, n_pages=128, max_batch=1, max_rows=128, max_span=128, max_context=1024)
    ctx = workloads.uniform_context(seed, 848, shape.vocab)
    first = int(SpecLoop(v, 1, 8).prefill([ctx])[0])
    om = oracle.DenseDecoder(shape, lambda n: host[n], cache_weights=False)
    cache = oracle.SeqCache(shape, 900, kv_dtype="bf16")
    ref_pre = om.forward([cache], [ctx], last_row_logits=True)[0]
    if margins(ref_pre)[0] > MARGIN:
        assert first == int(ref_pre.argmax())
    span = [int(ref_pre.argmax())] + [int(t) for t in workloads.uniform_drafts(seed, 0, 7, shape.vocab)]
    ref = om.forward([cache], [span])[0]
    v.ensure_capacity(_t([856]), 1)
    am = _t(np.zeros(8))
    lg = torch.zeros(8, shape.vocab, dtype=torch.float32, device="cuda")
    v.spec_forward(_t(span), _t([0, 8]), 1, 8, 8, am, lg)
    torch.cuda.synchronize()
    assert v.get_status() == 0
    flips, d = check_rows(lg.cpu().numpy(), am.cpu().numpy(), ref, "36-layer verify")
    # The same step against an oracle whose cache keeps K/V exactly (the literal fp32 reading of the
    # bar): the bf16 K/V storage costs up to EXACT_KV_BOUND on the logits at 36 layers, and every row
    # whose exact-KV top-2 margin exceeds twice the measured difference keeps its argmax.
    exact = oracle.SeqCache(shape, 900)
    om.forward([exact], [ctx], last_row_logits=True)
    ref64 = om.forward([exact], [span])[0]
    g = lg.cpu().numpy().astype(np.float64)
    d64 = float(np.abs(g - ref64).max())
    assert d64 <= EXACT_KV_BOUND, f"exact-KV oracle: max |dlogit| {d64:.4g} > {EXACT_KV_BOUND}"
    sure = margins(ref64) > 2 * d64
    np.testing.assert_array_equal(am.cpu().numpy()[sure], ref64.argmax(-1)[sure])
    print(f"36-layer verify at 848: max |dlogit| {d:.3e} (bf16 KV oracle), {d64:.3e} (exact-KV oracle, "
          f"{int(sure.sum())}/8 rows argmax-checked), near-tie flips {flips}")


@pytest.mark.parametrize("L,S", [(32768, 8), (1020, 8), (2040, 16)])
def test_attention_long_context(L, S):
    """Paged attention of an S-row span over an L-token cache: 32768 + 8 (33 key groups of 1024
    positions), and spans straddling a key group (1020 + 8, 2040 + 16), whose first rows see no
    key of the last group, so that group's state is empty for them and must contribute nothing to
    the merge across groups; 2040 + 16 also takes two launches of 8 span rows."""
    attention_long_context(L, S)


def attention_long_context(L, S):
    """Paged attention of an S-row span over an L-token cache (synthetic K/V and
    q), every output against the oracle's attention on the same bf16 values."""
    import torch
    import speculative_decoding_verify_02_gb300 as sdv
    shape = synth.Shape("attn-4b-heads", 1, 256, 32, 8, 128, 256, 256)     # the 4B model's heads
    weights = {n: torch.zeros(d, dtype=torch.bfloat16, device="cuda") for n, d in shape.tensor_shapes().items()}
    P = 16
    n_pages = (L + S) // P + 2
    v = sdv.Verifier(shape, weights, page_size=P, n_pages=n_pages, max_batch=1, max_rows=128, max_span=16,
                     max_context=n_pages * P)
    v.ensure_capacity(_t([L + S]), 1)
    tab, npg, top = _t(np.zeros(v.pages_per_seq)), _t([0]), _t([0])
    v.page_table(tab, npg, top)
    torch.cuda.synchronize()
    tab = tab.cpu().numpy()
    nkv, nq, D = 8, 32, 128
    T = L + S
    kv = synth.normal_bf16(4, "long.kv", 2 * T * nkv * D, 1.0).reshape(2, T, nkv, D)
    pool = v.pool.view(torch.bfloat16).view(n_pages, 2, nkv, P, D)
    kv_dev = sdv.upload_bf16(kv)                                            # [2][T][nkv][D]
    for p in range(-(-T // P)):
        pos = np.arange(p * P, min((p + 1) * P, T))
        pool[tab[p], :, :, :len(pos)] = kv_dev[:, pos].permute(0, 2, 1, 3)
    q = synth.normal_bf16(4, "long.q", S * nq * D, 1.0)
    out = torch.zeros(S, nq * D, dtype=torch.bfloat16, device="cuda")
    v.op_attention(0, sdv.upload_bf16(q), _t([0, S]), _t([L]), 1, S, out)
    torch.cuda.synchronize()
    assert v.get_status() == 0
    f64 = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = oracle.attention_rows(f64(q).reshape(S, nq, D), f64(kv[0]), f64(kv[1]), np.arange(L, L + S),
                                1 / np.sqrt(D))
    got = out.float().cpu().numpy().reshape(S, nq, D)
    err = np.abs(got - ref).max()
    print(f"attention over {L} + {S}: max |d| {err:.3e}")
    assert err <= 2e-2

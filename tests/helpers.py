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

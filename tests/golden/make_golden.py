"""Writes tests/golden/tiny_ngram_k4_oracle.txt from the oracle alone.

Run from the repository root:  python tests/golden/make_golden.py
The file records the oracle's greedy spec loop on the tiny decoder (seed 1,
128-token motif prompt, 2-gram lookup, fixed K=4, 32 tokens) with each verify
row's argmax and top-2 logit margin.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402
from synth import workloads  # noqa: E402


def main():
    W = synth.weights(synth.TINY, 1)
    model = oracle.DenseDecoder(synth.TINY, lambda n: W[n])
    streams, recs, _ = oracle.generate(model, [workloads.motif_prompt(1)], 32, drafter="ngram", k=4,
                                       keep_logits=True)
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_ngram_k4_oracle.txt")
    with open(out, "w") as f:
        f.write("# Oracle output, tiny decoder (seed 1), 128-token motif prompt, 2-gram lookup, K=4, 32 tokens.\n")
        f.write("# Written by tests/golden/make_golden.py (oracle only).\n")
        f.write("stream | " + " ".join(map(str, streams[0])) + "\n")
        for r in recs:
            lg = r.logits[0]
            top2 = np.sort(lg, axis=-1)[:, -2:]
            margins = " ".join(f"{x:.6f}" for x in (top2[:, 1] - top2[:, 0]))
            f.write("step | " + " ".join(map(str, r.spans[0])) + " | " + " ".join(map(str, r.argmax[0]))
                    + f" | {r.m[0]} | {r.new_len[0]} | {margins}\n")


if __name__ == "__main__":
    main()

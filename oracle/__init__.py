"""CPU oracle for the speculative-decoding verify path.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports, calls or
links this package: only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it. It
shares no code with the CUDA path; the only common dependency is the seeded
input generator package ``synth``.

It is plain and slow on purpose: numpy in float64, the steps in the order the
pages give them, a library matmul as the only borrowed primitive.

Sources (named by page title and section):
  [TS] TensorSharp, "Speculative decoding" (docs/speculative_decoding.md):
       the shared loop and trunk seam; the protocol (draft, verify, rollback,
       commit); n-gram prompt lookup; sliding-window caches and rollback.
  [PI] pegainfer, "Qwen3 DFlash speculative decoding"
       (docs/models/qwen3/dflash-speculative-decoding.md): the transaction
       (propose, verify, accept, commit/roll back); draft-seed alignment;
       the losslessness gate; the capture-shape gotcha (span truncation).
  [CA] CoreAI model zoo, "spec-decode n-gram on a dense target"
       (knowledge/spec-decode-ngram-dense): dense rollback by position,
       the rows gate, adaptive K, the prompt-lookup minimum match.

Pins: every function is checked in tests/test_oracle_*.py against closed
forms, library routines (torch float64), brute force on tiny inputs and the
invariants the pages state. Parity of the decoder's logits is pinned by those
library cross-checks and invariants only; the pages print no logits that could
pin values for these synthetic models.
"""
from .model import DenseDecoder, SeqCache, rmsnorm, silu, rope_neox, attention_rows, argmax_lowest, round_bf16
from .pages import PagePool, CapacityError
from .spec import accept_greedy, ngram_propose, adapt_k, ngram_propose_multi, required_order, NgramIndex
from .loop import generate, StepRecord
from .sampling import draw_rows, perturbed, gumbel, uniforms

__all__ = [
    "DenseDecoder", "SeqCache", "round_bf16", "rmsnorm", "silu", "rope_neox", "attention_rows", "argmax_lowest",
    "PagePool", "CapacityError", "accept_greedy", "ngram_propose", "adapt_k", "generate", "StepRecord",
    "draw_rows", "perturbed", "gumbel", "uniforms", "ngram_propose_multi", "required_order", "NgramIndex",
]

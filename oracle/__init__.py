"""Oracle for the shared-round verify step: plain, slow, float64 CPU code.

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it. The
product path (the CUDA library and its Python binding) never imports, calls or
links anything here, and this package imports nothing from the product.

Sources (web pages about the TensorFold project):
  * PR #1377 "LFM2: shared-round decode": the commits "a verify's greedy rows
    take the GPU's pick of their logits" (the greedy pick), "a shared round runs
    each layer's conv and attention once over all its streams" (segment table,
    per-stream partials, and checks against float64 attention and against
    the conv's steps replayed on the host), and
    the commit on the kernel contract and its planted controls.
  * PR #1391 "lfm2: draft with LiquidAI's DSpark drafter (--drafter)": the
    target checks every draft; its attention stays causal.
  * The same PR's drafter side (``oracle/draft.py``): the Markov head's pick
    and the kernel that fills the verify's ids from the drafter's picks.
  * Issue #1374 "LFM2.5-24B-A2B on Metal: drafts with LiquidAI's DSpark drafter
    (proposal and gate)", section "What": a drafted reply equals its plain one.

The pages print no formulas; every reading taken where they are silent is
stated in the docstring of the function that takes it.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, invariants, hand-worked fixtures under ``tests/golden/`` and
brute force on tiny inputs), except what the docstring of ``step`` marks as
"parity unpinned".
"""

from .step import (  # noqa: F401
    NQ, NKV, D, H, CIN, KW, SCALE,
    bf16_to_f64, f64_to_bf16_rne,
    short_conv_stream, conv_layer,
    attention_stream, attention_partials_stream, merge_partials, attention_layer,
    argmax_rows, accept_stream, accept_all, rewind_state,
    verify_step,
)
from .draft import (  # noqa: F401
    f64_to_bf16_rne_any, markov_step, markov_chain, markov_all,
    DFLAG_BAD_PENDING, DFLAG_BAD_DRAFT, draft_ids_all,
)

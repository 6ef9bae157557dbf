"""CPU oracle for the DeltaNet verify / accept / commit / prefill-checkpoint path
and for drafting from the request's own context.

TEST INFRASTRUCTURE ONLY. This package is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py``, and by nothing else. The product path
(``deltanet_recurrent_state_gb300``) never imports, calls or links it; the two
share no code, and the oracle imports nothing from the product package.

Everything is plain NumPy in float64. Each function follows the definition it
cites, token by token, with no blocking, fusion or reordering: a reader can
check it against the formula by eye. Values that the product stores in fp16
are rounded to fp16 here at exactly the same places (round-to-nearest-even,
numpy's direct float64 -> float16 conversion), and nowhere else.

Sources (cited by page title and section):

* "HyperQwen: 1,000 tok/s on a Single RTX 3090 Through Aggressive
  Recurrent-State Speculation" (starlog), section "Technical Insight": the
  DeltaNet recurrent state grows with the verify-block width (per-position
  state copies), fp16 DeltaNet state, and recurrent-state checkpoints for
  prefix caching.
* "Qwen3.8-27B on a Single RTX 3090: How Calibrated Quantization and
  Speculative Decoding Hit 1,000 tok/s" (starlog), section "Technical
  Insight": greedy verification of a draft block (compare logits, keep the
  accepted prefix, discard the rejected drafts).
* "HyperQwen on one RTX 3090: a first-time developer's guide to the 381-token
  claim", section "What actually became faster?": a verify block of up to 16
  tokens; prefix caching of a ~25,000-token document.
* "HyperQwen: 1,000 tok/s ..." (Technical Insight) and "HyperQwen on one RTX 3090
  ..." (What actually became faster?): later verify positions are drafted by copying
  from the request's own context (``context_lookup.py`` states the reading used).
* The pages name DeltaNet but never print its update. The update used here is
  the published gated delta rule (Yang, Kautz and Hatamizadeh, "Gated Delta
  Networks: Improving Mamba2 with Delta Rule", 2024):
  S_t = g_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,  o_t = S_t q_t,
  with S a dv x dk matrix.

Pins: every function here is checked in ``tests/test_oracle_pins.py`` against
closed forms, invariants, hand-worked golden values and brute force, never
against itself. No function is "parity unpinned".
"""

from .recurrence import (  # noqa: F401
    round_to,
    gated_delta_step,
    verify_block,
    commit,
    prefill_checkpoint,
)
from .accept import argmax_lowest, accept_greedy  # noqa: F401
from .context_lookup import context_drafts_row, context_drafts  # noqa: F401

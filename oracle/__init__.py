"""CPU oracle for the fused cascaded-reduction hot path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this
package: only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.  It shares no code with the
CUDA library (``cascaded_reductions_gb300``) and imports nothing from it.

What it computes is the *unfused, multi-pass* definition of each cascade, in
float64 (numpy), exactly as the pages state the stages:

* attention (single-row decode, split-KV decode, causal prefill) --
  safe softmax in three stages (row max, then the exp-sum denominator, then the
  weighted sum with V, divided at the end).  RedFuser episode transcript,
  cue 9 (safe softmax's three stages) and cue 19 (the weighted sum with V).
  Per-segment states and their merge follow cue 21 and cue 39
  (Multi-Segment strategy) and the episode viz page's widget "Merging partial
  states across blocks (FlashDecoding-style)".
* MoE routing -- softmax then top-k (transcript cue 11; "Online normalizer
  calculation for softmax", abstract on its citation page: softmax and top-k
  fused).
* FP8 per-token quantisation then GEMM -- abs-max, scale = absmax / 448, e4m3
  encode, then the GEMM sum (transcript cue 33).
* single-row cascades -- safe softmax of a row, variance, moment of inertia
  (transcript cue 47).
* multi-latent attention decode -- the attention cascade with every query
  head reading one shared latent cache (transcript cues 41 and 55).

Every floating-point step is float64 unless the step itself is a rounding to a
narrower format the method fixes (fp32 scale and fp32 quotient before the e4m3
encode, the e4m3 encode itself).

Parity pins (tests under ``tests/test_oracle_*.py``) tie each function to
something other than itself: the pages' worked example, closed forms, the merge
invariant and identity element, library routines (torch float64 softmax and
scaled-dot-product attention, torch's own float8/bfloat16 casts), the e4m3
definition checked exhaustively, and brute force on tiny inputs.
"""

from . import attention, routing, fp8, bf16, rowcascades, mla  # noqa: F401

"""MoE routing cascade oracle: softmax over experts, then top-k.

Definitions followed:

* RedFuser episode transcript, cue 11 -- MoE routing is softmax followed by
  top-k, a cascade of reductions of the same shape as attention's.
* "Online normalizer calculation for softmax" (citation page, abstract) --
  softmax and top-k computed together from one read of the row.

Readings of points the pages leave open (transcript cue 59 says the text does
not show exactly what is fused for routing):

* the k experts are the k largest probabilities; equal logits are ordered by
  lower expert index first; the output list is sorted by that order;
* with ``renormalize`` the weights are the probabilities renormalised over the
  selected experts, w_i = p_i / sum_{j in sel} p_j; without it they are the
  plain probabilities p_i.

float64 throughout.
"""

import numpy as np


def softmax(x):
    """Row softmax in float64, three passes: max, exp-sum, divide."""
    x = np.asarray(x, dtype=np.float64)
    m = x.max(axis=1, keepdims=True)
    e = np.exp(x - m)
    return e / e.sum(axis=1, keepdims=True)


def softmax_topk(logits, k, renormalize=True):
    """logits [T, E] -> (idx [T, k] int32, w [T, k] float64).

    The ordering key is (-p, expert index): a stable sort on -p keeps equal
    probabilities in index order.  p in float64 is strictly increasing in
    distinct float32 logits, so ordering by p equals ordering by the logits.
    """
    p = softmax(logits)
    order = np.argsort(-p, axis=1, kind="stable")[:, :k]
    sel = np.take_along_axis(p, order, axis=1)
    if renormalize:
        sel = sel / sel.sum(axis=1, keepdims=True)
    return order.astype(np.int32), sel

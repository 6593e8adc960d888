"""MoE routing cascade oracle: softmax over experts, then top-k.

Definitions followed:

* RedFuser episode transcript, cue 11 -- MoE routing is softmax followed by
  top-k, a cascade of reductions of the same shape as attention's.
* "Online normalizer calculation for softmax" (citation page, abstract) --
  softmax and top-k computed together from one read of the row.

Readings of points the pages leave open (transcript cue 59 says the text does
not show exactly what is fused for routing):

* the k experts are the k largest logits (so the k largest probabilities),
  listed in descending order of logit; equal logits are ordered by lower
  expert index first;
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

    The ordering key is (-logit, expert index), taken on the logits widened
    exactly to float64: a stable sort on -x keeps equal logits in index
    order (and -0 equal to +0).  The key is the logit itself, not p:
    exp(x - m) underflows to zero (or to equal subnormals) once a logit lies
    more than about 745 below the row maximum, and such experts must still
    be ordered by their logits.  Where p does not underflow the two orders
    agree, since exp is increasing.
    """
    x = np.asarray(logits, dtype=np.float64)
    p = softmax(x)
    order = np.argsort(-x, axis=1, kind="stable")[:, :k]
    sel = np.take_along_axis(p, order, axis=1)
    if renormalize:
        sel = sel / sel.sum(axis=1, keepdims=True)
    return order.astype(np.int32), sel

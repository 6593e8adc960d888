"""Attention cascade oracle: safe softmax then the weighted sum with V.

Definitions followed (page titles and their sections):

* RedFuser episode transcript, cue 9 -- safe softmax is three dependent
  stages: the row max m, the sum of exp(x - m), then the divide.
* Transcript cue 19 -- the second reduction is the weighted sum
  sum_j exp(x_j - m) * v_j, divided by the denominator once at the end.
* Transcript cue 21 and the episode viz page's widget "Merging partial states
  across blocks (FlashDecoding-style)" -- two partial states, each relative to
  its own max, combine by rescaling to the larger max.
* Transcript cue 39 -- Multi-Segment: the key sequence is split into segments
  whose partial states are merged.
* Transcript cue 27/29 -- the state monoid has an identity element; a segment
  with no keys carries that identity, (m, l, acc) = (-inf, 0, 0).

Readings of points the pages leave open:

* scores are s_j = scale * <q, k_j>; the exponential base is e, so ``m`` and
  ``lse`` are in natural-log units;
* segments are contiguous blocks of ceil(L / S) keys: segment s holds keys
  [s*c, min(L, (s+1)*c)), c = ceil(L/S); a segment past the end is empty;
* causal prefill is top-left aligned: query i sees keys 0..i (equal query and
  key lengths).

Everything accumulates in float64.  Inputs are float64 arrays holding the exact
values of the fp32/bf16 inputs (widening is exact).
"""

import math

import numpy as np


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def softmax_v(q, K, V, scale):
    """Single query row, unfused multi-pass definition.

    q: [D], K: [L, D], V: [L, Dv]  ->  (out [Dv], m, l)
    pass 1 scores, pass 2 max, pass 3 denominator, pass 4 weighted sum / l.
    """
    q, K, V = _f64(q), _f64(K), _f64(V)
    s = scale * (K @ q)                 # pass 1: the contraction over D
    m = s.max()                         # pass 2: reduction 1 (max)
    e = np.exp(s - m)
    l = e.sum()                         # pass 3: reduction 2 (sum of exp)
    out = (e @ V) / l                   # pass 4: reduction 3 (weighted sum), one divide
    return out, m, l


def softmax_v_rows(q, K, V, scale):
    """Many independent rows: q [R, D], K [R, L, D], V [R, L, Dv].

    Returns out [R, Dv], m [R], l [R] (same four passes, batched over rows).
    """
    q, K, V = _f64(q), _f64(K), _f64(V)
    s = scale * np.einsum("rld,rd->rl", K, q)
    m = s.max(axis=1)
    e = np.exp(s - m[:, None])
    l = e.sum(axis=1)
    out = np.einsum("rl,rld->rd", e, V) / l[:, None]
    return out, m, l


def segment_bounds(L, S):
    """Contiguous split of L keys into S segments of ceil(L/S) keys each."""
    c = -(-L // S) if L > 0 else 0
    return [(min(L, s * c), min(L, (s + 1) * c)) for s in range(S)]


def segment_states(q, K, V, scale, S):
    """Per-segment unnormalised states for many rows, by definition.

    For each row and each segment [a, b): m_s = max of the segment's scores,
    l_s = sum exp(s_j - m_s), acc_s = sum exp(s_j - m_s) * v_j.  An empty
    segment gives the identity state (-inf, 0, 0).

    q [R, D], K [R, L, D], V [R, L, Dv] -> m [R, S], l [R, S], acc [R, S, Dv]
    """
    q, K, V = _f64(q), _f64(K), _f64(V)
    R, L, _ = K.shape
    Dv = V.shape[2]
    m = np.full((R, S), -np.inf)
    l = np.zeros((R, S))
    acc = np.zeros((R, S, Dv))
    s_all = scale * np.einsum("rld,rd->rl", K, q) if L > 0 else np.zeros((R, 0))
    for s, (a, b) in enumerate(segment_bounds(L, S)):
        if b <= a:
            continue
        sc = s_all[:, a:b]
        ms = sc.max(axis=1)
        e = np.exp(sc - ms[:, None])
        m[:, s] = ms
        l[:, s] = e.sum(axis=1)
        acc[:, s, :] = np.einsum("rl,rld->rd", e, V[:, a:b, :])
    return m, l, acc


def merge_states(m, l, acc):
    """Combine S partial states per row into the final output.

    M = max_s m_s; each state is rescaled by exp(m_s - M) (taken as 0 for an
    identity state, m_s = -inf); l = sum of rescaled l_s, acc likewise;
    out = acc / l; lse = M + ln(l).

    m [R, S], l [R, S], acc [R, S, Dv] -> out [R, Dv], lse [R]
    """
    m, l, acc = _f64(m), _f64(l), _f64(acc)
    M = m.max(axis=1)
    w = np.zeros_like(m)
    live = np.isfinite(m)
    Mb = np.broadcast_to(M[:, None], m.shape)
    w[live] = np.exp(m[live] - Mb[live])
    L_tot = (w * l).sum(axis=1)
    A = np.einsum("rs,rsd->rd", w, acc)
    out = A / L_tot[:, None]
    lse = M + np.log(L_tot)
    return out, lse


def causal_attention(Q, K, V, scale, causal=True):
    """Prefill attention for one (batch, head): Q, K, V [N, D] -> out [N, D], lse [N].

    Four passes per row as in ``softmax_v``; with ``causal`` row i only sees
    keys 0..i (top-left aligned mask).
    """
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    N = Q.shape[0]
    s = scale * (Q @ K.T)                               # pass 1
    if causal:
        mask = np.tril(np.ones((N, K.shape[0]), dtype=bool))
        s = np.where(mask, s, -np.inf)
    m = s.max(axis=1)                                   # pass 2
    e = np.exp(s - m[:, None])
    l = e.sum(axis=1)                                   # pass 3
    out = (e @ V) / l[:, None]                          # pass 4
    return out, m + np.log(l)


def causal_attention_row(q, K, V, scale, i, causal=True):
    """One query row i of prefill attention (for sampled checks at full size)."""
    n = i + 1 if causal else K.shape[0]
    out, m, l = softmax_v(q, _f64(K)[:n], _f64(V)[:n], scale)
    return out, m + math.log(l)

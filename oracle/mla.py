"""Multi-latent attention (MLA) decode oracle.

TEST INFRASTRUCTURE ONLY (see the package header).

What the pages give: the RedFuser episode transcript names multi-latent
attention as one of the four evaluated workloads and reports the generated
MLA kernel within 2 percent of DeepSeek's FlashMLA on an H800 (cue 41), a
comparison made on decode shapes with one query row (cue 55); decode splits
the key sequence into segments whose partial states are merged (cue 39).
The pages give no formulas or shapes for MLA itself.

Reading taken (the plainest one consistent with "DeepSeek's FlashMLA" on
decode shapes): the cascade is ordinary safe-softmax attention in which every
query head of a sequence reads ONE shared latent cache C [L, Dk]:

    s_hj = scale * <q_h, c_j>            (q_h [Dk], c_j [Dk])
    p_hj = softmax_j(s_hj)               (max, then exp-sum, then divide)
    o_h  = sum_j p_hj * c_j[:Dv]         (the value is the first Dv latent dims)

with Dk = 576 = 512 latent dims + 64 rotary dims and Dv = 512 (DeepSeek-V2's
compressed-KV layout with the key/value up-projections absorbed into the
query and the output).  The softmax scale is a parameter.

Segments follow ``attention.segment_bounds`` (contiguous blocks of ceil(L/S)
keys) and the per-segment states are the same (m, l, acc) as for ordinary
split-KV decode, so ``attention.merge_states`` merges them.

Everything accumulates in float64.
"""

import numpy as np

from .attention import segment_bounds


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def mla_decode(q, C, dv, scale):
    """q [B, H, Dk], C [B, L, Dk] -> (out [B, H, dv], m [B, H], l [B, H]).

    Unfused multi-pass definition: pass 1 scores against the shared latent
    rows, pass 2 max, pass 3 exp-sum, pass 4 weighted sum of the first dv
    latent dims, divided once.
    """
    q, C = _f64(q), _f64(C)
    s = scale * np.einsum("bhd,bld->bhl", q, C)        # pass 1
    m = s.max(axis=2)                                   # pass 2
    e = np.exp(s - m[:, :, None])
    l = e.sum(axis=2)                                   # pass 3
    out = np.einsum("bhl,blv->bhv", e, C[:, :, :dv]) / l[:, :, None]   # pass 4
    return out, m, l


def mla_segment_states(q, C, dv, scale, S):
    """Per-segment states: m [B, H, S], l [B, H, S], acc [B, H, S, dv].

    For every sequence, head and segment [a, b): m = max score of the segment,
    l = sum exp(s - m), acc = sum exp(s - m) c[:dv]; an empty segment is the
    identity (-inf, 0, 0).
    """
    q, C = _f64(q), _f64(C)
    B, H, _ = q.shape
    L = C.shape[1]
    m = np.full((B, H, S), -np.inf)
    l = np.zeros((B, H, S))
    acc = np.zeros((B, H, S, dv))
    s_all = scale * np.einsum("bhd,bld->bhl", q, C)
    for s, (a, b) in enumerate(segment_bounds(L, S)):
        if b <= a:
            continue
        sc = s_all[:, :, a:b]
        ms = sc.max(axis=2)
        e = np.exp(sc - ms[:, :, None])
        m[:, :, s] = ms
        l[:, :, s] = e.sum(axis=2)
        acc[:, :, s, :] = np.einsum("bhl,blv->bhv", e, C[:, a:b, :dv])
    return m, l, acc

"""Parity of rf_softmax_topk with the oracle through the C ABI.

Indices bit-exact (ties by lower expert index), weights within the fp32
tolerance.  Both routing workloads at full size ([16384 x 256] top-8 and
[65536 x 64] top-2, element by element), plus edge cases: constructed ties,
E = 2 with k = 1, E not a multiple of 4, k = E, k = 32, E = 1024, T = 1,
and renormalize off.
"""

import numpy as np
import pytest
import torch

from helpers import assert_close_f32
from oracle import routing as Rt
import synthetic_inputs as si

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rf():
    import cascaded_reductions_gb300 as m
    return m


def check(rf, x, k, renorm, what):
    idx, w = rf.softmax_topk(x.cuda(), k, renorm)
    torch.cuda.synchronize()
    ridx, rw = Rt.softmax_topk(x.numpy(), k, renorm)
    gi = idx.cpu().numpy()
    bad = np.argwhere(gi != ridx)
    assert bad.size == 0, f"{what}: {len(bad)} index mismatches, first {bad[0]}: {gi[bad[0][0]]} vs {ridx[bad[0][0]]}"
    assert_close_f32(w.cpu().numpy(), rw, what)


@pytest.mark.parametrize("name", ["route_256", "route_64"])
def test_full_size(rf, name):
    cfg = si.FULL[name]
    x = si.routing_logits(cfg["T"], cfg["E"], seed=si.SEEDS[name])
    check(rf, x, cfg["k"], True, name)


@pytest.mark.parametrize("E,k", [(2, 1), (2, 2), (3, 2), (33, 5), (64, 16), (64, 17), (100, 32),
                                 (128, 8), (130, 3), (256, 32), (511, 9), (1024, 32), (1024, 1)])
@pytest.mark.parametrize("renorm", [True, False])
def test_shapes(rf, E, k, renorm):
    x = si.routing_logits(37, E, seed=E * 7 + k)
    check(rf, x, k, renorm, f"E={E} k={k}")


def test_ties_lower_index_first(rf):
    T, E = 64, 256
    g = torch.Generator().manual_seed(9)
    # few distinct values -> many exact ties, including at the k-th place
    x = torch.randint(-3, 4, (T, E), generator=g).float()
    x[5] = 0.0
    check(rf, x, 8, True, "ties")
    x2 = torch.randint(0, 2, (T, 64), generator=g).float()
    check(rf, x2, 2, False, "ties E=64")


def test_single_token(rf):
    x = si.routing_logits(1, 256, seed=1)
    check(rf, x, 8, True, "T=1")


@pytest.mark.parametrize("E,k", [(64, 1), (64, 3), (64, 4), (60, 4), (61, 2), (64, 8), (47, 6),
                                 (128, 16), (120, 9), (256, 1), (256, 5), (200, 8), (253, 8)])
def test_merge_shapes(rf, E, k):
    x = si.routing_logits(301, E, seed=E * 13 + k)
    check(rf, x, k, True, f"E={E} k={k}")
    check(rf, x, k, False, f"E={E} k={k} no renorm")


@pytest.mark.parametrize("E,k", [(256, 8), (64, 2), (64, 4), (128, 16)])
def test_top_values_in_one_lane(rf, E, k):
    # every one of the k largest logits sits in the slots of one lane, so that
    # lane wins round after round and must rescan its untaken slots
    T = 96
    x = si.routing_logits(T, E, seed=5)
    G, W = {256: 32, 64: 4 if k <= 4 else 8, 128: 16}[E], 4
    nv = E // G
    for t in range(T):
        lane = t % G
        slots = [(i // W) * G * W + lane * W + (i % W) for i in range(nv)]
        for j, e in enumerate(slots[:k]):
            x[t, e] = 50.0 - j if t % 2 else 50.0 - (k - 1 - j)   # both orders
    check(rf, x, k, True, f"one-lane E={E} k={k}")


def test_neg_inf_logits(rf):
    x = si.routing_logits(64, 256, seed=6)
    x[:, ::3] = -float("inf")
    x[7, :] = -float("inf")
    x[7, 200] = 1.0       # one finite logit: the rest are -inf ties, lower index first
    check(rf, x, 8, True, "-inf logits")


@pytest.mark.parametrize("E,k", [(256, 8), (64, 2), (64, 4), (128, 8), (1024, 32)])
def test_masked_experts_far_below_the_max(rf, E, k):
    # masked experts at large finite negatives (their probabilities underflow
    # to zero), mixed with exact ties among the live ones and among the
    # masked ones: the order must still follow the logits
    T = 256
    g = torch.Generator().manual_seed(E + k)
    x = torch.randint(-2, 3, (T, E), generator=g).float()
    mask = torch.rand((T, E), generator=g) < 0.6
    fill = torch.tensor([-1e4, -3e38, -900.0, -800.0])[torch.randint(0, 4, (T, E), generator=g)]
    x = torch.where(mask, fill, x)
    x[3, :] = -1e4                       # every logit masked: all ties
    x[4, :] = -3e38
    x[4, E - 1] = -1e4                    # one survivor, the rest tied far below
    x[5, :] = torch.where(torch.arange(E) % 2 == 0, -900.0, -800.0)
    x[6, :k + 1] = 3.0                    # the k-th place decided by a tie among the live
    check(rf, x, k, True, f"masked E={E} k={k}")
    check(rf, x, k, False, f"masked E={E} k={k} no renorm")


@pytest.mark.parametrize("E", [32, 64, 96, 128])
@pytest.mark.parametrize("k", [1, 2])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 1000])
def test_one_thread_per_token_shapes(rf, E, k, T):
    # k <= 2 with E a multiple of 32 up to 128: one thread per token over a
    # row staged in shared memory; T around the 64-token block (ragged tails)
    x = si.routing_logits(T, E, seed=1000 * E + 10 * k + T)
    check(rf, x, k, True, f"E={E} k={k} T={T}")
    check(rf, x, k, False, f"E={E} k={k} T={T} no renorm")


@pytest.mark.parametrize("E", [32, 64, 128])
def test_one_thread_per_token_ties_and_order(rf, E):
    T = 200
    g = torch.Generator().manual_seed(E)
    x = torch.randint(-2, 3, (T, E), generator=g).float()   # ties everywhere
    x[0, :] = 1.0                                          # all tied: experts 0, 1
    x[1, :] = -1e4
    x[1, E - 1] = 5.0
    x[1, E - 2] = 5.0                                      # the two best tie at the end
    x[2, :] = torch.arange(E, dtype=torch.float32)         # increasing: E-1, E-2
    x[3, :] = -torch.arange(E, dtype=torch.float32)        # decreasing: 0, 1
    x[4, :] = 0.0
    x[4, 5] = -0.0                                         # -0 ties with +0
    for k in (1, 2):
        check(rf, x, k, True, f"ties E={E} k={k}")
        check(rf, x, k, False, f"ties E={E} k={k} no renorm")


@pytest.mark.parametrize("k", [1, 2, 3, 5, 7, 8])
@pytest.mark.parametrize("T", [1, 15, 16, 17, 1000])
def test_two_threads_per_token_shapes(rf, k, T):
    # E = 256, k <= 8: two threads per token over a staged row; T around the
    # 16-token block (ragged tails), renormalisation on and off
    x = si.routing_logits(T, 256, seed=500 + 10 * k + T)
    check(rf, x, k, True, f"E=256 k={k} T={T}")
    check(rf, x, k, False, f"E=256 k={k} T={T} no renorm")


def test_two_threads_per_token_structure(rf):
    T, E = 64, 256
    x = si.routing_logits(T, E, seed=77)
    x[0, :] = 0.5                             # every value a candidate, all tied
    x[1, 128:] += 40.0                        # the top 8 all in the second half
    x[2, :128] += 40.0                        # ... all in the first half
    x[3, :] = -float("inf")
    x[3, 5] = 2.0                             # one finite value, the rest -inf ties
    x[4, :] = -float("inf")
    x[4, 200:203] = 1.0                       # three finite, ties among the -inf after them
    x[5, ::2] = -float("inf")                 # half the row at -inf
    x[6, 127] = x[6, 128] = 30.0              # a tie across the two halves
    x[7, 0] = x[7, 255] = 30.0
    for k in (1, 4, 8):
        check(rf, x, k, True, f"structure k={k}")
        check(rf, x, k, False, f"structure k={k} no renorm")

"""Single-row cascade oracles: safe softmax of a row, variance, moment of
inertia, layer normalisation, RMS normalisation.

RedFuser episode transcript, cue 47: the paper measures safe softmax on rows
of 1K to 8K elements at several fusion levels, and also runs variance and
moment of inertia.  Each is a cascade: the second reduction needs the first
one's finished result (cue 9 for softmax: max, then sum of exp(x - max), then
the divide).  The oracle writes each out as its unfused multi-pass definition
in float64.

Readings (the pages give names, no formulas, for the last two):

* variance is the population variance of the row: mean = sum x / n, then
  var = sum (x - mean)^2 / n (the second reduction needs the first's mean);
* moment of inertia of a row of point masses m_i at positions r_i in R^3 is
  taken about the centre of mass: c = sum m_i r_i / sum m_i, then
  I = sum m_i |r_i - c|^2 (the second reduction needs the first's c).
  Positions are stored coordinate-major per row: pos[row, axis, i].
"""

import numpy as np


def row_softmax(x):
    """x [R, n] -> y [R, n]: pass 1 max, pass 2 sum of exp(x - max), pass 3 divide."""
    x = np.asarray(x, dtype=np.float64)
    m = x.max(axis=1, keepdims=True)
    e = np.exp(x - m)
    return e / e.sum(axis=1, keepdims=True)


def row_variance(x):
    """x [R, n] -> (mean [R], var [R]): pass 1 mean, pass 2 mean of squared deviations."""
    x = np.asarray(x, dtype=np.float64)
    mean = x.sum(axis=1) / x.shape[1]
    var = ((x - mean[:, None]) ** 2).sum(axis=1) / x.shape[1]
    return mean, var


def moment_of_inertia(mass, pos):
    """mass [R, n], pos [R, 3, n] -> (center [R, 3], inertia [R]).

    Pass 1: total mass and the mass-weighted position sum, c = sum m r / sum m.
    Pass 2: I = sum m |r - c|^2.
    """
    m = np.asarray(mass, dtype=np.float64)
    p = np.asarray(pos, dtype=np.float64)
    M = m.sum(axis=1)
    c = np.einsum("rn,rdn->rd", m, p) / M[:, None]
    d = p - c[:, :, None]
    inertia = np.einsum("rn,rdn->r", m, d * d)
    return c, inertia


def layer_norm(x, gamma, beta, eps):
    """x [R, n], gamma/beta [n] -> y [R, n].

    Pass 1: mean; pass 2: population variance; pass 3: y = (x - mean) /
    sqrt(var + eps) * gamma + beta (bookshelf explainer, "Problem":
    normalisation layers are cascaded reductions).
    """
    x = np.asarray(x, dtype=np.float64)
    mean, var = row_variance(x)
    return ((x - mean[:, None]) / np.sqrt(var[:, None] + eps) * np.asarray(gamma, np.float64)
            + np.asarray(beta, np.float64))


def rms_norm(x, gamma, eps):
    """x [R, n], gamma [n] -> y [R, n].

    Pass 1: the mean of squares ms = sum x^2 / n; pass 2: y = x / sqrt(ms +
    eps) * gamma (the normalisation needs the finished reduction; bookshelf
    explainer, "Problem": normalisation layers are cascaded reductions).
    """
    x = np.asarray(x, dtype=np.float64)
    ms = (x * x).sum(axis=1) / x.shape[1]
    return x / np.sqrt(ms[:, None] + eps) * np.asarray(gamma, np.float64)

"""Elementary operators of the block, float64 numpy (oracle; test infrastructure only).

None of these is printed on the Oases pages; each is the textbook definition of
the layer, written out:
  * LayerNorm over the hidden dimension with biased variance:
      u = (x - mean) / sqrt(var + eps) * gamma + beta.
    Pinned: rows of u have mean 0 and variance var/(var+eps) when gamma=1,
    beta=0; finite differences pin the backward.
  * GeLU, exact erf form: gelu(a) = a * Phi(a), Phi the standard normal CDF;
    gelu'(a) = Phi(a) + a * phi(a).  Pinned: gelu(0)=0, gelu'(0)=1/2,
    gelu(1)=Phi(1) (normal-table value), finite differences.
  * One attention head: O = softmax(Q K^T / sqrt(d) + mask) V with the causal
    mask (key j visible from query i iff j <= i).  Pinned: one-token sequence
    gives O = V, row 0 of a causal head is V[0], Q = 0 gives running means of V,
    finite differences pin the backward.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf

_SQRT2 = math.sqrt(2.0)
_INV_SQRT_2PI = 1.0 / math.sqrt(2.0 * math.pi)


def layer_norm(x: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float):
    """Row LayerNorm.  Returns (u, mean, rstd); mean and rstd have one entry per row."""
    mean = x.mean(axis=1)
    xc = x - mean[:, None]
    var = (xc * xc).mean(axis=1)
    rstd = 1.0 / np.sqrt(var + eps)
    u = xc * rstd[:, None] * gamma[None, :] + beta[None, :]
    return u, mean, rstd


def layer_norm_backward(du, x, mean, rstd, gamma):
    """Backward of ``layer_norm``.  Returns (dx, dgamma, dbeta).

    With xhat = (x - mean) * rstd and g = du * gamma:
      dx = rstd * (g - mean_row(g) - xhat * mean_row(g * xhat)),
      dgamma = sum_rows(du * xhat), dbeta = sum_rows(du).
    """
    xhat = (x - mean[:, None]) * rstd[:, None]
    gh = du * gamma[None, :]
    dx = rstd[:, None] * (gh - gh.mean(axis=1, keepdims=True)
                          - xhat * (gh * xhat).mean(axis=1, keepdims=True))
    return dx, (du * xhat).sum(axis=0), du.sum(axis=0)


def normal_cdf(a):
    return 0.5 * (1.0 + erf(a / _SQRT2))


def gelu(a):
    """gelu(a) = a * Phi(a) (exact erf form)."""
    return a * normal_cdf(a)


def gelu_grad(a):
    """d gelu / da = Phi(a) + a * phi(a), phi the standard normal density."""
    return normal_cdf(a) + a * _INV_SQRT_2PI * np.exp(-0.5 * a * a)


def attention_head(q: np.ndarray, k: np.ndarray, v: np.ndarray, causal: bool):
    """One head of one sequence: q, k, v are [S, d].  Returns (O [S, d], P [S, S])."""
    S, d = q.shape
    s = (q @ k.T) * (1.0 / math.sqrt(d))
    if causal:
        s = np.where(np.tril(np.ones((S, S), dtype=bool)), s, -np.inf)
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=1, keepdims=True)
    return p @ v, p


def attention_head_backward(do, q, k, v, p):
    """Backward of ``attention_head`` given its probabilities P.  Returns (dq, dk, dv).

    dV = P^T dO;  dP = dO V^T;  dS = P * (dP - rowsum(dP * P));
    dQ = dS K / sqrt(d);  dK = dS^T Q / sqrt(d).
    """
    d = q.shape[1]
    scale = 1.0 / math.sqrt(d)
    dv = p.T @ do
    dp = do @ v.T
    ds = p * (dp - (dp * p).sum(axis=1, keepdims=True))
    return (ds @ k) * scale, (ds.T @ q) * scale, dv

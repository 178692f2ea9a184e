"""Literal matrix forms of one EFLA token and one DeltaNet token -- TEST INFRASTRUCTURE ONLY.

These build the d x d matrices the pages write down and multiply them, with no
rearrangement, so that the factored C oracle can be checked against the
formula as printed.  Small d only (O(d^3) per token).
"""
from __future__ import annotations

import math

import numpy as np


def efla_gate_literal(beta: float, lam: float) -> float:
    """alpha = (1 - e^{-beta*lam}) / lam exactly as printed.

    ["Exact Flow Linear Attention" (gist.science), Metodologia 3;
     "Error-Free Linear Attention is a Free Lunch" (howistudyai), Step 1.]
    Uses exp, not expm1, so that it is an independent evaluation; valid away
    from lam == 0 where the printed quotient is defined.
    """
    return (1.0 - math.exp(-beta * lam)) / lam


def efla_step_literal(S: np.ndarray, q: np.ndarray, k: np.ndarray, v: np.ndarray, beta: float):
    """S_t = (I - alpha k k^T) S_{t-1} + alpha k v^T;  o_t = S_t^T q_t.

    [gist.science, Metodologia 3; howistudyai, Steps 2-3.]
    """
    k = np.asarray(k, dtype=np.float64)
    lam = float(k @ k)
    a = efla_gate_literal(beta, lam)
    d = k.shape[0]
    S_new = (np.eye(d) - a * np.outer(k, k)) @ S + a * np.outer(k, v)
    return S_new.T @ q, S_new


def deltanet_step_literal(S: np.ndarray, q: np.ndarray, k: np.ndarray, v: np.ndarray, beta: float):
    """Euler (delta-rule) step S <- (I - beta k k^T) S + beta k v^T; o = S^T q.

    ["Error-Free Linear Attention is a Free Lunch" (howistudyai), "Delta Rule
     (Linear Attention as Online Learning)"; the page calls it the explicit Euler
     step of the same ODE.]
    """
    d = k.shape[0]
    S_new = (np.eye(d) - beta * np.outer(k, k)) @ S + beta * np.outer(k, v)
    return S_new.T @ q, S_new


def run_literal(step, S0, q, k, v, beta):
    """Apply ``step`` token by token to one head: q,k [T,dk]; v [T,dv]; beta [T]."""
    S = np.array(S0, dtype=np.float64, copy=True)
    outs = []
    for t in range(q.shape[0]):
        o, S = step(S, q[t], k[t], v[t], float(beta[t]))
        outs.append(o)
    return np.stack(outs) if outs else np.zeros((0, S.shape[1])), S

"""Brute-force numerics for pinning the EFLA closed form -- TEST INFRASTRUCTURE ONLY.

The pages obtain the EFLA update as the exact solution, over one token window
of length beta, of the zero-order-hold ODE

    dS/dt = -A S + F,   A = k k^T,   F = k v^T

["Exact Flow Linear Attention" (gist.science), Metodologia 1;
 "Error-Free Linear Attention is a Free Lunch" (howistudyai), "The Concept
 (EFLA)" recipe steps 1-3].  These routines solve that ODE without the rank-1
closed form, so that the closed form can be checked against them:

* ``expm_taylor``: truncated Taylor series with scaling and squaring.
* ``zoh_exact_step``: the Van Loan block exponential (C. F. Van Loan, "Computing
  integrals involving the matrix exponential", IEEE TAC 23(3), 1978):
  exp(beta [[-A, F], [0, 0]]) = [[e^{-beta A}, int_0^beta e^{-(beta-s) A} F ds], [0, I]].
* ``rk4_step``: classical fourth-order Runge-Kutta with n substeps.
"""
from __future__ import annotations

import numpy as np


def expm_taylor(M: np.ndarray, terms: int = 40) -> np.ndarray:
    """exp(M) by scaling and squaring a truncated Taylor series (fp64)."""
    M = np.asarray(M, dtype=np.float64)
    norm = np.linalg.norm(M, 1)
    s = 0
    while norm / (2 ** s) > 0.25:
        s += 1
    X = M / (2 ** s)
    n = M.shape[0]
    E = np.eye(n)
    term = np.eye(n)
    for j in range(1, terms + 1):
        term = term @ X / j
        E = E + term
    for _ in range(s):
        E = E @ E
    return E


def zoh_exact_step(S: np.ndarray, k: np.ndarray, v: np.ndarray, beta: float, expm=expm_taylor):
    """Exact ODE solution over [0, beta] from S by the Van Loan block exponential."""
    dk, dv = k.shape[0], v.shape[0]
    Z = np.zeros((dk + dv, dk + dv))
    Z[:dk, :dk] = -np.outer(k, k)
    Z[:dk, dk:] = np.outer(k, v)
    E = expm(beta * Z)
    return E[:dk, :dk] @ S + E[:dk, dk:]


def rk4_step(S: np.ndarray, k: np.ndarray, v: np.ndarray, beta: float, n: int) -> np.ndarray:
    """Integrate dS/dt = -k k^T S + k v^T over [0, beta] with n RK4 substeps."""
    A = np.outer(k, k)
    F = np.outer(k, v)

    def f(X):
        return -A @ X + F

    h = beta / n
    X = np.array(S, dtype=np.float64, copy=True)
    for _ in range(n):
        k1 = f(X)
        k2 = f(X + 0.5 * h * k1)
        k3 = f(X + 0.5 * h * k2)
        k4 = f(X + h * k3)
        X = X + (h / 6.0) * (k1 + 2 * k2 + 2 * k3 + k4)
    return X

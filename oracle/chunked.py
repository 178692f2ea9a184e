"""Chunkwise (WY/UT) evaluation of the EFLA recurrence in fp64 -- TEST INFRASTRUCTURE ONLY.

The pages state that EFLA keeps the rank-1 algebraic form of the delta rule and
therefore its hardware-efficient WY/UT chunkwise parallel form
["Exact Flow Linear Attention" (gist.science), Metodologia 3;
 "Error-Free Linear Attention is a Free Lunch" (howistudyai), Step 4].  They do
not write the chunk equations out; this module derives them from the update
rule and evaluates them plainly, one chunk after another.

Derivation, for one chunk of C tokens starting from state S0 (dk x dv).
Write the per-token update as S_t = S_{t-1} + k_t u_t^T with
u_t^T = alpha_t (v_t^T - k_t^T S_{t-1}).  Unrolling S_{t-1} = S0 + sum_{i<t} k_i u_i^T:

    u_t + alpha_t sum_{i<t} (k_t . k_i) u_i = alpha_t v_t - alpha_t S0^T k_t

so with A = strictly-lower(diag(alpha) K K^T) and T = (I + A)^{-1}:

    U  = T diag(alpha) V - T diag(alpha) K S0 = U~ - W S0
    S_C = S0 + K^T U
    O  = Q S0 + (Q K^T o M) U          (M lower-triangular INCLUDING the diagonal,
                                        because o_t reads S_t, the updated state)

The last chunk of a sequence may be shorter than C.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


def _alpha_vec(beta: np.ndarray, lam: np.ndarray) -> np.ndarray:
    a = np.empty_like(lam)
    pos = lam > 0
    a[pos] = -np.expm1(-beta[pos] * lam[pos]) / lam[pos]
    a[~pos] = beta[~pos]
    return a


def chunk_step(S0, Q, K, V, beta):
    """One chunk: Q,K [c,dk], V [c,dv], beta [c], S0 [dk,dv] -> (O [c,dv], S_C)."""
    c = K.shape[0]
    lam = np.einsum("ti,ti->t", K, K)
    a = _alpha_vec(beta, lam)
    A = np.tril(a[:, None] * (K @ K.T), -1)
    I = np.eye(c)
    # T = (I + A)^{-1}; applied through a unit lower-triangular solve
    W = solve_triangular(I + A, a[:, None] * K, lower=True, unit_diagonal=True)
    Ut = solve_triangular(I + A, a[:, None] * V, lower=True, unit_diagonal=True)
    U = Ut - W @ S0
    M = np.tril(np.ones((c, c)))
    O = Q @ S0 + ((Q @ K.T) * M) @ U
    S_C = S0 + K.T @ U
    return O, S_C


def fwd_head(S0, q, k, v, beta, chunk: int):
    """One head, one sequence: q,k [T,dk]; v [T,dv]; beta [T]."""
    T = q.shape[0]
    S = np.array(S0, dtype=np.float64, copy=True)
    O = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, chunk):
        c1 = min(T, c0 + chunk)
        O[c0:c1], S = chunk_step(S, q[c0:c1], k[c0:c1], v[c0:c1], beta[c0:c1])
    return O, S


def fwd(q, k, v, beta, S0=None, cu_seqlens=None, *, chunk: int = 64):
    """Chunked fp64 forward with the layouts of ``oracle.fwd``."""
    q, k, v, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, beta))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is None:
        bounds = [(b, 0, T) for b in range(B)]
    else:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        bounds = [(0, int(cu[n]), int(cu[n + 1])) for n in range(cu.shape[0] - 1)]
    N = len(bounds)
    o = np.zeros((B, T, H, dv))
    S_T = np.zeros((N, H, dk, dv))
    for n, (b, t0, t1) in enumerate(bounds):
        for h in range(H):
            s0 = np.zeros((dk, dv)) if S0 is None else np.asarray(S0, dtype=np.float64)[n, h]
            o[b, t0:t1, h], S_T[n, h] = fwd_head(s0, q[b, t0:t1, h], k[b, t0:t1, h],
                                                 v[b, t0:t1, h], beta[b, t0:t1, h], chunk)
    return o, S_T

"""EFLA oracle -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct CPU implementations of what the EFLA token
mixer computes, used to check the CUDA path.  Only ``tests/``, the smoke
entry point and the CPU-baseline leg of ``bench.py`` may import this package;
the library in ``exact_delta_rule_gb300`` never does, and the two share no
code.

Contents:

* ``fwd`` / ``decode_step`` -- the sequential recurrence in fp64 (plain C in
  ``efla_oracle.c``, loaded with ctypes):
  lam = ||k||^2, alpha = -expm1(-beta*lam)/lam, S <- (I - alpha k k^T) S + alpha k v^T,
  o = S^T q with the updated S.
  ["Exact Flow Linear Attention" (gist.science), Metodologia 2-3;
   "Error-Free Linear Attention is a Free Lunch" (howistudyai), Steps 1-3.]
* ``alpha`` -- the gate alone (same C function).
* ``literal`` -- the update written with explicit d x d matrices (numpy), and the
  Euler (DeltaNet) step the pages compare against.
* ``chunked`` -- the chunkwise WY/UT evaluation of the same recurrence in fp64
  (numpy), derived from the update rule (the pages only name the technique).
* ``numerics`` -- a brute-force Taylor matrix exponential, the Van Loan block
  exponential for the zero-order-hold input integral, and RK4 on the ODE.

Pins (each checked by ``tests/test_oracle_*.py``, none of them re-types a
formula of this package): the worked example printed on the howistudyai page,
the matrix exponential of the ODE (Van Loan), RK4 convergence, the decay
invariant along k, the small-key (DeltaNet) limit, chunked == sequential,
linearity in (S0, V), orthogonal-key commutation, state hand-off, and varlen
packing == separate calls.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "efla_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

__all__ = ["build", "fwd", "decode_step", "alpha", "max_threads"]


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (-O2, no fast-math, OpenMP over heads)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            lp = ctypes.POINTER(ctypes.c_int64)
            lib.efla_oracle_alpha.restype = ctypes.c_double
            lib.efla_oracle_alpha.argtypes = [ctypes.c_double, ctypes.c_double]
            lib.efla_oracle_fwd_mode.restype = ctypes.c_int
            lib.efla_oracle_fwd_mode.argtypes = [dp, dp, dp, dp, dp, lp, dp, dp] + [ctypes.c_int] * 8
            lib.efla_oracle_decode_mode.restype = ctypes.c_int
            lib.efla_oracle_decode_mode.argtypes = [dp, dp, dp, dp, dp, dp] + [ctypes.c_int] * 6
            lib.efla_oracle_bwd_mode.restype = ctypes.c_int
            lib.efla_oracle_bwd_mode.argtypes = [dp] * 12 + [ctypes.c_int] * 7
            lib.efla_oracle_gate_grad.restype = None
            lib.efla_oracle_gate_grad.argtypes = [ctypes.c_double, ctypes.c_double, ctypes.c_int,
                                                  ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]
            lib.efla_oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor (CPU)
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a, ctype=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def alpha(beta: float, lam: float) -> float:
    """The EFLA gate (1 - exp(-beta*lam))/lam, beta at lam == 0."""
    return _load().efla_oracle_alpha(float(beta), float(lam))


def max_threads() -> int:
    return _load().efla_oracle_max_threads()


_UPDATES = {"exact": 0, "euler": 1}


def fwd(q, k, v, beta, S0=None, cu_seqlens=None, *, threads: int = 0, update: str = "exact"):
    """Sequential fp64 EFLA forward (``update="euler"``: the DeltaNet step, alpha = beta).

    q, k: [B, T, H, dk]; v: [B, T, H, dv]; beta: [B, T, H]; S0: [N, H, dk, dv] or None;
    cu_seqlens: [N+1] or None (then N = B).  Inputs of any float dtype are
    upcast exactly to fp64.  Returns (o [B, T, H, dv], S_T [N, H, dk, dv]) as
    fp64 numpy arrays.  ``threads`` > 0 sets the OpenMP thread count.
    """
    q, k, v, beta, S0 = (_f64(x) for x in (q, k, v, beta, S0))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    cu = None
    if cu_seqlens is not None:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().cpu().numpy()
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
        N = cu.shape[0] - 1
    else:
        N = B
    o = np.zeros((B, T, H, dv), dtype=np.float64)
    S_T = np.zeros((N, H, dk, dv), dtype=np.float64)
    rc = _load().efla_oracle_fwd_mode(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(S0),
                                      _ptr(cu, ctypes.c_int64), _ptr(o), _ptr(S_T),
                                      B, T, H, dk, dv, N, int(threads), _UPDATES[update])
    if rc != 0:
        raise ValueError(f"efla_oracle_fwd failed with code {rc}")
    return o, S_T


def decode_step(q, k, v, beta, S, *, threads: int = 0, update: str = "exact"):
    """One fp64 decode step.  q,k: [B,H,dk]; v: [B,H,dv]; beta: [B,H]; S: [B,H,dk,dv].

    Returns (o [B,H,dv], S_new [B,H,dk,dv]); the input S is not modified.
    """
    q, k, v, beta = (_f64(x) for x in (q, k, v, beta))
    S = _f64(S).copy()
    B, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, H, dv), dtype=np.float64)
    rc = _load().efla_oracle_decode_mode(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(S), _ptr(o),
                                         B, H, dk, dv, int(threads), _UPDATES[update])
    if rc != 0:
        raise ValueError(f"efla_oracle_decode failed with code {rc}")
    return o, S


def gate_grad(beta: float, lam: float, update: str = "exact"):
    """(d alpha / d beta, d alpha / d lam) of the gate (oracle/efla_oracle.c)."""
    a, b = ctypes.c_double(0.0), ctypes.c_double(0.0)
    _load().efla_oracle_gate_grad(float(beta), float(lam), _UPDATES[update], ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def bwd(q, k, v, beta, S0, do, dS_T, *, threads: int = 0, update: str = "exact"):
    """Reverse-mode gradients of ``fwd`` (no cu_seqlens): given do [B,T,H,dv] and dS_T
    [B,H,dk,dv] (or None), returns dict dq, dk [B,T,H,dk], dv [B,T,H,dv], dbeta [B,T,H],
    dS0 [B,H,dk,dv] as fp64 numpy arrays."""
    q, k, v, beta, S0, do, dS_T = (_f64(x) for x in (q, k, v, beta, S0, do, dS_T))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    out = {"dq": np.zeros((B, T, H, dk)), "dk": np.zeros((B, T, H, dk)), "dv": np.zeros((B, T, H, dv)),
           "dbeta": np.zeros((B, T, H)), "dS0": np.zeros((B, H, dk, dv))}
    rc = _load().efla_oracle_bwd_mode(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(S0), _ptr(do), _ptr(dS_T),
                                      _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dbeta"]),
                                      _ptr(out["dS0"]), B, T, H, dk, dv, int(threads), _UPDATES[update])
    if rc != 0:
        raise RuntimeError(f"efla_oracle_bwd_mode failed ({rc})")
    return out

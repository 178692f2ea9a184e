"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: numbers the
howistudyai page prints, the exact ODE solution computed without the rank-1
closed form, RK4 convergence, invariants the pages state, limits, and
brute-force evaluations of the formula as printed.  A dropped term, a wrong
sign, a transposed operand or a read-out of the pre-update state fails at
least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.linalg

import oracle
from oracle import chunked, literal, numerics

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _head(seed, T, dk, dv, key_scale=1.0, beta_lo=0.05, beta_hi=1.0):
    r = _rng(seed)
    q = r.standard_normal((T, dk))
    k = key_scale * r.standard_normal((T, dk)) * r.lognormal(0, 0.5, (T, 1))
    v = r.standard_normal((T, dv))
    beta = r.uniform(beta_lo, beta_hi, T)
    S0 = 0.3 * r.standard_normal((dk, dv))
    return q, k, v, beta, S0


def _fwd1(S0, q, k, v, beta):
    """Oracle forward on a single head given as [T, d] arrays."""
    o, S = oracle.fwd(q[None, :, None, :], k[None, :, None, :], v[None, :, None, :],
                      beta[None, :, None], S0[None, None])
    return o[0, :, 0], S[0, 0]


# ---------------------------------------------------------------- worked example
def test_worked_example_gate_and_write():
    """howistudyai Steps 1-3: k=[1,2], beta=0.2 -> lambda=5, alpha ~ 0.1264."""
    g = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    k = np.array(g["k"])
    lam = float(k @ k)
    assert lam == g["lambda"]
    assert g["beta"] * lam == pytest.approx(g["beta_times_lambda"])
    a = oracle.alpha(g["beta"], lam)
    tol = 0.5 * 10 ** (-g["printed_decimals"])
    assert abs(a - g["alpha"]) <= tol
    assert abs(math.exp(-g["beta"] * lam) - g["exp_minus_beta_lambda"]) <= tol
    assert abs(a * lam - g["one_minus_exp"]) <= tol
    # one token from S_{t-1} = 0: S_t = alpha k v^T (the printed outer product),
    # o_t = S_t^T q with the UPDATED state (a read-out of S_{t-1} would give 0).
    v, q = np.array(g["v"]), np.array(g["q"])
    o, S = oracle.decode_step(q[None, None], k[None, None], v[None, None],
                              np.array([[g["beta"]]]), np.zeros((1, 1, 2, 2)))
    kvT = np.array(g["k_vT"])
    rel = tol / g["alpha"]
    np.testing.assert_allclose(S[0, 0], g["alpha"] * kvT, rtol=rel, atol=0)
    np.testing.assert_allclose(o[0, 0], g["alpha"] * kvT.T @ q, rtol=rel, atol=0)
    assert np.all(np.abs(o[0, 0]) > 0.1)


# ------------------------------------------------------- (1) closed-form exponential
def test_rank1_power_identity_and_taylor_exponential():
    """A^n = lam^{n-1} A and e^{-beta A} = I - alpha A vs a brute-force Taylor series."""
    r = _rng(1)
    for d in (1, 2, 3, 5, 8):
        for _ in range(4):
            k = r.standard_normal(d) * r.lognormal(0, 1.0)
            beta = r.uniform(0.01, 2.0)
            A = np.outer(k, k)
            lam = float(k @ k)
            for n in (2, 3, 5):
                np.testing.assert_allclose(np.linalg.matrix_power(A, n), lam ** (n - 1) * A,
                                           rtol=1e-12, atol=1e-12 * lam ** n)
            a = oracle.alpha(beta, lam)
            E = numerics.expm_taylor(-beta * A)
            np.testing.assert_allclose(np.eye(d) - a * A, E, rtol=0, atol=1e-12)
            np.testing.assert_allclose(scipy.linalg.expm(-beta * A), E, rtol=0, atol=1e-12)


@pytest.mark.parametrize("d", [1, 2, 4, 8])
def test_update_equals_exact_zoh_solution(d):
    """The oracle's step equals e^{-beta A} S + int_0^beta e^{-(beta-s)A} k v^T ds
    computed by the Van Loan block exponential (no rank-1 shortcut)."""
    r = _rng(10 + d)
    for trial in range(6):
        dv = d + trial % 3
        k = r.standard_normal(d) * r.lognormal(0, 0.8)
        v = r.standard_normal(dv)
        q = r.standard_normal(d)
        beta = r.uniform(0.01, 1.5)
        S = r.standard_normal((d, dv))
        for expm in (numerics.expm_taylor, scipy.linalg.expm):
            S_exact = numerics.zoh_exact_step(S, k, v, beta, expm=expm)
            o, S_new = oracle.decode_step(q[None, None], k[None, None], v[None, None],
                                          np.array([[beta]]), S[None, None])
            scale = 1 + np.abs(S_exact).max()
            np.testing.assert_allclose(S_new[0, 0], S_exact, rtol=0, atol=1e-11 * scale)
            np.testing.assert_allclose(o[0, 0], S_exact.T @ q, rtol=0, atol=1e-10 * scale)


# --------------------------------------------------------------------- (2) RK4
def test_update_matches_rk4_with_fourth_order_convergence():
    r = _rng(2)
    d, dv = 6, 5
    k = r.standard_normal(d) * 1.5
    v = r.standard_normal(dv)
    beta = 0.7
    S = r.standard_normal((d, dv))
    lam = float(k @ k)
    assert beta * lam > 5  # stiff enough that Euler would be far off
    _, S_new = oracle.decode_step(np.zeros((1, 1, d)), k[None, None], v[None, None],
                                  np.array([[beta]]), S[None, None])
    S_new = S_new[0, 0]
    errs = []
    for n in (50, 100, 200, 400):
        assert beta / n * lam < 2.78  # RK4 stability bound on the stiff direction
        errs.append(np.abs(numerics.rk4_step(S, k, v, beta, n) - S_new).max())
    for e0, e1 in zip(errs, errs[1:]):
        assert 12.0 < e0 / e1 < 20.0  # ratio 2^4 = 16 for a fourth-order method
    assert np.abs(numerics.rk4_step(S, k, v, beta, 20000) - S_new).max() < 1e-12


def test_rk4_very_stiff_window():
    """beta*lambda ~ 100 (the stiff workload's range): RK4 with h*lambda < 2.78."""
    r = _rng(22)
    d, dv = 4, 3
    k = r.standard_normal(d)
    k = 10.0 * k / np.linalg.norm(k)
    v = r.standard_normal(dv)
    beta = 0.98
    S = r.standard_normal((d, dv))
    _, S_new = oracle.decode_step(np.zeros((1, 1, d)), k[None, None], v[None, None],
                                  np.array([[beta]]), S[None, None])
    S_rk = numerics.rk4_step(S, k, v, beta, 4000)
    np.testing.assert_allclose(S_new[0, 0], S_rk, rtol=0, atol=1e-10)


# ----------------------------------------------------- (3) decay invariant along k
def test_decay_invariant_along_key():
    """k_t^T S_t = e^{-beta lam} k_t^T S_{t-1} + (1 - e^{-beta lam}) v_t^T at every step
    (gist.science "Stabilita Teorica"; howistudyai Step 5)."""
    q, k, v, beta, S0 = _head(3, 40, 7, 5, key_scale=1.3)
    S = S0.copy()
    for t in range(40):
        _, S_new = oracle.decode_step(q[t][None, None], k[t][None, None], v[t][None, None],
                                      np.array([[beta[t]]]), S[None, None])
        S_new = S_new[0, 0]
        lam = float(k[t] @ k[t])
        decay = math.exp(-beta[t] * lam)
        lhs = k[t] @ S_new
        rhs = decay * (k[t] @ S) + (1 - decay) * v[t]
        np.testing.assert_allclose(lhs, rhs, rtol=0, atol=1e-12 * (1 + np.abs(rhs).max()))
        # directions orthogonal to k are untouched
        P = np.eye(7) - np.outer(k[t], k[t]) / lam
        np.testing.assert_allclose(P @ S_new, P @ S, rtol=0, atol=1e-12)
        S = S_new


def test_large_lambda_projection_limit():
    """beta*lam -> infinity: the state along k is replaced, k^T S_t -> v_t^T."""
    r = _rng(33)
    d, dv = 8, 4
    k = r.standard_normal(d)
    k *= 40.0 / np.linalg.norm(k)
    v = r.standard_normal(dv)
    S = r.standard_normal((d, dv))
    _, S_new = oracle.decode_step(np.zeros((1, 1, d)), k[None, None], v[None, None],
                                  np.array([[0.9]]), S[None, None])
    np.testing.assert_allclose(k @ S_new[0, 0], v, rtol=0, atol=1e-12)


# ---------------------------------------------------------- (4) DeltaNet limit
def test_small_key_limit_alpha_to_beta():
    beta = 0.6
    for lam in (1e-2, 1e-4, 1e-6, 1e-8):
        a = oracle.alpha(beta, lam)
        # alpha/beta = (1 - e^{-x})/x = 1 - x/2 + x^2/6 - ... with x = beta*lam
        x = beta * lam
        # alternating series: x/2 - x^2/6 <= 1 - alpha/beta <= x/2 (plus rounding)
        gap = 1 - a / beta
        assert 0.5 * x - x * x / 6 - 1e-15 <= gap <= 0.5 * x + 1e-15
    assert oracle.alpha(beta, 0.0) == beta
    # away from zero the expm1 form agrees with the printed exp quotient
    for lam in (0.3, 1.0, 5.0, 50.0):
        assert oracle.alpha(beta, lam) == pytest.approx(literal.efla_gate_literal(beta, lam),
                                                        rel=1e-13)


def test_efla_recovers_deltanet_for_small_keys():
    """With keys scaled by eps the EFLA and Euler (DeltaNet) trajectories differ by
    O(eps^4) in the state increment relative to O(eps^2): slope 2 in eps."""
    q, k, v, beta, S0 = _head(4, 24, 6, 4)
    diffs = []
    for eps in (1e-2, 1e-3, 1e-4):
        ke = eps * k
        _, S_e = _fwd1(S0, q, ke, v, beta)
        _, S_d = literal.run_literal(literal.deltanet_step_literal, S0, q, ke, v, beta)
        inc = np.abs(S_d - S0).max()
        diffs.append(np.abs(S_e - S_d).max() / inc)
    assert diffs[0] < 0.01
    for d0, d1 in zip(diffs, diffs[1:]):
        assert 80 < d0 / d1 < 125  # relative gap shrinks like eps^2


# ------------------------------------------------------ literal (brute-force) form
@pytest.mark.parametrize("seed,T,dk,dv", [(5, 1, 3, 2), (6, 17, 5, 4), (7, 33, 8, 8)])
def test_oracle_matches_literal_matrix_form(seed, T, dk, dv):
    q, k, v, beta, S0 = _head(seed, T, dk, dv)
    o, S = _fwd1(S0, q, k, v, beta)
    o_l, S_l = literal.run_literal(literal.efla_step_literal, S0, q, k, v, beta)
    np.testing.assert_allclose(o, o_l, rtol=0, atol=1e-12 * (1 + np.abs(o_l).max()))
    np.testing.assert_allclose(S, S_l, rtol=0, atol=1e-12 * (1 + np.abs(S_l).max()))


# ------------------------------------------------------- (5) chunked == sequential
@pytest.mark.parametrize("chunk", [1, 2, 3, 16, 64])
def test_chunked_equals_sequential(chunk):
    r = _rng(50 + chunk)
    B, T, H, dk, dv = 2, 101, 2, 8, 6
    q = r.standard_normal((B, T, H, dk))
    k = r.standard_normal((B, T, H, dk)) * r.lognormal(0, 0.7, (B, T, H, 1)) / 2
    v = r.standard_normal((B, T, H, dv))
    beta = r.uniform(0.05, 1.0, (B, T, H))
    S0 = 0.2 * r.standard_normal((B, H, dk, dv))
    o, S = oracle.fwd(q, k, v, beta, S0)
    o_c, S_c = chunked.fwd(q, k, v, beta, S0, chunk=chunk)
    np.testing.assert_allclose(o_c, o, rtol=0, atol=1e-11 * (1 + np.abs(o).max()))
    np.testing.assert_allclose(S_c, S, rtol=0, atol=1e-11 * (1 + np.abs(S).max()))


def test_chunked_equals_sequential_stiff_and_zero_keys():
    """Norms over two decades and some exactly-zero keys (alpha = beta, no-op update)."""
    r = _rng(77)
    T, dk, dv = 150, 16, 8
    q = r.standard_normal((1, T, 1, dk))
    kd = r.standard_normal((1, T, 1, dk))
    kd /= np.linalg.norm(kd, axis=-1, keepdims=True)
    k = kd * r.uniform(0.1, 10.0, (1, T, 1, 1))
    k[0, ::13] = 0.0
    v = r.standard_normal((1, T, 1, dv))
    beta = 1 / (1 + np.exp(-(2 + r.standard_normal((1, T, 1)))))
    S0 = 0.1 * r.standard_normal((1, 1, dk, dv))
    o, S = oracle.fwd(q, k, v, beta, S0)
    o_c, S_c = chunked.fwd(q, k, v, beta, S0, chunk=64)
    np.testing.assert_allclose(o_c, o, rtol=0, atol=1e-10 * (1 + np.abs(o).max()))
    np.testing.assert_allclose(S_c, S, rtol=0, atol=1e-10 * (1 + np.abs(S).max()))


# ------------------------------------------------------------------ invariants
def test_linear_in_initial_state_and_values():
    """(S0, V) -> (O, S_T) is linear for fixed q, k, beta."""
    q, k, v, beta, S0 = _head(8, 30, 6, 5)
    r = _rng(88)
    v2 = r.standard_normal(v.shape)
    S02 = r.standard_normal(S0.shape)
    a, b = 0.7, -1.9
    o1, S1 = _fwd1(S0, q, k, v, beta)
    o2, S2 = _fwd1(S02, q, k, v2, beta)
    o3, S3 = _fwd1(a * S0 + b * S02, q, k, a * v + b * v2, beta)
    np.testing.assert_allclose(o3, a * o1 + b * o2, rtol=0, atol=1e-11)
    np.testing.assert_allclose(S3, a * S1 + b * S2, rtol=0, atol=1e-11)


def test_orthogonal_keys_commute():
    """Updates with mutually orthogonal keys commute: S_T is order-independent."""
    r = _rng(9)
    d, dv = 8, 3
    Qm, _ = np.linalg.qr(r.standard_normal((d, d)))
    k = (Qm.T * r.uniform(0.3, 3.0, d)[:, None])  # rows orthogonal
    v = r.standard_normal((d, dv))
    beta = r.uniform(0.1, 1.0, d)
    q = r.standard_normal((d, d))
    S0 = r.standard_normal((d, dv))
    _, S_a = _fwd1(S0, q, k, v, beta)
    perm = r.permutation(d)
    _, S_b = _fwd1(S0, q[perm], k[perm], v[perm], beta[perm])
    np.testing.assert_allclose(S_a, S_b, rtol=0, atol=1e-12)
    # closed form: each orthogonal direction relaxes independently toward v/|k|
    kh = k / np.linalg.norm(k, axis=1, keepdims=True)
    expect = S0.copy()
    for t in range(d):
        lam = float(k[t] @ k[t])
        g = 1 - math.exp(-beta[t] * lam)
        expect = expect + np.outer(kh[t], g * (v[t] / math.sqrt(lam) - kh[t] @ S0))
    np.testing.assert_allclose(S_a, expect, rtol=0, atol=1e-12)


def test_forward_then_decode_equals_longer_forward():
    q, k, v, beta, S0 = _head(12, 20, 5, 4)
    o_full, S_full = _fwd1(S0, q, k, v, beta)
    o_a, S = _fwd1(S0, q[:15], k[:15], v[:15], beta[:15])
    outs = [o_a]
    for t in range(15, 20):
        o_t, S4 = oracle.decode_step(q[t][None, None], k[t][None, None], v[t][None, None],
                                     np.array([[beta[t]]]), S[None, None])
        S = S4[0, 0]
        outs.append(o_t[0])
    np.testing.assert_allclose(np.concatenate(outs), o_full, rtol=0, atol=1e-12)
    np.testing.assert_allclose(S, S_full, rtol=0, atol=1e-12)


def test_varlen_packing_equals_separate_calls():
    r = _rng(13)
    lens = [5, 1, 0, 37, 12]
    H, dk, dv = 2, 6, 3
    Tt = sum(lens)
    q = r.standard_normal((1, Tt, H, dk))
    k = r.standard_normal((1, Tt, H, dk))
    v = r.standard_normal((1, Tt, H, dv))
    beta = r.uniform(0.1, 1.0, (1, Tt, H))
    S0 = r.standard_normal((len(lens), H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, S = oracle.fwd(q, k, v, beta, S0, cu)
    for n, (t0, t1) in enumerate(zip(cu[:-1], cu[1:])):
        o_n, S_n = oracle.fwd(q[:, t0:t1], k[:, t0:t1], v[:, t0:t1], beta[:, t0:t1], S0[n:n + 1])
        np.testing.assert_array_equal(o[:, t0:t1], o_n)
        np.testing.assert_array_equal(S[n], S_n[0])
    np.testing.assert_array_equal(S[2], S0[2])  # empty sequence: S_T = S0
    o_c, S_c = chunked.fwd(q, k, v, beta, S0, cu, chunk=4)
    np.testing.assert_allclose(o_c, o, rtol=0, atol=1e-11)
    np.testing.assert_allclose(S_c, S, rtol=0, atol=1e-11)


def test_threads_do_not_change_results():
    r = _rng(14)
    q = r.standard_normal((2, 9, 4, 5))
    k = r.standard_normal((2, 9, 4, 5))
    v = r.standard_normal((2, 9, 4, 3))
    beta = r.uniform(0.1, 1, (2, 9, 4))
    a = oracle.fwd(q, k, v, beta, threads=1)
    b = oracle.fwd(q, k, v, beta, threads=4)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_oracle_rejects_bad_bounds():
    q = np.zeros((1, 4, 1, 2))
    with pytest.raises(ValueError):
        oracle.fwd(q, q, q, np.zeros((1, 4, 1)), None, np.array([0, 3, 2, 4]))
    with pytest.raises(ValueError):
        oracle.fwd(q, q, q, np.zeros((1, 4, 1)), None, np.array([0, 3]))


# ------------------------------------------------------------- Euler (DeltaNet) mode
def test_euler_mode_matches_literal_deltanet():
    """update="euler" is the delta-rule step S <- (I - beta k k^T) S + beta k v^T
    (howistudyai, "Delta Rule"), checked against the literal matrix form."""
    q, k, v, beta, S0 = _head(60, 29, 6, 5)
    o, S = oracle.fwd(q[None, :, None], k[None, :, None], v[None, :, None], beta[None, :, None],
                      S0[None, None], update="euler")
    o_l, S_l = literal.run_literal(literal.deltanet_step_literal, S0, q, k, v, beta)
    np.testing.assert_allclose(o[0, :, 0], o_l, rtol=0, atol=1e-11 * (1 + np.abs(o_l).max()))
    np.testing.assert_allclose(S[0, 0], S_l, rtol=0, atol=1e-11 * (1 + np.abs(S_l).max()))
    o_d, S_d = oracle.decode_step(q[0][None, None], k[0][None, None], v[0][None, None],
                                  np.array([[beta[0]]]), S0[None, None], update="euler")
    o_l1, S_l1 = literal.deltanet_step_literal(S0, q[0], k[0], v[0], beta[0])
    np.testing.assert_allclose(S_d[0, 0], S_l1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o_d[0, 0], o_l1, rtol=0, atol=1e-12)


def test_euler_and_exact_differ_for_large_keys():
    """The two updates are different methods: with beta*lambda ~ 4 they disagree."""
    q, k, v, beta, S0 = _head(61, 10, 4, 3, key_scale=2.0)
    _, S_e = _fwd1(S0, q, k, v, beta)
    _, S_d = oracle.fwd(q[None, :, None], k[None, :, None], v[None, :, None], beta[None, :, None],
                        S0[None, None], update="euler")
    assert np.abs(S_e - S_d[0, 0]).max() > 0.1


# ----------------------------------------------------------------- backward
def _fd_case(seed=3, T=6, H=2, dk=3, dv=2):
    rng = np.random.default_rng(seed)
    q = rng.normal(size=(1, T, H, dk))
    k = rng.normal(size=(1, T, H, dk))
    k[0, 2, 0] = 0.0                      # lambda = 0: the gate's limit value
    v = rng.normal(size=(1, T, H, dv))
    beta = rng.uniform(0.2, 1.5, size=(1, T, H))
    beta[0, 4, 1] = 1e-5                  # beta*lambda below 1e-3: the gate derivative's series branch
    S0 = rng.normal(size=(1, H, dk, dv))
    W = rng.normal(size=(1, T, H, dv))    # L = sum(o * W) + sum(S_T * V)
    V = rng.normal(size=(1, H, dk, dv))
    return q, k, v, beta, S0, W, V


@pytest.mark.parametrize("update", ["exact", "euler"])
def test_bwd_matches_finite_differences(update):
    """Every gradient of L = <o, W> + <S_T, V> against central differences of the forward oracle."""
    q, k, v, beta, S0, W, V = _fd_case()
    g = oracle.bwd(q, k, v, beta, S0, W, V, update=update)

    def loss(qq, kk, vv, bb, ss):
        o, S_T = oracle.fwd(qq, kk, vv, bb, ss, update=update)
        return float(np.sum(o * W) + np.sum(S_T * V))

    args = [q, k, v, beta, S0]
    names = ["dq", "dk", "dv", "dbeta", "dS0"]
    h = 1e-6
    for ai, name in enumerate(names):
        base = args[ai]
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            if name == "dk" and base[idx] == 0.0 and update == "exact":
                pass  # k = 0 is inside the domain from both sides: central differences are fine
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[ai][idx] += h
            minus[ai][idx] -= h
            fd[idx] = (loss(*plus) - loss(*minus)) / (2 * h)
        np.testing.assert_allclose(g[name], fd, rtol=2e-6, atol=2e-7, err_msg=f"{name} ({update})")


def test_gate_derivatives_match_finite_differences():
    h = 1e-7
    for beta in (0.3, 1.7, -0.4):
        for lam in (1e-6 / abs(beta), 5e-4 / abs(beta), 2e-3 / abs(beta), 0.5, 5.0, 30.0):
            dfdb, dfdl = oracle.gate_grad(beta, lam)
            fb = (oracle.alpha(beta + h, lam) - oracle.alpha(beta - h, lam)) / (2 * h)
            hl = h * max(lam, 1e-3)
            fl = (oracle.alpha(beta, lam + hl) - oracle.alpha(beta, lam - hl)) / (2 * hl)
            assert abs(dfdb - fb) <= 1e-6 * max(1.0, abs(fb)), (beta, lam, dfdb, fb)
            assert abs(dfdl - fl) <= 2e-5 * max(1.0, abs(fl)), (beta, lam, dfdl, fl)
        # at lam = 0 the gate is beta and its lam-slope is the limit -beta^2/2
        dfdb, dfdl = oracle.gate_grad(beta, 0.0)
        assert dfdb == 1.0 and abs(dfdl + beta * beta / 2) < 1e-15
        fl = (oracle.alpha(beta, 1e-7) - oracle.alpha(beta, 0.0)) / 1e-7
        assert abs(dfdl - fl) < 1e-6


def test_bwd_zero_step_size_closed_form():
    """beta = 0: the state never moves, so o_t = S0^T q_t, dq_t = S0 do_t, dS0 = dS_T + sum q_t do_t^T,
    dv = 0, dk = 0, and dbeta_t = du_t . (v_t - x_t) with du_t = G_t^T k_t, x_t = S0^T k_t and
    G_t = dS_T + sum_{s >= t} q_s do_s^T (df/dbeta = 1 at beta = 0)."""
    rng = np.random.default_rng(8)
    T, dk, dv = 5, 4, 3
    q, k = rng.normal(size=(1, T, 1, dk)), rng.normal(size=(1, T, 1, dk))
    v, do = rng.normal(size=(1, T, 1, dv)), rng.normal(size=(1, T, 1, dv))
    S0, dST = rng.normal(size=(1, 1, dk, dv)), rng.normal(size=(1, 1, dk, dv))
    g = oracle.bwd(q, k, v, np.zeros((1, T, 1)), S0, do, dST)
    s0 = S0[0, 0]
    np.testing.assert_allclose(g["dq"][0, :, 0], do[0, :, 0] @ s0.T, atol=1e-12)
    np.testing.assert_allclose(g["dS0"][0, 0], dST[0, 0] + np.einsum("ti,tj->ij", q[0, :, 0], do[0, :, 0]),
                               atol=1e-12)
    assert np.abs(g["dv"]).max() == 0 and np.abs(g["dk"]).max() == 0
    for t in range(T):
        Gt = dST[0, 0] + np.einsum("si,sj->ij", q[0, t:, 0], do[0, t:, 0])
        du = Gt.T @ k[0, t, 0]
        x = s0.T @ k[0, t, 0]
        assert abs(g["dbeta"][0, t, 0] - du @ (v[0, t, 0] - x)) < 1e-12


def test_bwd_is_linear_in_output_gradients():
    q, k, v, beta, S0, W, V = _fd_case(seed=5, T=9, H=2, dk=5, dv=4)
    g1 = oracle.bwd(q, k, v, beta, S0, W, V)
    g2 = oracle.bwd(q, k, v, beta, S0, 2.5 * W, None)
    g3 = oracle.bwd(q, k, v, beta, S0, np.zeros_like(W), 2.5 * V)
    for name in g1:
        np.testing.assert_allclose(2.5 * g1[name], g2[name] + g3[name], rtol=1e-12, atol=1e-12)

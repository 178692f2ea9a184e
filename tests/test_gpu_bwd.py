"""GPU parity of the backward passes (efla_bwd_recurrent, efla_bwd_chunked) against the fp64
reverse-mode oracle.

Tolerance: the kernels evaluate every gradient in fp32 on CUDA cores from exactly
representable inputs (the oracle sees the same values upcast), so the bar is the fp32
one used for the forward, relative Frobenius error <= 1e-4 per gradient tensor.  The chunked
path takes its chunk-start states from the forward kernels (for bf16 with d = 128 the
tensor-core kernel, whose split-bf16 products leave about 1e-5 of relative error in them);
the same bar holds."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
REL = 1e-4


@pytest.fixture(scope="module")
def efla():
    import exact_delta_rule_gb300 as m
    from exact_delta_rule_gb300 import build
    build.build()
    m.load()
    return m


def _rel(got, ref):
    got = got.detach().double().cpu().numpy()
    assert np.all(np.isfinite(got))
    n = np.linalg.norm(ref)
    return np.linalg.norm(got - ref) / (n if n > 0 else 1.0)


def _case(dtype, B, T, H, dk, dv, seed, s0=True, dst=True):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, T, H, dk), generator=g)
    k = torch.nn.functional.normalize(torch.randn((B, T, H, dk), generator=g), dim=-1)
    k = k * torch.exp(0.5 * torch.randn((B, T, H, 1), generator=g))
    v = torch.randn((B, T, H, dv), generator=g)
    beta = torch.sigmoid(torch.randn((B, T, H), generator=g))
    S0 = 0.1 * torch.randn((B, H, dk, dv), generator=g) if s0 else None
    dO = torch.randn((B, T, H, dv), generator=g)
    dST = torch.randn((B, H, dk, dv), generator=g) if dst else None
    if dtype == "bf16":
        q, k, v = (x.to(torch.bfloat16) for x in (q, k, v))
    return dict(q=q.contiguous(), k=k.contiguous(), v=v.contiguous(), beta=beta, S0=S0, dO=dO, dST=dST)


def _check(efla, c, update="exact", kind="recurrent"):
    d = {x: (y.to(DEV) if y is not None else None) for x, y in c.items()}
    fn = efla.bwd_recurrent if kind == "recurrent" else efla.bwd_chunked
    got = fn(d["q"], d["k"], d["v"], d["beta"], d["S0"], d["dO"], d["dST"], update=update)
    torch.cuda.synchronize()
    ref = oracle.bwd(c["q"], c["k"], c["v"], c["beta"], c["S0"], c["dO"], c["dST"], update=update)
    for name in ("dq", "dk", "dv", "dbeta", "dS0"):
        r = _rel(got[name], ref[name])
        assert r <= REL, f"{name}: rel-fro {r:.3e}"


KINDS = ["recurrent", "chunked"]


@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 64), (128, 128), (64, 32), (32, 128)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bwd_small(efla, dk, dv, dtype):
    _check(efla, _case(dtype, 2, 37, 2, dk, dv, seed=dk + dv))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [37, 64, 200])
def test_bwd_chunked_small(efla, d, dtype, T):
    """One partial chunk, one full chunk, and several chunks with a ragged tail."""
    _check(efla, _case(dtype, 2, T, 2, d, d, seed=d + T), kind="chunked")


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("f32", 128)])
def test_train_forward_then_saved_backward(efla, dtype, d):
    """fwd_chunked_train gives fwd_chunked's o and S_T bit for bit and keeps the chunk-start
    states (and T'') in the workspace; bwd_chunked(saved=True) on that workspace gives the
    gradients of bwd_chunked (which runs the forward again) and of the oracle."""
    c = _case(dtype, 2, 200, 3, d, d, seed=300 + d)
    g = {x: (y.to(DEV) if y is not None else None) for x, y in c.items()}
    o_ref, S_ref = efla.fwd_chunked(g["q"], g["k"], g["v"], g["beta"], g["S0"])
    o, S_T, ws = efla.fwd_chunked_train(g["q"], g["k"], g["v"], g["beta"], g["S0"])
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(S_T, S_ref)
    got = efla.bwd_chunked(g["q"], g["k"], g["v"], g["beta"], g["S0"], g["dO"], g["dST"], workspace=ws, saved=True)
    full = efla.bwd_chunked(g["q"], g["k"], g["v"], g["beta"], g["S0"], g["dO"], g["dST"])
    torch.cuda.synchronize()
    ref = oracle.bwd(c["q"], c["k"], c["v"], c["beta"], c["S0"], c["dO"], c["dST"])
    for name in ("dq", "dk", "dv", "dbeta", "dS0"):
        same = ((got[name] - full[name]).norm() / full[name].norm()).item()
        assert same <= 1e-6, f"{name}: saved vs full backward rel-fro {same:.3e}"
        r = _rel(got[name], ref[name])
        assert r <= REL, f"{name}: rel-fro {r:.3e}"
    assert efla.device_status() == 0


@pytest.mark.parametrize("B,T,H,s0,dst", [(1, 1, 1, True, True), (1, 64, 2, False, True), (2, 65, 3, True, False),
                                           (1, 129, 2, False, False)])
def test_train_pair_edge_shapes(efla, B, T, H, s0, dst):
    """The training pair (bf16, d = 128, every step on the tensor cores) on a single token, one
    full chunk, a full chunk and one token, and a ragged third chunk, with and without S0 and
    dS_T: o and S_T bit for bit those of fwd_chunked, the saved backward against the oracle, and
    the workspace reused by a second pair on other inputs of the same shape."""
    ws = None
    for seed in (400 + T, 500 + T):
        c = _case("bf16", B, T, H, 128, 128, seed=seed, s0=s0, dst=dst)
        g = {x: (y.to(DEV) if y is not None else None) for x, y in c.items()}
        o, S_T, ws = efla.fwd_chunked_train(g["q"], g["k"], g["v"], g["beta"], g["S0"], workspace=ws)
        got = efla.bwd_chunked(g["q"], g["k"], g["v"], g["beta"], g["S0"], g["dO"], g["dST"], workspace=ws, saved=True)
        o_ref, S_ref = efla.fwd_chunked(g["q"], g["k"], g["v"], g["beta"], g["S0"])
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(S_T, S_ref)
        ref = oracle.bwd(c["q"], c["k"], c["v"], c["beta"], c["S0"], c["dO"], c["dST"])
        for name in ("dq", "dk", "dv", "dbeta", "dS0"):
            r = _rel(got[name], ref[name])
            assert r <= REL, f"seed {seed} {name}: rel-fro {r:.3e}"
    assert efla.device_status() == 0


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_train_pair_delta_rule_gate(efla, dtype, d):
    """The training pair with the delta-rule gate (alpha = beta, unit-norm keys), against the
    oracle's reverse mode of the same recurrence."""
    c = _case(dtype, 2, 150, 2, d, d, seed=600 + d)
    kf = torch.nn.functional.normalize(c["k"].float(), dim=-1)
    c["k"] = (kf.to(torch.bfloat16) if dtype == "bf16" else kf).contiguous()
    g = {x: (y.to(DEV) if y is not None else None) for x, y in c.items()}
    o, S_T, ws = efla.fwd_chunked_train(g["q"], g["k"], g["v"], g["beta"], g["S0"], update="euler")
    got = efla.bwd_chunked(g["q"], g["k"], g["v"], g["beta"], g["S0"], g["dO"], g["dST"], workspace=ws, saved=True,
                           update="euler")
    o_ref, S_ref = efla.fwd_chunked(g["q"], g["k"], g["v"], g["beta"], g["S0"], update="euler")
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(S_T, S_ref)
    ref = oracle.bwd(c["q"], c["k"], c["v"], c["beta"], c["S0"], c["dO"], c["dST"], update="euler")
    for name in ("dq", "dk", "dv", "dbeta", "dS0"):
        r = _rel(got[name], ref[name])
        assert r <= REL, f"{name}: rel-fro {r:.3e}"
    assert efla.device_status() == 0


@pytest.mark.parametrize("kind", KINDS)
def test_bwd_no_state_no_state_gradient(efla, kind):
    _check(efla, _case("bf16", 1, 64, 3, 128, 128, seed=4, s0=False, dst=False), kind=kind)


@pytest.mark.parametrize("kind", KINDS)
def test_bwd_zero_keys_and_zero_steps(efla, kind):
    c = _case("f32", 1, 140, 2, 64, 64, seed=6)
    c["k"][:, 3::7] = 0
    c["beta"][:, 5::6] = 0
    c["beta"][:, 2::9] = 1e-4  # beta*lambda in the gate derivative's series range
    _check(efla, c, kind=kind)


@pytest.mark.parametrize("B,T,H", [(1, 1, 1), (1, 65, 1), (3, 333, 5), (2, 1000, 10)])
def test_bwd_chunked_tensor_core_shapes(efla, B, T, H):
    """bf16, d = 128 (every step on the tensor cores): a single token, one full chunk and one
    token, ragged tails on several units, and 320 chunk items, so that each persistent CTA of the
    gradient kernel walks two or three items and every mbarrier turns both parities."""
    _check(efla, _case("bf16", B, T, H, 128, 128, seed=100 + B * T + H), kind="chunked")


def test_bwd_chunked_tensor_core_path_zero_keys_zero_steps_and_euler(efla):
    """bf16 with d = 128 takes the tensor-core steps (the state pass's hand-over of G and -dR,
    the forward's T'' in both later steps): zero keys (whose T'' diagonal the gradient kernel
    sets), beta = 0, the gate derivative's series branch, a ragged tail and the delta-rule gate,
    against the oracle."""
    c = _case("bf16", 1, 150, 2, 128, 128, seed=8)
    k = c["k"].clone()
    k[:, 3::7] = 0
    c["k"] = k.contiguous()
    c["beta"][:, 5::6] = 0
    c["beta"][:, 2::9] = 1e-4
    _check(efla, c, kind="chunked")
    e = _case("bf16", 2, 100, 2, 128, 128, seed=9)
    e["k"] = torch.nn.functional.normalize(e["k"].float(), dim=-1).to(torch.bfloat16).contiguous()
    _check(efla, e, update="euler", kind="chunked")
    assert efla.device_status() == 0


@pytest.mark.parametrize("kind", KINDS)
def test_bwd_delta_rule_gate(efla, kind):
    c = _case("f32", 2, 150, 2, 64, 64, seed=7)
    c["k"] = torch.nn.functional.normalize(c["k"], dim=-1).contiguous()
    _check(efla, c, update="euler", kind=kind)


@pytest.mark.parametrize("kind", KINDS)
def test_bwd_longer_sequence_lm_law(efla, kind):
    inp = workloads.small_fwd("bf16", B=1, T=384, H=2, d=128, seed=19)
    g = torch.Generator().manual_seed(20)
    c = dict(q=inp["q"], k=inp["k"], v=inp["v"], beta=inp["beta"], S0=inp["S0"],
             dO=torch.randn((1, 384, 2, 128), generator=g), dST=torch.randn((1, 2, 128, 128), generator=g))
    _check(efla, c, kind=kind)
    assert efla.device_status() == 0


def test_bwd_chunked_stiff_keys(efla):
    """Key norms U[0.1, 10] and beta = sigmoid(N(2, 1)), as in the long-sequence workload."""
    g = torch.Generator().manual_seed(23)
    c = _case("bf16", 1, 256, 2, 128, 128, seed=22)
    kd = torch.nn.functional.normalize(torch.randn((1, 256, 2, 128), generator=g), dim=-1)
    c["k"] = (kd * (0.1 + 9.9 * torch.rand((1, 256, 2, 1), generator=g))).to(torch.bfloat16).contiguous()
    c["beta"] = torch.sigmoid(2.0 + torch.randn((1, 256, 2), generator=g))
    _check(efla, c, kind="chunked")


def test_bwd_chunked_equals_recurrent_lm_heads(efla):
    """B=8 H=16 T=2048 d=128 (the language-model-layer shape): the two backward paths agree on
    every head to rel-Frobenius <= 1e-4 (two fp32 evaluations of the same gradients)."""
    inp = workloads.make_fwd_inputs(workloads.FWD_WORKLOADS["lm"])
    g = torch.Generator().manual_seed(31)
    q, k, v, beta = (inp[x].to(DEV) for x in ("q", "k", "v", "beta"))
    B, T, H, d = q.shape
    dO = torch.randn((B, T, H, d), generator=g).to(DEV)
    dST = torch.randn((B, H, d, d), generator=g).to(DEV)
    a = efla.bwd_chunked(q, k, v, beta, None, dO, dST)
    b = efla.bwd_recurrent(q, k, v, beta, None, dO, dST)
    torch.cuda.synchronize()
    for name in ("dq", "dk", "dv", "dbeta", "dS0"):
        r = ((a[name] - b[name]).norm() / b[name].norm()).item()
        assert r <= REL, f"{name}: rel-fro {r:.3e}"
    assert efla.device_status() == 0


@pytest.mark.parametrize("kind", KINDS)
def test_bwd_empty(efla, kind):
    fn = efla.bwd_recurrent if kind == "recurrent" else efla.bwd_chunked
    e = torch.empty((2, 0, 2, 64), device=DEV)
    S0 = torch.randn((2, 2, 64, 64), device=DEV)
    dST = torch.randn((2, 2, 64, 64), device=DEV)
    out = fn(e, e, e, torch.empty((2, 0, 2), device=DEV), S0, e, dST)
    torch.cuda.synchronize()
    assert torch.equal(out["dS0"], dST)

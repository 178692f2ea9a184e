"""GPU parity of the delta-rule (Euler) update mode and of the prep kernel."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def efla():
    import exact_delta_rule_gb300 as m
    from exact_delta_rule_gb300 import build
    build.build()
    m.load()
    return m


def _unit_keys(inp):
    """The delta rule is used with L2-normalised keys (it is unstable for large
    beta*||k||^2); normalise the generated keys in place."""
    k = inp["k"].float()
    inp["k"] = (k / k.norm(dim=-1, keepdim=True).clamp_min(1e-6)).to(inp["k"].dtype)
    return inp


@pytest.mark.parametrize("fn", ["chunked", "recurrent"])
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_euler_forward(efla, fn, dtype, d):
    inp = _unit_keys(workloads.small_fwd(dtype, B=2, T=150, H=2, d=d, seed=71))
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    f = efla.fwd_chunked if fn == "chunked" else efla.fwd_recurrent
    o, S = f(g["q"], g["k"], g["v"], g["beta"], g["S0"], update="euler", o_dtype=torch.float32)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["S0"], update="euler")
    check(o, o_ref, in_dtype=dtype, what=f"euler o {fn}")
    check(S, S_ref, in_dtype=dtype, what=f"euler S_T {fn}")
    # and it is not the exact update
    o_x, _ = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["S0"])
    assert np.abs(o_x - o_ref).max() > 1e-2


def test_euler_decode(efla):
    cfg = workloads.DecodeWorkload("d", 4, 3, 128, 128, 5, 2, 0.1)
    S0 = workloads.make_decode_state(cfg)
    inp = workloads.make_decode_step(0, cfg)
    k = inp["k"].float()
    inp["k"] = (k / k.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    S = S0.to(DEV)
    o = efla.decode_step(*(inp[x].to(DEV) for x in ("q", "k", "v", "beta")), S, update="euler", o_dtype=torch.float32)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.decode_step(inp["q"], inp["k"], inp["v"], inp["beta"], S0, update="euler")
    check(o, o_ref, in_dtype="bf16", what="euler decode o")
    check(S, S_ref, in_dtype="bf16", what="euler decode S")


@pytest.mark.parametrize("dtype,dk,dv", [("bf16", 128, 128), ("bf16", 32, 64), ("f32", 64, 128)])
@pytest.mark.parametrize("update", ["exact", "euler"])
def test_prep_matches_oracle(efla, dtype, dk, dv, update):
    cfg = workloads.FwdWorkload("p", 2, 333, 3, dk, dv, dtype, 81, "uniform", 0.0, 10.0, 2.0, 0.0)
    inp = workloads.make_fwd_inputs(cfg)
    inp["k"][0, 5, 1] = 0  # a zero key: lambda = 0, alpha = beta
    k, v, beta = (inp[x].to(DEV) for x in ("k", "v", "beta"))
    out = efla.prep(k, beta, v, lam=True, alpha=True, ak=True, av=True, update=update)
    torch.cuda.synchronize()
    k64 = to64(inp["k"]).reshape(-1, dk)
    v64 = to64(inp["v"]).reshape(-1, dv)
    b64 = to64(inp["beta"]).reshape(-1)
    lam_ref = (k64 * k64).sum(-1)
    if update == "exact":
        a_ref = np.array([oracle.alpha(b, l) for b, l in zip(b64, lam_ref)])
    else:
        a_ref = b64
    lam = to64(out["lam"]).reshape(-1)
    a = to64(out["alpha"]).reshape(-1)
    np.testing.assert_allclose(lam, lam_ref, rtol=1e-5, atol=1e-30)
    np.testing.assert_allclose(a, a_ref, rtol=2e-5, atol=1e-30)
    rnd = 2.0 ** -8 if dtype == "bf16" else 1e-6
    ak_ref = a_ref[:, None] * k64
    av_ref = a_ref[:, None] * v64
    assert np.all(np.abs(to64(out["ak"]).reshape(-1, dk) - ak_ref) <= rnd * np.abs(ak_ref) + 1e-30)
    assert np.all(np.abs(to64(out["av"]).reshape(-1, dv) - av_ref) <= rnd * np.abs(av_ref) + 1e-30)
    zero_row = 5 * 3 + 1
    assert lam[zero_row] == 0 and a[zero_row] == pytest.approx(b64[zero_row])

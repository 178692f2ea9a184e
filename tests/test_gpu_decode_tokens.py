"""GPU parity of the multi-token decode (efla_decode_tokens) against the fp64 oracle.

m tokens appended to a resident state are the sequential recurrence over those
tokens with the state as S0, so the oracle is its forward over a length-m
sequence per (b, h)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def efla():
    import exact_delta_rule_gb300 as m
    from exact_delta_rule_gb300 import build
    build.build()
    m.load()
    return m


def _case(dk, dv, m, B=3, H=5, seed=91):
    cfg = workloads.DecodeWorkload("t", B, H, dk, dv, seed, 1, 0.1)
    return cfg, workloads.make_decode_state(cfg), workloads.make_decode_tokens(m, cfg)


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64), (32, 128), (128, 32)])
@pytest.mark.parametrize("m", [1, 5, 16, 37])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_tokens_small(efla, dk, dv, m, dtype):
    cfg, S0, inp = _case(dk, dv, m)
    if dtype == "f32":
        inp = {k: v.float() for k, v in inp.items()}
    S = S0.to(DEV)
    o = efla.decode_tokens(*(inp[x].to(DEV) for x in ("q", "k", "v", "beta")), S, o_dtype=torch.float32)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["beta"], S0, threads=0)
    check(o, o_ref, in_dtype=dtype, what=f"decode_tokens o m={m}")
    check(S, S_ref, in_dtype=dtype, what=f"decode_tokens S m={m}")


def test_decode_tokens_bf16_out_and_euler(efla):
    cfg, S0, inp = _case(128, 128, 7)
    # the delta-rule step (I - beta k k^T) is contractive only for beta ||k||^2 < 2: unit-norm keys
    kf = inp["k"].float()
    inp["k"] = (kf / kf.norm(dim=-1, keepdim=True)).to(torch.bfloat16).contiguous()
    S = S0.to(DEV)
    o = efla.decode_tokens(*(inp[x].to(DEV) for x in ("q", "k", "v", "beta")), S, o_dtype=torch.bfloat16,
                           update="euler")
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["beta"], S0, threads=0, update="euler")
    check(o, o_ref, in_dtype="bf16", what="decode_tokens euler o (bf16)", out_bf16=True)
    check(S, S_ref, in_dtype="bf16", what="decode_tokens euler S")


def test_decode_tokens_equals_chained_steps(efla):
    """m tokens at once and m single-token steps on the same inputs agree.

    With bf16 q, k, v and d = 128 the m tokens go through the tensor-core kernel, whose
    products split each non-bf16 operand into bf16 hi + lo parts (a residual of at most
    2^-16 of the operand), so the two paths agree to about 1e-5 of the values' scale
    rather than to fp32 rounding: relative Frobenius difference <= 1e-4."""
    cfg, S0, inp = _case(128, 128, 9, B=4, H=6)
    S1, S2 = S0.to(DEV), S0.to(DEV)
    g = {x: inp[x].to(DEV) for x in ("q", "k", "v", "beta")}
    o1 = efla.decode_tokens(g["q"], g["k"], g["v"], g["beta"], S1, o_dtype=torch.float32)
    o2 = torch.stack([efla.decode_step(g["q"][:, t].contiguous(), g["k"][:, t].contiguous(),
                                       g["v"][:, t].contiguous(), g["beta"][:, t].contiguous(), S2,
                                       o_dtype=torch.float32)
                      for t in range(9)], dim=1)
    torch.cuda.synchronize()
    for got, want in ((o1, o2), (S1, S2)):
        rel = (got - want).norm() / want.norm()
        assert rel <= 1e-4, rel


def test_decode_tokens_zero_tokens_and_empty_batch(efla):
    cfg, S0, inp = _case(64, 64, 0)
    S = S0.to(DEV)
    o = efla.decode_tokens(*(inp[x].to(DEV) for x in ("q", "k", "v", "beta")), S, o_dtype=torch.float32)
    torch.cuda.synchronize()
    assert o.shape == (3, 0, 5, 64)
    assert torch.equal(S.cpu(), S0)
    e = torch.empty((0, 4, 2, 64), dtype=torch.bfloat16, device=DEV)
    Se = torch.empty((0, 2, 64, 64), device=DEV)
    o = efla.decode_tokens(e, e, e, torch.empty((0, 4, 2), device=DEV), Se, o_dtype=torch.float32)
    assert o.shape == (0, 4, 2, 64)


def test_decode_tokens_full_size_sampled(efla):
    """B256 H32 d128, 16 tokens per call, two chained calls; sampled heads replayed by the oracle."""
    cfg = workloads.DECODE
    S0 = workloads.make_decode_state(cfg)
    S = S0.to(DEV)
    rng = np.random.default_rng(1)
    bs = rng.choice(cfg.B, 6, replace=False)
    hs = rng.choice(cfg.H, 6, replace=False)
    S_ref = S0[bs][:, hs].contiguous()
    for call in range(2):
        inp = workloads.make_decode_tokens(16, cfg, first_step=16 * call)
        o = efla.decode_tokens(*(inp[x].to(DEV) for x in ("q", "k", "v", "beta")), S, o_dtype=torch.float32)
        torch.cuda.synchronize()
        sub = {x: inp[x][bs][:, :, hs].contiguous() for x in ("q", "k", "v", "beta")}
        # the oracle's sequences are the (b, h) pairs of the sample
        o_ref, S_new = oracle.fwd(sub["q"], sub["k"], sub["v"], sub["beta"], S_ref, threads=0)
        got_o = o[torch.as_tensor(bs)][:, :, torch.as_tensor(hs)]
        check(got_o, o_ref, in_dtype="bf16", what=f"decode_tokens o call {call}")
        S_ref = torch.from_numpy(S_new)
        got_S = S[torch.as_tensor(bs)][:, torch.as_tensor(hs)]
        check(got_S, S_ref, in_dtype="bf16", what=f"decode_tokens S call {call}")
    assert efla.device_status() == 0

"""Seeded random sweep of shapes through the tensor-core paths (bf16, d = 128) and the
CUDA-core paths, against the fp64 oracle.

The cases are drawn once from a fixed seed, so the sweep is the same on every run: batch and
head counts that do not divide the SM count, lengths on and off the 64-token chunk grid, with
and without S0, varlen batches with empty and one-token sequences, multi-token decode of every
token count up to 16, and the chunked backward on ragged items.  Bars: tests/parity.py for
the forward and decode, relative Frobenius <= 1e-4 per gradient for the backward."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
_R = np.random.default_rng(20261203)
FWD_CASES = [dict(B=int(_R.integers(1, 4)), T=int(_R.integers(1, 700)), H=int(_R.integers(1, 6)),
                  s0=bool(_R.integers(0, 2)), seed=1000 + i) for i in range(8)]
VARLEN_CASES = [dict(lens=[int(x) for x in _R.choice([0, 1, 2, 63, 64, 65, 127, 129, 250], size=int(_R.integers(2, 9)))],
                     H=int(_R.integers(1, 4)), seed=2000 + i) for i in range(3)]
DECODE_CASES = [dict(B=int(_R.integers(1, 40)), H=int(_R.integers(1, 9)), m=int(_R.integers(1, 17)), seed=3000 + i)
                for i in range(5)]
BWD_CASES = [dict(B=int(_R.integers(1, 3)), T=int(_R.integers(1, 400)), H=int(_R.integers(1, 5)),
                  s0=bool(_R.integers(0, 2)), dst=bool(_R.integers(0, 2)), seed=4000 + i) for i in range(4)]


@pytest.fixture(scope="module")
def efla():
    import exact_delta_rule_gb300 as m
    from exact_delta_rule_gb300 import build
    build.build()
    m.load()
    return m


def _ids(cases):
    return ["-".join(f"{k}{v if not isinstance(v, list) else len(v)}" for k, v in c.items()) for c in cases]


@pytest.mark.parametrize("c", FWD_CASES, ids=_ids(FWD_CASES))
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_sweep_fwd_chunked(efla, c, dtype, d):
    inp = workloads.small_fwd(dtype, B=c["B"], T=c["T"], H=c["H"], d=d, seed=c["seed"], s0=c["s0"])
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    o, S = efla.fwd_chunked(g["q"], g["k"], g["v"], g["beta"], g["S0"], o_dtype=torch.float32)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["S0"], threads=0)
    check(o, o_ref, in_dtype=dtype, what=f"o {c}")
    check(S, S_ref, in_dtype=dtype, what=f"S_T {c}")


@pytest.mark.parametrize("c", VARLEN_CASES, ids=_ids(VARLEN_CASES))
def test_sweep_varlen(efla, c):
    inp = workloads.small_fwd("bf16", H=c["H"], d=128, seed=c["seed"], lengths=c["lens"])
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    o, S = efla.fwd_chunked(g["q"], g["k"], g["v"], g["beta"], g["S0"], g["cu_seqlens"])
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["S0"], inp["cu_seqlens"], threads=0)
    check(o, o_ref, in_dtype="bf16", what=f"o {c}", out_bf16=True)
    check(S, S_ref, in_dtype="bf16", what=f"S_T {c}")


@pytest.mark.parametrize("c", DECODE_CASES, ids=_ids(DECODE_CASES))
def test_sweep_decode_tokens(efla, c):
    cfg = workloads.DecodeWorkload("sweep", c["B"], c["H"], 128, 128, c["seed"], 1, 0.1)
    S0 = workloads.make_decode_state(cfg)
    inp = workloads.make_decode_tokens(c["m"], cfg)
    S = S0.to(DEV)
    o = efla.decode_tokens(*(inp[x].to(DEV) for x in ("q", "k", "v", "beta")), S, o_dtype=torch.float32)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["beta"], S0, threads=0)
    check(o, o_ref, in_dtype="bf16", what=f"decode_tokens o {c}")
    check(S, S_ref, in_dtype="bf16", what=f"decode_tokens S {c}")


@pytest.mark.parametrize("c", BWD_CASES, ids=_ids(BWD_CASES))
def test_sweep_bwd_chunked(efla, c):
    g = torch.Generator().manual_seed(c["seed"])
    B, T, H, d = c["B"], c["T"], c["H"], 128
    q = torch.randn((B, T, H, d), generator=g)
    k = torch.nn.functional.normalize(torch.randn((B, T, H, d), generator=g), dim=-1)
    k = k * torch.exp(0.5 * torch.randn((B, T, H, 1), generator=g))
    v = torch.randn((B, T, H, d), generator=g)
    beta = torch.sigmoid(torch.randn((B, T, H), generator=g))
    S0 = 0.1 * torch.randn((B, H, d, d), generator=g) if c["s0"] else None
    dO = torch.randn((B, T, H, d), generator=g)
    dST = torch.randn((B, H, d, d), generator=g) if c["dst"] else None
    q, k, v = (x.to(torch.bfloat16).contiguous() for x in (q, k, v))
    dev = lambda x: x.to(DEV) if x is not None else None  # noqa: E731
    got = efla.bwd_chunked(dev(q), dev(k), dev(v), dev(beta), dev(S0), dev(dO), dev(dST))
    torch.cuda.synchronize()
    ref = oracle.bwd(q, k, v, beta, S0, dO, dST)
    for name in ("dq", "dk", "dv", "dbeta", "dS0"):
        x = got[name].detach().double().cpu().numpy()
        assert np.all(np.isfinite(x))
        n = np.linalg.norm(ref[name])
        r = np.linalg.norm(x - ref[name]) / (n if n > 0 else 1.0)
        assert r <= 1e-4, f"{c} {name}: rel-fro {r:.3e}"
    assert efla.device_status() == 0

"""GPU parity of the time-split forward (efla_fwd_chunked_scan) against the fp64 oracle.

The split evaluation (segment maps, a scan over them, then every segment from its
start state) must reproduce the sequential recurrence, which the oracle runs
token by token over the whole sequence."""
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


def _dev(inp):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _scan(efla, inp, segments, **kw):
    g = _dev(inp)
    kw.setdefault("o_dtype", torch.float32)
    o, S = efla.fwd_chunked_scan(g["q"], g["k"], g["v"], g["beta"], g["S0"], segments=segments, **kw)
    torch.cuda.synchronize()
    return o, S


@pytest.mark.parametrize("T,segments", [(700, 3), (1000, 5), (512, 4), (640, 10), (130, 2)])
def test_scan_small(efla, T, segments):
    inp = workloads.small_fwd("bf16", B=2, T=T, H=2, d=128, seed=40 + segments)
    o, S = _scan(efla, inp, segments)
    o_ref, S_ref = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["S0"], threads=0)
    check(o, o_ref, in_dtype="bf16", what=f"scan o T={T} G={segments}")
    check(S, S_ref, in_dtype="bf16", what=f"scan S_T T={T} G={segments}")
    assert efla.device_status() == 0


def test_scan_stiff_norms_no_state_bf16_out(efla):
    inp = workloads.small_fwd("bf16", B=1, T=900, H=3, d=128, seed=8, key_norm="uniform", beta_mu=2.0, s0=False)
    o, S = _scan(efla, inp, 4, o_dtype=torch.bfloat16)
    o_ref, S_ref = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["beta"], None, threads=0)
    check(o, o_ref, in_dtype="bf16", what="scan stiff o (bf16)", out_bf16=True)
    check(S, S_ref, in_dtype="bf16", what="scan stiff S_T")


def test_scan_euler_unit_keys(efla):
    inp = workloads.small_fwd("bf16", B=1, T=600, H=2, d=128, seed=9)
    kf = inp["k"].float()
    inp["k"] = (kf / kf.norm(dim=-1, keepdim=True)).to(torch.bfloat16).contiguous()
    o, S = _scan(efla, inp, 3, update="euler")
    o_ref, S_ref = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["S0"], threads=0, update="euler")
    check(o, o_ref, in_dtype="bf16", what="scan euler o")
    check(S, S_ref, in_dtype="bf16", what="scan euler S_T")


def test_scan_matches_unsplit_and_one_piece_path(efla):
    inp = workloads.small_fwd("bf16", B=1, T=1500, H=4, d=128, seed=12)
    g = _dev(inp)
    o1, S1 = efla.fwd_chunked(g["q"], g["k"], g["v"], g["beta"], g["S0"], o_dtype=torch.float32)
    o2, S2 = _scan(efla, inp, 6)
    o3, S3 = _scan(efla, inp, 1)  # one piece: the plain path
    torch.cuda.synchronize()
    assert float((o1 - o2).norm() / o1.norm()) < 2e-3
    assert float((S1 - S2).norm() / S1.norm()) < 2e-3
    assert torch.equal(o1, o3) and torch.equal(S1, S3)


def test_scan_aliased_state_and_caller_workspace(efla):
    inp = workloads.small_fwd("bf16", B=1, T=400, H=2, d=128, seed=13)
    g = _dev(inp)
    need, G = efla.scan_workspace(1, 400, 2, segments=3)
    assert G == 3 and need > 0
    ws = torch.full((need,), 0x7f, dtype=torch.uint8, device=DEV)  # contents must not matter
    S = g["S0"].clone()
    o, S_out = efla.fwd_chunked_scan(g["q"], g["k"], g["v"], g["beta"], S, S_T=S, segments=3, workspace=ws, o_dtype=torch.float32)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["S0"], threads=0)
    check(o, o_ref, in_dtype="bf16", what="scan o, S0 aliased with S_T")
    check(S, S_ref, in_dtype="bf16", what="scan S_T aliased with S0")


def test_scan_stiff_config_sampled(efla):
    """The stiff/long configuration (B1 H16 T65536) split over the SMs; two heads replayed by the oracle."""
    cfg = workloads.FWD_WORKLOADS["stiff"]
    inp = workloads.make_fwd_inputs(cfg)
    o, S = _scan(efla, inp, 0)
    assert torch.isfinite(o).all() and torch.isfinite(S).all()
    for h in (0, 11):
        sl = (slice(0, 1), slice(None), slice(h, h + 1))
        S0 = None if inp["S0"] is None else inp["S0"][0:1, h:h + 1]
        o_ref, S_ref = oracle.fwd(inp["q"][sl], inp["k"][sl], inp["v"][sl], inp["beta"][sl], S0, threads=0)
        check(o[sl[0], sl[1], sl[2]], o_ref, in_dtype="bf16", what=f"stiff scan o head {h}")
        check(S[0:1, h:h + 1], S_ref, in_dtype="bf16", what=f"stiff scan S_T head {h}")
    assert efla.device_status() == 0

"""Device-side failure paths, exercised without any GPU fault.

* A bounded wait that runs out: a test hook makes a tensor-core kernel's issuing thread (the
  chunk kernel's, or the backward state pass's or gradient kernel's) wait on a barrier that
  nothing completes, with a short wait bound.  The kernel
  must abandon its work, let its own copies and tensor-core operations finish, record
  EFLA_ERR_DEVICE_TIMEOUT in the device status word and return; the context stays usable
  and the next normal call is correct.
* Malformed cu_seqlens (decreasing, or past T): the kernels write nothing for that
  sequence and record EFLA_ERR_INVALID_ARG; memory around the outputs is untouched, and a
  sequence that no other range overlaps is still correct.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TIMEOUT, INVALID = 4, 1


@pytest.fixture(scope="module")
def efla():
    import exact_delta_rule_gb300 as m
    from exact_delta_rule_gb300 import build
    build.build()
    m.load()
    yield m
    m.set_debug_stall(False)
    m.set_wait_limit_ns(0)


def _dev(inp):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


@pytest.mark.parametrize("T", [128, 150])
def test_wait_expiry_reports_timeout_and_context_survives(efla, T):
    inp = workloads.small_fwd("bf16", B=1, T=T, H=2, d=128, seed=71)
    g = _dev(inp)
    assert efla.device_status() == 0
    efla.set_wait_limit_ns(50_000_000)  # 50 ms
    efla.set_debug_stall(True)
    try:
        efla.fwd_chunked(g["q"], g["k"], g["v"], g["beta"], g["S0"], o_dtype=torch.float32)
        torch.cuda.synchronize()
    finally:
        efla.set_debug_stall(False)
        efla.set_wait_limit_ns(0)
    assert efla.device_status() == TIMEOUT
    assert efla.device_status() == 0  # reading clears the word
    o, S = efla.fwd_chunked(g["q"], g["k"], g["v"], g["beta"], g["S0"], o_dtype=torch.float32)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["S0"], threads=0)
    check(o, o_ref, in_dtype="bf16", what="o after a timed-out launch")
    check(S, S_ref, in_dtype="bf16", what="S_T after a timed-out launch")
    assert efla.device_status() == 0


@pytest.mark.parametrize("stall,which", [(2, "state pass"), (4, "gradient kernel")])
def test_backward_wait_expiry_reports_timeout_and_context_survives(efla, stall, which):
    """The same for the backward's two tensor-core kernels (bf16, d = 128): a stalled state
    pass or per-chunk gradient kernel records EFLA_ERR_DEVICE_TIMEOUT and returns; the next
    backward call is correct."""
    g = torch.Generator().manual_seed(79)
    B, T, H, d = 1, 150, 2, 128
    q = torch.randn((B, T, H, d), generator=g).to(torch.bfloat16)
    k = torch.nn.functional.normalize(torch.randn((B, T, H, d), generator=g), dim=-1).to(torch.bfloat16)
    v = torch.randn((B, T, H, d), generator=g).to(torch.bfloat16)
    beta = torch.sigmoid(torch.randn((B, T, H), generator=g))
    dO = torch.randn((B, T, H, d), generator=g)
    dST = torch.randn((B, H, d, d), generator=g)
    args = [x.to(DEV) for x in (q, k, v, beta)] + [None, dO.to(DEV), dST.to(DEV)]
    assert efla.device_status() == 0
    efla.set_wait_limit_ns(50_000_000)  # 50 ms
    efla.set_debug_stall(stall)
    try:
        efla.bwd_chunked(*args)
        torch.cuda.synchronize()
    finally:
        efla.set_debug_stall(False)
        efla.set_wait_limit_ns(0)
    assert efla.device_status() == TIMEOUT, which
    assert efla.device_status() == 0
    got = efla.bwd_chunked(*args)
    torch.cuda.synchronize()
    ref = oracle.bwd(q, k, v, beta, None, dO, dST)
    for name in ("dq", "dk", "dv", "dbeta"):
        a = got[name].double().cpu().numpy()
        r = np.linalg.norm(a - ref[name]) / np.linalg.norm(ref[name])
        assert r <= 1e-4, f"{name} after a timed-out {which}: rel-fro {r:.3e}"
    assert efla.device_status() == 0


@pytest.mark.parametrize("fn", ["chunked", "recurrent"])
@pytest.mark.parametrize("cu", [[0, 100, 60, 200], [0, 100, 300], [0, 120, 200, 201]])
def test_malformed_cu_seqlens_flagged(efla, fn, cu):
    T, H, d = 200, 2, 128
    N = len(cu) - 1
    inp = workloads.small_fwd("bf16", H=H, d=d, seed=73, lengths=[T])
    g = _dev(inp)
    pad, sentinel = 4096, 777.25
    ob = torch.full((pad + T * H * d + pad,), sentinel, device=DEV)
    sb = torch.full((pad + N * H * d * d + pad,), sentinel, device=DEV)
    o = ob[pad:pad + T * H * d].view(1, T, H, d)
    S = sb[pad:pad + N * H * d * d].view(N, H, d, d)
    cu_t = torch.tensor(cu, dtype=torch.int32, device=DEV)
    f = efla.fwd_chunked if fn == "chunked" else efla.fwd_recurrent
    assert efla.device_status() == 0
    f(g["q"], g["k"], g["v"], g["beta"], None, cu_t, o=o, S_T=S)
    torch.cuda.synchronize()
    assert efla.device_status() == INVALID
    for buf in (ob, sb):
        assert torch.all(buf[:pad] == sentinel) and torch.all(buf[-pad:] == sentinel)
    # When no other range overlaps it, the well-formed first sequence is still computed correctly
    # (ranges that overlap write the same rows of o: their outputs are unspecified).
    n0 = cu[1]
    if all(c >= n0 for c in cu[2:]):
        o_ref, S_ref = oracle.fwd(inp["q"][:, :n0], inp["k"][:, :n0], inp["v"][:, :n0], inp["beta"][:, :n0], None,
                                  threads=0)
        check(o[:, :n0], o_ref, in_dtype="bf16", what="o of the valid sequence")
        check(S[:1], S_ref, in_dtype="bf16", what="S_T of the valid sequence")
    assert efla.device_status() == 0


def test_error_strings(efla):
    assert efla.error_string(TIMEOUT).startswith("EFLA_ERR_DEVICE_TIMEOUT")
    assert efla.error_string(0) == "EFLA_OK"

"""The boundary calls with their exact C signatures, through ctypes on the raw library:
efla_fwd_chunked and efla_decode_step with o in the dtype of q, against the fp64 oracle.

With bf16 o the tolerance adds half a bf16 ulp of the reference value to the max-abs
bound: the output's own rounding (the outputs reach |o| ~ 27 on these workloads, where one
bf16 rounding alone is up to 0.06)."""
import ctypes

import pytest
import torch

import oracle
import workloads
from parity import check

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
BF16, F32 = 0, 1


@pytest.fixture(scope="module")
def lib():
    from exact_delta_rule_gb300 import build
    L = ctypes.CDLL(build.build())
    vp, ip = ctypes.c_void_p, ctypes.c_int
    L.efla_fwd_chunked.restype = ip
    L.efla_fwd_chunked.argtypes = [vp] * 8 + [ip] * 8 + [vp]
    L.efla_decode_step.restype = ip
    L.efla_decode_step.argtypes = [vp] * 6 + [ip] * 5 + [vp]
    L.efla_device_status.restype = ip
    L.efla_device_status.argtypes = [vp]
    L.efla_last_error.restype = ctypes.c_char_p
    return L


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("dtype,d,T,varlen", [("bf16", 128, 200, False), ("bf16", 128, 0, True),
                                              ("f32", 64, 130, False), ("bf16", 32, 77, False)])
def test_fwd_chunked_exact_signature(lib, dtype, d, T, varlen):
    if varlen:
        inp = workloads.small_fwd(dtype, H=2, d=d, seed=81, lengths=[65, 0, 130, 7])
    else:
        inp = workloads.small_fwd(dtype, B=2, T=T, H=3, d=d, seed=82)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    B, T, H, N = inp["B"], inp["T"], inp["H"], inp["N"]
    o = torch.empty((B, T, H, d), dtype=g["q"].dtype, device=DEV)
    S_T = torch.empty((N, H, d, d), dtype=torch.float32, device=DEV)
    code = lib.efla_fwd_chunked(_p(g["q"]), _p(g["k"]), _p(g["v"]), _p(g["beta"]), _p(g["S0"]),
                                _p(g["cu_seqlens"]), _p(o), _p(S_T), B, T, H, d, d, N,
                                BF16 if dtype == "bf16" else F32, 64, _stream())
    assert code == 0, lib.efla_last_error()
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["S0"], inp["cu_seqlens"], threads=0)
    check(o, o_ref, in_dtype=dtype, what="o", out_bf16=dtype == "bf16")
    check(S_T, S_ref, in_dtype=dtype, what="S_T")
    assert lib.efla_device_status(_stream()) == 0


def test_decode_step_exact_signature(lib):
    cfg = workloads.DecodeWorkload("d", 16, 8, 128, 128, 83, 3, 0.1)
    S0 = workloads.make_decode_state(cfg)
    S = S0.to(DEV)
    S_ref = S0.double().numpy()
    for step in range(3):
        inp = workloads.make_decode_step(step, cfg)
        g = {x: inp[x].to(DEV) for x in ("q", "k", "v", "beta")}
        o = torch.empty((cfg.B, cfg.H, cfg.dv), dtype=torch.bfloat16, device=DEV)
        code = lib.efla_decode_step(_p(g["q"]), _p(g["k"]), _p(g["v"]), _p(g["beta"]), _p(S), _p(o), cfg.B, cfg.H,
                                    cfg.dk, cfg.dv, BF16, _stream())
        assert code == 0, lib.efla_last_error()
        torch.cuda.synchronize()
        o_ref, S_ref = oracle.decode_step(inp["q"], inp["k"], inp["v"], inp["beta"], S_ref)
        check(o, o_ref, in_dtype="bf16", what=f"decode o step {step}", out_bf16=True)
        check(S, S_ref, in_dtype="bf16", what=f"decode S step {step}")

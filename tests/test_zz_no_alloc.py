"""efla_fwd_chunked_scan_static -- the time-split forward on the library's own fixed
scratch -- against efla_fwd_chunked_scan with a caller workspace and against the fp64
oracle, on two calls in a row.

The static call is for callers that cannot allocate device memory at call time (code
running inside a captured region or an allocator-free runtime, for instance); with its
outputs passed in it allocates nothing.  Both calls run the same kernels on the same
split, so their results are identical.  Collected last: it uses the library's scratch,
which persists between calls."""
import ctypes

import pytest
import torch

import oracle
import workloads
from parity import check

DEV = "cuda:0"


@pytest.fixture(scope="module")
def efla():
    import exact_delta_rule_gb300 as m
    from exact_delta_rule_gb300 import build
    build.build()
    m.load()
    return m


@pytest.mark.gpu
def test_static_scratch_matches_workspace_call_twice(efla):
    cases = [dict(B=1, T=1300, H=4, seed=61, segments=5), dict(B=2, T=777, H=3, seed=62, segments=0)]
    for c in cases:  # two calls in a row on the shared scratch, different sizes
        inp = workloads.small_fwd("bf16", B=c["B"], T=c["T"], H=c["H"], d=128, seed=c["seed"])
        g = {x: inp[x].to(DEV) for x in ("q", "k", "v", "beta", "S0")}
        o1, S1 = efla.fwd_chunked_scan(g["q"], g["k"], g["v"], g["beta"], g["S0"], segments=c["segments"],
                                       o_dtype=torch.float32)
        o2 = torch.empty_like(o1)
        S2 = torch.empty_like(S1)
        efla.fwd_chunked_scan_static(g["q"], g["k"], g["v"], g["beta"], g["S0"], segments=c["segments"],
                                     o=o2, S_T=S2)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(S1, S2), c
        o_ref, S_ref = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["S0"], threads=0)
        check(o2, o_ref, in_dtype="bf16", what=f"static o {c}")
        check(S2, S_ref, in_dtype="bf16", what=f"static S_T {c}")
    assert efla.device_status() == 0


@pytest.mark.gpu
def test_static_call_allocates_nothing(efla):
    """With o and S_T passed in, a static call changes neither torch's allocation count nor
    the device's free memory (after one call has resolved the scratch's address)."""
    inp = workloads.small_fwd("bf16", B=1, T=900, H=4, d=128, seed=63)
    g = {x: inp[x].to(DEV) for x in ("q", "k", "v", "beta", "S0")}
    o = torch.empty((1, 900, 4, 128), dtype=torch.bfloat16, device=DEV)
    S = torch.empty((1, 4, 128, 128), dtype=torch.float32, device=DEV)
    efla.fwd_chunked_scan_static(g["q"], g["k"], g["v"], g["beta"], g["S0"], segments=4, o=o, S_T=S)
    torch.cuda.synchronize()
    n0 = torch.cuda.memory_stats()["allocation.all.allocated"]
    free0, _ = torch.cuda.mem_get_info()
    efla.fwd_chunked_scan_static(g["q"], g["k"], g["v"], g["beta"], g["S0"], segments=4, o=o, S_T=S)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_stats()["allocation.all.allocated"] == n0
    assert free1 == free0
    o_ref, S_ref = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["S0"], threads=0)
    check(o, o_ref, in_dtype="bf16", what="static o (bf16)", out_bf16=True)
    check(S, S_ref, in_dtype="bf16", what="static S_T")


def test_static_scratch_rejects_oversize_split():
    """An explicit split needing more than the 32 MiB scratch is refused before any CUDA call."""
    from exact_delta_rule_gb300 import build
    L = ctypes.CDLL(build.build())
    vp, ip = ctypes.c_void_p, ctypes.c_int
    f = L.efla_fwd_chunked_scan_static
    f.restype = ip
    f.argtypes = [vp] * 7 + [ip] * 8 + [ip, vp]
    fake = [0x10000000 * (i + 1) for i in range(7)]
    fake[4] = None  # S0
    # B=1, H=300, 4 pieces: (3*4-2)*300 pieces of 64 KiB = 187.5 MiB
    assert f(*fake, 1, 256, 300, 128, 128, 0, 1, 4, 0, None) == 2
    L.efla_last_error.restype = ctypes.c_char_p
    assert b"static scratch" in L.efla_last_error()

"""efla_fwd_chunked_scan_static (library-owned scratch, no allocation per call) against
efla_fwd_chunked_scan with a caller workspace: the same kernels on the same split,
so the results are identical.  Collected last: it uses the library's fixed scratch."""
import ctypes

import pytest
import torch

import workloads

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
        o1, S1 = efla.fwd_chunked_scan(g["q"], g["k"], g["v"], g["beta"], g["S0"], segments=c["segments"])
        o2, S2 = efla.fwd_chunked_scan_static(g["q"], g["k"], g["v"], g["beta"], g["S0"], segments=c["segments"])
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(S1, S2), c
    assert efla.device_status() == 0


def test_static_scratch_rejects_oversize_split():
    """A split needing more than the 32 MiB scratch is refused before any CUDA call."""
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

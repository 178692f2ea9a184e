"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small cases compare every output element; the full-size workloads run in the
launch configuration the benchmark times and compare sampled (sequence, head)
units, each computed completely by the oracle.
"""
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


def _dev(inp):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _run(efla, fn, inp, o_dtype=torch.float32):
    g = _dev(inp)
    f = efla.fwd_chunked if fn == "chunked" else efla.fwd_recurrent
    o, S = f(g["q"], g["k"], g["v"], g["beta"], g["S0"], g["cu_seqlens"], o_dtype=o_dtype)
    torch.cuda.synchronize()
    return o, S


def _oracle(inp):
    return oracle.fwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["S0"], inp["cu_seqlens"], threads=0)


# ----------------------------------------------------------------- small cases
@pytest.mark.parametrize("fn", ["chunked", "recurrent"])
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("bf16", 32), ("f32", 32), ("f32", 128)])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
def test_fwd_small(efla, fn, dtype, d, T):
    inp = workloads.small_fwd(dtype, B=2, T=T, H=3, d=d, seed=100 + T + d, s0=(T % 2 == 1))
    o, S = _run(efla, fn, inp)
    o_ref, S_ref = _oracle(inp)
    check(o, o_ref, in_dtype=dtype, what=f"o {fn} {dtype} d{d} T{T}")
    check(S, S_ref, in_dtype=dtype, what=f"S_T {fn} {dtype} d{d} T{T}")


@pytest.mark.parametrize("chunk", [16, 32, 64])
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64), ("bf16", 32), ("f32", 128)])
def test_fwd_chunk_lengths(efla, chunk, dtype, d):
    """Every chunk length the boundary accepts (16 and 32 run the CUDA-core chunkwise kernel,
    64 the tensor-core kernel for bf16 d128), ragged lengths and a packed batch."""
    inp = workloads.small_fwd(dtype, B=2, T=150, H=2, d=d, seed=300 + chunk + d)
    g = _dev(inp)
    o, S = efla.fwd_chunked(g["q"], g["k"], g["v"], g["beta"], g["S0"], chunk=chunk, o_dtype=torch.float32)
    torch.cuda.synchronize()
    o_ref, S_ref = _oracle(inp)
    check(o, o_ref, in_dtype=dtype, what=f"o chunk {chunk}")
    check(S, S_ref, in_dtype=dtype, what=f"S_T chunk {chunk}")
    inp = workloads.small_fwd(dtype, H=2, d=d, seed=400 + chunk, lengths=[31, 0, 70, 16, 5])
    g = _dev(inp)
    o, S = efla.fwd_chunked(g["q"], g["k"], g["v"], g["beta"], g["S0"], g["cu_seqlens"], chunk=chunk,
                            o_dtype=torch.float32)
    torch.cuda.synchronize()
    o_ref, S_ref = _oracle(inp)
    check(o, o_ref, in_dtype=dtype, what=f"o varlen chunk {chunk}")
    check(S, S_ref, in_dtype=dtype, what=f"S_T varlen chunk {chunk}")


@pytest.mark.parametrize("fn", ["chunked", "recurrent"])
def test_fwd_bf16_output(efla, fn):
    inp = workloads.small_fwd("bf16", B=2, T=300, H=2, d=128, seed=7)
    o, S = _run(efla, fn, inp, o_dtype=torch.bfloat16)
    assert o.dtype == torch.bfloat16
    o_ref, S_ref = _oracle(inp)
    check(o, o_ref, in_dtype="bf16", what="o bf16", out_bf16=True)
    check(S, S_ref, in_dtype="bf16", what="S_T")


@pytest.mark.parametrize("fn", ["chunked", "recurrent"])
def test_fwd_varlen_small(efla, fn):
    lens = [1, 0, 64, 65, 130, 7, 0, 200, 63]
    inp = workloads.small_fwd("bf16", H=2, d=128, seed=9, lengths=lens)
    o, S = _run(efla, fn, inp)
    o_ref, S_ref = _oracle(inp)
    check(o, o_ref, in_dtype="bf16", what="o varlen")
    check(S, S_ref, in_dtype="bf16", what="S_T varlen")
    # empty sequences return their initial state exactly
    np.testing.assert_array_equal(to64(S[1]), to64(inp["S0"][1]))
    np.testing.assert_array_equal(to64(S[6]), to64(inp["S0"][6]))


@pytest.mark.parametrize("fn", ["chunked", "recurrent"])
def test_fwd_stiff_norms_small(efla, fn):
    inp = workloads.small_fwd("bf16", B=1, T=700, H=2, d=128, seed=5, key_norm="uniform", beta_mu=2.0)
    o, S = _run(efla, fn, inp)
    o_ref, S_ref = _oracle(inp)
    check(o, o_ref, in_dtype="bf16", what="o stiff")
    check(S, S_ref, in_dtype="bf16", what="S_T stiff")


def test_zero_keys_and_zero_beta(efla):
    inp = workloads.small_fwd("bf16", B=1, T=130, H=2, d=128, seed=21)
    inp["k"][:, ::5] = 0
    inp["beta"][:, 3::7] = 0
    for fn in ("chunked", "recurrent"):
        o, S = _run(efla, fn, inp)
        o_ref, S_ref = _oracle(inp)
        check(o, o_ref, in_dtype="bf16", what=f"o zero keys {fn}")
        check(S, S_ref, in_dtype="bf16", what=f"S_T zero keys {fn}")


def test_empty_inputs(efla):
    inp = workloads.small_fwd("bf16", B=2, T=0, H=2, d=128, seed=1)
    o, S = _run(efla, "chunked", inp)
    assert o.shape[1] == 0
    np.testing.assert_array_equal(to64(S), to64(inp["S0"]))
    inp = workloads.small_fwd("bf16", B=2, T=0, H=2, d=128, seed=1, s0=False)
    o, S = _run(efla, "chunked", inp)
    assert float(S.abs().max()) == 0.0


def test_state_alias_and_no_state(efla):
    inp = workloads.small_fwd("bf16", B=2, T=100, H=2, d=128, seed=31)
    g = _dev(inp)
    S = g["S0"].clone()
    o, S_out = efla.fwd_chunked(g["q"], g["k"], g["v"], g["beta"], S, S_T=S, o_dtype=torch.float32)
    torch.cuda.synchronize()
    assert S_out.data_ptr() == S.data_ptr()
    o_ref, S_ref = _oracle(inp)
    check(S, S_ref, in_dtype="bf16", what="S_T aliased with S0")
    o2, none = efla.fwd_chunked(g["q"], g["k"], g["v"], g["beta"], g["S0"], return_state=False, o_dtype=torch.float32)
    torch.cuda.synchronize()
    assert none is None
    check(o2, o_ref, in_dtype="bf16", what="o without S_T")


def test_guard_bands_untouched(efla):
    inp = workloads.small_fwd("bf16", B=2, T=77, H=3, d=128, seed=41)
    g = _dev(inp)
    B, T, H, d = 2, 77, 3, 128
    pad = 4096
    sentinel = 1234.5
    ob = torch.full((pad + B * T * H * d + pad,), sentinel, device=DEV)
    sb = torch.full((pad + B * H * d * d + pad,), sentinel, device=DEV)
    o = ob[pad:pad + B * T * H * d].view(B, T, H, d)
    S = sb[pad:pad + B * H * d * d].view(B, H, d, d)
    efla.fwd_chunked(g["q"], g["k"], g["v"], g["beta"], g["S0"], o=o, S_T=S)
    torch.cuda.synchronize()
    for buf in (ob, sb):
        assert torch.all(buf[:pad] == sentinel) and torch.all(buf[-pad:] == sentinel)
    o_ref, S_ref = _oracle(inp)
    check(o, o_ref, in_dtype="bf16", what="o guard")


def test_deterministic(efla):
    inp = workloads.small_fwd("bf16", B=2, T=333, H=2, d=128, seed=51)
    a = _run(efla, "chunked", inp)
    b = _run(efla, "chunked", inp)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# ---------------------------------------------------------------------- decode
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64), (32, 32), (128, 32), (32, 128)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_small(efla, dk, dv, dtype):
    cfg = workloads.DecodeWorkload("d", 3, 5, dk, dv, 77, 3, 0.1)
    S0 = workloads.make_decode_state(cfg)
    S = S0.to(DEV)
    S_ref = S0.double().numpy()
    for step in range(3):
        inp = workloads.make_decode_step(step, cfg)
        if dtype == "f32":
            inp = {k: v.float() for k, v in inp.items()}
        o = efla.decode_step(*(inp[x].to(DEV) for x in ("q", "k", "v", "beta")), S, o_dtype=torch.float32)
        torch.cuda.synchronize()
        o_ref, S_ref = oracle.decode_step(inp["q"], inp["k"], inp["v"], inp["beta"], S_ref)
        check(o, o_ref, in_dtype=dtype, what=f"decode o step {step}")
        check(S, S_ref, in_dtype=dtype, what=f"decode S step {step}")


def test_decode_full_chained(efla):
    """B256 H32 d128, 1000 chained steps; all heads run on the GPU, sampled heads
    are replayed by the oracle and compared after steps 1, 10 and 1000."""
    cfg = workloads.DECODE
    S0 = workloads.make_decode_state(cfg)
    S = S0.to(DEV)
    rng = np.random.default_rng(0)
    bs = rng.choice(cfg.B, 8, replace=False)
    hs = rng.choice(cfg.H, 8, replace=False)
    S_ref = S0[bs][:, hs].double().numpy()
    o = torch.empty((cfg.B, cfg.H, cfg.dv), device=DEV)
    for step in range(cfg.steps):
        inp = workloads.make_decode_step(step, cfg)
        efla.decode_step(*(inp[x].to(DEV, non_blocking=True) for x in ("q", "k", "v", "beta")), S, o=o)
        sub = {x: inp[x][bs][:, hs] for x in ("q", "k", "v", "beta")}
        o_ref, S_ref = oracle.decode_step(sub["q"], sub["k"], sub["v"], sub["beta"], S_ref)
        if step + 1 in (1, 10, cfg.steps):
            torch.cuda.synchronize()
            got_S = S[torch.as_tensor(bs)][:, torch.as_tensor(hs)]
            got_o = o[torch.as_tensor(bs)][:, torch.as_tensor(hs)]
            check(got_o, o_ref, in_dtype="bf16", what=f"decode o after {step + 1}")
            check(got_S, S_ref, in_dtype="bf16", what=f"decode S after {step + 1}")
    assert torch.isfinite(S).all()
    assert efla.device_status() == 0


# ------------------------------------------------------------ full workloads
def test_tiny_config(efla):
    cfg = workloads.FWD_WORKLOADS["tiny"]
    inp = workloads.make_fwd_inputs(cfg)
    o, S = _run(efla, "chunked", inp)
    o_ref, S_ref = _oracle(inp)
    check(o, o_ref, in_dtype="f32", what="tiny o")
    check(S, S_ref, in_dtype="f32", what="tiny S_T")


def _sampled(inp, units):
    """Oracle on selected (sequence, head) units of a full-size input."""
    out = []
    cu = inp["cu_seqlens"]
    for (n, h) in units:
        if cu is None:
            sl = (slice(n, n + 1), slice(None), slice(h, h + 1))
        else:
            t0, t1 = int(cu[n]), int(cu[n + 1])
            sl = (slice(0, 1), slice(t0, t1), slice(h, h + 1))
        S0 = None if inp["S0"] is None else inp["S0"][n:n + 1, h:h + 1]
        o_ref, S_ref = oracle.fwd(inp["q"][sl], inp["k"][sl], inp["v"][sl], inp["beta"][sl], S0, threads=0)
        out.append((sl, o_ref, S_ref))
    return out


@pytest.mark.parametrize("name,units", [
    ("lm", [(0, 0), (3, 7), (7, 15), (5, 2)]),
    ("stiff", [(0, 0), (0, 11)]),
    ("varlen", [(0, 0), (17, 3), (40, 7), (63, 5)]),
])
def test_full_workload_sampled(efla, name, units):
    cfg = workloads.FWD_WORKLOADS[name]
    inp = workloads.make_fwd_inputs(cfg)
    o, S = _run(efla, "chunked", inp)
    assert torch.isfinite(o).all() and torch.isfinite(S).all()
    for (sl, o_ref, S_ref), (n, h) in zip(_sampled(inp, units), units):
        got_o = o[sl[0], sl[1], sl[2]]
        check(got_o, o_ref, in_dtype="bf16", what=f"{name} o unit {(n, h)}")
        check(S[n:n + 1, h:h + 1], S_ref, in_dtype="bf16", what=f"{name} S_T unit {(n, h)}")
    assert efla.device_status() == 0


def test_chunked_matches_recurrent_on_lm_shape(efla):
    """Two independent GPU evaluations agree on the full LM workload (all heads)."""
    inp = workloads.make_fwd_inputs(workloads.FWD_WORKLOADS["lm"])
    o1, S1 = _run(efla, "chunked", inp)
    o2, S2 = _run(efla, "recurrent", inp)
    rel_o = float((o1 - o2).norm() / o2.norm())
    rel_S = float((S1 - S2).norm() / S2.norm())
    assert rel_o <= 5e-3 and rel_S <= 5e-3, (rel_o, rel_S)
    assert float((o1 - o2).abs().max()) <= 4e-2

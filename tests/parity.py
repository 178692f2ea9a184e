"""Tolerance checks of the CUDA path against the fp64 oracle.

Tolerances (stated for the method's workloads): bf16 inputs with fp32
accumulation -- max-abs error <= 2e-2 and relative Frobenius error <= 5e-3 on
o and S_T; fp32 inputs -- relative Frobenius error <= 1e-4.  When o is
requested in bf16 its own rounding is added to the max-abs bound (half a bf16
ulp of the reference value), since a bf16 output of magnitude above 10 cannot
be closer than that to the exact value.
"""
import numpy as np
import torch

MAX_ABS_BF16 = 2e-2
REL_FRO_BF16 = 5e-3
REL_FRO_F32 = 1e-4


def to64(x):
    if isinstance(x, torch.Tensor):
        return x.detach().double().cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def bf16_half_ulp(ref: np.ndarray) -> np.ndarray:
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


def errors(got, ref):
    got, ref = to64(got), to64(ref)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite values in the GPU result"
    d = np.abs(got - ref)
    nr = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / nr if nr > 0 else np.linalg.norm(got - ref)
    return d, rel


def check(got, ref, *, in_dtype: str, what: str, out_bf16: bool = False):
    d, rel = errors(got, ref)
    ref64 = to64(ref)
    if in_dtype == "f32":
        assert rel <= REL_FRO_F32, f"{what}: rel-fro {rel:.3e} > {REL_FRO_F32}"
        return float(d.max(initial=0.0)), float(rel)
    bound = MAX_ABS_BF16 + (bf16_half_ulp(ref64) if out_bf16 else 0.0)
    excess = d - bound
    worst = float(excess.max(initial=-1.0))
    assert worst <= 0, f"{what}: max-abs excess {worst:.3e} (max err {d.max():.3e})"
    assert rel <= REL_FRO_BF16, f"{what}: rel-fro {rel:.3e} > {REL_FRO_BF16}"
    return float(d.max(initial=0.0)), float(rel)

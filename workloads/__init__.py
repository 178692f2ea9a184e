"""Seeded synthetic inputs for the EFLA token mixer.

This module is shared by the oracle-side tests and the GPU path's tests and
benchmark.  It only draws random numbers and shapes them (key directions and
key norms, step sizes, initial states, sequence lengths); it holds none of the
method's arithmetic (no norms are consumed, no gate, no state update).

Shapes follow the activation layout of a linear-attention token mixer:
q, k: [B, T, H, d_k]; v: [B, T, H, d_v]; beta: [B, T, H]; S0: [N, H, d_k, d_v].
For packed variable-length batches B == 1 and ``cu_seqlens`` ([N+1], int32)
holds the sequence boundaries along T.

Distributions are those of the five workloads used for parity and
measurement:

* ``tiny``      B1 H2 T256 d32, fp32, q,k,v ~ N(0,1), key norms LogNormal(0,0.5),
                beta = sigmoid(N(0,1)), S0 = 0, chunk 64.
* ``lm``        B8 H16 T2048 d128, bf16, q,v ~ N(0,1), unit key directions times
                LogNormal(0,0.5) norms, beta = sigmoid(N(0,1)), S0 = 0.
* ``stiff``     B1 H16 T65536 d128, bf16, unit key directions times U[0.1,10]
                norms, beta = sigmoid(N(2,1)), S0 ~ 0.1 N(0,1).
* ``decode``    B256 H32 d128 single-token steps, bf16 q,k,v ~ N(0,1),
                beta = sigmoid(N(0,1)), fp32 state S ~ 0.1 N(0,1).
* ``varlen``    64 sequences with lengths U{1..8192} packed along T, H8 d128 bf16,
                unit key directions times LogNormal(0,1) norms,
                beta = sigmoid(N(0,1)), per-sequence S0 ~ 0.1 N(0,1).

The shape of the language-model workload stands in for the language-model
experiments the method was evaluated on; no dataset item is used.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import torch

__all__ = [
    "FwdWorkload", "DecodeWorkload", "FWD_WORKLOADS", "DECODE", "make_fwd_inputs",
    "make_decode_state", "make_decode_step", "varlen_lengths", "small_fwd",
]


@dataclasses.dataclass(frozen=True)
class FwdWorkload:
    name: str
    B: int
    T: int
    H: int
    dk: int
    dv: int
    dtype: str               # "f32" or "bf16"
    seed: int
    key_norm: str            # "lognormal" or "uniform"
    key_norm_a: float        # sigma for lognormal, low for uniform
    key_norm_b: float        # unused for lognormal, high for uniform
    beta_mu: float           # beta = sigmoid(N(beta_mu, 1))
    s0_std: float            # 0 means S0 is absent (zeros)
    chunk: int = 64
    n_seqs: int = 0          # > 0: packed variable-length batch of this many sequences
    max_len: int = 0         # lengths ~ U{1..max_len}

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    H: int
    dk: int
    dv: int
    seed: int
    steps: int
    s_std: float


FWD_WORKLOADS = {
    "tiny": FwdWorkload("tiny", 1, 256, 2, 32, 32, "f32", 1, "lognormal", 0.5, 0.0, 0.0, 0.0),
    "lm": FwdWorkload("lm", 8, 2048, 16, 128, 128, "bf16", 2, "lognormal", 0.5, 0.0, 0.0, 0.0),
    "stiff": FwdWorkload("stiff", 1, 65536, 16, 128, 128, "bf16", 3, "uniform", 0.1, 10.0, 2.0, 0.1),
    "varlen": FwdWorkload("varlen", 1, 0, 8, 128, 128, "bf16", 5, "lognormal", 1.0, 0.0, 0.0, 0.1,
                          n_seqs=64, max_len=8192),
}

DECODE = DecodeWorkload("decode", 256, 32, 128, 128, 4, 1000, 0.1)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def varlen_lengths(cfg: FwdWorkload) -> list:
    """Sequence lengths of a packed workload, drawn U{1..max_len} from its seed."""
    g = _gen(cfg.seed * 7919 + 1)
    return torch.randint(1, cfg.max_len + 1, (cfg.n_seqs,), generator=g).tolist()


def _keys(g: torch.Generator, shape, cfg: FwdWorkload) -> torch.Tensor:
    """Unit directions times a per-token norm drawn from the workload's law."""
    direction = torch.randn(shape, generator=g, dtype=torch.float32)
    direction = direction / direction.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    if cfg.key_norm == "lognormal":
        norm = torch.exp(cfg.key_norm_a * torch.randn(shape[:-1], generator=g))
    else:
        norm = cfg.key_norm_a + (cfg.key_norm_b - cfg.key_norm_a) * torch.rand(shape[:-1], generator=g)
    return direction * norm.unsqueeze(-1)


def make_fwd_inputs(cfg: FwdWorkload, *, lengths: Optional[Sequence[int]] = None,
                    T: Optional[int] = None, B: Optional[int] = None, H: Optional[int] = None,
                    seed: Optional[int] = None) -> dict:
    """Draw the inputs of a chunked-forward workload on the CPU.

    Returns a dict with q, k, v (cfg dtype), beta (fp32), S0 (fp32 or None),
    cu_seqlens (int32 or None) and the sizes B, T, H, N.  ``T``, ``B``, ``H``,
    ``lengths`` and ``seed`` override the workload's sizes to make smaller
    cases with the same value distributions.
    """
    seed = cfg.seed if seed is None else seed
    g = _gen(seed)
    H = cfg.H if H is None else H
    if cfg.n_seqs or lengths is not None:
        lens = list(varlen_lengths(cfg) if lengths is None else lengths)
        B_, T_ = 1, int(sum(lens))
        cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
        N = len(lens)
    else:
        B_ = cfg.B if B is None else B
        T_ = cfg.T if T is None else T
        cu = None
        N = B_
    q = torch.randn((B_, T_, H, cfg.dk), generator=g)
    k = _keys(g, (B_, T_, H, cfg.dk), cfg)
    v = torch.randn((B_, T_, H, cfg.dv), generator=g)
    beta = torch.sigmoid(cfg.beta_mu + torch.randn((B_, T_, H), generator=g))
    S0 = None
    if cfg.s0_std > 0:
        S0 = cfg.s0_std * torch.randn((N, H, cfg.dk, cfg.dv), generator=g)
    dt = cfg.torch_dtype
    return {
        "q": q.to(dt).contiguous(), "k": k.to(dt).contiguous(), "v": v.to(dt).contiguous(),
        "beta": beta.float().contiguous(), "S0": S0, "cu_seqlens": cu,
        "B": B_, "T": T_, "H": H, "N": N, "dk": cfg.dk, "dv": cfg.dv, "dtype": cfg.dtype,
    }


def small_fwd(dtype: str = "bf16", *, B: int = 2, T: int = 200, H: int = 3, d: int = 128,
              seed: int = 11, s0: bool = True, key_norm: str = "lognormal",
              lengths: Optional[Sequence[int]] = None, beta_mu: float = 0.0) -> dict:
    """A small forward case with the language-model value laws (for parity tests)."""
    cfg = FwdWorkload("small", B, T, H, d, d, dtype, seed, key_norm,
                      0.5 if key_norm == "lognormal" else 0.1,
                      0.0 if key_norm == "lognormal" else 10.0, beta_mu, 0.1 if s0 else 0.0)
    return make_fwd_inputs(cfg, lengths=lengths)


def make_decode_state(cfg: DecodeWorkload = DECODE, *, B: Optional[int] = None,
                      H: Optional[int] = None) -> torch.Tensor:
    """Initial fp32 state S ~ s_std * N(0,1), [B, H, d_k, d_v]."""
    B = cfg.B if B is None else B
    H = cfg.H if H is None else H
    g = _gen(cfg.seed)
    return (cfg.s_std * torch.randn((B, H, cfg.dk, cfg.dv), generator=g)).contiguous()


def make_decode_step(step: int, cfg: DecodeWorkload = DECODE, *, B: Optional[int] = None,
                     H: Optional[int] = None) -> dict:
    """Inputs of decode step ``step`` (0-based): bf16 q,k,v ~ N(0,1), beta = sigmoid(N(0,1))."""
    B = cfg.B if B is None else B
    H = cfg.H if H is None else H
    g = _gen((cfg.seed << 32) + step)
    q = torch.randn((B, H, cfg.dk), generator=g)
    k = torch.randn((B, H, cfg.dk), generator=g)
    v = torch.randn((B, H, cfg.dv), generator=g)
    beta = torch.sigmoid(torch.randn((B, H), generator=g))
    return {"q": q.to(torch.bfloat16).contiguous(), "k": k.to(torch.bfloat16).contiguous(),
            "v": v.to(torch.bfloat16).contiguous(), "beta": beta.float().contiguous()}


def make_decode_tokens(m: int, cfg: DecodeWorkload = DECODE, *, first_step: int = 0, B: Optional[int] = None,
                       H: Optional[int] = None) -> dict:
    """Inputs of m consecutive decode steps stacked along a token axis: q, k [B, m, H, d_k],
    v [B, m, H, d_v] (bf16), beta [B, m, H] (fp32) -- token t is decode step first_step + t."""
    B_ = cfg.B if B is None else B
    H_ = cfg.H if H is None else H
    if m == 0:
        e = lambda d: torch.empty((B_, 0, H_, d), dtype=torch.bfloat16)
        return {"q": e(cfg.dk), "k": e(cfg.dk), "v": e(cfg.dv), "beta": torch.empty((B_, 0, H_))}
    steps = [make_decode_step(first_step + t, cfg, B=B, H=H) for t in range(m)]
    out = {}
    for x in ("q", "k", "v", "beta"):
        out[x] = torch.stack([s[x] for s in steps], dim=1).contiguous()
    return out

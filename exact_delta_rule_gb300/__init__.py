"""Python binding of libefla.so -- the GB300 (sm_103a) EFLA token mixer.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/efla.h``.  PyTorch provides
device memory and streams.  If the shared library is missing, importing
works but every call raises ``RuntimeError`` -- there is no fallback path.

    o, S_T = fwd_chunked(q, k, v, beta, S0=None, cu_seqlens=None)
    o      = decode_step(q, k, v, beta, S)        # S updated in place
    o      = decode_tokens(q, k, v, beta, S)      # m tokens per sequence, S in place

Semantics (per head): lambda = ||k||^2, alpha = (1 - e^{-beta*lambda})/lambda,
S <- (I - alpha k k^T) S + alpha k v^T, o = S^T q with the updated S.
["Exact Flow Linear Attention" (gist.science), Metodologia 3;
 "Error-Free Linear Attention is a Free Lunch" (howistudyai), Steps 1-3.]
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

__all__ = ["EflaError", "lib_path", "load", "fwd_chunked", "fwd_chunked_scan", "fwd_chunked_scan_static",
           "scan_workspace", "fwd_recurrent", "decode_step", "decode_tokens", "bwd_recurrent", "bwd_chunked",
           "fwd_chunked_train",
           "bwd_workspace", "prep", "device_status", "error_string", "set_wait_limit_ns", "set_debug_stall", "abi_version", "STATUS", "UPDATES"]

_PKG = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_PKG, "libefla.so")

UPDATES = {"exact": 0, "euler": 1}
STATUS = {0: "EFLA_OK", 1: "EFLA_ERR_INVALID_ARG", 2: "EFLA_ERR_UNSUPPORTED", 3: "EFLA_ERR_CUDA",
          4: "EFLA_ERR_DEVICE_TIMEOUT"}
BF16, F32 = 0, 1

_lock = threading.Lock()
_lib = None


class EflaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


def load():
    """Load libefla.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(lib_path):
            raise RuntimeError(f"{lib_path} is not built; run `python -c 'import __graft_entry__ as g; "
                               f"g.build()'` (there is no non-CUDA fallback)")
        L = ctypes.CDLL(lib_path)
        vp, ip = ctypes.c_void_p, ctypes.c_int
        L.efla_fwd_chunked.restype = ip
        L.efla_fwd_chunked.argtypes = [vp] * 8 + [ip] * 8 + [vp]
        L.efla_fwd_recurrent.restype = ip
        L.efla_fwd_recurrent.argtypes = [vp] * 8 + [ip] * 7 + [vp]
        L.efla_decode_step.restype = ip
        L.efla_decode_step.argtypes = [vp] * 6 + [ip] * 5 + [vp]
        L.efla_fwd_chunked_ex.restype = ip
        L.efla_fwd_chunked_ex.argtypes = [vp] * 8 + [ip] * 10 + [vp]
        L.efla_fwd_recurrent_ex.restype = ip
        L.efla_fwd_recurrent_ex.argtypes = [vp] * 8 + [ip] * 9 + [vp]
        L.efla_decode_step_ex.restype = ip
        L.efla_decode_step_ex.argtypes = [vp] * 6 + [ip] * 7 + [vp]
        L.efla_fwd_chunked_scan.restype = ip
        L.efla_fwd_chunked_scan.argtypes = [vp] * 7 + [ip] * 8 + [vp, ctypes.c_size_t, ip, vp]
        L.efla_fwd_chunked_scan_static.restype = ip
        L.efla_fwd_chunked_scan_static.argtypes = [vp] * 7 + [ip] * 8 + [ip, vp]
        L.efla_fwd_scan_workspace.restype = ip
        L.efla_fwd_scan_workspace.argtypes = [ip] * 6 + [ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ip)]
        L.efla_bwd_recurrent.restype = ip
        L.efla_bwd_recurrent.argtypes = [vp] * 12 + [ip] * 7 + [vp]
        L.efla_bwd_chunked.restype = ip
        L.efla_bwd_chunked.argtypes = [vp] * 12 + [ip] * 7 + [vp, ctypes.c_size_t, vp]
        L.efla_bwd_workspace.restype = ip
        L.efla_bwd_workspace.argtypes = [ip] * 5 + [ctypes.POINTER(ctypes.c_size_t)]
        L.efla_bwd_chunked_saved.restype = ip
        L.efla_bwd_chunked_saved.argtypes = [vp] * 12 + [ip] * 7 + [vp, ctypes.c_size_t, vp]
        L.efla_fwd_chunked_train.restype = ip
        L.efla_fwd_chunked_train.argtypes = [vp] * 7 + [ip] * 7 + [vp, ctypes.c_size_t, vp]
        L.efla_decode_tokens.restype = ip
        L.efla_decode_tokens.argtypes = [vp] * 6 + [ip] * 8 + [vp]
        L.efla_prep.restype = ip
        L.efla_prep.argtypes = [vp] * 7 + [ctypes.c_longlong] + [ip] * 4 + [vp]
        L.efla_device_status.restype = ip
        L.efla_device_status.argtypes = [vp]
        L.efla_get_error_string.restype = ctypes.c_char_p
        L.efla_get_error_string.argtypes = [ip]
        L.efla_debug_set_wait_limit_ns.restype = None
        L.efla_debug_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
        L.efla_debug_set_stall.restype = None
        L.efla_debug_set_stall.argtypes = [ip]
        L.efla_last_error.restype = ctypes.c_char_p
        L.efla_last_error.argtypes = []
        L.efla_abi_version.restype = ip
        L.efla_abi_version.argtypes = []
        _lib = L
        return L


def abi_version() -> int:
    return load().efla_abi_version()


def _check(code: int):
    if code != 0:
        raise EflaError(code, load().efla_last_error().decode())


def _dt(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return BF16
    if t == torch.float32:
        return F32
    raise EflaError(1, f"unsupported dtype {t}")


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: Optional[torch.Tensor], name: str):
    if t is None:
        return
    if not t.is_cuda:
        raise EflaError(1, f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise EflaError(1, f"{name} must be contiguous")


def _check_fwd_inputs(q, k, v, beta, S0, N=None):
    """Shape and dtype checks shared by every forward wrapper (made before the device and
    layout checks); returns (B, T, H, dk, dv, N)."""
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4 or v.shape[:3] != q.shape[:3] \
            or beta.shape != q.shape[:3]:
        raise EflaError(1, f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)} "
                           f"beta{tuple(beta.shape)}")
    if q.dtype != k.dtype or q.dtype != v.dtype or beta.dtype != torch.float32:
        raise EflaError(1, "q, k, v must share a dtype and beta must be float32")
    _dt(q.dtype)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    N = B if N is None else N
    if S0 is not None and (S0.dtype != torch.float32 or tuple(S0.shape) != (N, H, dk, dv)):
        raise EflaError(1, f"S0 must be float32 [{N},{H},{dk},{dv}]")
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (beta, "beta"), (S0, "S0")):
        _need(t, n)
    return B, T, H, dk, dv, N


def _outputs(q, o, S_T, o_dtype, return_state, B, T, H, dk, dv, N):
    """The output tensors of a forward call: given ones are checked, missing ones allocated."""
    o_dtype = q.dtype if o_dtype is None else o_dtype
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=o_dtype, device=q.device)
    else:
        _need(o, "o")
        if tuple(o.shape) != (B, T, H, dv):
            raise EflaError(1, f"o must be [{B},{T},{H},{dv}]")
        _dt(o.dtype)
    if S_T is None and return_state:
        S_T = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device)
    elif S_T is not None:
        _need(S_T, "S_T")
        if S_T.dtype != torch.float32 or tuple(S_T.shape) != (N, H, dk, dv):
            raise EflaError(1, f"S_T must be float32 [{N},{H},{dk},{dv}]")
    return o, S_T


def _fwd(entry, q, k, v, beta, S0, cu_seqlens, o, S_T, o_dtype, chunk, stream, return_state, update="exact"):
    L = load()
    _need(cu_seqlens, "cu_seqlens")
    if cu_seqlens is not None:
        if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1:
            raise EflaError(1, "cu_seqlens must be a 1-D int32 tensor")
        N = cu_seqlens.shape[0] - 1
    else:
        N = None
    B, T, H, dk, dv, N = _check_fwd_inputs(q, k, v, beta, S0, N)
    o, st = _outputs(q, o, S_T, o_dtype, return_state, B, T, H, dk, dv, N)
    args = [_p(q), _p(k), _p(v), _p(beta), _p(S0), _p(cu_seqlens), _p(o), _p(st), B, T, H, dk, dv, N,
            _dt(q.dtype), _dt(o.dtype)]
    if update not in UPDATES:
        raise EflaError(1, f"unknown update rule {update!r}")
    if entry == "chunked":
        _check(L.efla_fwd_chunked_ex(*args, int(chunk), UPDATES[update], _stream(stream)))
    else:
        _check(L.efla_fwd_recurrent_ex(*args, UPDATES[update], _stream(stream)))
    return o, st


def fwd_chunked(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
                S0: Optional[torch.Tensor] = None, cu_seqlens: Optional[torch.Tensor] = None, *,
                o: Optional[torch.Tensor] = None, S_T: Optional[torch.Tensor] = None,
                o_dtype: Optional[torch.dtype] = None, chunk: int = 64, stream=None,
                return_state: bool = True, update: str = "exact") -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """EFLA forward, chunkwise.  Layouts as in ``efla_fwd_chunked`` (include/efla.h).

    q, k [B,T,H,dk], v [B,T,H,dv] (bf16 or fp32); beta [B,T,H] fp32; S0 [N,H,dk,dv] fp32;
    cu_seqlens [N+1] int32 (then B == 1).  Returns (o [B,T,H,dv] in ``o_dtype`` -- q's dtype
    unless given, or the dtype of a given ``o`` --, S_T [N,H,dk,dv] fp32 or None when
    ``return_state`` is False).  ``update="euler"`` runs the delta-rule (DeltaNet) gate
    alpha = beta through the same kernels.
    """
    return _fwd("chunked", q, k, v, beta, S0, cu_seqlens, o, S_T, o_dtype, chunk, stream, return_state, update)


def scan_workspace(B: int, T: int, H: int, dk: int = 128, dv: int = 128, segments: int = 0) -> Tuple[int, int]:
    """(workspace bytes, pieces per sequence) of ``fwd_chunked_scan`` (``efla_fwd_scan_workspace``)."""
    L = load()
    nb, g = ctypes.c_size_t(0), ctypes.c_int(0)
    _check(L.efla_fwd_scan_workspace(B, T, H, dk, dv, int(segments), ctypes.byref(nb), ctypes.byref(g)))
    return nb.value, g.value


def fwd_chunked_scan(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
                     S0: Optional[torch.Tensor] = None, *, segments: int = 0,
                     workspace: Optional[torch.Tensor] = None, o: Optional[torch.Tensor] = None,
                     S_T: Optional[torch.Tensor] = None, o_dtype: Optional[torch.dtype] = None, stream=None,
                     return_state: bool = True, update: str = "exact") -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """``fwd_chunked`` with each sequence split along time into ``segments`` pieces
    (``efla_fwd_chunked_scan``): for few long sequences.  ``workspace`` (a CUDA tensor of at
    least ``scan_workspace(...)[0]`` bytes) is allocated here when not given."""
    L = load()
    _need(workspace, "workspace")
    B, T, H, dk, dv, N = _check_fwd_inputs(q, k, v, beta, S0)
    o, S_T = _outputs(q, o, S_T, o_dtype, return_state, B, T, H, dk, dv, N)
    if update not in UPDATES:
        raise EflaError(1, f"unknown update rule {update!r}")
    need, _ = scan_workspace(B, T, H, dk, dv, segments)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    nbytes = workspace.numel() * workspace.element_size()
    _check(L.efla_fwd_chunked_scan(_p(q), _p(k), _p(v), _p(beta), _p(S0), _p(o), _p(S_T), B, T, H, dk, dv,
                                   _dt(q.dtype), _dt(o.dtype), int(segments), _p(workspace), nbytes,
                                   UPDATES[update], _stream(stream)))
    return o, S_T


def fwd_chunked_scan_static(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
                            S0: Optional[torch.Tensor] = None, *, segments: int = 0, o: Optional[torch.Tensor] = None,
                            S_T: Optional[torch.Tensor] = None, o_dtype: Optional[torch.dtype] = None, stream=None,
                            return_state: bool = True, update: str = "exact"):
    """``fwd_chunked_scan`` on the library's fixed scratch (``efla_fwd_chunked_scan_static``):
    no workspace.  Calls that overlap in time race on that scratch.  Pass ``o`` (and ``S_T``)
    to make the call allocate nothing at all."""
    L = load()
    B, T, H, dk, dv, N = _check_fwd_inputs(q, k, v, beta, S0)
    o, S_T = _outputs(q, o, S_T, o_dtype, return_state, B, T, H, dk, dv, N)
    if update not in UPDATES:
        raise EflaError(1, f"unknown update rule {update!r}")
    _check(L.efla_fwd_chunked_scan_static(_p(q), _p(k), _p(v), _p(beta), _p(S0), _p(o), _p(S_T), B, T, H, dk, dv,
                                          _dt(q.dtype), _dt(o.dtype), int(segments), UPDATES[update],
                                          _stream(stream)))
    return o, S_T


def fwd_recurrent(q, k, v, beta, S0=None, cu_seqlens=None, *, o=None, S_T=None,
                  o_dtype: Optional[torch.dtype] = None, stream=None, return_state: bool = True,
                  update: str = "exact"):
    """Token-by-token fp32 evaluation on CUDA cores (``efla_fwd_recurrent``)."""
    return _fwd("recurrent", q, k, v, beta, S0, cu_seqlens, o, S_T, o_dtype, 0, stream, return_state, update)


def decode_step(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor, S: torch.Tensor, *,
                o: Optional[torch.Tensor] = None, o_dtype: Optional[torch.dtype] = None,
                stream=None, update: str = "exact") -> torch.Tensor:
    """One token per sequence; S [B,H,dk,dv] fp32 is updated in place.  Returns o [B,H,dv]
    (in q's dtype unless ``o_dtype`` or ``o`` says otherwise)."""
    L = load()
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (beta, "beta"), (S, "S"), (o, "o")):
        _need(t, n)
    if q.dim() != 3 or k.shape != q.shape or v.shape[:2] != q.shape[:2] or beta.shape != q.shape[:2]:
        raise EflaError(1, "shape mismatch")
    B, H, dk = q.shape
    dv = v.shape[-1]
    if S.dtype != torch.float32 or tuple(S.shape) != (B, H, dk, dv):
        raise EflaError(1, f"S must be float32 [{B},{H},{dk},{dv}]")
    if q.dtype != k.dtype or q.dtype != v.dtype or beta.dtype != torch.float32:
        raise EflaError(1, "q, k, v must share a dtype and beta must be float32")
    if o is None:
        o = torch.empty((B, H, dv), dtype=q.dtype if o_dtype is None else o_dtype, device=q.device)
    elif tuple(o.shape) != (B, H, dv):
        raise EflaError(1, "o has the wrong shape")
    if update not in UPDATES:
        raise EflaError(1, f"unknown update rule {update!r}")
    _check(L.efla_decode_step_ex(_p(q), _p(k), _p(v), _p(beta), _p(S), _p(o), B, H, dk, dv,
                                 _dt(q.dtype), _dt(o.dtype), UPDATES[update], _stream(stream)))
    return o


def decode_tokens(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor, S: torch.Tensor, *,
                  o: Optional[torch.Tensor] = None, o_dtype: Optional[torch.dtype] = None,
                  stream=None, update: str = "exact") -> torch.Tensor:
    """m tokens per sequence appended to the state; S [B,H,dk,dv] fp32 is updated in place.

    q, k [B,m,H,dk], v [B,m,H,dv] (bf16 or fp32), beta [B,m,H] fp32.  Returns o [B,m,H,dv].
    Equal to m successive ``decode_step`` calls (``efla_decode_tokens``).
    """
    L = load()
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (beta, "beta"), (S, "S"), (o, "o")):
        _need(t, n)
    if q.dim() != 4 or k.shape != q.shape or v.shape[:3] != q.shape[:3] or beta.shape != q.shape[:3]:
        raise EflaError(1, "shape mismatch")
    B, m, H, dk = q.shape
    dv = v.shape[-1]
    if S.dtype != torch.float32 or tuple(S.shape) != (B, H, dk, dv):
        raise EflaError(1, f"S must be float32 [{B},{H},{dk},{dv}]")
    if q.dtype != k.dtype or q.dtype != v.dtype or beta.dtype != torch.float32:
        raise EflaError(1, "q, k, v must share a dtype and beta must be float32")
    if o is None:
        o = torch.empty((B, m, H, dv), dtype=q.dtype if o_dtype is None else o_dtype, device=q.device)
    elif tuple(o.shape) != (B, m, H, dv):
        raise EflaError(1, "o has the wrong shape")
    if update not in UPDATES:
        raise EflaError(1, f"unknown update rule {update!r}")
    _check(L.efla_decode_tokens(_p(q), _p(k), _p(v), _p(beta), _p(S), _p(o), B, m, H, dk, dv,
                                _dt(q.dtype), _dt(o.dtype), UPDATES[update], _stream(stream)))
    return o


def bwd_workspace(B: int, T: int, H: int, dk: int = 128, dv: int = 128) -> int:
    """Workspace bytes of ``bwd_chunked`` (``efla_bwd_workspace``)."""
    L = load()
    nb = ctypes.c_size_t(0)
    _check(L.efla_bwd_workspace(B, T, H, dk, dv, ctypes.byref(nb)))
    return nb.value


def bwd_chunked(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
                S0: Optional[torch.Tensor], dO: torch.Tensor, dS_T: Optional[torch.Tensor] = None, *,
                need_dS0: bool = True, workspace: Optional[torch.Tensor] = None, stream=None,
                update: str = "exact", saved: bool = False) -> dict:
    """``bwd_recurrent`` evaluated in chunks of 64 tokens (``efla_bwd_chunked``); ``workspace``
    (a CUDA tensor of at least ``bwd_workspace(...)`` bytes) is allocated here when not given.
    ``saved=True`` (``efla_bwd_chunked_saved``) takes the workspace that ``fwd_chunked_train``
    filled for these inputs and does not run the forward again."""
    if saved and workspace is None:
        raise EflaError(1, "saved=True needs the workspace that fwd_chunked_train filled")
    return _bwd("saved" if saved else "chunked", q, k, v, beta, S0, dO, dS_T, need_dS0, workspace, stream, update)


def fwd_chunked_train(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
                      S0: Optional[torch.Tensor] = None, *, workspace: Optional[torch.Tensor] = None,
                      o: Optional[torch.Tensor] = None, S_T: Optional[torch.Tensor] = None, stream=None,
                      update: str = "exact") -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """``fwd_chunked`` (rows of [B, T], o in q's dtype) that also keeps, in ``workspace``, what
    ``bwd_chunked`` would recompute (``efla_fwd_chunked_train``).  Returns (o, S_T, workspace);
    pass the workspace to ``bwd_chunked(..., workspace=..., saved=True)`` with the same inputs."""
    L = load()
    _need(workspace, "workspace")
    B, T, H, dk, dv, N = _check_fwd_inputs(q, k, v, beta, S0)
    o, S_T = _outputs(q, o, S_T, None, True, B, T, H, dk, dv, N)
    if o.dtype != q.dtype:
        raise EflaError(1, "o must have q's dtype")
    if update not in UPDATES:
        raise EflaError(1, f"unknown update rule {update!r}")
    need = bwd_workspace(B, T, H, dk, dv)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check(L.efla_fwd_chunked_train(_p(q), _p(k), _p(v), _p(beta), _p(S0), _p(o), _p(S_T), B, T, H, dk, dv,
                                    _dt(q.dtype), UPDATES[update], _p(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream)))
    return o, S_T, workspace


def bwd_recurrent(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, beta: torch.Tensor,
                  S0: Optional[torch.Tensor], dO: torch.Tensor, dS_T: Optional[torch.Tensor] = None, *,
                  need_dS0: bool = True, stream=None, update: str = "exact") -> dict:
    """Gradients of ``fwd_chunked`` (no cu_seqlens) from dO [B,T,H,dv] fp32 and dS_T
    [B,H,dk,dv] fp32 (or None): returns dq, dk, dv, dbeta and dS0 (fp32), ``efla_bwd_recurrent``."""
    return _bwd("recurrent", q, k, v, beta, S0, dO, dS_T, need_dS0, None, stream, update)


def _bwd(kind, q, k, v, beta, S0, dO, dS_T, need_dS0, workspace, stream, update):
    L = load()
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (beta, "beta"), (S0, "S0"), (dO, "dO"), (dS_T, "dS_T")):
        _need(t, n)
    if q.dim() != 4 or k.shape != q.shape or v.shape[:3] != q.shape[:3] or beta.shape != q.shape[:3]:
        raise EflaError(1, "shape mismatch")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if dO.dtype != torch.float32 or tuple(dO.shape) != (B, T, H, dv):
        raise EflaError(1, f"dO must be float32 [{B},{T},{H},{dv}]")
    for t, n in ((S0, "S0"), (dS_T, "dS_T")):
        if t is not None and (t.dtype != torch.float32 or tuple(t.shape) != (B, H, dk, dv)):
            raise EflaError(1, f"{n} must be float32 [{B},{H},{dk},{dv}]")
    if update not in UPDATES:
        raise EflaError(1, f"unknown update rule {update!r}")
    f32 = dict(dtype=torch.float32, device=q.device)
    out = {"dq": torch.empty((B, T, H, dk), **f32), "dk": torch.empty((B, T, H, dk), **f32),
           "dv": torch.empty((B, T, H, dv), **f32), "dbeta": torch.empty((B, T, H), **f32),
           "dS0": torch.empty((B, H, dk, dv), **f32) if need_dS0 else None}
    args = (_p(q), _p(k), _p(v), _p(beta), _p(S0), _p(dO), _p(dS_T), _p(out["dq"]), _p(out["dk"]), _p(out["dv"]),
            _p(out["dbeta"]), _p(out["dS0"]), B, T, H, dk, dv, _dt(q.dtype), UPDATES[update])
    if kind == "recurrent":
        _check(L.efla_bwd_recurrent(*args, _stream(stream)))
        return out
    _need(workspace, "workspace")
    need = bwd_workspace(B, T, H, dk, dv)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    fn = L.efla_bwd_chunked_saved if kind == "saved" else L.efla_bwd_chunked
    _check(fn(*args, _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def prep(k: torch.Tensor, beta: torch.Tensor, v: Optional[torch.Tensor] = None, *, lam: bool = True,
         alpha: bool = True, ak: bool = False, av: bool = False, update: str = "exact", stream=None) -> dict:
    """Per-token lambda = ||k||^2, gate alpha, and optionally alpha*k, alpha*v (``efla_prep``).

    k [..., d_k], v [..., d_v] (bf16 or fp32), beta [...] fp32 with matching leading
    dimensions.  Returns a dict with the requested outputs, shaped like beta
    (lam, alpha) or like k / v (ak, av).
    """
    L = load()
    for t, n in ((k, "k"), (beta, "beta"), (v, "v")):
        _need(t, n)
    if beta.dtype != torch.float32 or tuple(beta.shape) != tuple(k.shape[:-1]):
        raise EflaError(1, "beta must be float32 with k's leading shape")
    if av and v is None:
        raise EflaError(1, "av requested without v")
    if v is not None and (v.dtype != k.dtype or tuple(v.shape[:-1]) != tuple(k.shape[:-1])):
        raise EflaError(1, "v must match k's dtype and leading shape")
    if update not in UPDATES:
        raise EflaError(1, f"unknown update rule {update!r}")
    n = beta.numel()
    dk = k.shape[-1]
    dv = v.shape[-1] if v is not None else dk
    out = {}
    if lam:
        out["lam"] = torch.empty_like(beta)
    if alpha:
        out["alpha"] = torch.empty_like(beta)
    if ak:
        out["ak"] = torch.empty_like(k)
    if av:
        out["av"] = torch.empty_like(v)
    _check(L.efla_prep(_p(k), _p(v), _p(beta), _p(out.get("lam")), _p(out.get("alpha")), _p(out.get("ak")),
                       _p(out.get("av")), n, dk, dv, _dt(k.dtype), UPDATES[update], _stream(stream)))
    return out


def device_status(stream=None) -> int:
    """Read and clear the current device's status word (synchronises ``stream``)."""
    return load().efla_device_status(_stream(stream))


def error_string(code: int) -> str:
    """Static description of a status code (``efla_get_error_string``)."""
    return load().efla_get_error_string(int(code)).decode()


def set_wait_limit_ns(ns: int) -> None:
    """Test hook: bound on the chunk kernel's waits between warp roles, in ns (0 = the 2 s default)."""
    load().efla_debug_set_wait_limit_ns(int(ns))


def set_debug_stall(on) -> None:
    """Test hook (``efla_debug_set_stall``): make tensor-core kernels' waits run out on purpose.
    True (or 1) names the chunk kernel; an int is the header's set of kernel bits (1 chunk
    kernel, 2 backward state pass, 4 backward gradient kernel)."""
    load().efla_debug_set_stall(int(on) & 7)

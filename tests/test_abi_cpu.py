"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "efla.h")


@pytest.fixture(scope="module")
def lib():
    from exact_delta_rule_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(efla_[a-z_]+)\s*\(", text)))


def declared_params(name):
    """Parameter names of a function declared in the header, in order."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    m = re.search(r"\b" + name + r"\s*\(([^)]*)\)\s*;", text)
    assert m, name
    params = [p.strip() for p in m.group(1).split(",")]
    return [re.findall(r"[A-Za-z_][A-Za-z_0-9]*", p)[-1] for p in params if p and p != "void"]


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("efla_fwd_chunked", "efla_decode_step", "efla_get_error_string", "efla_fwd_recurrent",
              "efla_device_status", "efla_last_error", "efla_abi_version"):
        assert n in names


def test_boundary_signatures():
    """The two calls of the boundary take exactly these arguments, in this order (o has the
    dtype of q; no output-dtype argument)."""
    assert declared_params("efla_fwd_chunked") == [
        "q", "k", "v", "beta", "S0", "cu_seqlens", "o", "S_T", "B", "T", "H", "d_k", "d_v", "N", "dtype",
        "chunk", "stream"]
    assert declared_params("efla_decode_step") == [
        "q", "k", "v", "beta", "S", "o", "B", "H", "d_k", "d_v", "dtype", "stream"]
    assert declared_params("efla_get_error_string") == ["status"]
    text = open(HEADER).read()
    assert re.search(r"EFLA_OK\s*=\s*0,\s*EFLA_ERR_INVALID_ARG\s*=\s*1,", text)
    assert re.search(r"EFLA_BF16\s*=\s*0,\s*EFLA_F32\s*=\s*1", text)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in efla.h but not exported"


def test_abi_version_matches_header(lib):
    m = re.search(r"#define\s+EFLA_ABI_VERSION\s+(\d+)", open(HEADER).read())
    lib.efla_abi_version.restype = ctypes.c_int
    assert lib.efla_abi_version() == int(m.group(1))


def test_status_strings(lib):
    lib.efla_get_error_string.restype = ctypes.c_char_p
    lib.efla_get_error_string.argtypes = [ctypes.c_int]
    for code, name in enumerate(["EFLA_OK", "EFLA_ERR_INVALID_ARG", "EFLA_ERR_UNSUPPORTED", "EFLA_ERR_CUDA",
                                 "EFLA_ERR_DEVICE_TIMEOUT"]):
        assert lib.efla_get_error_string(code).decode().startswith(name)
    assert lib.efla_get_error_string(99)


# Fake, never-dereferenced device addresses: validation rejects before any CUDA call.
Q, K, V, BETA, O, S0, ST, CU = (0x10000000 * (i + 1) for i in range(8))


def _fwd(lib, **kw):
    a = dict(q=Q, k=K, v=V, beta=BETA, S0=None, cu=None, o=O, S_T=None, B=2, T=64, H=4, dk=128, dv=128, N=2,
             dt=0, chunk=64, stream=None)
    a.update(kw)
    vp, ip = ctypes.c_void_p, ctypes.c_int
    f = lib.efla_fwd_chunked
    f.restype = ip
    f.argtypes = [vp] * 8 + [ip] * 8 + [vp]
    return f(a["q"], a["k"], a["v"], a["beta"], a["S0"], a["cu"], a["o"], a["S_T"], a["B"], a["T"], a["H"],
             a["dk"], a["dv"], a["N"], a["dt"], a["chunk"], a["stream"])


def _last(lib):
    lib.efla_last_error.restype = ctypes.c_char_p
    return lib.efla_last_error().decode()


INVALID, UNSUPPORTED = 1, 2


@pytest.mark.parametrize("kw,code,msg", [
    (dict(B=-1), INVALID, "bad sizes"),
    (dict(H=0), INVALID, "bad sizes"),
    (dict(dk=0), INVALID, "positive"),
    (dict(dk=48), UNSUPPORTED, "supported head sizes"),
    (dict(dv=256), UNSUPPORTED, "supported head sizes"),
    (dict(chunk=48), UNSUPPORTED, "chunk"),
    (dict(chunk=128), UNSUPPORTED, "chunk"),
    (dict(chunk=-64), UNSUPPORTED, "chunk"),
    (dict(dt=7), INVALID, "dtype"),
    (dict(N=3), INVALID, "must equal B"),
    (dict(cu=CU, B=2), INVALID, "must be 1"),
    (dict(q=None), INVALID, "non-NULL"),
    (dict(beta=None), INVALID, "non-NULL"),
    (dict(k=K + 8), INVALID, "aligned"),
    (dict(S0=S0 + 4), INVALID, "aligned"),
    (dict(o=Q + 1024), INVALID, "overlaps"),
    (dict(S_T=O + 64), INVALID, "overlaps"),
    (dict(T=1 << 30), UNSUPPORTED, "exceeds"),
])
def test_fwd_rejects(lib, kw, code, msg):
    assert _fwd(lib, **kw) == code
    assert msg in _last(lib)


def test_fwd_recurrent_rejects(lib):
    vp, ip = ctypes.c_void_p, ctypes.c_int
    f = lib.efla_fwd_recurrent
    f.restype = ip
    f.argtypes = [vp] * 8 + [ip] * 7 + [vp]
    assert f(Q, K, V, BETA, None, None, O, None, 2, 64, 4, 128, 96, 2, 0, None) == UNSUPPORTED
    assert f(None, K, V, BETA, None, None, O, None, 2, 64, 4, 128, 128, 2, 0, None) == INVALID


def _dec(lib, **kw):
    a = dict(q=Q, k=K, v=V, beta=BETA, S=S0, o=O, B=4, H=2, dk=128, dv=128, dt=0, stream=None)
    a.update(kw)
    vp, ip = ctypes.c_void_p, ctypes.c_int
    f = lib.efla_decode_step
    f.restype = ip
    f.argtypes = [vp] * 6 + [ip] * 5 + [vp]
    return f(a["q"], a["k"], a["v"], a["beta"], a["S"], a["o"], a["B"], a["H"], a["dk"], a["dv"], a["dt"],
             a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(B=-2), INVALID), (dict(H=0), INVALID), (dict(dk=16), UNSUPPORTED), (dict(dv=100), UNSUPPORTED),
    (dict(S=None), INVALID), (dict(S=S0 + 8), INVALID), (dict(o=S0 + 4096), INVALID), (dict(dt=5), INVALID),
])
def test_decode_rejects(lib, kw, code):
    assert _dec(lib, **kw) == code
    assert _last(lib)


def test_product_package_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "exact_delta_rule_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"\boracle\b", text), f"{f} mentions the oracle"
                assert "efla_oracle" not in text


def test_binding_raises_without_library(tmp_path, monkeypatch):
    import exact_delta_rule_gb300 as efla
    monkeypatch.setattr(efla, "lib_path", str(tmp_path / "missing.so"))
    monkeypatch.setattr(efla, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        efla.load()


def test_update_rule_validated(lib):
    vp, ip = ctypes.c_void_p, ctypes.c_int
    f = lib.efla_fwd_chunked_ex
    f.restype = ip
    f.argtypes = [vp] * 8 + [ip] * 10 + [vp]
    assert f(Q, K, V, BETA, None, None, O, None, 2, 64, 4, 128, 128, 2, 0, 1, 64, 7, None) == INVALID
    assert "update" in _last(lib)
    g = lib.efla_decode_step_ex
    g.restype = ip
    g.argtypes = [vp] * 6 + [ip] * 7 + [vp]
    assert g(Q, K, V, BETA, S0, O, 4, 2, 128, 128, 0, 1, 3, None) == INVALID


def _prep(lib, **kw):
    a = dict(k=K, v=V, beta=BETA, lam=O, alpha=ST, ak=S0, av=CU, n=1000, dk=128, dv=128, dt=0, upd=0)
    a.update(kw)
    vp, ip = ctypes.c_void_p, ctypes.c_int
    f = lib.efla_prep
    f.restype = ip
    f.argtypes = [vp] * 7 + [ctypes.c_longlong] + [ip] * 4 + [vp]
    return f(a["k"], a["v"], a["beta"], a["lam"], a["alpha"], a["ak"], a["av"], a["n"], a["dk"], a["dv"],
             a["dt"], a["upd"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(n=-1), INVALID), (dict(dk=100), UNSUPPORTED), (dict(k=None), INVALID), (dict(v=None), INVALID),
    (dict(beta=BETA + 8), INVALID), (dict(lam=K + 64), INVALID), (dict(alpha=O + 16), INVALID),
    (dict(upd=9), INVALID), (dict(dt=4), INVALID),
])
def test_prep_rejects(lib, kw, code):
    assert _prep(lib, **kw) == code
    assert _last(lib)


def _dect(lib, **kw):
    a = dict(q=Q, k=K, v=V, beta=BETA, S=S0, o=O, B=4, m=3, H=2, dk=128, dv=128, ind=0, od=1, upd=0)
    a.update(kw)
    vp, ip = ctypes.c_void_p, ctypes.c_int
    f = lib.efla_decode_tokens
    f.restype = ip
    f.argtypes = [vp] * 6 + [ip] * 8 + [vp]
    return f(a["q"], a["k"], a["v"], a["beta"], a["S"], a["o"], a["B"], a["m"], a["H"], a["dk"], a["dv"], a["ind"],
             a["od"], a["upd"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(m=-1), INVALID), (dict(B=-1), INVALID), (dict(H=0), INVALID), (dict(dk=48), UNSUPPORTED),
    (dict(S=None), INVALID), (dict(q=None), INVALID), (dict(S=S0 + 8), INVALID), (dict(o=Q + 256), INVALID),
    (dict(S=O + 64), INVALID), (dict(upd=5), INVALID), (dict(od=3), INVALID),
])
def test_decode_tokens_rejects(lib, kw, code):
    assert _dect(lib, **kw) == code
    assert _last(lib)


def test_decode_tokens_empty_is_ok_without_gpu_work(lib):
    # m == 0 launches nothing: only S is needed
    assert _dect(lib, m=0, q=None, k=None, v=None, beta=None, o=None) == 0


def test_scan_workspace_query(lib):
    f = lib.efla_fwd_scan_workspace
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int] * 6 + [ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_int)]
    nb, g = ctypes.c_size_t(0), ctypes.c_int(0)
    assert f(1, 65536, 16, 128, 128, 9, ctypes.byref(nb), ctypes.byref(g)) == 0
    assert g.value == 9 and nb.value == (3 * 9 - 2) * 16 * 128 * 128 * 4
    assert f(1, 700, 2, 128, 128, 3, ctypes.byref(nb), ctypes.byref(g)) == 0
    assert g.value == 3  # 11 chunks -> pieces of 4, 4, 3 chunks
    assert f(2, 100, 2, 128, 128, 50, ctypes.byref(nb), ctypes.byref(g)) == 0
    assert g.value == 2  # capped at the chunk count
    assert f(8, 2048, 16, 128, 128, 1, ctypes.byref(nb), ctypes.byref(g)) == 0
    assert nb.value == 0 and g.value == 1
    assert f(1, 64, 0, 128, 128, 2, ctypes.byref(nb), ctypes.byref(g)) == INVALID


def _scanc(lib, **kw):
    a = dict(q=Q, k=K, v=V, beta=BETA, S0=None, o=O, S_T=None, B=1, T=700, H=2, dk=128, dv=128, ind=0, od=1,
             seg=3, ws=CU, wsb=1 << 30, upd=0)
    a.update(kw)
    vp, ip = ctypes.c_void_p, ctypes.c_int
    f = lib.efla_fwd_chunked_scan
    f.restype = ip
    f.argtypes = [vp] * 7 + [ip] * 8 + [vp, ctypes.c_size_t, ip, vp]
    return f(a["q"], a["k"], a["v"], a["beta"], a["S0"], a["o"], a["S_T"], a["B"], a["T"], a["H"], a["dk"],
             a["dv"], a["ind"], a["od"], a["seg"], a["ws"], a["wsb"], a["upd"], None)


@pytest.mark.parametrize("kw,msg", [
    (dict(ws=None), "workspace"), (dict(wsb=1000), "workspace"), (dict(ws=CU + 8), "aligned"),
    (dict(ws=O), "overlaps"), (dict(upd=4), "update"), (dict(H=0), "bad sizes"),
])
def test_scan_rejects(lib, kw, msg):
    assert _scanc(lib, **kw) == INVALID
    assert msg in _last(lib)


def _bw(lib, **kw):
    a = dict(q=Q, k=K, v=V, beta=BETA, S0=None, dO=CU, dST=None, dq=O, dk=ST, dv=S0, db=0x90000000, dS0=None,
             B=1, T=64, H=2, dk_=128, dv_=128, ind=0, upd=0)
    a.update(kw)
    vp, ip = ctypes.c_void_p, ctypes.c_int
    f = lib.efla_bwd_recurrent
    f.restype = ip
    f.argtypes = [vp] * 12 + [ip] * 7 + [vp]
    return f(a["q"], a["k"], a["v"], a["beta"], a["S0"], a["dO"], a["dST"], a["dq"], a["dk"], a["dv"], a["db"],
             a["dS0"], a["B"], a["T"], a["H"], a["dk_"], a["dv_"], a["ind"], a["upd"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(T=-1), INVALID), (dict(H=0), INVALID), (dict(dk_=48), UNSUPPORTED), (dict(dq=None), INVALID),
    (dict(dO=None), INVALID), (dict(dk=O + 256), INVALID), (dict(dq=Q + 1024), INVALID), (dict(upd=3), INVALID),
    (dict(db=0x90000000 + 4), INVALID), (dict(ind=5), INVALID),
])
def test_bwd_rejects(lib, kw, code):
    assert _bw(lib, **kw) == code
    assert _last(lib)


def _bwd_need(lib, B, T, H, dk, dv):
    f = lib.efla_bwd_workspace
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(ctypes.c_size_t)]
    n = ctypes.c_size_t(0)
    return n.value if f(B, T, H, dk, dv, ctypes.byref(n)) == 0 else 1 << 20


def _bwc(lib, ws=0xA0000000, ws_bytes=None, entry="efla_bwd_chunked", **kw):
    a = dict(q=Q, k=K, v=V, beta=BETA, S0=None, dO=CU, dST=None, dq=O, dk=ST, dv=S0, db=0x90000000, dS0=None,
             B=1, T=64, H=2, dk_=128, dv_=128, ind=0, upd=0)
    a.update(kw)
    vp, ip = ctypes.c_void_p, ctypes.c_int
    f = getattr(lib, entry)
    f.restype = ip
    f.argtypes = [vp] * 12 + [ip] * 7 + [vp, ctypes.c_size_t, vp]
    need = _bwd_need(lib, a["B"], max(a["T"], 0), max(a["H"], 1), a["dk_"], a["dv_"])
    return f(a["q"], a["k"], a["v"], a["beta"], a["S0"], a["dO"], a["dST"], a["dq"], a["dk"], a["dv"], a["db"],
             a["dS0"], a["B"], a["T"], a["H"], a["dk_"], a["dv_"], a["ind"], a["upd"], ws,
             need if ws_bytes is None else ws_bytes, None)


@pytest.mark.parametrize("entry", ["efla_bwd_chunked", "efla_bwd_chunked_saved"])
@pytest.mark.parametrize("kw,code", [
    (dict(T=-1), INVALID), (dict(H=0), INVALID), (dict(dk_=64, dv_=128), UNSUPPORTED),
    (dict(dk_=32, dv_=32), UNSUPPORTED), (dict(dq=None), INVALID), (dict(upd=3), INVALID),
    (dict(ws=None), INVALID), (dict(ws_bytes=1024), INVALID), (dict(ws=0xA0000000 + 8), INVALID),
    (dict(ws=Q), INVALID),
])
def test_bwd_chunked_rejects(lib, entry, kw, code):
    """efla_bwd_chunked and efla_bwd_chunked_saved validate sizes, the supported shapes
    (d_k = d_v in {64, 128}) and their workspace (present, large enough, aligned, overlapping no
    argument) before any launch."""
    assert _bwc(lib, entry=entry, **kw) == code
    assert _last(lib)


def _fwt(lib, ws=0xA0000000, ws_bytes=None, **kw):
    a = dict(q=Q, k=K, v=V, beta=BETA, S0=None, o=O, S_T=ST, B=1, T=64, H=2, dk_=128, dv_=128, ind=0, upd=0)
    a.update(kw)
    vp, ip = ctypes.c_void_p, ctypes.c_int
    f = lib.efla_fwd_chunked_train
    f.restype = ip
    f.argtypes = [vp] * 7 + [ip] * 7 + [vp, ctypes.c_size_t, vp]
    need = _bwd_need(lib, a["B"], max(a["T"], 0), max(a["H"], 1), a["dk_"], a["dv_"])
    return f(a["q"], a["k"], a["v"], a["beta"], a["S0"], a["o"], a["S_T"], a["B"], a["T"], a["H"], a["dk_"],
             a["dv_"], a["ind"], a["upd"], ws, need if ws_bytes is None else ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(T=-1), INVALID), (dict(H=0), INVALID), (dict(dk_=32, dv_=32), UNSUPPORTED),
    (dict(dk_=64, dv_=128), UNSUPPORTED), (dict(o=None), INVALID), (dict(upd=3), INVALID),
    (dict(ws=None), INVALID), (dict(ws_bytes=1024), INVALID), (dict(ws=0xA0000000 + 8), INVALID),
    (dict(ws=Q), INVALID),
])
def test_fwd_chunked_train_rejects(lib, kw, code):
    """efla_fwd_chunked_train validates as efla_fwd_chunked does, plus the backward's supported
    shapes and its workspace, before any launch."""
    assert _fwt(lib, **kw) == code
    assert _last(lib)


def test_bwd_workspace_size(lib):
    f = lib.efla_bwd_workspace
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(ctypes.c_size_t)]
    n = ctypes.c_size_t(0)
    assert f(8, 2048, 16, 128, 128, ctypes.byref(n)) == 0
    # per chunk: start state, end-state gradient, T''; per token: dO hi/lo, G, -dR hi/lo
    assert n.value == 8 * 16 * 32 * (2 * 128 * 128 + 64 * 64) * 4 + 8 * 2048 * 16 * 128 * (4 + 4 + 4)
    assert f(1, 65, 1, 64, 64, ctypes.byref(n)) == 0 and n.value == 2 * (2 * 64 * 64 + 64 * 64) * 4 + 65 * 64 * 12
    assert f(1, 64, 1, 32, 32, ctypes.byref(n)) == UNSUPPORTED
    assert f(1, 64, 1, 128, 128, None) == INVALID


def test_binding_checks_dtypes_and_shapes_before_any_device_call():
    """The forward wrappers (plain, split and static-scratch) reject a non-fp32 beta, a
    wrongly shaped S0 and mismatched q/k/v before touching a device."""
    import torch

    import exact_delta_rule_gb300 as efla
    B, T, H, d = 1, 8, 2, 128
    q = torch.zeros((B, T, H, d), dtype=torch.bfloat16)
    beta = torch.zeros((B, T, H))
    S0 = torch.zeros((B, H, d, d))
    for fn in (efla.fwd_chunked, efla.fwd_chunked_scan, efla.fwd_chunked_scan_static):
        with pytest.raises(efla.EflaError, match="beta must be float32"):
            fn(q, q, q, beta.bfloat16(), S0)
        with pytest.raises(efla.EflaError, match="S0 must be float32"):
            fn(q, q, q, beta, S0[:, :1])
        with pytest.raises(efla.EflaError, match="S0 must be float32"):
            fn(q, q, q, beta, S0.double())
        with pytest.raises(efla.EflaError, match="share a dtype"):
            fn(q, q.float(), q, beta, S0)
        with pytest.raises(efla.EflaError, match="shape mismatch"):
            fn(q, q[:, :4], q, beta, S0)
        with pytest.raises(efla.EflaError, match="CUDA tensor"):
            fn(q, q, q, beta, S0)


def test_status_word_is_resolved_per_device():
    """The status word's device address is cached per device index, under a lock."""
    src = open(os.path.join(ROOT, "exact_delta_rule_gb300", "csrc", "efla_api.cu")).read()
    body = src[src.index("int *device_status_ptr() {"):]
    body = body[:body.index("\n}\n")]
    assert "cudaGetDevice(&dev)" in body and "ptrs[dev]" in body and "lock_guard" in body

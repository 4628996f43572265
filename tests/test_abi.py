"""The C-ABI library builds, loads and exports what include/linattn.h
declares, and its host-side argument checks reject bad calls before anything
touches a GPU (these tests need no GPU: every call here returns during
validation, so nothing is enqueued; the workspace-size query asks the CUDA
runtime for the SM count and falls back to one SM without a device)."""
import ctypes
import os
import re

import pytest

import linear_attention_feature_gb300 as la
from linear_attention_feature_gb300 import build as labuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "linattn.h")

INVALID, UNSUPPORTED, OK = 1, 2, 0


@pytest.fixture(scope="module")
def lib():
    labuild.build()
    return la.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(la_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("la_forward", "la_decode_step", "la_check_device_status",
              "la_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared but not exported"
    assert set(declared_functions()) <= set(la.EXPORTED) | {"la_forward_ex"}


def test_status_strings_and_version(lib):
    for code, name in la.STATUS.items():
        assert lib.la_status_string(code).decode() == name
    assert lib.la_status_string(99).decode() == "LA_ERR_UNKNOWN"
    assert lib.la_abi_version() == 1


P = ctypes.c_void_p(0x1000)   # never dereferenced: validation fails first
P2 = ctypes.c_void_p(0x2000)
P3 = ctypes.c_void_p(0x3000)
OUT = ctypes.c_void_p(0x4000)


def fwd(lib, q=P, k=P2, v=P3, out=OUT, B=1, H=2, N=8, d=64, causal=1,
        decay=None, dtype=1, path=0, seg=0):
    return lib.la_forward_ex(q, k, v, out, B, H, N, d, causal, decay, dtype,
                             path, seg, None)


def floats(*xs):
    return (ctypes.c_float * len(xs))(*xs)


@pytest.mark.parametrize("kw, code, msg", [
    (dict(q=None), INVALID, "null"),
    (dict(out=None), INVALID, "null"),
    (dict(B=-1), INVALID, "negative"),
    (dict(N=-3), INVALID, "negative"),
    (dict(d=0), INVALID, "d must"),
    (dict(d=257), INVALID, "d must"),
    (dict(causal=2), INVALID, "causal"),
    (dict(dtype=7), INVALID, "dtype"),
    (dict(out=P), INVALID, "alias"),
    (dict(causal=0, decay=floats(0.5, 0.5)), INVALID, "causal form only"),
    (dict(decay=floats(0.5, 1.5)), INVALID, "[0, 1]"),
    (dict(decay=floats(float("nan"), 0.5)), INVALID, "[0, 1]"),
    (dict(decay=floats(-0.1, 0.5)), INVALID, "[0, 1]"),
    (dict(path=3), INVALID, "path"),
    (dict(seg=-1), INVALID, "segment_chunks"),
    (dict(dtype=0, path=2), UNSUPPORTED, "tensor-core"),
    (dict(d=96, path=2), UNSUPPORTED, "tensor-core"),
])
def test_forward_rejects_bad_arguments(lib, kw, code, msg):
    assert fwd(lib, **kw) == code
    assert msg in lib.la_last_error().decode()


def test_forward_empty_problems_are_noops(lib):
    # nothing is enqueued, so no GPU is needed; an empty problem touches no
    # tensor element, so NULL pointers (zero-size tensors) are accepted
    assert fwd(lib, B=0) == OK
    assert fwd(lib, H=0) == OK
    assert fwd(lib, N=0) == OK
    assert fwd(lib, N=0, q=None, k=None, v=None, out=None) == OK


def test_forward_rejects_decay_for_too_many_heads(lib):
    H = 1025
    dec = (ctypes.c_float * H)(*([0.5] * H))
    assert fwd(lib, H=H, decay=dec) == UNSUPPORTED


def test_decode_rejects_bad_arguments(lib):
    f = lib.la_decode_step
    assert f(None, P, P, P, P, OUT, 1, 1, 64, 1, None) == INVALID
    assert f(P, P, P, P, P, None, 1, 1, 64, 1, None) == INVALID
    assert f(P, P, P, P, P, OUT, -1, 1, 64, 1, None) == INVALID
    assert f(P, P, P, P, P, OUT, 1, 1, 0, 1, None) == INVALID
    assert f(P, P, P, P, P, OUT, 1, 1, 300, 1, None) == INVALID
    assert f(P, P, P, P, P, OUT, 1, 1, 64, 5, None) == INVALID
    assert f(P, P, P, P, P, OUT, 0, 4, 64, 1, None) == OK


def test_python_binding_refuses_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 1, 4, 4)
    with pytest.raises(ValueError, match="CUDA"):
        la.forward(q, q.clone(), q.clone())
    S = torch.zeros(1, 1, 4, 4)
    z = torch.zeros(1, 1, 4)
    t = torch.zeros(1, 1, 4)
    with pytest.raises(ValueError, match="CUDA"):
        la.decode_step(S, z, t, t.clone(), t.clone())


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        la.load_library(str(tmp_path / "nope.so"))


WS = ctypes.c_void_p(0x100000)  # 256-byte aligned, never dereferenced


def fwd_host(lib, q=P, k=P2, v=P3, out=OUT, B=1, H=2, N=8, d=64, causal=1,
             decay=None, dtype=1, ws=WS, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = lib.la_forward_host_workspace_bytes(B, H, N, d, dtype)
    return lib.la_forward_host(q, k, v, out, B, H, N, d, causal, decay, dtype,
                               ws, ws_bytes, None)


@pytest.mark.parametrize("kw, code, msg", [
    (dict(q=None), INVALID, "null"),
    (dict(out=None), INVALID, "null"),
    (dict(B=-1, ws_bytes=0), INVALID, "negative"),
    (dict(d=0, ws_bytes=0), INVALID, "d must"),
    (dict(d=300, ws_bytes=0), INVALID, "d must"),
    (dict(causal=2), INVALID, "causal"),
    (dict(dtype=7, ws_bytes=0), INVALID, "dtype"),
    (dict(out=P2), INVALID, "alias"),
    (dict(causal=0, decay=floats(0.5, 0.5)), INVALID, "causal form only"),
    (dict(decay=floats(0.5, 2.0)), INVALID, "[0, 1]"),
    (dict(ws=None), INVALID, "workspace"),
    (dict(ws_bytes=1024), INVALID, "workspace"),
    (dict(ws=ctypes.c_void_p(0x100010)), INVALID, "aligned"),
])
def test_forward_host_rejects_bad_arguments(lib, kw, code, msg):
    assert fwd_host(lib, **kw) == code
    assert msg in lib.la_last_error().decode()


def test_forward_host_workspace_size_and_empty_problems(lib):
    # q, k, v, out (each rounded up to 256 bytes), plus the kernels' scratch
    # on the tensor-core path (none on the CUDA-core path)
    assert lib.la_forward_host_workspace_bytes(4, 16, 4096, 64, 1) > 4 * 4 * 16 * 4096 * 64 * 2
    assert lib.la_forward_host_workspace_bytes(1, 1, 3, 3, 0) == 4 * 256
    assert lib.la_forward_host_workspace_bytes(1, 1, 3, 0, 0) == 0
    assert lib.la_forward_host_workspace_bytes(1, 1, 3, 3, 9) == 0
    assert fwd_host(lib, B=0, ws=None, ws_bytes=0) == OK
    assert fwd_host(lib, N=0, ws=None, ws_bytes=0) == OK


def test_forward_host_python_binding_refuses_strided_tensors(lib):
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 1, 4, 4)
    with pytest.raises(ValueError, match="contiguous host"):
        la.forward_host(q.transpose(2, 3), q.clone(), q.clone())


def test_forward_causal_state_rejects_bad_arguments(lib):
    f = lib.la_forward_causal_state
    SA = ctypes.c_void_p(0x200000)   # 16-byte aligned, never dereferenced
    ZA = ctypes.c_void_p(0x300000)
    assert f(P, P2, P3, OUT, None, ZA, 1, 2, 8, 64, None, 1, None) == INVALID
    assert "null state" in lib.la_last_error().decode()
    assert f(P, P2, P3, OUT, SA, None, 1, 2, 8, 64, None, 1, None) == INVALID
    assert f(P, P2, P3, OUT, ctypes.c_void_p(0x200004), ZA, 1, 2, 8, 64, None, 1,
             None) == INVALID
    assert "aligned" in lib.la_last_error().decode()
    assert f(None, P2, P3, OUT, SA, ZA, 1, 2, 8, 64, None, 1, None) == INVALID
    assert f(P, P2, P3, OUT, SA, ZA, 1, 2, 8, 300, None, 1, None) == INVALID
    assert f(P, P2, P3, OUT, SA, ZA, 1, 2, 8, 64, floats(0.5, 1.5), 1, None) == INVALID
    assert f(P, P2, P3, OUT, SA, ZA, 0, 2, 8, 64, None, 1, None) == OK  # no heads


def test_decode_step_ex_rejects_bad_decay(lib):
    f = lib.la_decode_step_ex
    assert f(P, P, P, P, P, OUT, 1, 2, 64, floats(0.5, -0.1), 1, None) == INVALID
    assert "[0, 1]" in lib.la_last_error().decode()
    assert f(P, P, P, P, P, OUT, 1, 2, 64, floats(float("nan"), 0.5), 1, None) == INVALID
    H = 1025
    dec = (ctypes.c_float * H)(*([0.5] * H))
    assert f(P, P, P, P, P, OUT, 1, H, 64, dec, 1, None) == UNSUPPORTED
    assert f(P, P, P, P, P, OUT, 0, 2, 64, floats(0.5, 0.5), 1, None) == OK


_Var = la._Variant  # the binding's la_variant struct (ctypes type checks it)


@pytest.mark.parametrize("fmap, norm", [(2, 1), (-1, 0), (0, 2), (1, -1)])
def test_variant_entry_points_reject_unknown_variants(lib, fmap, norm):
    var = ctypes.byref(_Var(fmap, norm))
    assert lib.la_forward_variant(P, P2, P3, OUT, 1, 2, 8, 64, 1, None, 1, var,
                                  None) == INVALID
    assert "variant" in lib.la_last_error().decode()
    assert lib.la_decode_step_variant(P, P, P, P, P, OUT, 1, 2, 64, None, 1, var,
                                      None) == INVALID


def test_variant_null_and_valid_variants_pass_validation(lib):
    # NULL and the four valid variants get past validation: an empty problem
    # then returns LA_OK without touching a GPU
    for var in (None, ctypes.byref(_Var(0, 1)), ctypes.byref(_Var(1, 0)),
                ctypes.byref(_Var(0, 0)), ctypes.byref(_Var(1, 1))):
        assert lib.la_forward_variant(P, P2, P3, OUT, 0, 2, 8, 64, 1, None, 1, var,
                                      None) == OK
        assert lib.la_decode_step_variant(P, P, P, P, P, OUT, 0, 2, 64, None, 1, var,
                                          None) == OK


def test_gated_entry_points_reject_bad_arguments(lib):
    G = ctypes.c_void_p(0x500000)
    f = lib.la_forward_gated
    assert f(P, P2, P3, OUT, None, 1, 2, 8, 64, 1, None, None) == INVALID
    assert "null gates" in lib.la_last_error().decode()
    assert f(P, P2, P3, OUT, G, 1, 2, 8, 300, 1, None, None) == INVALID
    assert f(P, P2, P3, OUT, G, 1, 2, 8, 64, 1, ctypes.byref(la._Variant(5, 1)), None) == INVALID
    assert f(P, P2, P3, OUT, G, 0, 2, 8, 64, 1, None, None) == OK  # empty
    d = lib.la_decode_step_gated
    assert d(P, P, P, P, P, OUT, None, 1, 2, 64, 1, None, None) == INVALID
    assert d(P, P, P, P, P, OUT, G, 1, 2, 0, 1, None, None) == INVALID
    assert d(P, P, P, P, P, OUT, G, 0, 2, 64, 1, None, None) == OK


def test_decode_step_delta_rejects_bad_arguments(lib):
    f = lib.la_decode_step_delta
    BETA = ctypes.c_void_p(0x600000)
    assert f(P, P, P, P, OUT, None, None, 1, 2, 64, 1, None) == INVALID
    assert "null" in lib.la_last_error().decode()
    assert f(None, P, P, P, OUT, BETA, None, 1, 2, 64, 1, None) == INVALID
    assert f(P, P, P, P, OUT, BETA, None, -1, 2, 64, 1, None) == INVALID
    assert f(P, P, P, P, OUT, BETA, None, 1, 2, 300, 1, None) == INVALID
    assert f(P, P, P, P, OUT, BETA, None, 1, 2, 64, 4, None) == INVALID
    assert f(P, P, P, P, OUT, BETA, None, 0, 2, 64, 1, None) == OK

"""GB300-native kernelised (elu+1) linear attention.

Thin Python binding over the C ABI of ``liblinattn.so`` (declared in
``include/linattn.h``): argument marshalling only.  Every step of the
computation runs in the library's CUDA kernels; PyTorch is used for device
memory and streams.  There is no CPU fallback: if the library has not been
built (``python -m linear_attention_feature_gb300.build``) or a tensor is not
on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

__all__ = ["forward", "forward_variant", "forward_gated", "decode_step_gated",
           "decode_step_delta",
           "forward_causal_state", "forward_host",
           "host_workspace_bytes", "decode_step",
           "check_device_status",
           "kernel_launch_count", "LinAttnError",
           "load_library", "LA_F32", "LA_BF16", "STATUS", "EXPORTED"]

LA_F32 = 0
LA_BF16 = 1
STATUS = {0: "LA_OK", 1: "LA_ERR_INVALID_ARG", 2: "LA_ERR_UNSUPPORTED",
          3: "LA_ERR_CUDA", 4: "LA_ERR_NO_MEMORY", 5: "LA_ERR_TIMEOUT",
          6: "LA_ERR_INTERNAL"}
EXPORTED = ("la_forward", "la_forward_ex", "la_decode_step",
            "la_check_device_status", "la_status_string", "la_last_error",
            "la_abi_version", "la_kernel_launch_count",
            "la_forward_causal_noalloc", "la_forward_host",
            "la_forward_host_workspace_bytes", "la_forward_causal_state",
            "la_decode_step_ex", "la_forward_variant", "la_decode_step_variant",
            "la_forward_gated", "la_decode_step_gated", "la_decode_step_delta",
            "la_debug_inject_timeout", "la_debug_fail_next_allocs", "la_forward_delta")

FEATURE_MAPS = {"elu1": 0, "identity": 1}


class _Variant(ctypes.Structure):
    _fields_ = [("feature_map", ctypes.c_int), ("normalise", ctypes.c_int)]


def _variant(feature_map, normalise):
    if feature_map not in FEATURE_MAPS:
        raise ValueError(f"feature_map must be one of {sorted(FEATURE_MAPS)}")
    return ctypes.byref(_Variant(FEATURE_MAPS[feature_map], int(bool(normalise))))

_lib = None


class LinAttnError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__(f"{STATUS.get(status, status)}: {detail}")


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load liblinattn.so (built in-tree).  Raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"{p} is missing: build the CUDA library first "
            "(python -m linear_attention_feature_gb300.build)")
    lib = ctypes.CDLL(p)
    V, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_float)
    lib.la_forward.argtypes = [V, V, V, V, I, I, I, I, I, F, I, V]
    lib.la_forward_ex.argtypes = [V, V, V, V, I, I, I, I, I, F, I, I, I, V]
    lib.la_decode_step.argtypes = [V, V, V, V, V, V, I, I, I, I, V]
    lib.la_decode_step_ex.argtypes = [V, V, V, V, V, V, I, I, I, F, I, V]
    lib.la_forward_causal_state.argtypes = [V, V, V, V, V, V, I, I, I, I, F, I, V]
    VP = ctypes.POINTER(_Variant)
    lib.la_forward_variant.argtypes = [V, V, V, V, I, I, I, I, I, F, I, VP, V]
    lib.la_decode_step_variant.argtypes = [V, V, V, V, V, V, I, I, I, F, I, VP, V]
    lib.la_forward_gated.argtypes = [V, V, V, V, V, I, I, I, I, I, VP, V]
    lib.la_decode_step_gated.argtypes = [V, V, V, V, V, V, V, I, I, I, I, VP, V]
    lib.la_decode_step_delta.argtypes = [V, V, V, V, V, V, V, I, I, I, I, V]
    lib.la_forward_host.argtypes = [V, V, V, V, I, I, I, I, I, F, I, V,
                                    ctypes.c_size_t, V]
    lib.la_forward_host_workspace_bytes.argtypes = [I, I, I, I, I]
    lib.la_forward_host_workspace_bytes.restype = ctypes.c_size_t
    lib.la_forward_delta.argtypes = [V, V, V, V, V, V, V, I, I, I, I, I, V]
    lib.la_debug_inject_timeout.argtypes = [ctypes.c_longlong, I]
    lib.la_debug_fail_next_allocs.argtypes = [I]
    lib.la_check_device_status.argtypes = [V]
    lib.la_status_string.argtypes = [I]
    lib.la_status_string.restype = ctypes.c_char_p
    lib.la_last_error.argtypes = []
    lib.la_last_error.restype = ctypes.c_char_p
    lib.la_abi_version.argtypes = []
    lib.la_kernel_launch_count.argtypes = []
    lib.la_kernel_launch_count.restype = ctypes.c_ulonglong
    for n in ("la_forward", "la_forward_ex", "la_decode_step", "la_forward_host",
              "la_decode_step_ex", "la_forward_causal_state",
              "la_forward_variant", "la_decode_step_variant",
              "la_forward_gated", "la_decode_step_gated", "la_decode_step_delta",
              "la_debug_inject_timeout", "la_debug_fail_next_allocs",
              "la_forward_delta", "la_check_device_status", "la_abi_version"):
        getattr(lib, n).restype = I
    if path is None:
        _lib = lib
    return lib


def _raise_if(status: int):
    if status != 0:
        detail = load_library().la_last_error().decode(errors="replace")
        raise LinAttnError(status, detail)


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return LA_F32
    if t.dtype == torch.bfloat16:
        return LA_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _check_cuda(*ts):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("all tensors must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")


def _stream_ptr(stream, device):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _decay_arg(decay, H):
    if decay is None:
        return None
    vals = [float(x) for x in (decay.tolist() if hasattr(decay, "tolist") else decay)]
    if len(vals) != H:
        raise ValueError(f"decay must have H={H} entries")
    return (ctypes.c_float * H)(*vals)


def forward(q, k, v, causal: bool = True, decay=None, out=None, *,
            path: int = 0, segment_chunks: int = 0, stream=None):
    """Linear attention over full sequences; q, k, v [B, H, N, d] on CUDA.

    causal=False: phi(Q)[phi(K)^T V] / phi(Q)[phi(K)^T 1].
    causal=True : running-state recurrence with optional per-head decay
    (`decay`: H floats in [0, 1]).  Returns `out` ([B, H, N, d], q's dtype).
    """
    torch = _torch()
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    if out is None:
        out = torch.empty_like(q)
    _check_cuda(q, k, v, out)
    B, H, N, d = q.shape
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.la_forward_ex(
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
            ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
            B, H, N, d, int(bool(causal)), _decay_arg(decay, H),
            _dtype_code(q), int(path), int(segment_chunks),
            _stream_ptr(stream, q.device))
    _raise_if(st)
    return out


def forward_variant(q, k, v, causal: bool = True, decay=None, out=None, *,
                    feature_map: str = "elu1", normalise: bool = True,
                    stream=None):
    """forward() with the feature map ("elu1" or "identity") and the
    normaliser selectable.  feature_map="identity", normalise=False with a
    decay is retention: o_i = sum_{j<=i} g^(i-j) (q_i . k_j) v_j."""
    torch = _torch()
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    if out is None:
        out = torch.empty_like(q)
    _check_cuda(q, k, v, out)
    B, H, N, d = q.shape
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.la_forward_variant(
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
            ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
            B, H, N, d, int(bool(causal)), _decay_arg(decay, H), _dtype_code(q),
            _variant(feature_map, normalise), _stream_ptr(stream, q.device))
    _raise_if(st)
    return out


def forward_gated(q, k, v, gates, out=None, *, feature_map: str = "elu1",
                  normalise: bool = True, stream=None):
    """Causal recurrence with a data-dependent scalar gate per token and
    head: gates [B, H, N] float32 on the GPU, values in [0, 1]
    (S_t = gates_t S_{t-1} + phi(k_t) v_t^T, z likewise)."""
    torch = _torch()
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    B, H, N, d = q.shape
    if tuple(gates.shape) != (B, H, N) or gates.dtype != torch.float32:
        raise ValueError("gates must be float32 [B, H, N]")
    if out is None:
        out = torch.empty_like(q)
    _check_cuda(q, k, v, out, gates)
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.la_forward_gated(
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
            ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(gates.data_ptr()), B, H, N, d, _dtype_code(q),
            _variant(feature_map, normalise), _stream_ptr(stream, q.device))
    _raise_if(st)
    return out


def decode_step_gated(S, z, q, k, v, gates, out=None, *, feature_map="elu1",
                      normalise=True, stream=None):
    """decode_step with this token's gate per head: gates [B, H] float32 on
    the GPU (S <- gates S + phi(k) v^T, z likewise)."""
    torch = _torch()
    if q.dim() != 3 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one [B, H, d] shape")
    B, H, d = q.shape
    if tuple(S.shape) != (B, H, d, d) or tuple(z.shape) != (B, H, d):
        raise ValueError("S must be [B, H, d, d] and z [B, H, d]")
    if tuple(gates.shape) != (B, H) or gates.dtype != torch.float32:
        raise ValueError("gates must be float32 [B, H]")
    if out is None:
        out = torch.empty_like(q)
    _check_cuda(S, z, q, k, v, out, gates)
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.la_decode_step_gated(
            ctypes.c_void_p(S.data_ptr()), ctypes.c_void_p(z.data_ptr()),
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
            ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(gates.data_ptr()), B, H, d, _dtype_code(q),
            _variant(feature_map, normalise), _stream_ptr(stream, q.device))
    _raise_if(st)
    return out


def decode_step_delta(S, q, k, v, beta, alpha=None, out=None, *, stream=None):
    """One delta-rule step per head (Gated DeltaNet with `alpha`): S [B, H,
    d, d] fp32 (S[a][c], a key feature) updated in place; beta, alpha
    [B, H] fp32 on the GPU; returns o = S_t^T q [B, H, d]."""
    torch = _torch()
    if q.dim() != 3 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one [B, H, d] shape")
    B, H, d = q.shape
    if tuple(S.shape) != (B, H, d, d) or S.dtype != torch.float32:
        raise ValueError("S must be float32 [B, H, d, d]")
    for name, t in (("beta", beta), ("alpha", alpha)):
        if t is not None and (tuple(t.shape) != (B, H) or t.dtype != torch.float32):
            raise ValueError(f"{name} must be float32 [B, H]")
    if out is None:
        out = torch.empty_like(q)
    _check_cuda(S, q, k, v, out, beta, *([alpha] if alpha is not None else []))
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.la_decode_step_delta(
            ctypes.c_void_p(S.data_ptr()), ctypes.c_void_p(q.data_ptr()),
            ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
            ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(beta.data_ptr()),
            ctypes.c_void_p(alpha.data_ptr() if alpha is not None else None),
            B, H, d, _dtype_code(q), _stream_ptr(stream, q.device))
    _raise_if(st)
    return out


def forward_delta(q, k, v, beta, alpha=None, out=None, S=None, *, stream=None):
    """The delta rule over sequences q, k, v [B, H, N, d] (DeltaNet; Gated
    DeltaNet with `alpha`): beta, alpha [B, H, N] fp32 on the GPU, one per
    token; S [B, H, d, d] fp32 (S[a][c], a key feature) the start state,
    updated in place to the state after the last token (None: start from
    zero).  Returns out [B, H, N, d] with o_t = S_t q_t."""
    torch = _torch()
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    B, H, N, d = q.shape
    for name, t in (("beta", beta), ("alpha", alpha)):
        if t is not None and (tuple(t.shape) != (B, H, N) or t.dtype != torch.float32):
            raise ValueError(f"{name} must be float32 [B, H, N]")
    if S is not None and (tuple(S.shape) != (B, H, d, d) or S.dtype != torch.float32):
        raise ValueError("S must be float32 [B, H, d, d]")
    if out is None:
        out = torch.empty_like(q)
    _check_cuda(q, k, v, out, beta, *[t for t in (alpha, S) if t is not None])
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.la_forward_delta(
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
            ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(beta.data_ptr()),
            ctypes.c_void_p(alpha.data_ptr() if alpha is not None else None),
            ctypes.c_void_p(S.data_ptr() if S is not None else None),
            B, H, N, d, _dtype_code(q), _stream_ptr(stream, q.device))
    _raise_if(st)
    return out


def forward_causal_state(q, k, v, decay=None, out=None, S=None, z=None, *,
                         stream=None):
    """Causal forward that also returns the final state: (out, S, z) with
    S [B, H, d, d] and z [B, H, d] in fp32 -- the state after the last token,
    in the layout decode_step takes, so that a decode continues the
    sequence."""
    torch = _torch()
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    B, H, N, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if S is None:
        S = torch.empty(B, H, d, d, dtype=torch.float32, device=q.device)
    if z is None:
        z = torch.empty(B, H, d, dtype=torch.float32, device=q.device)
    if tuple(S.shape) != (B, H, d, d) or tuple(z.shape) != (B, H, d):
        raise ValueError("S must be [B, H, d, d] and z [B, H, d]")
    if S.dtype != torch.float32 or z.dtype != torch.float32:
        raise TypeError("S and z must be float32")
    _check_cuda(q, k, v, out, S, z)
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.la_forward_causal_state(
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
            ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(S.data_ptr()), ctypes.c_void_p(z.data_ptr()),
            B, H, N, d, _decay_arg(decay, H), _dtype_code(q),
            _stream_ptr(stream, q.device))
    _raise_if(st)
    return out, S, z


def decode_step(S, z, q, k, v, out=None, *, decay=None, feature_map="elu1",
                normalise=True, stream=None):
    """One decode step per head: S, z (fp32, [B, H, d, d] / [B, H, d]) are
    updated in place (S <- g S + phi(k) v^T, z <- g z + phi(k), with the
    per-head decay g from `decay`, H floats in [0, 1], or 1); q, k, v
    [B, H, d]; returns out [B, H, d].  feature_map / normalise as in
    forward_variant."""
    torch = _torch()
    if q.dim() != 3 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one [B, H, d] shape")
    B, H, d = q.shape
    if tuple(S.shape) != (B, H, d, d) or tuple(z.shape) != (B, H, d):
        raise ValueError("S must be [B, H, d, d] and z [B, H, d]")
    if S.dtype != torch.float32 or z.dtype != torch.float32:
        raise TypeError("S and z must be float32")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    if out is None:
        out = torch.empty_like(q)
    _check_cuda(S, z, q, k, v, out)
    lib = load_library()
    with torch.cuda.device(q.device):
        st = lib.la_decode_step_variant(
            ctypes.c_void_p(S.data_ptr()), ctypes.c_void_p(z.data_ptr()),
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
            ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
            B, H, d, _decay_arg(decay, H), _dtype_code(q),
            _variant(feature_map, normalise), _stream_ptr(stream, q.device))
    _raise_if(st)
    return out


def kernel_launch_count() -> int:
    """Kernels enqueued by the library in this process so far."""
    return int(load_library().la_kernel_launch_count())


def check_device_status(stream=None, device=None):
    """Synchronise the stream and raise if a kernel reported a device-side
    failure (a bounded wait that ran out)."""
    torch = _torch()
    dev = device if device is not None else torch.cuda.current_device()
    with torch.cuda.device(dev):
        st = load_library().la_check_device_status(_stream_ptr(stream, dev))
    _raise_if(st)


def host_workspace_bytes(shape, dtype) -> int:
    """Device workspace bytes that forward_host needs for [B, H, N, d]."""
    torch = _torch()
    code = LA_BF16 if dtype == torch.bfloat16 else LA_F32 if dtype == torch.float32 else -1
    if code < 0:
        raise TypeError(f"unsupported dtype {dtype} (float32 or bfloat16)")
    B, H, N, d = (int(x) for x in shape)
    return int(load_library().la_forward_host_workspace_bytes(B, H, N, d, code))


def forward_host(q, k, v, causal: bool = True, decay=None, out=None, *,
                 workspace=None, device=None, stream=None):
    """forward() on HOST tensors q, k, v [B, H, N, d] (page-locked for full
    speed): the library copies them to the GPU, runs the forward and copies
    the result into `out` (a host tensor, allocated page-locked if None),
    pipelined over groups of heads.  `workspace` is a uint8 CUDA tensor of at
    least host_workspace_bytes(q.shape, q.dtype) bytes (allocated if None).
    The call is asynchronous: `out` is complete once `stream` (default: the
    current stream of `device`) has passed it, e.g. after
    torch.cuda.current_stream().synchronize()."""
    torch = _torch()
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    for t in (q, k, v):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("forward_host takes contiguous host tensors")
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    if out.is_cuda or not out.is_contiguous() or out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("out must be a contiguous host tensor like q")
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    need = host_workspace_bytes(q.shape, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    if not workspace.is_cuda or workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace must be a CUDA tensor of at least {need} bytes")
    B, H, N, d = q.shape
    lib = load_library()
    with torch.cuda.device(workspace.device):
        st = lib.la_forward_host(
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
            ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
            B, H, N, d, int(bool(causal)), _decay_arg(decay, H),
            _dtype_code(q), ctypes.c_void_p(workspace.data_ptr()),
            ctypes.c_size_t(workspace.numel() * workspace.element_size()),
            _stream_ptr(stream, workspace.device))
    _raise_if(st)
    return out

"""Double-precision CPU oracle for kernelised (elu+1) linear attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import this package.  The
product path (``linear_attention_feature_gb300``) never imports it, and the
oracle shares no code with the CUDA library.

The arithmetic lives in ``la_oracle.c`` (plain C loops in double precision,
each routine citing the passage it follows); this module only compiles it
with gcc and marshals numpy arrays through ctypes.  Inputs of any float dtype
are widened to float64 before the call, so the oracle sees exactly the values
the GPU sees.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "la_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liblaoracle.so")
_lock = threading.Lock()
_lib = None

FMAP_ELU1 = 0
FMAP_IDENTITY = 1


def build(force: bool = False) -> str:
    """Compile la_oracle.c into a shared library (gcc, -O2, no fast-math)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        os.makedirs(_OUT_DIR, exist_ok=True)
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", "-Wall", "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    # LA_ORACLE_LIB: a separately built copy of la_oracle.c (the tests run
    # the oracle's pins against a copy built with address and
    # undefined-behaviour sanitizers)
    path = os.environ.get("LA_ORACLE_LIB") or build()
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    L = ctypes.c_long
    I = ctypes.c_int
    lib.ora_phi.restype = ctypes.c_double
    lib.ora_phi.argtypes = [ctypes.c_double]
    lib.ora_feature_map.restype = None
    lib.ora_feature_map.argtypes = [P, P, L, I]
    lib.ora_noncausal_state.argtypes = [P, P, P, P, L, L, L, I]
    lib.ora_state_read.argtypes = [P, P, P, P, L, L, L, I, I]
    lib.ora_noncausal.argtypes = [P, P, P, P, L, L, L, I, I, I]
    lib.ora_recurrent_step.argtypes = [P, P, P, P, P, P, L, ctypes.c_double, I, I]
    lib.ora_causal.argtypes = [P, P, P, P, L, L, L, P, I, I, I]
    lib.ora_causal_state.argtypes = [P, P, P, P, L, L, L, P, I]
    lib.ora_causal_gated.argtypes = [P, P, P, P, P, L, L, L, I, I, I]
    lib.ora_delta_step.argtypes = [P, P, P, P, P, P, P, L, L]
    lib.ora_delta_forward.argtypes = [P, P, P, P, P, P, P, L, L, L, I]
    lib.ora_decode_step.argtypes = [P, P, P, P, P, P, L, L, P, I]
    lib.ora_quadratic.argtypes = [P, P, P, P, L, L, L, P, I, I, P]
    lib.ora_chunked.argtypes = [P, P, P, P, L, L, L, P, L, L]
    for name in ("ora_noncausal_state", "ora_state_read", "ora_noncausal",
                 "ora_causal_state", "ora_causal_gated", "ora_delta_step",
                 "ora_delta_forward",
                 "ora_recurrent_step", "ora_causal", "ora_decode_step",
                 "ora_quadratic", "ora_chunked"):
        getattr(lib, name).restype = I
    _lib = lib
    return lib


def _f64(x) -> np.ndarray:
    """Widen any array-like (numpy, or a CPU torch tensor) to C-contiguous
    float64.  bf16 torch tensors are converted through float32 first, which is
    exact."""
    if hasattr(x, "detach"):  # torch tensor, without importing torch here
        x = x.detach().cpu()
        if str(x.dtype) == "torch.bfloat16":
            x = x.float()
        x = x.numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, name: str):
    if rc != 0:
        raise RuntimeError(f"oracle {name} failed with code {rc}")


def _seq_shape(q):
    """[..., N, d] -> (BH, N, d) with all leading dims flattened."""
    if q.ndim < 2:
        raise ValueError("expected at least [N, d]")
    N, d = q.shape[-2], q.shape[-1]
    BH = int(np.prod(q.shape[:-2])) if q.ndim > 2 else 1
    return BH, N, d


def _decay_per_head(decay, q_shape, BH):
    """Expand a per-head decay (length H, the second-to-last-but-one axis of
    a [B, H, N, d] input) to one value per flattened head."""
    if decay is None:
        return None
    g = np.asarray(decay, dtype=np.float64).reshape(-1)
    if g.size == BH:
        return np.ascontiguousarray(g)
    if len(q_shape) >= 3 and g.size == q_shape[-3]:
        reps = BH // g.size
        return np.ascontiguousarray(np.tile(g, reps))
    raise ValueError("decay must have H or B*H entries")


def phi(x) -> np.ndarray:
    """Feature map elu(x)+1 (alpha = 1) applied elementwise."""
    a = _f64(x)
    y = np.empty_like(a)
    _load().ora_feature_map(_ptr(a), _ptr(y), a.size, FMAP_ELU1)
    return y


def phi_scalar(x: float) -> float:
    return float(_load().ora_phi(float(x)))


def noncausal(q, k, v, *, fmap=FMAP_ELU1, normalise=True, nthreads=1):
    """phi(Q)[phi(K)^T V] / phi(Q)[phi(K)^T 1] per head; inputs [..., N, d]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    BH, N, d = _seq_shape(q)
    out = np.empty_like(q)
    _check(_load().ora_noncausal(_ptr(q), _ptr(k), _ptr(v), _ptr(out), BH, N,
                                 d, fmap, int(normalise), int(nthreads)),
           "noncausal")
    return out


def noncausal_state(k, v, *, fmap=FMAP_ELU1):
    """(S, z) with S = phi(K)^T V ([..., d, d]) and z = phi(K)^T 1."""
    k, v = _f64(k), _f64(v)
    BH, N, d = _seq_shape(k)
    S = np.empty(k.shape[:-2] + (d, d))
    z = np.empty(k.shape[:-2] + (d,))
    _check(_load().ora_noncausal_state(_ptr(k), _ptr(v), _ptr(S), _ptr(z), BH,
                                       N, d, fmap), "noncausal_state")
    return S, z


def state_read(S, z, q, *, fmap=FMAP_ELU1, normalise=True):
    """y_i = phi(q_i)^T S / phi(q_i)^T z for queries q [..., M, d]."""
    S, z, q = _f64(S), _f64(z), _f64(q)
    BH, M, d = _seq_shape(q)
    out = np.empty_like(q)
    _check(_load().ora_state_read(_ptr(S), _ptr(z), _ptr(q), _ptr(out), BH, M,
                                  d, fmap, int(normalise)), "state_read")
    return out


def causal(q, k, v, decay=None, *, fmap=FMAP_ELU1, normalise=True,
           nthreads=1):
    """Causal recurrence with optional per-head decay; inputs [..., N, d]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    BH, N, d = _seq_shape(q)
    g = _decay_per_head(decay, q.shape, BH)
    out = np.empty_like(q)
    _check(_load().ora_causal(_ptr(q), _ptr(k), _ptr(v), _ptr(out), BH, N, d,
                              _ptr(g) if g is not None else None, fmap,
                              int(normalise), int(nthreads)), "causal")
    return out


def causal_gated(q, k, v, alpha, *, fmap=FMAP_ELU1, normalise=True, nthreads=1):
    """Causal recurrence with a scalar gate per token and head: alpha
    [..., N] (the leading dimensions of q); inputs [..., N, d]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    BH, N, d = _seq_shape(q)
    a = np.ascontiguousarray(np.asarray(alpha, dtype=np.float64))
    if a.shape != q.shape[:-1]:
        raise ValueError("alpha must have the shape of q without its last axis")
    out = np.empty_like(q)
    _check(_load().ora_causal_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(out),
                                    BH, N, d, fmap, int(normalise), int(nthreads)),
           "causal_gated")
    return out


def delta_step(S, q, k, v, beta, alpha=None):
    """Delta-rule step on float64 state S [..., d, d] (S[a][c], a key feature,
    c value column; updated in place): S <- alpha S + beta k (v - alpha S^T k)^T
    in this layout; returns o = S^T q [..., d].  beta, alpha: one per head."""
    if S.dtype != np.float64 or not S.flags.c_contiguous:
        raise TypeError("S must be a C-contiguous float64 array (in place)")
    q, k, v = _f64(q), _f64(k), _f64(v)
    d = q.shape[-1]
    BH = q.size // d
    b = np.ascontiguousarray(np.asarray(beta, dtype=np.float64).reshape(-1))
    a = None if alpha is None else np.ascontiguousarray(
        np.asarray(alpha, dtype=np.float64).reshape(-1))
    if b.size != BH or (a is not None and a.size != BH):
        raise ValueError("beta and alpha need one entry per head")
    out = np.empty_like(q)
    _check(_load().ora_delta_step(_ptr(S), _ptr(q), _ptr(k), _ptr(v), _ptr(b),
                                  _ptr(a) if a is not None else None, _ptr(out),
                                  BH, d), "delta_step")
    return out


def delta_forward(q, k, v, beta, alpha=None, S0=None, *, nthreads=1):
    """The delta rule over sequences q, k, v [..., N, d]: token by token
    S <- alpha_t S + beta_t k_t (v_t - alpha_t S^T k_t)^T (S[a][c], a key
    feature), o_t = S^T q_t; beta, alpha [..., N] (alpha None: 1); S0
    [..., d, d] the start state (None: zero).  Returns (out [..., N, d], S
    after the last token)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    BH, N, d = _seq_shape(q)
    b = np.ascontiguousarray(np.asarray(beta, dtype=np.float64).reshape(-1))
    a = None if alpha is None else np.ascontiguousarray(
        np.asarray(alpha, dtype=np.float64).reshape(-1))
    if b.size != BH * N or (a is not None and a.size != BH * N):
        raise ValueError("beta and alpha need one entry per token and head")
    S = (np.zeros(q.shape[:-2] + (d, d)) if S0 is None
         else np.array(_f64(S0), dtype=np.float64, order="C", copy=True))
    out = np.empty_like(q)
    _check(_load().ora_delta_forward(_ptr(S), _ptr(q), _ptr(k), _ptr(v), _ptr(b),
                                     _ptr(a) if a is not None else None, _ptr(out),
                                     BH, N, d, int(nthreads)), "delta_forward")
    return out, S


def causal_state(k, v, decay=None, *, fmap=FMAP_ELU1):
    """Final (S, z) of the causal recurrence after all N tokens of k, v
    [..., N, d], with optional per-head decay: S [..., d, d], z [..., d]."""
    k, v = _f64(k), _f64(v)
    BH, N, d = _seq_shape(k)
    g = _decay_per_head(decay, k.shape, BH)
    S = np.empty(k.shape[:-2] + (d, d))
    z = np.empty(k.shape[:-2] + (d,))
    _check(_load().ora_causal_state(_ptr(k), _ptr(v), _ptr(S), _ptr(z), BH, N, d,
                                    _ptr(g) if g is not None else None, fmap),
           "causal_state")
    return S, z


def recurrent_step(S, z, q, k, v, g=1.0, *, fmap=FMAP_ELU1, normalise=True):
    """One in-place step of the recurrence on a single head's float64 state
    arrays S [d, d], z [d]; returns the output row."""
    if S.dtype != np.float64 or not S.flags.c_contiguous:
        raise TypeError("S must be a C-contiguous float64 array (in place)")
    if z.dtype != np.float64 or not z.flags.c_contiguous:
        raise TypeError("z must be a C-contiguous float64 array (in place)")
    q, k, v = _f64(q), _f64(k), _f64(v)
    d = q.shape[-1]
    out = np.empty(d)
    _check(_load().ora_recurrent_step(_ptr(S), _ptr(z), _ptr(q), _ptr(k),
                                      _ptr(v), _ptr(out), d, float(g), fmap,
                                      int(normalise)), "recurrent_step")
    return out


def decode_step(S, z, q, k, v, decay=None, *, nthreads=1):
    """Decode one token per head on float64 state S [..., d, d], z [..., d]
    (updated in place); q, k, v [..., d].  Returns out [..., d]."""
    for a, name in ((S, "S"), (z, "z")):
        if a.dtype != np.float64 or not a.flags.c_contiguous:
            raise TypeError(f"{name} must be a C-contiguous float64 array")
    q, k, v = _f64(q), _f64(k), _f64(v)
    d = q.shape[-1]
    BH = q.size // d
    g = None
    if decay is not None:
        g = np.ascontiguousarray(np.asarray(decay, dtype=np.float64).reshape(-1))
        if g.size != BH:
            raise ValueError("decay for decode must have one entry per head")
    out = np.empty_like(q)
    _check(_load().ora_decode_step(_ptr(S), _ptr(z), _ptr(q), _ptr(k), _ptr(v),
                                   _ptr(out), BH, d,
                                   _ptr(g) if g is not None else None,
                                   int(nthreads)), "decode_step")
    return out


def quadratic(q, k, v, decay=None, *, fmap=FMAP_ELU1, normalise=True,
              return_weights=False):
    """Masked parallel form; O(N^2 d), small N only."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    BH, N, d = _seq_shape(q)
    g = _decay_per_head(decay, q.shape, BH)
    out = np.empty_like(q)
    W = np.empty(q.shape[:-2] + (N, N)) if return_weights else None
    _check(_load().ora_quadratic(_ptr(q), _ptr(k), _ptr(v), _ptr(out), BH, N,
                                 d, _ptr(g) if g is not None else None, fmap,
                                 int(normalise),
                                 _ptr(W) if W is not None else None),
           "quadratic")
    return (out, W) if return_weights else out


def chunked(q, k, v, decay=None, *, block=64, segments=1):
    """Chunked block-algebra prototype (test-only cross-check)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    BH, N, d = _seq_shape(q)
    g = _decay_per_head(decay, q.shape, BH)
    out = np.empty_like(q)
    _check(_load().ora_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(out), BH, N, d,
                               _ptr(g) if g is not None else None, int(block),
                               int(segments)), "chunked")
    return out

"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (automatic kernel and segment choice).  The GPU computes every
head and the double-precision oracle recomputes EVERY head (threaded over all
host cores); the two are compared element by element (max row-relative error
over every row of every head: 1e-4 for fp32 inputs, 2e-2 for bf16).  Every
head is an independent recurrence ("Story of Attention - Part 5", section 1a,
causal and matrix forms), so every head's output is defined and checked: a
scheduling error that touched only some work items (a ticket decoded to the
wrong head or segment, a look-back chain in a later wave) would show here."""
import os

import numpy as np
import pytest

import oracle
import linear_attention_feature_gb300 as la
from linear_attention_feature_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
CORES = os.cpu_count() or 1


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.build.build()
    la.load_library()


def per_head_errors(y, q, k, v, causal, decay=None):
    """Row-relative error of every head of y [B, H, N, d] against the oracle,
    heads taken in groups of the host's core count (bounded host memory)."""
    B, H, N, d = q.shape
    BH = B * H
    flat = [t.reshape(BH, N, d) for t in (y, q, k, v)]
    g = None if decay is None else np.array([decay[i % H] for i in range(BH)])
    errs = np.empty(BH)
    step = max(CORES, 1)
    for h0 in range(0, BH, step):
        sl = slice(h0, min(BH, h0 + step))
        ys, qs, ks, vs = (t[sl].float().cpu() for t in flat)
        if causal:
            ref = oracle.causal(qs, ks, vs, None if g is None else g[sl],
                                nthreads=CORES)
        else:
            ref = oracle.noncausal(qs, ks, vs, nthreads=CORES)
        for i in range(ref.shape[0]):
            errs[h0 + i] = wl.max_row_rel_err(ys[i], ref[i])
    return errs


def full_parity(w, causal, decay=None, seed=0):
    q, k, v = wl.make_workload_qkv(w, seed=seed, device="cuda")
    y = la.forward(q, k, v, causal=causal, decay=decay)
    la.check_device_status()
    errs = per_head_errors(y, q, k, v, causal, decay)
    tol = wl.TOL[w.dtype]
    bad = np.nonzero(~(errs <= tol))[0]
    assert bad.size == 0, (
        f"{bad.size} of {errs.size} heads over {tol}: first (b, h) = "
        f"{divmod(int(bad[0]), w.H)}, error {errs[bad[0]]:.3e}")
    return float(errs.max())


def test_fp32_causal_small_full():
    w = wl.WORKLOADS["fp32_causal_small"]
    assert full_parity(w, True) <= wl.TOL["f32"]


@pytest.mark.parametrize("causal", [True, False])
def test_b4h16_n4096_d64_full(causal):
    w = wl.WORKLOADS["bf16_b4h16_n4096_d64"]
    assert full_parity(w, causal) <= wl.TOL["bf16"]


def test_b2h16_n32768_d128_full():
    w = wl.WORKLOADS["bf16_b2h16_n32768_d128"]
    assert full_parity(w, True) <= wl.TOL["bf16"]


def test_decay_b4h8_n16384_d128_full():
    w = wl.WORKLOADS["bf16_decay_b4h8_n16384_d128"]
    assert full_parity(w, True, decay=list(w.decay)) <= wl.TOL["bf16"]


def test_decode_b256h32_d128_full():
    """All 8192 heads, every step.  Prefill: 1024 steps from a zero state on
    both sides, every output compared, then the GPU's fp32 state against the
    oracle's.  The oracle's prefilled state, rounded to fp32, then becomes
    the starting state of both sides (so both continue from identical
    buffers), and the 1024 decode steps are compared at every step and on
    the final state."""
    w = wl.WORKLOADS["decode_b256h32_d128"]
    B, H, d = w.B, w.H, w.d
    P, T = w.extra["prefill"], w.extra["steps"]
    q, k, v = wl.make_decode_tokens(B, H, d, P + T, "bf16", seed=100, device="cuda")
    S = torch.zeros(B, H, d, d, device="cuda")
    z = torch.zeros(B, H, d, device="cuda")
    So = np.zeros((B, H, d, d))
    zo = np.zeros((B, H, d))
    out = torch.empty(B, H, d, dtype=torch.bfloat16, device="cuda")
    worst = 0.0

    def step(t):
        nonlocal worst
        la.decode_step(S, z, q[t], k[t], v[t], out=out)
        y = out.cpu()
        r = oracle.decode_step(So, zo, q[t].cpu(), k[t].cpu(), v[t].cpu(),
                               nthreads=CORES)
        err = wl.max_row_rel_err(y, r)
        assert err <= wl.TOL["bf16"], (t, err)
        worst = max(worst, err)

    for t in range(P):
        step(t)
    la.check_device_status()
    np.testing.assert_allclose(S.cpu().numpy(), So, rtol=1e-3, atol=1e-3)
    np.testing.assert_allclose(z.cpu().numpy(), zo, rtol=1e-3, atol=1e-3)
    # both sides continue from the oracle's prefill rounded to fp32
    S32 = torch.from_numpy(So.astype(np.float32))
    z32 = torch.from_numpy(zo.astype(np.float32))
    S.copy_(S32.cuda())
    z.copy_(z32.cuda())
    So[...] = S32.double().numpy()
    zo[...] = z32.double().numpy()
    for t in range(P, P + T):
        step(t)
    la.check_device_status()
    np.testing.assert_allclose(S.cpu().numpy(), So, rtol=1e-3, atol=1e-3)
    np.testing.assert_allclose(z.cpu().numpy(), zo, rtol=1e-3, atol=1e-3)
    assert worst <= wl.TOL["bf16"]


def test_one_million_token_sequence():
    """A single 2^20-token head (the largest case here): the look-back chains
    over hundreds of segments; every row must match the oracle."""
    N = 1 << 20
    q, k, v = wl.make_qkv(1, 1, N, 64, "bf16", seed=21, device="cuda")
    y = la.forward(q, k, v, causal=True)
    la.check_device_status()
    ref = oracle.causal(q.float().cpu(), k.float().cpu(), v.float().cpu())
    assert wl.max_row_rel_err(y[0, 0].cpu(), ref[0, 0]) <= wl.TOL["bf16"]

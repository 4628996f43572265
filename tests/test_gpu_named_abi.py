"""The two calls the boundary is named for, la_forward and la_decode_step,
invoked directly through ctypes on device buffers (no Python wrapper in
between) and compared with the double-precision oracle.

la_forward: the causal running-state form ("Linear Attention", causal
running statistics; "Story of Attention - Part 5", section 1a) with and
without a per-head decay, and the non-causal matrix form, for bf16 (tensor
cores) and fp32 (CUDA cores).  la_decode_step: update, then read, for a few
consecutive tokens on a caller-owned state."""
import ctypes

import numpy as np
import pytest

import oracle
import linear_attention_feature_gb300 as la
from linear_attention_feature_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.build.build()
    return la.load_library()


def ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("form", ["causal", "decay", "noncausal"])
def test_la_forward_direct(lib, dtype, d, form):
    B, H, N = 2, 3, 700
    q, k, v = wl.make_qkv(B, H, N, d, dtype, seed=40 + d)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out = torch.empty_like(qd)
    decay = [0.96875, 0.5, 0.999][:H] if form == "decay" else None
    dec = (ctypes.c_float * H)(*decay) if decay else None
    code = la.LA_BF16 if dtype == "bf16" else la.LA_F32
    st = lib.la_forward(ptr(qd), ptr(kd), ptr(vd), ptr(out), B, H, N, d,
                        0 if form == "noncausal" else 1, dec, code, stream())
    assert st == 0, lib.la_last_error().decode()
    assert lib.la_check_device_status(stream()) == 0
    if form == "noncausal":
        ref = oracle.noncausal(q, k, v, nthreads=8)
    else:
        ref = oracle.causal(q, k, v, decay, nthreads=8)
    assert wl.max_row_rel_err(out.cpu(), ref) <= wl.TOL[dtype]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d", [64, 128])
def test_la_decode_step_direct(lib, dtype, d):
    B, H, T = 3, 5, 6
    q, k, v = wl.make_decode_tokens(B, H, d, T, dtype, seed=50 + d)
    S = torch.zeros(B, H, d, d, device="cuda")
    z = torch.zeros(B, H, d, device="cuda")
    So, zo = np.zeros((B, H, d, d)), np.zeros((B, H, d))
    code = la.LA_BF16 if dtype == "bf16" else la.LA_F32
    for t in range(T):
        qd, kd, vd = q[t].cuda(), k[t].cuda(), v[t].cuda()
        out = torch.empty_like(qd)
        st = lib.la_decode_step(ptr(S), ptr(z), ptr(qd), ptr(kd), ptr(vd),
                                ptr(out), B, H, d, code, stream())
        assert st == 0, lib.la_last_error().decode()
        assert lib.la_check_device_status(stream()) == 0
        ref = oracle.decode_step(So, zo, q[t], k[t], v[t])
        assert wl.max_row_rel_err(out.cpu(), ref) <= wl.TOL[dtype]
    np.testing.assert_allclose(S.cpu().numpy(), So, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(z.cpu().numpy(), zo, rtol=1e-5, atol=1e-6)

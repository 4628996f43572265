"""The allocation-free causal entry point, la_forward_causal_noalloc.

It serves callers that must not allocate device memory while they run
(allocation-free graph capture, hosts that reserve all memory up front,
plug-in layers handed their buffers).  It runs the causal tensor-core kernel
with its workspace in a fixed static device array, so these tests check,
through the C ABI, that its outputs match la_forward's on the same inputs,
call after call (the array keeps the previous call's contents, which must
not leak into the next result).  The file is named to be collected last.
"""
import ctypes

import pytest

import linear_attention_feature_gb300 as la
from linear_attention_feature_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
TOL = wl.TOL["bf16"]


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.build.build()
    lib = la.load_library()
    V, I = ctypes.c_void_p, ctypes.c_int
    lib.la_forward_causal_noalloc.argtypes = [
        V, V, V, V, I, I, I, I, ctypes.POINTER(ctypes.c_float), V]
    lib.la_forward_causal_noalloc.restype = I
    return lib


def noalloc(lib, q, k, v, out, decay=None):
    B, H, N, d = q.shape
    dec = (ctypes.c_float * H)(*decay) if decay is not None else None
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.la_forward_causal_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
        B, H, N, d, dec, stream)
    return st


@pytest.mark.parametrize("d, decay", [
    (64, None), (128, None), (128, [0.96875, 0.5, 0.99, 1.0])])
def test_noalloc_matches_la_forward_two_calls_in_a_row(lib, d, decay):
    B, H, N = 2, 4, 1300
    ref_in = [wl.make_qkv(B, H, N, d, "bf16", seed=s) for s in (11, 12)]
    for q, k, v in ref_in:  # second call reuses the scratch of the first
        q, k, v = q.cuda(), k.cuda(), v.cuda()
        out = torch.empty_like(q)
        assert noalloc(lib, q, k, v, out, decay) == 0, \
            lib.la_last_error().decode()
        ref = la.forward(q, k, v, causal=True, decay=decay)
        la.check_device_status()
        assert wl.max_row_rel_err(out.cpu(), ref.cpu()) <= TOL


@pytest.mark.parametrize("d, decay", [(64, None), (128, [0.96875, 0.75, 1.0])])
def test_noalloc_matches_the_oracle(lib, d, decay):
    # parity of the allocation-free call on its own, independent of
    # la_forward: the double-precision oracle, every head, twice in a row
    import oracle
    B, H, N = 1, 3, 900
    q, k, v = wl.make_qkv(B, H, N, d, "bf16", seed=13)
    ref = oracle.causal(q, k, v, decay, nthreads=8)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    for _ in range(2):
        out = torch.empty_like(qd)
        assert noalloc(lib, qd, kd, vd, out, decay) == 0, \
            lib.la_last_error().decode()
        la.check_device_status()
        assert wl.max_row_rel_err(out.cpu(), ref) <= TOL


def test_noalloc_long_sequence_fits_by_longer_segments(lib):
    # 64 heads of d=128 over 16 chunks: the default segmentation would need
    # more than the static scratch, so segments are lengthened to fit.
    q, k, v = (t.cuda() for t in wl.make_qkv(4, 16, 2048, 128, "bf16", seed=3))
    out = torch.empty_like(q)
    for _ in range(2):
        assert noalloc(lib, q, k, v, out) == 0, lib.la_last_error().decode()
        ref = la.forward(q, k, v, causal=True)
        la.check_device_status()
        assert wl.max_row_rel_err(out.cpu(), ref.cpu()) <= TOL


def test_noalloc_rejects_what_it_cannot_run(lib):
    q = torch.zeros(1, 1, 8, 96, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    assert noalloc(lib, q, q.clone(), q.clone(), out) == 2  # d = 96
    assert "d must be 64 or 128" in lib.la_last_error().decode()
    big = torch.zeros(1, 5_000_000, 1, 64, dtype=torch.bfloat16, device="cuda")
    big_out = torch.empty_like(big)
    # 5M heads: even the per-item flags exceed the 16 MiB scratch
    assert noalloc(lib, big, big.clone(), big.clone(), big_out) == 2
    assert "more workspace" in lib.la_last_error().decode()


@pytest.mark.parametrize("d", [64, 128])
def test_noalloc_makes_no_workspace_allocation(lib, d):
    # with the next workspace allocation set to fail, an allocating call
    # would return LA_ERR_NO_MEMORY; the allocation-free call succeeds and
    # leaves the hook armed, which the ordinary call after it then consumes
    lib.la_debug_fail_next_allocs.argtypes = [ctypes.c_int]
    lib.la_debug_fail_next_allocs.restype = ctypes.c_int
    q, k, v = (t.cuda() for t in wl.make_qkv(1, 4, 1300, d, "bf16", seed=21))
    out = torch.empty_like(q)
    assert lib.la_debug_fail_next_allocs(1) == 0
    try:
        assert noalloc(lib, q, k, v, out) == 0, lib.la_last_error().decode()
        la.check_device_status()
        with pytest.raises(la.LinAttnError) as ei:
            la.forward(q, k, v, causal=True)
        assert ei.value.status == 4
    finally:
        lib.la_debug_fail_next_allocs(0)
    ref = la.forward(q, k, v, causal=True)
    la.check_device_status()
    assert wl.max_row_rel_err(out.cpu(), ref.cpu()) <= TOL

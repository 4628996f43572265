"""The debug build (liblinattn_debug.so, compiled with -DLA_DEBUG): its
tensor-core kernels check the computed indices of their global-memory
accesses (item decode, published states and flags, look-back reads, gate
slots, final state) and report a failed check as LA_ERR_INTERNAL without
trapping.  Over small and ragged shapes that reach every tail, mask and
segment path, no check may fail and every output must match the oracle."""
import pytest

import oracle
import linear_attention_feature_gb300 as la
from linear_attention_feature_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
TOL = wl.TOL["bf16"]


@pytest.fixture(scope="module")
def debug_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.build.build()
    la.load_library()
    path = la.build.build(debug=True)
    saved = la._lib
    la._lib = la.load_library(path)
    try:
        yield la._lib
    finally:
        la._lib = saved


def gates_for(B, H, N, seed):
    g = torch.Generator().manual_seed(seed)
    a = 0.85 + 0.15 * torch.rand(B, H, N, generator=g)
    a[:, :, ::53] = 1.0
    a[0, 0, min(70, N // 2)] = 0.0  # a reset
    return a


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 129, 1000])
@pytest.mark.parametrize("seg", [0, 1, 3])
def test_debug_build_causal(debug_lib, d, N, seg):
    q, k, v = wl.make_qkv(1, 3, N, d, "bf16", seed=900 + N + d)
    y = la.forward(q.cuda(), k.cuda(), v.cuda(), causal=True, path=2,
                   segment_chunks=seg).cpu()
    la.check_device_status()  # raises on LA_ERR_INTERNAL
    assert wl.max_row_rel_err(y, oracle.causal(q, k, v, nthreads=8)) <= TOL


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [300, 1000])
def test_debug_build_decay_and_state(debug_lib, d, N):
    q, k, v = wl.make_qkv(2, 2, N, d, "bf16", seed=950 + N + d)
    dec = [0.97, 0.6]
    y, S, z = la.forward_causal_state(q.cuda(), k.cuda(), v.cuda(), decay=dec)
    la.check_device_status()
    assert wl.max_row_rel_err(y.cpu(), oracle.causal(q, k, v, dec, nthreads=8)) <= TOL
    S_ref, z_ref = (torch.from_numpy(x) for x in oracle.causal_state(k, v, dec))
    assert float((S.cpu().double() - S_ref).abs().max()) <= TOL * float(S_ref.abs().max())
    assert float((z.cpu().double() - z_ref).abs().max()) <= TOL * float(z_ref.abs().max())


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [200, 700])
def test_debug_build_gated(debug_lib, d, N):
    q, k, v = wl.make_qkv(1, 2, N, d, "bf16", seed=970 + N + d)
    a = gates_for(1, 2, N, 971 + N)
    y = la.forward_gated(q.cuda(), k.cuda(), v.cuda(), a.cuda()).cpu()
    la.check_device_status()
    ref = oracle.causal_gated(q.float(), k.float(), v.float(), a.double().numpy(), nthreads=8)
    assert wl.max_row_rel_err(y, ref) <= TOL


@pytest.mark.parametrize("N", [1, 333, 2000])
def test_debug_build_noncausal(debug_lib, N):
    q, k, v = wl.make_qkv(2, 3, N, 64, "bf16", seed=990 + N)
    y = la.forward(q.cuda(), k.cuda(), v.cuda(), causal=False, path=2).cpu()
    la.check_device_status()
    assert wl.max_row_rel_err(y, oracle.noncausal(q, k, v, nthreads=8)) <= TOL

"""GPU parity of the tcgen05 non-causal kernel (phi(K)^T [V | 1] reduced over
the sequence, then read by phi(Q)) against the double-precision oracle;
tolerance 2e-2 max row-relative error (bf16 inputs, fp32 accumulation)."""
import pytest

import oracle
import linear_attention_feature_gb300 as la
from linear_attention_feature_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
TOL = wl.TOL["bf16"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.build.build()
    la.load_library()


def run_tc(q, k, v, seg=0):
    y = la.forward(q.cuda(), k.cuda(), v.cuda(), causal=False, path=2,
                   segment_chunks=seg)
    la.check_device_status()
    return y.cpu()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 100, 128, 129, 300, 1000])
def test_noncausal_tc_ragged(d, N):
    q, k, v = wl.make_qkv(2, 3, N, d, "bf16", seed=N + 7 * d)
    y = run_tc(q, k, v)
    assert wl.max_row_rel_err(y, oracle.noncausal(q, k, v, nthreads=8)) <= TOL


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("seg", [1, 3])
def test_noncausal_tc_segments(d, seg):
    q, k, v = wl.make_qkv(1, 4, 1100, d, "bf16", seed=seg)
    y = run_tc(q, k, v, seg=seg)
    assert wl.max_row_rel_err(y, oracle.noncausal(q, k, v, nthreads=8)) <= TOL


@pytest.mark.parametrize("d", [64, 128])
def test_noncausal_tc_constant_values(d):
    q, k, _ = wl.make_qkv(1, 2, 700, d, "bf16", seed=9)
    u = torch.randn(1, 2, 1, d).to(torch.bfloat16)
    v = u.expand(1, 2, 700, d).contiguous()
    y = run_tc(q, k, v, seg=2)
    torch.testing.assert_close(y.float(), v.float(), rtol=2e-2, atol=2e-2)


def test_noncausal_tc_deterministic():
    """Partials are added in segment order, so repeated calls are identical."""
    q, k, v = (t.cuda() for t in wl.make_qkv(2, 4, 1500, 128, "bf16", seed=4))
    a = la.forward(q, k, v, causal=False, path=2, segment_chunks=2)
    for _ in range(3):
        b = la.forward(q, k, v, causal=False, path=2, segment_chunks=2)
        la.check_device_status()
        assert torch.equal(a, b)


def test_noncausal_tc_matches_cuda_core_path():
    q, k, v = (t.cuda() for t in wl.make_qkv(2, 2, 777, 64, "bf16", seed=6))
    y_tc = la.forward(q, k, v, causal=False, path=2)
    y_cc = la.forward(q, k, v, causal=False, path=1)
    la.check_device_status()
    assert wl.max_row_rel_err(y_tc.cpu(), y_cc.cpu()) <= TOL

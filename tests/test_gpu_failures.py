"""Failure paths on the GPU, driven through the library's testing hooks
without faulting the GPU: a bounded wait that runs out (a segment that
never publishes its state, with a short wait bound) must come back as
LA_ERR_TIMEOUT from la_check_device_status, and a workspace allocation that
fails must come back as LA_ERR_NO_MEMORY with nothing enqueued.  After
either, the next ordinary call must still match the oracle."""
import pytest

import oracle
import linear_attention_feature_gb300 as la
from linear_attention_feature_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
TIMEOUT, NO_MEMORY = 5, 4


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.build.build()
    return la.load_library()


def ordinary_call_matches_oracle(q, k, v):
    y = la.forward(q, k, v, causal=True, path=2, segment_chunks=2)
    la.check_device_status()
    ref = oracle.causal(q.cpu(), k.cpu(), v.cpu(), nthreads=8)
    assert wl.max_row_rel_err(y.cpu(), ref) <= wl.TOL["bf16"]


@pytest.mark.parametrize("hold", [1, 2])
def test_wait_that_runs_out_is_reported(lib, hold):
    # four segments per head: segments 1 and 2 publish the states of
    # segments 0 and 1 (their phase A), which the segments after them need;
    # those wait for a state that is never published, with a wait bound of
    # 2^20 cycles
    q, k, v = (t.cuda() for t in wl.make_qkv(1, 4, 8 * 128, 128, "bf16", seed=17))
    assert lib.la_debug_inject_timeout(1 << 20, hold) == 0
    la.forward(q, k, v, causal=True, path=2, segment_chunks=2)
    with pytest.raises(la.LinAttnError) as ei:
        la.check_device_status()
    assert ei.value.status == TIMEOUT
    # the status word is cleared and the context is usable
    ordinary_call_matches_oracle(q, k, v)


def test_hook_applies_to_one_launch_only(lib):
    q, k, v = (t.cuda() for t in wl.make_qkv(1, 2, 4 * 128, 128, "bf16", seed=18))
    assert lib.la_debug_inject_timeout(1 << 20, -1) == 0  # nothing held back
    ordinary_call_matches_oracle(q, k, v)                 # consumes the hook
    ordinary_call_matches_oracle(q, k, v)


def test_rejects_a_tiny_wait_bound(lib):
    assert lib.la_debug_inject_timeout(100, 0) == 1


@pytest.mark.parametrize("d, causal, dtype", [
    (128, True, "bf16"), (64, True, "bf16"), (64, False, "bf16"),
    (64, True, "f32"), (96, False, "f32")])  # fp32: the segmented CUDA-core path
def test_failed_workspace_allocation(lib, d, causal, dtype):
    q, k, v = (t.cuda() for t in wl.make_qkv(1, 2, 3 * 128, d, dtype, seed=19))
    n0 = la.kernel_launch_count()
    assert lib.la_debug_fail_next_allocs(1) == 0
    with pytest.raises(la.LinAttnError) as ei:
        la.forward(q, k, v, causal=causal)
    assert ei.value.status == NO_MEMORY
    assert "workspace allocation" in str(ei.value)
    assert la.kernel_launch_count() == n0  # nothing was enqueued
    la.check_device_status()
    y = la.forward(q, k, v, causal=causal)
    la.check_device_status()
    ref = (oracle.causal if causal else oracle.noncausal)(q.cpu(), k.cpu(), v.cpu())
    assert wl.max_row_rel_err(y.cpu(), ref) <= wl.TOL[dtype]

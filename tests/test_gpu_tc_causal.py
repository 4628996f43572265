"""GPU parity of the tcgen05 chunkwise causal kernel (bf16 in, fp32
accumulate) against the double-precision oracle.

Sizes span several 128-token chunks with ragged tails; `segment_chunks`
forces many segments per head so that the cross-CTA look-back over
published segment states is exercised (including chains longer than one
hop).  Tolerance: 2e-2 max row-relative error (bf16 inputs)."""
import numpy as np
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


def run_tc(q, k, v, decay=None, seg=0):
    y = la.forward(q.cuda(), k.cuda(), v.cuda(), causal=True, decay=decay,
                   path=2, segment_chunks=seg)
    la.check_device_status()
    return y.cpu()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 100, 128, 129, 300, 1000])
def test_causal_tc_ragged(d, N):
    q, k, v = wl.make_qkv(2, 3, N, d, "bf16", seed=N + d)
    y = run_tc(q, k, v)
    assert wl.max_row_rel_err(y, oracle.causal(q, k, v, nthreads=8)) <= TOL


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("seg", [1, 2, 3, 5, 7])
def test_causal_tc_many_segments(d, seg):
    q, k, v = wl.make_qkv(1, 4, 1500, d, "bf16", seed=seg)
    y = run_tc(q, k, v, seg=seg)
    assert wl.max_row_rel_err(y, oracle.causal(q, k, v, nthreads=8)) <= TOL


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("seg", [1, 4, 0, 5])
def test_causal_tc_decay(d, seg):
    H = 4
    dec = [0.0, 0.5, 0.96875, 1.0]
    q, k, v = wl.make_qkv(2, H, 700, d, "bf16", seed=40 + seg)
    y = run_tc(q, k, v, decay=dec, seg=seg)
    ref = oracle.causal(q, k, v, dec, nthreads=8)
    assert wl.max_row_rel_err(y, ref) <= TOL
    # g = 0 forgets everything: out_t = v_t (up to bf16 rounding)
    torch.testing.assert_close(y[:, 0].float(), v[:, 0].float(), rtol=1e-2,
                               atol=1e-2)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [300, 700])
@pytest.mark.parametrize("seg", [0, 1, 3])
def test_causal_tc_decay_folded(d, N, seg):
    """Decays >= 0.77 weight Q and K before P is formed and rescale P by
    g^-n per chunk (d = 128: when every head's decay is; d = 64: per head);
    decays at the threshold, just below it and at 1."""
    dec = [0.77, 0.7699, 0.96875, 1.0] if d == 64 else [0.77, 0.8, 0.96875, 1.0]
    q, k, v = wl.make_qkv(2, 4, N, d, "bf16", seed=60 + seg)
    y = run_tc(q, k, v, decay=dec, seg=seg)
    assert wl.max_row_rel_err(y, oracle.causal(q, k, v, dec, nthreads=8)) <= TOL


def test_causal_tc_decay_schedule_long_heads():
    """The decay schedule g_h = 1 - 2^(-5-h) over 8 heads, several segments."""
    dec = list(wl.decay_schedule(8))
    q, k, v = wl.make_qkv(1, 8, 2200, 128, "bf16", seed=77)
    y = run_tc(q, k, v, decay=dec, seg=2)
    assert wl.max_row_rel_err(y, oracle.causal(q, k, v, dec, nthreads=8)) <= TOL


def test_causal_tc_matches_cuda_core_path():
    q, k, v = (t.cuda() for t in wl.make_qkv(2, 2, 513, 64, "bf16", seed=5))
    y_tc = la.forward(q, k, v, causal=True, path=2, segment_chunks=2)
    y_cc = la.forward(q, k, v, causal=True, path=1)
    la.check_device_status()
    assert wl.max_row_rel_err(y_tc.cpu(), y_cc.cpu()) <= TOL


@pytest.mark.parametrize("d", [64, 128])
def test_causal_tc_constant_values(d):
    q, k, _ = wl.make_qkv(1, 2, 600, d, "bf16", seed=9)
    u = torch.randn(1, 2, 1, d).to(torch.bfloat16)
    v = u.expand(1, 2, 600, d).contiguous()
    y = run_tc(q, k, v, seg=2)
    torch.testing.assert_close(y.float(), v.float(), rtol=2e-2, atol=2e-2)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("decay", [None, [0.96875, 0.5, 0.999, 1.0],
                                   [0.96875, 0.8, 0.999, 1.0]])
def test_causal_tc_repeated_calls_are_bit_identical(d, decay):
    """Every segment's start state is the decayed sum of its predecessors'
    published local states, added in a fixed order, so repeated calls give
    the same bits whatever the timing (many segments per head here)."""
    q, k, v = (t.cuda() for t in wl.make_qkv(2, 4, 2900, d, "bf16", seed=3))
    a = la.forward(q, k, v, causal=True, decay=decay, path=2, segment_chunks=2)
    for _ in range(4):
        b = la.forward(q, k, v, causal=True, decay=decay, path=2, segment_chunks=2)
        la.check_device_status()
        assert torch.equal(a, b)


def test_gated_repeated_calls_are_bit_identical():
    q, k, v = (t.cuda() for t in wl.make_qkv(2, 4, 2900, 64, "bf16", seed=4))
    gen = torch.Generator().manual_seed(7)
    ga = (0.8 + 0.2 * torch.rand(2, 4, 2900, generator=gen)).cuda()
    a = la.forward_gated(q, k, v, ga)
    for _ in range(4):
        b = la.forward_gated(q, k, v, ga)
        la.check_device_status()
        assert torch.equal(a, b)


def test_auto_path_uses_tensor_cores_for_bf16():
    q, k, v = (t.cuda() for t in wl.make_qkv(1, 2, 256, 64, "bf16", seed=1))
    n0 = la.kernel_launch_count()
    la.forward(q, k, v, causal=True)
    la.check_device_status()
    assert la.kernel_launch_count() == n0 + 2  # workspace clear + forward

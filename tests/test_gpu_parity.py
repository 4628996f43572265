"""GPU parity: the CUDA library against the double-precision oracle,
element by element, on seeded inputs at sizes the oracle finishes in
seconds (several chunks, ragged tails), plus the degenerate cases.

Error metric: per output row, ||y_i - r_i||_inf / ||r_i||_inf, maximum over
all rows; the bar is 1e-4 for fp32 inputs and 2e-2 for bf16 inputs with fp32
accumulation."""
import numpy as np
import pytest

import oracle
import linear_attention_feature_gb300 as la
from linear_attention_feature_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.build.build()
    la.load_library()


def run_forward(q, k, v, causal, decay=None, **kw):
    y = la.forward(q.cuda(), k.cuda(), v.cuda(), causal=causal, decay=decay,
                   **kw)
    torch.cuda.synchronize()
    la.check_device_status()
    return y.cpu()


def ref_forward(q, k, v, causal, decay=None):
    if causal:
        return oracle.causal(q, k, v, decay, nthreads=8)
    return oracle.noncausal(q, k, v, nthreads=8)


# ---------------------------------------------------------------- worked example


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_worked_example(golden, causal, dtype):
    g = golden("kernel_la_worked_example.json")
    t = wl.torch_dtype(dtype)
    Q, K, V = (torch.tensor(g[n], dtype=t).reshape(1, 1, 4, 4)
               for n in ("Q", "K", "V"))
    y = run_forward(Q, K, V, causal)
    ref = ref_forward(Q, K, V, causal)
    assert wl.max_row_rel_err(y, ref) <= wl.TOL[dtype]
    if not causal:
        exact = np.array(g["num_1"]) / g["denom_1"]
        np.testing.assert_allclose(y[0, 0, 0].float().numpy(), exact,
                                   rtol=wl.TOL[dtype])


# ---------------------------------------------------------------- CUDA-core path


def test_fp32_causal_small_workload():
    w = wl.WORKLOADS["fp32_causal_small"]
    q, k, v = wl.make_workload_qkv(w, seed=0)
    y = run_forward(q, k, v, True)
    assert wl.max_row_rel_err(y, ref_forward(q, k, v, True)) <= 1e-4


@pytest.mark.parametrize("N", [1, 31, 32, 33, 100])
@pytest.mark.parametrize("d", [4, 64, 65, 130])
@pytest.mark.parametrize("causal", [True, False])
def test_cuda_core_ragged_fp32(N, d, causal):
    q, k, v = wl.make_qkv(2, 3, N, d, "f32", 1.0, seed=N * 1000 + d)
    y = run_forward(q, k, v, causal, path=1)
    assert wl.max_row_rel_err(y, ref_forward(q, k, v, causal)) <= 1e-4


@pytest.mark.parametrize("N, d", [(77, 64), (200, 128), (45, 96)])
@pytest.mark.parametrize("causal", [True, False])
def test_cuda_core_bf16(N, d, causal):
    q, k, v = wl.make_qkv(1, 2, N, d, "bf16", seed=7 + N)
    y = run_forward(q, k, v, causal, path=1)
    assert wl.max_row_rel_err(y, ref_forward(q, k, v, causal)) <= 2e-2


@pytest.mark.parametrize("N", [33, 129])
def test_cuda_core_decay_fp32(N):
    H = 4
    dec = [0.0, 0.5, 0.96875, 1.0]
    q, k, v = wl.make_qkv(2, H, N, 64, "f32", 1.0, seed=N)
    y = run_forward(q, k, v, True, dec, path=1)
    assert wl.max_row_rel_err(y, ref_forward(q, k, v, True, dec)) <= 1e-4
    # g = 0 forgets everything: out_t = v_t
    torch.testing.assert_close(y[:, 0], v[:, 0], rtol=1e-6, atol=1e-6)


def test_cuda_core_max_d():
    q, k, v = wl.make_qkv(1, 1, 40, 256, "f32", 0.2, seed=3)
    for causal in (True, False):
        y = run_forward(q, k, v, causal, path=1)
        assert wl.max_row_rel_err(y, ref_forward(q, k, v, causal)) <= 1e-4


@pytest.mark.parametrize("causal", [True, False])
def test_constant_values_give_constant_output(causal):
    q, k, _ = wl.make_qkv(1, 2, 70, 64, "f32", 2.0, seed=11)
    u = torch.randn(1, 2, 1, 64)
    v = u.expand(1, 2, 70, 64).contiguous()
    y = run_forward(q, k, v, causal)
    torch.testing.assert_close(y, v, rtol=2e-6, atol=2e-6)


# ---------------------------------------------------------------- decode


@pytest.mark.parametrize("d", [64, 128, 256, 5])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_steps_match_oracle(d, dtype):
    B, H, T = 3, 5, 12
    q, k, v = wl.make_decode_tokens(B, H, d, T, dtype, seed=d)
    S = torch.zeros(B, H, d, d, device="cuda")
    z = torch.zeros(B, H, d, device="cuda")
    So = np.zeros((B, H, d, d))
    zo = np.zeros((B, H, d))
    for t in range(T):
        y = la.decode_step(S, z, q[t].cuda(), k[t].cuda(), v[t].cuda())
        r = oracle.decode_step(So, zo, q[t], k[t], v[t])
        assert wl.max_row_rel_err(y.cpu(), r) <= wl.TOL[dtype]
    np.testing.assert_allclose(S.cpu().numpy(), So, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(z.cpu().numpy(), zo, rtol=1e-5, atol=1e-5)


def test_decode_equals_forward_causal():
    """N decode steps from a zero state reproduce the causal forward rows."""
    B, H, N, d = 2, 2, 40, 64
    q, k, v = wl.make_qkv(B, H, N, d, "f32", 1.0, seed=5)
    yf = run_forward(q, k, v, True)
    S = torch.zeros(B, H, d, d, device="cuda")
    z = torch.zeros(B, H, d, device="cuda")
    for t in range(N):
        y = la.decode_step(S, z, q[:, :, t].contiguous().cuda(),
                           k[:, :, t].contiguous().cuda(),
                           v[:, :, t].contiguous().cuda())
        assert wl.max_row_rel_err(y.cpu(), yf[:, :, t]) <= 1e-4


def test_decode_checkpoint_resume():
    """Saving and restoring (S, z) mid-way gives the same outputs as an
    unbroken run."""
    B, H, d, T = 2, 3, 128, 10
    q, k, v = wl.make_decode_tokens(B, H, d, T, "bf16", seed=9)
    S = torch.zeros(B, H, d, d, device="cuda")
    z = torch.zeros(B, H, d, device="cuda")
    ys = [la.decode_step(S, z, q[t].cuda(), k[t].cuda(), v[t].cuda()).cpu()
          for t in range(T)]
    S2 = torch.zeros_like(S)
    z2 = torch.zeros_like(z)
    for t in range(5):
        la.decode_step(S2, z2, q[t].cuda(), k[t].cuda(), v[t].cuda())
    saved = (S2.cpu().clone(), z2.cpu().clone())
    S3, z3 = saved[0].cuda(), saved[1].cuda()
    for t in range(5, T):
        y = la.decode_step(S3, z3, q[t].cuda(), k[t].cuda(), v[t].cuda()).cpu()
        torch.testing.assert_close(y, ys[t], rtol=0, atol=0)

"""Prefill -> decode hand-off: la_forward_causal_state returns the final state
of the causal recurrence, and la_decode_step_ex continues from it with an
optional per-head decay.  Checked against the double-precision oracle: the
final state (max abs error over a head / max |S| of that head), the decode
outputs (max row-relative error), and the whole hand-off against a single
causal pass over the concatenated sequence."""
import numpy as np
import pytest

import oracle
import linear_attention_feature_gb300 as la
from linear_attention_feature_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

STATE_TOL = {"f32": 1e-4, "bf16": 1e-2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.build.build()
    la.load_library()


def state_err(S, ref):
    S = np.asarray(S, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    ax = tuple(range(2, ref.ndim))
    scale = np.abs(ref).max(axis=ax, keepdims=True)
    return float((np.abs(S - ref) / np.where(scale > 0, scale, 1.0)).max())


def dec_list(dec, H):
    return None if dec is None else list(dec[:H])


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [100, 1500, 3000])
@pytest.mark.parametrize("dec", [None, [0.0, 0.5, 0.96875, 1.0]])
def test_final_state_tensor_cores(d, N, dec):
    q, k, v = (t.cuda() for t in wl.make_qkv(1, 4, N, d, "bf16", seed=40 + N))
    out, S, z = la.forward_causal_state(q, k, v, decay=dec)
    la.check_device_status()
    Sr, zr = oracle.causal_state(k.float().cpu(), v.float().cpu(), dec)
    assert state_err(S.cpu(), Sr) <= STATE_TOL["bf16"]
    assert state_err(z.cpu(), zr) <= STATE_TOL["bf16"]
    # the outputs are those of la_forward
    ref = oracle.causal(q.float().cpu(), k.float().cpu(), v.float().cpu(), dec)
    assert wl.max_row_rel_err(out.cpu(), ref) <= wl.TOL["bf16"]


@pytest.mark.parametrize("dtype, d", [("f32", 64), ("bf16", 96), ("f32", 33)])
@pytest.mark.parametrize("dec", [None, [0.9, 0.5]])
def test_final_state_cuda_cores(dtype, d, dec):
    q, k, v = (t.cuda() for t in wl.make_qkv(2, 2, 333, d, dtype, seed=50 + d))
    out, S, z = la.forward_causal_state(q, k, v, decay=dec)
    la.check_device_status()
    Sr, zr = oracle.causal_state(k.float().cpu(), v.float().cpu(), dec)
    tol = STATE_TOL["f32"] if dtype == "f32" else STATE_TOL["bf16"]
    assert state_err(S.cpu(), Sr) <= tol
    assert state_err(z.cpu(), zr) <= tol


@pytest.mark.parametrize("dtype, d", [("bf16", 64), ("bf16", 128), ("f32", 64)])
@pytest.mark.parametrize("dec", [None, [0.96875, 0.5, 0.999]])
def test_decode_with_decay_matches_oracle(dtype, d, dec):
    B, H = 3, 3
    q, k, v = wl.make_decode_tokens(B, H, d, 5, dtype, seed=60 + d)
    S0 = np.random.default_rng(61).standard_normal((B, H, d, d)) * 0.1
    z0 = np.abs(np.random.default_rng(62).standard_normal((B, H, d))) + 1.0
    S = torch.tensor(S0, dtype=torch.float32).cuda()
    z = torch.tensor(z0, dtype=torch.float32).cuda()
    So, zo = S.double().cpu().numpy().copy(), z.double().cpu().numpy().copy()
    g = None if dec is None else np.tile(np.asarray(dec), B)
    tol = wl.TOL["f32"] if dtype == "f32" else wl.TOL["bf16"]
    for t in range(5):
        y = la.decode_step(S, z, q[t].cuda(), k[t].cuda(), v[t].cuda(), decay=dec)
        r = oracle.decode_step(So, zo, q[t].float(), k[t].float(), v[t].float(), g)
        assert wl.max_row_rel_err(y.cpu(), r) <= tol
    la.check_device_status()
    np.testing.assert_allclose(S.cpu().numpy(), So, rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(z.cpu().numpy(), zo, rtol=1e-4, atol=1e-4)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dec", [None, [0.96875, 0.5, 1.0, 0.0]])
def test_prefill_then_decode_equals_one_causal_pass(d, dec):
    # prefill N tokens on the tensor cores, then T single-token steps: the
    # decode outputs are the last T rows of one causal pass over N + T
    B, H, N, T = 2, 4, 1000, 16
    q, k, v = wl.make_qkv(B, H, N + T, d, "bf16", seed=70 + d)
    qd, kd, vd = (t[:, :, :N].contiguous().cuda() for t in (q, k, v))
    _, S, z = la.forward_causal_state(qd, kd, vd, decay=dec)
    ys = []
    for t in range(N, N + T):
        ys.append(la.decode_step(S, z, q[:, :, t].contiguous().cuda(),
                                 k[:, :, t].contiguous().cuda(),
                                 v[:, :, t].contiguous().cuda(), decay=dec).cpu())
    la.check_device_status()
    ref = oracle.causal(q.float(), k.float(), v.float(), dec)
    y = torch.stack(ys, dim=2)
    assert wl.max_row_rel_err(y, ref[:, :, N:]) <= wl.TOL["bf16"]
    Sr, zr = oracle.causal_state(k.float(), v.float(), dec)
    assert state_err(S.cpu(), Sr) <= STATE_TOL["bf16"]
    assert state_err(z.cpu(), zr) <= STATE_TOL["bf16"]


def test_empty_sequence_gives_zero_state():
    q = torch.zeros(2, 3, 0, 64, dtype=torch.bfloat16, device="cuda")
    S = torch.full((2, 3, 64, 64), 7.0, device="cuda")
    z = torch.full((2, 3, 64), 7.0, device="cuda")
    la.forward_causal_state(q, q.clone(), q.clone(), S=S, z=z)
    torch.cuda.synchronize()
    assert not S.any() and not z.any()

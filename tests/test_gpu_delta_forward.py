"""The delta rule over whole sequences (la_forward_delta): the page's worked
write reproduced exactly as a one-token sequence, and seeded sequences
against the double-precision oracle (fp32 and bf16 inputs, with and without
the Gated DeltaNet forget gate, given start states, every head dimension the
kernel templates cover), plus the hand-off to the delta-rule decode step."""
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


def make_inputs(B, H, N, d, dtype, seed, gated):
    q, k, v = wl.make_qkv(B, H, N, d, dtype, seed=seed)
    # DeltaNet writes with unit keys; normalise in fp32, then round
    kf = k.float()
    k = (kf / kf.norm(dim=-1, keepdim=True).clamp_min(1e-6)).to(k.dtype)
    g = torch.Generator().manual_seed(seed + 1)
    beta = 0.1 + 0.9 * torch.rand(B, H, N, generator=g)
    alpha = (0.5 + 0.5 * torch.rand(B, H, N, generator=g)) if gated else None
    return q, k, v, beta, alpha


def oracle_run(q, k, v, beta, alpha, S0=None):
    return oracle.delta_forward(q.float(), k.float(), v.float(), beta.double().numpy(),
                                None if alpha is None else alpha.double().numpy(),
                                S0=None if S0 is None else S0.double().numpy(), nthreads=8)


def test_delta_forward_worked_example(golden):
    g = golden("deltanet_worked_example.json")
    d = 2
    S = torch.tensor(g["S_prev"], dtype=torch.float32).t().contiguous().view(1, 1, d, d).cuda()
    k = torch.tensor(g["k"], dtype=torch.float32).view(1, 1, 1, d).cuda()
    v = torch.tensor(g["v"], dtype=torch.float32).view(1, 1, 1, d).cuda()
    beta = torch.full((1, 1, 1), float(g["beta"]), device="cuda")
    o = la.forward_delta(k.clone(), k, v, beta, S=S)
    la.check_device_status()
    np.testing.assert_array_equal(S[0, 0].t().cpu().numpy(), np.asarray(g["S_next"], np.float32))
    np.testing.assert_array_equal(o[0, 0, 0].cpu().numpy(), np.asarray(g["S_next_k"], np.float32))


@pytest.mark.parametrize("B, H, N, d", [(1, 2, 100, 16), (2, 3, 300, 64), (1, 2, 257, 100),
                                        (1, 2, 130, 128), (1, 1, 70, 200), (3, 1, 33, 5)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("gated", [False, True])
def test_delta_forward_matches_oracle(B, H, N, d, dtype, gated):
    q, k, v, beta, alpha = make_inputs(B, H, N, d, dtype, 70 + d, gated)
    y = la.forward_delta(q.cuda(), k.cuda(), v.cuda(), beta.cuda(),
                         None if alpha is None else alpha.cuda())
    la.check_device_status()
    ref, _ = oracle_run(q, k, v, beta, alpha)
    assert wl.max_row_rel_err(y.cpu(), ref) <= wl.TOL[dtype]


@pytest.mark.parametrize("d", [64, 128])
def test_delta_forward_state_in_and_out(d):
    # a given start state, and the final state against the oracle's
    B, H, N = 2, 2, 200
    q, k, v, beta, alpha = make_inputs(B, H, N, d, "f32", 90 + d, True)
    S0 = 0.1 * torch.randn(B, H, d, d, generator=torch.Generator().manual_seed(5))
    S = S0.clone().cuda()
    y = la.forward_delta(q.cuda(), k.cuda(), v.cuda(), beta.cuda(), alpha.cuda(), S=S)
    la.check_device_status()
    ref, S_ref = oracle_run(q, k, v, beta, alpha, S0)
    assert wl.max_row_rel_err(y.cpu(), ref) <= wl.TOL["f32"]
    assert float(np.abs(S.cpu().double().numpy() - S_ref).max() / np.abs(S_ref).max()) <= 1e-4


def test_delta_forward_then_decode_steps():
    # the forward's final state continues with la_decode_step_delta; together
    # they equal one forward over all tokens
    B, H, N, T, d = 1, 4, 150, 10, 64
    q, k, v, beta, alpha = make_inputs(B, H, N + T, d, "f32", 95, True)
    qc, kc, vc, bc, ac = (t.cuda() for t in (q, k, v, beta, alpha))
    S = torch.zeros(B, H, d, d, device="cuda")
    la.forward_delta(qc[:, :, :N].contiguous(), kc[:, :, :N].contiguous(),
                     vc[:, :, :N].contiguous(), bc[:, :, :N].contiguous(),
                     ac[:, :, :N].contiguous(), S=S)
    outs = [la.decode_step_delta(S, qc[:, :, t].contiguous(), kc[:, :, t].contiguous(),
                                 vc[:, :, t].contiguous(), bc[:, :, t].contiguous(),
                                 ac[:, :, t].contiguous()) for t in range(N, N + T)]
    la.check_device_status()
    y_all = la.forward_delta(qc, kc, vc, bc, ac)
    la.check_device_status()
    dec = torch.stack(outs, dim=2).cpu()
    assert wl.max_row_rel_err(dec, y_all[:, :, N:].cpu().double().numpy()) <= 1e-4


def test_delta_forward_rejects_bad_arguments():
    lib = la.load_library()
    q = torch.zeros(1, 1, 4, 8, device="cuda")
    b = torch.zeros(1, 1, 4, device="cuda")
    V = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    assert lib.la_forward_delta(V(q), V(q), V(q), V(q), V(b), None, None, 1, 1, 4, 300, 0, None) == 1
    assert lib.la_forward_delta(V(q), V(q), V(q), V(q), None, None, None, 1, 1, 4, 8, 0, None) == 1
    assert lib.la_forward_delta(None, None, None, None, None, None, None, 0, 1, 4, 8, 0, None) == 0

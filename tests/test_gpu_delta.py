"""Delta-rule decode step (la_decode_step_delta): the page's worked example
("Story of Attention - Part 5", section 7) reproduced exactly, and seeded
multi-step sequences against the double-precision oracle, with and without
the Gated DeltaNet forget gate."""
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


@pytest.mark.parametrize("d", [2, 64, 128])
def test_delta_worked_example_printed(golden, d):
    # the 2-dimensional example, zero-padded to d (the padding stays zero)
    g = golden("deltanet_worked_example.json")
    S = torch.zeros(1, 1, d, d, device="cuda")
    S[0, 0, :2, :2] = torch.tensor(g["S_prev"], dtype=torch.float32).t()  # library layout
    k = torch.zeros(1, 1, d, device="cuda")
    v = torch.zeros(1, 1, d, device="cuda")
    k[0, 0, :2] = torch.tensor(g["k"], dtype=torch.float32)
    v[0, 0, :2] = torch.tensor(g["v"], dtype=torch.float32)
    beta = torch.full((1, 1), float(g["beta"]), device="cuda")
    o = la.decode_step_delta(S, k.clone(), k, v, beta)   # query with the same key
    torch.cuda.synchronize()
    np.testing.assert_array_equal(S[0, 0, :2, :2].t().cpu().numpy(),
                                  np.asarray(g["S_next"], dtype=np.float32))
    assert not S[0, 0, 2:].any() and not S[0, 0, :, 2:].any()
    np.testing.assert_array_equal(o[0, 0, :2].cpu().numpy(),
                                  np.asarray(g["S_next_k"], dtype=np.float32))


@pytest.mark.parametrize("dtype, d", [("f32", 64), ("f32", 128), ("bf16", 128),
                                      ("bf16", 64), ("f32", 37)])
@pytest.mark.parametrize("gated", [False, True])
def test_delta_steps_match_oracle(dtype, d, gated):
    B, H, T = 2, 3, 8
    q, k, v = wl.make_decode_tokens(B, H, d, T, dtype, seed=170 + d)
    # unit-norm keys, as DeltaNet models use
    k = (k.float() / k.float().norm(dim=-1, keepdim=True)).to(k.dtype)
    gen = torch.Generator().manual_seed(171 + d)
    beta = torch.rand(T, B, H, generator=gen)
    alpha = 0.8 + 0.2 * torch.rand(T, B, H, generator=gen)
    S = torch.zeros(B, H, d, d, device="cuda")
    So = np.zeros((B, H, d, d))
    tol = 1e-4 if dtype == "f32" else wl.TOL["bf16"]
    for t in range(T):
        a = alpha[t].cuda() if gated else None
        o = la.decode_step_delta(S, q[t].cuda(), k[t].cuda(), v[t].cuda(),
                                 beta[t].cuda(), a)
        r = oracle.delta_step(So, q[t].float(), k[t].float(), v[t].float(),
                              beta[t].double().numpy(),
                              alpha[t].double().numpy() if gated else None)
        assert wl.max_row_rel_err(o.cpu(), r) <= tol, t
    la.check_device_status()
    np.testing.assert_allclose(S.cpu().numpy(), So, rtol=1e-4, atol=1e-4)


def test_delta_stores_the_value_for_a_unit_key():
    # beta = 1 with a unit key: afterwards S^T k = v (the state returns v_t)
    d = 128
    rng = np.random.default_rng(180)
    S = torch.tensor(rng.standard_normal((1, 2, d, d)), dtype=torch.float32).cuda()
    k = torch.tensor(rng.standard_normal((1, 2, d)), dtype=torch.float32)
    k = (k / k.norm(dim=-1, keepdim=True)).cuda()
    v = torch.tensor(rng.standard_normal((1, 2, d)), dtype=torch.float32).cuda()
    o = la.decode_step_delta(S, k.clone(), k, v, torch.ones(1, 2, device="cuda"))
    torch.cuda.synchronize()
    np.testing.assert_allclose(o.cpu().numpy(), v.cpu().numpy(), rtol=1e-4, atol=1e-4)

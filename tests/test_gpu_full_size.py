"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (automatic kernel and segment choice): the GPU computes every
head; the double-precision oracle recomputes sampled heads in full and they
are compared element by element (max row-relative error; 1e-4 for fp32
inputs, 2e-2 for bf16).  Inputs are generated on the GPU from the seeded
generator and the sampled heads copied to the host for the oracle."""
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


def sampled_parity(w, causal, heads, decay=None, seed=0):
    q, k, v = wl.make_workload_qkv(w, seed=seed, device="cuda")
    y = la.forward(q, k, v, causal=causal, decay=decay)
    la.check_device_status()
    worst = 0.0
    for b, h in heads:
        qs, ks, vs = (t[b, h].float().cpu() for t in (q, k, v))
        if causal:
            g = None if decay is None else [decay[h]]
            ref = oracle.causal(qs[None], ks[None], vs[None], g)[0]
        else:
            ref = oracle.noncausal(qs[None], ks[None], vs[None])[0]
        err = wl.max_row_rel_err(y[b, h].cpu(), ref)
        worst = max(worst, err)
    return worst


def test_fp32_causal_small_full():
    w = wl.WORKLOADS["fp32_causal_small"]
    assert sampled_parity(w, True, [(0, 0), (0, 1)]) <= wl.TOL["f32"]


@pytest.mark.parametrize("causal", [True, False])
def test_b4h16_n4096_d64_full(causal):
    w = wl.WORKLOADS["bf16_b4h16_n4096_d64"]
    heads = [(0, 0), (1, 7), (3, 15)]
    assert sampled_parity(w, causal, heads) <= wl.TOL["bf16"]


def test_b2h16_n32768_d128_full():
    w = wl.WORKLOADS["bf16_b2h16_n32768_d128"]
    assert sampled_parity(w, True, [(0, 3), (1, 15)]) <= wl.TOL["bf16"]


def test_decay_b4h8_n16384_d128_full():
    w = wl.WORKLOADS["bf16_decay_b4h8_n16384_d128"]
    heads = [(0, 0), (3, 7)]  # strongest and weakest decay
    assert sampled_parity(w, True, heads, decay=list(w.decay)) <= wl.TOL["bf16"]


def test_decode_b256h32_d128_full():
    """All 8192 heads decode on the GPU: 1024 prefill steps from a zero state,
    then 1024 steps; sampled heads are replayed by the oracle and compared
    at every 64th step and on the final state."""
    w = wl.WORKLOADS["decode_b256h32_d128"]
    B, H, d = w.B, w.H, w.d
    T = w.extra["prefill"] + w.extra["steps"]
    q, k, v = wl.make_decode_tokens(B, H, d, T, "bf16", seed=100, device="cuda")
    S = torch.zeros(B, H, d, d, device="cuda")
    z = torch.zeros(B, H, d, device="cuda")
    heads = [(0, 0), (131, 17), (255, 31)]
    outs = {bh: [] for bh in heads}
    for t in range(T):
        y = la.decode_step(S, z, q[t], k[t], v[t])
        if t % 64 == 63:
            for bh in heads:
                outs[bh].append(y[bh].float().cpu())
    la.check_device_status()
    for (b, h) in heads:
        So, zo = np.zeros((d, d)), np.zeros(d)
        checked = 0
        for t in range(T):
            r = oracle.recurrent_step(So, zo, q[t, b, h].float().cpu(),
                                      k[t, b, h].float().cpu(),
                                      v[t, b, h].float().cpu())
            if t % 64 == 63:
                err = wl.max_row_rel_err(outs[(b, h)][checked], r)
                assert err <= wl.TOL["bf16"], (b, h, t, err)
                checked += 1
        np.testing.assert_allclose(S[b, h].cpu().numpy(), So, rtol=1e-3, atol=1e-3)
        np.testing.assert_allclose(z[b, h].cpu().numpy(), zo, rtol=1e-3, atol=1e-3)


def test_one_million_token_sequence():
    """A single 2^20-token head (the largest case here): the look-back chains
    over hundreds of segments; the last rows must still match the oracle."""
    N = 1 << 20
    q, k, v = wl.make_qkv(1, 1, N, 64, "bf16", seed=21, device="cuda")
    y = la.forward(q, k, v, causal=True)
    la.check_device_status()
    ref = oracle.causal(q.float().cpu(), k.float().cpu(), v.float().cpu())
    idx = np.r_[0:256, N // 2 - 128:N // 2 + 128, N - 256:N]
    assert wl.max_row_rel_err(y[0, 0].cpu()[idx], ref[0, 0][idx]) <= wl.TOL["bf16"]

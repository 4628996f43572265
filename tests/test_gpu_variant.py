"""Method variants (la_forward_variant, la_decode_step_variant): the feature
map (elu(x) + 1 or the identity) and the normaliser are selectable, which
with a decay gives retention.  The RetNet worked example printed on the pages
("Story of Attention - Part 5", section 4) is reproduced exactly on every
path; larger seeded cases are compared with the double-precision oracle."""
import numpy as np
import pytest

import oracle
import linear_attention_feature_gb300 as la
from linear_attention_feature_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

ID = oracle.FMAP_IDENTITY


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.build.build()
    la.load_library()


def padded(x, d, dtype):
    """[n, 4] example matrix zero-padded to [1, 1, n, d]."""
    a = torch.zeros(1, 1, len(x), d, dtype=dtype)
    a[0, 0, :, :4] = torch.tensor(x, dtype=torch.float64).to(dtype)
    return a.cuda()


@pytest.mark.parametrize("dtype, d", [(torch.float32, 4), (torch.float32, 64),
                                      (torch.bfloat16, 64), (torch.bfloat16, 128)])
def test_retnet_worked_example_printed(golden, dtype, d):
    g = golden("retnet_worked_example.json")
    q, k, v = (padded(g[n], d, dtype) for n in ("Q", "K", "V"))
    y = la.forward_variant(q, k, v, causal=True, decay=[g["gamma"]],
                           feature_map="identity", normalise=False)
    la.check_device_status()
    np.testing.assert_array_equal(y[0, 0, :, :4].double().cpu().numpy(),
                                  np.asarray(g["output_parallel"], dtype=np.float64))
    assert not y[0, 0, :, 4:].any()


def test_retnet_worked_example_recurrent_states(golden):
    g = golden("retnet_worked_example.json")
    Q, K, V = (torch.tensor(g[n], dtype=torch.float32).cuda() for n in ("Q", "K", "V"))
    S = torch.zeros(1, 1, 4, 4, device="cuda")
    z = torch.zeros(1, 1, 4, device="cuda")
    outs = []
    for t in range(4):
        outs.append(la.decode_step(S, z, Q[t].view(1, 1, 4), K[t].view(1, 1, 4),
                                   V[t].view(1, 1, 4), decay=[g["gamma"]],
                                   feature_map="identity", normalise=False).cpu())
        if t < 3:
            np.testing.assert_array_equal(S[0, 0].cpu().numpy(),
                                          np.asarray(g[f"S_{t + 1}"], dtype=np.float32))
    np.testing.assert_array_equal(torch.cat(outs).view(4, 4).numpy(),
                                  np.asarray(g["output_parallel"], dtype=np.float32))


def ref_variant(q, k, v, causal, dec, fmap, norm):
    q, k, v = (t.float().cpu() for t in (q, k, v))
    if causal:
        return oracle.causal(q, k, v, dec, fmap=fmap, normalise=norm, nthreads=8)
    return oracle.noncausal(q, k, v, fmap=fmap, normalise=norm, nthreads=8)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [300, 2000])
@pytest.mark.parametrize("dec", [None, [0.5, 0.9, 0.96875, 1.0], [0.8, 0.9, 0.96875, 1.0]])
def test_retention_tensor_cores(d, N, dec):
    q, k, v = (t.cuda() for t in wl.make_qkv(1, 4, N, d, "bf16", seed=80 + N))
    y = la.forward_variant(q, k, v, causal=True, decay=dec,
                           feature_map="identity", normalise=False)
    la.check_device_status()
    assert wl.max_row_rel_err(y.cpu(), ref_variant(q, k, v, True, dec, ID, False)) <= wl.TOL["bf16"]


@pytest.mark.parametrize("fmap, norm", [("identity", False), ("elu1", False)])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("dtype, d", [("bf16", 64), ("f32", 64), ("bf16", 96)])
def test_variants_match_oracle(fmap, norm, causal, dtype, d):
    q, k, v = (t.cuda() for t in wl.make_qkv(2, 2, 700, d, dtype, seed=90 + d))
    y = la.forward_variant(q, k, v, causal=causal, feature_map=fmap, normalise=norm)
    la.check_device_status()
    fm = ID if fmap == "identity" else oracle.FMAP_ELU1
    tol = wl.TOL["f32"] if dtype == "f32" else wl.TOL["bf16"]
    assert wl.max_row_rel_err(y.cpu(), ref_variant(q, k, v, causal, None, fm, norm)) <= tol


def test_default_variant_is_la_forward():
    q, k, v = (t.cuda() for t in wl.make_qkv(1, 2, 500, 64, "bf16", seed=99))
    a = la.forward(q, k, v, causal=False)
    b = la.forward_variant(q, k, v, causal=False)  # non-causal is deterministic
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("dtype, d", [("bf16", 128), ("f32", 64), ("f32", 20)])
def test_retention_decode_matches_oracle(dtype, d):
    B, H = 2, 3
    dec = [0.5, 0.96875, 1.0]
    q, k, v = wl.make_decode_tokens(B, H, d, 6, dtype, seed=100 + d)
    S = torch.zeros(B, H, d, d, device="cuda")
    z = torch.zeros(B, H, d, device="cuda")
    So, zo = np.zeros((B, H, d, d)), np.zeros((B, H, d))
    tol = wl.TOL["f32"] if dtype == "f32" else wl.TOL["bf16"]
    for t in range(6):
        y = la.decode_step(S, z, q[t].cuda(), k[t].cuda(), v[t].cuda(), decay=dec,
                           feature_map="identity", normalise=False).cpu()
        for b in range(B):
            for h in range(H):
                r = oracle.recurrent_step(So[b, h], zo[b, h], q[t, b, h].float(),
                                          k[t, b, h].float(), v[t, b, h].float(),
                                          dec[h], fmap=ID, normalise=False)
                assert wl.max_row_rel_err(y[b, h], r) <= tol
    la.check_device_status()

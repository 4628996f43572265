"""Seeded random configurations across the forward paths against the
double-precision oracle: head size, sequence length (ragged tails, one
token, several chunks), batch and heads, dtype, causal or not, per-head
decays (including 0, 1 and values on both sides of the folded-weights
threshold), the feature map and normaliser switches, kernel selection and
forced segment lengths.  Each case is small enough for the oracle to finish
at once; together they cover combinations the targeted tests do not."""
import random

import pytest

import oracle
import linear_attention_feature_gb300 as la
from linear_attention_feature_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _cases(n=36, seed=2024):
    rng = random.Random(seed)
    out = []
    for i in range(n):
        dtype = rng.choice(["bf16", "bf16", "f32"])
        d = rng.choice([64, 128, 64, 128, 32, 96, 8]) if dtype == "bf16" else rng.choice([16, 64, 100])
        N = rng.choice([1, 7, 128, 129, 300, 513, 640])
        B, H = rng.choice([(1, 1), (1, 3), (2, 2), (3, 1)])
        causal = rng.random() < 0.75
        decay = None
        if causal and rng.random() < 0.5:
            decay = [rng.choice([0.0, 0.5, 0.76, 0.78, 0.9, 0.99, 1.0]) for _ in range(H)]
        variant = ("elu1", True)
        if rng.random() < 0.25:
            variant = rng.choice([("identity", False), ("elu1", False), ("identity", True)])
        path = rng.choice([0, 0, 1, 2])
        seg = rng.choice([0, 0, 1, 2, 3])
        out.append((i, B, H, N, d, dtype, causal, decay, variant, path, seg))
    return out


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.build.build()
    la.load_library()


@pytest.mark.parametrize("case", _cases(), ids=lambda c: f"case{c[0]}")
def test_random_configuration_matches_oracle(case):
    i, B, H, N, d, dtype, causal, decay, (fmap, norm), path, seg = case
    if fmap == "identity" and norm and dtype == "bf16":
        # the identity map's normaliser sum_j q.k_j can come close to zero, so
        # rows divided by it amplify the bf16 rounding of q and k without bound
        pytest.skip("identity map with the normaliser in bf16: no stable bound")
    q, k, v = wl.make_qkv(B, H, N, d, dtype, seed=500 + i)
    tc_ok = dtype == "bf16" and d in (64, 128)
    if (fmap, norm) == ("elu1", True):
        if path == 2 and not tc_ok:
            path = 0
        y = la.forward(q.cuda(), k.cuda(), v.cuda(), causal=causal, decay=decay,
                       path=path, segment_chunks=seg)
    else:
        y = la.forward_variant(q.cuda(), k.cuda(), v.cuda(), causal=causal, decay=decay,
                               feature_map=fmap, normalise=norm)
    la.check_device_status()
    fm = oracle.FMAP_ELU1 if fmap == "elu1" else oracle.FMAP_IDENTITY
    if causal:
        ref = oracle.causal(q, k, v, decay, fmap=fm, normalise=norm, nthreads=4)
    else:
        ref = oracle.noncausal(q, k, v, fmap=fm, normalise=norm, nthreads=4)
    assert wl.max_row_rel_err(y.cpu(), ref) <= wl.TOL[dtype], case

"""The CUDA-core (fp32 FMA) path with its sequences cut into segments: local
segment states, their scan in segment order, then the outputs of every
segment from its start state.  Parity with the double-precision oracle for
each segmentation (one chunk of 32 tokens per segment up to one segment per
head, ragged tails), for the causal form with and without decay and for the
non-causal form; repeated calls are bit-identical."""
import pytest

import oracle
import linear_attention_feature_gb300 as la
from linear_attention_feature_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
TOL32, TOL16 = wl.TOL["f32"], wl.TOL["bf16"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.build.build()
    la.load_library()


def oracle_for(form, q, k, v, dec):
    if form == "noncausal":
        return oracle.noncausal(q, k, v, nthreads=8)
    return oracle.causal(q, k, v, dec if form == "decay" else None, nthreads=8)


@pytest.mark.parametrize("seg", [1, 2, 3, 7, 100])
@pytest.mark.parametrize("form", ["causal", "decay", "noncausal"])
@pytest.mark.parametrize("d", [64, 100])
def test_segmented_fp32_matches_oracle(seg, form, d):
    B, H, N = 2, 3, 333  # 11 chunks, the last of 13 tokens
    q, k, v = wl.make_qkv(B, H, N, d, "f32", seed=40 + d)
    dec = [0.97, 0.5, 1.0]
    y = la.forward(q.cuda(), k.cuda(), v.cuda(), causal=form != "noncausal",
                   decay=dec if form == "decay" else None, path=1,
                   segment_chunks=seg)
    la.check_device_status()
    assert wl.max_row_rel_err(y.cpu(), oracle_for(form, q, k, v, dec)) <= TOL32


@pytest.mark.parametrize("seg", [1, 4])
def test_segmented_bf16_odd_width(seg):
    q, k, v = wl.make_qkv(1, 2, 290, 96, "bf16", seed=44)
    y = la.forward(q.cuda(), k.cuda(), v.cuda(), causal=True, path=1,
                   segment_chunks=seg)
    la.check_device_status()
    assert wl.max_row_rel_err(y.cpu(), oracle.causal(q, k, v)) <= TOL16


def test_config_one_uses_segments_and_is_deterministic():
    # B1 H2 N512 d64 fp32: automatic segmentation gives one chunk per
    # segment (three launches: local states, scan, outputs)
    w = wl.WORKLOADS["fp32_causal_small"]
    q, k, v = (t.cuda() for t in wl.make_workload_qkv(w, seed=0))
    n0 = la.kernel_launch_count()
    y1 = la.forward(q, k, v, causal=True)
    assert la.kernel_launch_count() - n0 == 3
    y2 = la.forward(q, k, v, causal=True)
    la.check_device_status()
    assert torch.equal(y1, y2)
    ref = oracle.causal(q.cpu(), k.cpu(), v.cpu(), nthreads=8)
    assert wl.max_row_rel_err(y1.cpu(), ref) <= TOL32
    # one segment per head: a single launch, same result within rounding
    n0 = la.kernel_launch_count()
    y3 = la.forward(q, k, v, causal=True, segment_chunks=16)
    assert la.kernel_launch_count() - n0 == 1
    la.check_device_status()
    assert wl.max_row_rel_err(y3.cpu(), ref) <= TOL32


def test_segmented_gated_and_final_state():
    # small heads get one chunk per segment automatically
    B, H, N, d = 1, 2, 250, 48
    q, k, v = wl.make_qkv(B, H, N, d, "f32", seed=46)
    gen = torch.Generator().manual_seed(7)
    g = 0.8 + 0.2 * torch.rand(B, H, N, generator=gen)
    g[0, 1, 100] = 0.0  # a zero gate: the state restarts there
    y = la.forward_gated(q.cuda(), k.cuda(), v.cuda(), g.cuda())
    la.check_device_status()
    ref = oracle.causal_gated(q, k, v, g, nthreads=4)
    assert wl.max_row_rel_err(y.cpu(), ref) <= TOL32
    dec = [0.9, 1.0]
    y2, S, z = la.forward_causal_state(q.cuda(), k.cuda(), v.cuda(), decay=dec)
    la.check_device_status()
    S_ref, z_ref = oracle.causal_state(k, v, dec)
    assert wl.max_row_rel_err(y2.cpu(), oracle.causal(q, k, v, dec)) <= TOL32
    for got, ref in ((S, S_ref), (z, z_ref)):
        g64 = got.cpu().double().numpy()
        assert abs(g64 - ref).max() / abs(ref).max() <= TOL32

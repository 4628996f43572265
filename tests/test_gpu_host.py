"""la_forward_host: host buffers in and out, copies pipelined over groups of
heads.  Each case checks the host result against the double-precision oracle
(sampled heads) and against forward() on device copies of the same inputs,
with the grouping exercised both ways: whole batches per group, and ranges of
heads inside one batch (with a per-head decay sliced to match)."""
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


def pinned(*ts):
    return tuple(t.contiguous().pin_memory() for t in ts)


def check(q, k, v, causal, decay, heads, tol):
    out = la.forward_host(q, k, v, causal=causal, decay=decay)
    torch.cuda.current_stream().synchronize()
    la.check_device_status()
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    ref_dev = la.forward(qd, kd, vd, causal=causal, decay=decay).cpu()
    assert wl.max_row_rel_err(out, ref_dev) <= tol
    for b, h in heads:
        qs, ks, vs = (t[b, h].float() for t in (q, k, v))
        if causal:
            g = None if decay is None else [decay[h]]
            ref = oracle.causal(qs[None], ks[None], vs[None], g)[0]
        else:
            ref = oracle.noncausal(qs[None], ks[None], vs[None])[0]
        assert wl.max_row_rel_err(out[b, h], ref) <= tol, (b, h)
    return out


def test_host_batch_groups_causal_bf16():
    # 50 MB of input: four groups of two batches each
    q, k, v = pinned(*wl.make_qkv(8, 4, 4096, 64, "bf16", seed=31))
    check(q, k, v, True, None, [(0, 0), (7, 3)], wl.TOL["bf16"])


def test_host_head_range_groups_with_decay():
    # one batch, 12 heads in two groups of 6 (19 MB of input): the decay is
    # sliced per group
    q, k, v = pinned(*wl.make_qkv(1, 12, 4096, 64, "bf16", seed=32))
    dec = [0.5, 0.9, 0.99, 1.0, 0.0, 0.75, 0.96875, 0.8, 1.0, 0.6, 0.999, 0.3]
    check(q, k, v, True, dec, [(0, 1), (0, 6), (0, 11)], wl.TOL["bf16"])


def test_host_batch_and_uneven_head_groups_noncausal_d128():
    # B=3 < groups wanted (4, 75 MB of input): one group per batch; then
    # B=1 with H=7: heads split 2 + 2 + 2 + 1
    q, k, v = pinned(*wl.make_qkv(3, 8, 4096, 128, "bf16", seed=33))
    check(q, k, v, False, None, [(0, 0), (2, 7)], wl.TOL["bf16"])
    q, k, v = pinned(*wl.make_qkv(1, 7, 8192, 128, "bf16", seed=38))
    check(q, k, v, False, None, [(0, 0), (0, 6)], wl.TOL["bf16"])


def test_host_fp32_small_single_group_ragged():
    q, k, v = pinned(*wl.make_qkv(1, 3, 333, 64, "f32", seed=34))
    check(q, k, v, True, None, [(0, 0), (0, 2)], wl.TOL["f32"])


def test_host_pageable_buffers():
    q, k, v = wl.make_qkv(2, 4, 1024, 64, "bf16", seed=35)
    out = torch.empty_like(q)  # pageable: the CUDA driver stages the copies
    la.forward_host(q.contiguous(), k.contiguous(), v.contiguous(), causal=True, out=out)
    torch.cuda.current_stream().synchronize()
    ref = la.forward(q.cuda(), k.cuda(), v.cuda(), causal=True).cpu()
    assert wl.max_row_rel_err(out, ref) <= wl.TOL["bf16"]


def test_host_back_to_back_calls_share_a_workspace():
    # the second call's copies may only start once the first call is done
    # with the workspace; both results must be intact
    shape = (4, 4, 4096, 64)
    ws = torch.empty(la.host_workspace_bytes(shape, torch.bfloat16),
                     dtype=torch.uint8, device="cuda")
    a = pinned(*wl.make_qkv(*shape, "bf16", seed=36))
    b = pinned(*wl.make_qkv(*shape, "bf16", seed=37))
    oa = la.forward_host(*a, causal=True, workspace=ws)
    ob = la.forward_host(*b, causal=True, workspace=ws)
    torch.cuda.current_stream().synchronize()
    for (q, k, v), o in ((a, oa), (b, ob)):
        ref = la.forward(q.cuda(), k.cuda(), v.cuda(), causal=True).cpu()
        assert wl.max_row_rel_err(o, ref) <= wl.TOL["bf16"]

"""Data-dependent scalar gate per token and head (la_forward_gated,
la_decode_step_gated): S_t = alpha_t S_{t-1} + phi(k_t) v_t^T with the
normaliser gated alike, compared with the double-precision oracle on seeded
inputs and gates (including exact zeros and ones)."""
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


def make_gates(B, H, N, seed, lo=0.8):
    g = torch.Generator().manual_seed(seed)
    a = lo + (1.0 - lo) * torch.rand(B, H, N, generator=g)
    a[:, :, ::97] = 1.0          # exact ones
    a[0, 0, min(40, N // 2)] = 0.0  # a reset
    return a


@pytest.mark.parametrize("dtype, d", [("f32", 64), ("bf16", 64), ("bf16", 128), ("f32", 37)])
@pytest.mark.parametrize("N", [31, 333, 1000])
def test_gated_forward_matches_oracle(dtype, d, N):
    q, k, v = wl.make_qkv(2, 2, N, d, dtype, seed=110 + N)
    a = make_gates(2, 2, N, 111 + N)
    y = la.forward_gated(q.cuda(), k.cuda(), v.cuda(), a.cuda())
    la.check_device_status()
    ref = oracle.causal_gated(q.float(), k.float(), v.float(), a.double().numpy(), nthreads=8)
    tol = wl.TOL["f32"] if dtype == "f32" else wl.TOL["bf16"]
    assert wl.max_row_rel_err(y.cpu(), ref) <= tol


def test_gated_forward_constant_gates_equal_decay():
    q, k, v = (t.cuda() for t in wl.make_qkv(1, 3, 500, 64, "f32", seed=120))
    dec = [0.9, 0.5, 1.0]
    a = torch.tensor(dec).view(1, 3, 1).expand(1, 3, 500).contiguous().cuda()
    y = la.forward_gated(q, k, v, a)
    r = la.forward(q, k, v, causal=True, decay=dec)
    torch.cuda.synchronize()
    assert wl.max_row_rel_err(y.cpu(), r.cpu()) <= 1e-5


def test_gated_retention_variant():
    q, k, v = wl.make_qkv(1, 2, 400, 64, "f32", seed=121)
    a = make_gates(1, 2, 400, 122)
    y = la.forward_gated(q.cuda(), k.cuda(), v.cuda(), a.cuda(),
                         feature_map="identity", normalise=False)
    ref = oracle.causal_gated(q, k, v, a.double().numpy(), fmap=oracle.FMAP_IDENTITY,
                              normalise=False)
    assert wl.max_row_rel_err(y.cpu(), ref) <= wl.TOL["f32"]


@pytest.mark.parametrize("dtype, d", [("bf16", 128), ("f32", 64)])
def test_gated_decode_continues_the_gated_forward(dtype, d):
    # decode steps with per-token gates equal the gated forward's last rows
    B, H, N = 2, 3, 24
    q, k, v = wl.make_qkv(B, H, N, d, dtype, seed=130 + d)
    a = make_gates(B, H, N, 131 + d, lo=0.6)
    S = torch.zeros(B, H, d, d, device="cuda")
    z = torch.zeros(B, H, d, device="cuda")
    ys = []
    for t in range(N):
        ys.append(la.decode_step_gated(S, z, q[:, :, t].contiguous().cuda(),
                                       k[:, :, t].contiguous().cuda(),
                                       v[:, :, t].contiguous().cuda(),
                                       a[:, :, t].contiguous().cuda()).cpu())
    la.check_device_status()
    ref = oracle.causal_gated(q.float(), k.float(), v.float(), a.double().numpy())
    tol = wl.TOL["f32"] if dtype == "f32" else wl.TOL["bf16"]
    assert wl.max_row_rel_err(torch.stack(ys, dim=2), ref) <= tol


def test_gated_bf16_runs_on_the_tensor_cores():
    q, k, v = (t.cuda() for t in wl.make_qkv(1, 2, 256, 64, "bf16", seed=140))
    a = make_gates(1, 2, 256, 141).cuda()
    n0 = la.kernel_launch_count()
    la.forward_gated(q, k, v, a)
    la.check_device_status()
    # the gate slots of every chunk (with the workspace clear), the tcgen05 kernel
    assert la.kernel_launch_count() == n0 + 2


@pytest.mark.parametrize("d", [64, 128])
def test_gated_tensor_cores_across_segments(d):
    # 12 heads x 40 chunks: several segments per head, so each segment's
    # gate product travels through the look-back; zero gates sit inside
    # middle segments and on a chunk boundary
    B, H, N = 2, 6, 5000
    q, k, v = wl.make_qkv(B, H, N, d, "bf16", seed=150 + d)
    a = make_gates(B, H, N, 151 + d, lo=0.97)
    a[1, 2, 2500] = 0.0
    a[0, 5, 1280] = 0.0
    y = la.forward_gated(q.cuda(), k.cuda(), v.cuda(), a.cuda())
    la.check_device_status()
    heads = [(0, 0), (0, 5), (1, 2), (1, 5)]
    for b, h in heads:
        ref = oracle.causal_gated(q[b, h][None].float(), k[b, h][None].float(),
                                  v[b, h][None].float(), a[b, h][None].double().numpy())[0]
        assert wl.max_row_rel_err(y[b, h].cpu(), ref) <= wl.TOL["bf16"], (b, h)


@pytest.mark.parametrize("d", [64, 128])
def test_gated_constant_gates_equal_decay_on_tensor_cores(d):
    q, k, v = (t.cuda() for t in wl.make_qkv(1, 4, 2000, d, "bf16", seed=160 + d))
    dec = [0.9, 0.5, 0.99, 1.0]
    a = torch.tensor(dec).view(1, 4, 1).expand(1, 4, 2000).contiguous().cuda()
    y = la.forward_gated(q, k, v, a)
    r = la.forward(q, k, v, causal=True, decay=dec)
    torch.cuda.synchronize()
    assert wl.max_row_rel_err(y.cpu(), r.cpu()) <= wl.TOL["bf16"]


@pytest.mark.parametrize("d", [64, 128])
def test_gated_retention_on_tensor_cores(d):
    q, k, v = wl.make_qkv(1, 3, 1500, d, "bf16", seed=190 + d)
    a = make_gates(1, 3, 1500, 191 + d, lo=0.9)
    y = la.forward_gated(q.cuda(), k.cuda(), v.cuda(), a.cuda(),
                         feature_map="identity", normalise=False)
    la.check_device_status()
    ref = oracle.causal_gated(q.float(), k.float(), v.float(), a.double().numpy(),
                              fmap=oracle.FMAP_IDENTITY, normalise=False, nthreads=3)
    assert wl.max_row_rel_err(y.cpu(), ref) <= wl.TOL["bf16"]


def test_gated_long_head_many_segments():
    # one head of 2^16 tokens: dozens of segments whose gate products chain
    # through the look-back; gates close to 1 keep old state alive, with a
    # reset in the middle
    N, d = 1 << 16, 64
    q, k, v = wl.make_qkv(1, 1, N, d, "bf16", seed=200)
    a = make_gates(1, 1, N, 201, lo=0.999)
    a[0, 0, N // 2 + 77] = 0.0
    y = la.forward_gated(q.cuda(), k.cuda(), v.cuda(), a.cuda())
    la.check_device_status()
    ref = oracle.causal_gated(q.float(), k.float(), v.float(), a.double().numpy())
    idx = np.r_[0:128, N // 2:N // 2 + 256, N - 256:N]
    assert wl.max_row_rel_err(y[0, 0].cpu()[idx], ref[0, 0][idx]) <= wl.TOL["bf16"]


@pytest.mark.parametrize("d", [64, 128])
def test_gated_tiny_gates_exceed_the_factored_range(d):
    # heads 0, 2: gates 2^-U(0, 8), whose 32-token spans of log2 overshoot
    # what a product of two normal floats covers, so the diagonal score
    # blocks form each weight directly; heads 1, 3: gates in [0.95, 1), the
    # factored form; a zero gate in one block of head 1
    N = 1000
    q, k, v = wl.make_qkv(1, 4, N, d, "bf16", seed=210 + d)
    g = torch.Generator().manual_seed(211 + d)
    a = 0.95 + 0.05 * torch.rand(1, 4, N, generator=g)
    a[:, 0::2] = torch.exp2(-8.0 * torch.rand(1, 2, N, generator=g))
    a[0, 1, 300] = 0.0
    y = la.forward_gated(q.cuda(), k.cuda(), v.cuda(), a.cuda())
    la.check_device_status()
    ref = oracle.causal_gated(q.float(), k.float(), v.float(), a.double().numpy(), nthreads=4)
    assert wl.max_row_rel_err(y.cpu(), ref) <= wl.TOL["bf16"]


@pytest.mark.parametrize("d", [64, 128])
def test_gated_chunks_on_both_sides_of_the_fold_threshold(d):
    # a chunk whose gate product is at least 2^-48 (and has no zero gate)
    # takes the weights into Q and K at once; heads 0 and 1 sit just above
    # and just below that product per 128-token chunk, head 2 mixes both
    # from chunk to chunk, head 3 has gates in [0.7, 1)
    N = 900
    q, k, v = wl.make_qkv(1, 4, N, d, "bf16", seed=220 + d)
    g = torch.Generator().manual_seed(221 + d)
    a = torch.empty(1, 4, N)
    a[0, 0] = 2.0 ** (-47.5 / 128)
    a[0, 1] = 2.0 ** (-48.5 / 128)
    a[0, 2] = torch.where((torch.arange(N) // 128) % 2 == 0,
                          torch.tensor(2.0 ** (-40.0 / 128)), torch.tensor(2.0 ** (-60.0 / 128)))
    a[0, 3] = 0.7 + 0.3 * torch.rand(N, generator=g)
    y = la.forward_gated(q.cuda(), k.cuda(), v.cuda(), a.cuda())
    la.check_device_status()
    ref = oracle.causal_gated(q.float(), k.float(), v.float(), a.double().numpy(), nthreads=4)
    assert wl.max_row_rel_err(y.cpu(), ref) <= wl.TOL["bf16"]

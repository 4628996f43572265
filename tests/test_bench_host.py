"""Host arithmetic of bench.py's roofline figures, checked against the
per-unit counts of the method (no GPU).

Compulsory bytes of a forward: q, k, v read once and out written once, 4*d
elements per token and head.  Decode step: the fp32 state S (d x d) and z (d)
read and written, q, k, v read and out written.  Chunked causal FLOPs with
full C x C blocks: per token and head, phi(Q)phi(K)^T and P~V give 2*C*d
MACs, the inter-chunk read phi(Q)S and the state update phi(K)^T V give
2*d^2 MACs.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("shape,elem,expect", [
    # causal and non-causal forward, B=4, H=16, N=4096, d=64, bf16: 134 MB
    ((4, 16, 4096, 64), 2, 134_217_728),
    # long-context causal, B=2, H=16, N=32768, d=128, bf16: 1.07 GB
    ((2, 16, 32768, 128), 2, 1_073_741_824),
    # causal with per-head decay, B=4, H=8, N=16384, d=128, bf16: 537 MB
    ((4, 8, 16384, 128), 2, 536_870_912),
    # fp32 causal, B=1, H=2, N=512, d=64: 1 MiB
    ((1, 2, 512, 64), 4, 1_048_576),
])
def test_forward_bytes_are_the_compulsory_traffic(shape, elem, expect):
    B, H, N, d = shape
    assert bench.forward_bytes(B, H, N, d, elem) == expect
    # one read of q, k and v and one write of out, token by token
    assert expect == sum(elem * d for _ in range(4)) * B * H * N


def test_decode_bytes_per_step():
    # 256 sequences x 32 heads, d = 128: 133,120 bytes per head and step
    per_head = 2 * (128 * 128 + 128) * 4 + 3 * 128 * 2 + 128 * 2
    assert per_head == 133_120
    assert bench.decode_bytes(256 * 32, 128, 2) == 8192 * 133_120
    assert bench.decode_bytes(256 * 32, 128, 2) == 1_090_519_040


@pytest.mark.parametrize("d,C,per_token", [
    (64, 64, 32_768),     # 64 FLOP per byte at bf16 (512 B per token and head)
    (128, 128, 131_072),  # 128 FLOP per byte (1024 B per token and head)
    (64, 128, 49_152),    # the d = 64 kernel runs C = 128 chunks
])
def test_chunk_flops_per_token(d, C, per_token):
    macs = 2 * d * d + 2 * C * d
    assert 2 * macs == per_token
    assert bench.chunk_flops(1, 1, 1, d, C) == per_token
    assert bench.chunk_flops(4, 16, 4096, d, C) == per_token * 4 * 16 * 4096


def test_roofline_fraction_and_units():
    # 1 GB in 1 ms is 1000 GB/s: half of a 2000 GB/s peak
    r = bench.roofline_hbm(1_000_000_000, 1.0, 2000.0, traffic=123)
    assert r == {"bound": "hbm", "achieved": 1000.0, "peak": 2000.0,
                 "unit": "GB/s", "frac": 0.5, "traffic": 123}
    # 2e12 FLOP in 2 ms is 1000 TFLOP/s
    t = bench.tensor_fraction(2e12, 2.0, 2000.0)
    assert t == {"achieved_tflops": 1000.0, "peak_tflops": 2000.0, "frac": 0.5}


def test_peaks_come_from_the_measured_file_or_the_stated_fallback():
    p = bench.load_peaks()
    assert p["source"] in ("measured", "fallback")
    assert p["hbm_gbs"] > 1000 and p["bf16_tflops"] > 100
    if p["source"] == "fallback":
        assert (p["hbm_gbs"], p["bf16_tflops"]) == (6800.0, 1900.0)


def test_bench_parity_reads_every_head_of_a_forward_leg():
    # the CPU-baseline leg's comparison: an exact output scores ~0, and a
    # planted error in the LAST head (the oracle side is exact) is found
    torch = pytest.importorskip("torch")
    import oracle
    from linear_attention_feature_gb300 import workloads as wl
    q, k, v = wl.make_qkv(2, 3, 40, 8, "f32", 1.0, seed=1)
    y = torch.from_numpy(oracle.causal(q, k, v)).float()
    leg = {"form": "causal", "qkv": (q, k, v), "y": y.clone(), "decay": None}
    e, _ = bench.leg_error(oracle, wl, leg, 2)
    assert e < 1e-6
    y2 = y.clone()
    y2[1, 2, 17, 3] += 1.0
    leg["y"] = y2
    e2, _ = bench.leg_error(oracle, wl, leg, 2)
    assert e2 > 0.1


def test_bench_parity_replays_decode_legs():
    torch = pytest.importorskip("torch")
    import numpy as np
    import oracle
    from linear_attention_feature_gb300 import workloads as wl
    T, nh, d = 5, 3, 8
    q, k, v = wl.make_decode_tokens(1, nh, d, T, "f32", 1.0, seed=2)
    q, k, v = q[:, 0], k[:, 0], v[:, 0]      # [T, heads, d]
    S, z = np.zeros((nh, d, d)), np.zeros((nh, d))
    for t in range(T):
        y = oracle.decode_step(S, z, q[t], k[t], v[t])
    leg = {"form": "decode", "q": q, "k": k, "v": v,
           "y": torch.from_numpy(y).float(), "S": torch.from_numpy(S).float(),
           "z": torch.from_numpy(z).float(), "decay": None, "heads": "all"}
    e, info = bench.leg_error(oracle, wl, leg, 2)
    assert e < 1e-6 and info["state_rel_err"] < 1e-6
    leg["S"] = leg["S"] * 1.01
    _, info = bench.leg_error(oracle, wl, leg, 2)
    assert info["state_rel_err"] > 5e-3

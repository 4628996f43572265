#!/usr/bin/env python
"""Benchmark of the linear-attention hot path on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one causal la_forward over one batch of the long-context workload
(bf16 q, k, v [B=2, H=16, N=32768, d=128], N(0,1)/sqrt(d), seed = rank), the
largest single-GPU forward configuration.  The other paths of the hot path
(causal and non-causal forms at B=4, H=16, N=4096, d=64; causal with per-head
decay; fp32 causal; recurrent decode) are timed in the same run and reported
under "paths".  Rank 0 prints one JSON line.

Timing: each step is captured once in a CUDA graph (so that host-side
launch work does not sit between the events); W untimed warm-up replays, then
K replays, each bracketed by CUDA events on the stream the library launches
on, with L2 flushed between steps (a 256 MiB buffer written, then another
256 MiB read, so that the flush leaves no dirty lines whose write-back would
fall inside the next timed step); barrier + synchronize on
both sides of the timed region; the max over ranks is taken.  `value` = tokens (B*N per step, summed over ranks) per
second.  `e2e` repeats the main step through the C ABI with pinned host
buffers, the host->device copies of q, k, v and the device->host copy of the
output inside the timed region.

The CPU-baseline leg times the CPU oracle (the slow double-precision
reference that the parity tests use) on a bounded sample of the main
workload, and compares the oracle with the output of every timed leg (every
head of the forward legs; a stated sample of heads, every step replayed, for
the decode legs): each leg's `max_rel_err` is the largest per-row
||y - r||_inf / ||r||_inf.

--impl reference times the CPU oracle on a bounded sample of the same
workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("causal linear-attn tokens/s and % tensor roofline; "
          "decode step % HBM peak")
MAIN = "bf16_b2h16_n32768_d128"
MID = "bf16_b4h16_n4096_d64"
FLUSH_BYTES = 256 << 20


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": float(j["hbm_gbs"]),
                "bf16_tflops": float(j["bf16_tflops"]),
                "bf16_tflops_sustained": float(j.get("bf16_tflops_sustained",
                                                     j["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
               "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "-i",
                 str(self.idx), "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0, "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        load = [r for r in self.rows if (num(r[3]) or 0) >= 50]
        use = load or self.rows
        sm = [num(r[0]) for r in use if num(r[0]) is not None]
        smax = [num(r[1]) for r in self.rows if num(r[1]) is not None]
        reasons = sorted({name for r in use
                          for name, val in zip(self.REASONS, r[4:8])
                          if val.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(self.rows),
                "samples_under_load": len(load)}


# ------------------------------------------------------------------ helpers


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's value (NCCL reduces a device tensor, gloo a host
    one)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def capture(fn):
    """Capture one call of `fn` in a CUDA graph; returns (replay, launches)
    where `launches` is the number of library kernels one call enqueues."""
    import torch
    import linear_attention_feature_gb300 as la
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        fn()
        torch.cuda.synchronize()
        n0 = la.kernel_launch_count()
        with torch.cuda.graph(g, stream=s):
            fn()
        launches = la.kernel_launch_count() - n0
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g.replay, launches


def timed_steps(fn, K, W, world, flush=None, name="timed"):
    """Per-step CUDA-event durations (ms) of K steps after W warm-ups, the
    warm-ups and the timed steps inside one NVTX range `la/<name>` (so that
    a profiler can select a leg's launches by range)."""
    import torch
    with torch.cuda.nvtx.range("la/" + name):
        return _timed_steps(fn, K, W, world, flush)


def _timed_steps(fn, K, W, world, flush):
    import torch
    for _ in range(W):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for s, e in ev:
        if flush is not None:
            flush()
        s.record(stream)
        fn()
        e.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in ev]


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from
# one ncu capture of a kernel, keyed by kernel and workload, valid only while
# the kernel's sources hash to the recorded digest (else reported as null).
KNOWN_TRAFFIC = {
    # ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum --clock-control none
    #     -k regex:<kernel> -s 3 -c 1 python bench.py --kernel-case B H N D FORM
    # (FORM causal, decay, noncausal, gated, retention or state;
    # dram__bytes_read.sum +
    # dram__bytes_write.sum of the captured launch; "sources":
    # kernel_sources_digest(kernel) at capture time)
    ("causal_wide_kernel<0>", "bf16_b2h16_n32768_d128"):
        {"sources": "a3c2a2e658e48689", "bytes": 1159936000 + 217027584},
    ("causal_wide_kernel<2>", "bf16_decay_b4h8_n16384_d128"):
        {"sources": "a3c2a2e658e48689", "bytes": 552642304 + 82396160},
    ("causal_kernel<64,0>", "bf16_b4h16_n4096_d64"):
        {"sources": "ddb510b143bbb274", "bytes": 100765696 + 4827392},
    ("causal_kernel<64,2>", "bf16_b4h16_n4096_d64"):
        {"sources": "ddb510b143bbb274", "bytes": 105593600 + 5026816},
    ("causal_kernel<64,0>+state", "bf16_b4h16_n4096_d64"):
        {"sources": "ddb510b143bbb274", "bytes": 100765952 + 4875008},
    ("causal_wide_kernel<1>", "bf16_decay_b4h8_n16384_d128"):
        {"sources": "a3c2a2e658e48689", "bytes": 559840512 + 82061824},
    ("noncausal_kernel<64>", "bf16_b4h16_n4096_d64"):
        {"sources": "c99e10d20fed1e5d", "bytes": 100719104 + 3817984},
}


# The source files that make up each profiled kernel (its translation unit
# and the device headers it includes); a recorded DRAM traffic stays valid
# while their digest is unchanged.
KERNEL_SOURCES = {
    "causal_kernel": ("la_causal_tc.cu", "la_tc_common.cuh", "la_tc_ptx.cuh", "la_tc_host.h"),
    "causal_wide_kernel": ("la_causal_wide.cu", "la_tc_common.cuh", "la_tc_ptx.cuh",
                           "la_tc_host.h"),
    "noncausal_kernel": ("la_noncausal_tc.cu", "la_tc_common.cuh", "la_tc_ptx.cuh", "la_tc_host.h"),
}


def kernel_sources_digest(kernel="causal_kernel"):
    import hashlib
    csrc = os.path.join(ROOT, "linear_attention_feature_gb300", "csrc")
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel.split("<")[0]]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def known_traffic(kernel, w):
    rec = KNOWN_TRAFFIC.get((kernel, w.name))
    if rec is None or rec["sources"] != kernel_sources_digest(kernel):
        return None
    return rec["bytes"]


def forward_bytes(B, H, N, d, elem):
    """Compulsory HBM bytes of one forward: q, k, v read once, out written
    once."""
    return 4 * B * H * N * d * elem


def roofline_hbm(bytes_per_launch, ms, peak_gbs, traffic=None):
    achieved = bytes_per_launch / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1),
            "peak": peak_gbs, "unit": "GB/s",
            "frac": round(achieved / peak_gbs, 4), "traffic": traffic}


def tensor_fraction(flops_per_launch, ms, peak_tflops):
    t = flops_per_launch / (ms * 1e-3) / 1e12
    return {"achieved_tflops": round(t, 2), "peak_tflops": peak_tflops,
            "frac": round(t / peak_tflops, 4)}


def chunk_flops(B, H, N, d, C):
    """FLOPs of the chunked causal method with full C x C blocks: per token
    2*(2 d^2 + 2 C d)."""
    return 2 * (2 * d * d + 2 * C * d) * B * H * N


# ------------------------------------------------------------------ our arm


MAIN_KERNEL = "causal_wide_kernel<0>"
MID_KERNEL = "causal_kernel<64,0>"


def host_copy(*ts):
    return tuple(t.detach().cpu() for t in ts)


def run_ours(args):
    import torch
    import linear_attention_feature_gb300 as la
    from linear_attention_feature_gb300 import workloads as wl

    rank, world, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    la.build.build()
    la.load_library()
    peaks = load_peaks()
    K, W = args.steps, args.warmup
    dev = torch.device("cuda", torch.cuda.current_device())
    flush_buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_rd = torch.zeros(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_acc = torch.empty((), dtype=torch.float32, device=dev)

    def flush():
        # Written, the buffer evicts every line the step used; the read of a
        # second buffer then writes the first one's dirty lines back before
        # the next step starts (else about 100 MB of write-back lands in it).
        flush_buf.zero_()
        torch.sum(flush_rd, dim=0, out=flush_acc)

    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else local
    sampler = ClockSampler(gpu_index).start()
    # host copies of each leg's inputs and output, compared with the oracle
    # by the CPU-baseline leg (rank 0, one GPU)
    keep = {} if (rank == 0 and world == 1 and not args.no_cpu) else None

    # ---------------- main: causal forward on the long-context workload
    w = wl.WORKLOADS[MAIN]
    q, k, v = (t.to(dev) for t in wl.make_workload_qkv(w, seed=rank))
    out = torch.empty_like(q)
    main_fn = lambda: la.forward(q, k, v, causal=True, out=out)  # noqa: E731
    replay, per_call = capture(main_fn)
    steps_ms = timed_steps(replay, K, W, world, flush, name=MAIN)
    launches = per_call * K  # library kernels inside the timed region
    la.check_device_status()
    ms = max_over_ranks(sum(steps_ms) / K, world)
    tokens_step = w.B * w.N
    value = tokens_step * world / (ms * 1e-3)
    byts = forward_bytes(w.B, w.H, w.N, w.d, 2)
    C = 128
    roof = roofline_hbm(byts, ms, peaks["hbm_gbs"], known_traffic(MAIN_KERNEL, w))
    tens = tensor_fraction(chunk_flops(w.B, w.H, w.N, w.d, C), ms,
                           peaks["bf16_tflops"])
    if keep is not None:
        keep["main"] = {"form": "causal", "qkv": host_copy(q, k, v),
                        "y": out.cpu()}

    # ---------------- e2e through the C ABI with host buffers
    # (la_forward_host: page-locked host q, k, v in, host out back; the
    # library pipelines the copies over groups of heads)
    qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
    oh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    ws = torch.empty(la.host_workspace_bytes(q.shape, q.dtype), dtype=torch.uint8,
                     device=dev)

    def e2e_fn():
        la.forward_host(qh, kh, vh, causal=True, out=oh, workspace=ws)
    e2e_ms = timed_steps(e2e_fn, K, W, world, name=MAIN + " e2e")
    e2e_t = max_over_ranks(sum(e2e_ms) / K, world)
    e2e = {"value": round(tokens_step * world / (e2e_t * 1e-3), 1),
           "unit": "tokens/s", "h2d_bytes_per_step": 3 * q.numel() * 2,
           "d2h_bytes_per_step": out.numel() * 2,
           "ms_per_step": round(e2e_t, 4)}
    del qh, kh, vh, oh, ws

    paths = {}
    if not args.main_only:
        paths = run_other_paths(args, la, wl, dev, flush, peaks, world, rank, keep)
    clocks = sampler.stop()

    # ---------------- CPU baseline (oracle) on rank 0: timing and parity
    cpu = None
    errs = {}
    if keep is not None:
        cpu = cpu_baseline(w, keep, args.cpu_seconds)
        errs = cpu.get("max_rel_err", {})
        for name, r in paths.items():
            if name in errs:
                r["max_rel_err"] = errs[name]

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
            "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": round(ms, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"{MAIN} causal", "B": w.B, "H": w.H,
                       "N": w.N, "d": w.d, "global_batch": w.B * world,
                       "seq_len": w.N, "parallelism": f"replicas{world}",
                       "inputs": "N(0,1)/sqrt(d), bf16, seed=rank",
                       "l2": "flushed between timed steps (256 MiB written, "
                             "then another 256 MiB read)"},
            "roofline": roof, "tensor": tens, "chunk": C,
            "max_rel_err": errs.get("main"), "tolerance": wl.TOL["bf16"],
            "e2e": e2e, "gpu_launches": launches,
            "clocks": clocks, "cpu_baseline": cpu, "paths": paths,
            "peaks": peaks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_other_paths(args, la, wl, dev, flush, peaks, world, rank, keep):
    import torch
    res = {}
    Kx, Wx = max(3, args.steps // 2), max(3, args.warmup)
    mid = {}

    def mid_inputs():
        if not mid:
            w = wl.WORKLOADS[MID]
            mid["qkv"] = tuple(t.to(dev) for t in wl.make_workload_qkv(w, seed=rank))
        return mid["qkv"]

    def fwd_path(name, wkey, causal, decay=None, inputs=None, elem=2, kernel=None,
                 state=False, retention=False, gated=False):
        w = wl.WORKLOADS[wkey]
        try:
            if inputs is None:
                qq, kk, vv = (t.to(dev) for t in wl.make_workload_qkv(w, seed=rank))
            else:
                qq, kk, vv = inputs
            oo = torch.empty_like(qq)
            fn = lambda: la.forward(qq, kk, vv, causal=causal, decay=decay, out=oo)  # noqa
            extra = 0
            form = "causal" if causal else "noncausal"
            ga = Ss = zs = None
            if retention:
                # identity feature map, no normaliser (retention)
                fn = lambda: la.forward_variant(qq, kk, vv, causal=causal, decay=decay,  # noqa
                                                out=oo, feature_map="identity",
                                                normalise=False)
                form = "retention"
            if gated:
                # a data-dependent gate per token, uniform in [0.9, 1)
                gen = torch.Generator(device="cpu").manual_seed(200 + rank)
                ga = (0.9 + 0.1 * torch.rand(w.B, w.H, w.N, generator=gen)).to(dev)
                fn = lambda: la.forward_gated(qq, kk, vv, ga, out=oo)  # noqa
                extra = 4 * w.B * w.H * w.N  # the gates
                form = "gated"
            if state:
                # forward plus the final state (the prefill of a decode)
                Ss = torch.empty(w.B, w.H, w.d, w.d, device=dev)
                zs = torch.empty(w.B, w.H, w.d, device=dev)
                fn = lambda: la.forward_causal_state(qq, kk, vv, decay=decay, out=oo,  # noqa
                                                     S=Ss, z=zs)
                extra = 4 * w.B * w.H * (w.d * w.d + w.d)
                form = "state"
            replay, _ = capture(fn)
            steps = timed_steps(replay, Kx, Wx, world, flush, name=f"{wkey} {form}")
            la.check_device_status()
            ms = max_over_ranks(sum(steps) / Kx, world)
            r = {"tokens_per_s": round(w.B * w.N * world / (ms * 1e-3), 1),
                 "ms_per_step": round(ms, 4), "steps": Kx,
                 "roofline": roofline_hbm(forward_bytes(w.B, w.H, w.N, w.d, elem) + extra,
                                          ms, peaks["hbm_gbs"],
                                          known_traffic(kernel, w) if kernel else None)}
            if causal and elem == 2:
                C = 128
                r["tensor"] = tensor_fraction(chunk_flops(w.B, w.H, w.N, w.d, C),
                                              ms, peaks["bf16_tflops"])
                r["chunk"] = C
            res[name] = r
            if keep is not None:
                keep[name] = {"form": form, "qkv": host_copy(qq, kk, vv),
                              "y": oo.cpu(), "decay": decay,
                              "gates": None if ga is None else ga.cpu(),
                              "S": None if Ss is None else Ss.cpu(),
                              "z": None if zs is None else zs.cpu()}
        except Exception as e:  # keep the main line; report the failure
            res[name] = {"error": f"{type(e).__name__}: {e}"}

    fwd_path(f"{MID} causal", MID, True, inputs=mid_inputs(), kernel=MID_KERNEL)
    fwd_path(f"{MID} noncausal", MID, False, inputs=mid_inputs(),
             kernel="noncausal_kernel<64>")
    wd = wl.WORKLOADS["bf16_decay_b4h8_n16384_d128"]
    fwd_path("bf16_decay_b4h8_n16384_d128 causal", wd.name, True,
             decay=list(wd.decay), kernel="causal_wide_kernel<2>")
    fwd_path("fp32_causal_small causal", "fp32_causal_small", True, elem=4)
    fwd_path(f"{MID} causal with final state", MID, True, inputs=mid_inputs(),
             state=True, kernel="causal_kernel<64,0>+state")
    fwd_path("bf16_decay_b4h8_n16384_d128 retention", wd.name, True,
             decay=list(wd.decay), retention=True, kernel="causal_wide_kernel<1>")
    fwd_path(f"{MID} gated", MID, True, inputs=mid_inputs(), gated=True,
             kernel="causal_kernel<64,2>")
    # the same gated problem in fp32 (the CUDA-core kernels)
    fwd_path(f"{MID} gated fp32", MID, True, elem=4, gated=True,
             inputs=tuple(t.float() for t in mid_inputs()))

    # the delta rule over the same sequences (Gated DeltaNet: beta = 0.5,
    # alpha_h = 1 - 2^(-5-h) for every token, unit-norm keys)
    name = f"{MID} gated delta rule forward"
    try:
        w = wl.WORKLOADS[MID]
        qq, kk, vv = mid_inputs()
        kn = (kk.float() / kk.float().norm(dim=-1, keepdim=True)).to(kk.dtype)
        beta = torch.full((w.B, w.H, w.N), 0.5, device=dev)
        alpha = torch.tensor(wl.decay_schedule(w.H), dtype=torch.float32, device=dev)
        alpha = alpha.view(1, w.H, 1).expand(w.B, w.H, w.N).contiguous()
        oo = torch.empty_like(qq)
        replay, _ = capture(lambda: la.forward_delta(qq, kn, vv, beta, alpha, out=oo))
        steps = timed_steps(replay, Kx, Wx, world, flush, name=name)
        la.check_device_status()
        ms = max_over_ranks(sum(steps) / Kx, world)
        res[name] = {"tokens_per_s": round(w.B * w.N * world / (ms * 1e-3), 1),
                     "ms_per_step": round(ms, 4), "steps": Kx,
                     "roofline": roofline_hbm(forward_bytes(w.B, w.H, w.N, w.d, 2)
                                              + 8 * w.B * w.H * w.N, ms, peaks["hbm_gbs"]),
                     "note": "recurrent form on CUDA cores, tokens in order: "
                             "latency-bound, not HBM-bound"}
        if keep is not None:
            keep[name] = {"form": "delta_forward", "qkv": host_copy(qq, kn, vv),
                          "y": oo.cpu(), "beta": beta.cpu(), "alpha": alpha.cpu()}
    except Exception as e:  # keep the main line; report the failure
        res[name] = {"error": f"{type(e).__name__}: {e}"}
    mid.clear()
    try:
        res["decode_b256h32_d128"] = run_decode(la, wl, dev, peaks, world, rank,
                                                args, keep=keep,
                                                name="decode_b256h32_d128")
    except Exception as e:
        res["decode_b256h32_d128"] = {"error": f"{type(e).__name__}: {e}"}
    try:
        # the same decode with the per-head decay g_h = 1 - 2^(-5-h)
        wdec = wl.WORKLOADS["decode_b256h32_d128"]
        res["decode_b256h32_d128 decay"] = run_decode(
            la, wl, dev, peaks, world, rank, args,
            decay=list(wl.decay_schedule(wdec.H)), keep=keep,
            name="decode_b256h32_d128 decay")
    except Exception as e:
        res["decode_b256h32_d128 decay"] = {"error": f"{type(e).__name__}: {e}"}
    try:
        res["decode_b256h32_d128 gated delta rule"] = run_delta_decode(
            la, wl, dev, peaks, world, rank, args, keep=keep,
            name="decode_b256h32_d128 gated delta rule")
    except Exception as e:
        res["decode_b256h32_d128 gated delta rule"] = {"error": f"{type(e).__name__}: {e}"}
    return res


def decode_sample(B, H):
    """Heads (b, b mod H) for every sequence b: every batch entry and every
    head index appear; the decode legs' parity sample."""
    return [(b, b % H) for b in range(B)]


def keep_decode(keep, name, form, q, k, v, o, S, z=None, decay=None, beta=None,
                alpha=None):
    """Host copies of the sampled heads' tokens (all steps), their last output
    and their final state, for the CPU-baseline leg's replay."""
    B, H = q.shape[1], q.shape[2]
    bs = [b for b, _ in decode_sample(B, H)]
    hs = [h for _, h in decode_sample(B, H)]
    sel = lambda t: t[:, bs, hs].cpu()  # noqa: E731  [T, heads, d]
    keep[name] = {"form": form, "q": sel(q), "k": sel(k), "v": sel(v),
                  "y": o[bs, hs].cpu(), "S": S[bs, hs].cpu(),
                  "z": None if z is None else z[bs, hs].cpu(),
                  "decay": None if decay is None else [decay[h] for h in hs],
                  "beta": None if beta is None else beta[bs, hs].cpu(),
                  "alpha": None if alpha is None else alpha[bs, hs].cpu(),
                  "heads": f"{len(bs)} of {B * H} heads, (b, b mod {H}) for every b"}


def run_delta_decode(la, wl, dev, peaks, world, rank, args, keep=None, name=None):
    """The decode workload with the Gated DeltaNet step: beta = 0.5, alpha_h
    = 1 - 2^(-5-h) per head, unit-norm keys; 1024 untimed prefill steps,
    then the timed steps as one graph."""
    import torch
    w = wl.WORKLOADS["decode_b256h32_d128"]
    B, H, d = w.B, w.H, w.d
    P, T = w.extra["prefill"], w.extra["steps"]
    if args.decode_steps:
        T = args.decode_steps
    q, k, v = wl.make_decode_tokens(B, H, d, P + T, "bf16", seed=300 + rank,
                                    device=dev)
    k = (k.float() / k.float().norm(dim=-1, keepdim=True)).to(k.dtype)
    S = torch.zeros(B, H, d, d, device=dev)
    o = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    beta = torch.full((B, H), 0.5, device=dev)
    alpha = torch.tensor(wl.decay_schedule(H), dtype=torch.float32,
                         device=dev).expand(B, H).contiguous()
    step = lambda t: la.decode_step_delta(S, q[t], k[t], v[t], beta, alpha, out=o)  # noqa
    for t in range(P):
        step(t)
    replay, _ = capture(lambda: [step(t) for t in range(P, P + T)])
    S.zero_()
    for t in range(P):
        step(t)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.nvtx.range("la/" + (name or "decode")):
        e0.record(st)
        replay()
        e1.record(st)
        torch.cuda.synchronize()
    barrier(world)
    la.check_device_status()
    ms_total = max_over_ranks(e0.elapsed_time(e1), world)
    ms = ms_total / T
    if keep is not None:
        keep_decode(keep, name, "delta", q[:P + T], k[:P + T], v[:P + T], o, S,
                    beta=beta, alpha=alpha)
    byts = B * H * (2 * d * d * 4 + 4 * d * 2 + 8)  # S read and written, q k v o, beta alpha
    return {"tokens_per_s": round(B * T * world / (ms_total * 1e-3), 1),
            "ms_per_step": round(ms, 5), "steps": T, "prefill": P,
            "roofline": roofline_hbm(byts, ms, peaks["hbm_gbs"])}


def decode_bytes(BH, d, elem):
    """Compulsory bytes of one decode step: S and z read and written (fp32),
    q, k, v read, out written."""
    return BH * (2 * (d * d + d) * 4 + 4 * d * elem)


def run_decode(la, wl, dev, peaks, world, rank, args, decay=None, keep=None,
               name=None):
    import torch
    w = wl.WORKLOADS["decode_b256h32_d128"]
    B, H, d = w.B, w.H, w.d
    P, T = w.extra["prefill"], w.extra["steps"]
    if args.decode_steps:
        T = args.decode_steps
    q, k, v = wl.make_decode_tokens(B, H, d, P + T, "bf16", seed=100 + rank,
                                    device=dev)
    S = torch.zeros(B, H, d, d, device=dev)
    z = torch.zeros(B, H, d, device=dev)
    o = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    for t in range(P):  # prefill from the 1024 seeded tokens (untimed)
        la.decode_step(S, z, q[t], k[t], v[t], out=o, decay=decay)
    # the T timed steps, captured once as one graph of T launches
    replay, _ = capture(lambda: [la.decode_step(S, z, q[t], k[t], v[t], out=o,
                                                decay=decay)
                                  for t in range(P, P + T)])
    # capturing ran the steps once: restore the prefilled state
    S.zero_()
    z.zero_()
    for t in range(P):
        la.decode_step(S, z, q[t], k[t], v[t], out=o, decay=decay)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.nvtx.range("la/" + (name or "decode")):
        e0.record(st)
        replay()
        e1.record(st)
        torch.cuda.synchronize()
    barrier(world)
    la.check_device_status()
    ms_total = max_over_ranks(e0.elapsed_time(e1), world)
    ms = ms_total / T
    # the same T steps launched one by one from Python (no graph), from the
    # same prefilled state: the graph hides the host's per-launch gaps
    S.zero_()
    z.zero_()
    for t in range(P):
        la.decode_step(S, z, q[t], k[t], v[t], out=o, decay=decay)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0.record(st)
    for t in range(P, P + T):
        la.decode_step(S, z, q[t], k[t], v[t], out=o, decay=decay)
    e1.record(st)
    torch.cuda.synchronize()
    barrier(world)
    la.check_device_status()
    ms_eager = max_over_ranks(e0.elapsed_time(e1), world)
    if keep is not None:
        keep_decode(keep, name, "decode", q[:P + T], k[:P + T], v[:P + T], o, S,
                    z=z, decay=decay)
    return {"tokens_per_s": round(B * T * world / (ms_total * 1e-3), 1),
            "ms_per_step": round(ms, 5), "steps": T, "prefill": P,
            "state_bytes": S.numel() * 4,
            "l2": "state (512 MiB) larger than L2; steps back to back",
            "roofline": roofline_hbm(decode_bytes(B * H, d, 2), ms,
                                     peaks["hbm_gbs"]),
            "eager": {"tokens_per_s": round(B * T * world / (ms_eager * 1e-3), 1),
                      "ms_per_step": round(ms_eager / T, 5),
                      "launch": "one call per step, no CUDA graph"}}


# ------------------------------------------------------------------ oracle


def _max_err_by_heads(wl, y, ref_fn, q, k, v, cores, extra=None):
    """Max row-relative error of y [..., N, d] against ref_fn on groups of
    `cores` flattened heads (bounded host memory)."""
    N, d = q.shape[-2], q.shape[-1]
    flat = [t.reshape(-1, N, d) for t in (y, q, k, v)]
    ex = None if extra is None else extra.reshape(flat[1].shape[0], -1)
    worst = 0.0
    for h0 in range(0, flat[1].shape[0], cores):
        sl = slice(h0, h0 + cores)
        ref = ref_fn(flat[1][sl], flat[2][sl], flat[3][sl],
                     None if ex is None else ex[sl], h0)
        worst = max(worst, wl.max_row_rel_err(flat[0][sl], ref))
    return worst


def leg_error(oracle, wl, leg, cores):
    """Max row-relative error of one kept leg against the oracle."""
    import numpy as np
    form = leg["form"]
    if form == "delta_forward":
        q, k, v = leg["qkv"]
        ref, _ = oracle.delta_forward(q.float(), k.float(), v.float(),
                                      leg["beta"].double().numpy(),
                                      leg["alpha"].double().numpy(), nthreads=cores)
        return wl.max_row_rel_err(leg["y"], ref), {}
    if form in ("decode", "delta"):
        qs, ks, vs = leg["q"], leg["k"], leg["v"]
        nh, d = qs.shape[1], qs.shape[2]
        So = np.zeros((nh, d, d))
        zo = np.zeros((nh, d))
        for t in range(qs.shape[0]):
            if form == "decode":
                r = oracle.decode_step(So, zo, qs[t], ks[t], vs[t], leg["decay"],
                                       nthreads=cores)
            else:
                r = oracle.delta_step(So, qs[t], ks[t], vs[t], leg["beta"].numpy(),
                                      leg["alpha"].numpy())
        err = wl.max_row_rel_err(leg["y"], r)
        s_err = float(np.abs(leg["S"].double().numpy() - So).max() / np.abs(So).max())
        return err, {"state_rel_err": s_err, "sample": leg["heads"]}
    q, k, v = leg["qkv"]
    H = q.shape[1]
    BH = q.shape[0] * H
    g = None
    if leg.get("decay") is not None:
        g = np.array([leg["decay"][i % H] for i in range(BH)])

    def ref(qs, ks, vs, ex, h0):
        gs = None if g is None else g[h0:h0 + qs.shape[0]]
        if form == "noncausal":
            return oracle.noncausal(qs, ks, vs, nthreads=cores)
        if form == "retention":
            return oracle.causal(qs, ks, vs, gs, fmap=oracle.FMAP_IDENTITY,
                                 normalise=False, nthreads=cores)
        if form == "gated":
            return oracle.causal_gated(qs, ks, vs, ex, nthreads=cores)
        return oracle.causal(qs, ks, vs, gs, nthreads=cores)

    err = _max_err_by_heads(wl, leg["y"], ref, q, k, v, cores,
                            extra=leg.get("gates"))
    info = {}
    if form == "state":
        So, zo = oracle.causal_state(k, v, None if g is None else g)
        info["state_rel_err"] = float(
            np.abs(leg["S"].double().numpy() - So).max() / np.abs(So).max())
    return err, info


def cpu_baseline(w, keep, seconds):
    """Time the oracle (as it stands) on a bounded sample of the main
    workload: whole heads of the causal form, on all host cores.  Then
    compare the oracle with every kept leg's output (`max_rel_err`)."""
    import oracle
    from linear_attention_feature_gb300 import workloads as wl
    cores = os.cpu_count() or 1
    qs, ks, vs = keep["main"]["qkv"]
    BH = w.B * w.H
    # calibrate on one head, then take as many heads as fit the budget
    t0 = time.perf_counter()
    oracle.causal(qs[0, :1], ks[0, :1], vs[0, :1], nthreads=1)
    per_head = time.perf_counter() - t0
    heads = int(max(1, min(BH, seconds * cores / max(per_head, 1e-6))))
    heads = max(cores, heads) if BH >= cores else BH
    heads = min(heads, BH)
    qf = qs.reshape(BH, w.N, w.d)[:heads]
    kf = ks.reshape(BH, w.N, w.d)[:heads]
    vf = vs.reshape(BH, w.N, w.d)[:heads]
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.causal(qf, kf, vf, nthreads=cores)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= seconds:
            break
    frac = heads / BH
    # the same oracle on one core: one head, one thread, for about 2 s
    reps1 = 0
    t1 = time.perf_counter()
    while True:
        oracle.causal(qf[:1], kf[:1], vf[:1], nthreads=1)
        reps1 += 1
        dt1 = time.perf_counter() - t1
        if dt1 >= min(2.0, seconds / 5):
            break
    # parity of every timed leg against the oracle
    errs, info = {}, {}
    t2 = time.perf_counter()
    for name, leg in keep.items():
        try:
            e, extra = leg_error(oracle, wl, leg, cores)
            errs[name] = round(e, 6)
            if extra:
                info[name] = extra
        except Exception as ex:  # report, do not lose the line
            info[name] = {"error": f"{type(ex).__name__}: {ex}"}
    dt2 = time.perf_counter() - t2
    return {"value": round(reps * frac * w.B * w.N / dt, 1), "unit": "tokens/s",
            "cores": min(cores, heads), "kind": "oracle",
            "sample": f"causal form, {heads} of {BH} heads of {MAIN} "
                      f"(N={w.N}, d={w.d}), fp64, {reps} passes in {dt:.1f} s; "
                      f"tokens/s scaled by the head fraction",
            "single_core": {"value": round(reps1 * w.B * w.N / BH / dt1, 1),
                            "unit": "tokens/s",
                            "sample": f"1 head, 1 thread, {reps1} passes in "
                                      f"{dt1:.1f} s; scaled by the head fraction"},
            "max_rel_err": errs, "parity_detail": info,
            "parity_seconds": round(dt2, 1),
            "parity": "oracle vs each timed leg's output: every head of the "
                      "forward legs; decode legs: the sampled heads replayed "
                      "over every step, last output and final state"}


def run_reference(args):
    rank, world, _ = dist_info()
    if rank != 0:
        return
    import oracle
    from linear_attention_feature_gb300 import workloads as wl
    w = wl.WORKLOADS[MAIN]
    q, k, v = wl.make_workload_qkv(w, seed=0)
    cores = os.cpu_count() or 1
    BH = w.B * w.H
    heads = min(BH, cores)  # one head per core per step
    qf = q.reshape(BH, w.N, w.d)[:heads]
    kf = k.reshape(BH, w.N, w.d)[:heads]
    vf = v.reshape(BH, w.N, w.d)[:heads]
    for _ in range(args.warmup):
        oracle.causal(qf, kf, vf, nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.causal(qf, kf, vf, nthreads=cores)
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    value = (heads / BH) * w.B * w.N / dt
    sample = (f"each step: causal form on {heads} of {BH} heads of {MAIN} "
              f"(N={w.N}, d={w.d}), fp64; tokens/s scaled by the head fraction")
    line = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
            "impl": "reference", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{MAIN} causal", "B": w.B, "H": w.H,
                       "N": w.N, "d": w.d, "global_batch": w.B,
                       "seq_len": w.N},
            "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s",
                             "cores": heads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 1), "unit": "tokens/s",
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_kernel_case(B, H, N, d, form):
    """Four calls of one forward (or, for FORM decode / delta, four decode
    steps on a [B, H, d, d] state; N is ignored) on seeded inputs (no timing,
    no output)."""
    import torch
    import linear_attention_feature_gb300 as la
    from linear_attention_feature_gb300 import workloads as wl
    B, H, N, d = int(B), int(H), int(N), int(d)
    la.build.build()
    la.load_library()
    if form in ("decode", "delta"):
        q, k, v = wl.make_decode_tokens(B, H, d, 4, "bf16", seed=0, device="cuda")
        S = torch.zeros(B, H, d, d, device="cuda")
        z = torch.zeros(B, H, d, device="cuda")
        beta = torch.full((B, H), 0.5, device="cuda")
        for t in range(4):
            if form == "decode":
                la.decode_step(S, z, q[t], k[t], v[t])
            else:
                la.decode_step_delta(S, q[t], k[t], v[t], beta)
        torch.cuda.synchronize()
        la.check_device_status()
        return
    q, k, v = wl.make_qkv(B, H, N, d, "bf16", seed=0, device="cuda")
    out = torch.empty_like(q)
    decay = list(wl.decay_schedule(H)) if form == "decay" else None
    gates = None
    if form == "gated":  # a gate per token, uniform in [0.9, 1), as the gated leg
        gen = torch.Generator(device="cpu").manual_seed(200)
        gates = (0.9 + 0.1 * torch.rand(B, H, N, generator=gen)).to("cuda")
    if form == "retention":  # identity feature map, no normaliser, the decay schedule
        decay = list(wl.decay_schedule(H))
    S = z = None
    if form == "state":  # the forward plus its final state
        S = torch.empty(B, H, d, d, device="cuda")
        z = torch.empty(B, H, d, device="cuda")
    for _ in range(4):
        if gates is not None:
            la.forward_gated(q, k, v, gates, out=out)
        elif form == "retention":
            la.forward_variant(q, k, v, causal=True, decay=decay, out=out,
                               feature_map="identity", normalise=False)
        elif form == "state":
            la.forward_causal_state(q, k, v, out=out, S=S, z=z)
        else:
            la.forward(q, k, v, causal=form != "noncausal", decay=decay, out=out)
    torch.cuda.synchronize()
    la.check_device_status()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--main-only", action="store_true",
                    help="time only the main causal step")
    ap.add_argument("--no-cpu", action="store_true",
                    help="skip the CPU-baseline timing of the oracle")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--decode-steps", type=int, default=0,
                    help="timed decode steps (default: the workload's 1024)")
    ap.add_argument("--kernel-case", nargs=5,
                    metavar=("B", "H", "N", "D", "FORM"),
                    help="run one forward (FORM: causal, noncausal, decay, gated, "
                         "retention or state) "
                         "or decode step (FORM: decode or delta) four times "
                         "and exit; a driver for ncu captures")
    args = ap.parse_args()
    if args.kernel_case:
        run_kernel_case(*args.kernel_case)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

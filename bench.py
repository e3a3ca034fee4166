#!/usr/bin/env python
"""Benchmark of the GLA forward on GB300: one JSON line per run (rank 0).

A step is one gla_fwd over one batch of the workload (every kernel of the path), inputs resident in HBM.
The default workload is the long-context one (B=1, H=32, T=65536, K=V=128, bf16).  L2 is flushed (a write of
a buffer twice the L2 size) before each timed step, outside the timed events; the steps are enqueued back to
back, each between its own pair of CUDA events, and the host synchronises once after the last, so host launch
latency stays outside the events.  ``value`` is the tokens of all timed steps over their summed time; the
line also gives the median step and the median launch of each kernel (the roofline uses the latter), and a
``warm`` figure from the same number of steps without the flush.
Per-kernel times come from CUDA events that libgla records around each of its launches on the call's
stream (gla_profile_events).  ``e2e`` repeats the measurement through the same public call with the inputs
copied host->device from pinned memory and o/ht copied back inside the timed region.

``--impl reference`` times the fp64 CPU oracle (the only reference this method has) on a bounded sample of
the same workload instead.  ``--pass bwd`` measures the backward (gla_bwd: dq, dk, dv, dg, dh0 for a random
upstream gradient of o and of the final state) on the same workload instead of the forward.

Multi-GPU (torchrun): the workload's sequences are independent problems, so each rank runs its own copy
(weak scaling, no collective on the data path); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GLA fwd tokens/s on 1 GB300; % of BF16 tensor peak or HBM roofline"
DEFAULT_WORKLOAD = "long_t64k_h32"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# kernel name -> source file that defines it (a traffic figure is only reused while that file is unchanged)
KERNEL_SOURCES = {"out_ffma": "csrc/ffma_kernels.cu", "state_ffma": "csrc/ffma_kernels.cu",
                  "scan_segments": "csrc/ffma_kernels.cu", "plan_varlen": "csrc/ffma_kernels.cu",
                  "fused_tc": "csrc/tc_fused.cu", "ttt_linear_fwd": "csrc/ttt_ffma.cu",
                  "wy_fwd_ffma": "csrc/wy_ffma.cu", "wy_fwd_tc": "csrc/wy_tc.cu",
                  "bwd_chunk_sums_tc": "csrc/bwd_tc.cu", "bwd_grads": "csrc/bwd_ffma.cu",
                  "bwd_grads_tc": "csrc/bwd_grads_tc.cu", "ttt_linear_tc": "csrc/ttt_tc.cu"}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-warm", action="store_true", help="skip the warm-L2 figure")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd", "ttt", "wy"], default="fwd")
    ap.add_argument("--ttt-chunk", type=int, default=16, help="mini-batch size of --pass ttt")
    return ap.parse_args(argv)


# ------------------------------------------------------------------------------------------------
# workload arithmetic (algorithmic bytes / flops)
# ------------------------------------------------------------------------------------------------

def work_units(inp):
    rows = inp.q.shape[0] * inp.q.shape[1]
    esz = 4 if inp.dtype == "f32" else 2
    K, V, H = inp.K, inp.V, inp.H
    token_heads = rows * H
    in_bytes = token_heads * esz * (3 * K + V)
    out_bytes = token_heads * 4 * V
    state = inp.N * H * K * V * 4
    state_bytes = (state if inp.h0 is not None else 0) + state   # h0 read (if any) + ht write
    flops = token_heads * (2 * inp.chunk * K + 2 * inp.chunk * V + 4 * K * V)
    return dict(tokens=rows, token_heads=token_heads, bytes=in_bytes + out_bytes + state_bytes,
                in_bytes=in_bytes, out_bytes=out_bytes, state_bytes=state_bytes, flops=flops)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def peak_hbm(peaks):
    for key in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs"):
        if key in peaks and peaks[key]:
            return float(peaks[key])
    return FALLBACK_PEAKS["hbm_gbs"]


def traffic_for(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source is unchanged since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    src = KERNEL_SOURCES.get(kernel)
    if not os.path.exists(path) or src is None:
        return None
    with open(path) as f:
        table = json.load(f)
    ent = table.get(f"{kernel}@{workload}")
    if not ent:
        return None
    with open(os.path.join(ROOT, "chunkwise_gated_linear_chunked_gb300", src), "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    return ent["dram_bytes_per_launch"] if ent.get("src_sha") == sha else None


# ------------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="gla_clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------------
# CPU oracle sample (cpu_baseline and the reference arm)
# ------------------------------------------------------------------------------------------------

def oracle_sample(inp, seconds, head_start=0):
    """Run the fp64 oracle over groups of heads (all sequences of each head) until about `seconds` of wall
    time; return (tokens/s in the workload's unit, threads used, description).  A token of the metric is
    one row with all H heads, so each (sequence, head) item of length L counts L / H tokens."""
    import oracle
    from chunkwise_gated_linear_chunked_gb300.inputs import stored_numpy
    cores = os.cpu_count() or 1
    H = inp.H
    per_group = max(1, min(H, -(-cores // max(inp.N, 1))))
    t0 = time.perf_counter()
    token_heads, threads, groups, h = 0, 1, 0, head_start % H
    while True:
        heads = [(h + i) % H for i in range(per_group)]
        sel = lambda x: x[:, :, heads].contiguous()
        args = [stored_numpy(sel(x)) for x in (inp.q, inp.k, inp.v, inp.g)]
        h0 = None if inp.h0 is None else inp.h0[:, heads].contiguous().numpy()
        cu = None if inp.cu_seqlens is None else inp.cu_seqlens.numpy()
        ts = time.perf_counter()
        _, _, threads = oracle.gla_fwd(*args, inp.scale, h0=h0, cu_seqlens=cu, nthreads=cores)
        token_heads += inp.q.shape[0] * inp.q.shape[1] * len(heads)
        groups += 1
        h = (h + per_group) % H
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    desc = (f"fp64 oracle over {groups} group(s) of {per_group} head(s) x all {inp.N} sequence(s) "
            f"({token_heads} token-heads, {el:.1f} s wall)")
    return token_heads / H / el, threads, desc


def oracle_single_thread(inp, max_rows=16384):
    """The fp64 oracle on one thread: the first sequence's first head, its first `max_rows` rows at most;
    tokens/s in the workload's unit (a token is one row with all H heads, so one head-row counts 1/H)."""
    import oracle
    from chunkwise_gated_linear_chunked_gb300.inputs import stored_numpy
    if inp.cu_seqlens is None:
        rows = min(inp.q.shape[1], max_rows)
        sel = lambda x: x[:1, :rows, :1].contiguous()
        cu = None
    else:
        a0, a1 = int(inp.cu_seqlens[0]), int(inp.cu_seqlens[1])
        rows = min(a1 - a0, max_rows)
        sel = lambda x: x[:, a0:a0 + rows, :1].contiguous()
        cu = None
    args = [stored_numpy(sel(x)) for x in (inp.q, inp.k, inp.v, inp.g)]
    h0 = None if inp.h0 is None else inp.h0[:1, :1].contiguous().numpy()
    t0 = time.perf_counter()
    oracle.gla_fwd(*args, inp.scale, h0=h0, cu_seqlens=cu, nthreads=1)
    el = time.perf_counter() - t0
    return rows / inp.H / el, f"fp64 oracle, 1 thread, one head of the first sequence ({rows} rows, {el:.2f} s)"


# ------------------------------------------------------------------------------------------------

def main(argv=None):
    args = parse_args(argv)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    import torch
    from chunkwise_gated_linear_chunked_gb300.inputs import WORKLOADS, workload_inputs

    if args.workload not in WORKLOADS:
        raise SystemExit(f"unknown workload {args.workload}; choose from {list(WORKLOADS)}")
    w = WORKLOADS[args.workload]

    if args.impl == "reference":
        return run_reference(args, w, world, rank)

    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    from chunkwise_gated_linear_chunked_gb300 import binding

    inp = workload_inputs(args.workload)
    if args.pass_ == "bwd":
        return run_backward(args, w, inp, dev, dist, world, rank)
    if args.pass_ == "ttt":
        return run_ttt(args, w, inp, dev, dist, world, rank)
    if args.pass_ == "wy":
        return run_wy(args, w, dev, dist, world, rank)
    wu = work_units(inp)
    q, k, v, g = (x.to(dev) for x in (inp.q, inp.k, inp.v, inp.g))
    h0 = None if inp.h0 is None else inp.h0.to(dev)
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.to(dev)
    B, T, H, K, V, N = inp.q.shape[0], inp.q.shape[1], inp.H, inp.K, inp.V, inp.N
    code = binding.GLA_F32 if inp.dtype == "f32" else binding.GLA_BF16
    o = torch.empty(B, T, H, V, dtype=torch.float32, device=dev)
    ht = torch.empty(N, H, K, V, dtype=torch.float32, device=dev)
    ws = torch.zeros(max(256, binding.workspace_size(B, T, H, K, V, N, inp.chunk, code)), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream()

    def step():
        rc = binding.fwd_into(q, k, v, g, o, inp.scale, h0, ht, cu, N, B, T, H, K, V, inp.chunk, code, ws,
                              stream)
        if rc != 0:
            raise binding.GlaError(rc)

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 64 << 20), dtype=torch.uint8, device=dev)

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    if binding.get_status(ws) != 0:
        raise RuntimeError("device status error during warm-up")

    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clocks:
        step_ms, per_kernel, launches = timed_steps(step, flush, stream, args.steps)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    total_ms = max_over_ranks(sum(step_ms), dist, dev)
    status = binding.get_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {binding.strerror(status)} in the timed region")

    value = whole_job_value(wu["tokens"], args.steps, world, total_ms)
    ms_per_step = total_ms / args.steps

    # the same steps without the L2 flush (inputs of the small workloads then partly stay in L2)
    warm = None
    if not args.no_warm:
        wstep_ms, wper_kernel, _ = timed_steps(step, None, stream, args.steps)
        torch.cuda.synchronize()
        if binding.get_status(ws) != 0:
            raise RuntimeError("device status error in the warm-L2 steps")
        warm = {"ms_per_step_median": round(statistics.median(wstep_ms), 5),
                "value": round(wu["tokens"] / (statistics.median(wstep_ms) / 1e3), 1),
                "kernels_ms": {n: round(statistics.median(v), 5) for n, v in wper_kernel.items()},
                "l2": "not flushed between steps"}

    # dominant kernel and its roofline (median launch time)
    peaks, peak_src = load_peaks()
    kern_tot = {n: sum(v) for n, v in per_kernel.items()}
    dom = max(kern_tot, key=kern_tot.get)
    dom_ms = statistics.median(per_kernel[dom])
    dom_bytes = kernel_algorithmic_bytes(dom, wu)
    hbm = peak_hbm(peaks)
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "peak_source": peak_src,
                "traffic": traffic_for(dom, args.workload),
                "algorithmic_bytes_per_launch": dom_bytes,
                "tensor_tflops_algorithmic": round(wu["flops"] / (ms_per_step / 1e3) / 1e12, 2)}

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(args, inp, binding, dev, stream, flush)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        val, threads, desc = oracle_sample(inp, args.cpu_seconds)
        v1, desc1 = oracle_single_thread(inp)
        cpu = {"value": round(val, 1), "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": desc,
               "hardware_concurrency": os.cpu_count(),
               "single_thread": {"value": round(v1, 1), "unit": "tokens/s", "sample": desc1}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "ms_per_step_median": round(statistics.median(step_ms), 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": compute_dtype(inp), "data": "synthetic",
            "config": {"workload": args.workload, "desc": w.note, "B": B, "T": T, "H": H, "K": K, "V": V,
                       "N": N, "chunk": inp.chunk, "input_dtype": inp.dtype, "h0": inp.h0 is not None,
                       "tokens_per_step": wu["tokens"], "algorithmic_bytes_per_step": wu["bytes"],
                       "l2": "flushed before every timed step (zero-fill of a 2x L2 buffer, outside the events)",
                       "parallelism": "replicas" if world == 1 else f"weak x{world} (independent sequences)"},
            "roofline": roofline,
            "kernels_ms": {n: round(statistics.median(v), 5) for n, v in per_kernel.items()},
            "warm": warm, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches, "clocks": clocks.summary(),
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


FP32_LANES_PER_SM = 128   # fp32 FMA lanes per SM (4 sub-partitions x 32)


def bwd_chunks(inp):
    if inp.cu_seqlens is None:
        return inp.q.shape[0] * -(-inp.q.shape[1] // inp.chunk)
    lens = (inp.cu_seqlens[1:] - inp.cu_seqlens[:-1]).tolist()
    return sum(max(1, -(-L // inp.chunk)) for L in lens)


def bwd_kernel_flops(name, inp):
    """Algorithmic flops of one launch of a backward kernel (2 per multiply-add, masked tiles counted)."""
    C, K, V, H = inp.chunk, inp.K, inp.V, inp.H
    nc = bwd_chunks(inp) * H
    if name in ("bwd_grads", "bwd_grads_tc"):
        return 2 * nc * (C * C * (3 * K + 2 * V) + 3 * C * K * V)
    if name in ("bwd_chunk_sums", "bwd_chunk_sums_tc"):
        return 2 * nc * 2 * C * K * V
    if name == "bwd_scan":
        return 2 * 2 * nc * K * V
    return 0


def bwd_kernel_bytes(name, inp):
    """Algorithmic HBM bytes of one launch of a tensor-core backward kernel: every input row read once, every
    fp32 output row written once, the per-chunk [K][V] fp32 tiles it reads or writes moved once."""
    K, V, H = inp.K, inp.V, inp.H
    rows = inp.q.shape[0] * inp.q.shape[1] * H
    nc = bwd_chunks(inp) * H
    isz = 2 if inp.dtype in ("bf16", "f16") else 4
    if name == "bwd_grads_tc":   # q, k, g, v, do in; S_c, R_c in; dq, dk, dg, dv out; chunk sums of dg out
        return rows * (isz * (3 * K + 2 * V) + 4 * (3 * K + V)) + nc * (2 * K * V * 4 + K * 4)
    if name == "bwd_chunk_sums_tc":   # q, k, g, v, do in; the two [K][V] contributions and G_l out
        return rows * isz * (3 * K + 2 * V) + nc * (2 * K * V * 4 + K * 4)
    return 0


def oracle_bwd_sample(inp, do, dht, seconds):
    """The fp64 backward oracle over groups of heads for about `seconds`; tokens/s, threads, description."""
    import oracle
    from chunkwise_gated_linear_chunked_gb300.inputs import stored_numpy
    cores = os.cpu_count() or 1
    H = inp.H
    per_group = max(1, min(H, -(-cores // max(inp.N, 1))))
    t0 = time.perf_counter()
    token_heads, threads, groups, h = 0, 1, 0, 0
    while True:
        heads = [(h + i) % H for i in range(per_group)]
        sel = lambda x: x[:, :, heads].contiguous()
        arrs = [stored_numpy(sel(x)) for x in (inp.q, inp.k, inp.v, inp.g, do)]
        st = lambda x: None if x is None else x[:, heads].contiguous().numpy()
        cu = None if inp.cu_seqlens is None else inp.cu_seqlens.numpy()
        oracle.gla_bwd(*arrs, inp.scale, h0=st(inp.h0), dht=st(dht), cu_seqlens=cu, nthreads=cores)
        threads = min(cores, inp.N * len(heads))
        token_heads += inp.q.shape[0] * inp.q.shape[1] * len(heads)
        groups += 1
        h = (h + per_group) % H
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    desc = (f"fp64 backward oracle over {groups} group(s) of {per_group} head(s) x all {inp.N} sequence(s) "
            f"({token_heads} token-heads, {el:.1f} s wall)")
    return token_heads / H / el, threads, desc


def run_backward(args, w, inp, dev, dist, world, rank):
    """The backward step: one gla_bwd over the workload with a seeded random upstream gradient of o (input
    dtype) and of the final state (fp32); inputs resident in HBM, L2 flushed before each step."""
    import torch
    from chunkwise_gated_linear_chunked_gb300 import binding
    B, T, H, K, V, N = inp.q.shape[0], inp.q.shape[1], inp.H, inp.K, inp.V, inp.N
    code = binding.GLA_F32 if inp.dtype == "f32" else binding.GLA_BF16
    gen = torch.Generator().manual_seed(w.seed + 7)
    do_cpu = torch.randn(tuple(inp.v.shape), generator=gen).to(inp.v.dtype)
    dht_cpu = torch.randn(N, H, K, V, generator=gen) * 0.5
    q, k, v, g, do = (x.to(dev) for x in (inp.q, inp.k, inp.v, inp.g, do_cpu))
    dht = dht_cpu.to(dev)
    h0 = None if inp.h0 is None else inp.h0.to(dev)
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.to(dev)
    f32 = dict(dtype=torch.float32, device=dev)
    dq, dk, dg = (torch.empty(B, T, H, K, **f32) for _ in range(3))
    dv = torch.empty(B, T, H, V, **f32)
    dh0 = torch.empty(N, H, K, V, **f32)
    ws = torch.zeros(max(256, binding.bwd_workspace_size(B, T, H, K, V, N, inp.chunk, code)), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream()

    def step():
        rc = binding.bwd_into(q, k, v, g, do, inp.scale, h0, dht, dq, dk, dv, dg, dh0, cu, N, B, T, H, K, V,
                              inp.chunk, code, ws, stream)
        if rc != 0:
            raise binding.GlaError(rc, "gla_bwd")

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 64 << 20), dtype=torch.uint8, device=dev)
    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    if binding.get_status(ws) != 0:
        raise RuntimeError("device status error during warm-up")
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clocks:
        step_ms, per_kernel, launches = timed_steps(step, flush, stream, args.steps)
    if dist is not None:
        dist.barrier()
    total_ms = max_over_ranks(sum(step_ms), dist, dev)
    if binding.get_status(ws) != 0:
        raise RuntimeError("device status error in the timed region")
    tokens = B * T
    value = whole_job_value(tokens, args.steps, world, total_ms)
    ms_per_step = total_ms / args.steps
    kern_tot = {n: sum(x) for n, x in per_kernel.items()}
    dom = max(kern_tot, key=kern_tot.get)
    dom_ms = statistics.median(per_kernel[dom])
    props = torch.cuda.get_device_properties(dev)
    csum = clocks.summary()
    mhz = csum.get("sm_max_mhz") or 2070.0
    peak = props.multi_processor_count * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12
    flops = bwd_kernel_flops(dom, inp)
    nbytes = bwd_kernel_bytes(dom, inp)
    if nbytes:   # a tensor-core kernel: its fp32-accurate products are far from the tensor peak; HBM bounds it
        peaks, src = load_peaks()
        hbm = peak_hbm(peaks)
        achieved = nbytes / (dom_ms / 1e3) / 1e9
        roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": hbm,
                    "unit": "GB/s", "frac": round(achieved / hbm, 4), "peak_source": f"{src} HBM copy",
                    "traffic": traffic_for(dom, args.workload), "algorithmic_bytes_per_launch": nbytes,
                    "algorithmic_flops_per_launch": flops}
    else:
        achieved = flops / (dom_ms / 1e3) / 1e12
        roofline = {"bound": "alu", "kernel": dom, "achieved": round(achieved, 2), "peak": round(peak, 1),
                    "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                    "peak_source": f"fp32 FMA: {props.multi_processor_count} SMs x {FP32_LANES_PER_SM} lanes x 2 x "
                                   f"{mhz:.0f} MHz", "traffic": traffic_for(dom, args.workload),
                    "algorithmic_flops_per_launch": flops}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        val, threads, desc = oracle_bwd_sample(inp, do_cpu, dht_cpu, args.cpu_seconds)
        cpu = {"value": round(val, 1), "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": desc}
    if rank == 0:
        line = {
            "metric": "GLA bwd tokens/s on 1 GB300 (dq, dk, dv, dg, dh0); % of fp32 CUDA-core peak",
            "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": args.workload, "pass": "bwd", "desc": w.note, "B": B, "T": T, "H": H,
                       "K": K, "V": V, "N": N, "chunk": inp.chunk, "input_dtype": inp.dtype,
                       "h0": inp.h0 is not None, "dht": True,
                       "l2": "flushed before every timed step (zero-fill of a 2x L2 buffer, outside the events)",
                       "parallelism": "replicas" if world == 1 else f"weak x{world} (independent sequences)"},
            "roofline": roofline,
            "kernels_ms": {n: round(statistics.median(x), 5) for n, x in per_kernel.items()},
            "cpu_baseline": cpu, "e2e": None, "gpu_launches": launches, "clocks": csum,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def ttt_inputs(w, inp):
    """TTT-linear inputs on the workload's q, k, v (K == V): seeded LayerNorm weight/bias and learning rate."""
    import torch
    gen = torch.Generator().manual_seed(w.seed + 11)
    H, D = inp.H, inp.K
    lw = 1.0 + 0.2 * torch.randn(H, D, generator=gen)
    lb = 0.1 * torch.randn(H, D, generator=gen)
    eta = 0.02 + 0.05 * torch.rand(tuple(inp.q.shape[:3]), generator=gen)
    return lw, lb, eta


def ttt_flops(inp, chunk):
    """Algorithmic flops of one TTT-linear launch (2 per multiply-add): per mini-batch of BT rows the
    k h and q h products (2 BT D^2), the masked scores and their use (~BT^2 D) and the state update (BT D^2)."""
    D, H = inp.K, inp.H
    if inp.cu_seqlens is None:
        lens = [inp.q.shape[1]] * inp.q.shape[0]
    else:
        lens = (inp.cu_seqlens[1:] - inp.cu_seqlens[:-1]).tolist()
    total = 0
    for L in lens:
        for r0 in range(0, L, chunk):
            bt = min(chunk, L - r0)
            total += 3 * bt * D * D + bt * bt * D
    return 2 * total * H


def run_ttt(args, w, inp, dev, dist, world, rank):
    """The TTT-linear forward step over the workload (one gla_ttt_linear_fwd), L2 flushed before each step."""
    import torch
    from chunkwise_gated_linear_chunked_gb300 import binding
    if inp.K != inp.V:
        raise SystemExit("--pass ttt needs a workload with K == V")
    lw, lb, eta = ttt_inputs(w, inp)
    q, k, v = (x.to(dev) for x in (inp.q, inp.k, inp.v))
    lwd, lbd, etad = lw.to(dev), lb.to(dev), eta.to(dev)
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.to(dev)
    scale = inp.K ** -0.5
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        binding.ttt_linear_fwd(q, k, v, lwd, lbd, etad, scale=scale, eps=1e-6, chunk=args.ttt_chunk,
                               cu_seqlens=cu, workspace=ws, stream=stream)

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 64 << 20), dtype=torch.uint8, device=dev)
    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clocks:
        step_ms, per_kernel, launches = timed_steps(step, flush, stream, args.steps)
    if dist is not None:
        dist.barrier()
    total_ms = max_over_ranks(sum(step_ms), dist, dev)
    if binding.get_status(ws) != 0:
        raise RuntimeError("device status error in the timed region")
    B, T = inp.q.shape[0], inp.q.shape[1]
    value = whole_job_value(B * T, args.steps, world, total_ms)
    dom = max(per_kernel, key=lambda n: sum(per_kernel[n]))   # ttt_linear_tc (bf16, D = 128) or ttt_linear_fwd
    dom_ms = statistics.median(per_kernel[dom])
    props = torch.cuda.get_device_properties(dev)
    csum = clocks.summary()
    mhz = csum.get("sm_max_mhz") or 2070.0
    flops = ttt_flops(inp, args.ttt_chunk)
    achieved = flops / (dom_ms / 1e3) / 1e12
    if dom == "ttt_linear_tc":   # the products on the tensor cores: against the measured bf16 peak
        peaks, psrc = load_peaks()
        peak = float(peaks.get("bf16_tflops") or FALLBACK_PEAKS["bf16_tflops"])
        bound, peak_source = "tensor", f"{psrc} bf16 dense (cuBLAS burst)"
    else:
        peak = props.multi_processor_count * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12
        bound = "alu"
        peak_source = f"fp32 FMA: {props.multi_processor_count} SMs x {FP32_LANES_PER_SM} lanes x 2 x {mhz:.0f} MHz"
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        from chunkwise_gated_linear_chunked_gb300.inputs import stored_numpy
        cores = os.cpu_count() or 1
        t0 = time.perf_counter()
        token_heads, h = 0, 0
        while True:
            heads = [(h + i) % inp.H for i in range(min(inp.H, cores))]
            sel = lambda x: x[:, :, heads].contiguous()
            oracle.ttt_linear_fwd(*(stored_numpy(sel(x)) for x in (inp.q, inp.k, inp.v)), lw[heads].numpy(),
                                  lb[heads].numpy(), sel(eta).numpy(), scale, 1e-6, args.ttt_chunk,
                                  cu_seqlens=None if inp.cu_seqlens is None else inp.cu_seqlens.numpy(),
                                  nthreads=cores)
            token_heads += B * T * len(heads)
            h = (h + len(heads)) % inp.H
            if time.perf_counter() - t0 >= args.cpu_seconds:
                break
        el = time.perf_counter() - t0
        cpu = {"value": round(token_heads / inp.H / el, 1), "unit": "tokens/s", "cores": min(cores, inp.N * inp.H),
               "kind": "oracle", "sample": f"fp64 TTT-linear oracle, {token_heads} token-heads, {el:.1f} s wall"}
    if rank == 0:
        line = {
            "metric": "TTT-linear fwd tokens/s on 1 GB300; % of fp32 CUDA-core peak",
            "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16x2 (fp32 state split in two bf16 terms for its products), f32 state and accumulate" if dom == "ttt_linear_tc" else "f32", "data": "synthetic",
            "config": {"workload": args.workload, "pass": "ttt", "chunk": args.ttt_chunk, "B": B, "T": T,
                       "H": inp.H, "D": inp.K, "input_dtype": inp.dtype,
                       "l2": "flushed before every timed step (zero-fill of a 2x L2 buffer, outside the events)",
                       "parallelism": "replicas" if world == 1 else f"weak x{world} (independent sequences)"},
            "roofline": {"bound": bound, "kernel": dom, "achieved": round(achieved, 2), "peak": round(peak, 1),
                         "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "peak_source": peak_source,
                         "traffic": traffic_for(dom, args.workload), "algorithmic_flops_per_launch": flops},
            "kernels_ms": {n: round(statistics.median(x), 5) for n, x in per_kernel.items()},
            "cpu_baseline": cpu, "e2e": None, "gpu_launches": launches, "clocks": csum,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def wy_bytes_flops(x):
    """Algorithmic bytes and flops of one WY launch: k read once per key head, v, beta, A, g read once,
    w and u written once; 2 flops per multiply-add of the chunk products (BT x BT by BT x (K + V))."""
    esz = 4 if x.dtype == "f32" else 2
    rows = x.B * x.T
    nbytes = rows * (x.H * x.K + x.HV * (x.V + 1 + x.BT)) * esz + rows * x.HV * 4 * (x.g is not None)
    nbytes += rows * x.HV * (x.K + x.V) * 4
    if x.cu_seqlens is None:
        lens = [x.T] * x.B
    else:
        lens = (x.cu_seqlens[1:] - x.cu_seqlens[:-1]).tolist()
    flops = 0
    for L in lens:
        for r0 in range(0, L, x.BT):
            m = min(x.BT, L - r0)
            flops += 2 * m * m * (x.K + x.V)
    return nbytes, flops * x.HV


def wy_roofline(dom, dom_ms, nbytes, flops, alu_peak, hbm_peak, hbm_src, props, mhz, workload):
    """The tensor-core kernel is bounded by HBM (its flops are cheap on tcgen05); the CUDA-core kernel by the
    fp32 FMA rate (about 20 flop per byte against a ridge of about 12)."""
    gbs = nbytes / (dom_ms / 1e3) / 1e9
    tflops = flops / (dom_ms / 1e3) / 1e12
    if dom == "wy_fwd_tc":
        return {"bound": "hbm", "kernel": dom, "achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(gbs / hbm_peak, 4), "peak_source": hbm_src, "traffic": traffic_for(dom, workload),
                "algorithmic_bytes_per_launch": nbytes, "achieved_tflops_fp32_equivalent": round(tflops, 2)}
    return {"bound": "alu", "kernel": dom, "achieved": round(tflops, 2), "peak": round(alu_peak, 1),
            "unit": "TFLOP/s", "frac": round(tflops / alu_peak, 4),
            "peak_source": f"fp32 FMA: {props.multi_processor_count} SMs x {FP32_LANES_PER_SM} lanes x 2 x {mhz:.0f} MHz",
            "traffic": traffic_for(dom, workload), "algorithmic_flops_per_launch": flops,
            "hbm": {"algorithmic_bytes_per_launch": nbytes, "achieved_gbs": round(gbs, 1), "peak_gbs": hbm_peak,
                    "peak_source": hbm_src}}


def run_wy(args, w, dev, dist, world, rank):
    """The WY-representation forward of the gated delta rule (one gla_wy_fwd) on the workload's shapes."""
    import torch
    from chunkwise_gated_linear_chunked_gb300 import binding
    from chunkwise_gated_linear_chunked_gb300.inputs import stored_numpy, wy_workload_inputs
    x = wy_workload_inputs(args.workload)
    k, v, beta, A, g = (t.to(dev) for t in (x.k, x.v, x.beta, x.A, x.g))
    cu = None if x.cu_seqlens is None else x.cu_seqlens.to(dev)
    N = x.B if cu is None else cu.numel() - 1
    ws = torch.zeros(max(int(binding.lib().gla_wy_workspace_size(x.T, N, x.BT, int(cu is not None))), 256),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    wo = torch.empty(x.B, x.T, x.HV, x.K, dtype=torch.float32, device=dev)
    uo = torch.empty(x.B, x.T, x.HV, x.V, dtype=torch.float32, device=dev)
    code = {"f32": binding.GLA_F32, "bf16": binding.GLA_BF16, "f16": binding.GLA_F16}[x.dtype]

    def step():
        rc = binding.wy_into(k, v, beta, A, g, wo, uo, cu, N, x.B, x.T, x.H, x.HV, x.K, x.V, x.BT, code, ws,
                             stream)
        if rc != 0:
            raise RuntimeError(f"gla_wy_fwd returned {rc}")

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 64 << 20), dtype=torch.uint8, device=dev)
    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clocks:
        step_ms, per_kernel, launches = timed_steps(step, flush, stream, args.steps)
    if dist is not None:
        dist.barrier()
    total_ms = max_over_ranks(sum(step_ms), dist, dev)
    if binding.get_status(ws) != 0:
        raise RuntimeError("device status error in the timed region")
    value = whole_job_value(x.B * x.T, args.steps, world, total_ms)
    dom = max((n_ for n_ in per_kernel if n_ != "plan_varlen"), key=lambda n_: statistics.median(per_kernel[n_]))
    dom_ms = statistics.median(per_kernel[dom])
    props = torch.cuda.get_device_properties(dev)
    csum = clocks.summary()
    mhz = csum.get("sm_max_mhz") or 2070.0
    peak = props.multi_processor_count * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12
    nbytes, flops = wy_bytes_flops(x)
    achieved = flops / (dom_ms / 1e3) / 1e12
    peaks, hbm_src = load_peaks()
    hbm_peak = peak_hbm(peaks)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        cores = os.cpu_count() or 1
        t0 = time.perf_counter()
        rows_done, n = 0, 0
        while True:   # whole sequences of the workload, in turn, until the time budget is used
            if x.cu_seqlens is None:
                sl = slice(n, n + 1)
                sub = [t[sl] for t in (x.k, x.v, x.beta, x.A, x.g)]
                cus = None
            else:
                a0, a1 = int(x.cu_seqlens[n]), int(x.cu_seqlens[n + 1])
                sub = [t[:, a0:a1] for t in (x.k, x.v, x.beta, x.A, x.g)]
                cus = np.array([0, a1 - a0], dtype=np.int32)
            oracle.wy_fwd(*(stored_numpy(t.contiguous()) for t in sub[:4]), sub[4].double().numpy(),
                          cu_seqlens=cus, nthreads=cores)
            rows_done += sub[0].shape[0] * sub[0].shape[1]
            n = (n + 1) % (x.B if x.cu_seqlens is None else x.cu_seqlens.numel() - 1)
            if time.perf_counter() - t0 >= args.cpu_seconds:
                break
        el = time.perf_counter() - t0
        cpu = {"value": round(rows_done / el, 1), "unit": "tokens/s", "cores": min(cores, x.HV),
               "kind": "oracle", "sample": f"fp64 WY oracle on whole sequences of the workload, {rows_done} rows, "
                                           f"{el:.1f} s wall"}
    if rank == 0:
        line = {
            "metric": "gated-delta WY forward tokens/s on 1 GB300",
            "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16x2 (fp32 operands split in two bf16 terms), f32 accumulate" if dom == "wy_fwd_tc" else "f32",
            "data": "synthetic",
            "config": {"workload": args.workload, "pass": "wy", "chunk": x.BT, "B": x.B, "T": x.T, "H": x.H,
                       "HV": x.HV, "K": x.K, "V": x.V, "input_dtype": x.dtype, "outputs": "fp32",
                       "l2": "flushed before every timed step (zero-fill of a 2x L2 buffer, outside the events)",
                       "parallelism": "replicas" if world == 1 else f"weak x{world} (independent sequences)"},
            "roofline": wy_roofline(dom, dom_ms, nbytes, flops, peak, hbm_peak, hbm_src, props, mhz, args.workload),
            "kernels_ms": {n_: round(statistics.median(t), 5) for n_, t in per_kernel.items()},
            "cpu_baseline": cpu, "e2e": None, "gpu_launches": launches, "clocks": csum,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def compute_dtype(inp):
    """Arithmetic type of the path: fp16 tensor-core operands (fp32 accumulation) for bf16 inputs with
    K == 128 and V a multiple of 128, fp32 CUDA-core arithmetic otherwise."""
    return "f16" if inp.dtype == "bf16" and inp.K == 128 and inp.V % 128 == 0 else "f32"


def timed_steps(step, flush, stream, steps):
    """Time `steps` calls of step() on the device.  Every step is preceded by an L2 flush (outside its
    events) and bracketed by its own pair of CUDA events and its own per-kernel event set on the launching
    stream; the steps are enqueued back to back and the host synchronises once at the end, so host launch
    latency does not sit inside a step's events.  Returns (per-step ms, {kernel: [ms per launch]}, launches)."""
    import torch
    from chunkwise_gated_linear_chunked_gb300 import binding
    timers = [binding.KernelTimer() for _ in range(steps)]
    events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for timer, (start, end) in zip(timers, events):
        if flush is not None:
            flush.zero_()
        with timer:
            start.record(stream)
            step()
            end.record(stream)
    torch.cuda.synchronize()
    step_ms, per_kernel, launches = [], {}, 0
    for timer, (start, end) in zip(timers, events):
        step_ms.append(start.elapsed_time(end))
        res = timer.results()
        launches += len(res)
        for name, ms in res:
            per_kernel.setdefault(name, []).append(ms)
    return step_ms, per_kernel, launches


def max_over_ranks(total_ms, dist=None, device=None):
    """The timed region's length: the maximum over ranks of each rank's timed total (ms)."""
    if dist is None:
        return total_ms
    import torch
    t = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(tokens_per_step, steps, world, total_ms):
    """Tokens per second over all ranks: every rank processes `tokens_per_step` each step (weak scaling)."""
    return tokens_per_step * steps * world / (total_ms / 1e3)


def kernel_algorithmic_bytes(name, wu):
    if name in ("out_ffma", "fused_tc"):
        return wu["bytes"]
    if name == "state_ffma":
        return wu["in_bytes"]   # upper bound: k, g, v of the non-final segments are a subset
    return wu["state_bytes"]


def measure_e2e(args, inp, binding, dev, stream, flush):
    """Same metric through the public host-buffer call gla_fwd_host: inputs in pinned host memory, o and ht
    back into pinned host memory, every copy inside the timed events.  The call pipelines head groups (the
    next group's inputs copied in while a group computes and the previous group's outputs are copied out)."""
    import torch
    host = [x.contiguous().pin_memory() for x in (inp.q, inp.k, inp.v, inp.g)]
    host_h0 = None if inp.h0 is None else inp.h0.pin_memory()
    host_cu = None if inp.cu_seqlens is None else inp.cu_seqlens.pin_memory()
    B, T, H, K, V, N = inp.q.shape[0], inp.q.shape[1], inp.H, inp.K, inp.V, inp.N
    ho = torch.empty(B, T, H, V, dtype=torch.float32).pin_memory()
    hht = torch.empty(N, H, K, V, dtype=torch.float32).pin_memory()
    code = binding.GLA_F32 if inp.dtype == "f32" else binding.GLA_BF16
    groups = next(gr for gr in (4, 2, 1) if H % gr == 0)   # measured on long_t64k_h32: 1 16.6 ms, 2 14.1, 4 14.0, 8 14.4, 16 19.5
    ws = torch.zeros(max(256, binding.host_workspace_size(B, T, H, K, V, N, inp.chunk, code, groups)),
                     dtype=torch.uint8, device=dev)
    h2d = sum(x.numel() * x.element_size() for x in host) + \
        sum(x.numel() * x.element_size() for x in (host_h0, host_cu) if x is not None)
    d2h = ho.numel() * ho.element_size() + hht.numel() * hht.element_size()

    def e2e_step():
        rc = binding.fwd_host_into(*host, ho, inp.scale, host_h0, hht, host_cu, N, B, T, H, K, V, inp.chunk, code,
                                   groups, ws, stream)
        if rc != 0:
            raise binding.GlaError(rc)

    for _ in range(max(args.warmup, 1)):
        e2e_step()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    tot = 0.0
    for _ in range(args.steps):
        flush.zero_()
        s.record(stream)
        e2e_step()
        e.record(stream)
        torch.cuda.synchronize()
        tot += s.elapsed_time(e)
    tokens = B * T
    return {"value": round(tokens * args.steps / (tot / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(tot / args.steps, 4),
            "api": f"gla_fwd_host, {groups} head groups"}


def run_reference(args, w, world, rank):
    """The fp64 CPU oracle as the reference arm: each step times a bounded sample of the workload."""
    if rank != 0:
        return
    from chunkwise_gated_linear_chunked_gb300.inputs import workload_inputs
    inp = workload_inputs(args.workload)
    per_step = max(1.0, min(args.cpu_seconds, 150.0 / max(args.steps + args.warmup, 1)))
    for i in range(args.warmup):
        oracle_sample(inp, 0.0, head_start=i)
    vals, threads, desc = [], 1, ""
    t0 = time.perf_counter()
    for i in range(args.steps):
        val, threads, desc = oracle_sample(inp, per_step, head_start=i)
        vals.append(val)
    el = time.perf_counter() - t0
    value = statistics.mean(vals)
    wu = work_units(inp)
    line = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el * 1e3 / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": args.workload, "desc": w.note, "tokens_per_step": wu["tokens"],
                       "sample": "each step: heads of the workload, all sequences, ~%.1f s of oracle time"
                                 % per_step},
            "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

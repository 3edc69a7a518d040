#!/usr/bin/env python3
"""Benchmark: exact attention forward + backward on GB300 through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--sweep]

A step is one pass of the whole hot path over one batch: fa_fwd (O, LSE) then
fa_bwd (D preprocess, the backward kernel, dQ conversion).  The default
workload is long-context causal training attention (B=4, H=32, N=8192,
d=128, causal, bf16, seeded synthetic N(0,1) inputs), a shape with N >= 4096
and d = 128, where the forward and backward are compared with the tensor
peak.  Its inputs (4 x 268 MB) exceed the 129 MB L2, so no L2 flush is
needed between steps.  --workload gpt2_medium gives the GPT-2-medium
attention shape of the paper review's Figure 2 (B=64, H=16, N=1024, d=64).

Printed (rank 0, one JSON line): fwd+bwd TFLOP/s with FLOPs counted as
4*B*H*N^2*d for the forward and 2.5x that for the backward (recomputation
included), the time per step, the roofline of the dominant call, the end-to-end
figure through host buffers, the clocks seen while timing, and the fp64 oracle
timed on the host cores as a baseline.

With --gpus N > 1 (launched under torch.distributed.run) every rank processes
its own copy of the workload (attention heads are independent: weak scaling,
no data-path collective); the time is the max over ranks and the value sums
the work of all ranks.  --impl reference times the fp64 CPU oracle instead.
--workload picks another workload of io_aware_exact_10_gb300.workloads.
--once runs one untimed fa_fwd and fa_bwd of the workload (with --batch to
cut B): the driver of a small ncu capture.  --sweep times the sequence-length
sweep (N = 512 ... 32768, d = 64 and 128, H = 16, B*N = 65536, causal):
forward and forward+backward TFLOP/s per point, printed as one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
# head groups of the end-to-end leg's host-memory call (copies of one group
# overlap the kernels of the others)
E2E_CHUNKS = 8
# DRAM bytes (read + write) of one fa_bwd call, summed over its three
# launches, per workload, from one ncu capture of `bench.py --once`, with the
# hash of the sources it measured.  A capture on a smaller batch (capture_B)
# is scaled to the workload's B: the heads are independent, so the bytes
# grow in proportion.  The bench line reports a figure only while the code
# of the fa_bwd call (the backward kernels, their launch layer and shared
# helpers, comments aside) is the code the capture measured.
NCU_TRAFFIC = {
    # captured on the whole workload (B = 64)
    "gpt2_medium_B64_H16_N1024_d64": {
        "bytes": 2148664320.0, "capture_B": 64,
        "sources_sha256": "621cb8a3620df2df464ef675c08f6ee11d4aa7a01cbcc1109ba35293045b71cc"},
    # captured at B = 1, scaled by B (the heads are independent)
    "long_causal_B4_H32_N8192_d128": {
        "bytes": 1010353152.0, "capture_B": 1,
        "sources_sha256": "621cb8a3620df2df464ef675c08f6ee11d4aa7a01cbcc1109ba35293045b71cc"},
}
BWD_SOURCES = ("fa_api.cu", "fa_bwd.cu", "fa_bwd_d64.cu", "fa_kernels.h", "sm103_ptx.cuh")
DEFAULT_WORKLOAD = "long_causal"


def strip_comments(text: str) -> str:
    """C/C++ source without comments and blank lines (trailing spaces cut)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.split("\n") if line.strip())


def kernel_sources_sha256() -> str:
    """Hash of the fa_bwd call's sources with their comments stripped."""
    import hashlib
    csrc = os.path.join(ROOT, "io_aware_exact_10_gb300", "csrc")
    h = hashlib.sha256()
    for name in BWD_SOURCES:
        with open(os.path.join(csrc, name)) as f:
            h.update(name.encode() + b"\0" + strip_comments(f.read()).encode())
    return h.hexdigest()


def ncu_traffic(w):
    """The captured DRAM bytes of one fa_bwd call on workload w, scaled from
    the capture's batch to w.B, while the kernel sources still match the
    capture; else None."""
    t = NCU_TRAFFIC.get(w.name)
    if not t or kernel_sources_sha256() != t["sources_sha256"]:
        return None
    return t["bytes"] * w.B / t["capture_B"]


def load_peaks():
    try:
        with open(PEAKS_PATH) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return FALLBACK_PEAKS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def oracle_heads(w, flops: float, most: int) -> int:
    """Heads of workload w whose forward + backward add up to about `flops`
    (at least 1, at most `most`): the fp64 oracle runs at a few tens of
    GFLOP/s on the host cores, so 1e11 flop is a few seconds."""
    one = W_head_flops(w)
    return max(1, min(most, int(flops // one)))


def W_head_flops(w) -> float:
    """Forward + backward FLOPs of one query head of w."""
    return (w.fwd_flops() + w.bwd_flops()) / (w.B * w.H)


def cpu_oracle_sample(w, cpu_inputs, n_heads: int):
    """Time the fp64 oracle (fwd + bwd) on the first n_heads heads of the
    workload's inputs; returns (seconds, flops of the sample, threads)."""
    import oracle
    from io_aware_exact_10_gb300 import workloads as W
    oracle.build()
    G = w.H // w.kv_heads  # query heads per key/value head
    n_heads = max(G, n_heads // G * G)  # whole groups
    sub = W.Workload(w.name, 1, n_heads, w.N, w.d, causal=w.causal, seed=w.seed, N_k=w.N_k,
                     block_pattern=w.block_pattern)
    flat = lambda t, n: t.reshape(-1, t.shape[-2], w.d)[:n].double().numpy()
    q, k, v, dO = cpu_inputs
    qs, dOs = flat(q, n_heads), flat(dO, n_heads)
    ks, vs = flat(k, n_heads // G), flat(v, n_heads // G)
    bm = W.block_mask(w) if w.block_pattern else None
    t0 = time.perf_counter()
    oracle.attn_fwd(qs, ks, vs, w.scale, w.causal, block_mask=bm)
    oracle.attn_bwd(qs, ks, vs, dOs, w.scale, w.causal, block_mask=bm)
    dt = time.perf_counter() - t0
    return dt, sub.fwd_flops() + sub.bwd_flops(), oracle.num_threads()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args, w):
    """The fp64 oracle timed on the host cores (rank 0 only)."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    heads_per_step = oracle_heads(w, 1.0e11, 8)
    import oracle
    from io_aware_exact_10_gb300 import workloads as W
    oracle.build()
    q, k, v, dO = W.make_inputs(w)
    G = w.H // w.kv_heads  # query heads per key/value head
    heads_per_step = max(G, heads_per_step // G * G)  # whole groups
    flat = lambda t: t.reshape(-1, t.shape[-2], w.d).double().numpy()
    qs, ks, vs, dOs = flat(q), flat(k), flat(v), flat(dO)
    sub = W.Workload(w.name, 1, heads_per_step, w.N, w.d, causal=w.causal, N_k=w.N_k,
                     seed=w.seed, block_pattern=w.block_pattern)
    flops_step = sub.fwd_flops() + sub.bwd_flops()
    bm = W.block_mask(w) if w.block_pattern else None

    def step(i):
        lo = (i * heads_per_step) % (w.B * w.H)
        sl, sk = slice(lo, lo + heads_per_step), slice(lo // G, (lo + heads_per_step) // G)
        oracle.attn_fwd(qs[sl], ks[sk], vs[sk], w.scale, w.causal, block_mask=bm)
        oracle.attn_bwd(qs[sl], ks[sk], vs[sk], dOs[sl], w.scale, w.causal, block_mask=bm)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = flops_step * args.steps / dt / 1e12
    cores = oracle.num_threads()
    sample = (f"{heads_per_step} heads (of {w.B * w.H}) of {w.name} per step, fwd+bwd, "
              "fp64 C oracle with OpenMP")
    line = {
        "impl": "reference", "metric": "attention fwd+bwd TFLOP/s", "value": value,
        "unit": "TFLOP/s", "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1), bf16-rounded)",
        "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def block_mask_of(w):
    from io_aware_exact_10_gb300 import workloads as W
    return W.block_mask(w)


def config_of(w):
    c = {"workload": f"{w.name}, forward+backward", "B": w.B, "H": w.H, "N": w.N, "d": w.d,
         "causal": w.causal, "scale": w.scale,
         "l2": "inputs larger than L2 (4 x %.0f MB bf16), no flush" % (w.B * w.H * w.N * w.d * 2 / 1e6),
         "flops": "fwd 4*B*H*N^2*d (x1/2 causal); bwd 2.5x fwd"}
    if w.block_pattern:
        bm = block_mask_of(w)
        c["block_pattern"] = w.block_pattern
        c["blocks_kept"] = round(float(bm.mean()), 4)
        c["flops"] = ("fwd 4*B*H*d*pairs, pairs = (query, key) pairs inside the kept 128x128 "
                      "blocks (and the causal rule); bwd 2.5x fwd")
    if w.kv_heads != w.H or w.kv_len != w.N:
        if w.kv_heads != w.H:
            c["H_kv"] = w.kv_heads
        if w.kv_len != w.N:
            c["N_k"] = w.kv_len
            c["flops"] = ("fwd 4*B*H*d*pairs, pairs = N*N_k (causal: N*N_k - N^2/2, the last "
                          "query aligned with the last key); bwd 2.5x fwd")
        qb = w.B * w.H * w.N * w.d * 2 / 1e6
        kb = w.B * w.kv_heads * w.kv_len * w.d * 2 / 1e6
        c["l2"] = ("inputs larger than L2 together (Q, dO %.0f MB, K, V %.0f MB bf16 each: "
                   "%.0f MB), no flush" % (qb, kb, 2 * qb + 2 * kb))
    return c


def run_ours(args, w):
    import torch
    import io_aware_exact_10_gb300 as fa
    from io_aware_exact_10_gb300 import workloads as W
    import __graft_entry__

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    __graft_entry__.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()

    B, H, Hkv, N, Nk, d = w.B, w.H, w.kv_heads, w.N, w.kv_len, w.d
    cpu_inputs = W.make_inputs(w)
    q, k, v, dO = (t.to(dev) for t in cpu_inputs)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = fa.fa_bwd_workspace_size(B, H, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    causal = int(w.causal)

    # fa_fwd_ex / fa_bwd_ex with H_kv = H and N_k = N are fa_fwd / fa_bwd; a
    # block-sparse workload goes through fa_fwd_sparse / fa_bwd_sparse with its
    # mask resident on the device (a fixed part of the configuration)
    bmask = (torch.from_numpy(W.block_mask(w)).to(dev) if w.block_pattern else None)

    def fwd():
        if bmask is None:
            fa.fa_fwd_ex(q, k, v, o, lse, B, H, Hkv, N, Nk, d, w.scale, causal, stream)
        else:
            fa.fa_fwd_sparse(q, k, v, o, lse, B, H, Hkv, N, Nk, d, w.scale, causal, bmask, stream)

    def bwd():
        if bmask is None:
            fa.fa_bwd_ex(q, k, v, o, lse, dO, dq, dk, dv, B, H, Hkv, N, Nk, d, w.scale, causal, ws,
                         ws_bytes, stream)
        else:
            fa.fa_bwd_sparse(q, k, v, o, lse, dO, dq, dk, dv, B, H, Hkv, N, Nk, d, w.scale, causal,
                             bmask, ws, ws_bytes, stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    from io_aware_exact_10_gb300.replicas import max_over_ranks as _max_over_ranks

    def max_over_ranks(x: float) -> float:
        return _max_over_ranks(x, device=dev)

    ev = lambda: torch.cuda.Event(enable_timing=True)
    for _ in range(args.warmup):
        fwd()
        bwd()
    barrier()

    # ---- timed region: K steps, device-resident inputs
    clocks = ClockSampler(dev.index if world == 1 else local)
    if rank == 0:
        clocks.start()
    barrier()
    e0, e1 = ev(), ev()
    fwd_ev = [(ev(), ev()) for _ in range(args.steps)]
    bwd_ev = [(ev(), ev()) for _ in range(args.steps)]
    e0.record(stream)
    for i in range(args.steps):
        fwd_ev[i][0].record(stream)
        fwd()
        fwd_ev[i][1].record(stream)
        bwd_ev[i][0].record(stream)
        bwd()
        bwd_ev[i][1].record(stream)
    e1.record(stream)
    barrier()
    clk = clocks.stop() if rank == 0 else None
    ms_total = max_over_ranks(e0.elapsed_time(e1))
    fwd_ms = statistics.mean(a.elapsed_time(b) for a, b in fwd_ev)
    bwd_ms = statistics.mean(a.elapsed_time(b) for a, b in bwd_ev)
    st = fa.fa_last_device_error(stream)
    if st != fa.FA_OK:
        raise RuntimeError(f"device error after the timed region: {fa.fa_strerror(st)}")

    flops_step = w.fwd_flops() + w.bwd_flops()
    ms_step = ms_total / args.steps
    from io_aware_exact_10_gb300.replicas import whole_job_rate
    value = whole_job_rate(flops_step, world, ms_step * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    peak_sus = float(peaks.get("bf16_tflops_sustained", peak))
    bwd_tf = w.bwd_flops() / (bwd_ms * 1e-3) / 1e12
    fwd_tf = w.fwd_flops() / (fwd_ms * 1e-3) / 1e12

    # ---- end to end: pinned host inputs -> device -> fwd + bwd -> host outputs,
    # through the host-memory entry point, which pipelines the copies of each
    # head group against the kernels of the others (a block mask, resident on
    # the device like the dense path's, applies to every group).
    hq, hk, hv, hdO = (t.cpu().pin_memory() for t in (q, k, v, dO))
    ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    hdq = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    hdk, hdv = (torch.empty(k.shape, dtype=k.dtype).pin_memory() for _ in range(2))
    e2e_chunks = E2E_CHUNKS
    stage_bytes = fa.fa_fwd_bwd_host_device_bytes(B, H, Hkv, N, Nk, d, e2e_chunks)
    stage = torch.empty(stage_bytes, dtype=torch.uint8, device=dev)
    e2e_path = f"fa_fwd_bwd_host, {e2e_chunks} head groups"

    def e2e_step():
        fa.fa_fwd_bwd_host(hq, hk, hv, hdO, ho, hl, hdq, hdk, hdv, B, H, Hkv, N, Nk, d, w.scale,
                           causal, stage, stage_bytes, e2e_chunks, stream, block_mask=bmask)

    e2e_steps = max(3, min(args.steps, 20))
    e2e_step()
    barrier()
    a, b = ev(), ev()
    a.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    b.record(stream)
    barrier()
    e2e_ms = max_over_ranks(a.elapsed_time(b)) / e2e_steps
    h2d = sum(t.numel() * t.element_size() for t in (q, k, v, dO))
    d2h = sum(t.numel() * t.element_size() for t in (o, lse, dq, dk, dv))

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    # ---- CPU baseline: the oracle on a bounded sample of the same workload
    cpu_heads = int(os.environ.get("FA_BENCH_CPU_HEADS", oracle_heads(w, 4.0e11, 128)))
    cpu_s, cpu_flops, cores = cpu_oracle_sample(w, cpu_inputs, cpu_heads)

    line = {
        "metric": "attention fwd+bwd TFLOP/s",
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) fp32 rounded to bf16)",
        "config": config_of(w),
        "pct_of_peak": 100.0 * value / world / peak,
        "fwd": {"ms": fwd_ms, "tflops": fwd_tf, "pct_of_peak": 100 * fwd_tf / peak},
        "bwd": {"ms": bwd_ms, "tflops": bwd_tf, "pct_of_peak": 100 * bwd_tf / peak},
        "roofline": {
            "kernel": "fa_bwd call (D preprocess + backward kernel + dQ convert), timed with "
                      "CUDA events per launch; its FLOPs are the backward's 5 N^2 d contractions",
            "bound": "tensor",
            "achieved": bwd_tf,
            "peak": peak,
            "unit": "TFLOP/s",
            "frac": bwd_tf / peak,
            "frac_sustained": bwd_tf / peak_sus,
            "peak_source": f"{peak_src} bf16 burst ({PEAKS_PATH if peak_src == 'measured' else 'recipe fallback'})",
            "traffic": ncu_traffic(w),
        },
        "e2e": {"value": world * flops_step / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "path": e2e_path},
        "gpu_launches": 4 * args.steps,
        "bars": bars_of(w, fwd_tf, bwd_tf, peak),
        "clocks": clk,
        "cpu_baseline": {"value": cpu_flops / cpu_s / 1e12, "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"first {cpu_heads} of {w.B * w.H} heads of {w.name}, "
                                   f"fwd+bwd in fp64 ({cpu_s:.1f} s)"},
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def bars_of(w, fwd_tf: float, bwd_tf: float, peak: float):
    """The throughput bars, stated for N >= 4096 and d = 128: the forward at
    >= 60 % and the backward at >= 40 % of the dense bf16 tensor peak (None
    for other shapes)."""
    if w.d != 128 or w.N < 4096:
        return None
    return {"fwd_min_pct": 60.0, "bwd_min_pct": 40.0,
            "fwd_pct": 100.0 * fwd_tf / peak, "bwd_pct": 100.0 * bwd_tf / peak,
            "fwd_met": fwd_tf >= 0.6 * peak, "bwd_met": bwd_tf >= 0.4 * peak}


def run_once(args, w):
    """One untimed fa_fwd and fa_bwd of workload w (B cut to --batch when
    given), drawn on the device: the driver of a small ncu capture."""
    import dataclasses
    import torch
    import io_aware_exact_10_gb300 as fa
    from io_aware_exact_10_gb300 import workloads as W
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    if args.batch:
        w = dataclasses.replace(w, B=args.batch)
    B, H, Hkv, N, Nk, d = w.B, w.H, w.kv_heads, w.N, w.kv_len, w.d
    q, k, v, dO = W.make_inputs_on_device(w, dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    wsb = fa.fa_bwd_workspace_size(B, H, N, d)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    fa.fa_fwd_ex(q, k, v, o, lse, B, H, Hkv, N, Nk, d, w.scale, int(w.causal), stream)
    fa.fa_bwd_ex(q, k, v, o, lse, dO, dq, dk, dv, B, H, Hkv, N, Nk, d, w.scale, int(w.causal),
                 ws, wsb, stream)
    if fa.fa_last_device_error(stream) != fa.FA_OK:
        raise RuntimeError("device error")
    print(f"{w.name} B={B}: one fa_fwd, one fa_bwd", flush=True)


def sweep_bytes(N: int, d: int, BH: int, causal: bool) -> dict:
    """DRAM bytes of one sweep point's forward and main backward kernel: the
    algorithmic minimum (every input read once, every output written once;
    for the backward the fp32 dQ accumulator read and written once) and the
    tiled model, i.e. what the kernels stream if L2 kept nothing between
    CTAs.  Forward: a CTA holds query tiles 2p, 2p+1 and streams K, V tiles
    0 .. nu_p - 1 (nu_p = min(2p + 2, nkv) when causal).  Backward: a CTA
    holds key tile kt, reads its K, V once, writes dK, dV once, and per
    visited query tile (from kt on when causal) streams Q, dO, 1 KB of row
    statistics and a read and write of the 128 x d fp32 dQ rows."""
    tile = 128 * d * 2                      # bf16 128-row tile
    nt = -(-N // 128)
    npairs = -(-nt // 2)
    fwd_min = BH * (8 * N * d + 4 * N)
    streamed = sum(min(2 * p + 2, nt) if causal else nt for p in range(npairs))
    fwd_model = BH * (4 * N * d + 4 * N + streamed * 2 * tile)
    bwd_min = BH * (8 * N * d + 8 * N + 4 * N * d + 8 * N * d)
    visits = sum(nt - kt if causal else nt for kt in range(nt))
    bwd_model = BH * (nt * 4 * tile + visits * (2 * tile + 1024 + 2 * 128 * d * 4))
    return {"fwd_min": fwd_min, "fwd_model": fwd_model, "bwd_kernel_min": bwd_min,
            "bwd_kernel_model": bwd_model}


def sweep_cpu_baseline(N: int, d: int, causal: bool):
    """The sweep's CPU baseline: the fp64 oracle's time for one head's forward
    + backward at a sweep point, measured on a whole head up to N = 4096, else
    extrapolated by FLOPs from 64 evenly spaced forward rows.  Returns (ms,
    how, threads)."""
    import numpy as np
    import oracle
    from io_aware_exact_10_gb300 import workloads as W
    oracle.build()
    w1 = W.Workload(f"oracle_N{N}_d{d}", 1, 1, N, d, causal=causal)
    q, k, v, dO = (t.reshape(N, d).double().numpy() for t in W.make_inputs(w1))
    head_flops = w1.fwd_flops() + w1.bwd_flops()
    if N <= 4096:
        t0 = time.perf_counter()
        oracle.attn_fwd(q, k, v, w1.scale, causal)
        oracle.attn_bwd(q, k, v, dO, w1.scale, causal)
        return 1e3 * (time.perf_counter() - t0), "one head, forward + backward", oracle.num_threads()
    rows = np.linspace(0, N - 1, 64).astype(np.int64)
    t0 = time.perf_counter()
    oracle.attn_fwd_rows(q, k, v, rows, w1.scale, causal)
    dt = time.perf_counter() - t0
    keys = (rows + 1) if causal else np.full_like(rows, N)
    sample_flops = float((4 * d * keys).sum())
    return (1e3 * dt * head_flops / sample_flops,
            "extrapolated by FLOPs from 64 forward rows of one head", oracle.num_threads())


def run_sweep_once(args):
    """One fa_fwd and one fa_bwd per sweep point, untimed: the driver of the
    per-point ncu capture (DRAM bytes and tensor-pipe activity per kernel)."""
    import torch
    import io_aware_exact_10_gb300 as fa
    from io_aware_exact_10_gb300 import workloads as W
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    for d in W.SWEEP_D:
        for N in W.SWEEP_N:
            w = W.sweep(N, d)
            B, H = w.B, w.H
            q, k, v, dO = W.make_inputs_on_device(w, dev)
            o = torch.empty_like(q)
            lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
            wsb = fa.fa_bwd_workspace_size(B, H, N, d)
            ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
            fa.fa_fwd(q, k, v, o, lse, B, H, N, d, w.scale, 1, stream)
            fa.fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, w.scale, 1, ws, wsb, stream)
            if fa.fa_last_device_error(stream) != fa.FA_OK:
                raise RuntimeError("device error during the sweep")
            print(f"N={N} d={d} B={B} H={H}: one fa_fwd, one fa_bwd", flush=True)
            del q, k, v, dO, o, lse, dq, dk, dv, ws


def run_sweep(args):
    """Forward and forward+backward TFLOP/s per sweep point (one JSON line),
    with each point's byte model and the oracle's time for one head."""
    import torch
    import io_aware_exact_10_gb300 as fa
    from io_aware_exact_10_gb300 import workloads as W
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    peaks, _ = load_peaks()
    peak = float(peaks["bf16_tflops"])
    points = []
    clocks = ClockSampler(0)
    clocks.start()
    for d in W.SWEEP_D:
        for N in W.SWEEP_N:
            w = W.sweep(N, d)
            B, H = w.B, w.H
            q, k, v, dO = W.make_inputs_on_device(w, dev)
            o = torch.empty_like(q)
            lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
            wsb = fa.fa_bwd_workspace_size(B, H, N, d)
            ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
            f = lambda: fa.fa_fwd(q, k, v, o, lse, B, H, N, d, w.scale, 1, stream)
            b = lambda: fa.fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, w.scale, 1, ws,
                                  wsb, stream)
            res = {}
            for name, fn, fl in (("fwd", f, w.fwd_flops()),
                                 ("fwd_bwd", lambda: (f(), b()), w.fwd_flops() + w.bwd_flops())):
                for _ in range(args.warmup):
                    fn()
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(args.steps):
                    fn()
                e1.record(stream)
                torch.cuda.synchronize()
                ms = e0.elapsed_time(e1) / args.steps
                res[name] = {"ms": ms, "tflops": fl / ms / 1e9, "pct_of_peak": 100 * fl / ms / 1e9 / peak}
            if fa.fa_last_device_error(stream) != fa.FA_OK:
                raise RuntimeError("device error during the sweep")
            points.append({"N": N, "d": d, "B": B, "H": H, **res,
                           "bytes": sweep_bytes(N, d, B * H, True)})
            del q, k, v, dO, o, lse, dq, dk, dv, ws
    clk = clocks.stop()
    # the CPU baseline (the oracle on the host cores), after the GPU timing
    for pt in points:
        ms, how, threads = sweep_cpu_baseline(pt["N"], pt["d"], True)
        pt["cpu_baseline"] = {"kind": "oracle", "ms_per_head": ms, "sample": how,
                              "cores": threads, "ms_all_heads": ms * pt["B"] * pt["H"]}
    print(json.dumps({"metric": "attention fwd / fwd+bwd TFLOP/s vs N (causal, H=16, B*N=65536)",
                      "unit": "TFLOP/s", "peak": peak, "steps": args.steps,
                      "warmup": args.warmup, "data": "synthetic (seeded on the device)",
                      "clocks": clk, "sweep": points}), flush=True)


TILE_LAYOUTS = ((256, 128), (256, 64), (128, 128), (128, 64))  # (Br, Bc)


def tile_layout_call(fa, q, k, v, o, lse, w, br, bc, causal, stream):
    """One forward of workload w's shape with Br query rows per CTA and Bc
    keys per K/V tile.  Br = 256 is the normal layout (a CTA holds two
    128-row query tiles of a head).  Br = 128 views every 128-row query tile
    as its own query head (N_q = 128, H N / 128 query heads on the H
    key/value heads): each CTA holds one tile, with the same arithmetic per
    row (non-causal only, since causal masking aligns on each head's last
    row).  Bc = 64 is fa_fwd_tiled's 64-key tile."""
    B, H, N, d = w.B, w.H, w.N, w.d
    if br == 256:
        return fa.fa_fwd_tiled(q, k, v, o, lse, B, H, H, N, N, d, w.scale, causal, bc, stream)
    nt = N // 128
    return fa.fa_fwd_tiled(q, k, v, o, lse, B, H * nt, H, 128, N, d, w.scale, 0, bc, stream)


def run_tile_sweep(args):
    """Forward time against the two tile sizes of the paper review's Fig. 2
    (middle panel: runtime against block size): query rows per CTA (Br = 128
    or 256) and keys per K/V tile (Bc = 64 or 128), non-causal, plus the Bc
    axis causal at Br = 256.  Layouts with the same Bc give o and lse bit for
    bit equal; the two Bc agree to rounding.  Prints one JSON line: forward
    time and TFLOP/s per (N, d, Br, Bc), with the K/V bytes a no-reuse model
    says each layout streams (a model, not a counter)."""
    import torch
    import io_aware_exact_10_gb300 as fa
    from io_aware_exact_10_gb300 import workloads as W
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    peaks, _ = load_peaks()
    peak = float(peaks["bf16_tflops"])
    points = []
    max_dev = {"o": 0.0, "lse": 0.0}
    for d in W.SWEEP_D:
        for N in (1024, 4096, 16384):
            for causal in (False, True):
                w = W.sweep(N, d, causal=causal)
                B, H = w.B, w.H
                q, k, v = W.make_inputs_on_device(w, dev, with_grad=False)
                res, outs = {}, {}
                layouts = TILE_LAYOUTS if not causal else ((256, 128), (256, 64))
                for br, bc in layouts:
                    o = torch.empty_like(q)
                    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
                    f = lambda: tile_layout_call(fa, q, k, v, o, lse, w, br, bc, int(causal), stream)
                    for _ in range(args.warmup):
                        f()
                    torch.cuda.synchronize()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    for _ in range(args.steps):
                        f()
                    e1.record(stream)
                    torch.cuda.synchronize()
                    ms = e0.elapsed_time(e1) / args.steps
                    tf = w.fwd_flops() / ms / 1e9
                    # K and V bytes the CTAs ask for from L2 or DRAM if nothing
                    # were reused between CTAs (each streams its head's K and V
                    # once, or up to its last visible tile when causal)
                    kv_model = B * H * 2 * N * d * 2 * (N // br if br <= N else 1)
                    if causal:
                        kv_model = kv_model // 2
                    res[f"br{br}_bc{bc}"] = {"ms": ms, "tflops": tf, "pct_of_peak": 100 * tf / peak,
                                             "kv_model_gb": kv_model / 1e9}
                    outs[(br, bc)] = (o, lse)
                    del o, lse, f
                if fa.fa_last_device_error(stream) != fa.FA_OK:
                    raise RuntimeError("device error during the tile sweep")
                for bc in (128, 64):
                    if (128, bc) in outs and not (torch.equal(outs[(256, bc)][0], outs[(128, bc)][0])
                                                  and torch.equal(outs[(256, bc)][1], outs[(128, bc)][1])):
                        raise RuntimeError(f"Br = 128 and Br = 256 disagree at N={N}, d={d}, Bc={bc}")
                do = (outs[(256, 64)][0].float() - outs[(256, 128)][0].float()).abs().max().item()
                dl = (outs[(256, 64)][1] - outs[(256, 128)][1]).abs().max().item()
                if do > 2e-2 or dl > 1e-3:
                    raise RuntimeError(f"Bc = 64 and Bc = 128 differ beyond rounding at N={N}, d={d}")
                max_dev["o"], max_dev["lse"] = max(max_dev["o"], do), max(max_dev["lse"], dl)
                points.append({"N": N, "d": d, "B": B, "H": H, "causal": causal, **res})
                del q, k, v, outs
    print(json.dumps({"metric": "attention fwd TFLOP/s vs query rows per CTA (Br) and keys per "
                                "K/V tile (Bc)",
                      "unit": "TFLOP/s", "peak": peak, "steps": args.steps,
                      "warmup": args.warmup, "same_bc_bitwise_equal": True,
                      "bc64_vs_bc128_max_abs": max_dev, "points": points}),
          flush=True)


def run_tile_once(args):
    """One untimed forward per tile layout at N = 4096, d = 128 (B = 16,
    H = 16, non-causal): the driver of the per-layout ncu capture."""
    import torch
    import io_aware_exact_10_gb300 as fa
    from io_aware_exact_10_gb300 import workloads as W
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    w = W.sweep(4096, 128, causal=False)
    q, k, v = W.make_inputs_on_device(w, dev, with_grad=False)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    for br, bc in TILE_LAYOUTS:
        tile_layout_call(fa, q, k, v, o, lse, w, br, bc, 0, stream)
        print(f"Br={br} Bc={bc}: one forward", flush=True)
    if fa.fa_last_device_error(stream) != fa.FA_OK:
        raise RuntimeError("device error")


def run_compare(args, w):
    """Standard attention against this library on one workload (the
    comparison of the paper review's Fig. 2): a forward+backward step of
    softmax(scale Q K^T) V computed the standard way, with S and P written to
    and read back from device memory (torch bf16 matmul, softmax and
    autograd: library kernels, the comparator), and the same step through
    fa_fwd/fa_bwd.  Prints one JSON line with each side's step time, FLOP
    rate and peak device memory.  HBM bytes come from an ncu launch list of
    this same command (the kernels of the two sides have distinct names)."""
    import torch
    import io_aware_exact_10_gb300 as fa
    from io_aware_exact_10_gb300 import workloads as W
    import __graft_entry__

    if w.kv_heads != w.H or w.kv_len != w.N or w.block_pattern:
        raise SystemExit("--compare takes a dense multi-head workload with N_k = N")
    torch.cuda.set_device(0)
    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    B, H, N, d = w.B, w.H, w.N, w.d
    q, k, v, dO = W.make_inputs_on_device(w, dev)
    causal = int(w.causal)
    ev = lambda: torch.cuda.Event(enable_timing=True)

    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = fa.fa_bwd_workspace_size(B, H, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    def ours_step():
        fa.fa_fwd(q, k, v, o, lse, B, H, N, d, w.scale, causal, stream)
        fa.fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, w.scale, causal, ws, ws_bytes,
                  stream)

    cmask = (torch.ones(N, N, dtype=torch.bool, device=dev).triu(1) if w.causal else None)

    def standard_step():
        qq, kk, vv = (t.detach().requires_grad_(True) for t in (q, k, v))
        s_ = torch.matmul(qq, kk.transpose(-1, -2)) * w.scale
        if cmask is not None:
            s_ = s_.masked_fill(cmask, float("-inf"))
        p_ = torch.softmax(s_, dim=-1)
        out = torch.matmul(p_, vv)
        out.backward(dO)
        return qq.grad, kk.grad, vv.grad

    def timed(step, reps):
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        base = torch.cuda.memory_allocated()
        torch.cuda.reset_peak_memory_stats()
        a, b = ev(), ev()
        a.record(stream)
        for _ in range(reps):
            step()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps, (torch.cuda.max_memory_allocated() - base) / 1e9

    reps = max(1, min(args.steps, 20))
    ours_ms, ours_peak = timed(ours_step, reps)
    std_ms, std_mem = timed(standard_step, reps)
    # device memory a step needs beyond its inputs: for this library the
    # outputs and the workspace, allocated once above (plus any peak during
    # the step); for standard attention the peak of the step, which holds S,
    # P, their gradients and the outputs
    ours_mem = ours_peak + sum(t.numel() * t.element_size() for t in (o, lse, dq, dk, dv, ws)) / 1e9
    if fa.fa_last_device_error(stream) != fa.FA_OK:
        raise RuntimeError("device error in the comparison")
    half = 0.5 if w.causal else 1.0
    nn = B * H * N * N * d * half
    # algorithmic FLOPs of each method: standard fwd 2 contractions, bwd 4;
    # this library recomputes S and P in the backward (5 contractions)
    std_flops, ours_flops = 2 * nn * 6, 2 * nn * 7
    line = {
        "mode": "compare", "workload": w.name, "steps": reps, "warmup": args.warmup,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1), drawn on the device)",
        "standard": {"impl": "torch bf16 matmul + softmax + matmul, autograd backward "
                             "(S and P materialised)",
                     "ms": std_ms, "gflop": std_flops / 1e9,
                     "tflops": std_flops / (std_ms * 1e-3) / 1e12, "extra_mem_gb": std_mem},
        "ours": {"impl": "fa_fwd + fa_bwd", "ms": ours_ms, "gflop": ours_flops / 1e9,
                 "tflops": ours_flops / (ours_ms * 1e-3) / 1e12, "extra_mem_gb": ours_mem},
        "speedup": std_ms / ours_ms,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--once", action="store_true",
                    help="one untimed fa_fwd and fa_bwd of the workload (ncu capture driver)")
    ap.add_argument("--batch", type=int, default=0,
                    help="with --once: the workload's B cut to this value")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--tile-sweep", action="store_true",
                    help="forward time against query rows per CTA (128 or 256) and keys per "
                         "K/V tile (64 or 128)")
    ap.add_argument("--tile-once", action="store_true",
                    help="one untimed forward per tile layout at N=4096, d=128 (ncu capture driver)")
    ap.add_argument("--sweep-once", action="store_true",
                    help="one untimed fa_fwd and fa_bwd per sweep point (ncu capture driver)")
    ap.add_argument("--compare", action="store_true",
                    help="standard attention (S, P in device memory) against this library")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    from io_aware_exact_10_gb300 import workloads as W
    if args.sweep_once:
        run_sweep_once(args)
        return
    if args.tile_sweep:
        run_tile_sweep(args)
        return
    if args.tile_once:
        run_tile_once(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    w = W.WORKLOADS[args.workload]
    if args.once:
        run_once(args, w)
        return
    if args.compare:
        run_compare(args, w)
        return
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()

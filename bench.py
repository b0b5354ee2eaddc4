#!/usr/bin/env python
"""Benchmark of the paged decode-attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--kv bf16|fp8] [--window W]

A step is one pass of the whole hot path over one batch: kv_append of the
step's new K/V, then paged decode attention (plus its LSE merge launch) over
every sequence.  The default workload is the Llama-3-8B-shaped GQA continuous
batch (64 sequences, contexts uniform in [128, 8192], 32 query / 8 KV heads,
head_dim 128, block 16), whose KV cache (~1.03 GB) is 8x the 129 MB L2, so
no flush is needed between steps.

Printed (rank 0, one JSON line): effective HBM GB/s of the step, where bytes =
resident KV + q + out, with microseconds per step, the fraction of the
measured HBM peak, the roofline of the attention launch, the end-to-end
figure through the public API with host buffers, the oracle as a CPU
baseline, and the SM clocks sampled while the steps ran.  The headline step
time is the CUDA-graph replay of the step (the three launches captured
once); the eagerly launched step is reported under "eager".

--kv fp8 times the same step over an 8-bit (e4m3) cache with per-KV-head
scales (the quantising append, then attention); --window W times
sliding-window attention.  Their bytes count what the step must move: the
e4m3 cache is one byte per element, and a window reads at most W + q_len - 1
tokens per sequence.  The default line (bf16, no window) is the headline.

Under torchrun (N > 1) every rank runs an independent replica of the
workload on its own GPU (no collective on the data path); the timing is the
maximum over ranks and `value` counts the bytes of all ranks.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attn effective HBM GB/s (% of GB300 peak) and μs per decode step"
UNIT = "GB/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "attn_traffic.json")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama3_8b_gqa")
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16")
    ap.add_argument("--window", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-soak", action="store_true",
                    help="skip the 1 s untimed load before the timed steps (profiling runs)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def tensor_peak():
    """Dense bf16 tensor peak: the sustained figure (the bench times long runs of steps)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["bf16_tflops_sustained"])
        return v, "measured (MEASURED_PEAKS.json bf16_tflops_sustained: cuBLAS bf16 GEMM)"
    except Exception:
        return 1700.0, "fallback (no MEASURED_PEAKS.json)"


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs: copy, read+write bytes)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (no MEASURED_PEAKS.json)"


def kernel_source_hash():
    """Hash of the attention kernel's sources, line comments and blank lines
    left out (a comment edit does not change the kernel the counters came from)."""
    h = hashlib.sha256()
    for name in ("decode_attn.cuh", "decode_attn.cu", "decode_attn_fp8.cu", "ptx.cuh",
                 "tcgen05.cuh", "pkv_internal.h"):
        with open(os.path.join(ROOT, "paged_kv_cache_256_gb300", "csrc", name)) as f:
            for line in f:
                code = line.split("//", 1)[0].strip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def profiled_traffic(key):
    """DRAM bytes per attention launch from the committed ncu summary, if still current."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("kernel_source_sha") != kernel_source_hash():
        return None
    return rec.get("bytes_per_launch", {}).get(key)


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while work runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    rows.append(dict(sm=float(p[1]), smax=float(p[2]), power=float(p[3]),
                                     hw=p[5], hwt=p[6], swt=p[7], cap=p[8]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("cap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["smax"] for r in rows),
                "power_w_max": max(r["power"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


def max_over_ranks(values, device=None):
    """Element-wise maximum of a list of floats over all ranks (identity at N = 1).

    Uses the process group's own backend: NCCL on GPU tensors for the bench,
    gloo on CPU tensors in the multi-process CPU tests.
    """
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def whole_job_gbps(bytes_per_rank, ms_per_step, world):
    """Whole-job throughput of N independent replicas timed by the slowest rank."""
    return world * bytes_per_rank / (ms_per_step * 1e-3) / 1e9


# ---------------------------------------------------------------------------
def step_bytes(wl, elem_bytes=2, window=0):
    """Algorithmic bytes of one decode step: the KV the step must read + q + out (bf16).

    Without a window that is every resident token; with one, a sequence needs
    only its last W + q_len - 1 tokens (the union of its rows' windows).
    """
    import numpy as np
    from paged_kv_cache_256_gb300 import pkv_kv_bytes
    ctx = wl.context_lens.astype(np.int64)
    if window > 0:
        ctx = np.minimum(ctx, window + wl.q_len - 1)
    kv = pkv_kv_bytes(1, wl.n_kv, wl.head_dim, elem_bytes, int(ctx.sum()))
    q = wl.q.nbytes
    return kv + q + q, kv


def step_flops(wl, window=0):
    """Algorithmic FLOPs of the attention: 4 * head_dim per (query row, visible key)
    (2 for q.k, 2 for p * v), summed over sequences, query heads and new tokens."""
    import numpy as np
    ctx = wl.context_lens.astype(np.int64)[:, None]
    pos = ctx - wl.q_len + np.arange(wl.q_len, dtype=np.int64)[None, :]
    hi = np.minimum(pos + 1, ctx)
    lo = np.maximum(pos - window + 1, 0) if window > 0 else np.zeros_like(pos)
    visible = np.where(pos >= 0, np.maximum(hi - lo, 0), 0)
    return int(4 * wl.head_dim * wl.n_q * visible.sum())


def cpu_baseline(wl, budget_s=12.0):
    """The oracle, as it stands, on the host cores: GB/s over a bounded sample."""
    import numpy as np
    import oracle
    orc = oracle.get()
    kw = dict(n_q=wl.n_q, n_kv=wl.n_kv, head_dim=wl.head_dim, block_size=wl.block_size,
              scale=wl.scale)
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    orc.kv_append(wl.k_new, wl.v_new, wl.slot_mapping, kc, vc, block_size=wl.block_size)
    total, kv = step_bytes(wl)
    reps, t_used = 0, 0.0
    while t_used < budget_s and reps < 50:
        t0 = time.perf_counter()
        orc.paged_attn(wl.q, kc, vc, wl.block_tables, wl.context_lens, **kw)
        t_used += time.perf_counter() - t0
        reps += 1
    return {"value": round(total * reps / t_used / 1e9, 3), "unit": UNIT,
            "cores": orc.num_threads(), "kind": "oracle",
            "sample": f"whole {wl.name} step (attention over {wl.resident_tokens()} resident "
                      f"tokens), {reps} repetitions, fp64, {t_used:.1f} s"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    from paged_kv_cache_256_gb300.workloads import make_workload
    wl = make_workload(args.workload)
    orc = oracle.get()
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    kw = dict(n_q=wl.n_q, n_kv=wl.n_kv, head_dim=wl.head_dim, block_size=wl.block_size,
              scale=wl.scale)
    # Size each step's sample so that warm-up + timed steps stay within ~2 minutes.
    t0 = time.perf_counter()
    orc.paged_attn(wl.q[:4], kc, vc, wl.block_tables[:4], wl.context_lens[:4], **kw)
    per_seq = (time.perf_counter() - t0) / 4
    budget = 120.0 / max(1, args.steps + args.warmup)
    nseq = int(max(1, min(wl.num_seqs, budget / max(per_seq, 1e-6))))
    sub_ctx = wl.context_lens[:nseq]
    kv = 2 * wl.n_kv * wl.head_dim * 2 * int(sub_ctx.astype(np.int64).sum())
    qb = wl.q[:nseq].nbytes
    total = kv + 2 * qb

    def step():
        orc.kv_append(wl.k_new[: nseq * wl.q_len], wl.v_new[: nseq * wl.q_len],
                      wl.slot_mapping[: nseq * wl.q_len], kc, vc, block_size=wl.block_size)
        orc.paged_attn(wl.q[:nseq], kc, vc, wl.block_tables[:nseq], sub_ctx, **kw)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    value = total / dt / 1e9
    sample = (f"first {nseq} of {wl.num_seqs} sequences of {wl.name} per step "
              f"({int(sub_ctx.sum())} resident tokens), kv_append + attention, fp64")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "sample_seqs": nseq},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": orc.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
def run_ours(args):
    import numpy as np
    import torch

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)

    import paged_kv_cache_256_gb300 as pkv
    from paged_kv_cache_256_gb300.device import fp8_to_device, to_device
    from paged_kv_cache_256_gb300.workloads import fp8_cache_for, make_workload

    wl = make_workload(args.workload)
    kv8 = args.kv == "fp8"
    total_bytes, kv_bytes = step_bytes(wl, 1 if kv8 else 2, args.window)
    dw = to_device(wl, device)
    d8 = fp8_to_device(fp8_cache_for(wl), device) if kv8 else None
    if kv8:  # the bf16 caches are not used by this step
        dw.k_cache = dw.v_cache = None
        torch.cuda.empty_cache()
    ws = pkv.alloc_workspace(wl.num_seqs, wl.q_len, wl.n_q, wl.n_kv, wl.head_dim,
                             wl.block_size, device=device)
    out = torch.empty(tuple(dw.q.shape), dtype=torch.bfloat16, device=device)
    stream = torch.cuda.current_stream(device)
    grid = torch.cuda.get_device_properties(device).multi_processor_count
    launches_per_step = 3 if grid > 1 else 2

    def append(s):
        if kv8:
            pkv.pkv_kv_append_fp8(dw.k_new, dw.v_new, dw.slot_mapping, d8.kv_cache, d8.k_scale,
                                  d8.v_scale, stream=s)
        else:
            pkv.pkv_kv_append(dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache,
                              stream=s)

    def attend(s):
        if kv8:
            pkv.pkv_paged_decode_attn_ex(dw.q, d8.kv_cache, None, dw.block_tables,
                                         dw.context_lens, wl.scale, out, ws, stream=s,
                                         window=args.window, k_scale=d8.k_scale,
                                         v_scale=d8.v_scale)
        elif args.window:
            pkv.pkv_paged_decode_attn_ex(dw.q, dw.k_cache, dw.v_cache, dw.block_tables,
                                         dw.context_lens, wl.scale, out, ws, stream=s,
                                         window=args.window)
        else:
            pkv.pkv_paged_decode_attn(dw.q, dw.k_cache, dw.v_cache, dw.block_tables,
                                      dw.context_lens, wl.scale, out, ws, stream=s)

    def step():
        append(stream)
        attend(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(device)
    st = pkv.pkv_check_error(ws)
    if st != pkv.PKV_OK:
        raise RuntimeError(f"warm-up reported {pkv.pkv_status_string(st)}")

    K = args.steps
    ev_step = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    ev_attn = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    clocks = ClockSampler(local)
    clocks.start()
    # Let the sampler see the GPU under load before and through the timed steps.
    t_soak = time.perf_counter()
    while not args.no_soak and time.perf_counter() - t_soak < 1.0:
        for _ in range(50):
            step()
        torch.cuda.synchronize(device)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    ev_step[0].record(stream)
    for k in range(K):
        append(stream)
        ev_attn[k].record(stream)
        attend(stream)
        ev_step[k + 1].record(stream)
    torch.cuda.synchronize(device)
    if world > 1:
        torch.distributed.barrier()
    st = pkv.pkv_check_error(ws)
    if st != pkv.PKV_OK:
        raise RuntimeError(f"timed steps reported {pkv.pkv_status_string(st)}")

    total_ms = ev_step[0].elapsed_time(ev_step[K])
    attn_ms = [ev_attn[k].elapsed_time(ev_step[k + 1]) for k in range(K)]
    step_ms = [ev_step[k].elapsed_time(ev_step[k + 1]) for k in range(K)]
    ms_per_step, attn_mean = max_over_ranks([total_ms / K, sum(attn_ms) / K], device)

    # ---- end to end through the public API, host buffers, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        host = {
            "q": torch.from_numpy(wl.q.view(np.int16)).pin_memory(),
            "k_new": torch.from_numpy(wl.k_new.view(np.int16)).pin_memory(),
            "v_new": torch.from_numpy(wl.v_new.view(np.int16)).pin_memory(),
            "slot_mapping": torch.from_numpy(wl.slot_mapping).pin_memory(),
            "block_tables": torch.from_numpy(wl.block_tables).pin_memory(),
            "context_lens": torch.from_numpy(wl.context_lens).pin_memory(),
        }
        out_host = torch.empty(tuple(out.shape), dtype=torch.int16).pin_memory()
        dev = {
            "q": dw.q.view(torch.int16), "k_new": dw.k_new.view(torch.int16),
            "v_new": dw.v_new.view(torch.int16), "slot_mapping": dw.slot_mapping,
            "block_tables": dw.block_tables, "context_lens": dw.context_lens,
        }
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out_host.numel() * out_host.element_size()

        def e2e_step():
            for k2, t in host.items():
                dev[k2].copy_(t, non_blocking=True)
            step()
            out_host.copy_(out.view(torch.int16), non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        e0.record(stream)
        for _ in range(K):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(device)
        e2e_ms = max_over_ranks([e0.elapsed_time(e1) / K], device)[0]
        e2e = {"value": round(whole_job_gbps(total_bytes, e2e_ms, world), 2), "unit": UNIT,
               "us_per_step": round(e2e_ms * 1e3, 2), "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h}

    # ---- the same step replayed from a CUDA graph (no host launch cost)
    graph = None
    if not args.no_graph:
        gs = torch.cuda.Stream(device)
        gs.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gs):
            append(gs)
            attend(gs)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize(device)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        g0.record(stream)
        for _ in range(K):
            g.replay()
        g1.record(stream)
        torch.cuda.synchronize(device)
        g_ms = max_over_ranks([g0.elapsed_time(g1) / K], device)[0]
        st = pkv.pkv_check_error(ws)
        if st != pkv.PKV_OK:
            raise RuntimeError(f"graph replay reported {pkv.pkv_status_string(st)}")
        graph = {"value": round(whole_job_gbps(total_bytes, g_ms, world), 2), "unit": UNIT,
                 "us_per_step": round(g_ms * 1e3, 2)}

    clk = clocks.stop()

    # The headline step is the CUDA-graph replay (how a decode loop is served);
    # the eagerly launched step is reported beside it.
    eager = {"value": round(whole_job_gbps(total_bytes, ms_per_step, world), 2), "unit": UNIT,
             "us_per_step": round(ms_per_step * 1e3, 2)}
    step_source = "eager launches"
    if graph is not None:
        ms_per_step = graph["us_per_step"] / 1e3
        step_source = "CUDA-graph replay of the step"
    peak, peak_src = hbm_peak()
    value = whole_job_gbps(total_bytes, ms_per_step, world)
    achieved = total_bytes / (attn_mean * 1e-3) / 1e9
    flops = step_flops(wl, args.window)
    prefill = wl.group * wl.q_len > 128  # many query rows per KV head: compute-bound
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "us_per_step": round(ms_per_step * 1e3, 2),
        "pct_of_peak": round(100.0 * value / world / peak, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 KV (f16 products, fp32 softmax)" if kv8 else "bf16",
        "data": "synthetic",
        "config": {
            "workload": wl.name, "num_seqs": wl.num_seqs, "n_q": wl.n_q, "n_kv": wl.n_kv,
            "head_dim": wl.head_dim, "block_size": wl.block_size, "q_len": wl.q_len,
            "resident_tokens": wl.resident_tokens(), "bytes_per_step": total_bytes,
            "kv_bytes": kv_bytes, "kv_dtype": args.kv, "window": args.window,
            "l2": f"no flush: resident KV {kv_bytes / L2_BYTES:.1f}x the 129 MB L2",
            "step": ("kv_append_fp8" if kv8 else "kv_append") +
                    " + paged_decode_attn (+ lse_merge)",
            "timed_as": step_source,
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
            "step_us_p10_p50_p90": [round(1e3 * x, 2) for x in
                                     statistics.quantiles(step_ms, n=10)[::4]] if K >= 10 else None,
        },
        "roofline": {
            "kernel": "paged_decode_attn (attention + merge launches of one call)",
            "bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "flops_per_launch": flops,
            "traffic": profiled_traffic(wl.name + ("/fp8" if kv8 else "") +
                                        (f"/w{args.window}" if args.window else "")),
            "peak_source": peak_src, "attn_us": round(attn_mean * 1e3, 2),
            "algorithmic_bytes_per_launch": total_bytes,
        },
        "e2e": e2e,
        "eager": eager,
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
    }
    if prefill:
        # A prefill chunk is a dense contraction: its roofline is the tensor peak.
        tpeak, tsrc = tensor_peak()
        tflops = flops / (attn_mean * 1e-3) / 1e12
        line["roofline"].update({"bound": "tensor", "achieved": round(tflops, 2), "peak": tpeak,
                                 "unit": "TFLOP/s", "frac": round(tflops / tpeak, 4),
                                 "peak_source": tsrc,
                                 "hbm_gbs_of_algorithmic_bytes": round(achieved, 2)})
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not kv8 and not args.window:
        line["cpu_baseline"] = cpu_baseline(wl)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())

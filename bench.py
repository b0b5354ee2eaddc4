#!/usr/bin/env python
"""Benchmark of the paged decode-attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--kv bf16|fp8] [--window W] [--only]

A step is one pass of the whole hot path over one batch: kv_append of the
step's new K/V, then paged decode attention (plus its LSE merge launch) over
every sequence.  Each step is captured once as a CUDA graph and replayed; the
attention call alone is captured as a second graph.  Before every timed
replay the L2 is flushed (a write of 2x the 129 MB L2, then a read of 2x the
L2), outside the replay's own pair of CUDA events, so every step starts cold
and its bytes come from HBM whatever the size of its working set.

Printed (rank 0, one JSON line):
  * the headline workload (default: the Llama-3-8B-shaped GQA continuous
    batch, 64 sequences, contexts uniform in [128, 8192], 32 query / 8 KV
    heads, head_dim 128, block 16): effective GB/s of exactly K timed steps,
    where bytes = resident KV + q + out, microseconds per step, and the
    fraction of the measured copy peak, of a measured read-stream peak and of
    the nominal HBM rate;
  * its roofline from the attention call's own replays (attention + merge
    launches) in the same mode, with percentiles over at least 200 steps;
  * the end-to-end figure through the public API with host buffers, the
    oracle as a CPU baseline, and the SM clocks sampled while the steps ran;
  * `per_workload`: the same step and attention figures for every other
    named workload -- tiny, the MHA layer, MQA speculative verify, 128k
    contexts, the 8-bit (e4m3) cache on GQA / MQA verify / prefill, and the
    chunked-prefill chunk (a tensor-core roofline) -- 200 flushed steps each.

--kv fp8 makes the headline the same step over an 8-bit (e4m3) cache (the
quantising append, then attention); --window W times sliding-window
attention.  Their bytes count what the step must move: the e4m3 cache is one
byte per element, and a window reads at most W + q_len - 1 tokens per
sequence.  --only skips the per-workload lines (profiling runs).

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
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "attn_traffic.json")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama3_8b_gqa")
    ap.add_argument("--kv", choices=["bf16", "fp8", "fp8blk"], default="bf16")
    ap.add_argument("--window", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-soak", action="store_true",
                    help="skip the 1 s untimed load before the timed steps (profiling runs)")
    ap.add_argument("--only", action="store_true",
                    help="time the chosen workload only (no per-workload lines)")
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
    for name in ("decode_attn.cuh", "decode_attn.cu", "decode_attn_fp8.cu",
                 "decode_attn_fp8_block.cu", "ptx.cuh", "tcgen05.cuh", "pkv_internal.h"):
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
    if dist.get_backend() == "nccl":
        dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    else:
        dev = "cpu"
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
# Workloads timed beside the headline, each as (key, workload, kv dtype, window).
PER_WORKLOAD = [
    ("tiny", "tiny", "bf16", 0),
    ("llama2_7b_mha", "llama2_7b_mha", "bf16", 0),
    ("mqa_spec_verify", "mqa_spec_verify", "bf16", 0),
    ("long_splitk", "long_splitk", "bf16", 0),
    ("llama3_8b_gqa/e4m3", "llama3_8b_gqa", "fp8", 0),
    ("llama3_8b_gqa/e4m3_block_scales", "llama3_8b_gqa", "fp8blk", 0),
    ("mqa_spec_verify/e4m3", "mqa_spec_verify", "fp8", 0),
    ("mqa_spec_verify/e4m3_block_scales", "mqa_spec_verify", "fp8blk", 0),
    ("llama3_8b_chunked_prefill", "llama3_8b_chunked_prefill", "bf16", 0),
    ("llama3_8b_chunked_prefill/e4m3", "llama3_8b_chunked_prefill", "fp8", 0),
]
DIST_STEPS = 200  # steps behind each percentile line


class L2Flush:
    """Evicts the L2 before a timed step: a write of 2x the L2, then a read of 2x the L2
    (the read evicts the dirty lines the write left, so their write-back lands here and
    not in the timed step that follows)."""

    def __init__(self, device):
        import torch
        import paged_kv_cache_256_gb300 as pkv
        self.pkv = pkv
        n = 2 * L2_BYTES
        self.wbuf = torch.empty(n, dtype=torch.uint8, device=device)
        self.rbuf = torch.zeros(n, dtype=torch.uint8, device=device)
        self.sink = torch.zeros(1, dtype=torch.int32, device=device)
        self.k = 0

    def __call__(self):
        self.k = (self.k + 1) & 0x7F
        self.wbuf.fill_(self.k)
        self.pkv.pkv_read_stream(self.rbuf, self.sink)

    describe = ("flushed before every timed step: a write of 2x the 129 MB L2, then a read "
                "of 2x the L2 (pkv_read_stream), outside the timed events")


def read_peak(device, nbytes=2 << 30, reps=8):
    """Best read rate of pkv_read_stream over a 2 GiB buffer (16x the L2), GB/s."""
    import torch
    import paged_kv_cache_256_gb300 as pkv
    buf = torch.zeros(nbytes, dtype=torch.uint8, device=device)
    sink = torch.zeros(1, dtype=torch.int32, device=device)
    best, best_c = 0.0, 0
    for c in (1, 2, 3, 4):
        pkv.pkv_read_stream(buf, sink, c)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        for a, b in ev:
            a.record()
            pkv.pkv_read_stream(buf, sink, c)
            b.record()
        torch.cuda.synchronize(device)
        gbs = nbytes / (min(a.elapsed_time(b) for a, b in ev) * 1e-3) / 1e9
        if gbs > best:
            best, best_c = gbs, c
    del buf
    return {"gbs": round(best, 1), "ctas_per_sm": best_c, "bytes": nbytes,
            "kernel": "pkv_read_stream (16-byte loads, 8 in flight per thread, 512-thread CTAs)"}


def pctl(xs):
    """p10, p50, p90 of a list (ms) in microseconds."""
    q = statistics.quantiles(xs, n=10) if len(xs) >= 10 else [min(xs)] * 4 + [max(xs)] * 5
    return [round(1e3 * q[0], 2), round(1e3 * statistics.median(xs), 2), round(1e3 * q[8], 2)]


class Case:
    """One workload on the device: its step (append + attention) and its attention call,
    eager and as CUDA graphs."""

    def __init__(self, name, kv, window, device):
        import torch
        import paged_kv_cache_256_gb300 as pkv
        from paged_kv_cache_256_gb300.device import fp8_to_device, to_device
        from paged_kv_cache_256_gb300.workloads import (fp8_block_scales_for, fp8_cache_for,
                                                        make_workload)
        self.pkv, self.device = pkv, device
        self.wl = wl = make_workload(name)
        self.kv8 = kv in ("fp8", "fp8blk")
        self.blk = kv == "fp8blk"
        self.kv_name = {"bf16": "bf16", "fp8": "e4m3", "fp8blk": "e4m3, per-block scales"}[kv]
        self.window = window
        self.total_bytes, self.kv_bytes = step_bytes(wl, 1 if self.kv8 else 2, window)
        if self.blk:  # each (block, KV head) read also brings its 16-byte scale entry
            import numpy as np
            nblk = (wl.context_lens.astype(np.int64) + wl.block_size - 1) // wl.block_size
            self.total_bytes += 16 * wl.n_kv * int(nblk.sum())
        self.flops = step_flops(wl, window)
        self.dw = to_device(wl, device)
        self.d8 = fp8_to_device(fp8_cache_for(wl), device) if self.kv8 else None
        self.dsc = (torch.from_numpy(fp8_block_scales_for(wl)).to(device) if self.blk
                    else None)
        if self.kv8:  # the bf16 caches are not used by this step
            self.dw.k_cache = self.dw.v_cache = None
            torch.cuda.empty_cache()
        self.ws = pkv.alloc_workspace(wl.num_seqs, wl.q_len, wl.n_q, wl.n_kv, wl.head_dim,
                                      wl.block_size, device=device)
        self.out = torch.empty(tuple(self.dw.q.shape), dtype=torch.bfloat16, device=device)
        grid = torch.cuda.get_device_properties(device).multi_processor_count
        self.launches_per_step = 3 if grid > 1 else 2
        self.prefill = wl.group * wl.q_len > 128  # many query rows per KV head: compute-bound

    def append(self, s):
        pkv, dw, d8 = self.pkv, self.dw, self.d8
        if self.blk:
            pkv.pkv_kv_append_fp8_block(dw.k_new, dw.v_new, dw.slot_mapping, d8.kv_cache,
                                        self.dsc, stream=s)
        elif self.kv8:
            pkv.pkv_kv_append_fp8(dw.k_new, dw.v_new, dw.slot_mapping, d8.kv_cache, d8.k_scale,
                                  d8.v_scale, stream=s)
        else:
            pkv.pkv_kv_append(dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache,
                              stream=s)

    def attend(self, s):
        pkv, dw, d8, wl = self.pkv, self.dw, self.d8, self.wl
        if self.blk:
            pkv.pkv_paged_decode_attn_ex(dw.q, d8.kv_cache, None, dw.block_tables,
                                         dw.context_lens, wl.scale, self.out, self.ws, stream=s,
                                         window=self.window, kv_scales=self.dsc)
        elif self.kv8:
            pkv.pkv_paged_decode_attn_ex(dw.q, d8.kv_cache, None, dw.block_tables,
                                         dw.context_lens, wl.scale, self.out, self.ws, stream=s,
                                         window=self.window, k_scale=d8.k_scale,
                                         v_scale=d8.v_scale)
        elif self.window:
            pkv.pkv_paged_decode_attn_ex(dw.q, dw.k_cache, dw.v_cache, dw.block_tables,
                                         dw.context_lens, wl.scale, self.out, self.ws, stream=s,
                                         window=self.window)
        else:
            pkv.pkv_paged_decode_attn(dw.q, dw.k_cache, dw.v_cache, dw.block_tables,
                                      dw.context_lens, wl.scale, self.out, self.ws, stream=s)

    def step(self, s):
        self.append(s)
        self.attend(s)

    def check(self, what):
        st = self.pkv.pkv_check_error(self.ws)
        if st != self.pkv.PKV_OK:
            raise RuntimeError(f"{self.wl.name}: {what} reported {self.pkv.pkv_status_string(st)}")

    def capture(self, warmup):
        """Eager warm-up steps, then the step and the attention call captured as graphs."""
        import torch
        stream = torch.cuda.current_stream(self.device)
        for _ in range(max(3, warmup)):
            self.step(stream)
        torch.cuda.synchronize(self.device)
        self.check("warm-up")
        self.graphs = {}
        for kind, fn in (("step", self.step), ("attn", self.attend)):
            gs = torch.cuda.Stream(self.device)
            gs.wait_stream(stream)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=gs):
                fn(gs)
            stream.wait_stream(gs)
            for _ in range(3):
                g.replay()
            self.graphs[kind] = g
        torch.cuda.synchronize(self.device)
        self.check("graph warm-up")

    def time_replays(self, kind, n, flush):
        """n replays of one graph, the L2 flushed before each, each timed by its own events."""
        import torch
        g = self.graphs[kind]
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for a, b in ev:
            flush()
            a.record()
            g.replay()
            b.record()
        torch.cuda.synchronize(self.device)
        return [a.elapsed_time(b) for a, b in ev]

    def release(self):
        import torch
        self.graphs = None
        self.dw = self.d8 = self.dsc = self.ws = self.out = None
        torch.cuda.synchronize(self.device)
        torch.cuda.empty_cache()


def roofline_of(case, attn_ms, hbm, rpeak):
    """Roofline of the attention call (attention + merge launches) from its mean time."""
    achieved = case.total_bytes / (attn_ms * 1e-3) / 1e9
    key = case.wl.name + ("/fp8blk" if case.blk else "/fp8" if case.kv8 else "") + \
        (f"/w{case.window}" if case.window else "")
    r = {"kernel": "paged_decode_attn (attention + merge launches of one call)", "bound": "hbm",
         "achieved": round(achieved, 2), "peak": hbm[0], "unit": "GB/s",
         "frac": round(achieved / hbm[0], 4),
         "frac_of_read_peak": round(achieved / rpeak, 4) if rpeak else None,
         "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
         "traffic": profiled_traffic(key), "peak_source": hbm[1],
         "attn_us": round(attn_ms * 1e3, 2), "algorithmic_bytes_per_launch": case.total_bytes,
         "flops_per_launch": case.flops}
    if case.prefill:
        # A prefill chunk is a dense contraction: its roofline is the tensor peak.
        tpeak, tsrc = tensor_peak()
        tflops = case.flops / (attn_ms * 1e-3) / 1e12
        r.update({"bound": "tensor", "achieved": round(tflops, 2), "peak": tpeak,
                  "unit": "TFLOP/s", "frac": round(tflops / tpeak, 4), "peak_source": tsrc,
                  "frac_of_read_peak": None, "frac_of_nominal": None,
                  "hbm_gbs_of_algorithmic_bytes": round(achieved, 2)})
    return r


def workload_line(case, step_ms, attn_ms, hbm, rpeak, world):
    """One per-workload entry: distributions of flushed graph replays of the step and of
    the attention call."""
    mean_step, mean_attn = max_over_ranks([statistics.fmean(step_ms), statistics.fmean(attn_ms)])
    wl = case.wl
    return {
        "config": {"workload": wl.name, "num_seqs": wl.num_seqs, "n_q": wl.n_q, "n_kv": wl.n_kv,
                   "head_dim": wl.head_dim, "block_size": wl.block_size, "q_len": wl.q_len,
                   "kv_dtype": case.kv_name, "window": case.window,
                   "resident_tokens": wl.resident_tokens(), "bytes_per_step": case.total_bytes},
        "us_per_step": round(mean_step * 1e3, 2),
        "step_us_p10_p50_p90": pctl(step_ms),
        "value": round(whole_job_gbps(case.total_bytes, mean_step, world), 2), "unit": UNIT,
        "pct_of_peak": round(100.0 * case.total_bytes / (mean_step * 1e-3) / 1e9 / hbm[0], 2),
        "attn_us": round(mean_attn * 1e3, 2),
        "attn_us_p10_p50_p90": pctl(attn_ms),
        "steps_timed": len(step_ms),
        "roofline": roofline_of(case, mean_attn, hbm, rpeak),
    }


def e2e_of(case, K, world):
    """The step through the public API with host buffers: this step's inputs copied from
    pinned host memory, the step, and `out` copied back, all inside the timed region.
    The inputs (q, new K/V rows, slots, block tables, context lengths) sit back to back in
    one pinned staging buffer, as a serving loop would pack them, and arrive by one copy
    into a device buffer of the same layout that the calls read."""
    import dataclasses
    import numpy as np
    import torch
    wl, device = case.wl, case.device
    stream = torch.cuda.current_stream(device)
    fields = [("q", wl.q.view(np.int16), torch.bfloat16), ("k_new", wl.k_new.view(np.int16), torch.bfloat16),
              ("v_new", wl.v_new.view(np.int16), torch.bfloat16),
              ("slot_mapping", wl.slot_mapping, torch.int32),
              ("block_tables", wl.block_tables, torch.int32),
              ("context_lens", wl.context_lens, torch.int32)]
    offs, size = [], 0
    for _, arr, _ in fields:
        offs.append(size)
        size = (size + arr.nbytes + 255) // 256 * 256  # each field 256-byte aligned
    host_stage = torch.zeros(size, dtype=torch.uint8).pin_memory()
    dev_stage = torch.empty(size, dtype=torch.uint8, device=device)
    views = {}
    for (name, arr, dt), off in zip(fields, offs):
        flat = np.ascontiguousarray(arr).view(np.uint8).ravel()
        host_stage[off:off + flat.size].copy_(torch.from_numpy(flat))
        views[name] = dev_stage[off:off + flat.size].view(dt).view(arr.shape)
    out_host = torch.empty(tuple(case.out.shape), dtype=torch.int16).pin_memory()
    h2d = size
    d2h = out_host.numel() * out_host.element_size()
    saved = case.dw
    case.dw = dataclasses.replace(saved, **views)

    def e2e_step():
        dev_stage.copy_(host_stage, non_blocking=True)
        case.step(stream)
        out_host.copy_(case.out.view(torch.int16), non_blocking=True)

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
    e2e_ms = max_over_ranks([e0.elapsed_time(e1) / K])[0]
    case.check("end-to-end steps")
    case.dw = saved
    return {"value": round(whole_job_gbps(case.total_bytes, e2e_ms, world), 2), "unit": UNIT,
            "us_per_step": round(e2e_ms * 1e3, 2), "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "timed_as": "eager launches, back to back; per step one host-to-device copy of the "
                        "packed inputs and one device-to-host copy of out, in the timed region"}


def run_ours(args):
    import torch

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)

    hbm = hbm_peak()
    flush = L2Flush(device)
    rpk = read_peak(device)
    rpeak = max_over_ranks([-rpk["gbs"]])[0] * -1.0  # the slowest rank's read peak

    clocks = ClockSampler(local)
    clocks.start()
    # ---- the headline workload: exactly K timed steps, then its distributions
    case = Case(args.workload, args.kv, args.window, device)
    case.capture(args.warmup)
    # Let the sampler see the GPU under load before the timed steps.
    t_soak = time.perf_counter()
    while not args.no_soak and time.perf_counter() - t_soak < 1.0:
        case.time_replays("step", 20, flush)
    K = args.steps
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    step_ms_k = case.time_replays("step", K, flush)
    torch.cuda.synchronize(device)
    if world > 1:
        torch.distributed.barrier()
    case.check("timed steps")
    ms_per_step = max_over_ranks([statistics.fmean(step_ms_k)])[0]
    n_dist = max(K, DIST_STEPS)
    step_ms = step_ms_k + case.time_replays("step", n_dist - K, flush) if n_dist > K else step_ms_k
    attn_ms = case.time_replays("attn", n_dist, flush)
    case.check("distribution steps")
    head = workload_line(case, step_ms, attn_ms, hbm, rpeak, world)
    wl = case.wl
    launches = case.launches_per_step * K
    headline_case = (wl.name, args.kv, case.window)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not case.kv8 and \
            not args.window:
        cpu = cpu_baseline(wl)

    # ---- the other workloads: the same flushed graph replays, DIST_STEPS of each
    per = {}
    if not args.only:
        for key, name, kv, window in PER_WORKLOAD:
            if (name, kv, window) == headline_case:
                continue
            c = Case(name, kv, window, device)
            c.capture(args.warmup)
            s_ms = c.time_replays("step", DIST_STEPS, flush)
            a_ms = c.time_replays("attn", DIST_STEPS, flush)
            c.check("timed steps")
            per[key] = workload_line(c, s_ms, a_ms, hbm, rpeak, world)
            c.release()
    clk = clocks.stop()
    # The end-to-end figure runs eager launches from the host, after the clock
    # sampler has stopped: its polling of the driver can stall the host's
    # launches (the device-timed replays above do not wait on the host).
    e2e = None if args.no_e2e else e2e_of(case, K, world)
    case.release()

    total_bytes = case.total_bytes
    value = whole_job_gbps(total_bytes, ms_per_step, world)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "us_per_step": round(ms_per_step * 1e3, 2),
        "pct_of_peak": round(100.0 * value / world / hbm[0], 2),
        "pct_of_read_peak": round(100.0 * value / world / rpeak, 2),
        "pct_of_nominal": round(100.0 * value / world / NOMINAL_HBM_GBS, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 KV (f16 products, fp32 softmax)" if case.kv8 else "bf16",
        "data": "synthetic",
        "config": {
            "workload": wl.name, "num_seqs": wl.num_seqs, "n_q": wl.n_q, "n_kv": wl.n_kv,
            "head_dim": wl.head_dim, "block_size": wl.block_size, "q_len": wl.q_len,
            "resident_tokens": wl.resident_tokens(), "bytes_per_step": total_bytes,
            "kv_bytes": case.kv_bytes, "kv_dtype": case.kv_name,
            "window": case.window, "l2": L2Flush.describe,
            "step": ("kv_append_fp8_block" if case.blk else "kv_append_fp8" if case.kv8
                     else "kv_append") +
                    " + paged_decode_attn (+ lse_merge)",
            "timed_as": "CUDA-graph replay of the step, one pair of events per step",
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
            "step_us_p10_p50_p90": head["step_us_p10_p50_p90"],
            "attn_us_p10_p50_p90": head["attn_us_p10_p50_p90"],
            "percentiles_over_steps": n_dist,
        },
        "roofline": head["roofline"],
        "read_peak_gbs": rpeak,
        "read_peak": rpk,
        "nominal_hbm_gbs": NOMINAL_HBM_GBS,
        "e2e": e2e,
        "gpu_launches": launches,
        "per_workload": per,
        "clocks": clk,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
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

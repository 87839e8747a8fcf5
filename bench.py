#!/usr/bin/env python3
"""Benchmark: shared-KV multi-decoder paged decode attention on GB300.

One step = one shkv_decode_attention call (one layer of one decode step for
the whole batch: every decoder's stacked queries against the shared paged
cache).  The headline value is KV GB/s: the algorithmic bytes of a step
(unique KV pages + Q + O, each read or written once) divided by the step
time, summed over ranks.  Also reported: decode steps/s, fraction of the
measured HBM peak, the same kernel run once per decoder without sharing,
an end-to-end figure through the C ABI with host buffers, and the fp64
oracle timed on the host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl shkv|reference]

The default workload is Qwen3-14B attention (128 requests, 8 decoders,
contexts from a truncated log-normal with mean 27K tokens, ~14.5 GB of KV per
step), the largest configuration.  Under torchrun the global batch is N
batches of the configuration; the host partitioner (shkv_partition_requests)
gives each rank its requests, balanced by unique KV bytes, and each rank
holds and streams only its own pages: the path shards by request with no
exchange step, per-GPU work stays about one batch (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from cross_model_shared_gb300 import workloads as W  # noqa: E402

METRIC = "shared-KV decode attention: KV GB/s (% of HBM peak) and decode steps/s"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
# The decode kernel each consumer runs, the source files that define it, and
# the stem of its committed ncu summaries under profiles/.
_CSRC = "cross_model_shared_gb300/csrc/"
KERNELS = {
    "mma.sync": {"name": "shkv_decode_kernel", "stem": "decode_attn",
                 "sources": [_CSRC + "decode_attn.cu", _CSRC + "decode_common.cuh", _CSRC + "shkv_device.cuh"]},
    "tcgen05": {"name": "shkv_decode_umma_kernel", "stem": "decode_umma",
                "sources": [_CSRC + "decode_umma.cu", _CSRC + "decode_common.cuh", _CSRC + "shkv_device.cuh"]},
}


# ---------------------------------------------------------------------------
def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="qwen14b", choices=W.CONFIG_ORDER)
    ap.add_argument("--batch", type=int, default=0,
                    help="use only the first B requests of the workload (reduced case for profiling)")
    ap.add_argument("--impl", default="shkv", choices=["shkv", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--isolated", type=int, default=20,
                    help="single decode launches timed one at a time, each after an L2 flush (0: skip)")
    ap.add_argument("--prefix-pages", action="store_true",
                    help="host-side page-manager run: a seeded multi-agent workflow over the prefix pool")
    ap.add_argument("--prefill-tokens", type=int, default=0,
                    help="time the causal partial prefill of this many new tokens per request "
                         "(appended after the workload's cached prefixes)")
    ap.add_argument("--tail-tokens", type=int, default=0,
                    help="give every decoder its own unique tail of about this many tokens (seeded, "
                         "uniform in [T/2, 3T/2]) and time the decode with tails")
    return ap.parse_args()


def load_workload(args, replica: int = 0) -> W.Workload:
    wl = W.make_workload(args.config, replica)
    if args.batch and args.batch < wl.B:
        wl = W.custom_workload(f"{wl.name}[:{args.batch}]", B=args.batch, N=wl.N, Hq=wl.Hq, Hkv=wl.Hkv, D=wl.D,
                               P=wl.P, lens_prefill=wl.lens_prefill[:args.batch], n_append=wl.n_append, seed=wl.seed)
    return wl


class Job:
    """The whole job's requests and this rank's share of them.  One rank: the
    configuration itself.  N ranks: N batches of the configuration (replica
    r drawn with its own seed), divided among the ranks by the library's
    host partitioner, each rank holding only its own requests' pages."""

    def __init__(self, args, world_size: int, rank: int, partition: bool = True):
        self.base = load_workload(args)
        parts = [self.base] + [load_workload(args, r) for r in range(1, world_size)]
        self.lens_prefill = np.concatenate([w.lens_prefill for w in parts]).astype(np.int32)
        self.lens_final = np.concatenate([w.lens_final for w in parts]).astype(np.int32)
        self.world_size, self.rank = world_size, rank
        b = self.base
        self.page_bytes = b.P * b.Hkv * b.D * 2 * 2
        self.qo_bytes_per_request = 2 * b.rows * b.D * 2
        self.kv_bytes = int(((self.lens_final.astype(np.int64) + b.P - 1) // b.P).sum()) * self.page_bytes
        if not partition:
            return
        if world_size == 1:
            self.owner = np.zeros(b.B, np.int32)
            self.rank_pages = np.array([int(b.pages_per_request().sum())], np.int64)
            self.local = b
        else:
            from cross_model_shared_gb300 import _native as N
            self.owner, self.rank_pages = N.shkv_partition_requests(self.lens_final, b.P, world_size)
            mine = np.flatnonzero(self.owner == rank)
            self.local = W.custom_workload(f"{b.name} shard {rank}/{world_size}", B=len(mine), N=b.N, Hq=b.Hq,
                                           Hkv=b.Hkv, D=b.D, P=b.P, lens_prefill=self.lens_prefill[mine],
                                           n_append=b.n_append, seed=1000 * b.seed + rank + 1)

    def rank_requests(self):
        return [int((self.owner == r).sum()) for r in range(self.world_size)]

    def rank_bytes(self):
        """Algorithmic bytes of one step on each rank: its unique KV pages +
        its queries read + its outputs written."""
        return [int(self.rank_pages[r]) * self.page_bytes + n * self.qo_bytes_per_request
                for r, n in enumerate(self.rank_requests())]

    def total_bytes(self) -> int:
        """Algorithmic bytes of one step of the whole job (every rank's)."""
        return self.kv_bytes + len(self.lens_final) * self.qo_bytes_per_request


def workload_config(job: "Job"):
    """The `config` object of both arms' JSON lines: the workload by name
    and shape, the job's global batch, and how L2 reuse between timed steps
    is excluded."""
    per_rank_kv = job.kv_bytes // job.world_size
    l2 = l2_label(per_rank_kv, pool_copies_for(per_rank_kv))
    b = job.base
    return {
        "workload": b.name, "batch": int(len(job.lens_final)), "decoders": b.N, "hq_per_decoder": b.Hq,
        "hkv": b.Hkv, "head_dim": b.D, "page_size": b.P, "rows_per_kv_head": b.R,
        "mean_context": float(job.lens_final.mean()), "kv_bytes_per_step": job.kv_bytes,
        "step_bytes": job.total_bytes(),
        "l2": l2, "parallelism": f"request shards x{job.world_size}",
    }


L2_BYTES = 129 * 2**20
ROTATE_BELOW_BYTES = 10**9


def pool_copies_for(kv_bytes: int) -> int:
    """Copies of a pool to rotate through so that consecutive steps read
    different memory: enough to pass 1 GB of KV, at most 16."""
    if kv_bytes >= ROTATE_BELOW_BYTES:
        return 1
    return int(min(16, -(-ROTATE_BELOW_BYTES // max(1, kv_bytes))))


def l2_label(kv_bytes: int, copies: int) -> str:
    if copies == 1:
        return f"inputs larger than L2: {kv_bytes / 1e9:.2f} GB of KV per step vs 129 MB of L2"
    total = copies * kv_bytes
    resident = "larger than L2" if total > 2 * L2_BYTES else "L2-resident (warm)"
    return f"{copies} pool copies rotated step by step ({total / 1e9:.2f} GB, {resident})"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_sha(consumer: str) -> str:
    h = hashlib.sha256()
    for rel in KERNELS[consumer]["sources"]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(consumer: str, config: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel on
    this workload, if it was taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"{KERNELS[consumer]['stem']}_{config}_traffic.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.lstrip().startswith("#"):
                    k, _, v = line.partition(":")
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha") != kernel_sha(consumer):
            return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


def max_over_ranks(value: float, world_size: int, device) -> float:
    """Largest value over all ranks (the slowest rank's time sets the job's
    time); identity on one rank."""
    if world_size == 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput_gbs(bytes_per_step: int, steps: int, world_size: int, seconds: float) -> float:
    """Whole-job GB/s: every rank processes its own replica of the step."""
    return world_size * bytes_per_step * steps / seconds / 1e9


def step_bytes(wl: W.Workload) -> int:
    """Algorithmic bytes of one step: unique KV pages + Q read + O written."""
    qo = 2 * wl.B * wl.rows * wl.D * 2
    return W.unique_kv_bytes(wl) + qo


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        t0, t1 = (self.marks[0], self.marks[-1]) if len(self.marks) >= 2 else (0, float("inf"))
        rows = [s for t, s in self.samples if t0 <= t <= t1 + 0.06] or [s for _, s in self.samples]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
def quantile_requests(lens, n: int = 8):
    """A fixed subset of up to n requests at evenly spaced length quantiles
    (shortest, ..., median, ..., longest)."""
    order = np.argsort(np.asarray(lens), kind="stable")
    idx = np.unique(np.rint(np.linspace(0, len(order) - 1, min(n, len(order)))).astype(int))
    return [int(order[i]) for i in idx]


def cpu_oracle_sample(wl: W.Workload, q_bits, fetch_pages, budget_s: float, step_kv_bytes: int):
    """Time the fp64 oracle on whole requests (all rows, full context): a
    fixed subset of 8 requests at the workload's length quantiles, cycled
    until the budget is spent.  The rate (KV GB/s) is extrapolated to a whole
    step.  Returns the cpu_baseline object."""
    import oracle
    picks = quantile_requests(wl.lens_final)
    kv_bytes, elapsed, done = 0, 0.0, []
    cache = {}
    i = 0
    while elapsed < budget_s and i < 64 * len(picks):
        b = picks[i % len(picks)]
        if b not in cache:
            cache[b] = fetch_pages(b)
        kb, vb, npg = cache[b]
        bt = np.arange(npg, dtype=np.int32)[None, :]
        t0 = time.perf_counter()
        oracle.decode_attention(q_bits[b:b + 1], kb, vb, bt, np.array([wl.lens_final[b]], np.int32),
                                n_models=wl.N, hq=wl.Hq, scale=wl.scale)
        elapsed += time.perf_counter() - t0
        kv_bytes += npg * wl.P * wl.Hkv * wl.D * 4
        done.append(b)
        i += 1
    value = kv_bytes / elapsed / 1e9
    lens = [int(wl.lens_final[b]) for b in picks]
    desc = (f"{len(picks)} whole requests of {wl.name} at its length quantiles ({min(lens)}..{max(lens)} tokens; "
            f"all {wl.rows} stacked rows, full context), {len(done)} oracle calls, fp64, "
            f"{oracle.num_threads()} threads; rate extrapolated to the whole step")
    return {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle", "sample": desc,
            "seconds": round(elapsed, 2), "extrapolated_step_s": step_kv_bytes / (value * 1e9)}


def run_reference(args):
    """The oracle as the reference arm, on the host cores (rank 0 only): each
    step is one whole request of the workload (all stacked rows, full
    context), cycling through the 8 requests at its length quantiles like the
    cpu_baseline sample; their pages are drawn on the host (untimed)."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    job = Job(args, ws, 0, partition=False)      # the GPU arm's global batch at this world size
    wl = job.base
    q = W.gen_q(wl)
    rng = np.random.default_rng(wl.seed + 77)
    picks = quantile_requests(wl.lens_final)
    cache = {}

    def pages(b):
        if b not in cache:
            npg = int((wl.lens_final[b] + wl.P - 1) // wl.P)
            shape = (npg, wl.Hkv, wl.P, wl.D)
            cache[b] = (W.bf16_bits_from_f32(rng.standard_normal(shape, dtype=np.float32)),
                        W.bf16_bits_from_f32(rng.standard_normal(shape, dtype=np.float32)), npg)
        return cache[b]

    kv_bytes, elapsed, done = 0, 0.0, []
    wall0 = time.perf_counter()
    total_steps = args.steps + args.warmup
    for s in range(total_steps):
        b = picks[s % len(picks)]
        kb, vb, npg = pages(b)
        bt = np.arange(npg, dtype=np.int32)[None, :]
        t0 = time.perf_counter()
        oracle.decode_attention(q[b:b + 1], kb, vb, bt, np.array([wl.lens_final[b]], np.int32),
                                n_models=wl.N, hq=wl.Hq, scale=wl.scale)
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            elapsed += dt
            kv_bytes += npg * wl.P * wl.Hkv * wl.D * 4
            done.append(b)
        if time.perf_counter() - wall0 > 240.0 and len(done) > 0:
            break                      # keep the arm within a few minutes
    value = kv_bytes / elapsed / 1e9
    lens = [int(wl.lens_final[b]) for b in picks]
    desc = (f"{len(done)} timed steps, each one whole request of {wl.name} from the {len(picks)} at its length "
            f"quantiles ({min(lens)}..{max(lens)} tokens; all {wl.rows} stacked rows, full context), fp64 oracle, "
            f"{oracle.num_threads()} threads")
    kv_step = job.kv_bytes
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * elapsed / max(1, len(done)),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(job),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": desc, "extrapolated_step_s": kv_step / (value * 1e9)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
class E2EPipeline:
    """End-to-end steps through the C ABI: each step copies its queries from
    pinned host memory to the device, runs the decode, and copies its output
    back to pinned host memory.  The copies run on their own streams with two
    buffers of each, so step i+1's upload and step i-1's download overlap
    step i's kernel, as a serving loop would; every step still moves its own
    bytes in both directions."""

    def __init__(self, q, run):
        import torch
        self.run = run
        self.q_host = [torch.empty(q.shape, dtype=q.dtype, pin_memory=True) for _ in range(2)]
        self.out_host = [torch.empty(q.shape, dtype=q.dtype, pin_memory=True) for _ in range(2)]
        for h in self.q_host:
            h.copy_(q.cpu())
        self.q_dev = [torch.empty_like(q) for _ in range(2)]
        self.out_dev = [torch.empty_like(q) for _ in range(2)]
        self.main = torch.cuda.current_stream()
        self.s_in, self.s_out = torch.cuda.Stream(), torch.cuda.Stream()
        self.ev_in = [torch.cuda.Event() for _ in range(2)]
        self.ev_done = [torch.cuda.Event() for _ in range(2)]
        self.ev_out = [torch.cuda.Event() for _ in range(2)]
        for ev in self.ev_done + self.ev_out:
            ev.record(self.main)
        self.i = 0

    def step(self):
        import torch
        j = self.i & 1
        with torch.cuda.stream(self.s_in):
            self.s_in.wait_event(self.ev_done[j])          # the decode two steps back has read q_dev[j]
            self.q_dev[j].copy_(self.q_host[j], non_blocking=True)
            self.ev_in[j].record(self.s_in)
        self.main.wait_event(self.ev_in[j])
        self.main.wait_event(self.ev_out[j])                # out_dev[j] of two steps back is on the host
        self.run(self.q_dev[j], self.out_dev[j])
        self.ev_done[j].record(self.main)
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_event(self.ev_done[j])
            self.out_host[j].copy_(self.out_dev[j], non_blocking=True)
            self.ev_out[j].record(self.s_out)
        self.i += 1


def tail_lengths(wl: W.Workload, T: int) -> np.ndarray:
    rng = np.random.default_rng(wl.seed + 4242)
    return rng.integers(max(0, T // 2), T + T // 2 + 1, size=(wl.B, wl.N)).astype(np.int32)


def run_gpu_tails(args):
    """Decode where every decoder also attends its own unique tail
    (PrefillShare Eq. 9: one shared prefix, N unique tails)."""
    import torch
    from cross_model_shared_gb300 import DecoderTails, SharedKVPool

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    base = load_workload(args)
    probe = tail_lengths(base, args.tail_tokens)
    wl = W.custom_workload(f"{base.name}+tails{args.tail_tokens}", B=base.B, N=base.N, Hq=base.Hq, Hkv=base.Hkv,
                           D=base.D, P=base.P, lens_prefill=base.lens_prefill, n_append=base.n_append,
                           seed=base.seed, spare_pages=W.tails_spare_pages(probe, base.P))
    tt, tl = W.make_tails(wl, probe, seed=wl.seed + 1)
    q_bits = W.gen_q(wl)
    k_dev, v_dev = W.gen_pool_device(wl, device=dev)
    pool = SharedKVPool(wl.num_pages, wl.P, wl.Hkv, wl.D, max_batch=wl.B, max_pages_per_seq=wl.max_pages_per_seq,
                        device=dev, k_pages=k_dev, v_pages=v_dev, initial_seq_lens=wl.lens_final)
    pool.block_table.copy_(torch.from_numpy(wl.block_table).to(dev))
    tails = DecoderTails(pool, wl.B, wl.N, tt.shape[2], initial_tail_lens=tl)
    tails.block_table.copy_(torch.from_numpy(tt).to(dev))
    q = torch.from_numpy(q_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    out = torch.empty_like(q)
    lse = torch.empty((wl.B, wl.rows), dtype=torch.float32, device=dev)
    torch.cuda.synchronize()

    def step():
        tails.decode_attention(q, scale=wl.scale, out=out, lse=lse)

    for _ in range(max(3, args.warmup)):
        step()
    if pool.check_errors():
        raise RuntimeError("device error bits during warm-up")
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.2)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    sampler.mark()
    clocks = sampler.stop()
    ms = ev0.elapsed_time(ev1)
    if pool.check_errors():
        raise RuntimeError("device error bits in the timed region")
    shared_kv = W.unique_kv_bytes(wl)
    tail_kv = int(((tl.astype(np.int64) + wl.P - 1) // wl.P).sum()) * wl.P * wl.Hkv * wl.D * 4
    nbytes = shared_kv + tail_kv + 2 * wl.B * wl.rows * wl.D * 2
    ms_per_step = ms / args.steps
    per_gpu = nbytes / (ms_per_step * 1e-3) / 1e9
    value = job_throughput_gbs(nbytes, args.steps, 1, ms * 1e-3)

    # end to end through the C ABI: pinned host q in, host out back, per step
    e_steps = max(200, min(args.steps, 1000))     # host-timed: enough steps that a host stall is noise
    pipe = E2EPipeline(q, lambda qd, od: tails.decode_attention(qd, scale=wl.scale, out=od, lse=lse))
    e2e_step = pipe.step

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e_steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_value = nbytes * e_steps / (time.perf_counter() - t0) / 1e9

    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        order = np.argsort(wl.lens_final, kind="stable")
        kv_b, elapsed, done = 0, 0.0, []
        i = 0
        while elapsed < args.cpu_budget_s and i < 64 * wl.B:
            b = int(order[(len(order) // 2 + i) % len(order)])
            npg = int((wl.lens_final[b] + wl.P - 1) // wl.P)
            tpg = ((tl[b].astype(np.int64) + wl.P - 1) // wl.P).astype(int)
            ids = np.concatenate([wl.block_table[b, :npg]] + [tt[b, m, :tpg[m]] for m in range(wl.N)]).astype(np.int64)
            idt = torch.from_numpy(ids).to(dev)
            kb = k_dev.index_select(0, idt).view(torch.int16).cpu().numpy().view(np.uint16)
            vb = v_dev.index_select(0, idt).view(torch.int16).cpu().numpy().view(np.uint16)
            bt = np.arange(npg, dtype=np.int32)[None, :]
            ttl = np.full((1, wl.N, max(1, int(tpg.max()))), -1, np.int32)
            off = npg
            for m in range(wl.N):
                ttl[0, m, :tpg[m]] = np.arange(off, off + tpg[m])
                off += tpg[m]
            t0 = time.perf_counter()
            oracle.decode_attention_tails(q_bits[b:b + 1], kb, vb, bt, np.array([wl.lens_final[b]], np.int32), ttl,
                                          tl[b:b + 1], n_models=wl.N, hq=wl.Hq, scale=wl.scale)
            elapsed += time.perf_counter() - t0
            kv_b += len(ids) * wl.P * wl.Hkv * wl.D * 4
            done.append(b)
            i += 1
        cpu = {"value": kv_b / elapsed / 1e9, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
               "sample": f"{len(done)} whole requests of {wl.name} with their {wl.N} tails, fp64, "
                         f"{oracle.num_threads()} threads", "seconds": round(elapsed, 2)}

    peak, peak_kind = measured_peaks()
    consumer = pool.decode_consumer(wl.N, wl.Hq)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.B, "decoders": wl.N, "hq_per_decoder": wl.Hq, "hkv": wl.Hkv,
                   "head_dim": wl.D, "page_size": wl.P, "rows_per_kv_head": wl.R,
                   "mean_context": float(wl.lens_final.mean()), "mean_tail": float(tl.mean()),
                   "shared_kv_bytes": shared_kv, "tail_kv_bytes": tail_kv, "step_bytes": nbytes,
                   "l2": "inputs larger than L2" if shared_kv + tail_kv > 2 * 129e6 else "L2-resident working set",
                   "parallelism": "replicas x1"},
        "steps_per_s": 1e3 / ms_per_step,
        "pct_of_hbm_peak": {"measured_copy": 100 * per_gpu / peak, "nominal_8tbs": 100 * per_gpu / NOMINAL_HBM_GBS},
        "roofline": {"bound": "hbm", "achieved": per_gpu, "peak": peak, "unit": "GB/s", "frac": per_gpu / peak,
                     "peak_kind": peak_kind, "traffic": None, "kernel": KERNELS[consumer]["name"],
                     "consumer": consumer, "note": "whole step: the unit-table kernel and one decode pass over shared pages and tails"},
        "unshared": None,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": q.numel() * 2,
                "d2h_bytes_per_step": q.numel() * 2, "steps": e_steps,
                "copies": "own streams, two buffers: overlap the neighbouring steps' kernels"},
        "gpu_launches": 2 * args.steps,     # the tails-unit kernel and the decode, per step
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def run_prefix_pages(args):
    """Seeded agent workflow over the prefix pool (PrFaaS hybrid prefix cache
    pool; ICaRus key design 2: prompts cached for one agent are hits for the
    others).  Per session, every round each of the N agents sends the
    session context plus its own instruction; its output (the next round's
    context growth) is appended afterwards.  Compares pages held and tokens
    prefilled with the pool against every request holding private pages."""
    from cross_model_shared_gb300 import PrefixPages
    wl = load_workload(args)
    rng = np.random.default_rng(wl.seed + 99)
    P, n_agents = wl.P, wl.N
    sessions, rounds, instr, out_tok = 16, 4, 64, 256
    ctx = [rng.integers(0, 32000, size=int(L)).astype(np.int32) for L in wl.lens_prefill[:sessions]]
    max_tokens = max(len(c) for c in ctx) + rounds * (n_agents * out_tok + instr) + instr
    num_pages = sessions * n_agents * ((max_tokens + P - 1) // P)
    pages = PrefixPages(num_pages, P)
    ops, t_ops = 0, 0.0
    prefilled = total = 0
    peak_pool = peak_private = 0
    for r in range(rounds):
        held = []
        for s_ in range(sessions):
            for a in range(n_agents):
                prompt = np.concatenate([ctx[s_], np.full(instr, 100000 + a, np.int32)])
                t0 = time.perf_counter()
                pg, cached = pages.acquire(prompt)
                pages.publish(prompt, pg)
                t_ops += time.perf_counter() - t0
                ops += 2
                held.append(pg)
                prefilled += len(prompt) - cached
                total += len(prompt)
        st = pages.stats()
        peak_pool = max(peak_pool, st["referenced_pages"])
        peak_private = max(peak_private, sum(len(h) for h in held))
        t0 = time.perf_counter()
        for pg in held:
            pages.release(pg)
        t_ops += time.perf_counter() - t0
        ops += len(held)
        for s_ in range(sessions):
            for a in range(n_agents):
                ctx[s_] = np.concatenate([ctx[s_], rng.integers(0, 32000, size=out_tok).astype(np.int32)])
    st = pages.stats()
    line = {
        "metric": "prefix pool: pages held and prefill tokens saved (host page manager)",
        "value": 1.0 - prefilled / total, "unit": "fraction of prompt tokens served from cached pages",
        "higher_is_better": True, "data": "synthetic", "dtype": "int32",
        "config": {"workload": f"{wl.name} sessions={sessions} agents={n_agents} rounds={rounds} "
                               f"instruction={instr} output={out_tok}", "page_size": P},
        "pages_held_peak": {"prefix_pool": peak_pool, "private_pages": peak_private,
                            "ratio": peak_private / max(1, peak_pool)},
        "prefill_tokens": {"with_pool": prefilled, "without_pool": total},
        "block_hit_rate": st["block_hits"] / max(1, st["block_lookups"]),
        "host_ops_per_s": ops / t_ops, "ops": ops,
    }
    print(json.dumps(line), flush=True)


def measured_tensor_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def measured_tensor_peak_sustained():
    """cuBLAS bf16 GEMMs run back to back for seconds, under the power cap:
    the denominator for a dense kernel looped as long as the timed region is."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 1700.0, "fallback"


def run_gpu_prefill(args):
    """Causal partial prefill of T new tokens over each request's cached
    prefix (PrefillShare Sec. 3.3), on the tensor cores."""
    import torch
    from cross_model_shared_gb300 import SharedKVPool

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    base = load_workload(args)
    T = args.prefill_tokens
    wl = W.custom_workload(f"{base.name}+prefill{T}", B=base.B, N=1, Hq=base.Hq, Hkv=base.Hkv, D=base.D, P=base.P,
                           lens_prefill=base.lens_prefill, n_append=T, seed=base.seed)
    k_dev, v_dev = W.gen_pool_device(wl, device=dev)
    pool = SharedKVPool(wl.num_pages, wl.P, wl.Hkv, wl.D, max_batch=wl.B, max_pages_per_seq=wl.max_pages_per_seq,
                        device=dev, k_pages=k_dev, v_pages=v_dev, initial_seq_lens=wl.lens_final)
    pool.block_table.copy_(torch.from_numpy(wl.block_table).to(dev))
    g = torch.Generator(device=dev).manual_seed(wl.seed + 5)
    q = torch.randn((wl.B, T, wl.Hq, wl.D), generator=g, device=dev).to(torch.bfloat16)
    out = torch.empty_like(q)
    lse = torch.empty((wl.B, T, wl.Hq), dtype=torch.float32, device=dev)

    def step():
        pool.prefill_attention(q, scale=wl.scale, out=out, lse=lse)

    for _ in range(max(3, args.warmup)):
        step()
    if pool.check_errors():
        raise RuntimeError("device error bits during warm-up")
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.2)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    sampler.mark()
    clocks = sampler.stop()
    if pool.check_errors():
        raise RuntimeError("device error bits in the timed region")
    ms = ev0.elapsed_time(ev1) / args.steps
    prefix = wl.lens_final.astype(np.int64) - T
    keys_b = prefix * T + T * (T + 1) // 2                                   # per request: keys attended, summed
    flops_b = 4.0 * keys_b * wl.Hq * wl.D                                    # QK and PV, 2 flops per MAC
    flops = float(flops_b.sum())
    kv_bytes = W.unique_kv_bytes(wl)
    tflops = flops / (ms * 1e-3) / 1e12
    peak, kind = measured_tensor_peak()
    peak_s, _ = measured_tensor_peak_sustained()

    # end to end through the C ABI: pinned host q in, host out back, per step
    e_steps = max(10, min(args.steps, 200))
    pipe = E2EPipeline(q, lambda qd, od: pool.prefill_attention(qd, scale=wl.scale, out=od, lse=lse))
    for _ in range(3):
        pipe.step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e_steps):
        pipe.step()
    torch.cuda.synchronize()
    e2e_value = flops * e_steps / (time.perf_counter() - t0) / 1e12

    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        order = np.argsort(wl.lens_final, kind="stable")
        q_bits = q.view(torch.int16).cpu().numpy().view(np.uint16)
        fl, elapsed, done = 0.0, 0.0, []
        i = 0
        while elapsed < args.cpu_budget_s and i < wl.B:
            b = int(order[(len(order) // 2 + i) % len(order)])
            npg = int((wl.lens_final[b] + wl.P - 1) // wl.P)
            idt = torch.from_numpy(wl.block_table[b, :npg].astype(np.int64)).to(dev)
            kb = k_dev.index_select(0, idt).view(torch.int16).cpu().numpy().view(np.uint16)
            vb = v_dev.index_select(0, idt).view(torch.int16).cpu().numpy().view(np.uint16)
            t0 = time.perf_counter()
            oracle.prefill_attention(q_bits[b:b + 1], kb, vb, np.arange(npg, dtype=np.int32)[None, :],
                                     np.array([wl.lens_final[b]], np.int32), scale=wl.scale)
            elapsed += time.perf_counter() - t0
            fl += float(flops_b[b])
            done.append(b)
            i += 1
        cpu = {"value": fl / elapsed / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
               "sample": f"{len(done)} whole requests of {wl.name} ({T} new tokens each), fp64, "
                         f"{oracle.num_threads()} threads", "seconds": round(elapsed, 2)}
    line = {
        "metric": "partial-prefill attention: TFLOP/s (% of bf16 tensor peak)", "value": tflops, "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.B, "new_tokens": T, "hq": wl.Hq, "hkv": wl.Hkv,
                   "head_dim": wl.D, "page_size": wl.P, "mean_prefix": float(prefix.mean()),
                   "kv_bytes": kv_bytes, "flops": flops, "parallelism": "replicas x1"},
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                     "peak_kind": kind, "traffic": None, "kernel": "shkv_prefill_umma_kernel",
                     "kv_gbs": kv_bytes / (ms * 1e-3) / 1e9,
                     # the timed region is args.steps launches back to back, as
                     # long as the sustained GEMM loop: its fraction, for context
                     "peak_sustained": peak_s, "frac_of_sustained": tflops / peak_s,
                     "timed_s": ms * args.steps / 1e3},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": q.numel() * 2,
                "d2h_bytes_per_step": q.numel() * 2, "steps": e_steps,
                "copies": "own streams, two buffers: overlap the neighbouring steps' kernels"},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def run_gpu(args):
    import torch
    import torch.distributed as dist
    from cross_model_shared_gb300 import SharedKVPool

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", init_method="env://")

    job = Job(args, ws, rank)
    wl = job.local
    q_bits = W.gen_q(wl)
    k_dev, v_dev = W.gen_pool_device(wl, device=dev)
    pool = SharedKVPool(wl.num_pages, wl.P, wl.Hkv, wl.D, max_batch=wl.B, max_pages_per_seq=wl.max_pages_per_seq,
                        device=dev, k_pages=k_dev, v_pages=v_dev, initial_seq_lens=wl.lens_prefill)
    pool.block_table.copy_(torch.from_numpy(wl.block_table).to(dev))
    append = None
    if wl.n_append:
        g = torch.Generator(device=dev).manual_seed(404)
        shape = (wl.B, wl.n_append, wl.Hkv, wl.D)
        kn = torch.randn(shape, generator=g, device=dev).to(torch.bfloat16)
        vn = torch.randn(shape, generator=g, device=dev).to(torch.bfloat16)
        pool.append_kv(kn, vn)
        # the append timed on its own: lengths reset to the cached prefixes and
        # the same tokens appended again (the same bytes land in the same
        # slots), each launch between events after an L2 flush
        flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
        times = []
        for i in range(10):
            pool.set_seq_lens(wl.lens_prefill)
            flush.fill_(i & 0xff)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            pool.append_kv(kn, vn)
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        del flush, kn, vn
        ab = 4 * wl.B * wl.n_append * wl.Hkv * wl.D * 2          # K and V, read and written
        ams = statistics.median(times)
        append = {"ms": ams, "bytes": ab, "gbs": ab / (ams * 1e-3) / 1e9, "launches": len(times),
                  "how": "median of single launches after an L2 flush (lengths reset, same tokens appended)"}
    # Small pools are rotated: step i reads copy i % n, so consecutive steps
    # never find each other's pages in L2.
    n_copies = pool_copies_for(job.kv_bytes // ws)
    pools = [pool]
    for _ in range(1, n_copies):
        p2 = SharedKVPool(wl.num_pages, wl.P, wl.Hkv, wl.D, max_batch=wl.B, max_pages_per_seq=wl.max_pages_per_seq,
                          device=dev, k_pages=k_dev.clone(), v_pages=v_dev.clone(), initial_seq_lens=wl.lens_final)
        p2.block_table.copy_(pool.block_table)
        pools.append(p2)
    q = torch.from_numpy(q_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    out = torch.empty_like(q)
    for p_ in pools:
        p_.workspace(wl.B, wl.N, wl.Hq)
    torch.cuda.synchronize()
    it = [0]

    def step():
        pools[it[0] % n_copies].decode_attention(q, wl.N, scale=wl.scale, out=out)
        it[0] += 1

    for _ in range(max(3, args.warmup)):
        step()
    for p_ in pools:
        flags = p_.check_errors()
        if flags:
            raise RuntimeError(f"device error bits 0x{flags:x} during warm-up")

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.2)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    sampler.mark()
    if ws > 1:
        dist.barrier()
    clocks = sampler.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1), ws, dev)
    for p_ in pools:
        flags = p_.check_errors()
        if flags:
            raise RuntimeError(f"device error bits 0x{flags:x} in the timed region")

    ms_per_step = ms / args.steps
    nbytes = job.total_bytes()
    value = nbytes * args.steps / (ms * 1e-3) / 1e9
    local_bytes = job.rank_bytes()[rank]
    local_ms = ev0.elapsed_time(ev1) / args.steps
    per_gpu = local_bytes / (local_ms * 1e-3) / 1e9

    # --- isolated launches: each one after an L2 flush (a write over twice
    # the L2 size, itself a kernel between consecutive decode launches, so no
    # launch overlaps its predecessor), timed on its own
    isolated = None
    if args.isolated > 0:
        flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.isolated)]
        for i, (a, b) in enumerate(evs):
            flush.fill_(i & 0xff)
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        iso_ms = sorted(a.elapsed_time(b) for a, b in evs)
        med = statistics.median(iso_ms)
        # the same after a flush that reads the buffer instead: L2 is left
        # full of clean lines, so the launch does not also pay the write-back
        # of the dirty ones the write flush leaves behind
        flush32 = flush.view(torch.int32)
        for a, b in evs:
            torch.amax(flush32)          # int32 max: reads the buffer, no cast, one tiny write
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        rd_ms = statistics.median(a.elapsed_time(b) for a, b in evs)
        isolated = {"ms": med, "min_ms": iso_ms[0], "max_ms": iso_ms[-1], "launches": len(iso_ms),
                    "gbs": local_bytes / (med * 1e-3) / 1e9, "frac": None,
                    "how": "median of single launches, each after an L2 flush (a 258 MB write kernel)",
                    "after_read_flush": {"ms": rd_ms, "gbs": local_bytes / (rd_ms * 1e-3) / 1e9, "frac": None,
                                         "how": "the same after a kernel that reads the 258 MB buffer"}}
        del flush, flush32

    # --- the same kernel once per decoder, without sharing (N launches/step)
    q_models = [q[:, m * wl.Hq:(m + 1) * wl.Hq].contiguous() for m in range(wl.N)]
    out_m = [torch.empty_like(x) for x in q_models]
    u_steps = max(10, min(args.steps, 500))
    for m in range(wl.N):
        pool.decode_attention(q_models[m], 1, scale=wl.scale, out=out_m[m])
    torch.cuda.synchronize()
    ev0.record(stream)
    for i in range(u_steps):
        p_ = pools[i % n_copies]
        for m in range(wl.N):
            p_.decode_attention(q_models[m], 1, scale=wl.scale, out=out_m[m])
    ev1.record(stream)
    torch.cuda.synchronize()
    unshared_ms = ev0.elapsed_time(ev1) / u_steps

    # --- end to end through the C ABI: pinned host q in, host out back, per step
    e_steps = max(10, min(args.steps, 1000))
    pipe = E2EPipeline(q, lambda qd, od: pools[pipe.i % n_copies].decode_attention(qd, wl.N, scale=wl.scale,
                                                                                     out=od))
    for _ in range(3):
        pipe.step()
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(e_steps):
        pipe.step()
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, ws, dev)
    e2e_value = nbytes * e_steps / e2e_s / 1e9
    qbytes = len(job.lens_final) * wl.rows * wl.D * 2

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        def fetch(b):
            npg = int((wl.lens_final[b] + wl.P - 1) // wl.P)
            ids = torch.from_numpy(wl.block_table[b, :npg].astype(np.int64)).to(dev)
            kb = k_dev.index_select(0, ids).view(torch.int16).cpu().numpy().view(np.uint16)
            vb = v_dev.index_select(0, ids).view(torch.int16).cpu().numpy().view(np.uint16)
            return kb, vb, npg
        cpu = cpu_oracle_sample(wl, q_bits, fetch, args.cpu_budget_s, job.kv_bytes)

    peak, peak_kind = measured_peaks()
    if isolated is not None:
        isolated["frac"] = isolated["gbs"] / peak
        isolated["after_read_flush"]["frac"] = isolated["after_read_flush"]["gbs"] / peak
    consumer = pool.decode_consumer(wl.N, wl.Hq)
    traffic = profiled_traffic(consumer, job.base.name) if ws == 1 else None
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(job),
            "steps_per_s": 1e3 / ms_per_step,
            "decoder_tokens_per_s": len(job.lens_final) * wl.N * 1e3 / ms_per_step,
            "pct_of_hbm_peak": {"measured_copy": 100 * per_gpu / peak, "nominal_8tbs": 100 * per_gpu / NOMINAL_HBM_GBS},
            "roofline": {"bound": "hbm", "achieved": per_gpu, "peak": peak, "unit": "GB/s",
                         "frac": per_gpu / peak, "peak_kind": peak_kind, "traffic": traffic,
                         "kernel": KERNELS[consumer]["name"], "consumer": consumer,
                         "bytes_per_launch": local_bytes},
            "isolated": isolated,
            "unshared": {"ms_per_step": unshared_ms, "launches_per_step": wl.N,
                         "speedup_of_sharing": unshared_ms / local_ms},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": qbytes, "d2h_bytes_per_step": qbytes,
                    "steps": e_steps, "copies": "own streams, two buffers: overlap the neighbouring steps' kernels"},
            "shards": {"requests": job.rank_requests(), "step_bytes": job.rank_bytes(),
                       "partitioner": "shkv_partition_requests (longest first, fewest pages)"},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        if append is not None:
            append["frac_of_copy"] = append["gbs"] / peak
            line["append"] = append
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.prefix_pages:
        run_prefix_pages(args)
        return
    if args.prefill_tokens and args.impl == "shkv":
        run_gpu_prefill(args)
        return
    if args.tail_tokens and args.impl == "shkv":
        run_gpu_tails(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()

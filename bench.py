#!/usr/bin/env python
"""Benchmark of paged chunk attention forward + backward on GB300.

One step = one attention layer's whole chunk-recurrent sweep over a sequence
("Out of the Memory Barrier", gist.science/de §2.A-B): reset the sequence,
then for every chunk append its K/V into the paged pool and run the forward,
then run the backward over the chunks in reverse (dQ written, dK/dV added in
place into the paged fp32 gradient pool). Default workload: the Qwen2.5-7B
attention shape (28 q heads, 4 KV heads, d 128), bf16, page 128, 32K tokens in
chunks of 4096.

value = algorithmic fwd+bwd FLOPs (14 * Hq * d * attended pairs; pairs =
N(N+1)/2 for dense causal) / device time, in TFLOP/s. Prints one JSON line.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged chunk-attn fwd+bwd TFLOP/s & tokens/s/layer; % of bf16 TC peak"
UNIT = "TFLOP/s"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--workload", default="qwen7b_dense_32k")
    ap.add_argument("--context", type=int, default=0,
                    help="override the workload's context length N (a multiple of its chunk "
                         "length; 0 = the workload's own), e.g. for small profiling runs")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-sparse", action="store_true",
                    help="dense line only: skip its sub-record of the page-sparse 256K workload")
    ap.add_argument("--sparse-steps", type=int, default=5,
                    help="timed steps of the page-sparse sub-record (2 warm-up steps)")
    ap.add_argument("--flags", type=int, default=0, help="pool flags (1 = CUDA cores only)")
    ap.add_argument("--offload-chunks", type=int, default=8,
                    help="offload workload: chunks measured at the end of the sequence")
    ap.add_argument("--slots", type=int, default=0,
                    help="offload workload: device page slots (0 = the context's page count)")
    ap.add_argument("--layer-loop", action="store_true",
                    help="train one attention block (hidden 3584, random weights) chunk by "
                         "chunk with recomputation at 32K, 64K and 128K (or --context) and "
                         "report time and device memory per context length")
    ap.add_argument("--study", default="", choices=["", "topk-error"],
                    help="topk-error: sparse-vs-dense output and gradient error against "
                         "the top-K budget on a page-sparse workload, and the paged pool's "
                         "device footprint against the bytes its pages need")
    ap.add_argument("--overlap-proj", action="store_true",
                    help="offload workload: also run a synthetic bf16 K/V projection GEMM per "
                         "chunk on the main stream while the selected pages stream in, and "
                         "report how much of it the transfer hides")
    ap.add_argument("--offload-layers", type=int, default=0,
                    help="dense workload: measure L layers in pinned host memory, the next "
                         "layer's pages staged while the current one computes (0 = off)")
    return ap.parse_args()


def bench_workload(args):
    """The named workload, with --context replacing its context length."""
    from paged_kv_chunk_chunked_gb300 import synth
    w = synth.workload(args.workload)
    if args.context:
        if args.context <= 0 or args.context % w.C:
            raise SystemExit(f"--context must be a positive multiple of the chunk length {w.C}")
        w = w.with_(N=args.context, name=f"{w.name} at context {args.context}")
    return w


def ensure_library(world: int, rank: int):
    """Rank 0 builds libpkv (a no-op when it is up to date) while the others
    wait, so replicas never write the same objects at once; then every rank
    loads it."""
    from paged_kv_chunk_chunked_gb300 import binding as B
    from paged_kv_chunk_chunked_gb300 import build as pkv_build
    if rank == 0 or world == 1:
        pkv_build.build()
    barrier(world)
    B.lib()


def pairs_dense(N: int) -> int:
    return N * (N + 1) // 2


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples (200 ms) during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ distributed (replicas)

def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def reduce_max(x: float, world: int) -> float:
    """Max over ranks (replicas): the job's time is its slowest rank's."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_rate(units_per_rank: float, ms_local: float, world: int):
    """Whole-job rate over `world` independent replicas: every rank processes
    units_per_rank per step; the job's step time is the slowest rank's.
    Returns (units per second summed over ranks, max ms per step)."""
    ms = reduce_max(ms_local, world)
    return world * units_per_rank / (ms * 1e-3), ms


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ CPU oracle sample

def oracle_sample(w, n_queries: int):
    """Oracle fwd+bwd of the last chunk's last n_queries queries, one query head,
    against every key before them. Returns (algorithmic FLOPs, seconds, desc)."""
    import numpy as np
    import oracle
    from paged_kv_chunk_chunked_gb300 import synth
    c = w.n_chunks - 1
    s, e = w.chunk_range(c)
    ks = np.concatenate([synth.chunk_k(w, i)[:, :1] for i in range(w.n_chunks)])
    vs = np.concatenate([synth.chunk_v(w, i)[:, :1] for i in range(w.n_chunks)])
    q = synth.chunk_q(w, c)[-n_queries:, :1]
    do = synth.chunk_do(w, c)[-n_queries:, :1]
    q0 = e - n_queries
    t = time.perf_counter()
    o, lse = oracle.attention_forward(q, ks[:e], vs[:e], q0)
    oracle.attention_backward(q, ks[:e], vs[:e], o, do, lse, q0)
    dt = time.perf_counter() - t
    pairs = sum(q0 + i + 1 for i in range(n_queries))
    flops = 14 * w.d * pairs
    desc = (f"oracle fp64 fwd+bwd of the last {n_queries} queries of chunk {c}, 1 of {w.Hq} "
            f"query heads, against all {e} earlier keys ({pairs} pairs)")
    return flops, dt, desc


def cpu_threads() -> int:
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


# ------------------------------------------------------------------ roofline traffic

def traffic_for(kernel: str, source: str):
    """dram bytes per launch from the committed ncu summary, if the kernel's
    source is unchanged since the counters were taken; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        ent = t[kernel]
        sha = hashlib.sha256(open(os.path.join(ROOT, source), "rb").read()).hexdigest()[:16]
        return ent["bytes_per_launch"] if ent.get("source_sha") == sha else None
    except (OSError, KeyError, ValueError):
        return None


def dense_config(w, world: int) -> dict:
    """The `config` of the dense line; the reference arm reports the same."""
    return {"workload": w.name, "N": w.N, "C": w.C, "P": w.P, "Hq": w.Hq, "Hkv": w.Hkv,
            "d": w.d, "block_table": w.table, "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (Q, dO, O, dQ: 4 x 235 MB per step)"}


def tensor_peak(pk: dict, kind: str):
    """The bf16 tensor peak for kernels timed in a timed region of about a
    second or less at full clocks: MEASURED_PEAKS' burst figure (a cuBLAS GEMM
    timed alone); the sustained figure was taken under the power cap at lower
    clocks."""
    return pk.get("bf16_tflops", pk.get("bf16_tflops_sustained")), \
        f"{kind} bf16_tflops (burst: the kernels run at full clocks in a short timed region)"


# ------------------------------------------------------------------ pkv arm

def run_pkv(args, world, rank):
    import torch
    from paged_kv_chunk_chunked_gb300 import binding as B
    from paged_kv_chunk_chunked_gb300 import synth
    from paged_kv_chunk_chunked_gb300.sweep import ChunkSweep

    ensure_library(world, rank)
    w = bench_workload(args)
    sw = ChunkSweep(w, flags=args.flags).load_inputs()
    stream = torch.cuda.current_stream()
    n = w.n_chunks
    ev = lambda: torch.cuda.Event(enable_timing=True)
    fwd_ev = [[(ev(), ev()) for _ in range(n)] for _ in range(args.steps)]
    bwd_ev = [[(ev(), ev()) for _ in range(n)] for _ in range(args.steps)]

    def step(k=None):
        """One sweep; k = timed step index (records per-call events) or None."""
        sw.reset()
        for c in range(n):
            s, e = w.chunk_range(c)
            B.pkv_append(sw.seq, sw.k[c], sw.v[c], e - s, stream)
            if k is not None:
                fwd_ev[k][c][0].record(stream)
            B.pkv_chunk_attn_fwd(sw.seq, sw.q[c], s, e - s, sw.o[c], sw.lse[c], None, stream)
            if k is not None:
                fwd_ev[k][c][1].record(stream)
        for c in reversed(range(n)):
            if k is not None:
                bwd_ev[k][c][0].record(stream)
            sw.backward(c, stream)
            if k is not None:
                bwd_ev[k][c][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    B.pkv_check(sw.pool)
    barrier(world)
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    t0, t1 = ev(), ev()
    B.pkv_profile_enable(True)
    t0.record(stream)
    for k in range(args.steps):
        step(k)
    t1.record(stream)
    torch.cuda.synchronize()
    prof = B.pkv_profile_collect()
    B.pkv_profile_enable(False)
    fwd_ms = [sum(a.elapsed_time(b) for a, b in fwd_ev[k]) for k in range(args.steps)]
    bwd_ms = [sum(a.elapsed_time(b) for a, b in bwd_ev[k]) for k in range(args.steps)]
    clk = clocks.stop()
    barrier(world)
    B.pkv_check(sw.pool)
    flops_fwd = 4 * w.Hq * w.d * pairs_dense(w.N)
    flops_bwd = 10 * w.Hq * w.d * pairs_dense(w.N)
    flops_s, ms_step = replica_rate(flops_fwd + flops_bwd, t0.elapsed_time(t1) / args.steps, world)
    tflops = flops_s / 1e12
    pk, pk_kind = peaks()
    peak_tc, peak_kind = tensor_peak(pk, pk_kind)
    fwd_call = statistics.mean(fwd_ms) / n
    bwd_call = statistics.mean(bwd_ms) / n
    fwd_ach = flops_fwd / n / (fwd_call * 1e-3) / 1e12
    bwd_ach = flops_bwd / n / (bwd_call * 1e-3) / 1e12
    # Per-kernel device time from the library's event pairs (launching stream).
    # Algorithmic FLOPs attributed per kernel: forward 4 (S, PV); the backward's
    # 10 split as dK/dV kernel 8 (S^T, dP^T, dV, dK) and dQ kernel 2 (dQ; its
    # recomputed S and dP are not counted again) -- times Hq * d * pairs.
    per_step = {"fwd_tc_kernel": 4, "bwd_kv_tc_kernel": 8, "bwd_q_tc_kernel": 2,
                "fwd_simt": 4, "bwd_dkdv_simt": 8, "bwd_dq_simt": 2}
    sources = {"fwd_tc_kernel": "paged_kv_chunk_chunked_gb300/csrc/attn_tc_fwd.cu",
               "bwd_kv_tc_kernel": "paged_kv_chunk_chunked_gb300/csrc/attn_tc_bwd.cu",
               "bwd_q_tc_kernel": "paged_kv_chunk_chunked_gb300/csrc/attn_tc_bwd.cu"}
    total_prof = sum(v[1] for v in prof.values()) or 1.0
    kernels = {name: {"launches": cnt, "ms_per_step": round(ms / args.steps, 3),
                      "share": round(ms / total_prof, 4)} for name, (cnt, ms) in prof.items()}
    dom = max(prof, key=lambda k: prof[k][1])
    dom_cnt, dom_ms = prof[dom]
    roof = {
        "bound": "tensor", "unit": "TFLOP/s", "peak": peak_tc, "peak_kind": peak_kind,
        "kernel": dom,
    }
    if dom in per_step:
        ach = per_step[dom] * w.Hq * w.d * pairs_dense(w.N) * args.steps / (dom_ms * 1e-3) / 1e12
        src = sources.get(dom)
        roof.update(achieved=round(ach, 2), frac=round(ach / peak_tc, 4),
                    flops_per_launch=per_step[dom] * w.Hq * w.d * pairs_dense(w.N) * args.steps / dom_cnt,
                    ms_per_launch=round(dom_ms / dom_cnt, 4),
                    traffic=traffic_for(dom, src) if src else None)
    gpu_launches = sum(v[0] for v in prof.values())

    out = {
        "metric": METRIC, "value": round(tflops, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) Q/K/V/dO, bf16-rounded)",
        "config": dense_config(w, world),
        "tokens_per_s_per_layer": round(world * w.N / (ms_step * 1e-3), 1),
        "pct_bf16_peak": round(100 * tflops / world / peak_tc, 2),
        "fwd_ms_per_step": round(statistics.mean(fwd_ms), 3),
        "bwd_ms_per_step": round(statistics.mean(bwd_ms), 3),
        "fwd_ms_per_chunk": [round(statistics.mean(fwd_ev[k][c][0].elapsed_time(fwd_ev[k][c][1])
                                                   for k in range(args.steps)), 4) for c in range(n)],
        "bwd_ms_per_chunk": [round(statistics.mean(bwd_ev[k][c][0].elapsed_time(bwd_ev[k][c][1])
                                                   for k in range(args.steps)), 4) for c in range(n)],
        "fwd_tflops": round(fwd_ach, 2), "bwd_tflops": round(bwd_ach, 2),
        "roofline": roof,
        "kernels": kernels,
        "gpu_launches": gpu_launches,
        "clocks": clk,
    }

    if not args.no_e2e:
        out["e2e"] = run_e2e(args, w, sw, step, world)
    out["hbm_kernels"] = hbm_kernels(args, w, sw, prof, pk)
    sw.close()
    if world == 1 and not args.no_sparse:
        out["sparse"] = sparse_subrecord(args, world, rank)
    if rank == 0 and world == 1 and not args.no_cpu:
        flops, dt, desc = oracle_sample(w, REF_SAMPLE_QUERIES(w))
        out["cpu_baseline"] = {"value": round(flops / dt / 1e12, 6), "unit": UNIT,
                               "cores": cpu_threads(), "kind": "oracle", "sample": desc,
                               "seconds": round(dt, 2)}
    return out


def hbm_kernels(args, w, sw, prof, pk):
    """HBM-bound kernels of the path against the measured copy bandwidth.

    grad_accumulate_kernel: a standalone read-modify-write of the whole
    sequence's fp32 dK/dV pages (pkv_grad_accumulate over rows [0, N)), 12
    bytes per element (delta read, pool read and write). Each launch is timed
    alone with CUDA events on the launching stream, after a 512 MB write that
    flushes L2. append_kernel: from the timed step's per-kernel event times;
    per launch it reads the chunk's K and V, writes them into the pages, writes
    the representatives and zeroes the fresh pages' fp32 gradients."""
    import torch
    from paged_kv_chunk_chunked_gb300 import binding as B

    hbm = pk.get("hbm_gbs")
    stream = torch.cuda.current_stream()
    sw.reset()
    for c in range(w.n_chunks):
        s, e = w.chunk_range(c)
        B.pkv_append(sw.seq, sw.k[c], sw.v[c], e - s, stream)
    gen = torch.Generator(device="cuda").manual_seed(w.seed)
    dk = torch.randn((w.N, w.Hkv, w.d), device="cuda", generator=gen)
    dv = torch.randn((w.N, w.Hkv, w.d), device="cuda", generator=gen)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(3):
        B.pkv_grad_accumulate(sw.seq, 0, w.N, dk, dv, stream)
    n_it = max(args.steps, 5)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_it)]
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        B.pkv_grad_accumulate(sw.seq, 0, w.N, dk, dv, stream)
        b.record(stream)
    torch.cuda.synchronize()
    B.pkv_check(sw.pool)
    ms = statistics.median(a.elapsed_time(b) for a, b in evs)
    acc_bytes = 12 * w.N * w.Hkv * w.d * 2
    out = {"grad_accumulate_kernel": {
        "bound": "hbm", "unit": "GB/s", "bytes_per_launch": acc_bytes,
        "ms_per_launch": round(ms, 4), "achieved": round(acc_bytes / (ms * 1e-3) / 1e9, 1),
        "peak": hbm, "peak_kind": "measured hbm_gbs (copy, timed alone)",
        "rows": w.N, "l2": "flushed (512 MB write) before each launch",
        "traffic": traffic_for("grad_accumulate_kernel", "paged_kv_chunk_chunked_gb300/csrc/append.cu")}}
    if hbm:
        out["grad_accumulate_kernel"]["frac"] = round(out["grad_accumulate_kernel"]["achieved"] / hbm, 4)
    if "append_kernel" in prof:
        cnt, tot = prof["append_kernel"]
        el = 2 if w.dtype == "bf16" else 4
        per = w.C * w.Hkv * w.d
        a_bytes = 2 * per * el * 2 + (w.C // w.P) * w.Hkv * w.d * 4 + 2 * per * 4
        ach = a_bytes / (tot / cnt * 1e-3) / 1e9
        out["append_kernel"] = {"bound": "hbm", "unit": "GB/s", "bytes_per_launch": a_bytes,
                                "ms_per_launch": round(tot / cnt, 4), "achieved": round(ach, 1),
                                "peak": hbm, "frac": round(ach / hbm, 4) if hbm else None,
                                "peak_kind": "measured hbm_gbs (copy)"}
    del flush, dk, dv
    return out


def run_e2e(args, w, sw, step, world):
    """Same step with inputs in pinned host memory: H2D of every chunk's Q, K,
    V, dO and D2H of every chunk's dQ and the gathered dK, dV inside the
    timed region, through ChunkSweep.run_from_host (side-stream copies
    overlapped with the kernels)."""
    import torch
    host_in = [[t.cpu().pin_memory() for t in lst] for lst in (sw.q, sw.k, sw.v, sw.do)]
    host_dq = [t.cpu().pin_memory() for t in sw.dq]
    dk = torch.empty((w.N, w.Hkv, w.d), dtype=torch.float32, device="cuda")
    dv = torch.empty_like(dk)
    host_dk = torch.empty(dk.shape, dtype=torch.float32).pin_memory()
    host_dv = torch.empty_like(host_dk).pin_memory()
    h2d = sum(t.numel() * t.element_size() for lst in host_in for t in lst)
    d2h = sum(t.numel() * t.element_size() for t in host_dq) + 2 * dk.numel() * 4

    host = dict(zip(("q", "k", "v", "do"), host_in))
    out = {"dq": host_dq, "dk": host_dk, "dv": host_dv}
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_step():
        # The package's host-buffer sweep: copies overlapped with the kernels.
        sw.run_from_host(host, out, dk, dv, h2d_stream, d2h_stream)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    torch.cuda.synchronize()
    flops = 14 * w.Hq * w.d * pairs_dense(w.N)
    flops_s, ms = replica_rate(flops, (time.perf_counter() - t0) * 1e3 / args.steps, world)
    return {"value": round(flops_s / 1e12, 3), "unit": UNIT,
            "ms_per_step": round(ms, 3), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


# ------------------------------------------------------------------ reference arm (the oracle)

def REF_SAMPLE_QUERIES(w) -> int:
    """Queries of the oracle's sample (cpu_baseline and the reference arm): the
    last chunk's, one query head, against every earlier key."""
    return w.C


def run_reference(args, world, rank):
    w = bench_workload(args)
    n_q = REF_SAMPLE_QUERIES(w)
    for _ in range(args.warmup):
        oracle_sample(w, n_q)
    times, flops, desc = [], 0, ""
    for _ in range(args.steps):
        flops, dt, desc = oracle_sample(w, n_q)
        times.append(dt)
    dt = statistics.mean(times)
    val = flops / dt / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": round(val, 6), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1) Q/K/V/dO, bf16-rounded)",
        "config": dense_config(w, world),
        "cpu_baseline": {"value": round(val, 6), "unit": UNIT, "cores": cpu_threads(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(val, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------ page-sparse workloads

def sparse_pairs(sel_host, P: int, g: int) -> int:
    """Attended (query, key) pairs of one chunk for all query heads, from its
    selection [n_qp, Hkv, kmax]: P*P per listed earlier page, P(P+1)/2 for the
    query page itself (causal), times the g query heads of each KV head."""
    import numpy as np
    listed = (sel_host >= 0).sum(axis=-1)                   # [n_qp, Hkv]
    return int(g * ((listed - 1) * P * P + P * (P + 1) // 2).sum())


def run_sparse(args, world, rank):
    """Page-sparse chunk sweep: per chunk append, page top-K, sparse forward;
    then the sparse backward over the chunks in reverse. Also times the dense
    sweep of the same context once for the sparse/dense speedup."""
    import torch
    from paged_kv_chunk_chunked_gb300 import binding as B
    from paged_kv_chunk_chunked_gb300 import synth
    from paged_kv_chunk_chunked_gb300.sweep import ChunkSweep

    ensure_library(world, rank)
    w = bench_workload(args)
    K, ns, nl = w.topk if w.topk else (0,) + tuple(w.local)
    sw = ChunkSweep(w, flags=args.flags).load_inputs()
    stream = torch.cuda.current_stream()
    n = w.n_chunks
    sels = [torch.empty(((e - s + w.P - 1) // w.P, w.Hkv, K + ns + nl), dtype=torch.int32,
                        device="cuda") for s, e in (w.chunk_range(c) for c in range(n))]

    def step(sparse=True):
        sw.reset()
        for c in range(n):
            s, e = w.chunk_range(c)
            B.pkv_append(sw.seq, sw.k[c], sw.v[c], e - s, stream)
            if sparse and w.local:
                B.pkv_page_local(sw.seq, s, e - s, ns, nl, sels[c], None, stream)
            elif sparse:
                B.pkv_page_topk(sw.seq, sw.q[c], s, e - s, K, ns, nl, sels[c], None, stream)
            B.pkv_chunk_attn_fwd(sw.seq, sw.q[c], s, e - s, sw.o[c], sw.lse[c],
                                 sels[c] if sparse else None, stream)
        for c in reversed(range(n)):
            sw.backward(c, stream, sel=sels[c] if sparse else None)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    B.pkv_check(sw.pool)
    pairs = sum(sparse_pairs(x.cpu().numpy(), w.P, w.g) for x in sels)
    ev = lambda: torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    t0, t1 = ev(), ev()
    B.pkv_profile_enable(True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    prof = B.pkv_profile_collect()
    B.pkv_profile_enable(False)
    clk = clocks.stop()
    B.pkv_check(sw.pool)
    ms = t0.elapsed_time(t1) / args.steps
    # the dense sweep of the same context, once, for the speedup of page sparsity
    step(sparse=False)
    torch.cuda.synchronize()
    d0, d1 = ev(), ev()
    d0.record(stream)
    step(sparse=False)
    d1.record(stream)
    torch.cuda.synchronize()
    dense_ms = d0.elapsed_time(d1)
    flops = 14 * w.d * pairs
    flops_s, ms = replica_rate(flops, ms, world)
    tflops = flops_s / 1e12
    pk, pk_kind = peaks()
    peak_tc, peak_kind = tensor_peak(pk, pk_kind)
    kernels = {k: {"launches": c, "ms_per_step": round(t / args.steps, 3)} for k, (c, t) in prof.items()}
    # Dominant kernel (by device time) with the FLOPs it runs over the attended
    # pairs: dK/dV kernel 8 (S^T, dP^T, dV, dK), dQ kernel 6, forward 4, times d.
    units = {"bwd_kv_tc_kernel": 8, "bwd_q_tc_kernel": 6, "fwd_tc_kernel": 4}
    dom = max(prof, key=lambda k: prof[k][1])
    dom_cnt, dom_ms = prof[dom]
    dom_flops = units.get(dom, 0) * w.d * pairs * args.steps
    dom_ach = dom_flops / (dom_ms * 1e-3) / 1e12 if dom in units else None
    out = {
        "metric": METRIC, "value": round(tflops, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": f"synthetic (seeded {w.keys} keys, N(0,1) Q/V/dO, bf16-rounded)",
        "config": {"workload": w.name, "N": w.N, "C": w.C, "P": w.P, "Hq": w.Hq, "Hkv": w.Hkv,
                   "d": w.d, **({"topk": list(w.topk)} if w.topk else {"local": list(w.local)}),
                   "block_table": w.table,
                   "flops": "14*d*attended pairs (from the selections)"},
        "attended_pairs_per_step": pairs,
        "dense_pairs": w.Hq * pairs_dense(w.N),
        "tokens_per_s_per_layer": round(w.N / (ms * 1e-3), 1),
        "pct_bf16_peak": round(100 * tflops / peak_tc, 2),
        "dense_ms_per_step": round(dense_ms, 3),
        "sparse_speedup_vs_dense": round(dense_ms / ms, 2),
        "roofline": {"bound": "tensor", "kernel": dom, "unit": "TFLOP/s",
                     "achieved": round(dom_ach, 2) if dom_ach else None, "peak": peak_tc,
                     "frac": round(dom_ach / peak_tc, 4) if dom_ach else None,
                     "flops_per_launch": dom_flops / max(dom_cnt, 1),
                     "peak_kind": peak_kind, "traffic": None},
        "kernels": kernels, "gpu_launches": sum(v[0] for v in prof.values()),
        "clocks": clk,
    }
    sel = selection_record(w, prof, args.steps, pk, pk_kind, K + ns + nl)
    if sel:
        out["selection"] = sel
    return out


# Kernels of the page-selection chain (page queries, scores, top-K).
SELECTION_KERNELS = ("topk_fused_kernel",)


def selection_bytes(w, kmax: int) -> int:
    """Algorithmic bytes of one sweep's page selection: per chunk, its queries
    read once (n_q * Hq * d bf16), the representative of every candidate page
    read once (fp32 [Hkv, d]) with its block-table entry, and the selection
    written ([n_qp, Hkv, kmax] int32)."""
    K, ns, nl = w.topk
    el = 2 if w.dtype == "bf16" else 4
    total = 0
    for c in range(w.n_chunks):
        s, e = w.chunk_range(c)
        n_qp = (e - s + w.P - 1) // w.P
        n_cand = max(0, s // w.P + n_qp - 1 - nl - ns + 1)
        total += (e - s) * w.Hq * w.d * el + n_cand * (w.Hkv * w.d * 4 + 4) \
            + n_qp * w.Hkv * kmax * 4
    return total


def selection_record(w, prof, steps, pk, pk_kind, kmax):
    """HBM roofline of the page-selection chain over the timed steps: its
    algorithmic bytes against the summed event time of its kernels."""
    names = [k for k in SELECTION_KERNELS if k in prof]
    if not w.topk or not names:
        return None
    ms = sum(prof[k][1] for k in names) / steps
    byts = selection_bytes(w, kmax)
    gbs = byts / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "unit": "GB/s", "kernels": names,
            "bytes_per_step": byts, "ms_per_step": round(ms, 4),
            "us_per_chunk": round(1e3 * ms / w.n_chunks, 2),
            "achieved": round(gbs, 1), "peak": pk["hbm_gbs"],
            "frac": round(gbs / pk["hbm_gbs"], 4), "peak_kind": f"{pk_kind} hbm_gbs",
            "per_kernel_us_per_chunk": {k: round(1e3 * prof[k][1] / steps / w.n_chunks, 2)
                                        for k in names}}


def sparse_subrecord(args, world, rank):
    """The page-sparse 256K workload, shortened (args.sparse_steps timed steps,
    2 warm-up), for the dense line: its step time, TFLOP/s over attended
    pairs, the dense sweep of the same context, the dominant kernel's tensor
    roofline and the page-selection chain's HBM roofline."""
    sub = argparse.Namespace(**vars(args))
    sub.workload, sub.context = "qwen7b_sparse_256k", 0
    sub.steps, sub.warmup = max(1, args.sparse_steps), 2
    r = run_sparse(sub, world, rank)
    keep = ("value", "unit", "steps", "warmup", "ms_per_step", "config", "tokens_per_s_per_layer",
            "attended_pairs_per_step", "dense_ms_per_step", "sparse_speedup_vs_dense", "roofline",
            "selection", "page_query_roofline", "select_kernel_us_per_launch", "kernels", "clocks",
            "gpu_launches")
    return {k: r[k] for k in keep if k in r}


def run_topk_error_study(args, world, rank):
    """Gradient approximation error of page-level top-K against its budget.

    One dense sweep and one sparse sweep per K of the same seeded workload,
    all on the GPU through the library; errors are relative Frobenius norms of
    the sparse result against the dense one over the whole sequence (O, dQ of
    every chunk; dK, dV of the whole gradient pool). The pages report that the
    gradient error stays small at adequate retrieval budgets (gist.science/de
    §4 "Genauigkeit"; gist.science/ja §4). Also the device bytes the paged
    pool took against what its pages need (the pages' Fig. 4: a non-paged
    cache can take ~3x the theoretical requirement)."""
    import numpy as np
    import torch
    from paged_kv_chunk_chunked_gb300 import binding as B
    from paged_kv_chunk_chunked_gb300 import synth
    from paged_kv_chunk_chunked_gb300.sweep import ChunkSweep, to_device

    ensure_library(world, rank)
    name = args.workload if synth.workload(args.workload).topk else "qwen7b_sparse_256k"
    w = synth.workload(name)
    _, ns, nl = w.topk
    ChunkSweep(synth.workload("tiny_dense_f32")).load_inputs([0]).close()   # device code loaded
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    sw = ChunkSweep(w).load_inputs([])
    torch.cuda.synchronize()
    pool_bytes = free0 - torch.cuda.mem_get_info()[0]
    el = 2 if w.dtype == "bf16" else 4
    need = w.n_phys * w.Hkv * w.P * w.d * (2 * el + 2 * 4) + w.n_phys * w.Hkv * w.d * 4
    sw.load_inputs()
    stream = torch.cuda.current_stream()

    def sweep(K):
        sw.reset()
        sels = []
        for c in range(w.n_chunks):
            s, e = w.chunk_range(c)
            B.pkv_append(sw.seq, sw.k[c], sw.v[c], e - s, stream)
            sel = None
            if K is not None:
                sel = torch.empty(((e - s + w.P - 1) // w.P, w.Hkv, K + ns + nl),
                                  dtype=torch.int32, device="cuda")
                B.pkv_page_topk(sw.seq, sw.q[c], s, e - s, K, ns, nl, sel, None, stream)
            sels.append(sel)
            B.pkv_chunk_attn_fwd(sw.seq, sw.q[c], s, e - s, sw.o[c], sw.lse[c], sel, stream)
        for c in reversed(range(w.n_chunks)):
            sw.backward(c, stream, sel=sels[c])
        g = sw.gather()
        pairs = sum(sparse_pairs(x.cpu().numpy(), w.P, w.g) for x in sels) if K is not None \
            else w.Hq * pairs_dense(w.N)
        return (torch.cat([x.float() for x in sw.o]), torch.cat([x.float() for x in sw.dq]),
                g["dk"], g["dv"], pairs)

    rel = lambda a, b: float(torch.linalg.vector_norm(a - b) / torch.linalg.vector_norm(b))
    rows = []
    for queries in ("normal", "coherent"):
        sw.w = w = w.with_(queries=queries)
        sw.q = [to_device(synth.chunk_q(w, c), w.dtype) for c in range(w.n_chunks)]
        dense = sweep(None)
        for K in (4, 8, 16, 32, 64, 128, 256):
            sp = sweep(K)
            rows.append({"queries": queries, "K": K,
                         "attended_frac": round(sp[4] / dense[4], 5),
                         **{f"{n}_rel": round(rel(a, b), 5)
                            for n, a, b in zip(("o", "dq", "dk", "dv"), sp[:4], dense[:4])}})
            del sp
        del dense
    B.pkv_check(sw.pool)
    sw.close()
    return {"study": "topk_gradient_error", "workload": w.name, "n_sink": ns, "n_local": nl,
            "data": "synthetic (seeded clustered keys; queries N(0,1) ('normal') or a "
                    "(query page, KV group) centre N(0,1) + N(0,1) ('coherent'); V, dO "
                    "N(0,1); bf16-rounded)",
            "error": "relative Frobenius norm, sparse vs dense, both on the GPU",
            "rows": rows,
            "memory": {"pool_device_bytes": int(pool_bytes), "page_bytes_needed": int(need),
                       "ratio": round(pool_bytes / need, 4),
                       "what": "K, V, dK, dV pages and representatives of the context"}}


def run_layer_loop(args, world, rank):
    """Chunk-recurrent training of one attention block (``layer.ChunkRecurrentBlock``):
    forward chunk by chunk, backward in reverse with the chunk's Q and attention
    recomputed; projections are cuBLAS GEMMs, attention runs in the library.
    Per context length: step time, tokens/s, the bytes of the paged pool, and
    the transient device memory of a step beyond its inputs and outputs, which
    the pages say chunk-recurrent recomputation keeps constant in the context
    (gist.science/de §2.A; sciencestack.ai Fig. 1 caption)."""
    import torch
    from paged_kv_chunk_chunked_gb300 import binding as B
    from paged_kv_chunk_chunked_gb300 import synth
    from paged_kv_chunk_chunked_gb300.layer import ChunkRecurrentBlock
    from paged_kv_chunk_chunked_gb300.sweep import to_device

    ensure_library(world, rank)
    w0 = synth.workload(args.workload)
    hidden = 3584
    ChunkRecurrentBlock(w0.with_(N=w0.C), 64).close()     # device code loaded before measuring
    contexts = [args.context] if args.context else [32768, 65536, 131072]
    rows = []
    for N in contexts:
        w = w0.with_(N=N)
        blk = ChunkRecurrentBlock(w, hidden)
        pool_bytes = blk.pool_device_bytes
        xs = [to_device(synth.block_x(w, c, hidden), w.dtype) for c in range(w.n_chunks)]
        dys = [to_device(synth.block_dy(w, c, hidden), w.dtype) for c in range(w.n_chunks)]
        for _ in range(args.warmup):
            ys = blk.forward(xs)
            dxs, g = blk.backward(xs, dys)
            del ys, dxs, g
        torch.cuda.synchronize()
        B.pkv_check(blk.pool)
        torch.cuda.reset_peak_memory_stats()
        base = torch.cuda.memory_allocated()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        out_bytes = 0
        for _ in range(args.steps):
            ys = blk.forward(xs)
            dxs, g = blk.backward(xs, dys)
            out_bytes = sum(t.numel() * t.element_size() for t in ys + dxs) + \
                sum(t.numel() * 4 for t in g.values())
            del ys, dxs, g
        b.record()
        torch.cuda.synchronize()
        B.pkv_check(blk.pool)
        ms = a.elapsed_time(b) / args.steps
        peak = torch.cuda.max_memory_allocated() - base
        rows.append({"N": N, "ms_per_step": round(ms, 3),
                     "tokens_per_s": round(N / (ms * 1e-3), 1),
                     "kv_pool_bytes": int(pool_bytes),
                     "kv_pool_bytes_per_token": round(pool_bytes / N, 1),
                     "step_transient_bytes": int(peak - out_bytes),
                     "step_output_bytes": int(out_bytes)})
        blk.close()
        del xs, dys
        torch.cuda.empty_cache()
    return {"metric": "chunk-recurrent training step of one attention block: time and device memory vs context",
            "unit": "ms/step", "value": rows[-1]["ms_per_step"], "higher_is_better": False,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "dtype": w0.dtype,
            "data": "synthetic (seeded N(0,1) inputs and upstream gradients, random weights)",
            "config": {"workload": w0.name, "C": w0.C, "P": w0.P, "Hq": w0.Hq, "Hkv": w0.Hkv,
                       "d": w0.d, "hidden": hidden, "block": "x + attention(x wq, x wk, x wv) wo"},
            "rows": rows,
            "memory_note": "step_transient_bytes = peak torch allocation during a step minus the "
                           "step's outputs (y, dx, weight gradients); the paged pool is outside "
                           "torch's allocator and reported separately"}


def run_offload(args, world, rank):
    """Pinned-host offload of the 1M-token page-sparse workload. All 128 chunks'
    K/V are appended into pinned host pages; the measured step is the sparse
    forward + backward of the last `--offload-chunks` chunks. Each chunk stages
    its selected pages (K/V, then K/V + gradients) into the sequence's slot
    cache on a side stream: pages already staged by an earlier chunk stay, so
    only the difference crosses the host link; the gradients go back once, at
    the end of the backward sweep, when the step releases the slots (every
    step starts with an empty cache). Each step first zeroes the gradient
    pool, as a training step does: on the device-resident pool a write of
    every gradient page, on the pinned-host pool a per-page record in HBM, so
    the backward's first staging of a page fills zeros in HBM instead of
    copying stale host pages. The same step on a device-resident pool gives
    the staging overhead.

    --overlap-proj adds the computations the pages overlap with the transfer
    (gist.science/de §2.C: with sparse attention, the key/value projections
    that follow): the next chunk's Q and K/V projections while a chunk's pages
    stream in for its forward, and the chunk's recomputed projections while
    its pages and gradients stream in for its backward (bf16 cuBLAS GEMMs,
    hidden 3584). It reports the copy time (the staging kernels' own event time), the
    part of it the step exposes (pinned-host step minus device-resident step,
    both with the GEMMs) and overlap = 1 - exposed / copy time."""
    import numpy as np
    import torch
    from paged_kv_chunk_chunked_gb300 import binding as B
    from paged_kv_chunk_chunked_gb300 import synth
    from paged_kv_chunk_chunked_gb300.sweep import to_device

    ensure_library(world, rank)
    w = bench_workload(args)
    K, ns, nl = w.topk
    n = w.n_chunks
    meas = list(range(n - args.offload_chunks, n))
    main_s = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    bt = synth.block_table(w)
    if args.slots <= 0:
        args.slots = w.n_pages
    hidden = 3584
    res = {}
    for mode in ("pinned_host", "device"):
        host = mode == "pinned_host"
        pool = B.pkv_pool_create(w.P, w.Hkv, w.Hq, w.d, B.PKV_BF16, w.n_phys,
                                 residency=B.PKV_RES_PINNED_HOST if host else B.PKV_RES_DEVICE,
                                 n_device_slots=args.slots if host else 0)
        seq = B.pkv_seq_create(pool)
        q = {c: to_device(synth.chunk_q(w, c), "bf16") for c in meas}
        do = {c: to_device(synth.chunk_do(w, c), "bf16") for c in meas}
        o = {c: torch.empty_like(q[c]) for c in meas}
        dq = {c: torch.empty_like(q[c]) for c in meas}
        lse = {c: torch.empty((w.Hq, w.C), dtype=torch.float32, device="cuda") for c in meas}
        sel = {c: torch.empty((w.C // w.P, w.Hkv, K + ns + nl), dtype=torch.int32, device="cuda")
               for c in meas}
        # synthetic projections of a chunk (Qwen2.5-7B: hidden 3584; K/V 2 x Hkv x d
        # columns, Q Hq x d), random weights; plain cuBLAS GEMMs on the main stream
        gen = torch.Generator(device="cuda").manual_seed(w.seed)
        x_proj = torch.randn((w.C, hidden), device="cuda", generator=gen).to(torch.bfloat16)
        w_kv = (torch.randn((hidden, 2 * w.Hkv * w.d), device="cuda", generator=gen) / 60.0).to(torch.bfloat16)
        w_q = (torch.randn((hidden, w.Hq * w.d), device="cuda", generator=gen) / 60.0).to(torch.bfloat16)

        def fill():
            B.pkv_seq_reset(seq)
            B.pkv_set_block_table(seq, bt)
            for c in range(n):
                s, e = w.chunk_range(c)
                k = to_device(synth.chunk_k(w, c), "bf16")
                v = to_device(synth.chunk_v(w, c), "bf16")
                B.pkv_append(seq, k, v, e - s, main_s)
            torch.cuda.synchronize()

        mk = lambda: torch.cuda.Event(enable_timing=True)

        def step(proj=False, rec=None):
            """rec: dict collecting per-chunk event pairs (main-stream span of
            the chunk from its prefetch to its attention call; side-stream span
            of its staging)."""
            B.pkv_grad_zero(seq, main_s)      # a training step starts from zero gradients
            for phase, chunks in (("fwd", meas), ("bwd", list(reversed(meas)))):
                for c in chunks:
                    s, e = w.chunk_range(c)
                    if phase == "fwd":
                        B.pkv_page_topk(seq, q[c], s, e - s, K, ns, nl, sel[c], None, main_s)
                    m0, m1, c0, c1 = mk(), mk(), mk(), mk()
                    if rec is not None:
                        m0.record(main_s)
                    if host:
                        if rec is not None:
                            side.wait_stream(main_s)
                            c0.record(side)
                        what = B.PKV_STAGE_KV if phase == "fwd" else B.PKV_STAGE_KV | B.PKV_STAGE_GRADS
                        B.pkv_prefetch(seq, sel[c], sel[c].numel(), what, side)
                        if rec is not None:
                            c1.record(side)
                    if proj:      # fwd: the next chunk's Q, K, V projections; bwd: the recomputed ones
                        torch.matmul(x_proj, w_q)
                        torch.matmul(x_proj, w_kv)
                    if host:
                        B.pkv_wait(seq, main_s, 0)
                    if phase == "fwd":
                        B.pkv_chunk_attn_fwd(seq, q[c], s, e - s, o[c], lse[c], sel[c], main_s)
                    else:
                        B.pkv_chunk_attn_bwd(seq, q[c], o[c], do[c], lse[c], s, e - s, dq[c], sel[c], main_s)
                    if rec is not None:
                        m1.record(main_s)
                        rec.setdefault(phase, []).append((m0, m1, c0, c1) if host else (m0, m1))
            if host:
                B.pkv_release_slots(seq, side)        # gradients back once; cold cache next step
                B.pkv_wait(seq, main_s, 0)

        fill()
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        B.pkv_check(pool)
        st0 = B.pkv_stage_stats(seq) if host else None
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        clocks = ClockSampler(torch.cuda.current_device())
        clocks.start()
        B.pkv_profile_enable(True)
        ev0.record(main_s)
        for _ in range(args.steps):
            step()
        ev1.record(main_s)
        torch.cuda.synchronize()
        prof = B.pkv_profile_collect()
        B.pkv_profile_enable(False)
        clk = clocks.stop()
        B.pkv_check(pool)
        res[mode] = dict(ms=ev0.elapsed_time(ev1) / args.steps, prof=prof, clocks=clk)
        if host:
            st1 = B.pkv_stage_stats(seq)
            res[mode]["moved"] = {k: (st1[k] - st0[k]) / args.steps for k in st1}
            res[mode]["union_pages"] = sum(int((np.unique(sel[c].cpu().numpy()) >= 0).sum())
                                           for c in meas)
        if args.overlap_proj:
            step(proj=True)
            B.pkv_profile_enable(True)
            ev0.record(main_s)
            for _ in range(args.steps):
                step(proj=True)
            ev1.record(main_s)
            torch.cuda.synchronize()
            res[mode]["prof_proj"] = B.pkv_profile_collect()
            B.pkv_profile_enable(False)
            B.pkv_check(pool)
            res[mode]["ms_proj"] = ev0.elapsed_time(ev1) / args.steps
            rec = {}
            step(proj=True, rec=rec)
            torch.cuda.synchronize()
            res[mode]["chunks"] = {ph: [[round(ev[0].elapsed_time(ev[1]), 4)] +
                                        ([round(ev[2].elapsed_time(ev[3]), 4)] if host else [])
                                        for ev in evs] for ph, evs in rec.items()}
            if not host:      # the step's GEMMs alone, back to back
                ev0.record(main_s)
                for _ in range(args.steps):
                    for _c in range(2 * len(meas)):
                        torch.matmul(x_proj, w_q)
                        torch.matmul(x_proj, w_kv)
                ev1.record(main_s)
                torch.cuda.synchronize()
                res[mode]["gemm_ms"] = ev0.elapsed_time(ev1) / args.steps
        B.pkv_pool_destroy(pool)
        del q, do, o, dq, lse, sel
        torch.cuda.empty_cache()
    hp = res["pinned_host"]
    kv_ph = w.P * w.d * 2 * 2          # K + V of one page of one KV head
    g_ph = w.P * w.d * 4 * 2           # dK + dV
    mv = hp["moved"]
    bytes_moved = mv["kv_in"] * kv_ph + (mv["grads_in"] + mv["grads_out"]) * g_ph
    # without the slot cache: every chunk's selection staged afresh, K/V for the
    # forward, K/V and gradients in and gradients out for the backward
    bytes_afresh = hp["union_pages"] * w.Hkv * (2 * kv_ph + 2 * g_ph)
    stage_names = ("stage_plan_kernel", "stage_copy_kernel", "stage_writeback_kernel")

    def copy_ms(prof):
        return sum(prof.get(k, (0, 0.0))[1] for k in stage_names) / args.steps

    overhead = hp["ms"] / res["device"]["ms"] - 1.0
    extra = {}
    if args.overlap_proj:
        cp = copy_ms(hp["prof_proj"])
        exposed = hp["ms_proj"] - res["device"]["ms_proj"]
        # Per chunk with a warm slot cache (every chunk but the first of each
        # sweep): main-stream time pinned-host minus device-resident (the
        # exposed part of the staging) against the staging's own time.
        per = {}
        for ph in ("fwd", "bwd"):
            hc, dc = hp["chunks"][ph], res["device"]["chunks"][ph]
            cp_w = sum(x[1] for x in hc[1:])
            ex_w = sum(max(0.0, hx[0] - dx[0]) for hx, dx in zip(hc[1:], dc[1:]))
            per[ph] = {"copy_ms_per_chunk": [x[1] for x in hc],
                       "exposed_ms_per_chunk": [round(hx[0] - dx[0], 4) for hx, dx in zip(hc, dc)],
                       "warm_copy_ms": round(cp_w, 4), "warm_exposed_ms": round(ex_w, 4),
                       "warm_overlap": round(1.0 - ex_w / cp_w, 3) if cp_w > 0 else None}
        extra["projection_overlap_per_chunk"] = per
        extra["projection_overlap"] = {
            "gemms": f"per measured chunk and sweep: a chunk's Q and K/V projections [{w.C}, {hidden}] x "
                     f"[{hidden}, {w.Hq * w.d}] and x [{hidden}, {2 * w.Hkv * w.d}] (the next chunk's in "
                     f"the forward, the recomputed ones in the backward), cuBLAS bf16",
            "gemm_ms_per_step": round(res["device"]["gemm_ms"], 3),
            "copy_ms_per_step": round(cp, 3),
            "ms_per_step_pinned_host_with_projection": round(hp["ms_proj"], 3),
            "ms_per_step_device_with_projection": round(res["device"]["ms_proj"], 3),
            "exposed_copy_ms_per_step": round(exposed, 3),
            "overlap": round(1.0 - exposed / cp, 3) if cp > 0 else None}
    return {
        "metric": "page-sparse offload step: staged pages over the host link, overhead vs HBM-resident",
        "value": round(overhead * 100, 2), "unit": "% step-time overhead", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": False,
        "ms_per_step_pinned_host": round(hp["ms"], 3), "ms_per_step_device": round(res["device"]["ms"], 3),
        "config": {"workload": w.name, "N": w.N, "C": w.C, "P": w.P, "Hq": w.Hq, "Hkv": w.Hkv,
                   "d": w.d, "topk": list(w.topk), "measured_chunks": meas, "device_slots": args.slots},
        "page_heads_moved_per_step": mv, "bytes_moved_per_step": bytes_moved,
        "bytes_per_step_without_slot_cache": bytes_afresh,
        "copy_ms_per_step": round(copy_ms(hp["prof"]), 3),
        "link_gbs_in_copy_kernels": round(bytes_moved / (copy_ms(hp["prof"]) * 1e-3) / 1e9, 1)
        if copy_ms(hp["prof"]) > 0 else None,
        "kernels_pinned_host": {k: {"launches": c, "ms_per_step": round(t / args.steps, 3)}
                                for k, (c, t) in hp["prof"].items()},
        "data": "synthetic (seeded clustered keys)",
        "clocks": {"pinned_host": hp["clocks"], "device": res["device"]["clocks"]},
        **extra,
    }


def run_offload_dense(args, world, rank):
    """Dense offload across layers: every layer's K/V pages and fp32 gradient
    pages live in pinned host memory. The measured step is the last chunk's
    forward + backward in each of L layers; layer l + 1's pages (K, V, dK, dV)
    are staged into its HBM slots on a side stream while layer l computes, and
    layer l's gradients go back after it. The same step with HBM-resident
    layers gives the overhead."""
    import torch
    from paged_kv_chunk_chunked_gb300 import binding as B
    from paged_kv_chunk_chunked_gb300 import synth
    from paged_kv_chunk_chunked_gb300.sweep import to_device

    ensure_library(world, rank)
    w = bench_workload(args)
    L = args.offload_layers
    c = w.n_chunks - 1
    s, e = w.chunk_range(c)
    main_s = torch.cuda.current_stream()
    side, side_out = torch.cuda.Stream(), torch.cuda.Stream()   # host-to-device, device-to-host
    q = to_device(synth.chunk_q(w, c), w.dtype)
    do = to_device(synth.chunk_do(w, c), w.dtype)
    o, dq = torch.empty_like(q), torch.empty_like(q)
    lse = torch.empty((w.Hq, e - s), dtype=torch.float32, device="cuda")
    kv = [(to_device(synth.chunk_k(w, i), w.dtype), to_device(synth.chunk_v(w, i), w.dtype))
          for i in range(w.n_chunks)]
    res, clk = {}, {}
    for mode in ("pinned_host", "device"):
        host = mode == "pinned_host"
        pools, seqs = [], []
        for _ in range(L):
            pool = B.pkv_pool_create(w.P, w.Hkv, w.Hq, w.d, B.PKV_BF16, w.n_phys,
                                     residency=B.PKV_RES_PINNED_HOST if host else B.PKV_RES_DEVICE,
                                     n_device_slots=w.n_pages if host else 0)
            seq = B.pkv_seq_create(pool)
            for i, (k_, v_) in enumerate(kv):
                a, b_ = w.chunk_range(i)
                B.pkv_append(seq, k_, v_, b_ - a, main_s)
            pools.append(pool)
            seqs.append(seq)
        torch.cuda.synchronize()

        def step():
            if host:
                B.pkv_prefetch(seqs[0], None, 0, B.PKV_STAGE_KV | B.PKV_STAGE_GRADS, side)
            for l in range(L):
                if host:
                    if l + 1 < L:
                        B.pkv_prefetch(seqs[l + 1], None, 0, B.PKV_STAGE_KV | B.PKV_STAGE_GRADS, side)
                    B.pkv_wait(seqs[l], main_s, 0)
                B.pkv_chunk_attn_fwd(seqs[l], q, s, e - s, o, lse, None, main_s)
                B.pkv_chunk_attn_bwd(seqs[l], q, o, do, lse, s, e - s, dq, None, main_s)
                if host:
                    B.pkv_writeback_grads(seqs[l], side_out)
            if host:
                for l in range(L):
                    B.pkv_wait(seqs[l], main_s, 0)

        for _ in range(max(1, args.warmup)):
            step()
        torch.cuda.synchronize()
        for pool in pools:
            B.pkv_check(pool)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        clocks = ClockSampler(torch.cuda.current_device())
        clocks.start()
        ev0.record(main_s)
        for _ in range(args.steps):
            step()
        ev1.record(main_s)
        torch.cuda.synchronize()
        clk[mode] = clocks.stop()
        for pool in pools:
            B.pkv_check(pool)
        res[mode] = ev0.elapsed_time(ev1) / args.steps
        for pool in pools:
            B.pkv_pool_destroy(pool)
    page_kv = w.Hkv * w.P * w.d * 2 * 2
    page_g = w.Hkv * w.P * w.d * 4 * 2
    bytes_moved = L * w.n_pages * (page_kv + 2 * page_g)
    overhead = res["pinned_host"] / res["device"] - 1.0
    return {
        "metric": "dense layer offload: next layer's pages staged over the host link while the "
                  "current layer computes, overhead vs HBM-resident",
        "value": round(overhead * 100, 2), "unit": "% step-time overhead", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": False,
        "ms_per_step_pinned_host": round(res["pinned_host"], 3),
        "ms_per_step_device": round(res["device"], 3),
        "config": {"workload": w.name, "N": w.N, "C": w.C, "P": w.P, "Hq": w.Hq, "Hkv": w.Hkv,
                   "d": w.d, "layers": L, "measured_chunk": c},
        "bytes_moved_per_step": bytes_moved,
        "link_gbs_needed_to_hide": round(bytes_moved / (res["device"] * 1e-3) / 1e9, 1),
        "data": "synthetic (seeded N(0,1) K/V/Q/dO, the same for every layer)",
        "clocks": clk,
    }


def json_safe(x):
    """The result with every non-finite float replaced by None: the line must
    be strict JSON (NaN and Infinity are not)."""
    if isinstance(x, float):
        return x if math.isfinite(x) else None
    if isinstance(x, dict):
        return {k: json_safe(v) for k, v in x.items()}
    if isinstance(x, (list, tuple)):
        return [json_safe(v) for v in x]
    return x


def main():
    args = parse_args()
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return 0
        print(json.dumps(json_safe(run_reference(args, int(os.environ.get("WORLD_SIZE", "1")), rank)), allow_nan=False))
        return 0
    world, rank, _ = dist_setup(args)
    from paged_kv_chunk_chunked_gb300 import synth
    wl = bench_workload(args)
    if args.study == "topk-error":
        out = run_topk_error_study(args, world, rank)
    elif args.layer_loop:
        out = run_layer_loop(args, world, rank)
    elif args.offload_layers > 0:
        out = run_offload_dense(args, world, rank)
    elif wl.offload:
        out = run_offload(args, world, rank)
    elif wl.topk or wl.local:
        out = run_sparse(args, world, rank)
    else:
        out = run_pkv(args, world, rank)
    if rank == 0:
        print(json.dumps(json_safe(out), allow_nan=False), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

#!/usr/bin/env python3
"""Benchmark: DSA-layer forward+backward tokens/s on one GB300.

Workload (default): the L=131072 bf16 layer with a 10% needle -- Hq=16 query
heads sharing one K/V head of d=128, an indexer of 8 heads x 64, 32768 pools
of 4 tokens, top-512 pools per query, indexer chunks of 8192 queries.
Synthetic seeded inputs (dsa_inputs.py); no dataset, no trained weights.

One step = the whole layer: pool keys, for each 8192-query chunk the fused
indexer scores + top-k selection, sparse attention forward, then the backward
(dQ, dK, dV).  It calls the C-ABI entry points one by one on one stream, with CUDA
events between them, so the per-kernel durations (and the roofline of the
dominant kernel) are measured live in the same run.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

--impl reference times the CPU oracle (fp64, single thread, on this host's
cores) on a bounded sample of the same workload: that is the only place the
benchmark runs the oracle.  With N > 1 (torchrun), every rank runs an
independent replica of the layer (the layer has no exchange step on one
GPU); value = the sum over ranks of tokens / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import dsa_inputs  # noqa: E402

METRIC = "DSA-layer tokens/s fwd+bwd at L=128k on 1 GB300"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return {k: float(j[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(PEAKS_FALLBACK), "fallback"


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one
# ncu capture of the bench at the full 128k workload (one-pass metrics).  A
# figure is reported only while the kernel's source files hash as they did
# when it was captured; after any change to them the bench reports null until
# it is captured again.
TRAFFIC = {
    ("bf16_128k_needle", "attn_bwd"): {"bytes": 11616282624 + 9580551936,
                                       "sources": {"attn_bwd.cu": "6114a89bda28ac3a", "gather.cuh": "9c5588b13d0916cd", "common.cuh": "4c65dfd5da7caf78"}},
    ("bf16_128k_needle", "attn_fwd"): {"bytes": 1271921920 + 1564575744,
                                       "sources": {"attn_fwd.cu": "ffdff854d43dc7cb", "gather.cuh": "9c5588b13d0916cd", "common.cuh": "4c65dfd5da7caf78"}},
    # mean over the 16 chunk launches of one step
    ("bf16_128k_needle", "indexer"): {"bytes": 36841456 + 477152544,
                                      "sources": {"indexer_tc.cu": "4152b6e7fe6b5292", "common.cuh": "4c65dfd5da7caf78"}},
    ("bf16_128k_needle", "topk"): {"bytes": 538500512 + 11403616,
                                   "sources": {"topk.cu": "7e34eb4699bcd34b", "common.cuh": "4c65dfd5da7caf78"}},
}


def measured_traffic(workload: str, kernel: str):
    import hashlib
    rec = TRAFFIC.get((workload, kernel))
    if rec is None:
        return None
    csrc = os.path.join(ROOT, "long_context_sparse_dsa_gb300", "csrc")
    for name, digest in rec["sources"].items():
        try:
            with open(os.path.join(csrc, name), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest()[:16] != digest:
                    return None
        except OSError:
            return None
    return rec["bytes"]


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ algorithmic work
def algorithmic(wl):
    """Per-launch algorithmic bytes / flops of each kernel (causal, selected work only)."""
    L, P, k, Hq, d, Hi, di = wl.L, wl.P, wl.k, wl.Hq, wl.d, wl.Hi, wl.di
    t = torch.arange(L, dtype=torch.float64)
    elig = torch.floor((t + 1) / 4)
    pairs = float(elig.sum())
    partial = torch.where(t % 4 == 3, 0.0, t % 4 + 1)
    nkeys = float((4 * torch.minimum(elig, torch.tensor(float(k))) + partial).sum())
    eb = 2 if wl.dtype == "bf16" else 4
    # with a backward the forward also writes the fp32 output (o_acc) and the
    # backward reads it instead of re-forming D from K and V
    acc = 4.0 * L * Hq * d if wl.passes == "fwd+bwd" else 0.0
    return {
        "pool_keys": {"bytes": L * di * eb + P * di * eb},
        "indexer": {"flops": 2.0 * Hi * di * pairs, "score_bytes": 4.0 * pairs},
        "topk": {"bytes": 4.0 * pairs + 4.0 * L * k},
        # gathered K and V rows; Q read, O written, idx read, LSE written
        "attn_fwd": {"bytes": nkeys * 2 * d * eb + L * Hq * d * eb * 2 + L * k * 4 + L * Hq * 4 + acc,
                     "l2_bytes": nkeys * 2 * d * eb,
                     "flops": 4.0 * Hq * d * nkeys},
        # gathered K and V rows, fp32 dK and dV reductions; Q, dO, o_acc read, dQ written; idx, LSE read
        "attn_bwd": {"bytes": nkeys * 2 * d * eb + nkeys * 2 * d * 4 + L * Hq * d * (2 * eb + 4) + acc
                     + L * k * 4 + L * Hq * 4,
                     "l2_bytes": nkeys * 2 * d * eb + nkeys * 2 * d * 4,
                     "flops": 10.0 * Hq * d * nkeys},
        "nkeys": nkeys, "pairs": pairs,
    }


# ------------------------------------------------------------ replicas
def aggregate_replicas(local_ms: float, local_tokens: int, world: int, device=None):
    """Whole-job throughput of N independent replicas: every rank's tokens
    divided by the slowest rank's time.  Returns (tokens/s, max ms, tokens)."""
    if world > 1:
        t = torch.tensor([local_ms, float(local_tokens)], dtype=torch.float64, device=device)
        mx = t[:1].clone()
        torch.distributed.all_reduce(mx, op=torch.distributed.ReduceOp.MAX)
        tot = t[1:].clone()
        torch.distributed.all_reduce(tot, op=torch.distributed.ReduceOp.SUM)
        local_ms, local_tokens = float(mx.item()), int(tot.item())
    return local_tokens / (local_ms / 1e3), local_ms, local_tokens


# -------------------------------------------------------------------- ours
def run_ours(args, rank, world):
    import long_context_sparse_dsa_gb300 as dsa
    from long_context_sparse_dsa_gb300 import build as lib_build

    wl = dsa_inputs.WORKLOADS[args.workload]
    with_bwd = wl.passes == "fwd+bwd"
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or not os.path.exists(dsa.LIB_PATH):
        lib_build.build()
    if world > 1:
        torch.distributed.barrier()
    dsa.library()

    names = ("Q", "K", "V", "q_I", "k_I", "w") + (("dO",) if with_bwd else ())
    torch.cuda.reset_peak_memory_stats(dev)
    host = dsa_inputs.make(wl, names, pin=True)
    inputs_sha = inputs_digest(host, names)
    d_in = {n: host[n].to(dev, non_blocking=True) for n in names}
    dims = dsa.make_dims(wl.L, wl.Hq, wl.d, wl.Hi, wl.di, wl.k, q_chunk=wl.q_chunk, scale=wl.scale, dtype=wl.dtype)
    # with a backward, the forward keeps its fp32 output for it (the backward
    # then forms D from it and needs no workspace)
    bufs = dsa.alloc_forward_buffers(dims, dev, o_acc=with_bwd)
    dq = torch.empty((wl.L, wl.Hq, wl.d), device=dev) if with_bwd else None
    dk = torch.empty((wl.L, wl.d), device=dev) if with_bwd else None
    dv = torch.empty((wl.L, wl.d), device=dev) if with_bwd else None
    dsa.set_indexer_topk_route(args.indexer_route)
    dsa.set_attn_fwd_route(args.attn_fwd_route)
    det = with_bwd and args.backward == "det"
    bws = dsa.alloc_bwd_det_workspace(dims, dev) if det else None
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # 256 MiB > L2
    stream = torch.cuda.current_stream(dev)
    C = wl.q_chunk
    chunks = [(q0, min(C, wl.L - q0)) for q0 in range(0, wl.L, C)]
    # kernels per step: pool keys; per chunk the fused indexer + top-k (sampled
    # scores when the chunk has rows of more than 2048 pools, thresholds,
    # candidates, selection, fallback scores, fallback top-k; fp32 layers: the
    # indexer and the top-k); the forward; the backward
    # per chunk: route 1 (and fp32 layers) the indexer and the top-k; route 0
    # the sampled scores when a row has more than 2048 pools, thresholds,
    # candidate indexer, selection, fallback indexer, fallback top-k
    if wl.dtype != "bf16" or args.indexer_route == 1:
        per_chunk = [2 for _ in chunks]
    else:
        per_chunk = [(1 if ((q0 + n) >> 2) > 2048 else 0) + 5 for q0, n in chunks]
    # the deterministic backward: dQ pass, 5 inversion kernels, 3 per 4096-query band
    bwd_launches = (1 + 5 + 3 * ((wl.L + 4095) // 4096)) if det else 1
    launches_per_step = 1 + sum(per_chunk) + 1 + (bwd_launches if with_bwd else 0)

    split_pair = args.indexer_route == 1 or wl.dtype != "bf16"
    scores = bufs.ws.view(torch.float32)   # the score block of route 1 (the workspace holds it)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    def step(timers=None):
        marks = []
        if timers is not None:
            marks.append(("start", timers.pop()))
            marks[-1][1].record(stream)
        dsa.pool_keys(dims, d_in["k_I"], bufs.kpool, stream)
        if timers is not None:
            marks.append(("pool_keys", timers.pop()))
            marks[-1][1].record(stream)
        for q0, n in chunks:
            if split_pair:
                # route 1 is the indexer's score block and the row-wise top-k:
                # the same two kernels through their own entry points, so that
                # each gets its own time and roofline
                dsa.indexer_score(dims, d_in["q_I"], bufs.kpool, d_in["w"], q0, n, scores, stream=stream)
                if timers is not None:
                    marks.append(("indexer", timers.pop()))
                    marks[-1][1].record(stream)
                dsa.topk(dims, scores, q0, n, bufs.idx, stream=stream)
                if timers is not None:
                    marks.append(("topk", timers.pop()))
                    marks[-1][1].record(stream)
                continue
            dsa.indexer_topk(dims, d_in["q_I"], bufs.kpool, d_in["w"], q0, n, bufs.idx, bufs.ws, stream=stream)
            if timers is not None:
                marks.append(("indexer_topk", timers.pop()))
                marks[-1][1].record(stream)
        dsa.sparse_attn_fwd(dims, d_in["Q"], d_in["K"], d_in["V"], bufs.idx, bufs.o, bufs.lse, stream,
                            o_acc=bufs.o_acc)
        if timers is not None:
            marks.append(("attn_fwd", timers.pop()))
            marks[-1][1].record(stream)
        if with_bwd:
            if det:
                dsa.sparse_attn_bwd_det(dims, d_in["Q"], d_in["K"], d_in["V"], bufs.idx, bufs.o, bufs.lse,
                                        d_in["dO"], dq, dk, dv, bws, None, stream, o_acc=bufs.o_acc)
            else:
                dsa.sparse_attn_bwd(dims, d_in["Q"], d_in["K"], d_in["V"], bufs.idx, bufs.o, bufs.lse, d_in["dO"],
                                    dq, dk, dv, bws, None, stream, o_acc=bufs.o_acc)
            if timers is not None:
                marks.append(("attn_bwd_det" if det else "attn_bwd", timers.pop()))
                marks[-1][1].record(stream)
        return marks

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    dsa.check_device_error(stream)

    per_kernel = {}
    step_ms = []
    n_marks = 2 + 2 * len(chunks) + 2 + 1
    with ClockSampler(local) as clk:
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        for _ in range(args.steps):
            flush.fill_(1)                                  # evict L2 between steps (outside the events)
            timers = [ev() for _ in range(n_marks)]
            marks = step(timers)
            torch.cuda.synchronize(dev)
            for (nm, e0), (nm1, e1) in zip(marks[:-1], marks[1:]):
                per_kernel.setdefault(nm1, []).append(e0.elapsed_time(e1))
            step_ms.append(marks[0][1].elapsed_time(marks[-1][1]))
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
    dsa.check_device_error(stream)

    value, total_ms, tokens = aggregate_replicas(sum(step_ms), wl.L * args.steps, world, dev)

    # kernel totals per step (sum over chunk launches) and per-launch means
    steps = args.steps
    k_ms = {nm: sum(v) / steps for nm, v in per_kernel.items()}
    launch_ms = {nm: sum(v) / len(v) for nm, v in per_kernel.items()}
    alg = algorithmic(wl)
    peaks, peak_kind = load_peaks()
    ceilings = l2_ceilings(dsa, dims, wl, d_in["K"], d_in["V"], bufs.idx, stream, dev, with_bwd)
    dominant = max(k_ms, key=k_ms.get)
    rl = roofline(dominant, alg, launch_ms, k_ms, peaks, peak_kind, wl, len(chunks), ceilings)
    kernels = {nm: {"ms_per_step": round(k_ms[nm], 4), "calls_per_step": len(per_kernel[nm]) // steps,
                    **roofline(nm, alg, launch_ms, k_ms, peaks, peak_kind, wl, len(chunks), ceilings)} for nm in k_ms}

    # device memory of the layer: every buffer is a torch allocation (the library allocates nothing)
    flush_bytes = flush.numel()
    peak = torch.cuda.max_memory_allocated(dev)
    memory = {"peak_allocated_gib": round((peak - flush_bytes) / 2**30, 3),
              "indexer_topk_workspace_gib": round(bufs.ws.numel() / 2**30, 3),
              "what": "torch.cuda.max_memory_allocated over inputs, outputs and workspaces, less the 256 MiB "
                      "L2-flush buffer; the library allocates no device memory"}

    # end-to-end through the C ABI with host buffers: H2D of the inputs, the layer, D2H of the results
    e2e = end_to_end(dsa, dims, wl, host, d_in, bufs, dq, dk, dv, bws, stream, args, with_bwd, world, dev, det)
    clocks = clk.summary()
    return {
        "metric": METRIC if args.workload == "bf16_128k_needle" else f"DSA-layer tokens/s ({wl.passes}) {wl.name}",
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if wl.dtype == "bf16" else "f32", "data": "synthetic (seeded)",
        "config": {"workload": wl.name, "L": wl.L, "Hq": wl.Hq, "d": wl.d, "Hi": wl.Hi, "di": wl.di, "k": wl.k,
                   "q_chunk": wl.q_chunk, "pass": wl.passes, "needle": wl.needle,
                   "indexer_topk_route": args.indexer_route, "attn_fwd_route": args.attn_fwd_route,
                   "backward": args.backward if with_bwd else None,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "256 MiB buffer written before every timed step, outside the events"},
        "roofline": rl,
        "kernels": kernels,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "memory": memory,
        "inputs_sha256": inputs_sha,
    }


def roofline(nm, alg, launch_ms, k_ms, peaks, peak_kind, wl, nchunks, ceilings=None):
    """Roofline of one kernel from its mean CUDA-event launch time.

    The indexer is a tensor-core contraction (burst bf16 peak); top-k and the
    pool keys stream from HBM (measured copy bandwidth).  The attention kernels
    gather K/V rows from a table that stays in L2 and the backward adds fp32
    dK/dV rows into one: their bound is L2 traffic, so they are measured
    against a ceiling taken in the same run -- a replay of the same gathers and
    bulk reductions with no arithmetic (dsa_probe_traffic) -- with the HBM and
    tensor-core fractions beside it."""
    ms = launch_ms[nm]
    hbm = peaks["hbm_gbs"]
    traffic = measured_traffic(wl.name, nm)
    if nm in ("indexer", "indexer_topk"):
        # one call = one chunk (average); the work counted is the indexer's
        # causal flops (the sampled pass and the selection are overhead)
        flops = alg["indexer"]["flops"] / nchunks
        a = flops / (ms * 1e-3) / 1e12
        pk = peaks["bf16_tflops"]
        out = {"bound": "tensor", "achieved": round(a, 2), "peak": pk, "unit": "TFLOP/s", "frac": round(a / pk, 4),
               "traffic": traffic, "peak_source": f"{peak_kind} bf16 dense (burst)"}
        if traffic is not None:
            out["hbm_frac"] = round(traffic / (ms * 1e-3) / 1e9 / hbm, 4)
        return out
    if nm in ("attn_fwd", "attn_bwd", "attn_bwd_det") and ceilings and nm.replace("_det", "") in ceilings:
        # the deterministic backward is held to the same ceiling as the atomic
        # one: the replay of the query-major gathers and reductions
        c = ceilings[nm.replace("_det", "")]
        b = alg[nm.replace("_det", "")]["l2_bytes"]
        a = b / (ms * 1e-3) / 1e9
        fl = alg[nm.replace("_det", "")]["flops"] / (ms * 1e-3) / 1e12
        tpk = peaks["bf16_tflops_sustained"]
        out = {"bound": "l2", "achieved": round(a, 1), "peak": round(c["gbs"], 1), "unit": "GB/s",
               "frac": round(a / c["gbs"], 4), "traffic": traffic,
               "peak_source": c["what"],
               "tensor": {"achieved_tflops": round(fl, 2), "peak": tpk, "frac": round(fl / tpk, 4),
                          "peak_source": f"{peak_kind} bf16 dense (sustained)"}}
        if traffic is not None:
            out["hbm"] = {"achieved_gbs": round(traffic / (ms * 1e-3) / 1e9, 1), "peak": hbm,
                          "frac": round(traffic / (ms * 1e-3) / 1e9 / hbm, 4),
                          "peak_source": f"{peak_kind} HBM copy"}
        return out
    if nm == "topk":
        b = alg["topk"]["bytes"] / nchunks
    elif nm == "pool_keys":
        b = alg["pool_keys"]["bytes"]
    else:
        b = alg[nm]["bytes"]
    a = b / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(a, 1), "peak": hbm, "unit": "GB/s", "frac": round(a / hbm, 4),
            "traffic": traffic, "peak_source": f"{peak_kind} HBM copy"}


def l2_ceilings(dsa, dims, wl, k, v, idx, stream, dev, with_bwd, reps=3):
    """Same-run ceilings for the attention kernels: dsa_probe_traffic replays
    the kernels' own steps over the layer's own selection (the same pool
    gathers and, for the backward, the same fp32 bulk reductions, with the
    same occupancy) and does no arithmetic.  Best of `reps`; the bytes are the
    kernels' logical L2 bytes, so ceiling / achieved = kernel time / replay time."""
    alg = algorithmic(wl)
    out = {}
    scratch = None
    if with_bwd:
        scratch = (torch.zeros((wl.L, wl.d), device=dev), torch.zeros((wl.L, wl.d), device=dev))
    for nm, red in (("attn_fwd", False), ("attn_bwd", True)):
        if red and not with_bwd:
            continue
        dk, dv = scratch if red else (None, None)
        best = None
        for r in range(reps + 1):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            dsa.probe_traffic(dims, k, v, idx, dk, dv, stream=stream)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ms = e0.elapsed_time(e1)
            if r > 0:
                best = ms if best is None else min(best, ms)
        b = alg[nm]["l2_bytes"]
        what = ("same-run replay of this kernel's steps over the layer's own selection, no arithmetic "
                "(dsa_probe_traffic): the same 16-byte cp.async pool gathers of K and V"
                + (" and one fp32 bulk reduction per pool slot into each of dK and dV" if red else "")
                + f", same occupancy; best of {reps}: {best:.3f} ms for {b / 1e9:.1f} GB")
        out[nm] = {"gbs": b / (best * 1e-3) / 1e9, "ms": best, "bytes": b, "what": what}
    dsa.check_device_error(stream)
    return out


def end_to_end(dsa, dims, wl, host, d_in, bufs, dq, dk, dv, bws, stream, args, with_bwd, world, dev, det=False):
    """Tokens/s through the public entry points with host buffers: every step
    copies its inputs in from pinned host memory, runs the layer and copies its
    outputs (O, LSE and, with a backward, dQ, dK, dV) back to pinned memory.

    The layer runs as its three phases, each through its own entry points:
    pool keys and indexer + top-k per query chunk (what dsa_layer_fwd does
    first), the attention forward, the backward.  Consecutive steps are
    pipelined with two device buffer sets, the phases on one stream and the
    copies on another (_e2e_pipelined): a phase waits only for its own inputs
    (k_I, q_I, w; then Q, K, V; then dO), the next step's inputs go in while
    this one runs, and O and LSE go back as soon as the forward is done.
    --e2e-steps steps (10
    by default) are timed, pipeline fill and drain included, and the box's
    measured copy rates are reported beside the figure.  If the pipelined run
    raises, the serialised run is reported and "mode" says why."""
    names = list(d_in.keys())
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    outs = [bufs.o, bufs.lse] + ([dq, dk, dv] if with_bwd else [])
    d2h = sum(t.numel() * t.element_size() for t in outs)
    steps = max(1, args.e2e_steps)
    phases = layer_phases(dsa, dims, wl, bufs, bws, with_bwd, det)
    assert sorted(n for ph in phases for n in ph[0]) == sorted(names)
    overlap = None
    try:
        ms, overlap = _e2e_pipelined(host, d_in, outs, phases, steps, dev)
        mode = "pipelined: a run stream and one copy stream, 2 device buffer sets, per-phase copies"
    except Exception as exc:   # reported in the JSON line, never silent
        torch.cuda.synchronize(dev)
        ms = _e2e_serial(host, names, d_in, outs, phases, steps, stream, dev)
        mode = f"serialised on one stream (pipelined run raised {type(exc).__name__}: {exc})"[:240]
    value, ms, _ = aggregate_replicas(ms, wl.L * steps, world, dev)
    return {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": round(ms / steps, 3), "mode": mode,
            "overlap": overlap,
            "copy_bandwidth": copy_bandwidth(host, names, d_in, outs, stream, dev),
            # the runtime's hardware work queues per device (unset: the runtime's default)
            "cuda_device_max_connections": os.environ.get("CUDA_DEVICE_MAX_CONNECTIONS")}


def layer_phases(dsa, dims, wl, bufs, bws, with_bwd, det=False):
    """The layer as (inputs it needs, run(d, o, stream), indices into the
    outputs [O, LSE, dQ, dK, dV] it completes), in order: pool keys and
    indexer + top-k per query chunk (the first part of dsa_layer_fwd), the
    attention forward, the backward."""
    C = int(dims.q_chunk)
    chunks = [(q0, min(C, wl.L - q0)) for q0 in range(0, wl.L, C)]

    def select(d, o, s):       # writes kpool, idx (and the indexer workspace)
        dsa.pool_keys(dims, d["k_I"], bufs.kpool, s)
        for q0, n in chunks:
            dsa.indexer_topk(dims, d["q_I"], bufs.kpool, d["w"], q0, n, bufs.idx, bufs.ws, stream=s)

    def forward(d, o, s):      # writes O, LSE, o_acc
        dsa.sparse_attn_fwd(dims, d["Q"], d["K"], d["V"], bufs.idx, o[0], o[1], s, o_acc=bufs.o_acc)

    def backward(d, o, s):     # writes dQ, dK, dV
        if det:
            dsa.sparse_attn_bwd_det(dims, d["Q"], d["K"], d["V"], bufs.idx, o[0], o[1], d["dO"], o[2], o[3], o[4],
                                    bws, stream=s, o_acc=bufs.o_acc)
        else:
            dsa.layer_bwd(dims, d["Q"], d["K"], d["V"], bufs.idx, o[0], o[1], d["dO"], o[2], o[3], o[4], bws,
                          stream=s, o_acc=bufs.o_acc)

    phases = [(["k_I", "q_I", "w"], select, []), (["Q", "K", "V"], forward, [0, 1])]
    if with_bwd:
        phases.append((["dO"], backward, [2, 3, 4]))
    return phases


def copy_bandwidth(host, names, d_in, outs, stream, dev):
    """The host<->device copy rates this box gives the end-to-end leg: the
    step's input copies from pinned memory alone, then its output copies to
    pinned memory alone, each timed with CUDA events on one stream (best of 3)."""
    pinned = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    h2d_b = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h_b = sum(t.numel() * t.element_size() for t in outs)

    def timed(fn):
        best = None
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            e0.record(stream)
            with torch.cuda.stream(stream):
                fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        return best

    ms_in = timed(lambda: [d_in[n].copy_(host[n], non_blocking=True) for n in names])
    ms_out = timed(lambda: [dst.copy_(src, non_blocking=True) for src, dst in zip(outs, pinned)])
    return {"h2d_gbs": round(h2d_b / (ms_in * 1e-3) / 1e9, 1), "h2d_ms": round(ms_in, 3),
            "d2h_gbs": round(d2h_b / (ms_out * 1e-3) / 1e9, 1), "d2h_ms": round(ms_out, 3)}


def _e2e_pipelined(host, d_in, outs, phases, steps, dev, sink=None):
    """Total ms of `steps` pipelined steps (see end_to_end) and where it went.
    sink (a list): receives the pinned host copies of the last step's outputs.

    Two streams: the layer's phases run on one, every copy on the other, in
    the order the copies are needed.  When step i starts, step i-1 -- the last
    user of the other buffer set -- is done, so the inputs of step i+1 go into
    that set; O and LSE of step i go out when its forward is done, its
    gradients when its backward is done.  So copies never run at the same time
    as one another -- concurrent copies in both directions slowed each other
    several-fold on some boxes -- while each overlaps the kernels."""
    names = [n for ph in phases for n in ph[0]]
    sets = [(d_in, outs), ({n: torch.empty_like(d_in[n]) for n in names}, [torch.empty_like(t) for t in outs])]
    pinned = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs] for _ in sets]
    s_run, s_cp = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    P = len(phases)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    in_done = [[ev() for _ in range(P)] for _ in range(steps)]     # a phase's inputs are in
    ph_done = [[ev() for _ in range(P)] for _ in range(steps)]     # a phase has run
    out_done = [[ev() for _ in range(P)] for _ in range(steps)]    # a phase's outputs are out

    def copy_in(i):
        d = sets[i % 2][0]
        for p, (inputs, _, _) in enumerate(phases):
            with torch.cuda.stream(s_cp):
                for n in inputs:
                    d[n].copy_(host[n], non_blocking=True)
            in_done[i][p].record(s_cp)

    # one untimed pass of every copy over every buffer: freshly allocated
    # pinned memory is slow on its first transfers
    with torch.cuda.stream(s_cp):
        for d, o in sets:
            for n in names:
                d[n].copy_(host[n], non_blocking=True)
        for k in range(len(sets)):
            for src, dst in zip(outs, pinned[k]):
                dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize(dev)
    start = ev()
    start.record(s_cp)
    copy_in(0)
    for i in range(steps):
        d, o = sets[i % 2]
        for p, (_, run, outputs) in enumerate(phases):
            s_run.wait_event(in_done[i][p])
            if i >= 2 and outputs:
                s_run.wait_event(out_done[i - 2][p])   # step i-2's outputs in this set have been copied out
            run(d, o, s_run)
            ph_done[i][p].record(s_run)
        if i + 1 < steps:
            if i >= 1:
                s_cp.wait_event(ph_done[i - 1][-1])    # step i-1 has finished reading the next step's set
            copy_in(i + 1)
        for p, (_, _, outputs) in enumerate(phases):
            if outputs:
                s_cp.wait_event(ph_done[i][p])
                with torch.cuda.stream(s_cp):
                    for j in outputs:
                        pinned[i % 2][j].copy_(o[j], non_blocking=True)
                out_done[i][p].record(s_cp)
    torch.cuda.synchronize(dev)
    # Where the time went, from the same events: a phase can begin once its
    # inputs are in, its buffer set's previous outputs are out and the phase
    # before it is done; from then to its end is its time inside the pipeline,
    # and the run stream's wait before it is copy time the pipeline did not hide.
    t = start.elapsed_time
    last_out = max(p for p in range(P) if phases[p][2])
    layer_ms, wait_ms = [], []
    for i in range(steps):
        run_ms = waited = 0.0
        for p, (_, _, outputs) in enumerate(phases):
            ready = t(in_done[i][p])
            if i >= 2 and outputs:
                ready = max(ready, t(out_done[i - 2][p]))
            anchor = t(ph_done[i][p - 1]) if p > 0 else (t(ph_done[i - 1][-1]) if i > 0 else None)
            begin = ready if anchor is None else max(ready, anchor)
            if anchor is not None:
                waited += begin - anchor
            run_ms += t(ph_done[i][p]) - begin
        layer_ms.append(run_ms)
        wait_ms.append(waited)
    overlap = {"layer_ms_mean": round(sum(layer_ms) / steps, 3), "layer_ms_max": round(max(layer_ms), 3),
               "run_stream_wait_ms_mean": round(sum(wait_ms) / steps, 3),
               "fill_ms": round(t(in_done[0][0]), 3),
               "drain_ms": round(t(out_done[-1][last_out]) - t(ph_done[-1][-1]), 3)}
    if sink is not None:
        sink.append(pinned[(steps - 1) % 2])
    return t(out_done[-1][last_out]), overlap


def _e2e_serial(host, names, d_in, outs, phases, steps, stream, dev):
    """Total ms of `steps` steps with every copy and launch on one stream."""
    pinned = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]

    def one():
        with torch.cuda.stream(stream):
            for n in names:
                d_in[n].copy_(host[n], non_blocking=True)
        for _, run, _ in phases:
            run(d_in, outs, stream)
        with torch.cuda.stream(stream):
            for src, dst in zip(outs, pinned):
                dst.copy_(src, non_blocking=True)

    one()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1)


def inputs_digest(host: dict, names) -> str:
    """SHA-256 over the host input arrays, in the given tensor order."""
    import hashlib
    h = hashlib.sha256()
    for n in names:
        t = host[n].contiguous()
        h.update(n.encode())
        h.update(t.view(torch.uint8).numpy().tobytes() if t.dtype != torch.bfloat16
                 else t.view(torch.int16).numpy().tobytes())
    return h.hexdigest()


ARM_PARTS = {"0xd4f": "Arm Neoverse-V2", "0xd40": "Arm Neoverse-V1", "0xd0c": "Arm Neoverse-N1",
             "0xd49": "Arm Neoverse-N2", "0xd84": "Arm Neoverse-V3"}


def host_cpu() -> dict:
    """The host's logical CPU count and a model string (best effort; Arm
    hosts list only implementer and part numbers in /proc/cpuinfo)."""
    model = platform.processor() or platform.machine()
    try:
        with open("/proc/cpuinfo") as f:
            fields = {}
            for ln in f:
                if ":" in ln:
                    key, val = (x.strip() for x in ln.split(":", 1))
                    fields.setdefault(key.lower(), val)
        if "model name" in fields:
            model = fields["model name"]
        elif "cpu part" in fields:
            part = fields["cpu part"].lower()
            model = f"{ARM_PARTS.get(part, 'Arm CPU part ' + part)} ({platform.machine()})"
    except OSError:
        pass
    return {"host_cpus": os.cpu_count(), "cpu_model": model}


def oracle_sample(wl, n_rows: int, seed: int = 7):
    """Time the CPU oracle (single thread) on n_rows query rows of the workload:
    pool keys, the rows' indexer scores and top-k, their attention forward and
    backward.  Returns (seconds, rows, description)."""
    import numpy as np
    import oracle

    oracle.build()
    with_bwd = wl.passes == "fwd+bwd"
    names = ("Q", "K", "V", "q_I", "k_I", "w") + (("dO",) if with_bwd else ())
    host = dsa_inputs.make(wl, names)
    g = torch.Generator().manual_seed(seed)
    rows = np.sort(torch.randint(wl.L // 2, wl.L, (n_rows,), generator=g).numpy()).astype(np.int64)
    f = {n: host[n].to(torch.float32).numpy() for n in ("K", "V", "q_I", "k_I", "w")}
    Qr = host["Q"][rows].to(torch.float32).numpy()
    dOr = host["dO"][rows].to(torch.float32).numpy() if with_bwd else None
    t0 = time.perf_counter()
    kp = oracle.pool_keys(f["k_I"], wl.dtype == "bf16")
    t_pool = time.perf_counter() - t0
    t1 = time.perf_counter()
    sc = oracle.indexer_scores(f["q_I"], kp, f["w"], rows)
    sel = oracle.topk(sc, wl.L, wl.k, rows)
    idx = np.full((wl.L, wl.k), -1, np.int32)
    idx[rows] = sel
    oracle.attn_fwd(Qr, f["K"], f["V"], idx, wl.scale, rows, q_compact=True)
    if with_bwd:
        oracle.attn_bwd(Qr, f["K"], f["V"], idx, dOr, wl.scale, rows, with_dkv=True, threads=1, q_compact=True)
    t_rows = time.perf_counter() - t1
    # the pool-key pass is per layer: charge it in proportion to the rows sampled
    secs = t_rows + t_pool * (n_rows / wl.L)
    desc = (f"extrapolated from {n_rows} sampled query rows (drawn uniformly from the second half of the "
            f"sequence): indexer scores over all eligible pools, top-{wl.k}, attention {wl.passes} with dK/dV; "
            f"pool keys once, charged per row; tokens/s = rows / their single-core time")
    return secs, n_rows, desc


def oracle_full_tiny():
    """The oracle's whole forward on the smallest workload (L=4096, fp32),
    single-threaded, every row: a measured (not extrapolated) CPU time."""
    import oracle

    oracle.build()
    wl = dsa_inputs.WORKLOADS["tiny_fp32_fwd"]
    host = dsa_inputs.make(wl, ("Q", "K", "V", "q_I", "k_I", "w"))
    f = {n: host[n].to(torch.float32).numpy() for n in host}
    t0 = time.perf_counter()
    oracle.layer_fwd(f["Q"], f["K"], f["V"], f["q_I"], f["k_I"], f["w"], wl.k, wl.scale, False)
    secs = time.perf_counter() - t0
    return {"workload": wl.name, "L": wl.L, "pass": wl.passes, "seconds": round(secs, 3),
            "value": round(wl.L / secs, 1), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": "every row of the workload (measured, not extrapolated)"}


def run_reference(args):
    wl = dsa_inputs.WORKLOADS[args.workload]
    per_step_rows = max(1, args.ref_rows)
    times = []
    for s in range(args.warmup + args.steps):
        secs, n, desc = oracle_sample(wl, per_step_rows, seed=100 + s)
        if s >= args.warmup:
            times.append(secs)
    total = sum(times)
    value = per_step_rows * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC if args.workload == "bf16_128k_needle" else wl.name,
        "value": round(value, 3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / args.steps, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": wl.name, "L": wl.L, "k": wl.k, "pass": wl.passes},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": desc, **host_cpu()},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="bf16_128k_needle", choices=sorted(dsa_inputs.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-rows", type=int, default=24, help="oracle rows per reference step")
    ap.add_argument("--cpu-rows", type=int, default=384,
                    help="oracle rows for the cpu_baseline field (384: about 10 s of one host core at 128k)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10, help="end-to-end steps (at least 1; 10 by default)")
    ap.add_argument("--indexer-route", type=int, default=1, choices=[0, 1],
                    help="indexer + top-k route: 1 score block + row-wise top-k (default), 0 candidate lists")
    ap.add_argument("--backward", default="atomic", choices=["atomic", "det"],
                    help="backward: atomic (default) or the deterministic key-major one")
    ap.add_argument("--attn-fwd-route", type=int, default=0, choices=[0, 1],
                    help="attention forward: 0 warp-level kernel (default), 1 tcgen05 kernel")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl")
    line = run_ours(args, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            wl = dsa_inputs.WORKLOADS[args.workload]
            secs, n, desc = oracle_sample(wl, args.cpu_rows)
            line["cpu_baseline"] = {"value": round(n / secs, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                    "sample": desc, "seconds": round(secs, 2), "extrapolated": True,
                                    **host_cpu(), "full_run_tiny_fwd": oracle_full_tiny()}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

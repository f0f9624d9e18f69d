"""Benchmark: MSA forward + backward on the packed-document T=16384 workload.

One step = the whole hot path on one batch: plan build (q2k -> CSR -> tasks),
forward (O, LSE) and backward (dQ, dK, dV), inputs resident in HBM.  L2 is
flushed (256 MiB write) before every timed step; each step is bracketed by
CUDA events on the launching stream.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line.  FLOPs are the method's own: 4*d per attended
(query, head, key) triple forward and 10*d backward, counted exactly by the
plan builder.  Under torchrun (N > 1) every rank runs its own replica of the
workload (weak scaling, no data-path collective); rank 0 prints the
aggregate.  ``--impl reference`` times the fp64 CPU oracle (the reference arm)
on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_sparse_gqa_msa_gb300 import inputs  # noqa: E402

HEAD_DIM = 128
FWD_FLOP_PER_PAIR = 4 * HEAD_DIM
BWD_FLOP_PER_PAIR = 10 * HEAD_DIM
METRIC = "MSA fwd+bwd sparse TFLOP/s & tokens/s at T=16k; % of GB300 BF16 tensor peak"
WORKLOAD = 3  # packed 16k row of documents
# every kernel family the library launches on the plan / forward / backward path
KERNELS = ("plan_docs", "plan_count", "plan_scan", "plan_scatter", "plan_emit", "plan_ftasks",
           "fwd_kmax", "fwd_v16", "fwd_rows", "fwd_group", "fwd_main", "fwd_finalize",
           "fwd_fallback", "bwd_delta", "bwd_main", "bwd_finalize")
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.path = os.path.join("/tmp", f"msa_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- recorded DRAM traffic
def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of ``kernel`` from the committed ncu record in
    profiles/, or None when there is none for this workload or the kernel's
    sources changed since the counters were taken (hash mismatch)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"{kernel}_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("workload") != workload:
        return None
    h = hashlib.sha256()
    for src in rec.get("source_files", []):
        p = os.path.join(ROOT, src)
        if not os.path.exists(p):
            return None
        with open(p, "rb") as f:
            h.update(f.read())
    if h.hexdigest()[:16] != rec.get("source_sha256_16"):
        return None
    return rec.get("bytes_per_launch")


# ---------------------------------------------------------------- adjacent steps
def measure_packing(dev, peaks):
    """Padded packed rows <-> compact THD for the query tensor of eight packed
    rows of 16384 tokens (each row losing a U(0, 0.15) trailing fraction to
    padding, as in the eight-row workload): device time per call with CUDA
    events (inputs of 2 GB, far above L2), algorithmic bytes = the rows read
    and written, against the measured copy bandwidth."""
    from block_sparse_gqa_msa_gb300 import api
    B, S = 8, 16384
    rng = np.random.default_rng(4004)
    lens = (S - np.floor(rng.uniform(0.0, 0.15, size=B) * S)).astype(np.int32)
    row_len = torch.from_numpy(lens).to(dev)
    x = torch.empty((B, S, 64, 128), dtype=torch.bfloat16, device=dev).normal_()
    T = int(lens.sum())
    row_bytes = 64 * 128 * 2
    stream = torch.cuda.current_stream()
    out = {}
    y, offs = api.pack_thd(x, row_len, total=T)
    back = api.unpack_bshd(y, row_len, offs, S)
    for name, fn, nbytes in (
            ("pack_thd", lambda: api.pack_thd(x, row_len, total=T), 2 * T * row_bytes),
            ("unpack_bshd", lambda: api.unpack_bshd(y, row_len, offs, S, out=back),
             (T + B * S) * row_bytes)):
        for _ in range(3):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(10):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / 10
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"ms": ms, "bytes": nbytes, "GB_s": gbs,
                     "frac_of_hbm": gbs / float(peaks["hbm_gbs"]),
                     "shape": f"[{B},{S},64,128] bf16, T={T}"}
    del x, y, back
    out["select_blocks"] = measure_selection(dev, peaks)
    return out


def measure_selection(dev, peaks, dim: int = 64):
    """Block scorer + top-16 on the packed-document T=16384 row with index
    dim 64 (synthetic N(0,1) index queries / keys): device time per call and
    the scoring FMA rate against the fp32 FMA peak (SMs x 128 lanes x the
    maximum SM clock)."""
    from block_sparse_gqa_msa_gb300 import api
    w = inputs.config(WORKLOAD)
    T = w.T
    g = torch.Generator().manual_seed(7007)
    iq = torch.randn(T, 4, dim, generator=g).to(torch.bfloat16).to(dev)
    ik = torch.randn(T, 4, dim, generator=g).to(torch.bfloat16).to(dev)
    offs = w.doc_offsets.to(dev)
    q2k = torch.empty((4, T, 16), dtype=torch.int32, device=dev)
    ws = torch.empty(api.select_workspace_bytes(T, w.num_docs, dim), dtype=torch.uint8,
                     device=dev)
    # scoring work: every (token, index head) with more than 16 candidate blocks
    # scores blocks 1 .. b-1 (blocks 0 and b are always kept)
    fma = 0
    for ln in np.diff(w.doc_offsets.numpy()):
        b = np.arange(int(ln)) // 128
        fma += int(np.where(b + 1 > 16, b - 1, 0).sum()) * 4 * dim
    fma += T * 4 * dim  # block sums
    stream = torch.cuda.current_stream()
    for _ in range(3):
        api.msa_select_blocks(iq, ik, offs, q2k=q2k, workspace=ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(10):
        api.msa_select_blocks(iq, ik, offs, q2k=q2k, workspace=ws)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / 10
    api.profile_enable(True)
    api.profile_reset()
    api.msa_select_blocks(iq, ik, offs, q2k=q2k, workspace=ws)
    split = {k: api.profile_read(k)[1] for k in ("sel_summary", "sel_topk")}
    api.profile_enable(False)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peak = sms * 128 * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6
    return {"ms": ms, "fma": fma, "TFMA_s": fma / (ms * 1e-3) / 1e12,
            "frac_of_fp32_fma": fma / (ms * 1e-3) / peak, "bound": "alu",
            "kernels_ms": {k: round(v, 4) for k, v in split.items()},
            "shape": f"T={T}, {w.num_docs} documents, index dim {dim}"}


# ---------------------------------------------------------------- multi-rank
def reduce_over_ranks(x: float, world: int, op: str = "max") -> float:
    """Max (the slowest rank's time) or sum (work done by all ranks) of one
    number over the ranks of the default process group; identity at N=1."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64)
    red = torch.distributed.ReduceOp.MAX if op == "max" else torch.distributed.ReduceOp.SUM
    torch.distributed.all_reduce(t, op=red)
    return float(t.item())


def aggregate(total_ms: float, steps: int, flop_step: float, tokens: int, world: int):
    """Whole-job figures of a weak-scaling run: every rank processed its own
    replica; the job took as long as its slowest rank.  Returns
    (ms_per_step, TFLOP/s over all ranks, tokens/s over all ranks)."""
    ms = reduce_over_ranks(total_ms, world, "max") / steps
    flop = reduce_over_ranks(flop_step, world, "sum")
    tok = reduce_over_ranks(tokens, world, "sum")
    return ms, flop / (ms * 1e-3) / 1e12, tok / (ms * 1e-3)


# ---------------------------------------------------------------- reference arm
def cpu_sample(w, budget_s: float = 20.0, max_doc_tokens: int = 0):
    """Time the fp64 oracle's forward + backward on whole documents of the
    workload (documents are independent, so each is a faithful sample).  With
    ``max_doc_tokens`` each document is cut to that prefix, which is itself a
    valid document (causal attention never looks past a query)."""
    import oracle
    offs = w.doc_offsets.numpy()
    lens = np.diff(offs)
    order = np.argsort(np.abs(lens - np.median(lens)))  # typical documents first
    flops = 0.0
    pairs_total = 0
    spent = 0.0
    used = []
    for d in order:
        s, e = int(offs[d]), int(offs[d + 1])
        if max_doc_tokens > 0:
            e = min(e, s + max_doc_tokens)
        sub = inputs.Workload(
            name="doc", q=w.q[s:e], k=w.k[s:e], v=w.v[s:e], do=w.do[s:e],
            q2k=w.q2k[:, s:e].contiguous(),
            doc_offsets=torch.tensor([0, e - s], dtype=torch.int32), scale=w.scale)
        P = oracle.Problem.from_workload(sub)
        pairs = P.pair_count()
        t0 = time.perf_counter()
        P.forward()
        P.backward()
        dt = time.perf_counter() - t0
        spent += dt
        pairs_total += pairs
        flops += pairs * (FWD_FLOP_PER_PAIR + BWD_FLOP_PER_PAIR)
        used.append(e - s)
        if spent >= budget_s * 0.5:
            break
    return {
        "flops": flops, "seconds": spent, "tokens": int(sum(used)), "docs": len(used),
        "pairs": pairs_total, "cores": oracle.threads(),
        "sample": f"{len(used)} {'document prefix(es)' if max_doc_tokens > 0 else 'whole document(s)'}"
                  f" ({sum(used)} tokens, lengths {used}) of the packed T=16384 row: oracle "
                  f"forward + backward in fp64",
    }


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = inputs.config(WORKLOAD)
    budget = args.sample_seconds or max(3.0, 30.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_sample(w, budget, args.sample_max_tokens)
    times, flops, last = [], 0.0, None
    for _ in range(args.steps):
        last = cpu_sample(w, budget, args.sample_max_tokens)
        times.append(last["seconds"])
        flops += last["flops"]
    total = sum(times)
    value = flops / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "docs": w.num_docs},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": last["cores"],
                         "kind": "oracle", "sample": last["sample"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- streaming kernels
def streaming_bytes(T: int, n_ungrouped: int, NB: int, dq_esz: int = 2) -> dict:
    """Algorithmic bytes per launch of the HBM-bound kernels: what each must
    read and write by its definition (n_ungrouped: (token, index head) pairs
    whose octet is not grouped; NB: key blocks; dq_esz: bytes per dQ pool
    element)."""
    kv = T * 4 * 128 * 2  # one of K, V as bf16
    rows_q = T * 64 * 128 * 2  # one of Q, O, dO as bf16
    return {
        "fwd_kmax": 3 * kv + 2 * 4 * NB * 4,                 # K, V read; fp16 V, maxima written
        "fwd_v16": 4 * NB * 4 + 4 * 4,                       # max |v| read, scales written (the
                                                             # copy is rewritten only if a head
                                                             # needs a scale: not here)
        "fwd_rows": n_ungrouped * (4096 + 64 + 128 + 8192),  # Q, q2k read; shifts, sums, pool zeroed
        "fwd_finalize": n_ungrouped * (8192 + 128 + 4096 + 64),  # pool, shifts, sums read; O, LSE
        "bwd_delta": 2 * rows_q + T * 64 * 4 + T * 64 * 128 * dq_esz + 2 * T * 512 * 4,
        "bwd_finalize": T * 64 * 128 * dq_esz + 2 * T * 512 * 4 + rows_q + 2 * kv,
    }


def measure_workload(api, dev, n: int, steps: int = 5) -> dict:
    """plan + forward + backward of workload n with inputs resident and L2
    flushed before each timed step: TFLOP/s of the method's FLOPs."""
    w = inputs.config(n)
    q, k, v, do = (x.to(dev) for x in (w.q, w.k, w.v, w.do))
    q2k, offs = w.q2k.to(dev), w.doc_offsets.to(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        p = api.msa_build_plan(q2k, offs)
        o, lse = api.msa_forward(p, q, k, v, w.scale)
        api.msa_backward(p, q, k, v, o, lse, do, w.scale)
        return p

    for _ in range(3):
        p = step()
    torch.cuda.synchronize()
    pairs = api.msa_plan_counts(p)["pairs"]
    ms = []
    for _ in range(steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    m = statistics.mean(ms)
    flop = pairs * (FWD_FLOP_PER_PAIR + BWD_FLOP_PER_PAIR)
    return {"workload": w.name, "T": w.T, "ms_per_step": m, "TFLOP_s": flop / (m * 1e-3) / 1e12,
            "steps": steps}


# ---------------------------------------------------------------- GPU arm
def run_gpu(args, rank, world):
    from block_sparse_gqa_msa_gb300 import api

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = inputs.config(WORKLOAD, seed=inputs.CONFIG_SEEDS[WORKLOAD] + rank)
    T = w.T
    stream = torch.cuda.current_stream()
    q, k, v, do = (x.to(dev) for x in (w.q, w.k, w.v, w.do))
    q2k, offs = w.q2k.to(dev), w.doc_offsets.to(dev)
    plan = api.msa_build_plan(q2k, offs, super_block=args.super_block)
    pws = plan.workspace
    fws = torch.empty(api.forward_workspace_bytes(plan), dtype=torch.uint8, device=dev)
    bws = torch.empty(api.backward_workspace_bytes(plan), dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((T, 64), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def step():
        p = api.msa_build_plan(q2k, offs, super_block=args.super_block,
                                 workspace=pws)
        api.msa_forward(p, q, k, v, w.scale, o=o, lse=lse, workspace=fws)
        api.msa_backward(p, q, k, v, o, lse, do, w.scale, dq=dq, dk=dk, dv=dv, workspace=bws)
        return p

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if api.msa_read_status(plan) != 0:
        raise RuntimeError(f"device status {api.msa_read_status(plan)}")
    counts = api.msa_plan_counts(plan)
    pairs = counts["pairs"]
    flop_fwd = pairs * FWD_FLOP_PER_PAIR
    flop_bwd = pairs * BWD_FLOP_PER_PAIR

    # ---- device-timed loop (inputs resident, L2 flushed before each step)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = ClockSampler() if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
        time.sleep(0.3)
    launches0 = api.launch_count()
    for i in range(args.steps):
        flush.zero_()
        e = evs[i]
        e[0].record(stream)
        p = api.msa_build_plan(q2k, offs, super_block=args.super_block,
                                 workspace=pws)
        api.msa_forward(p, q, k, v, w.scale, o=o, lse=lse, workspace=fws)
        api.msa_backward(p, q, k, v, o, lse, do, w.scale, dq=dq, dk=dk, dv=dv, workspace=bws)
        e[3].record(stream)
    torch.cuda.synchronize()
    launches = api.launch_count() - launches0
    clk = clocks.stop() if clocks else None
    step_ms = [e[0].elapsed_time(e[3]) for e in evs]
    # ---- per-kernel times: a separate loop of the same steps with the
    # library's per-launch events (they keep launches apart, so the timed
    # loop above runs without them)
    psteps = min(args.steps, 5)
    api.profile_enable(True)
    api.profile_reset()
    pevs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(psteps)]
    for i in range(psteps):
        flush.zero_()
        e = pevs[i]
        e[0].record(stream)
        p = api.msa_build_plan(q2k, offs, super_block=args.super_block, workspace=pws)
        e[1].record(stream)
        api.msa_forward(p, q, k, v, w.scale, o=o, lse=lse, workspace=fws)
        e[2].record(stream)
        api.msa_backward(p, q, k, v, o, lse, do, w.scale, dq=dq, dk=dk, dv=dv, workspace=bws)
        e[3].record(stream)
    torch.cuda.synchronize()
    kern = {}
    for name in KERNELS:
        n, ms = api.profile_read(name)
        if n:
            kern[name] = {"launches": n / psteps, "ms_per_step": ms / psteps}
    api.profile_enable(False)
    if world > 1:
        torch.distributed.barrier()
    # the plan / forward / backward split, from the profiled loop
    plan_ms = [e[0].elapsed_time(e[1]) for e in pevs]
    fwd_ms = [e[1].elapsed_time(e[2]) for e in pevs]
    bwd_ms = [e[2].elapsed_time(e[3]) for e in pevs]
    flop_step = flop_fwd + flop_bwd
    ms_per_step, value, tok_s = aggregate(sum(step_ms), args.steps, flop_step, T, world)

    # ---- end to end through the public API with host buffers.  Every step
    # copies its inputs from pinned host memory and all of its results back;
    # the copies run on their own streams so step i+1's upload and step i-1's
    # download overlap step i's kernels (two device buffer sets).
    pin = lambda x: x.pin_memory()  # noqa: E731
    hq, hk, hv, hdo, hq2k, hoffs = (pin(x) for x in (w.q, w.k, w.v, w.do, w.q2k, w.doc_offsets))
    ho, hlse = pin(torch.empty_like(w.q)), pin(torch.empty((T, 64), dtype=torch.float32))
    hdq, hdk, hdv = pin(torch.empty_like(w.q)), pin(torch.empty_like(w.k)), pin(torch.empty_like(w.v))
    h_in = (hq, hk, hv, hdo, hq2k, hoffs)
    h_out = (ho, hlse, hdq, hdk, hdv)
    h2d = sum(x.numel() * x.element_size() for x in h_in)
    d2h = sum(x.numel() * x.element_size() for x in h_out)
    e2e_steps = max(4, args.steps)  # as many steps as the device-timed loop
    e2e_ms = float("nan")
    if not args.no_e2e:
        sets_in = [tuple(torch.empty_like(x, device=dev) for x in h_in) for _ in range(2)]
        sets_out = [(torch.empty_like(q), torch.empty((T, 64), dtype=torch.float32, device=dev),
                     torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
                    for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        comp_done = [None, None]
        out_done = [None, None]

        def e2e_step(i):
            b = i & 1
            dq_, dk_, dv_ = sets_out[b][2], sets_out[b][3], sets_out[b][4]
            with torch.cuda.stream(s_in):
                if comp_done[b] is not None:  # step i-2's kernels read this set
                    s_in.wait_event(comp_done[b])
                for d_, h_ in zip(sets_in[b], h_in):
                    d_.copy_(h_, non_blocking=True)
                in_ready = ev()
                in_ready.record(s_in)
            stream.wait_event(in_ready)
            if out_done[b] is not None:  # step i-2's results were copied out
                stream.wait_event(out_done[b])
            qq, kk, vv, dd, q2, of = sets_in[b]
            oo, ll = sets_out[b][0], sets_out[b][1]
            pp = api.msa_build_plan(q2, of, super_block=args.super_block,
                                 workspace=pws)
            api.msa_forward(pp, qq, kk, vv, w.scale, o=oo, lse=ll, workspace=fws)
            api.msa_backward(pp, qq, kk, vv, oo, ll, dd, w.scale, dq=dq_, dk=dk_, dv=dv_,
                             workspace=bws)
            comp_done[b] = ev()
            comp_done[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[b])
                for h_, d_ in zip(h_out, sets_out[b]):
                    h_.copy_(d_, non_blocking=True)
                out_done[b] = ev()
                out_done[b].record(s_out)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize()
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ea.record(stream)
        s_in.wait_event(ea)
        for i in range(e2e_steps):
            e2e_step(i)
        stream.wait_stream(s_out)
        eb.record(stream)
        torch.cuda.synchronize()
        e2e_ms = ea.elapsed_time(eb) / e2e_steps
    _, e2e_value, _ = aggregate(e2e_ms, 1, flop_step, T, world)
    e2e_ms = reduce_over_ranks(e2e_ms, world, "max")
    if rank != 0:
        return

    # ---- roofline of the dominant kernel
    peaks, peak_src = load_peaks()
    dom = max(("fwd_main", "bwd_main"), key=lambda n: kern.get(n, {}).get("ms_per_step", 0.0))
    dom_flop = flop_fwd if dom == "fwd_main" else flop_bwd
    per_launch_ms = kern[dom]["ms_per_step"] / kern[dom]["launches"]
    achieved = dom_flop / (per_launch_ms * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    traffic = recorded_traffic(dom, w.name)

    adjacent = measure_packing(dev, peaks) if not args.no_adjacent else None
    if adjacent is not None and WORKLOAD != 2:
        # the pages' own operator benchmark setting: one document of 16k tokens
        adjacent["single_doc_16k"] = measure_workload(api, dev, 2)
        adjacent["single_doc_16k"]["pct_of_peak"] = (
            100.0 * adjacent["single_doc_16k"]["TFLOP_s"] / float(peaks["bf16_tflops"]))
    # HBM-bound kernels: algorithmic bytes per launch against the copy bandwidth
    grouped, _, _ = api.msa_plan_export_groups(plan)
    sbytes = streaming_bytes(T, int((grouped == 0).sum()), int(api.msa_plan_counts(plan)["NB"]))
    streaming = {}
    for name, nbytes in sbytes.items():
        if name in kern:
            ms_l = kern[name]["ms_per_step"] / kern[name]["launches"]
            gbs = nbytes / (ms_l * 1e-3) / 1e9
            streaming[name] = {"bytes": nbytes, "ms": round(ms_l, 4), "GB_s": round(gbs, 1),
                               "frac_of_hbm": round(gbs / float(peaks["hbm_gbs"]), 3)}
    # the main kernels' times in clock cycles (box-to-box comparisons at equal work)
    mhz = (clk or {}).get("sm_mhz") or float(peaks.get("sm_max_mhz", 2070.0))
    mcycles = {n_: round(kern[n_]["ms_per_step"] / kern[n_]["launches"] * mhz / 1e3, 3)
               for n_ in ("fwd_group", "fwd_main", "bwd_main") if n_ in kern}
    cpu = cpu_sample(w, budget_s=20.0) if not args.no_cpu_baseline else None
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "T": T, "docs": w.num_docs, "heads": "64q/4kv/4idx",
                   "head_dim": 128, "block": 128, "topk": 16, "super_block": args.super_block, "o_pool": "f32",
                   "pairs": pairs, "flop_per_step": flop_step,
                   "l2": "flushed before each timed step (256 MiB write)"},
        "tokens_per_s": tok_s,
        "pct_of_peak": 100.0 * value / world / peak,
        "pct_of_sustained_peak": 100.0 * value / world / float(peaks["bf16_tflops_sustained"]),
        "ms": {"plan": statistics.mean(plan_ms), "fwd": statistics.mean(fwd_ms),
               "bwd": statistics.mean(bwd_ms)},
        "kernels_ms_per_step": {k_: round(v_["ms_per_step"], 4) for k_, v_ in kern.items()},
        "kernels_mcycles_per_launch": mcycles,
        "streaming": streaming,
        "clocks": clk,
        "gpu_launches": launches,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "roofline": {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_src} bf16 burst (MEASURED_PEAKS.json)"
                     if peak_src == "measured" else "fallback 1.9 PFLOP/s"},
    }
    if adjacent:
        line["adjacent"] = adjacent
    if cpu:
        line["cpu_baseline"] = {"value": cpu["flops"] / cpu["seconds"] / 1e12, "unit": "TFLOP/s",
                                "cores": cpu["cores"], "kind": "oracle", "sample": cpu["sample"]}
    print(json.dumps(line), flush=True)


def main():
    global WORKLOAD
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--super-block", type=int, default=64)
    ap.add_argument("--workload", type=int, default=WORKLOAD, choices=[1, 2, 3, 4, 5],
                    help="synthetic workload (default: the packed 16k row the metric is quoted on)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-adjacent", action="store_true",
                    help="skip the THD packing measurement")
    ap.add_argument("--sample-seconds", type=float, default=0.0,
                    help="reference arm: CPU seconds per step (default: about 30 s per run)")
    ap.add_argument("--sample-max-tokens", type=int, default=0,
                    help="reference arm: cut sampled documents to this prefix (0 = whole)")
    args = ap.parse_args()
    WORKLOAD = args.workload
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        torch.distributed.init_process_group(backend="gloo")
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_gpu(args, rank, world)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

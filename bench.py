#!/usr/bin/env python3
"""Benchmark: exact attention forward + backward on the GQA causal 8K workload.

One step = one pass of the whole hot path over one batch of synthetic input:
attn_fwd (O, LSE) then attn_bwd (row sums D, dK/dV kernel, dQ kernel) on
B=1, Hq=64, Hkv=8, N=8192, d=128, causal, bf16 (the Llama-3-70B attention
shape).  Throughput counts algorithmic FLOPs: 4*B*Hq*d*(allowed pairs) for
the forward and 2.5x that for the backward.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]
  python bench.py --workload causal_mha_2k|flex_mods_4k|tiny_mha|fp8_outliers_16k|...

Prints ONE JSON line (rank 0); the default workload is the one the metric is
quoted on, the others are the smaller parity workloads timed the same way
(tiny_mha: forward only; fp8_outliers_16k: Hadamard + e4m3 prologue and the
e4m3 forward).  ``--impl reference`` times the fp64 CPU
oracle (the reference arm) on bounded row slices of the same
workload.  Under torchrun each rank runs an independent replica (weak
scaling, no data-path collective; the process group only carries the
timing barrier and max).
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

import numpy as np  # noqa: E402
import torch  # noqa: E402

import attn_inputs as gen  # noqa: E402

WORKLOAD = "gqa_causal_8k"
METRIC = "attention TFLOPS fwd/bwd (bf16 causal N=8K d=128) & % of GB300 dense peak"
UNIT = "TFLOP/s"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(PEAKS_FALLBACK), "fallback"


def bf16_peak(peaks, src, clk):
    """The bf16 dense peak a kernel timed in this run is held against.

    The measured burst figure holds for a short timed region at the maximum SM
    clock with no power cap (the case of every line this script prints: tens
    of milliseconds of work).  When the clock record shows a lower median SM
    clock, or sw_power_cap, the burst figure is scaled by median / max MHz.
    Returns (TFLOP/s, description)."""
    burst = peaks["bf16_tflops"]
    med, smax = (clk or {}).get("sm_mhz"), (clk or {}).get("sm_max_mhz")
    capped = "sw_power_cap" in (clk or {}).get("reasons", [])
    if med and smax and (med < 0.97 * smax or capped):
        return burst * med / smax, (f"{src} bf16_tflops (burst) x {med:.0f}/{smax:.0f} MHz "
                                    f"(median SM clock under load{', sw_power_cap' if capped else ''})")
    return burst, f"{src} bf16_tflops (burst: timed region at the maximum SM clock, no power cap)"


def causal_pairs(N: int) -> int:
    return N * (N + 1) // 2


def allowed_pairs(cfg, doc_ids=None) -> int:
    """Number of (query, key) pairs the workload's mask allows, summed over the
    batch (the FLOP count's unmasked fraction times N^2 times B)."""
    N, B = cfg["N"], cfg["B"]
    causal, W = cfg.get("causal", False), cfg.get("window")
    if doc_ids is None and W is None:
        return B * (causal_pairs(N) if causal else N * N)
    if not causal:
        raise ValueError("pair count implemented for causal masks with window / documents")
    total = 0
    for b in range(B):
        lens = np.bincount(doc_ids[b]) if doc_ids is not None else np.array([N])
        for L in lens.tolist():
            i = np.arange(L, dtype=np.int64)
            total += int(np.minimum(i + 1, W if W is not None else L).sum())
    return total


def flops(cfg, doc_ids=None):
    fwd = 4.0 * cfg["Hq"] * cfg["d"] * allowed_pairs(cfg, doc_ids)
    return fwd, 2.5 * fwd


# ---------------------------------------------------------------- clocks ----
class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ----------------------------------------------------------- distributed ----
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allmax(world, x: float) -> float:
    """Largest of the ranks' values (the slowest replica's time sets the step)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_seed(cfg, rank: int) -> int:
    """Each replica draws its own inputs (replicas do not repeat one another's work)."""
    return cfg["seed"] + 97 * rank


def job_throughput(world: int, work_per_rank: float, max_ms: float) -> float:
    """Whole-job throughput of weak-scaled replicas: every rank does the same work per
    step, and the step lasts as long as the slowest rank (per second)."""
    return world * work_per_rank / (max_ms * 1e-3)


# ------------------------------------------------------- oracle baseline ----
def row_pairs(cfg, doc_ids, b, rows):
    """Allowed keys of each query row in ``rows`` (of batch entry b)."""
    N = cfg["N"]
    rows = np.asarray(rows, np.int64)
    cnt = rows + 1 if cfg.get("causal") else np.full(rows.shape, N, np.int64)
    if cfg.get("window") is not None:
        cnt = np.minimum(cnt, cfg["window"])
    if doc_ids is not None:
        start = np.searchsorted(doc_ids[b], doc_ids[b][rows], side="left")
        cnt = np.minimum(cnt, rows - start + 1)
    return cnt


def oracle_sample(cfg, x, budget_s: float, rows_per_slice: int, fwd_only=False):
    """Time the fp64 oracle on row slices of query heads of the workload.

    Runs slices (forward rows + their backward contributions) until
    ``budget_s`` seconds have passed (at least one).  Returns (TFLOP/s,
    seconds, description)."""
    from oracle import attn64
    docs = x.get("doc_ids")
    mods = attn64.Mods(causal=cfg.get("causal", False), window=cfg.get("window"), doc_ids=docs,
                       softcap=cfg.get("softcap"), alibi=cfg.get("alibi", False))
    scale = 1.0 / math.sqrt(cfg["d"])
    N, d = cfg["N"], cfg["d"]
    rows_per_slice = min(rows_per_slice, N)
    per_pair = (1.0 if fwd_only else 3.5) * 4.0 * d
    done_flops, t0, n = 0.0, time.perf_counter(), 0
    starts = list(range(N - rows_per_slice, -1, -rows_per_slice))
    while True:
        b = (n // cfg["Hq"]) % cfg["B"]
        hq = n % cfg["Hq"]
        r0 = starts[n % len(starts)]
        rows = np.arange(r0, r0 + rows_per_slice)
        attn64.head_forward(x["q"], x["k"], x["v"], scale, mods, b, hq, rows=rows)
        if not fwd_only:
            attn64.head_rows_backward(x["q"], x["k"], x["v"], x["do"], scale, mods, b, hq, rows)
        done_flops += per_pair * float(row_pairs(cfg, docs, b, rows).sum())
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    what = "forward" if fwd_only else "forward + their backward contributions"
    desc = (f"{n} slices of {rows_per_slice} query rows ({what}, fp64 numpy) of "
            f"{cfg.get('name', WORKLOAD)}; {done_flops:.3e} algorithmic FLOP")
    return done_flops / el / 1e12, el, desc


def cpu_info():
    cores = os.cpu_count() or 1
    return cores


# ---------------------------------------------------------------- ours -----
def traffic_record(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    source is unchanged since it was captured (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    h = sources_sha(rec["source"])
    return rec["bytes_per_launch"] if h is not None and h == rec.get("source_sha") else None


def sources_sha(names) -> str | None:
    """First 16 hex digits of the SHA-256 of the named kernel sources (one file
    name or a list, concatenated in the given order)."""
    names = [names] if isinstance(names, str) else list(names)
    m = hashlib.sha256()
    try:
        for n in names:
            with open(os.path.join(ROOT, "exact_attention_66_gb300", "csrc", n), "rb") as f:
                m.update(f.read())
    except OSError:
        return None
    return m.hexdigest()[:16]


def computed_pairs(ea, cfg, mods, dev) -> int:
    """(query, key) pairs inside the 128 x 128 tiles the kernels compute (the
    non-skipped tiles of the block map), summed over the batch, per query
    head: the same unit as allowed_pairs."""
    B, N = cfg["B"], cfg["N"]
    nT = (N + 127) // 128
    if cfg.get("window") or cfg.get("doc"):
        tiles = int((ea.block_map(B, N, mods, device=dev) > 0).sum().item())
    elif cfg.get("causal"):
        tiles = B * nT * (nT + 1) // 2
    else:
        tiles = B * nT * nT
    return tiles * 128 * 128


def workload_mods(ea, cfg, x, dev):
    docs = x.get("doc_ids")
    ddocs = torch.from_numpy(docs).to(dev) if docs is not None else None
    m = ea.make_mods(causal=cfg.get("causal", False), window=cfg.get("window"), doc_ids=ddocs,
                     softcap=cfg.get("softcap"), alibi=cfg.get("alibi", False))
    return m, docs


def mods_label(cfg):
    parts = [k for k in ("causal", "window", "doc", "softcap", "alibi") if cfg.get(k)]
    return "+".join(parts) or "none"


def l2_note(cfg):
    q_bytes = cfg["B"] * cfg["Hq"] * cfg["N"] * cfg["d"] * 2
    if q_bytes * 4 > 130 * 2**20:
        return f"inputs larger than L2 (Q/O/dO/dQ {q_bytes / 2**20:.0f} MiB each)"
    return f"inputs fit in L2 (Q {q_bytes / 2**10:.0f} KiB): warm-cache timing"


def link_gbs(stream, host_src, dev_dst, dev_src, host_dst) -> dict:
    """Host link bandwidth right after the end-to-end steps: one pinned
    host -> device copy and one device -> host copy, each timed alone with
    CUDA events (GB/s).  The machine's host link is shared, and the end-to-end
    figure follows it."""
    out = {}
    for name, dst, src in (("h2d", dev_dst, host_src), ("d2h", host_dst, dev_src)):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            dst.copy_(src, non_blocking=True)
            e1.record(stream)
        torch.cuda.synchronize()
        out[name] = round(src.numel() * src.element_size() / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)
    return out


def pipelined_e2e(dev, compute_stream, ins, outs, compute, steps, world):
    """Time ``steps`` end-to-end steps through the public API, pipelined.

    Every step copies its inputs from pinned host memory into one of two
    device buffer sets (``ins``: [(host, (dev0, dev1))]), runs ``compute(b)``
    on ``compute_stream`` with buffer set b, and copies its results back into
    pinned host memory (``outs``: [((dev0, dev1), (host0, host1))]).  The
    copies run on their own streams, so step i's inputs arrive while step
    i - 1 computes and its results leave while step i + 1 computes; events
    keep a buffer set from being overwritten before its step has read it and
    its results have left.  Returns ms per step (CUDA events, from before the
    first copy in to after the last copy out)."""
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def one(i, t=None):
        b = i & 1
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_comp[b])  # step i - 2 has read buffer set b
            if t is not None:
                t[0].record(s_in)
            for host, bufs in ins:
                bufs[b].copy_(host, non_blocking=True)
            ev_in[b].record(s_in)
        compute_stream.wait_event(ev_in[b])
        if i >= 2:
            compute_stream.wait_event(ev_out[b])  # step i - 2's results have left
        compute(b)
        ev_comp[b].record(compute_stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            if t is not None:
                t[2].record(s_out)
            for bufs, hosts in outs:
                hosts[b].copy_(bufs[b], non_blocking=True)
            ev_out[b].record(s_out)
        if t is not None:
            t[1].record(s_in)
            t[3].record(s_out)

    for i in range(2):  # warm-up
        one(i)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    ts = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for i in range(steps):
        one(i, ts[i])
    s_out.wait_stream(compute_stream)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    pipelined_e2e.copy_ms = (sum(t[0].elapsed_time(t[1]) for t in ts) / steps,
                             sum(t[2].elapsed_time(t[3]) for t in ts) / steps)
    return e0.elapsed_time(e1) / steps


def copy_gbs_in_pipeline(ms_in, ms_out, h2d, d2h) -> dict:
    """Bandwidth the pipelined copies got inside the timed end-to-end steps
    (bytes of a step's copies / the mean time its copy group took), rounded."""
    return {"h2d": round(h2d / (ms_in * 1e-3) / 1e9, 1), "d2h": round(d2h / (ms_out * 1e-3) / 1e9, 1)}


def run_ours(args, world, rank, local):
    import exact_attention_66_gb300 as ea

    if args.workload == "fp8_outliers_16k":
        return run_fp8(args, world, rank, local)
    if gen.WORKLOADS[args.workload].get("varlen"):
        return run_varlen(args, world, rank, local)
    if gen.WORKLOADS[args.workload].get("paged"):
        return run_paged(args, world, rank, local)
    if gen.WORKLOADS[args.workload].get("decode"):
        return run_decode(args, world, rank, local)
    name = args.workload
    cfg = dict(gen.WORKLOADS[name])
    if args.heads:  # smaller case of the same shape family (profiling); 8 query heads per KV head
        cfg["Hq"], cfg["Hkv"] = args.heads, max(1, args.heads // 8)
    B, Hq, Hkv, N, d = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["N"], cfg["d"]
    fwd_only = name == "tiny_mha"
    scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    x = gen.make_inputs(**dict(cfg, seed=replica_seed(cfg, rank)))
    host = {k: x[k].pin_memory() for k in ("q", "k", "v", "do")}
    q, k, v, do = (host[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    mods, docs = workload_mods(ea, cfg, x, dev)
    nws_f = ea.attn_workspace_size(ea.OP_FWD, B, Hq, Hkv, N, d, mods)
    ws_f = torch.empty(max(nws_f, 1), dtype=torch.uint8, device=dev)
    # --bwd-fp8: the opt-in mixed e4m3 backward (d = 128, at most the causal mask)
    bwd_fp8 = bool(args.bwd_fp8) and not fwd_only
    bmods = ea.make_mods(causal=cfg.get("causal", False), bwd_fp8=True) if bwd_fp8 else mods
    nws = ea.attn_workspace_size(ea.OP_BWD, B, Hq, Hkv, N, d, bmods)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    with_map = bool(cfg.get("window") or cfg.get("doc"))
    fused_bwd = bool(cfg.get("causal")) and with_map and d == 128  # the library's one-kernel backward

    def mk_events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record(stream)  # create the handles before passing them to the library
        return evs

    def fwd():
        ea.attn_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, mods, ws_f if nws_f else None, nws_f, stream)

    def step(ev=None):
        if ev is None:
            fwd()
            if not fwd_only:
                ea.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale, bmods, ws, nws, stream)
        else:
            ev[0].record(stream)
            fwd()
            ev[1].record(stream)
            if not fwd_only:
                ea.attn_bwd_profiled(q, k, v, o, do, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale, bmods,
                                     ws, nws, stream, ev[2:6])

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    ea.attn_status(stream)

    # The timed steps are the public calls a user makes (attn_fwd, attn_bwd),
    # events only around the loop; the per-kernel times come from a separate
    # pass through attn_bwd_profiled afterwards (its events between the
    # kernels cost about 1 % and keep the dQ kernel from starting in the dK/dV
    # kernel's tail).
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize(dev)
    t_start.record(stream)
    for s in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    barrier(world)
    ea.attn_status(stream)
    total_ms = t_start.elapsed_time(t_end)
    total_ms = allmax(world, total_ms)
    evs = [mk_events(6) for _ in range(max(3, min(args.steps, 20)))]
    for ev in evs:
        step(ev)
    torch.cuda.synchronize(dev)
    ea.attn_status(stream)
    mean = lambda a: sum(a) / len(a)  # noqa: E731
    k_fwd = [e[0].elapsed_time(e[1]) for e in evs]
    if fwd_only:
        k_pre = k_kv = k_dq = [0.0]
    else:
        k_pre = [e[2].elapsed_time(e[3]) for e in evs]
        k_kv = [e[3].elapsed_time(e[4]) for e in evs]
        k_dq = [e[4].elapsed_time(e[5]) for e in evs]

    # end to end through the public API: every step's inputs in from pinned host
    # memory and its results out, pipelined over two buffer sets
    in_names = ("q", "k", "v") if fwd_only else ("q", "k", "v", "do")
    out_names = ("o", "lse") if fwd_only else ("o", "lse", "dq", "dk", "dv")
    e2e_steps = 0 if args.no_e2e else max(3, min(args.steps, 20))
    h2d = sum(host[n].numel() * host[n].element_size() for n in in_names)
    d2h = sum(t.numel() * t.element_size() for t in (o, lse, dq, dk, dv)[:len(out_names)])
    e2e_ms = float("nan")
    link = in_pipe = None
    if e2e_steps:
        dev_in = {n: (t, torch.empty_like(t)) for n, t in zip(("q", "k", "v", "do"), (q, k, v, do))}
        dev_out = {n: (t, torch.empty_like(t)) for n, t in zip(("o", "lse", "dq", "dk", "dv"), (o, lse, dq, dk, dv))}
        host_out = {n: tuple(torch.empty(dev_out[n][0].shape, dtype=dev_out[n][0].dtype, pin_memory=True)
                             for _ in range(2)) for n in out_names}

        def compute(b):
            qb, kb, vb, dob = (dev_in[n][b] for n in ("q", "k", "v", "do"))
            ob, lb, dqb, dkb, dvb = (dev_out[n][b] for n in ("o", "lse", "dq", "dk", "dv"))
            fo, fl = ea.forward(qb, kb, vb, scale, mods, out=ob, lse=lb, stream=stream)
            if not fwd_only:
                ea.attn_bwd(qb, kb, vb, fo, dob, fl, dqb, dkb, dvb, B, Hq, Hkv, N, d, scale, bmods, ws, nws, stream)

        e2e_ms = pipelined_e2e(dev, stream, [(host[n], dev_in[n]) for n in in_names],
                               [(dev_out[n], host_out[n]) for n in out_names], compute, e2e_steps, world)
        e2e_ms = allmax(world, e2e_ms)
        in_pipe = copy_gbs_in_pipeline(*pipelined_e2e.copy_ms, h2d, d2h)
        link = link_gbs(stream, host[in_names[0]], dev_in[in_names[0]][0], dev_out[out_names[0]][0],
                        host_out[out_names[0]][0])
    ea.attn_status(stream)

    fwd_f, bwd_f = flops(cfg, docs)
    allowed = allowed_pairs(cfg, docs)
    computed = computed_pairs(ea, cfg, mods, dev)
    if fwd_only:
        bwd_f = 0.0
    ms = total_ms / args.steps
    value = job_throughput(world, fwd_f + bwd_f, ms) / 1e12
    peaks, src = load_peaks()
    peak, peak_src = bf16_peak(peaks, src, clk)
    fwd_t = fwd_f / (mean(k_fwd) * 1e-3) / 1e12
    bwd_ms = mean(k_pre) + mean(k_kv) + mean(k_dq)
    bwd_t = bwd_f / (bwd_ms * 1e-3) / 1e12 if not fwd_only else 0.0
    # Causal masks with window / document parts at d = 128 run the one-kernel
    # backward: all 5 GEMMs (S and dP recomputed, dV, dK, dQ) in one kernel,
    # between the bounds / row-statistics kernels and the dQ conversion.
    # Otherwise the dK/dV kernel does 4 of the 5 (= 2x the forward FLOPs) and
    # the dQ kernel the fifth (S and dP recomputed again, 2 more GEMMs).
    kernels = {"fwd_bf16": (mean(k_fwd), fwd_f)}
    if not fwd_only and fused_bwd:
        kernels.update({"bwd_fused": (mean(k_kv), bwd_f), "bwd_pre": (mean(k_pre), 0.0),
                        "bwd_dq_convert": (mean(k_dq), 0.0)})
    elif not fwd_only:
        kernels.update({"bwd_dkdv_e4m3" if bwd_fp8 else "bwd_dkdv": (mean(k_kv), 0.8 * bwd_f),
                        "bwd_dq": (mean(k_dq), 0.2 * bwd_f),
                        "bwd_quant_and_pre" if bwd_fp8 else "bwd_pre": (mean(k_pre), 0.0)})
    dom = max(kernels, key=lambda n: kernels[n][0])
    dom_ms, dom_flops = kernels[dom]
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    roofline = {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 1),
                "peak": round(peak, 1), "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "traffic": traffic_record(dom) if name == WORKLOAD and not args.heads else None,
                "peak_source": peak_src}
    if fwd_only:
        # a forward this small is latency / HBM bound: bytes Q+K+V in, O + LSE out
        nbytes = 2 * (B * Hq * N * d + 2 * B * Hkv * N * d + B * Hq * N * d) + 4 * B * Hq * N
        gbs = nbytes / (mean(k_fwd) * 1e-3) / 1e9
        roofline = {"kernel": "fwd_bf16", "bound": "hbm", "achieved": round(gbs, 1),
                    "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 5),
                    "traffic": None, "bytes_per_launch": nbytes,
                    "peak_source": f"{src} hbm_gbs (inputs stay in L2 between steps: warm)"}
    map_launches = (3 if cfg.get("doc") else 2) if with_map else 0  # document runs, block map, tile ranges
    bwd_launches = 0 if fwd_only else (4 if fused_bwd else 3) + map_launches + (3 if bwd_fp8 else 0)
    launches = 1 + map_launches + bwd_launches
    line = {
        "metric": (METRIC if name == WORKLOAD and not bwd_fp8 else
                   f"attention TFLOPS fwd{'' if fwd_only else '/bwd'} ({name}"
                   + (", mixed e4m3 backward: e4m3 dP and dV GEMMs)" if bwd_fp8 else ")")),
        "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 + e4m3 (dP, dV)" if bwd_fp8 else "bf16",
        "data": "synthetic",
        "config": {"workload": name, "B": B, "Hq": Hq, "Hkv": Hkv, "N": N, "d": d,
                   "mask": mods_label(cfg), "parallelism": f"replicas{world}" if world > 1 else "single",
                   "l2": l2_note(cfg)},
        "fwd_tflops": round(fwd_t, 1), "bwd_tflops": round(bwd_t, 1),
        "fwd_frac_peak": round(fwd_t / peak, 4), "bwd_frac_peak": round(bwd_t / peak, 4),
        "kernel_ms": {n: round(t, 4) for n, (t, _) in kernels.items()},
        "roofline": roofline,
        "tile_efficiency": {
            "allowed_pairs": allowed, "computed_pairs": computed, "ratio": round(allowed / computed, 4),
            "note": "allowed (i, j) pairs / pairs inside the non-skipped 128 x 128 tiles; the rest of the "
                    "gap to the peak is kernel time"},
        "e2e": None if not e2e_steps else {
            "value": round(job_throughput(world, fwd_f + bwd_f, e2e_ms) / 1e12, 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
            "pipelined": "copies in and out on their own streams, two device buffer sets",
            "link_gbs": link, "copy_gbs_in_steps": in_pipe},
        "gpu_launches": launches * args.steps,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, el, desc = oracle_sample(dict(cfg, name=name), x, args.cpu_seconds, 512, fwd_only)
        line["cpu_baseline"] = {"value": round(tf, 5), "unit": UNIT, "cores": cpu_info(),
                                "kind": "oracle", "sample": desc, "seconds": round(el, 2)}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_varlen(args, world, rank, local):
    """Packed variable-length sequences through attn_fwd_varlen /
    attn_bwd_varlen (causal inside each sequence), timed per call."""
    import exact_attention_66_gb300 as ea

    name = args.workload
    cfg = dict(gen.WORKLOADS[name])
    B, Hq, Hkv, N, d = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["N"], cfg["d"]
    scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    x = gen.make_inputs(**dict(cfg, seed=replica_seed(cfg, rank)))
    ids = x["doc_ids"][0]
    cu = np.concatenate([[0], np.cumsum(np.bincount(ids))]).astype(np.int32)
    n_seqs = len(cu) - 1
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    dcu = torch.from_numpy(cu).to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((1, Hq, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    mods = ea.make_mods(causal=True)
    nf = ea.attn_workspace_size(ea.OP_FWD_VARLEN, 1, Hq, Hkv, N, d, mods)
    nb = ea.attn_workspace_size(ea.OP_BWD_VARLEN, 1, Hq, Hkv, N, d, mods)
    wf = torch.empty(nf, dtype=torch.uint8, device=dev)
    wb = torch.empty(nb, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        ea.attn_fwd_varlen(q, k, v, o, lse, dcu, n_seqs, Hq, Hkv, N, d, scale, mods, wf, nf, stream)
        if ev is not None:
            ev[1].record(stream)
        ea.attn_bwd_varlen(q, k, v, o, do, lse, dq, dk, dv, dcu, n_seqs, Hq, Hkv, N, d, scale, mods,
                           wb, nb, stream)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    ea.attn_status(stream)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize(dev)
    t0.record(stream)
    for s in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    barrier(world)
    ea.attn_status(stream)
    ms = allmax(world, t0.elapsed_time(t1)) / args.steps
    # per-call times from a separate pass with events between the calls
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(max(3, min(args.steps, 20)))]
    for ev in evs:
        step(ev)
    torch.cuda.synchronize(dev)
    k_fwd = sum(e[0].elapsed_time(e[1]) for e in evs) / len(evs)
    k_bwd = sum(e[1].elapsed_time(e[2]) for e in evs) / len(evs)
    peaks, src = load_peaks()
    peak, peak_src = bf16_peak(peaks, src, clk)
    fwd_f, bwd_f = flops(cfg, x["doc_ids"])
    fwd_t = fwd_f / (k_fwd * 1e-3) / 1e12
    bwd_t = bwd_f / (k_bwd * 1e-3) / 1e12
    line = {
        "metric": f"attention TFLOPS fwd/bwd ({name})",
        "value": round(world * (fwd_f + bwd_f) / (ms * 1e-3) / 1e12, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": name, "B": 1, "Hq": Hq, "Hkv": Hkv, "N": N, "d": d, "n_seqs": n_seqs,
                   "mask": "causal within each packed sequence",
                   "parallelism": "single" if world == 1 else f"replicas{world}", "l2": l2_note(cfg)},
        "fwd_tflops": round(fwd_t, 1), "bwd_tflops": round(bwd_t, 1),
        "fwd_frac_peak": round(fwd_t / peak, 4), "bwd_frac_peak": round(bwd_t / peak, 4),
        "kernel_ms": {"fwd_varlen (ids, map, runs, forward)": round(k_fwd, 4),
                      "bwd_varlen (ids, map, runs, row stats, dK/dV, dQ)": round(k_bwd, 4)},
        "roofline": {"kernel": "bwd_varlen", "bound": "tensor", "achieved": round(bwd_t, 1),
                     "peak": round(peak, 1), "unit": "TFLOP/s", "frac": round(bwd_t / peak, 4), "traffic": None,
                     "peak_source": peak_src},
        "e2e": None, "gpu_launches": 10 * args.steps, "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_paged(args, world, rank, local):
    """Causal prefill forward with K/V read through a block table from a
    shuffled cache of 16-row blocks (attn_fwd_paged), beside the same forward
    on contiguous K/V."""
    import exact_attention_66_gb300 as ea

    name = args.workload
    cfg = dict(gen.WORKLOADS[name])
    if args.heads:  # smaller case of the same workload (profiling)
        cfg["Hq"] = cfg["Hkv"] = args.heads
    B, Hq, Hkv, N, d = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["N"], cfg["d"]
    scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    x = gen.make_inputs(**dict(cfg, seed=replica_seed(cfg, rank), need_do=False))
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    nb = N // 16
    num_blocks = B * nb
    perm = torch.from_numpy(np.random.default_rng(cfg["seed"]).permutation(num_blocks).astype(np.int32))
    table = perm.reshape(B, nb).to(dev)
    kc = torch.empty(num_blocks, Hkv, 16, d, dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    kc[table.reshape(-1).long()] = k.reshape(B, Hkv, nb, 16, d).permute(0, 2, 1, 3, 4).reshape(-1, Hkv, 16, d)
    vc[table.reshape(-1).long()] = v.reshape(B, Hkv, nb, 16, d).permute(0, 2, 1, 3, 4).reshape(-1, Hkv, 16, d)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    mods = ea.make_mods(causal=True)
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ea.attn_status(stream)
        return e0.elapsed_time(e1) / args.steps

    barrier(world)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ms = timed(lambda: ea.attn_fwd_paged(q, kc, vc, table, num_blocks, o, lse, B, Hq, Hkv, N, d, scale, mods,
                                         None, 0, stream))
    clk = clocks.stop()
    ms_contig = timed(lambda: ea.attn_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, mods, None, 0, stream))
    ms = allmax(world, ms)
    peaks, src = load_peaks()
    peak, peak_src = bf16_peak(peaks, src, clk)
    fwd_f, _ = flops(cfg)
    t = fwd_f / (ms * 1e-3) / 1e12
    line = {
        "metric": f"attention TFLOPS fwd ({name}, paged K/V)", "value": round(world * t, 2), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": name, "B": B, "Hq": Hq, "Hkv": Hkv, "N": N, "d": d, "mask": "causal",
                   "block_size": 16, "num_blocks": num_blocks,
                   "parallelism": "single" if world == 1 else f"replicas{world}", "l2": l2_note(cfg)},
        "fwd_tflops": round(t, 1), "fwd_frac_peak": round(t / peak, 4),
        "kernel_ms": {"fwd_paged": round(ms, 4), "fwd_contiguous_same_inputs": round(ms_contig, 4)},
        "roofline": {"kernel": "fwd_paged", "bound": "tensor", "achieved": round(t, 1), "peak": round(peak, 1),
                     "unit": "TFLOP/s", "frac": round(t / peak, 4), "traffic": None,
                     "peak_source": peak_src},
        "e2e": None, "gpu_launches": args.steps, "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def decode_bytes(B, Hq, Hkv, d, lens, T=1):
    """Algorithmic HBM bytes of one decode step: every cached K and V row of
    every sequence once, the block-table entries used, Q read, O and LSE
    written (T new tokens per sequence)."""
    lens = np.asarray(lens, np.int64)
    kv = 2 * int(lens.sum()) * Hkv * d * 2
    table = 4 * int(((lens + 15) // 16).sum()) + 4 * B
    return kv + table + 2 * B * Hq * T * d * 2 + 4 * B * Hq * T


def run_decode(args, world, rank, local):
    """One decode step per sequence over a shuffled paged K/V cache
    (attn_decode_paged): HBM-bound, reported in GB/s of algorithmic bytes
    against the measured copy bandwidth."""
    import exact_attention_66_gb300 as ea

    name = args.workload
    cfg = dict(gen.WORKLOADS[name])
    if args.batch:  # smaller case of the same workload (profiling)
        cfg["B"] = args.batch
    B, Hq, Hkv, N, d = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["N"], cfg["d"]
    T = cfg.get("q_len", 1)
    scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    x = gen.paged_decode_inputs(**dict(cfg, seed=replica_seed(cfg, rank)))
    q_host = x["q"].pin_memory()
    q = q_host.to(dev)
    kc, vc = x["k_cache"].to(dev), x["v_cache"].to(dev)
    table = torch.from_numpy(x["block_table"]).to(dev)
    lens = torch.from_numpy(x["seqlens"]).to(dev)
    num_blocks, max_blocks = kc.shape[0], table.shape[1]
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, T) if T > 1 else (B, Hq), dtype=torch.float32, device=dev)
    nws = ea.attn_decode_workspace_size(B, Hq, Hkv, T, max_blocks, d, None)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(bufs=None):
        qq, oo, ll = bufs if bufs is not None else (q, o, lse)
        ea.attn_decode_paged(qq, kc, vc, table, max_blocks, lens, num_blocks, oo, ll, B, Hq, Hkv, T, d, scale,
                             None, ws, nws, stream)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        barrier(world)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        ea.attn_status(stream)
        return e0.elapsed_time(e1) / args.steps

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ms = timed(step)
    clk = clocks.stop()
    # end to end: the new tokens' queries in, outputs back (the cache stays
    # resident), pipelined over two buffer sets
    q2, o2, l2 = (q, torch.empty_like(q)), (o, torch.empty_like(o)), (lse, torch.empty_like(lse))
    pin2 = lambda t: tuple(torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for _ in range(2))  # noqa: E731
    ms_e2e = pipelined_e2e(dev, stream, [(q_host, q2)], [(o2, pin2(o)), (l2, pin2(lse))],
                           lambda b: step((q2[b], o2[b], l2[b])), max(3, args.steps), world)
    ea.attn_status(stream)
    ms, ms_e2e = allmax(world, ms), allmax(world, ms_e2e)
    peaks, src = load_peaks()
    nbytes = decode_bytes(B, Hq, Hkv, d, x["seqlens"], T)
    gbs = nbytes / (ms * 1e-3) / 1e9
    hbm = peaks["hbm_gbs"]
    bytes_io = q.numel() * 2 + o.numel() * 2 + lse.numel() * 4
    line = {
        "metric": f"paged decode HBM throughput ({name})", "value": round(world * gbs, 1), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": name, "B": B, "Hq": Hq, "Hkv": Hkv, "d": d, "new_tokens": T, "max_context": N,
                   "context_lengths": f"uniform in [{cfg['min_len']}, {N}], total {int(x['seqlens'].sum())}",
                   "block_size": 16, "num_blocks": num_blocks,
                   "parallelism": "single" if world == 1 else f"replicas{world}",
                   "l2": f"cache larger than L2 ({2 * kc.numel() * 2 / 2**20:.0f} MiB of K and V)"},
        "tokens_per_s": round(world * B * T / (ms * 1e-3), 1),
        "algorithmic_bytes_per_step": nbytes,
        "roofline": {"kernel": "decode_paged (setup, main and merge launches together)", "bound": "hbm",
                     "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4),
                     "traffic": traffic_record("decode_paged") if not args.batch and T == 1 else None,
                     "peak_source": f"{src} hbm_gbs"},
        "e2e": {"value": round(world * nbytes / (ms_e2e * 1e-3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": q.numel() * 2, "d2h_bytes_per_step": bytes_io - q.numel() * 2,
                "ms_per_step": round(ms_e2e, 4),
                "pipelined": "copies in and out on their own streams, two device buffer sets"},
        "gpu_launches": 3 * args.steps, "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_fp8(args, world, rank, local):
    """The FP8 workload: signed-Hadamard + e4m3 prologue, then the e4m3
    forward (non-causal), timed per kernel group with CUDA events."""
    import exact_attention_66_gb300 as ea

    name = args.workload
    cfg = dict(gen.WORKLOADS[name])
    if args.heads:  # smaller case of the same workload (profiling)
        cfg["Hq"] = cfg["Hkv"] = args.heads
    B, Hq, Hkv, N, d = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["N"], cfg["d"]
    scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    x = gen.make_inputs(**dict(cfg, seed=replica_seed(cfg, rank), need_do=False))
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    signs = torch.from_numpy(gen.hadamard_signs(Hkv, d, cfg["seed"] + 20)).to(dev)
    q8 = torch.empty(q.shape, dtype=torch.uint8, device=dev)
    k8 = torch.empty(k.shape, dtype=torch.uint8, device=dev)
    v8 = torch.empty(v.shape, dtype=torch.uint8, device=dev)
    sc = torch.empty(B * Hq + 2 * B * Hkv, dtype=torch.float32, device=dev)
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    nq = ea.attn_workspace_size(ea.OP_QUANT_FP8, B, Hq, Hkv, N, d, None)
    wq = torch.empty(nq, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        ea.attn_hadamard_quant_fp8(q, k, v, q8, k8, v8, sc, signs, B, Hq, Hkv, N, d, wq, nq, stream)
        if ev is not None:
            ev[1].record(stream)
        ea.attn_fwd_fp8(q8, k8, v8, sc, o, lse, B, Hq, Hkv, N, d, scale, None, None, 0, stream)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    ea.attn_status(stream)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize(dev)
    t0.record(stream)
    for s in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    barrier(world)
    ea.attn_status(stream)
    ms = allmax(world, t0.elapsed_time(t1)) / args.steps
    # per-call times from a separate pass with events between the calls
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(max(3, min(args.steps, 20)))]
    for ev in evs:
        step(ev)
    torch.cuda.synchronize(dev)
    k_pro = sum(e[0].elapsed_time(e[1]) for e in evs) / len(evs)
    k_fwd = sum(e[1].elapsed_time(e[2]) for e in evs) / len(evs)
    # the same prologue with RoPE fused in front of the rotation
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for rep in range(2):
        if rep:
            r0.record(stream)
        for _ in range(args.steps):
            ea.attn_rope_hadamard_quant_fp8(q, k, v, q8, k8, v8, sc, signs, B, Hq, Hkv, N, d, 10000.0,
                                            wq, nq, stream)
    r1.record(stream)
    torch.cuda.synchronize(dev)
    ea.attn_status(stream)
    k_rope = r0.elapsed_time(r1) / args.steps
    peaks, src = load_peaks()
    bf16p, peak_src = bf16_peak(peaks, src, clk)
    fp8_peak = 2.0 * bf16p  # dense e4m3 = 2x bf16 (nominal ratio)
    fwd_f = 4.0 * Hq * d * allowed_pairs(cfg)
    fwd_t = fwd_f / (k_fwd * 1e-3) / 1e12
    rows = B * Hq * N + 2 * B * Hkv * N
    pro_bytes = rows * (2 * d + d)  # algorithmic: every bf16 row read once, its e4m3 row written
    moved = rows * (2 * 2 * d + d)  # what the two passes move (the amax pass reads every row too)
    pro_gbs = pro_bytes / (k_pro * 1e-3) / 1e9
    line = {
        "metric": f"attention TFLOPS fwd ({name}, e4m3)", "value": round(world * fwd_f / (ms * 1e-3) / 1e12, 2),
        "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3", "data": "synthetic (0.1 % of entries x50)",
        "config": {"workload": name, "B": B, "Hq": Hq, "Hkv": Hkv, "N": N, "d": d, "mask": "none",
                   "parallelism": "single" if world == 1 else f"replicas{world}", "l2": l2_note(cfg)},
        "fwd_tflops": round(fwd_t, 1), "fwd_frac_fp8_peak": round(fwd_t / fp8_peak, 4),
        "kernel_ms": {"hadamard_quant": round(k_pro, 4), "fwd_fp8": round(k_fwd, 4)},
        "roofline": {"kernel": "fwd_fp8", "bound": "tensor", "achieved": round(fwd_t, 1), "peak": fp8_peak,
                     "unit": "TFLOP/s", "frac": round(fwd_t / fp8_peak, 4),
                     "traffic": traffic_record("fwd_fp8") if not args.heads else None,
                     "peak_source": f"{peak_src}, x 2 (nominal e4m3/bf16 ratio)"},
        "prologue": {"achieved": round(pro_gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(pro_gbs / peaks["hbm_gbs"], 4), "bytes": pro_bytes,
                     "traffic": traffic_record("hadamard_quant") if not args.heads else None,
                     "bytes_moved_two_passes": moved, "moved_gbs": round(moved / (k_pro * 1e-3) / 1e9, 1),
                     "with_rope_ms": round(k_rope, 4),
                     "with_rope_gbs": round(pro_bytes / (k_rope * 1e-3) / 1e9, 1)},
        "e2e": None, "gpu_launches": 4 * args.steps, "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args, world, rank):
    """The fp64 CPU oracle as the reference arm, on bounded slices per step."""
    if rank != 0:
        return
    cfg = dict(gen.WORKLOADS[WORKLOAD])
    x = gen.make_inputs(cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["N"], cfg["d"], seed=cfg["seed"])
    # size each step's slice so the whole run stays within about two minutes
    per_step = max(0.05, min(2.0, 120.0 / max(1, args.steps + args.warmup)))
    t0 = time.perf_counter()
    oracle_sample(cfg, x, 0.0, 64)
    t64 = time.perf_counter() - t0
    rows = int(max(16, min(2048, 64 * per_step / max(t64, 1e-3))) // 16 * 16)
    for _ in range(args.warmup):
        oracle_sample(cfg, x, 0.0, rows)
    tf_all, el_all = [], 0.0
    for _ in range(args.steps):
        tf, el, desc = oracle_sample(cfg, x, 0.0, rows)
        tf_all.append(tf)
        el_all += el
    value = statistics.mean(tf_all)
    ms = 1e3 * el_all / args.steps
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": cfg["B"], "Hq": cfg["Hq"], "Hkv": cfg["Hkv"],
                   "N": cfg["N"], "d": cfg["d"], "mask": "causal"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cpu_info(), "kind": "oracle",
                         "sample": f"per step: one slice of {rows} query rows (forward + their "
                                   f"backward contributions) of {WORKLOAD}"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="time budget of the oracle CPU baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host copies) leg")
    ap.add_argument("--workload", choices=sorted(gen.WORKLOADS), default=WORKLOAD,
                    help="workload to time; the default is the one the metric is quoted on")
    ap.add_argument("--batch", type=int, default=0,
                    help="paged decode workloads only: this many sequences instead of the workload's (profiling)")
    ap.add_argument("--bwd-fp8", action="store_true",
                    help="time the opt-in mixed e4m3 backward (ATTN_MOD_BWD_FP8; d = 128, at most a causal mask)")
    ap.add_argument("--heads", type=int, default=0,
                    help="query heads for a smaller profiling case (8 per KV head; fp8_outliers_16k: as many KV "
                         "heads); default: the workload's")
    args = ap.parse_args()
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, world, rank)
        return
    world, rank, local = dist_setup()
    run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python3
"""Benchmark of the GQA attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {ours,reference}]

One step = one decode token through the 80 attention layers of a Llama3-70B
shaped model at S_kv = 8192 (B=1, H_q=64, H_kv=8, d=128 per layer; 80 KV
caches, 2.7 GB resident in HBM, so L2 never holds a layer's cache between
uses), replayed as one CUDA graph of 80 ``gqa_attn_decode`` calls, followed by
one 8K causal prefill call (B=1, T_q=S_kv=8192; 335 MB of operands, larger than
L2). ``value`` is decode KV GB/s; the prefill TFLOPS are in ``prefill``.

For N > 1 (torchrun) every rank runs the same work on its own GPU with no
data-path collective (weak scaling); a barrier and a max over ranks bracket
the timed region. ``--impl reference`` times the fp64 CPU oracle on a bounded
sample of the same workloads instead.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode KV GB/s (% of 8 TB/s) & tok/s; prefill TFLOPS (% bf16 peak)"
NOMINAL_HBM_GBS = 8000.0
NOMINAL_BF16_TFLOPS = 2250.0
LAYERS = 80  # Llama3-70B decoder layers
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_traffic():
    """Per-launch DRAM bytes from the committed ncu summaries, kept only while the
    profiled kernel source is unchanged (sha256 match); else None."""
    import hashlib

    out = {}
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return out
    for key, rec in json.load(open(path)).items():
        if not isinstance(rec, dict) or "sha256" not in rec:
            continue
        src = os.path.join(ROOT, rec["source"])
        if os.path.exists(src) and hashlib.sha256(open(src, "rb").read()).hexdigest() == rec["sha256"]:
            out[key] = rec["bytes_per_launch"]
    return out


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


# ---------------------------------------------------------------- workloads


def decode_bytes(B, H_q, H_kv, d, seqlens):
    """Algorithmic bytes of one decode call: K and V rows read, q read, O and lse written."""
    kv = 2 * H_kv * d * 2 * int(sum(seqlens))
    return kv, kv + B * H_q * d * 2 * 2 + B * H_q * 4


def prefill_flops(B, H_q, d, T_q, S_kv, q_offset, causal):
    """4 * d flops per visible (query, key) pair (Q K^T and P V), visible pairs only."""
    if causal:
        pairs = sum(min(S_kv, q_offset + t + 1) for t in range(T_q))
    else:
        pairs = T_q * S_kv
    return 4.0 * d * H_q * B * pairs


def prefill_bytes(B, H_q, H_kv, d, T_q, S_kv):
    return (2 * B * H_q * T_q * d * 2) + (2 * B * H_kv * S_kv * d * 2) + B * H_q * T_q * 4


# ------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples every 10 ms; stop(window)
    keeps the samples taken inside the timed region (wall-clock seconds)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "10"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, window=None):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        lines = open(self.path).read().splitlines()
        os.unlink(self.path)
        return self.summarise(lines, window)

    @classmethod
    def summarise(cls, lines, window=None):
        """Median SM clock, max clock and active throttle reasons of the samples
        whose timestamps fall in `window` (t0, t1) (all samples if none do)."""
        import datetime

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        def stamp(x):
            try:
                return datetime.datetime.strptime(x, "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                return None

        rows = [[x.strip() for x in ln.split(",")] for ln in lines]
        rows = [r for r in rows if len(r) >= 10]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "samples_total": 0}
        inside = rows
        if window is not None:
            t0, t1 = window
            inside = [r for r in rows
                      if stamp(r[0]) is not None and t0 - 0.005 <= stamp(r[0]) <= t1 + 0.005]
        use = inside or rows
        sm = [num(r[2]) for r in use if num(r[2]) is not None]
        mx = [num(r[3]) for r in use if num(r[3]) is not None]
        reasons = sorted({cls.REASONS[i] for r in use for i in range(4) if r[6 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "samples_total": len(rows),
                "window": "timed region" if inside else "whole run (no sample inside it)"}


# --------------------------------------------------------------- CPU oracle


def cpu_oracle_sample(seconds: float, steps: int = 1, procs: int = 1):
    """Times the fp64 oracle, as it stands, on rows of the two workloads.

    Runs `procs` fresh single-threaded worker processes side by side (each on
    its own rows); each of `steps` samples spends about `seconds` of CPU time
    per process. Returns one dict per step with decode GB/s (KV bytes of whole
    decode calls, pro rata per query head) and prefill TFLOPS over all
    processes (rows summed, the slowest process's time), and the process count.
    """
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    running = [subprocess.Popen(
        [sys.executable, os.path.abspath(__file__), "--cpu-worker", str(seconds),
         "--cpu-worker-steps", str(steps), "--cpu-worker-offset", str(i)],
        env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
        for i in range(procs)]
    per_proc = []
    for pr in running:
        out, err = pr.communicate(timeout=300 + 3 * seconds * steps)
        if pr.returncode != 0:
            raise RuntimeError(err[-2000:])
        per_proc.append(json.loads(out.strip().splitlines()[-1]))
    res = []
    for st in range(steps):
        xs = [pp[st] for pp in per_proc]
        dec_s = max(x["decode_s"] for x in xs)
        pre_s = max(x["prefill_s"] for x in xs)
        res.append({"decode_gbs": sum(x["decode_bytes"] for x in xs) / dec_s / 1e9,
                    "decode_rows": sum(x["decode_rows"] for x in xs), "decode_s": dec_s,
                    "prefill_tflops": sum(x["prefill_flops"] for x in xs) / pre_s / 1e12,
                    "prefill_rows": sum(x["prefill_rows"] for x in xs), "prefill_s": pre_s,
                    "threads": procs})
    return res


def cpu_worker(seconds: float, steps: int, offset: int = 0):
    import torch

    torch.set_num_threads(1)
    import oracle
    from gqa_attention_split_gb300 import workloads as wl

    w = wl.LLAMA70B_DECODE_8K
    q, k, v, sl = wl.decode_inputs(w)
    kv_bytes, _ = decode_bytes(w.B, w.H_q, w.H_kv, w.d, sl.tolist())
    p = wl.CAUSAL_PREFILL_8K
    qp, kp, vp = wl.prefill_inputs(p)
    res = []
    rows = n = 0
    for _ in range(steps):
        t0 = time.perf_counter()
        r0 = rows
        while time.perf_counter() - t0 < seconds / 2 or rows == r0:
            h = (rows + 7 * offset) % w.H_q
            oracle.attention_rows(q[:, :, None], k, v, [(0, h, 0)], scale=w.scale,
                                  seqlens=sl.tolist())
            rows += 1
        td = time.perf_counter() - t0
        t0 = time.perf_counter()
        flops = 0.0
        n0 = n
        while time.perf_counter() - t0 < seconds / 2 or n == n0:
            m = n + 131 * offset
            t = (m * 997) % p.T_q  # spread over the causal triangle
            oracle.attention_rows(qp, kp, vp, [(0, (m * 13) % p.H_q, t)], scale=p.scale,
                                  causal=True, q_offset=p.q_offset)
            flops += 4.0 * p.d * min(p.S_kv, p.q_offset + t + 1)
            n += 1
        tp = time.perf_counter() - t0
        res.append({"decode_bytes": kv_bytes * (rows - r0) / w.H_q, "decode_rows": rows - r0,
                    "decode_s": td, "prefill_flops": flops, "prefill_rows": n - n0,
                    "prefill_s": tp})
    print(json.dumps(res))


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def bench_config(world: int) -> dict:
    """The workload both arms run (the reference arm prints the same dict)."""
    from gqa_attention_split_gb300 import workloads as wl

    w, p = wl.LLAMA70B_DECODE_8K, wl.CAUSAL_PREFILL_8K
    return {"workload": f"{LAYERS} x {w.name} decode (graph) + {p.name}",
            "decode": {"B": w.B, "H_q": w.H_q, "H_kv": w.H_kv, "d": w.d, "S_kv": w.S_max,
                       "layers": LAYERS},
            "prefill": {"B": p.B, "H_q": p.H_q, "H_kv": p.H_kv, "d": p.d, "T_q": p.T_q,
                        "S_kv": p.S_kv, "causal": True},
            "l2": "inputs larger than L2: 80 distinct 33.5 MB KV caches per step; "
                  "prefill operands 335 MB",
            "parallelism": f"replicas x{world}"}


# ------------------------------------------------------------------ GPU arm


def aggregate_max(values, device, world):
    """Element-wise max over ranks (the slowest rank sets the time)."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist

    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def run_ours(args, rank, world, local_rank):
    import torch

    from gqa_attention_split_gb300 import api
    from gqa_attention_split_gb300 import build as _build
    from gqa_attention_split_gb300 import workloads as wl

    _build.build()
    api.lib()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peaks, peak_kind = load_peaks()

    # ---- decode: 80 layers of the Llama3-70B 8K decode shape
    w = wl.LLAMA70B_DECODE_8K
    q0, k0, v0, sl0 = wl.decode_inputs(w)
    gen = torch.Generator(device=dev).manual_seed(w.seed * 1000 + rank)
    qs = torch.empty((LAYERS,) + tuple(q0.shape), dtype=torch.bfloat16, device=dev)
    ks = torch.empty((LAYERS,) + tuple(k0.shape), dtype=torch.bfloat16, device=dev)
    vs = torch.empty_like(ks)
    qs.copy_(torch.randn(qs.shape, generator=gen, device=dev).to(torch.bfloat16))
    for L_ in range(LAYERS):  # layer by layer to bound the fp32 temporaries
        ks[L_].copy_(torch.randn(k0.shape, generator=gen, device=dev).to(torch.bfloat16))
        vs[L_].copy_(torch.randn(v0.shape, generator=gen, device=dev).to(torch.bfloat16))
    qs[0].copy_(q0)
    ks[0].copy_(k0)
    vs[0].copy_(v0)
    seqlens = sl0.to(dev)
    os_ = torch.empty_like(qs)
    lses = torch.empty((LAYERS, w.B, w.H_q), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ns = args.num_splits or api.gqa_attn_pick_num_splits(w.B, w.H_kv, w.S_max, sms)

    def decode_layers():
        for L_ in range(LAYERS):
            api.decode(qs[L_], ks[L_], vs[L_], seqlens, num_splits=ns, out=os_[L_],
                       lse=lses[L_])

    with torch.cuda.stream(stream):
        decode_layers()  # allocates the stream's workspace before capture
    stream.synchronize()
    api.check(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        decode_layers()
    kv_b, alg_b = decode_bytes(w.B, w.H_q, w.H_kv, w.d, sl0.tolist())

    # ---- prefill: one 8K causal call (if the library has the prefill kernel)
    p = wl.CAUSAL_PREFILL_8K
    qp, kp, vp = (t.to(dev) for t in wl.prefill_inputs(p))
    op = torch.empty_like(qp)
    lsep = torch.empty((p.B, p.H_q, p.T_q), dtype=torch.float32, device=dev)
    have_prefill = True
    try:
        with torch.cuda.stream(stream):
            api.prefill(qp, kp, vp, q_offset=p.q_offset, causal=True, out=op, lse=lsep)
    except api.GqaError as e:
        if e.code != api.GQA_ERR_UNSUPPORTED:
            raise
        have_prefill = False
    pf_flops = prefill_flops(p.B, p.H_q, p.d, p.T_q, p.S_kv, p.q_offset, True)

    def prefill_call():
        api.prefill(qp, kp, vp, q_offset=p.q_offset, causal=True, out=op, lse=lsep)

    splits_active = sum(math.ceil(int(s) / math.ceil(w.S_max / ns)) for s in sl0.tolist())
    # the combine kernel runs only when a row spans several clusters
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    combine = ns // api.gqa_attn_decode_cluster_size(w.B, w.H_kv, ns, sms) > 1
    launches_decode = LAYERS * (1 + (1 if combine else 0))
    launches_prefill = 1 if have_prefill else 0

    def one_step(ev):
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            graph.replay()
            ev[1].record(stream)
            if have_prefill:
                prefill_call()
            ev[2].record(stream)

    for _ in range(args.warmup):
        one_step([torch.cuda.Event(enable_timing=True) for _ in range(3)])
    stream.synchronize()
    api.check(stream)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)  # let the sampler take its first readings
    t_wall0 = time.perf_counter()
    t_epoch0 = time.time()
    for i in range(args.steps):
        one_step(evs[i])
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    t_epoch1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    time.sleep(0.05)  # the sampler's last readings of the region
    clk = clocks.stop(window=(t_epoch0, t_epoch1))
    api.check(stream)

    # the same 80 decode calls as plain launches (no graph), after the timed
    # region, for reference
    with torch.cuda.stream(stream):
        pl0, pl1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        pl0.record(stream)
        for _ in range(3):
            decode_layers()
        pl1.record(stream)
    stream.synchronize()
    api.check(stream)
    plain_call_us = pl0.elapsed_time(pl1) * 1e3 / (3 * LAYERS)

    # one decode call alone, L2 flushed before it (a 256 MB write), as a decode
    # step whose neighbours are not attention calls sees it. A GPU-side sleep
    # (~100 us) ahead of the start event keeps the host's launch work for the
    # call out of the timed interval; no other kernel overlaps the call.
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    lone = []
    with torch.cuda.stream(stream):
        for i in range(23):
            flush.fill_(i & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            stream.synchronize()
            torch.cuda._sleep(200_000)
            e0.record(stream)
            api.decode(qs[i % LAYERS], ks[i % LAYERS], vs[i % LAYERS], seqlens, num_splits=ns,
                       out=os_[0], lse=lses[0])
            e1.record(stream)
            stream.synchronize()
            if i >= 3:
                lone.append(e0.elapsed_time(e1) * 1e3)
    api.check(stream)
    del flush
    lone_call_us = statistics.median(lone)

    dec_ms = sum(e[0].elapsed_time(e[1]) for e in evs)
    pre_ms = sum(e[1].elapsed_time(e[2]) for e in evs)
    dec_ms, pre_ms, tot_ms = aggregate_max([dec_ms, pre_ms, dec_ms + pre_ms], dev, world)
    K = args.steps
    dec_call_s = dec_ms / 1e3 / (K * LAYERS)
    dec_gbs_rank = kv_b / dec_call_s / 1e9
    value = dec_gbs_rank * world  # every rank decodes its own batch (weak scaling)
    pre_s = pre_ms / 1e3 / K if have_prefill else None
    pre_tflops = pf_flops / pre_s / 1e12 if have_prefill else None

    # ---- end to end through the same entry points, host buffers in pinned memory
    e2e = run_e2e(api, torch, dev, stream, w, ns, p, have_prefill, args, world)

    hbm_peak = float(peaks["hbm_gbs"])
    tc_peak = float(peaks["bf16_tflops"])  # burst: the prefill call is ~1 ms
    traffic = load_traffic()
    roof_decode = {"bound": "hbm", "achieved": alg_b / dec_call_s / 1e9, "peak": hbm_peak,
                   "unit": "GB/s", "frac": alg_b / dec_call_s / 1e9 / hbm_peak,
                   "traffic": traffic.get("decode"),
                   "kernel": "split_kernel (one per gqa_attn_decode call; combine_kernel "
                             + ("also launched" if combine else "not launched: one cluster "
                                "covers each row") + ")",
                   "algorithmic_bytes_per_launch": alg_b,
                   "peak_kind": peak_kind + " copy bandwidth"}
    res = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": tot_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic N(0,1) bf16, seeded; random KV caches (no trained weights)",
        "config": bench_config(world),
        "decode": {"kv_GBps": value, "pct_of_8TBps": 100 * dec_gbs_rank / NOMINAL_HBM_GBS,
                   "pct_of_measured_hbm": 100 * dec_gbs_rank / hbm_peak,
                   "us_per_layer_call": dec_call_s * 1e6,
                   "num_splits": ns, "active_splits": splits_active,
                   "plain_loop_us_per_layer_call": plain_call_us,
                   "lone_call_us": lone_call_us,
                   "lone_call_GBps": kv_b / lone_call_us / 1e3,
                   "lone_call_note": "one call alone after an L2 flush (host launch work "
                                     "hidden behind a GPU sleep), median of 20; the graph "
                                     "figure overlaps consecutive calls",
                   "tok_per_s_one_layer": w.B / dec_call_s,
                   "tok_per_s_80_layers": w.B / (dec_call_s * LAYERS)},
        "prefill": None if not have_prefill else {
            "TFLOPS": pre_tflops * world, "ms_per_call": pre_s * 1e3,
            "pct_of_nominal_2250": 100 * pre_tflops / NOMINAL_BF16_TFLOPS,
            "pct_of_measured_bf16": 100 * pre_tflops / float(peaks["bf16_tflops"]),
            "flops_per_call": pf_flops},
        "roofline": roof_decode,
        "e2e": e2e,
        "gpu_launches": K * (launches_decode + launches_prefill),
        "clocks": clk,
        "wall_s_timed_region": t_wall,
    }
    if have_prefill:
        # `roofline` describes the kernel with the larger share of the measured
        # step; the other one is reported beside it as roofline_<name>.
        pk = ("prefill_pair_kernel<false> (head pairs)" if (p.H_q // p.H_kv) % 2 == 0
              else "prefill_pair_kernel<true> (block pairs)")
        roof_prefill = {
            "bound": "tensor", "achieved": pre_tflops, "peak": tc_peak, "unit": "TFLOP/s",
            "frac": pre_tflops / tc_peak, "traffic": traffic.get("prefill"), "kernel": pk,
            "algorithmic_flops_per_launch": pf_flops,
            "peak_kind": peak_kind + " bf16 matmul burst"}
        if pre_ms >= dec_ms:
            res["roofline"], res["roofline_decode"] = roof_prefill, roof_decode
        else:
            res["roofline"], res["roofline_prefill"] = roof_decode, roof_prefill
        res["step_share"] = {"decode": dec_ms / tot_ms, "prefill": pre_ms / tot_ms}
    return res


def run_e2e(api, torch, dev, stream, w, ns, p, have_prefill, args, world):
    """Same metric through the public API with pinned host inputs/outputs (one layer/call)."""
    from gqa_attention_split_gb300 import workloads as wl

    q, k, v, sl = wl.decode_inputs(w)
    hq, hk, hv, hs = (t.pin_memory() for t in (q, k, v, sl))
    dq, dk, dv, ds = (torch.empty_like(t, device=dev) for t in (q, k, v, sl))
    ho = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    hl = torch.empty((w.B, w.H_q), dtype=torch.float32).pin_memory()
    do = torch.empty_like(dq)
    dl = torch.empty((w.B, w.H_q), dtype=torch.float32, device=dev)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hs))
    d2h = ho.numel() * 2 + hl.numel() * 4
    kv_b, _ = decode_bytes(w.B, w.H_q, w.H_kv, w.d, sl.tolist())
    steps = max(3, min(args.steps, 50))

    def step():
        for src, dst in ((hq, dq), (hk, dk), (hv, dv), (hs, ds)):
            dst.copy_(src, non_blocking=True)
        api.decode(dq, dk, dv, ds, num_splits=ns, out=do, lse=dl)
        ho.copy_(do, non_blocking=True)
        hl.copy_(dl, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
    stream.synchronize()
    t = e0.elapsed_time(e1) / 1e3 / steps
    out = {"value": kv_b / t / 1e9 * world, "unit": "GB/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "what": f"one {w.name} decode call per step"}
    if have_prefill:
        qp, kp, vp = wl.prefill_inputs(p)
        hqp, hkp, hvp = (x.pin_memory() for x in (qp, kp, vp))
        dqp, dkp, dvp = (torch.empty_like(x, device=dev) for x in (qp, kp, vp))
        hop = torch.empty(qp.shape, dtype=torch.bfloat16).pin_memory()
        hlp = torch.empty((p.B, p.H_q, p.T_q), dtype=torch.float32).pin_memory()
        dop = torch.empty_like(dqp)
        dlp = torch.empty((p.B, p.H_q, p.T_q), dtype=torch.float32, device=dev)

        def pstep():
            for src, dst in ((hqp, dqp), (hkp, dkp), (hvp, dvp)):
                dst.copy_(src, non_blocking=True)
            api.prefill(dqp, dkp, dvp, q_offset=p.q_offset, causal=True, out=dop, lse=dlp)
            hop.copy_(dop, non_blocking=True)
            hlp.copy_(dlp, non_blocking=True)

        psteps = max(3, min(args.steps, 10))
        with torch.cuda.stream(stream):
            pstep()
            stream.synchronize()
            e0.record(stream)
            for _ in range(psteps):
                pstep()
            e1.record(stream)
        stream.synchronize()
        tp = e0.elapsed_time(e1) / 1e3 / psteps
        flops = prefill_flops(p.B, p.H_q, p.d, p.T_q, p.S_kv, p.q_offset, True)
        out["prefill"] = {"value": flops / tp / 1e12 * world, "unit": "TFLOP/s",
                          "h2d_bytes_per_step": sum(x.numel() * 2 for x in (qp, kp, vp)),
                          "d2h_bytes_per_step": hop.numel() * 2 + hlp.numel() * 4}
    return out


def run_reference(args, rank, world):
    """The fp64 CPU oracle as the reference arm, on this arm's config and metric,
    on every host core (one single-threaded process per core, own rows each)."""
    if rank != 0:
        return None
    # The whole run stays within a few minutes: about 150 s of CPU work per core.
    per = max(0.2, min(args.ref_seconds, 150.0 / (args.warmup + args.steps)))
    procs = host_cores()
    per_step = cpu_oracle_sample(per, args.warmup + args.steps, procs=procs)
    timed = per_step[args.warmup:]
    info = timed[-1]
    dec = statistics.mean(x["decode_gbs"] for x in timed)
    pre = statistics.mean(x["prefill_tflops"] for x in timed)
    sample = (f"per step: {info['decode_rows']} query-head rows of the 8K decode "
              f"({info['decode_s']:.1f}s) and {info['prefill_rows']} rows of the 8K causal "
              f"prefill ({info['prefill_s']:.1f}s), fp64 oracle, {procs} single-threaded "
              "processes")
    return {"impl": "reference", "metric": METRIC, "value": dec, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.mean(x["decode_s"] + x["prefill_s"] for x in timed),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic N(0,1) bf16 widened to fp64, seeded",
            "config": bench_config(world),
            "prefill": {"TFLOPS": pre},
            "cpu_baseline": {"value": dec, "unit": "GB/s", "cores": procs,
                             "host_cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": dec, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_case(args):
    """One workload alone: plain launches for profiling and quick timing, and for the
    decode cases also back-to-back calls in a CUDA graph over rotating caches."""
    import torch

    from gqa_attention_split_gb300 import api
    from gqa_attention_split_gb300 import build as _build
    from gqa_attention_split_gb300 import workloads as wl

    _build.build()
    api.lib()
    dev = torch.device("cuda", 0)
    graph_call = None  # decode cases: the same call in a CUDA graph over rotating caches
    extra = None
    if args.case in ("decode8k_q8", "ragged128k_q8", "decode8k_q4", "ragged128k_q4"):
        # INT8 / INT4 cache: bytes read are the codes plus one fp32 scale per
        # token for K and for V; the rate is also given as the bf16 bytes it
        # replaces
        int4 = args.case.endswith("_q4")
        quant = api.quantize_kv_q4 if int4 else api.quantize_kv_q8
        dec = api.decode_q4 if int4 else api.decode_q8
        w = wl.RAGGED_DECODE_128K if args.case.startswith("ragged") else wl.LLAMA70B_DECODE_8K
        q, k, v, sl = (t.to(dev) for t in wl.decode_inputs(w))
        caches = [quant(k, v)]
        del k, v
        tokens = sum(min(int(x), w.S_max) for x in sl.tolist())
        q8_bytes = tokens * w.H_kv * ((w.d if int4 else 2 * w.d) + 8)
        bf16_bytes = tokens * w.H_kv * 2 * w.d * 2
        per_set = sum(t.numel() * t.element_size() for t in caches[0])
        for _ in range(max(1, -(-300_000_000 // per_set)) - 1):
            kk = torch.randn(w.B, w.H_kv, w.S_max, w.d, device=dev).to(torch.bfloat16)
            vv = torch.randn(w.B, w.H_kv, w.S_max, w.d, device=dev).to(torch.bfloat16)
            caches.append(quant(kk, vv))
            del kk, vv
        torch.cuda.synchronize()
        api.check()

        def one(cset):
            dec(q, *cset, sl, num_splits=args.num_splits)

        def call():
            one(caches[0])

        gs = torch.cuda.Stream()
        with torch.cuda.stream(gs):
            for cset in caches:
                one(cset)
        gs.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            for cset in caches:
                one(cset)

        def graph_call():
            graph.replay()

        graph_calls = len(caches)
        work, unit = q8_bytes / 1e9, "GB/s"
        extra = {("int4" if int4 else "int8") + "_bytes_per_call": q8_bytes,
                 "bf16_equivalent_bytes_per_call": bf16_bytes}
    elif args.case in ("decode8k", "ragged128k", "ring8k", "decode128k"):
        w = {"ragged128k": wl.RAGGED_DECODE_128K,
             "decode128k": wl.LLAMA70B_DECODE_128K_B1}.get(args.case, wl.LLAMA70B_DECODE_8K)
        q, k, v, sl = (t.to(dev) for t in wl.decode_inputs(w))
        ring = args.case == "ring8k"
        if ring:
            # ring-buffer cache with 4 sinks and 8192 slots; the rows have produced
            # 3 x 8192 + 7 tokens, so every slot is live (same bytes as decode8k)
            sl = torch.full((w.B,), 3 * w.S_max + 7, dtype=torch.int32, device=dev)
        live = [min(int(x), w.S_max) for x in sl.tolist()]
        kv_b, _ = decode_bytes(w.B, w.H_q, w.H_kv, w.d, live)

        def one(kk, vv):
            if ring:
                api.decode_ring(q, kk, vv, sl, n_sink=4, num_splits=args.num_splits)
            else:
                api.decode(q, kk, vv, sl, num_splits=args.num_splits)

        def call():
            one(k, v)

        # enough distinct caches that L2 (129 MB) never holds the next one
        n_sets = max(1, -(-300_000_000 // (2 * k.numel() * k.element_size())))
        sets = [(k, v)] + [(torch.randn(k.shape, device=dev).to(torch.bfloat16),
                            torch.randn(v.shape, device=dev).to(torch.bfloat16))
                           for _ in range(n_sets - 1)]
        gs = torch.cuda.Stream()
        with torch.cuda.stream(gs):
            for kk, vv in sets:
                one(kk, vv)  # sizes the stream's workspace before capture
        gs.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            for kk, vv in sets:
                one(kk, vv)

        def graph_call():
            graph.replay()

        graph_calls = len(sets)
        work, unit = kv_b / 1e9, "GB/s"
    elif args.case in ("prefill8k", "chunked32k", "prefill8k_mha"):
        p = {"prefill8k": wl.CAUSAL_PREFILL_8K, "chunked32k": wl.CHUNKED_PREFILL_32K,
             "prefill8k_mha": wl.CAUSAL_PREFILL_8K_MHA}[args.case]
        q, k, v = (t.to(dev) for t in wl.prefill_inputs(p))

        def call():
            api.prefill(q, k, v, q_offset=p.q_offset, causal=True)

        work = prefill_flops(p.B, p.H_q, p.d, p.T_q, p.S_kv, p.q_offset, True) / 1e12
        unit = "TFLOP/s"
    else:
        raise SystemExit(f"unknown case {args.case}")
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    api.check()
    times = []
    for _ in range(args.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / 1e3)
    api.check()
    med = statistics.median(times)
    res = {"case": args.case, "median_us": med * 1e6, "value": work / med, "unit": unit,
           "steps": args.steps, "note": "plain launches, warm L2 possible; not a bench value"}
    if graph_call is not None:
        gt = []
        for _ in range(max(3, args.steps)):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            graph_call()
            e1.record()
            torch.cuda.synchronize()
            gt.append(e0.elapsed_time(e1) / 1e3 / graph_calls)
        api.check()
        gmed = statistics.median(gt)
        res["graph"] = {"us_per_call": gmed * 1e6, "value": work / gmed, "calls_per_graph":
                        graph_calls, "note": "back-to-back calls in a CUDA graph over distinct "
                        "caches larger than L2 together"}
        if extra:
            res["graph"]["bf16_equivalent_GBps"] = extra["bf16_equivalent_bytes_per_call"] / gmed / 1e9
            res.update(extra)
    print(json.dumps(res))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU work for the cpu_baseline leg")
    ap.add_argument("--ref-seconds", type=float, default=4.0,
                    help="CPU work per step of --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", default=None,
                    help="one workload alone: decode8k | ragged128k | ring8k | decode128k | "
                         "decode8k_q8 | ragged128k_q8 | decode8k_q4 | ragged128k_q4 | prefill8k "
                         "| chunked32k | prefill8k_mha")
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--cpu-worker", type=float, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-worker-steps", type=int, default=1, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-worker-offset", type=int, default=0, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_worker is not None:
        cpu_worker(args.cpu_worker, args.cpu_worker_steps, args.cpu_worker_offset)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.case:
        run_case(args)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            # the oracle on every host core (one single-threaded process each),
            # and on one thread
            procs = host_cores()
            cb = cpu_oracle_sample(args.cpu_seconds, procs=procs)[0]
            c1 = cpu_oracle_sample(args.cpu_seconds)[0]
            res["cpu_baseline"] = {
                "value": cb["decode_gbs"], "unit": "GB/s", "cores": procs,
                "host_cores": os.cpu_count(), "kind": "oracle",
                "sample": f"{cb['decode_rows']} query-head rows of the 8K decode in "
                          f"{cb['decode_s']:.1f}s on {procs} single-threaded processes (fp64 "
                          f"oracle, own rows each); prefill: {cb['prefill_rows']} rows",
                "prefill_TFLOPS": cb["prefill_tflops"],
                "single_thread": {"value": c1["decode_gbs"], "unit": "GB/s",
                                  "prefill_TFLOPS": c1["prefill_tflops"],
                                  "sample": f"{c1['decode_rows']} decode rows in "
                                            f"{c1['decode_s']:.1f}s, {c1['prefill_rows']} "
                                            "prefill rows, 1 thread"}}
        else:
            res["cpu_baseline"] = None
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()

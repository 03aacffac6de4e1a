#!/usr/bin/env python
"""Benchmark: MLA decode µs/call and KV-read GB/s against the GB300 HBM roofline.

One step = one full decode call over the batch of the
headline workload: fp8 e4m3 KV cache (per-tensor scale), batch 256 x 1 query
token, kv_len 8192 per sequence, bf16 queries -- 1.21 GB of KV streamed per
call, larger than the 129 MB L2, so consecutive calls read HBM.

Prints ONE JSON line (rank 0). value = KV-read GB/s over all ranks
(algorithmic KV bytes / time); us_per_call alongside. Under torchrun each rank
runs its own copy of the workload (weak scaling, no collective on the data
path; a barrier and a max over ranks bracket the timing).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the fp64 CPU oracle (the reference semantics) on the
same workload and metric, one bounded sample per step, on the host cores.
"""
from __future__ import annotations

import argparse
import dataclasses
import datetime
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "fp8kv_bs256_kv8192"
METRIC = "MLA decode µs/call and KV-read GB/s vs GB300 HBM peak, per (batch, kv_len, dtype)"
STAGE1_SOURCES = ["mla_stage1_tc.cu", "mla_tc_common.cuh", "mla_tcgen05.cuh", "mla_device.cuh", "mla_partition.cuh",
                  "mla_internal.h"]


def _code_only(src: str) -> str:
    """The source with its comments and blank space removed (the sources hold no string
    literal with a comment marker in it), so that editing a comment does not invalidate a
    capture taken on the same code."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def _stage1_source_sha() -> str:
    h = hashlib.sha256()
    for f in STAGE1_SOURCES:
        with open(os.path.join(ROOT, "mla_decode_attention_split_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def _measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _ncu_traffic(workload: str):
    """DRAM bytes per stage-1 launch from the committed ncu summary, if it was
    taken on the current stage-1 source; else None. A capture of a smaller case
    is scaled to the workload by KV rows (traffic grows with the rows)."""
    path = os.path.join(ROOT, "profiles", "stage1_dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("source_sha") == _stage1_source_sha():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 100 ms in the background."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self, t0: float, t1: float):
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(inside)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _barrier_max(value: float, world: int, device):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate_gbs(kv_bytes_per_step: int, steps: int, world: int, ms_total: float) -> float:
    """Whole-job KV-read GB/s: every rank streams kv_bytes_per_step per step
    (weak scaling), over the slowest rank's time for all steps."""
    return kv_bytes_per_step * steps * world / (ms_total * 1e-3) / 1e9


def kv_bytes(inp) -> int:
    return inp.kv_bytes()


def workload_by_name(synth, name):
    if name in synth.WORKLOADS:
        return synth.WORKLOADS[name]
    # profiling shapes: kvfp8_bs64_kv8192, kvbf16_bs8_kv4096, kvmx_bs64_kv8192 (bf16 q, one token per
    # segment); kvfp8a8_...: fp8 q; an optional q<N> field sets the tokens per segment (kvfp8_bs64_q2_kv8192)
    parts = name.split("_")
    fmt, bs, kvl = parts[0], parts[1], parts[-1]
    q_len = int(parts[2][1:]) if len(parts) == 4 else 1
    kv_dtype = {"kvfp8": synth.FP8_E4M3, "kvfp8a8": synth.FP8_E4M3, "kvbf16": synth.BF16, "kvmx": synth.MXFP4}[fmt]
    q_dtype = synth.FP8_E4M3 if fmt == "kvfp8a8" else synth.BF16
    return synth.Workload(name, int(bs[2:]), q_len, int(kvl[2:]), q_dtype, kv_dtype)


L2_FLUSHED = "flushed (256 MB write) before each call"


def l2_flush(buf, i):
    """Evicts the timed call's inputs from L2: writes a 256 MB buffer (twice the L2)."""
    buf.fill_(i & 0xFF)


BACK_TO_BACK = "back to back: the calls issued without a host synchronisation, timed as a sequence"


def time_calls(m, torch, call, steps, warmup, flush_l2: bool) -> float:
    """Device µs per call. Cold: L2 flushed before each call, CUDA events around the call (the
    GPU is busy with the flush while the host prepares the launch), median over steps. Warm:
    `steps` calls back to back with no host synchronisation in between (consecutive launches
    overlap through programmatic dependent launch), events at the two ends of the sequence."""
    if flush_l2:
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        tot = []
        for i in range(warmup + steps):
            l2_flush(flush, i)
            call(ev)
            torch.cuda.synchronize()
            if i >= warmup:
                tot.append(m.elapsed_ms(ev[0], ev[2]) * 1e3)
        del flush
        return statistics.median(tot)
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        call()
    t1.record()
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) * 1e3 / steps


def time_workload(m, synth, torch, name, steps, warmup, flush_l2: bool, quantize_q: bool = False, w=None,
                  token_group: int = 0):
    """Per-call device time of one workload (stage-1 and total), median over steps.
    quantize_q: pass bf16 q and let the call quantise it (the pages' a8w8 flow).
    w: a Workload instead of a named one; token_group: a segment's tokens share KV tiles in groups of 2 or 4."""
    w = synth.WORKLOADS[name] if w is None else w
    if quantize_q:
        w = synth.Workload(w.name, w.batch, w.q_len, w.kv_len, synth.BF16, w.kv_dtype, w.ragged_max, w.seed)
    inp = synth.make_inputs(w, "cuda")
    out = torch.empty((inp.total_q, 16, 512), dtype=torch.bfloat16, device="cuda")
    ws = m.alloc_group_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, token_group)

    def call(events=None):
        m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, out, inp.kv_dtype, workspace=ws,
                 q_dtype=inp.q_dtype, q_scale=inp.q_scale, events=events, quantize_q=quantize_q,
                 token_group=token_group)

    us = time_calls(m, torch, call, steps, warmup, flush_l2)
    st, flags = m.device_error(ws)
    assert st == m.MLA_OK, (name, flags)
    return {"us_per_call": round(us, 2), "kv_gbs": round(kv_bytes(inp) / (us * 1e-6) / 1e9, 1),
            "kv_bytes": kv_bytes(inp), "l2": L2_FLUSHED if flush_l2 else BACK_TO_BACK}


def time_paged_workload(m, synth, torch, name, page_size, steps, warmup, flush_l2: bool, in_order: bool = False):
    """Per-call device time of a workload with its fp8 cache in pages of `page_size` rows,
    scattered over the pool in random order, or in pool order (the pages' identity table)
    when in_order. The page table is built once, outside the timing."""
    w = synth.WORKLOADS[name]
    pin = synth.make_paged_inputs(w, "cuda", kv_lens=synth.make_lengths(w), page_size=page_size)
    if in_order:
        pin = dataclasses.replace(pin, page_indices=torch.sort(pin.page_indices).values.contiguous())
    out = torch.empty((pin.total_q, 16, 512), dtype=torch.bfloat16, device="cuda")
    ws = m.alloc_paged_workspace(pin.batch, pin.total_q, pin.total_kv, synth.FP8_E4M3)

    def call(events=None):
        m.decode_paged(pin.q, pin.kv_pages, pin.kv_scale, pin.qo_indptr, pin.page_indptr, pin.page_indices,
                       pin.last_page_len, page_size, out, synth.FP8_E4M3, total_kv=pin.total_kv, workspace=ws,
                       q_dtype=pin.q_dtype, q_scale=pin.q_scale, events=events)

    us = time_calls(m, torch, call, steps, warmup, flush_l2)
    st, flags = m.device_error(ws)
    assert st == m.MLA_OK, (name, page_size, flags)
    kvb = pin.total_kv * synth.D_QK  # the rows read (the pool's spare pages are not)
    return {"us_per_call": round(us, 2), "kv_gbs": round(kvb / (us * 1e-6) / 1e9, 1), "kv_bytes": kvb,
            "page_size": page_size, "pages": pin.num_pages, "page_order": "pool order" if in_order else "random",
            "l2": L2_FLUSHED if flush_l2 else BACK_TO_BACK}


def _first_rows(h, rows):
    """A one-segment host input cut to its first `rows` KV rows (rows <= 0: all)."""
    if rows <= 0 or rows >= h["kv"].shape[0]:
        return h
    g = dict(h)
    g["kv"] = h["kv"][:rows].copy()
    if h["kv_dtype"] == 2:  # mxfp4 scales go with their rows
        g["kv_scale"] = h["kv_scale"][:rows].copy()
    g["kv_indptr"] = h["kv_indptr"].copy()
    g["kv_indptr"][-1] = rows
    return g


def _oracle_segment(h, sm_scale):
    """One segment through the oracle (a worker of the host-core pool). Returns its KV rows."""
    import oracle
    oracle.mla_decode(h["q"], h["q_dtype"], h["q_scale"], h["kv"], h["kv_dtype"], h["kv_scale"], h["qo_indptr"],
                      h["kv_indptr"], heads=16, dqk=576, dv=512, sm_scale=sm_scale)
    return int(h["kv"].shape[0])


def _host_pool():
    """A process pool over the host cores (spawned: a forked CUDA process can hang)."""
    import multiprocessing as mp
    n = max(1, os.cpu_count() or 1)
    return mp.get_context("spawn").Pool(n), n


def cpu_baseline(inp, synth, oracle, target_s=15.0):
    """The oracle as it stands (fp64 C, one segment per worker) on all host cores, over a bounded
    sample of the workload's segments (all 16 heads each); throughput in KV-read GB/s."""
    rowb = inp.kv_bytes() / max(1, inp.total_kv)
    pool, n = _host_pool()
    try:
        sm = synth.sm_scale_default()
        pool.starmap(_oracle_segment, [(_first_rows(synth.to_host_codes(inp, [0]), 64), sm)] * n)  # workers up
        done, nbytes, b = 0, 0, 0
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < target_s and b < inp.batch:
            segs = list(range(b, min(inp.batch, b + n)))
            rows = pool.starmap(_oracle_segment, [(synth.to_host_codes(inp, [s]), sm) for s in segs])
            nbytes += int(sum(rows) * rowb)
            done += len(segs)
            b += len(segs)
        wall = time.perf_counter() - t0
    finally:
        pool.close()
        pool.join()
    gbs = nbytes / wall / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": f"{done} of {inp.batch} segments x 16 heads (fp64 C, one segment per process on {n} host "
                      f"cores), {wall:.1f} s wall",
            "us_per_call_equiv": round(inp.kv_bytes() / (gbs * 1e9) * 1e6, 1)}


def run_reference(args):
    world, rank, local = _dist()
    if rank != 0:
        return 0
    import torch
    import oracle
    from mla_decode_attention_split_gb300 import synth
    oracle.build()
    w = synth.WORKLOADS[HEADLINE]
    # segments are i.i.d.: a sub-batch of the workload's own shape, cycled
    sub = min(w.batch, 16)
    inp = synth.make_inputs(synth.Workload(w.name, sub, w.q_len, w.kv_len, w.q_dtype, w.kv_dtype, seed=w.seed), "cpu")
    rowb = inp.kv_bytes() / inp.total_kv
    sm = synth.sm_scale_default()
    hosts = [synth.to_host_codes(inp, [b]) for b in range(inp.batch)]
    pool, ncores = _host_pool()
    try:
        # one step = one sample segment per host core; the sample length keeps the whole run
        # near two minutes whatever --steps is (calibrated on one full segment)
        pool.starmap(_oracle_segment, [(_first_rows(hosts[0], 64), sm)] * ncores)  # workers up, oracle loaded
        t0 = time.perf_counter()
        pool.starmap(_oracle_segment, [(hosts[j % inp.batch], sm) for j in range(ncores)])  # one full step
        per_row = (time.perf_counter() - t0) / w.kv_len
        rows = int(min(w.kv_len, max(64, 90.0 / max(1, args.steps + args.warmup) / per_row)))
        cut = [_first_rows(h, rows) for h in hosts]
        times, nbytes = [], 0
        for i in range(args.warmup + args.steps):
            jobs = [(cut[(i * ncores + j) % inp.batch], sm) for j in range(ncores)]
            t0 = time.perf_counter()
            done = pool.starmap(_oracle_segment, jobs)
            dt = time.perf_counter() - t0
            if i >= args.warmup:
                times.append(dt)
                nbytes += int(sum(done) * rowb)
    finally:
        pool.close()
        pool.join()
    total = sum(times)
    gbs = nbytes / total / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / len(times) * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": HEADLINE, "batch": w.batch, "q_len": 1, "kv_len": w.kv_len, "q_dtype": "bf16",
                       "kv_dtype": "fp8_e4m3",
                       "step": f"{ncores} segments (16 heads x the first {rows} of their {w.kv_len} KV rows), one "
                               f"per host core, per step, cycling over {sub} seeded segments"},
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": ncores, "kind": "oracle",
                             "sample": f"{len(times)} steps x {ncores} segments x {rows} KV rows x 16 heads, fp64 C, "
                                       f"one process per host core"},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="skip the per-workload table")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end measurement")
    ap.add_argument("--workload", default=HEADLINE,
                    help="workload name (the five benchmark workloads, or kv{fp8,fp8a8,bf16,mx}_bs<B>[_q<N>]_kv<L> "
                         "for profiling)")
    ap.add_argument("--token-pairs", action="store_true", help="same as --token-group 2")
    ap.add_argument("--token-group", type=int, default=0,
                    help="the tokens of a segment share each KV tile in groups of 2 (fp8 or bf16 KV) or 4 (fp8 KV "
                         "and fp8 q); for q_len > 1")
    args = ap.parse_args()
    if args.token_pairs and not args.token_group:
        args.token_group = 2
    if args.impl == "reference":
        return run_reference(args)

    world, rank, local = _dist()
    import torch
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    from mla_decode_attention_split_gb300 import build as _build
    _build.build()
    import mla_decode_attention_split_gb300 as m
    from mla_decode_attention_split_gb300 import synth

    w = workload_by_name(synth, args.workload)
    inp = synth.make_inputs(w, device)
    torch.cuda.empty_cache()
    kvb = kv_bytes(inp)
    out = torch.empty((inp.total_q, 16, 512), dtype=torch.bfloat16, device=device)
    splits = m.plan(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype)
    ws = m.alloc_group_workspace(inp.batch, inp.total_q, inp.total_kv, inp.kv_dtype, args.token_group,
                                 num_splits=splits)
    stream = torch.cuda.current_stream()
    K, W = args.steps, args.warmup
    # the per-launch profile events run in a second, shorter pass: an event
    # recorded between two decode launches keeps the second from starting
    # while the first ends (programmatic dependent launch), so the timed pass
    # has events at its two ends only
    KP = min(K, 200)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(KP)]

    def step(events=None):
        m.decode(inp.q, inp.kv, inp.kv_scale, inp.qo_indptr, inp.kv_indptr, out, inp.kv_dtype, workspace=ws,
                 q_dtype=inp.q_dtype, q_scale=inp.q_scale, num_splits=splits, events=events, stream=stream,
                 token_group=args.token_group)

    for _ in range(W):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    _barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(K):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    for i in range(KP):  # per-launch kernel time for the roofline
        step(ev[i])
    torch.cuda.synchronize()
    _barrier(world)
    sampler.stop()
    st, flags = m.device_error(ws)
    assert st == m.MLA_OK, (m.status_string(st), flags)
    ms_total = t0.elapsed_time(t1)
    ms_total = _barrier_max(ms_total, world, device)
    stage1_ms = [m.elapsed_ms(e[0], e[1]) for e in ev]
    stage2_ms = [m.elapsed_ms(e[1], e[2]) for e in ev]
    s1_avg_s = sum(stage1_ms) / KP * 1e-3
    ms_step = ms_total / K
    value = aggregate_gbs(kvb, K, world, ms_total)
    peak, peak_kind = _measured_peaks()
    achieved = kvb / s1_avg_s / 1e9
    clocks = sampler.summary(t_wall0, t_wall1)

    # end to end through the host-buffer entry point: every input H2D from
    # pinned memory and the output D2H inside the timed region, every step
    e2e = None if (args.no_e2e or args.token_group > 1) else measure_e2e(m, torch, inp, out, ws, splits, stream, K,
                                                                       world, device, kvb)
    line = build_line(args, w, inp, kvb, splits, world, K, W, value, ms_step, achieved, peak, peak_kind, s1_avg_s,
                      stage2_ms, clocks, e2e)
    finish(args, line, rank, world, w, m, synth, torch, inp)
    return 0


def measure_e2e(m, torch, inp, out, ws, splits, stream, K, world, device, kvb):
    pin = (lambda t: None if t is None else t.cpu().pin_memory())
    h = {"q": pin(inp.q), "kv": pin(inp.kv), "kv_scale": pin(inp.kv_scale), "q_scale": pin(inp.q_scale),
         "qo_indptr": pin(inp.qo_indptr), "kv_indptr": pin(inp.kv_indptr),
         "out": torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()}
    dev = {k: (None if v is None else torch.empty_like(v, device=device)) for k, v in h.items()}
    e2e_steps = max(3, min(K, 50))
    for _ in range(2):
        m.decode_from_host(h, dev, inp.kv_dtype, q_dtype=inp.q_dtype, workspace=ws, num_splits=splits, stream=stream)
    torch.cuda.synchronize()
    _barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(e2e_steps):
        m.decode_from_host(h, dev, inp.kv_dtype, q_dtype=inp.q_dtype, workspace=ws, num_splits=splits, stream=stream)
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = _barrier_max(a.elapsed_time(b), world, device)
    h2d = sum(v.numel() * v.element_size() for k, v in h.items() if v is not None and k != "out")
    d2h = h["out"].numel() * 2
    return {"value": round(kvb * e2e_steps * world / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
            "us_per_call": round(e2e_ms / e2e_steps * 1e3, 1),
            "path": "mla_decode_from_host: q, KV cache, scales and indptrs H2D from pinned host memory, out D2H"}


def _kernel_name(synth, w) -> str:
    k = {synth.FP8_E4M3: "stage1_tc_kernel (tcgen05, e4m3 codes)", synth.MXFP4: "stage1_mx_kernel (tcgen05, e5m2 rebase)",
         synth.BF16: "stage1_bf_kernel (tcgen05 kind::f16)"}[w.kv_dtype]
    return k + f" <{synth.DTYPE_NAMES[w.kv_dtype]} KV, {synth.DTYPE_NAMES[w.q_dtype]} q>"


def _dtype_desc(synth, w) -> str:
    q = ("bf16 q as a hi+lo e4m3 pair per element (exact for elements within about 2^-13 of the token's "
         "max |q|; smaller ones rounded to the e4m3 subnormal step)" if w.q_dtype == synth.BF16 else "e4m3 q codes")
    return {synth.FP8_E4M3: f"e4m3 x e4m3 -> f32 (fp8 KV codes; {q})",
            synth.MXFP4: f"e5m2 x e4m3 -> f32 (mxfp4 KV rebased to e5m2 per row; {q})",
            synth.BF16: "bf16 x bf16 -> f32"}[w.kv_dtype]


def _launches_per_call(synth, w) -> int:
    # stage 1 merges split tokens itself: one launch per call
    return 1


def build_line(args, w, inp, kvb, splits, world, K, W, value, ms_step, achieved, peak, peak_kind, s1_avg_s,
               stage2_ms, clocks, e2e):
    from mla_decode_attention_split_gb300 import synth
    line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": round(ms_step, 4), "us_per_call": round(ms_step * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": _dtype_desc(synth, w),
            "data": "synthetic (seeded N(0,1), quantised as the pages' harness does)",
            "config": {"workload": w.name, "batch": w.batch, "q_len": w.q_len, "kv_len": w.kv_len,
                       "q_dtype": synth.DTYPE_NAMES[w.q_dtype], "kv_dtype": synth.DTYPE_NAMES[w.kv_dtype],
                       "kv_bytes_per_call": kvb, "num_splits": splits,
                       "l2": (f"inputs larger than L2 ({kvb / 1e9:.2f} GB KV per call, L2 129 MB); no flush"
                              if kvb > 129e6 else "KV fits in L2: back-to-back calls, warm"),
                       "parallelism": f"{world} independent replicas (weak scaling)"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": _ncu_traffic(w.name),
                         "kernel": {2: ("token pairs in " if w.kv_dtype == synth.BF16
                                        else "stage1_duo_kernel (tcgen05, token pairs, softmax in two warp groups) "
                                        if w.q_dtype == synth.FP8_E4M3
                                        else "stage1_pair_kernel (tcgen05, token pairs) "),
                                    4: "stage1_quad_kernel (tcgen05, groups of four tokens) "}.get(args.token_group, "")
                                   + _kernel_name(synth, w),
                         "algorithmic_bytes": f"{kvb} per launch = {kvb // inp.total_kv} B x {inp.total_kv} KV rows",
                         "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                         "stage1_us": round(s1_avg_s * 1e6, 2),
                         "stage2_us": round(sum(stage2_ms) / len(stage2_ms) * 1e3, 2),
                         "launch_timing": f"CUDA events around each launch, {len(stage2_ms)} launches right after "
                                          "the timed region"},
            "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"], "reasons": clocks["reasons"],
                       "samples_in_timed_region": clocks["samples"]},
            "gpu_launches": _launches_per_call(synth, w) * K,
            "e2e": e2e}
    return line


def finish(args, line, rank, world, w, m, synth, torch, inp):
    if rank == 0 and world == 1:
        if not args.no_workloads:
            table = {}
            for name in synth.WORKLOADS:
                try:
                    table[name] = {"cold": time_workload(m, synth, torch, name, 30, 5, True),
                                   "warm": time_workload(m, synth, torch, name, 30, 5, False)}
                except m.MlaError as e:
                    table[name] = {"unsupported": str(e)}
            # the a8w8 workload with q quantised inside the call (one extra small launch)
            qq = "a8w8_bs64_kv1024+in_call_q_quantisation"
            table[qq] = {"cold": time_workload(m, synth, torch, "a8w8_bs64_kv1024", 30, 5, True, quantize_q=True),
                         "warm": time_workload(m, synth, torch, "a8w8_bs64_kv1024", 30, 5, False, quantize_q=True)}
            # several query tokens per segment (multi-token decode), one token per KV pass
            # and tokens sharing each pass in pairs or groups of four
            for kd, kn, bs, ql, qd, qn, groups in ((synth.FP8_E4M3, "fp8kv", 128, 2, synth.BF16, "bf16q", (0, 2)),
                                                   (synth.FP8_E4M3, "fp8kv", 128, 2, synth.FP8_E4M3, "fp8q", (0, 2)),
                                                   (synth.BF16, "bf16kv", 32, 2, synth.BF16, "bf16q", (0, 2)),
                                                   (synth.FP8_E4M3, "fp8kv", 64, 4, synth.FP8_E4M3, "fp8q",
                                                    (0, 2, 4))):
                wq = synth.Workload(f"{kn}_bs{bs}_q{ql}_kv8192_{qn}", bs, ql, 8192, qd, kd)
                for g in groups:
                    key = wq.name + {0: "", 2: "+token_pairs", 4: "+token_group4"}[g]
                    table[key] = {"cold": time_workload(m, synth, torch, None, 30, 5, True, w=wq, token_group=g),
                                  "warm": time_workload(m, synth, torch, None, 30, 5, False, w=wq, token_group=g)}
            # the headline shape with the cache in pages scattered over a pool
            for ps, in_order in ((1, True), (1, False), (16, False), (64, False)):
                key = f"fp8kv_bs256_kv8192+paged_ps{ps}_{'in_order' if in_order else 'random'}"
                table[key] = {"cold": time_paged_workload(m, synth, torch, "fp8kv_bs256_kv8192", ps, 30, 5, True,
                                                          in_order),
                              "warm": time_paged_workload(m, synth, torch, "fp8kv_bs256_kv8192", ps, 30, 5, False,
                                                          in_order)}
            line["workloads"] = table
        if not args.no_cpu_baseline:
            import oracle
            oracle.build()
            line["cpu_baseline"] = cpu_baseline(inp, synth, oracle)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())

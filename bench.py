"""Benchmark: batch decode attention over a paged KV cache on GB300.

Workload (default ``uniform``): batch 64, kv_len ~ U{512..4096}, page 16, 32 qo / 8 kv heads,
head_dim 128, bf16 q/K/V/o, NHD, one plan reused over 32 layers of independent KV pools.
One step = plan() + run() on each of the 32 layers (one decode launch per layer; a split
request's chunks are merged inside that launch).  Every layer reads its own 1.2 GB pool, so a
step streams ~19 GB: inputs are far larger than L2 and each layer starts cold.  Smaller
workloads flush L2 between calls.

Prints one JSON line.  ``value`` is algorithmic GB/s: per call, the K and V bytes of every
attended token plus q and o, summed over the step and divided by the step time.
``--impl reference`` times the fp64 CPU oracle on the host cores on a bounded sample of the
same workload instead.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention: µs/call and KV-read GB/s as % of GB300 HBM peak"
ELT = {"f16": 2, "bf16": 2, "e4m3": 1}
L2_BYTES = 129 * 1024 * 1024


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one decode-kernel launch, from
# the ncu captures summarised in profiles/, and the digest of the kernel sources they were
# taken on: once the sources differ, the figure no longer describes the kernel and the line
# reports null.
MEASURED_TRAFFIC = {
    "sources_sha256": "134407828756dd62eb8d6960a5b70d9cc75e14acec9c502223049aec2a3e52dd",
    # profiles/decode_paged_kernel_traffic.md (one launch each, 1-pass ncu metric set, bytes)
    "uniform": 618856704.0,
    "mix": 418319872.0,
    "long": 2150457344.0,
    "lognormal": 3525971712.0,
}


# The files that decide what the decode kernel reads and writes: its device code and the
# planner that cuts its work list (host API and no-allocation code are left out).
KERNEL_SOURCES = ("decode_kernels.cuh", "pkd_device.cuh", "pkd_internal.h", "decode_f16.cu",
                  "decode_bf16.cu", "decode_e4m3.cu", "planner.cpp")


def kernel_sources_digest() -> str:
    return sources_digest(KERNEL_SOURCES)


# The same for the tcgen05 MLA kernel on the `mla` workload (profiles/mla_tc_kernel_mla.md).
MLA_KERNEL_SOURCES = ("mla_tc_kernels.cuh", "pkd_device.cuh", "pkd_internal.h", "mla_tc.cu",
                      "planner.cpp")
MLA_MEASURED_TRAFFIC = {
    "sources_sha256": "b4d2850a9d1ffc9d305864ac64921a53489fecf2b8ea347eb719e21fcde01957",
    "mla_tc_kernel": 151589376.0,
}


def sources_digest(names) -> str:
    csrc = os.path.join(ROOT, "paged_kv_decode_23_gb300", "csrc")
    h = hashlib.sha256()
    for name in names:
        h.update(name.encode())
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def mla_measured_traffic(kernel: str):
    if MLA_MEASURED_TRAFFIC.get("sources_sha256") != sources_digest(MLA_KERNEL_SOURCES):
        return None
    return MLA_MEASURED_TRAFFIC.get(kernel)


def max_over_ranks(values, world: int, device=None):
    """Element-wise maximum of `values` over all ranks of the process group: the slowest
    replica's times set the job's time (every rank gets the result)."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def replica_value(bytes_per_rank_step: float, world: int, ms_step: float) -> float:
    """Whole-job GB/s of `world` replicas, each moving `bytes_per_rank_step` per step, timed by
    the slowest rank's ms per step."""
    return world * bytes_per_rank_step / (ms_step * 1e-3) / 1e9


def measured_traffic(name: str):
    if MEASURED_TRAFFIC.get("sources_sha256") != kernel_sources_digest():
        return None
    return MEASURED_TRAFFIC.get(name)


def algorithmic_bytes(w) -> int:
    """K and V of every attended token, plus q and o, for one call."""
    lens = np.asarray(w.kv_lens, dtype=np.int64)
    att = lens if w.window_left < 0 else np.minimum(lens, w.window_left + 1)
    kv = int(att.sum()) * w.num_kv_heads * w.head_dim * ELT[w.kv_dtype] * 2
    qo = w.batch * w.num_qo_heads * w.head_dim * (ELT[w.q_dtype] + ELT[w.o_dtype])
    return kv + qo


def describe(w) -> str:
    extra = []
    if w.logits_soft_cap:
        extra.append(f"soft cap {w.logits_soft_cap:g}")
    if w.window_left >= 0:
        extra.append(f"window_left {w.window_left}")
    if w.fixed_split_size:
        extra.append(f"fixed split {w.fixed_split_size} pages")
    lens = np.asarray(w.kv_lens)
    return (f"{w.name}: batch {w.batch}, kv_len {lens.min()}..{lens.max()} (sum {lens.sum()}), "
            f"page {w.page_size}, {w.num_qo_heads}/{w.num_kv_heads} heads, D {w.head_dim}, "
            f"q {w.q_dtype} kv {w.kv_dtype} o {w.o_dtype}, {w.layout}"
            + (", " + ", ".join(extra) if extra else "")
            + (f", {w.layers} layers of independent pools, one plan per step" if w.layers > 1 else ""))


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples nvidia-smi every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.idx)], stdout=open(self.path, "w"),
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------------------- oracle arm
def _host_sample(w, budget_s: float, seed: int = 0):
    """A bounded sample of the workload for the CPU oracle: the first requests (in a seeded
    order) whose total attended tokens fit the time budget at the oracle's measured speed."""
    import oracle
    import workloads as W

    rng = np.random.default_rng(seed)
    order = rng.permutation(w.batch)

    def build(reqs):
        lens = np.asarray(w.kv_lens)[reqs]
        sw = W.custom(lens, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size,
                      layout=w.layout, q_dtype=w.q_dtype, kv_dtype=w.kv_dtype,
                      seed=w.seed + 1, pool_factor=1.0, logits_soft_cap=w.logits_soft_cap,
                      window_left=w.window_left, kv_store_scale=w.kv_store_scale,
                      k_scale=w.k_scale, v_scale=w.v_scale, sm_scale=w.sm_scale,
                      o_dtype=w.o_dtype)
        return sw, W.make_q(sw), W.make_pool(sw)

    def run(sw, q, pool):
        code = {"f16": oracle.F16, "bf16": oracle.BF16, "e4m3": oracle.E4M3}
        t0 = time.perf_counter()
        oracle.batch_decode_pool(sw.indptr, sw.indices, sw.last_page_len, W.raw_bits(q),
                                 code[sw.q_dtype], W.raw_bits(pool), code[sw.kv_dtype], sw.layout,
                                 sm_scale=sw.sm_scale, logits_soft_cap=sw.logits_soft_cap,
                                 window_left=sw.window_left, k_scale=sw.k_scale,
                                 v_scale=sw.v_scale)
        return time.perf_counter() - t0

    # calibrate on one request, then size the sample to the budget
    cal = build(order[:1])
    t_cal = max(run(*cal), 1e-4)
    rate = algorithmic_bytes(cal[0]) / t_cal
    target = rate * budget_s
    acc, take = 0, []
    full = algorithmic_bytes(w) / max(1, w.batch)
    for i in order:
        take.append(int(i))
        acc += full
        if acc >= target:
            break
    sw, q, pool = build(np.asarray(take))
    return sw, q, pool, run


def cpu_baseline(w, budget_s: float):
    import oracle
    sw, q, pool, run = _host_sample(w, budget_s)
    t = run(sw, q, pool)
    # a sample shorter than the budget (a whole layer can take well under a second) is run
    # again until the budget is spent, so the figure rests on seconds of CPU work
    passes = 1
    while t < budget_s and passes < 1000:
        t += run(sw, q, pool)
        passes += 1
    b = algorithmic_bytes(sw) * passes
    return {"value": b / t / 1e9, "unit": "GB/s", "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"{sw.batch} of {w.batch} requests of one layer "
                      f"({int(np.sum(sw.kv_lens))} tokens) x {passes} passes, fp64 oracle, "
                      f"{t:.1f} s"}


def reference_arm(args, w):
    import oracle
    steps, warmup = args.steps, args.warmup
    per_step = max(1.0, min(20.0, 150.0 / max(1, steps + warmup)))
    sw, q, pool, run = _host_sample(w, per_step)
    for _ in range(warmup):
        run(sw, q, pool)
    times = [run(sw, q, pool) for _ in range(steps)]
    t = sum(times)
    b = algorithmic_bytes(sw) * steps
    val = b / t / 1e9
    out = {
        "metric": METRIC, "impl": "reference", "value": val, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": steps, "warmup": warmup, "ms_per_step": t / steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(w, args),
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": oracle.max_threads(),
                         "kind": "oracle",
                         "sample": f"{sw.batch} of {w.batch} requests of one layer per step "
                                   f"({int(np.sum(sw.kv_lens))} tokens)"},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out))


def config_of(w, args):
    extra = {} if getattr(args, "pos_encoding", "NONE") == "NONE" else \
        {"pos_encoding_mode": args.pos_encoding}
    return {"workload": describe(w), **extra, "batch": w.batch, "layers": w.layers,
            "kv_tokens": int(np.sum(w.kv_lens)),
            "l2": "inputs larger than L2 (each call streams its own pool)"
            if algorithmic_bytes(w) > 4 * L2_BYTES else
            "L2 flushed between calls (2x L2 written, then 2x L2 of other data read, so no dirty "
            "line is written back inside a timed call)",
            "parallelism": f"replicas x{args.gpus}" if args.gpus > 1 else "single GPU"}


# ----------------------------------------------------------------------------- GPU arm
def gpu_arm(args, w, rank, world):
    import torch

    import workloads as W
    from paged_kv_decode_23_gb300 import BatchDecodePagedKV

    local = int(os.environ.get("LOCAL_RANK", 0))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    layers = w.layers
    qs = [W.make_q(w, device=dev, layer=l) for l in range(layers)]
    pools = [W.make_pool(w, device=dev, layer=l) for l in range(layers)]
    outs = [torch.empty_like(qs[0], dtype=W.TORCH_DTYPES[w.o_dtype]) for _ in range(layers)]
    lses = [torch.empty(w.batch, w.num_qo_heads, dtype=torch.float32, device=dev)
            for _ in range(layers)]
    indices = torch.from_numpy(w.indices).to(dev)
    indptr_t = torch.from_numpy(w.indptr)
    lpl_t = torch.from_numpy(w.last_page_len)
    ws = torch.zeros(256 << 20, dtype=torch.uint8, device=dev)
    dec = BatchDecodePagedKV(ws, w.layout, int_workspace_buffer=torch.zeros(
        16 << 20, dtype=torch.uint8, device=dev))
    plan_kw = dict(q_data_type=W.TORCH_DTYPES[w.q_dtype], kv_data_type=W.TORCH_DTYPES[w.kv_dtype],
                   o_data_type=W.TORCH_DTYPES[w.o_dtype], sm_scale=w.sm_scale,
                   logits_soft_cap=w.logits_soft_cap or None, window_left=w.window_left,
                   fixed_split_size=w.fixed_split_size or None,
                   disable_split_kv=w.disable_split_kv)
    if args.pos_encoding != "NONE":
        plan_kw["pos_encoding_mode"] = args.pos_encoding
    if args.kernel != "auto":
        plan_kw["use_tensor_cores"] = args.kernel == "tc"
    flush = None
    if algorithmic_bytes(w) <= 4 * L2_BYTES:
        # Writing a buffer larger than L2 evicts the inputs but leaves L2 full of dirty lines,
        # whose write-back would then land inside the next timed call; reading a second such
        # buffer afterwards replaces them with clean lines.
        flush_w = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        flush_r = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        flush_sum = torch.empty((), dtype=torch.float32, device=dev)

        def flush(v):
            flush_w.fill_(v)
            torch.sum(flush_r, dim=0, out=flush_sum)

    # Every timed step records events around its plan() upload and around its runs, so the
    # decode kernel's time is read off the same steps the step time comes from: with several
    # layers the runs segment holds the layers' launches back to back (programmatic dependent
    # launch on, as in use); with an L2 flush between calls each call is a segment of its own
    # and the flushes stay outside every segment.  Per-launch events in a second, untimed pass
    # (PDL off, so each pair brackets exactly one kernel) give the isolated launch beside it.
    def new_events(n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for a, b in evs:  # torch creates the CUDA event on first record; the C ABI records it again
            a.record(stream)
            b.record(stream)
        return evs

    plan_ev = new_events(args.steps)
    run_ev = new_events(args.steps * (layers if flush is not None else 1))
    iso_ev = new_events(args.steps * layers)
    iso_pass = [False]

    def step(k=None):
        timed = k is not None and not iso_pass[0]
        if timed:
            plan_ev[k][0].record(stream)
        dec.plan(indptr_t, indices, lpl_t, w.num_qo_heads, w.num_kv_heads, w.head_dim,
                 w.page_size, **plan_kw)
        if timed:
            plan_ev[k][1].record(stream)
            if flush is None:
                run_ev[k][0].record(stream)
        for l in range(layers):
            if flush is not None:
                flush(float(l))
                if timed:
                    run_ev[k * layers + l][0].record(stream)
            e = iso_ev[k * layers + l] if (k is not None and iso_pass[0]) else None
            dec.run(qs[l], pools[l], k_scale=w.k_scale, v_scale=w.v_scale, out=outs[l],
                    lse=lses[l], timing_events=e, enable_pdl=not iso_pass[0])
            if timed and flush is not None:
                run_ev[k * layers + l][1].record(stream)
        if timed and flush is None:
            run_ev[k][1].record(stream)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert dec.check_status() == 0, "device status word reports a failure"

    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("timed")  # lets a profiler restrict itself to the timed steps
    t_start.record(stream)
    for k in range(args.steps):
        step(k)
    t_end.record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    barrier()
    clk = clocks.stop()
    plan_ms = sum(a.elapsed_time(b) for a, b in plan_ev)
    run_ms = sum(a.elapsed_time(b) for a, b in run_ev)
    # with flushes the step is its timed segments; without, the whole timed loop
    ms_total = plan_ms + run_ms if flush is not None else t_start.elapsed_time(t_end)
    seg_detail = {"plan_us_per_step": plan_ms * 1e3 / args.steps,
                  "run_us_per_call": run_ms * 1e3 / (args.steps * layers)}
    # second pass, untimed for the step: each launch alone between its own events
    iso_pass[0] = True
    for k in range(args.steps):
        step(k)
    torch.cuda.synchronize()
    iso_pass[0] = False
    # the planner's own host cost: plan() calls with the GPU idle (inside the timed loop the
    # host runs ahead of the GPU and plan() would also measure the queue's back-pressure)
    torch.cuda.synchronize()
    t_h = time.perf_counter()
    for _ in range(20):
        dec.plan(indptr_t, indices, lpl_t, w.num_qo_heads, w.num_kv_heads, w.head_dim,
                 w.page_size, **plan_kw)
    host_plan_us = (time.perf_counter() - t_h) * 1e6 / 20
    torch.cuda.synchronize()
    iso_ms = statistics.mean(a.elapsed_time(b) for a, b in iso_ev)
    assert dec.check_status() == 0, "device status word reports a failure"

    # End to end through the public API with host buffers: every step copies all layers' q and
    # the page ids in from pinned host memory (one copy each) and all layers' o and lse out.
    q_all_host = torch.stack([q.cpu() for q in qs]).pin_memory()
    q_all_dev = torch.empty_like(q_all_host, device=dev)
    o_all_dev = torch.empty((layers,) + tuple(outs[0].shape), dtype=outs[0].dtype, device=dev)
    l_all_dev = torch.empty((layers,) + tuple(lses[0].shape), dtype=torch.float32, device=dev)
    o_all_host = torch.empty(o_all_dev.shape, dtype=o_all_dev.dtype).pin_memory()
    l_all_host = torch.empty(l_all_dev.shape, dtype=torch.float32).pin_memory()
    idx_host = torch.from_numpy(w.indices).pin_memory()
    idx_dev = torch.empty_like(indices)

    # With one layer the L2 flush runs before each step's clock starts (every step still starts
    # cold); with several it stays between the layers, inside the step.
    flush_before = flush is not None and layers == 1

    def e2e_step():
        idx_dev.copy_(idx_host, non_blocking=True)
        q_all_dev.copy_(q_all_host, non_blocking=True)
        dec.plan(indptr_t, idx_dev, lpl_t, w.num_qo_heads, w.num_kv_heads, w.head_dim,
                 w.page_size, **plan_kw)
        for l in range(layers):
            if flush is not None and not flush_before:
                flush(float(l))
            dec.run(q_all_dev[l], pools[l], k_scale=w.k_scale, v_scale=w.v_scale,
                    out=o_all_dev[l], lse=l_all_dev[l])
        o_all_host.copy_(o_all_dev, non_blocking=True)
        l_all_host.copy_(l_all_dev, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for _ in range(args.warmup):
        e2e_step()
    barrier()
    e2e_s = 0.0
    for k in range(args.steps):
        if flush_before:
            flush(float(k))
            torch.cuda.current_stream().synchronize()
        t0 = time.perf_counter()
        e2e_step()
        e2e_s += time.perf_counter() - t0
    barrier()
    h2d = q_all_host.numel() * q_all_host.element_size() + idx_host.numel() * 4
    d2h = o_all_host.numel() * o_all_host.element_size() + l_all_host.numel() * 4

    ms_total, e2e_s = max_over_ranks([ms_total, e2e_s], world, device=dev)

    bytes_call = algorithmic_bytes(w)
    bytes_step = bytes_call * layers
    ms_step = ms_total / args.steps
    value = replica_value(bytes_step, world, ms_step)
    peak, peak_kind = load_peaks()
    # the decode kernel's time per call inside the timed steps (cannot exceed the step's share)
    kern_avg_ms = run_ms / (args.steps * layers)
    achieved = bytes_call / (kern_avg_ms * 1e-3) / 1e9
    res = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": w.kv_dtype if w.kv_dtype == w.q_dtype else f"{w.q_dtype}/{w.kv_dtype}",
        "data": "synthetic", "config": config_of(w, args),
        "us_per_call": ms_step * 1e3 / layers,
        "pct_of_hbm_peak": 100.0 * (value / world) / peak,
        "peak_kind": peak_kind,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": args.traffic if args.traffic is not None else
                     measured_traffic(w.name)
                     if (args.kernel, args.pos_encoding, args.qo_heads, args.kv_dtype,
                         args.head_dim, args.fixed_split_size)
                     == ("auto", "NONE", None, None, None, None)
                     else None,
                     "kernel": "decode_paged_kernel", "kernel_us": kern_avg_ms * 1e3,
                     "kernel_us_source": "CUDA events around the runs of the timed steps "
                                         "(plan upload and L2 flushes outside), per call",
                     "kernel_us_isolated": iso_ms * 1e3,
                     "algorithmic_bytes_per_launch": bytes_call},
        "e2e": {"value": replica_value(bytes_step, world, e2e_s / args.steps * 1e3), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_s / args.steps * 1e3,
                "l2": ("flushed before each step, outside its clock" if flush_before else
                       "flushed between layers, inside the step" if flush is not None else
                       "every layer reads its own pool, far larger than L2")},
        "gpu_launches": args.steps * layers,
        "clocks": clk,
        "host_plan_us": host_plan_us,
    }
    res["segments"] = seg_detail
    res["launch"] = dec.plan_info()
    return res


# ----------------------------------------------------------------------------- MLA
def mla_bytes_flops(w):
    """Algorithmic bytes (latent rows of every attended token, plus q and o) and flops
    (QK over 576 dims and PV over 512, per head and token) of one MLA decode call."""
    toks = int(np.sum(w.kv_lens))
    kv = toks * (w.head_dim_ckv + w.head_dim_kpe) * 2
    qo = w.batch * w.num_heads * (w.head_dim_ckv * 2 + w.head_dim_kpe) * 2
    flops = toks * w.num_heads * (w.head_dim_ckv + w.head_dim_kpe + w.head_dim_ckv) * 2
    return kv + qo, flops


def mla_describe(w) -> str:
    return (f"mla: batch {w.batch}, kv_len {int(w.kv_lens.min())}..{int(w.kv_lens.max())} "
            f"(sum {int(np.sum(w.kv_lens))}), page {w.page_size}, {w.num_heads} heads, ckv 512 + "
            f"kpe 64, {w.dtype}, sm_scale 1/sqrt(192) (the MLA wrapper's example)")


def _mla_sample(w, budget_s: float):
    """A bounded sample of the MLA workload for the CPU oracle (its first requests)."""
    import oracle
    import workloads as W
    code = {"bf16": oracle.BF16, "f16": oracle.F16}[w.dtype]

    def build(n):
        sub = W.mla_custom(w.kv_lens[:n], w.num_heads, w.page_size, w.dtype, seed=w.seed + 1,
                           pool_factor=1.0)
        return sub, W.make_mla_q(sub), W.make_mla_cache(sub)

    def run(sub, q, c):
        t0 = time.perf_counter()
        oracle.mla_decode(sub.kv_indptr, sub.kv_indices, sub.kv_lens, W.raw_bits(q[0]),
                          W.raw_bits(q[1]), code, W.raw_bits(c[0]), W.raw_bits(c[1]), code,
                          sub.page_size, sub.sm_scale)
        return time.perf_counter() - t0

    cal = build(1)
    t1 = max(run(*cal), 1e-4)
    n = int(max(1, min(w.batch, budget_s / t1)))
    return build(n), run


def mla_cpu_baseline(w, budget_s: float):
    import oracle
    (sub, q, c), run = _mla_sample(w, budget_s)
    t = run(sub, q, c)
    passes = 1  # as in cpu_baseline: repeat a sample shorter than the budget
    while t < budget_s and passes < 1000:
        t += run(sub, q, c)
        passes += 1
    b, _ = mla_bytes_flops(sub)
    b *= passes
    return {"value": b / t / 1e9, "unit": "GB/s", "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"{sub.batch} of {w.batch} requests ({int(np.sum(sub.kv_lens))} tokens) "
                      f"x {passes} passes, fp64 MLA oracle, {t:.1f} s"}


def mla_reference_arm(args, w):
    import oracle
    steps, warmup = args.steps, args.warmup
    per_step = max(1.0, min(20.0, 150.0 / max(1, steps + warmup)))
    (sub, q, c), run = _mla_sample(w, per_step)
    for _ in range(warmup):
        run(sub, q, c)
    t = sum(run(sub, q, c) for _ in range(steps))
    b, _ = mla_bytes_flops(sub)
    value = b * steps / t / 1e9
    sample = (f"{sub.batch} of {w.batch} requests ({int(np.sum(sub.kv_lens))} tokens) per step, "
              f"fp64 MLA oracle")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
        "steps": steps, "warmup": warmup, "ms_per_step": t / steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": mla_describe(w), "batch": w.batch},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}))


def mla_kernel_name(args, w) -> str:
    tc = args.mla_backend == "tcgen05" or (args.mla_backend == "auto" and w.num_heads > 32)
    return "mla_tc_kernel" if tc else "mla_decode_kernel"


def mla_roofline(flops, nbytes, kern_ms, tf_peak, tf_kind, hbm_peak, traffic, kernel):
    """The roofline that binds one MLA launch: HBM when its arithmetic intensity (algorithmic
    flops per algorithmic byte) lies below the ridge point of the two measured peaks, else the
    tensor cores; the other roof is reported beside it."""
    tflops = flops / (kern_ms * 1e-3) / 1e12
    gbs = nbytes / (kern_ms * 1e-3) / 1e9
    intensity = flops / nbytes
    ridge = tf_peak * 1e12 / (hbm_peak * 1e9)
    hbm = {"achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
           "algorithmic_bytes_per_launch": nbytes}
    tensor = {"achieved": tflops, "peak": tf_peak, "unit": "TFLOP/s", "frac": tflops / tf_peak,
              "algorithmic_flops_per_launch": flops, "peak_kind": tf_kind}
    main, other, bound = (hbm, tensor, "hbm") if intensity < ridge else (tensor, hbm, "tensor")
    out = {"bound": bound, **main, "traffic": traffic, "kernel": kernel,
           "kernel_us": kern_ms * 1e3, "intensity_flop_per_byte": intensity,
           "ridge_flop_per_byte": ridge}
    out["tensor" if bound == "hbm" else "hbm"] = other
    return out


def mla_gpu_arm(args, w, rank, world):
    import torch

    import workloads as W
    from paged_kv_decode_23_gb300 import BatchMLAPagedAttention

    local = int(os.environ.get("LOCAL_RANK", 0))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    qn, qp = W.make_mla_q(w, device=dev)
    ckv, kpe = W.make_mla_cache(w, device=dev)
    out = torch.empty_like(qn)
    lse = torch.empty(w.batch, w.num_heads, dtype=torch.float32, device=dev)
    idx = torch.from_numpy(w.kv_indices).to(dev)
    qo_ip = torch.arange(w.batch + 1, dtype=torch.int32)
    kv_ip, kv_len = torch.from_numpy(w.kv_indptr), torch.from_numpy(w.kv_lens)
    mla = BatchMLAPagedAttention(torch.zeros(256 << 20, dtype=torch.uint8, device=dev),
                                 backend=args.mla_backend)
    dt = W.TORCH_DTYPES[w.dtype]
    flush_w = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    flush_r = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sum = torch.empty((), dtype=torch.float32, device=dev)

    def flush(v):
        flush_w.fill_(v)
        torch.sum(flush_r, dim=0, out=flush_sum)

    def plan(indices):
        mla.plan(qo_ip, kv_ip, indices, kv_len, w.num_heads, 512, 64, w.page_size, False,
                 w.sm_scale, dt, dt)

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    seg = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(2 * args.steps)]
    for a, b in ev + seg:
        a.record(stream)
        b.record(stream)

    def step(k=None, kernel_pass=False):
        if k is not None and not kernel_pass:
            seg[2 * k][0].record(stream)
        plan(idx)
        if k is not None and not kernel_pass:
            seg[2 * k][1].record(stream)
        flush(float(k or 0))
        if k is not None and not kernel_pass:
            seg[2 * k + 1][0].record(stream)
        mla.run(qn, qp, ckv, kpe, out=out, lse=lse,
                timing_events=ev[k] if (k is not None and kernel_pass) else None,
                enable_pdl=not kernel_pass)
        if k is not None and not kernel_pass:
            seg[2 * k + 1][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert mla.check_status() == 0, "device status word reports a failure"
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("timed")
    for k in range(args.steps):
        step(k)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    ms_total = sum(a.elapsed_time(b) for a, b in seg)
    plan_ms = sum(seg[2 * k][0].elapsed_time(seg[2 * k][1]) for k in range(args.steps))
    for k in range(args.steps):
        step(k, kernel_pass=True)
    torch.cuda.synchronize()
    assert mla.check_status() == 0, "device status word reports a failure"
    kern_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)

    # end to end with host buffers: q and the page ids in, o and lse out, every step
    qn_h, qp_h = qn.cpu().pin_memory(), qp.cpu().pin_memory()
    idx_h = torch.from_numpy(w.kv_indices).pin_memory()
    qn_d, qp_d, idx_d = torch.empty_like(qn), torch.empty_like(qp), torch.empty_like(idx)
    o_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    l_h = torch.empty(lse.shape, dtype=torch.float32).pin_memory()

    def e2e_step():
        idx_d.copy_(idx_h, non_blocking=True)
        qn_d.copy_(qn_h, non_blocking=True)
        qp_d.copy_(qp_h, non_blocking=True)
        plan(idx_d)
        mla.run(qn_d, qp_d, ckv, kpe, out=out, lse=lse)
        o_h.copy_(out, non_blocking=True)
        l_h.copy_(lse, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    # the L2 flush runs before each step's clock starts: every step starts cold
    for _ in range(args.warmup):
        flush(1.0)
        e2e_step()
    e2e_s = 0.0
    for k in range(args.steps):
        flush(float(k))
        torch.cuda.current_stream().synchronize()
        t0 = time.perf_counter()
        e2e_step()
        e2e_s += time.perf_counter() - t0
    ms_total, e2e_s = max_over_ranks([ms_total, e2e_s], world, device=dev)
    bytes_call, flops_call = mla_bytes_flops(w)
    ms_step = ms_total / args.steps
    hbm_peak, peak_kind = load_peaks()
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tf_peak, tf_kind = float(json.load(f)["bf16_tflops"]), "measured (burst)"
    except Exception:
        tf_peak, tf_kind = 1900.0, "fallback"
    h2d = (qn_h.numel() + qp_h.numel()) * qn_h.element_size() + idx_h.numel() * 4
    d2h = o_h.numel() * o_h.element_size() + l_h.numel() * 4
    return {
        "metric": METRIC, "value": replica_value(bytes_call, world, ms_step), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": mla_describe(w), "batch": w.batch, "layers": 1,
                   "mla_kernel": mla_kernel_name(args, w),
                   "kv_tokens": int(np.sum(w.kv_lens)),
                   "l2": "L2 flushed between calls (2x L2 written, then 2x L2 of other data "
                         "read, outside the timed segments)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "us_per_call": ms_step * 1e3,
        "pct_of_hbm_peak": 100.0 * (bytes_call / (ms_step * 1e-3) / 1e9) / hbm_peak,
        "peak_kind": peak_kind,
        "roofline": mla_roofline(flops_call, bytes_call, kern_ms, tf_peak, tf_kind, hbm_peak,
                                 mla_measured_traffic(mla_kernel_name(args, w))
                                 if w.name == "mla" else None, mla_kernel_name(args, w)),
        "e2e": {"value": replica_value(bytes_call, world, e2e_s / args.steps * 1e3), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_s / args.steps * 1e3,
                "l2": "flushed before each step, outside its clock"},
        "gpu_launches": args.steps,
        "clocks": clk,
        "segments": {"plan_us_per_step": plan_ms * 1e3 / args.steps,
                     "run_us_per_call": (ms_total - plan_ms) * 1e3 / args.steps},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="uniform",
                    choices=["worked", "uniform", "lognormal", "long", "mix", "mla"])
    ap.add_argument("--layers", type=int, default=None, help="override the layer count")
    ap.add_argument("--qo-heads", type=int, default=None,
                    help="override num_qo_heads (a GQA-group variant of the workload)")
    ap.add_argument("--kv-dtype", choices=["f16", "bf16", "e4m3"], default=None,
                    help="override the KV dtype (e4m3 stores values / 0.5, k_scale = v_scale = 0.5)")
    ap.add_argument("--head-dim", type=int, choices=[64, 128, 256], default=None,
                    help="override head_dim")
    ap.add_argument("--fixed-split-size", type=int, default=None,
                    help="override the plan's fixed_split_size (pages; 0 = the heuristic)")
    ap.add_argument("--kernel", choices=["auto", "tc", "cc"], default="auto")
    ap.add_argument("--pos-encoding", choices=["NONE", "ROPE_LLAMA", "ALIBI"], default="NONE",
                    help="plan's pos_encoding_mode (rope_theta 1e4, rope_scale 1)")
    ap.add_argument("--mla-backend", choices=["auto", "fa2", "tcgen05"], default="auto",
                    help="MLA kernel (--workload mla): auto picks tcgen05 for > 32 heads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per decode launch from an ncu capture of this kernel")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    import workloads as W
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.workload == "mla":
        w = W.mla_workload()
        if args.impl == "reference":
            if rank == 0:
                mla_reference_arm(args, w)
            return
        if world > 1:
            import torch
            torch.distributed.init_process_group("nccl")
        res = mla_gpu_arm(args, w, rank, world)
        if rank == 0:
            if not args.no_cpu_baseline:
                res["cpu_baseline"] = mla_cpu_baseline(w, args.cpu_budget)
            print(json.dumps(res))
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
        return
    w = W.workload(args.workload)
    if args.layers:
        w.layers = args.layers
    if args.qo_heads:
        if args.qo_heads % w.num_kv_heads:
            ap.error("--qo-heads must be a multiple of the workload's kv heads")
        w.num_qo_heads = args.qo_heads
    if args.head_dim:
        w.head_dim = args.head_dim
        w.sm_scale = None
    if args.fixed_split_size is not None:
        w.fixed_split_size = args.fixed_split_size
    if args.kv_dtype:
        w.kv_dtype = args.kv_dtype
        if args.kv_dtype == "e4m3":
            w.kv_store_scale, w.k_scale, w.v_scale = 0.5, 0.5, 0.5
    if args.impl == "reference":
        if rank == 0:
            reference_arm(args, w)
        return
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    res = gpu_arm(args, w, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(w, args.cpu_budget)
        print(json.dumps(res))
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

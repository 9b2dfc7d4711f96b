"""Benchmark: one data-parallel-attention rank's MLA decode step on one GB300.

A step is the whole hot path over one batch: for each of the workload's layers,
append this step's new latent row of every sequence into that layer's paged
cache, then decode every request over its full context (planned once per step,
since all layers share the sequence lengths and block table).  Default
workload: 20 sequences x 4096 tokens, 61 layers, 128 heads, page 64 (the
rank's share of a 159 x 4096 node batch; 5.76 GB of cache read per step).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 3] [--impl reference]

Prints one JSON line (rank 0).  `value` = cache bytes read per step / step
time (GB/s), the throughput form of the step latency also reported as
ms_per_step.  For N > 1 (torchrun) each rank runs an independent replica of
the rank workload on its own GPU (no collective on the data path; a barrier
and a max-reduction of the timings only).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import mla_inputs as mi  # noqa: E402

METRIC = "MLA decode step latency & cache GB/s at 1 GB300; % of roofline"
ROW_BYTES = mi.ROW * 2


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def reduce_max(x, world, device=None):
    """Max of a per-rank float over all ranks (the slowest rank sets the time)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput_gbs(world, bytes_per_rank_step, ms_per_step):
    """Whole-job GB/s: every rank processes its own replica of the workload."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- workload

def build_device_workload(w, device):
    import torch
    bt = mi.make_block_table(mi.rng_for(w.config_id, 0, 1), w.seq_lens, w.block_size,
                             w.num_blocks())
    layers = []
    for l in range(w.layers):
        d = mi.make_device_layer(w, l, device, block_table=bt)
        layers.append(d)
    shared = layers[0]
    B = w.batch
    outs = [torch.empty((B, 128, 512), dtype=torch.bfloat16, device=device) for _ in layers]
    lses = [torch.empty((B, 128), dtype=torch.float32, device=device) for _ in layers]
    return dict(layers=layers, bt=shared["block_table"], seq=shared["seq_lens"],
                slots=shared["slot_mapping"], outs=outs, lses=lses, bt_host=bt)


def algorithmic_bytes_per_layer(w):
    """(cache rows read, decode kernel's algorithmic bytes = cache + q, out written,
    appended rows written) per layer."""
    cache = sum(w.seq_lens) * ROW_BYTES
    q = w.batch * 128 * mi.ROW * 2
    out = w.batch * 128 * 512 * 2
    append = w.batch * ROW_BYTES if w.append else 0
    return cache, cache + q, out, append


KERNEL_SOURCES = ("mla_latent_cache_decode_gb300/csrc/decode_tc.cu",
                  "mla_latent_cache_decode_gb300/csrc/sm100.cuh",
                  "mla_latent_cache_decode_gb300/csrc/common.cuh",
                  "mla_latent_cache_decode_gb300/csrc/fp8.cuh")
KERNEL_HEADER = "include/mla.h"
# the header's constants that reach the decode kernel (its declarations,
# comments, ABI version and the no-allocation entry point's limits do not)
KERNEL_CONSTANTS = ("MLA_ROW_DIM", "MLA_KV_LORA_RANK", "MLA_ROPE_DIM", "MLA_NUM_HEADS")
TRAFFIC_PROFILE = "profiles/decode_tc_dp_rank_layer_b20x4096_dram.md"


def kernel_source_hash():
    """sha256 of the decode kernel's sources and of the header constants that
    reach it."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    with open(os.path.join(ROOT, KERNEL_HEADER)) as fh:
        consts = [ln.strip() for ln in fh
                  if ln.startswith("#define ") and ln.split()[1] in KERNEL_CONSTANTS]
    h.update("\n".join(consts).encode())
    return h.hexdigest()


def e2e_chunk_bounds(layers, growth=1.6):
    """Layer boundaries of the e2e step's copy chunks: the input chunks start
    at one layer and grow by `growth` (the decodes of layers [a, b) wait for
    the inputs of layers < b); the output chunks mirror them, shrinking
    towards the last layer.  Both lists run from 0 to `layers`."""
    b = [0]
    while b[-1] < layers:
        b.append(min(layers, max(b[-1] + 1, math.ceil(growth * b[-1]))))
    return b, [layers - x for x in reversed(b)]


def measured_traffic(w):
    """DRAM bytes per decode launch from the committed ncu capture, if it was taken
    on this workload's layer shape with the kernel as it is now; else None."""
    path = os.path.join(ROOT, TRAFFIC_PROFILE)
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.startswith("- "):
                k, v = line[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
    base = w.name.split("_first")[0]  # a --layers run has the same per-layer launch
    if fields.get("workload") != base or fields.get("kernel_source_sha256") != kernel_source_hash():
        return None
    try:
        return int(fields["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def algorithmic_flops_per_layer(w):
    return sum(w.seq_lens) * 2 * 128 * (mi.ROW + 512)


# ----------------------------------------------------------------------------- GPU arm

def run_mine(args, w, rank, world, local_rank):
    import torch
    import mla_latent_cache_decode_gb300 as mla

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    W = build_device_workload(w, device)
    ws = mla.make_workspace(w.batch, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    # all work on one non-default stream (capturable into a CUDA graph)
    stream = torch.cuda.Stream(device)
    torch.cuda.set_stream(stream)
    sh = stream.cuda_stream
    L = w.layers
    scale = mi.SOFTMAX_SCALE

    nvtx = torch.cuda.nvtx

    def step(timing_events=None):
        mla.mla_decode_plan(W["seq"], W["bt"], w.block_size, ws, dev_status=status, stream=sh,
                            num_blocks=w.num_blocks())
        for l in range(L):
            d = W["layers"][l]
            nvtx.range_push(f"layer {l}")
            # mla_decode_append_planned (the append of this step's row fused
            # into the decode kernel), as its two launches so that the decode
            # kernel can be timed on its own
            if timing_events is not None:
                timing_events[l][0].record(stream)
            mla.mla_decode_partial(d["q"], d["cache"], W["bt"], W["seq"], scale, W["outs"][l],
                                   W["lses"][l], workspace=ws, dev_status=status, stream=sh,
                                   kv_new=d["kv_new"] if w.append else None)
            if timing_events is not None:
                timing_events[l][1].record(stream)
            mla.mla_combine_planned(ws, w.batch, W["outs"][l], W["lses"][l], stream=sh)
            nvtx.range_pop()

    launches_per_step = 1 + L * 2

    # Between timed steps the L2 is flushed (a write of 2x its size, outside the
    # timed events) when one step's cache is small enough to stay partly
    # resident; a step reading many times L2 flushes it by itself.
    l2_bytes = torch.cuda.get_device_properties(device).L2_cache_size
    step_cache = algorithmic_bytes_per_layer(w)[0] * L
    flush_l2 = step_cache < 8 * l2_bytes
    flush_buf = (torch.empty(2 * l2_bytes, dtype=torch.uint8, device=device)
                 if flush_l2 else None)

    def flush():
        if flush_buf is not None:
            flush_buf.fill_(0x5A)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # ---- timed region: exactly K steps, device events on the launching stream
    clocks = ClockSampler(local_rank)
    if rank == 0:
        clocks.start()
    barrier()
    torch.cuda.synchronize()
    # each step between its own pair of events; with the flush, the flush
    # runs between a step's end event and the next step's start event
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for k in range(args.steps):
        flush()
        ev[k][0].record(stream)
        if graph is not None:
            graph.replay()
        else:
            step()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop() if rank == 0 else None
    per_step = [a.elapsed_time(b) for a, b in ev]
    ms_total = reduce_max(sum(per_step), world, device)
    ms_step = ms_total / args.steps
    per_step_sorted = sorted(per_step)

    def pct(p):
        return per_step_sorted[min(len(per_step_sorted) - 1, int(p * len(per_step_sorted)))]
    step_stats = {"median": round(statistics.median(per_step), 4), "p10": round(pct(0.10), 4),
                  "p90": round(pct(0.90), 4), "min": round(per_step_sorted[0], 4),
                  "max": round(per_step_sorted[-1], 4)}
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    # ---- the same step uncaptured (eager launches), reported beside the graph's
    eager_ms = None
    if graph is not None:
        k_eager = max(1, min(args.steps, 20))
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        eager = []
        for _ in range(k_eager):
            flush()
            g0.record(stream)
            step()
            g1.record(stream)
            torch.cuda.synchronize()
            eager.append(g0.elapsed_time(g1))
        eager_ms = reduce_max(statistics.mean(eager), world, device)

    # ---- per-launch duration of the decode kernel (events around each launch)
    kev = [[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
           for _ in range(L)]
    ksteps = max(1, min(args.steps, 20))
    kms = []
    for _ in range(ksteps):
        flush()
        step(kev)
        torch.cuda.synchronize()
        kms += [a.elapsed_time(b) for a, b in kev]
    decode_ms = statistics.mean(kms)

    # ---- e2e through the C ABI with host buffers (pinned), copies inside the timed region
    q_host = [d["q"].cpu().pin_memory() for d in W["layers"]]
    kv_host = [d["kv_new"].cpu().pin_memory() for d in W["layers"]]
    seq_host = W["seq"].cpu().pin_memory()
    bt_host = W["bt"].cpu().pin_memory()
    out_host = [torch.empty_like(o, device="cpu").pin_memory() for o in W["outs"]]
    qd = [torch.empty_like(d["q"]) for d in W["layers"]]
    kvd = [torch.empty_like(d["kv_new"]) for d in W["layers"]]
    seqd, btd = torch.empty_like(W["seq"]), torch.empty_like(W["bt"])
    h2d = sum(t.numel() * t.element_size() for t in q_host + kv_host + [seq_host, bt_host])
    d2h = sum(t.numel() * t.element_size() for t in out_host)

    # The step's copies run on their own streams so that they overlap the
    # decode: a chunk of layers waits only for its own q / kv_new, and its
    # outputs are read back as soon as its decodes are done.  Captured in a CUDA graph
    # (unless --no-graph), copies included, as a serving step would run it.
    hs, ds = torch.cuda.Stream(device), torch.cuda.Stream(device)

    # Dependencies between the copy streams and the compute stream are set
    # per chunk of layers rather than per layer: each cross-stream edge in the
    # graph adds ~2 us of scheduling latency in front of a kernel.  The host
    # link moves a layer's q in about half a layer's decode time, so the
    # inputs run ahead of the decodes: input chunks start at one layer and
    # grow by 1.6x (the decodes of layers [a, b) wait for the inputs of
    # layers < b, which arrive before the decodes reach layer a).  Output
    # chunks mirror them and shrink towards the end, where the last layer's
    # outputs cannot overlap any decode.  (Per-layer edges: +13% on the
    # 61-layer step; uniform chunks of three: +4% against this schedule.)
    in_bounds, out_bounds = e2e_chunk_bounds(L)
    in_chunks = list(zip(in_bounds[:-1], in_bounds[1:]))
    out_start = {b: a for a, b in zip(out_bounds[:-1], out_bounds[1:])}

    def e2e_step():
        hs.wait_stream(stream)
        with torch.cuda.stream(hs):
            seqd.copy_(seq_host, non_blocking=True)
            btd.copy_(bt_host, non_blocking=True)
            ev_in = {}
            for c0, c1 in in_chunks:
                for l in range(c0, c1):
                    qd[l].copy_(q_host[l], non_blocking=True)
                    kvd[l].copy_(kv_host[l], non_blocking=True)
                e = torch.cuda.Event()
                e.record(hs)
                ev_in[c0] = e
        ds.wait_stream(stream)
        for l in range(L):
            if l in ev_in:
                stream.wait_event(ev_in[l])
            if l == 0:
                mla.mla_decode_plan(seqd, btd, w.block_size, ws, dev_status=status, stream=sh,
                                    num_blocks=w.num_blocks())
            d = W["layers"][l]
            if w.append:
                mla.mla_decode_append_planned(qd[l], d["cache"], kvd[l], btd, seqd, scale,
                                              W["outs"][l], W["lses"][l], workspace=ws,
                                              dev_status=status, stream=sh)
            else:
                mla.mla_decode_planned(qd[l], d["cache"], btd, seqd, scale, W["outs"][l],
                                       W["lses"][l], workspace=ws, dev_status=status,
                                       stream=sh)
            if l + 1 in out_start:
                e = torch.cuda.Event()
                e.record(stream)
                ds.wait_event(e)
                with torch.cuda.stream(ds):
                    for k in range(out_start[l + 1], l + 1):
                        out_host[k].copy_(W["outs"][k], non_blocking=True)
        stream.wait_stream(hs)
        stream.wait_stream(ds)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e2e_graph = None
    if not args.no_graph:
        e2e_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(e2e_graph, stream=stream):
            e2e_step()
        for _ in range(2):
            e2e_graph.replay()
        torch.cuda.synchronize()
    esteps = max(1, min(args.steps, 50))
    barrier()
    t0 = time.perf_counter()
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(esteps):
        if e2e_graph is not None:
            e2e_graph.replay()
        else:
            e2e_step()
    a1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(max(a0.elapsed_time(a1), (time.perf_counter() - t0) * 1e3) / esteps,
                        world, device)
    assert int(status.item()) == 0

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return None

    cache_b, decode_b, out_b, append_b = algorithmic_bytes_per_layer(w)
    step_cache_bytes = cache_b * L
    value = job_throughput_gbs(world, step_cache_bytes, ms_step)
    hbm_peak, tf_peak, src = measured_peaks()
    achieved = decode_b / (decode_ms * 1e-3) / 1e9
    step_bytes = (decode_b + out_b + append_b) * L
    roofline_step_us = max(step_bytes / (hbm_peak * 1e9),
                           algorithmic_flops_per_layer(w) * L / (tf_peak * 1e12)) * 1e6
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "step_latency_us": round(ms_step * 1e3, 1), "step_ms": step_stats,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "seq_len": w.seq_lens[0]
                   if len(set(w.seq_lens)) == 1 else "mixed", "layers": L, "heads": 128,
                   "block_size": w.block_size, "cache_gb_per_step": round(step_cache_bytes / 1e9, 4),
                   "l2": (f"flushed: {2 * l2_bytes / 1e6:.0f} MB written between timed steps "
                          f"(outside their events)") if flush_l2 else
                         f"inputs larger than L2: {step_cache_bytes / 1e9:.2f} GB of cache per step",
                   "cuda_graph": graph is not None,
                   "parallelism": "dp-attention rank per GPU; replicas only"},
        "step_roofline_frac": round(roofline_step_us / (ms_step * 1e3), 4),
        "ms_per_step_uncaptured": round(eager_ms, 4) if eager_ms is not None else None,
        # all algorithmic bytes of the step (cache rows + q + out + appended
        # rows) per second, and against the nominal ~8 TB/s of GB300's HBM3e
        "algorithmic_gbs": round(world * step_bytes / (ms_step * 1e-3) / 1e9, 2),
        "step_frac_of_nominal_8tbs": round(step_bytes / (ms_step * 1e-3) / 8e12, 4),
        "roofline": {"bound": "hbm", "kernel": "decode_tc_kernel (mla_decode_partial)",
                     "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "peak_source": src,
                     "traffic": measured_traffic(w),
                     "algorithmic_bytes_per_launch": decode_b,
                     "launch_us": round(decode_ms * 1e3, 2)},
        "e2e": {"value": round(job_throughput_gbs(world, step_cache_bytes, e2e_ms), 2),
                "unit": "GB/s", "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "cuda_graph": e2e_graph is not None,
                "copies": "pinned host memory, on their own streams, overlapping the decode"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if not args.no_absorption:
        result["absorption"] = measure_absorption(w, device, stream, hbm_peak)
    if not args.no_tp_compare and world == 1 and w.name.startswith("dp_rank"):
        result["tp_rank"] = measure_tp_rank(device, stream, hbm_peak, ms_step, L)
    if not args.no_fp8 and world == 1:
        result["fp8"] = measure_fp8(w, device, stream, hbm_peak, tf_peak, ms_step)
    if not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, W, budget_s=args.cpu_budget)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return result


def measure_absorption(w, device, stream, hbm_peak, reps=20):
    """The absorption GEMMs of the same layers, timed beside the step (not in
    it): per layer q = [q_nope . W_UK ; q_pe] and o = out . W_UV over the
    rank's batch, each layer with its own random bf16 weights (33.6 MB a layer:
    the step streams them from HBM once, as a model does)."""
    import torch
    import mla_latent_cache_decode_gb300 as mla
    L, B = w.layers, w.batch
    g = torch.Generator(device=device).manual_seed(20261202)
    bf = torch.bfloat16
    w_uk = [torch.randn((128, 128, 512), generator=g, device=device).mul_(128 ** -0.5).to(bf)
            for _ in range(L)]
    w_uv = [torch.randn((128, 512, 128), generator=g, device=device).mul_(512 ** -0.5).to(bf)
            for _ in range(L)]
    q_nope = torch.randn((B, 128, 128), generator=g, device=device).to(bf)
    q_pe = torch.randn((B, 128, 64), generator=g, device=device).to(bf)
    out = torch.randn((B, 128, 512), generator=g, device=device).to(bf)
    q = torch.empty((B, 128, mi.ROW), dtype=bf, device=device)
    o = torch.empty((B, 128, 128), dtype=bf, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    sh = stream.cuda_stream

    def layers():
        for l in range(L):
            mla.mla_absorb_q(q_nope, q_pe, w_uk[l], q, dev_status=status, stream=sh)
            mla.mla_absorb_out(out, w_uv[l], o, dev_status=status, stream=sh)

    with torch.cuda.stream(stream):
        for _ in range(3):
            layers()
    torch.cuda.synchronize()
    # captured like the step (a model's layer runs them as graph nodes)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        layers()
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"absorption device status {int(status.item())}"
    us_layer = e0.elapsed_time(e1) * 1e3 / (reps * L)
    per_layer = 2 * (128 * 128 * 512 * 2) + B * 128 * (128 + 64 + 576 + 512 + 128) * 2
    gbs = per_layer / (us_layer * 1e-6) / 1e9
    return {"what": "q = [q_nope . W_UK ; q_pe] and o = out . W_UV per layer (absorb_kernel, "
                    "one launch each, back to back in a CUDA graph), not part of the step's value",
            "us_per_layer": round(us_layer, 2), "us_per_step": round(us_layer * L, 1),
            "bytes_per_layer": per_layer, "achieved_gbs": round(gbs, 1),
            "frac_of_hbm_peak": round(gbs / hbm_peak, 4), "launches_per_layer": 2}


def measure_tp_rank(device, stream, hbm_peak, dp_ms_step, layers, distinct=4, reps=5):
    """The same node batch under tensor-parallel attention (TP = 8): one rank
    decodes all 159 x 4096 sequences for its 16 of the 128 heads, so it reads
    the whole node's cache, against the DP rank's 20 sequences for all heads
    [dp-attention-expert-parallel-mla-kv-replication (inferenceinterviews.com),
    "A strong answer": 45.8 GB against 5.7 GB per step].  The step decodes
    `layers` layers in a CUDA graph; their caches cycle through `distinct`
    layers of 0.75 GB each (each far larger than L2, so every layer's cache is
    read from HBM, as with 61 caches)."""
    import torch
    import mla_latent_cache_decode_gb300 as mla
    heads, B, L_tok = 16, 159, 4096
    w = mi.custom_workload([L_tok] * B, block_size=64, layers=distinct, append=False,
                           pool_factor=1.0)
    lay = [mi.make_device_layer(w, l, device, num_heads=heads) for l in range(distinct)]
    bt, seq = lay[0]["block_table"], lay[0]["seq_lens"]
    out = torch.empty((B, heads, 512), dtype=torch.bfloat16, device=device)
    lse = torch.empty((B, heads), dtype=torch.float32, device=device)
    ws = mla.make_workspace(B, heads, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    sh = stream.cuda_stream

    def step():
        mla.mla_decode_plan(seq, bt, w.block_size, ws, num_heads=heads, dev_status=status,
                            stream=sh, num_blocks=w.num_blocks())
        for l in range(layers):
            d = lay[l % distinct]
            mla.mla_decode_planned(d["q"], d["cache"], bt, seq, mi.SOFTMAX_SCALE, out, lse,
                                   workspace=ws, dev_status=status, stream=sh)

    with torch.cuda.stream(stream):
        for _ in range(2):
            step()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    with torch.cuda.stream(stream):  # replays run on the current stream
        graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    # the decode kernel alone (no plan, no combine), eager, events around each launch
    kern = []
    with torch.cuda.stream(stream):
        for r in range(2 * distinct):
            d = lay[r % distinct]
            k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            k0.record(stream)
            mla.mla_decode_partial(d["q"], d["cache"], bt, seq, mi.SOFTMAX_SCALE, out, lse,
                                   workspace=ws, dev_status=status, stream=sh)
            k1.record(stream)
            kern.append((k0, k1))
    torch.cuda.synchronize()
    kern_us = sum(a.elapsed_time(b) for a, b in kern[distinct:]) * 1e3 / distinct
    layer_bytes = B * L_tok * mi.ROW * 2 + B * heads * mi.ROW * 2  # cache rows + q
    cache_bytes = B * L_tok * mi.ROW * 2 * layers
    return {"what": "one TP=8 rank: the node batch of 159 x 4096 sequences, 16 heads "
                    "(the few-head kernel), decoded over every layer's full cache",
            "heads": heads, "batch": B, "layers": layers, "ms_per_step": round(ms, 3),
            "cache_gb_per_step": round(cache_bytes / 1e9, 3),
            "cache_gbs": round(cache_bytes / (ms * 1e-3) / 1e9, 1),
            "frac_of_hbm_peak": round(cache_bytes / (ms * 1e-3) / 1e9 / hbm_peak, 4),
            "vs_dp_rank_step": round(ms / dp_ms_step, 2) if dp_ms_step else None,
            "decode_kernel_us": round(kern_us, 2),
            "decode_kernel_frac_of_hbm_peak": round(layer_bytes / (kern_us * 1e-6) / 1e9 / hbm_peak, 4),
            "caches": f"{distinct} distinct layer caches of {B * L_tok * mi.ROW * 2 / 1e9:.2f} GB, "
                      f"cycled"}


def measure_fp8(w, device, stream, hbm_peak, tf_peak, bf16_ms_step, reps=20):
    """The same step with an FP8 (E4M3) cache: each of the workload's layers
    has its own cache of one byte per latent element (576 bytes per token per
    layer), and the step is one plan, then per layer the fused quantising
    append + decode and the split combine, in a CUDA graph.  Reported beside
    the bf16 step, not part of the line's value."""
    import torch
    import mla_latent_cache_decode_gb300 as mla
    bt = mi.make_block_table(mi.rng_for(w.config_id, 0, 1), w.seq_lens, w.block_size,
                             w.num_blocks())
    layers = [mi.make_device_layer_fp8(w, l, device, block_table=bt) for l in range(w.layers)]
    L, B = w.layers, w.batch
    ws = mla.make_workspace(B, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    outs = [torch.empty((B, 128, 512), dtype=torch.bfloat16, device=device) for _ in range(L)]
    lses = [torch.empty((B, 128), dtype=torch.float32, device=device) for _ in range(L)]
    sh = stream.cuda_stream
    kv_scale = 1.0

    def step():
        d0 = layers[0]
        mla.mla_decode_plan(d0["seq_lens"], d0["block_table"], w.block_size, ws,
                            dev_status=status, stream=sh, num_blocks=w.num_blocks())
        for l, d in enumerate(layers):
            mla.mla_decode_fp8_planned(d["q"], d["cache8"], d["block_table"], d["seq_lens"],
                                       d["softmax_scale"], outs[l], lses[l], kv_scale=kv_scale,
                                       workspace=ws, dev_status=status, stream=sh,
                                       kv_new=d["kv_new"] if w.append else None)

    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"fp8 device status {int(status.item())}"
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    graph.replay()
    torch.cuda.synchronize()
    cache_bytes = sum(w.seq_lens) * mi.ROW * L               # one byte per element
    l2_bytes = torch.cuda.get_device_properties(device).L2_cache_size
    flush_buf = (torch.empty(2 * l2_bytes, dtype=torch.uint8, device=device)
                 if cache_bytes < 8 * l2_bytes else None)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for a, b in ev:
        if flush_buf is not None:
            with torch.cuda.stream(stream):
                flush_buf.fill_(0x5A)
        a.record(stream)
        graph.replay()
        b.record(stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"fp8 device status {int(status.item())}"
    per = [a.elapsed_time(b) for a, b in ev]
    ms = statistics.mean(per)
    step_bytes = (sum(w.seq_lens) * mi.ROW + B * 128 * mi.ROW * 2 + B * 128 * 512 * 2 +
                  (B * mi.ROW if w.append else 0)) * L
    flops = algorithmic_flops_per_layer(w) * L
    roof_us = max(step_bytes / (hbm_peak * 1e9), flops / (tf_peak * 1e12)) * 1e6
    return {"what": "the same step over an FP8 (E4M3) cache, fused quantising append, "
                    "CUDA graph; not part of the line's value",
            "ms_per_step": round(ms, 4), "step_ms_median": round(statistics.median(per), 4),
            "cache_gb_per_step": round(cache_bytes / 1e9, 4),
            "cache_gbs": round(cache_bytes / (ms * 1e-3) / 1e9, 1),
            "frac_of_hbm_peak": round(cache_bytes / (ms * 1e-3) / 1e9 / hbm_peak, 4),
            "roofline_us": round(roof_us, 1),
            "roofline_bound": "tensor" if flops / (tf_peak * 1e12) > step_bytes / (hbm_peak * 1e9)
            else "hbm",
            "step_roofline_frac": round(roof_us / (ms * 1e3), 4),
            "vs_bf16_step": round(ms / bf16_ms_step, 3), "kv_scale": kv_scale,
            "l2": "flushed between timed steps" if flush_buf is not None else "inputs larger than L2"}


# ----------------------------------------------------------------------------- oracle on the host

def _host_layer_for_oracle(w, d, bt):
    import oracle  # noqa: F401
    return dict(q=mi.to_bits(d["q"]), cache=mi.to_bits(d["cache"]), bt=bt,
                seq=d["seq_lens"].cpu().numpy(), kv=mi.to_bits(d["kv_new"]),
                slots=d["slot_mapping"].cpu().numpy())


def cpu_baseline(w, W, budget_s=15.0):
    """The fp64 oracle, as it stands, on the host cores over a bounded sample."""
    import oracle
    done_bytes, t_used, layers_done = 0, 0.0, 0
    for l in range(w.layers):
        h = _host_layer_for_oracle(w, W["layers"][l], W["bt_host"])
        t0 = time.perf_counter()
        cache = h["cache"]
        if w.append:
            oracle.append(h["kv"], h["slots"], cache)
        oracle.decode(h["q"], cache, h["bt"], h["seq"], mi.SOFTMAX_SCALE)
        t_used += time.perf_counter() - t0
        done_bytes += sum(w.seq_lens) * ROW_BYTES
        layers_done += 1
        if t_used >= budget_s:
            break
    return {"value": round(done_bytes / t_used / 1e9, 4), "unit": "GB/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{layers_done} of {w.layers} layers (append + decode of all {w.batch} "
                      f"requests), {t_used:.1f} s"}


def run_reference(args, w, rank, world):
    """Reference arm: the oracle, timed on the host cores, on the same workload and metric."""
    if rank != 0:
        return None
    import oracle
    rng = mi.rng_for(w.config_id, 0, 1)
    bt = mi.make_block_table(rng, w.seq_lens, w.block_size, w.num_blocks())
    # one request of one layer per step: bounded so K + W steps finish in minutes
    b = 0
    L = w.seq_lens[b]
    need = -(-L // w.block_size)
    g = np.random.default_rng(mi.BASE_SEED + w.config_id)
    cache = np.full((w.num_blocks(), w.block_size, mi.ROW), mi.BF16_NAN, np.uint16)
    blocks = bt[b, :need]
    cache[blocks] = mi.f32_to_bf16_bits(
        g.standard_normal((need, w.block_size, mi.ROW), dtype=np.float32))
    q = mi.make_queries(g, 1)
    kv = mi.f32_to_bf16_bits(g.standard_normal((1, mi.ROW), dtype=np.float32))
    slots = np.array([mi.slot_of(bt, b, L - 1, w.block_size)], np.int64)
    seq = np.array([L], np.int32)

    def step():
        oracle.append(kv, slots, cache)
        oracle.decode(q, cache, bt[b:b + 1], seq, mi.SOFTMAX_SCALE)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = L * ROW_BYTES / dt / 1e9
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "layers": w.layers,
                       "heads": 128, "block_size": w.block_size,
                       "parallelism": "dp-attention rank per GPU; replicas only"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s",
                             "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": f"each step: append + decode of 1 of {w.batch} requests "
                                       f"({L} tokens, 128 heads) of 1 of {w.layers} layers"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=3)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-absorption", action="store_true",
                    help="skip the separate timing of the absorption GEMMs")
    ap.add_argument("--no-tp-compare", action="store_true",
                    help="skip timing one TP=8 rank's step over the same node batch (16 heads)")
    ap.add_argument("--no-fp8", action="store_true",
                    help="skip timing the same step over an FP8 (E4M3) cache")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--layers", type=int, default=0,
                    help="run only the first N layers of the workload (for profiling captures)")
    ap.add_argument("--tp-only", action="store_true",
                    help="time only one TP=8 rank's step (16 heads; --layers sets its layers) "
                         "and print that object")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local_rank = dist_env()
    if args.tp_only:
        import torch
        torch.cuda.set_device(local_rank)
        device = torch.device("cuda", local_rank)
        hbm_peak = measured_peaks()[0]
        res = measure_tp_rank(device, torch.cuda.Stream(), hbm_peak, None, args.layers or 61)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return
    w = mi.workload(args.config)
    if args.layers and args.layers < w.layers:
        import dataclasses
        w = dataclasses.replace(w, layers=args.layers, name=f"{w.name}_first{args.layers}")
    if args.impl == "reference":
        res = run_reference(args, w, rank, world)
    else:
        res = run_mine(args, w, rank, world, local_rank)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()

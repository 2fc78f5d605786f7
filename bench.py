#!/usr/bin/env python3
"""Benchmark: params/s through the partition-aware ZeRO step on one GB300.

One step is the whole hot path over every bucket in one pass, with no bucket
buffer (zr_step_direct_range): each emulated rank's per-parameter bf16
gradients are read where they lie, sliced by partition as the IPG bucket
would hold them, reduce-scattered with the 1/N predivide, and AdamW and the
bf16 cast run on each partition, consecutive buckets sharing launches. The
same step with the bucket materialised (planned pack, then the fused
reduce-scatter + AdamW + cast per bucket) is reported beside it. Default workload: the
irregular layout (10,000 log-uniform params, 718,175,492 elements, 16 emulated
ranks, 2^24-element buckets, integer-valued grads), each rank's gradients laid
out as separately allocated tensors (512-byte aligned starts). Inputs are
synthetic, drawn on the device; every bucket's working set (~1 GB) exceeds
L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0). ``--impl reference`` times the CPU oracle on
the host instead (a bounded sample of the same workload per step).
Under torchrun each rank runs its own copy of the workload on its own GPU
("replicas only": the emulated data-parallel group lives on one GPU and
nothing crosses GPUs); only a host-side gloo barrier and max are used.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "params/s through fused reduce-scatter+AdamW shard step; HBM GB/s vs peak"
UNIT = "params/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="zr", choices=["zr", "reference"])
    ap.add_argument("--workload", default="irregular_10k")
    ap.add_argument("--world", type=int, default=0, help="override the workload's emulated replica count")
    ap.add_argument("--bucket", type=int, default=0, help="override the workload's reduce_bucket_size")
    ap.add_argument("--arrival", default="flat", choices=["flat", "reverse"],
                    help="gradient arrival order that fills the buckets (reverse: backward's order)")
    ap.add_argument("--max-norm", type=float, default=1.0,
                    help="clip norm of the step with the global gradient check (<= 0: check without clipping)")
    ap.add_argument("--no-clipped", action="store_true", help="skip timing the step with the gradient check")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle sample budget")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class Dist:
    """Host-side barrier / max over ranks (gloo); no data-path collective."""

    def __init__(self, world):
        self.world = world
        self.pg = None
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
            self.dist = dist

    def barrier(self):
        if self.world > 1:
            self.dist.barrier()

    def max(self, x: float) -> float:
        if self.world == 1:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.world > 1:
            self.dist.destroy_process_group()


# ----------------------------------------------------------------------------
# clocks
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def code_only(src: str) -> str:
    """C/C++/CUDA source without its comments, blank lines and trailing blanks
    (the sources have no comment markers inside string literals)."""
    import re
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def kernel_source_hash() -> str:
    """Hash of what the profiled DRAM traffic belongs to: the device code, the
    host code that plans and launches it (grids, shared memory, launch shapes)
    and the compiler flags, with comments removed; comment changes leave it."""
    from zero_partition_aware_gb300 import build as zb
    h = hashlib.sha256()
    for rel in ("zero_partition_aware_gb300/csrc/zr_kernels.cuh", "zero_partition_aware_gb300/csrc/zr_internal.h",
                "zero_partition_aware_gb300/csrc/kernels.cu", "include/zr.h"):
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    h.update(" ".join(zb.ARCH + zb.COMMON_FLAGS).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if it matches this source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e


# ----------------------------------------------------------------------------
# the GPU arm
# ----------------------------------------------------------------------------

def build_state(wl, device, arrival="flat"):
    import torch
    from zero_partition_aware_gb300 import workloads as W
    from zero_partition_aware_gb300.engine import DPGroup
    order = list(range(len(wl.numel) - 1, -1, -1)) if arrival == "reverse" else None
    grp = DPGroup(list(wl.numel), wl.world, wl.bucket, device=device, arrival=order)
    gen = W.generator(device, 0)
    T = wl.total
    master = torch.randn(T, generator=gen, device=device).mul_(wl.master_std)
    # each rank's grads: per-parameter tensors at 512-byte aligned starts of one arena
    offs = W.arena_offsets(wl.numel, 256)
    arena_n = offs[-1] + wl.numel[-1]
    arenas = [W.draw_grad(wl, arena_n, gen, device) for _ in range(wl.world)]
    m = W.draw_state(wl, T, gen, device)
    v = W.draw_state(wl, T, gen, device)
    grp.load_flat(master, m, v)
    del master, m, v
    views = [[a[o:o + n] for o, n in zip(offs, wl.numel)] for a in arenas]
    table = grp.grad_table(views)
    plan = grp.pack_plan(table)  # packing descriptors, built once like the gradient tensors
    return grp, arenas, table, plan


def bucket_bytes(grp, b, world):
    """Algorithmic bytes of the pack and of the fused kernel for bucket b."""
    L = grp.layout
    _, nb = L.bucket(b)
    pad = L.P - L.T if L.n_params and L.param(L.n_params - 1)[1] == b else 0
    real = nb - pad                               # elements that come from parameter grads
    pack = world * (2 * real + 2 * nb)            # read real grads, write the whole bucket
    fused = nb * (2 * world + 12 + 12 + 2)        # N bf16 grads + p,m,v read + p,m,v write + bf16 param
    return pack, fused


def timed_steps(args, nbk, launch_a, launch_b, stream, dist):
    """K steps bracketed by barrier + synchronize; CUDA events around every
    launch_a(b) and launch_b(b) (launch_b may be None). Returns the step time
    (max over ranks), the per-kernel totals and the libzr launch count."""
    import torch
    from zero_partition_aware_gb300 import zr
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * nbk + 1)] for _ in range(args.steps)]
    start_ev, end_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    n0 = zr.zr_launch_count()
    start_ev.record(stream)
    for k in range(args.steps):
        for b in range(nbk):
            evs[k][2 * b].record(stream)
            launch_a(b)
            evs[k][2 * b + 1].record(stream)
            if launch_b is not None:
                launch_b(b)
        evs[k][2 * nbk].record(stream)
    end_ev.record(stream)
    torch.cuda.synchronize()
    launches = zr.zr_launch_count() - n0
    dist.barrier()
    t_a = sum(evs[k][2 * b].elapsed_time(evs[k][2 * b + 1]) for k in range(args.steps) for b in range(nbk))
    t_b = sum(evs[k][2 * b + 1].elapsed_time(evs[k][2 * b + 2]) for k in range(args.steps) for b in range(nbk))
    ms_step = dist.max(start_ev.elapsed_time(end_ev) / args.steps)
    per_step = sorted(evs[k][0].elapsed_time(evs[k][2 * nbk]) for k in range(args.steps))
    timed_steps.last = {"median": round(dist.max(per_step[len(per_step) // 2]), 4), "best": round(dist.max(per_step[0]), 4)}
    return ms_step, t_a, t_b, launches


def timed_clipped(args, grp, dplan, hp, stream, dist):
    """K steps of the two-pass step with the global gradient check: every
    bucket averaged into the gradient partitions with the norm sums, then the
    check and the clipped AdamW + cast. CUDA events around the norm pass, the
    check and the update. Returns (ms/step, norm ms, check ms, update ms,
    launches, the last outcome)."""
    import torch
    from zero_partition_aware_gb300 import zr
    nbk = grp.layout.n_buckets
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start_ev, end_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    n0 = zr.zr_launch_count()
    start_ev.record(stream)
    for k in range(args.steps):
        ev[k][0].record(stream)
        zr.zr_rs_direct_norm_range(dplan, 0, nbk, grp.scale, grp._p_grad, grp.check, stream=stream)
        ev[k][1].record(stream)
        zr.zr_grad_check_finalize(grp.check, args.max_norm, stream=stream)
        ev[k][2].record(stream)
        zr.zr_adam_clip_step(grp.layout, grp._p_master, grp._p_m, grp._p_v, grp._p_grad, hp, grp.check,
                             grp.param, stream=stream)
        ev[k][3].record(stream)
    end_ev.record(stream)
    torch.cuda.synchronize()
    launches = zr.zr_launch_count() - n0
    dist.barrier()
    t = [sum(ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(args.steps)) for i in range(3)]
    ms_step = dist.max(start_ev.elapsed_time(end_ev) / args.steps)
    return ms_step, t[0], t[1], t[2], launches, zr.zr_gradcheck_read(grp.check, stream)


def run_gpu(args, rank, nranks, local, dist):
    import torch
    from zero_partition_aware_gb300 import workloads as W
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    wl = W_lookup(args)
    grp, arenas, table, plan = build_state(wl, device, args.arrival)
    dplan = grp.direct_plan(table)
    L = grp.layout
    hp = W.AdamW(step=wl.adam.step)
    nbk = L.n_buckets
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    pack_b, fused_b = zip(*[bucket_bytes(grp, b, wl.world) for b in range(nbk)])
    pack_bytes, fused_bytes = sum(pack_b), sum(fused_b)
    peak, peak_kind = measured_peaks()
    W_ = max(args.warmup, 3)

    direct = lambda b: grp.direct(b, dplan, hp, stream=stream)
    direct_all = lambda _: grp.step_direct(dplan, hp, stream=stream)
    pack = lambda b: grp.pack_planned(b, plan, stream)
    fused = lambda b: grp.fused(b, hp, stream=stream)

    # the headline step: steps 1-4 in one pass for every bucket (no bucket buffer), consecutive
    # buckets sharing launches (zr_step_direct_range)
    for _ in range(W_):
        direct_all(0)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ms_step, t_direct, _, launches = timed_steps(args, 1, direct_all, None, stream, dist)
    step_stats = timed_steps.last
    clk = clocks.stop()

    # the same step captured once in a CUDA graph and replayed
    graph_ms = None
    try:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            grp.step_direct(dplan, hp)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg):
            grp.step_direct(dplan, hp)
        for _ in range(2):
            cg.replay()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record()
        for _ in range(args.steps):
            cg.replay()
        g1.record()
        torch.cuda.synchronize()
        graph_ms = dist.max(g0.elapsed_time(g1) / args.steps)
        del cg
    except RuntimeError as e:  # reported, not fatal: the eager step is the measured one
        graph_ms = f"capture failed: {e}"

    # the same step with one launch per bucket (zr_step_direct), as buckets reduced while backward fills them
    for _ in range(W_):
        for b in range(nbk):
            direct(b)
    torch.cuda.synchronize()
    ms_pb, t_pb, _, launches_pb = timed_steps(args, nbk, direct, None, stream, dist)

    # the same step with the bucket materialised: planned pack, then the fused kernel
    for _ in range(W_):
        for b in range(nbk):
            pack(b)
            fused(b)
    torch.cuda.synchronize()
    ms_two, t_pack, t_fused, launches_two = timed_steps(args, nbk, pack, fused, stream, dist)

    # the same packed buckets reduced in flat order: the direct kernel over their param slices
    reduce_flat = lambda b: grp.reduce_packed(b, hp, stream=stream)
    for _ in range(W_):
        for b in range(nbk):
            pack(b)
            reduce_flat(b)
    torch.cuda.synchronize()
    ms_two_f, _, t_red_f, _ = timed_steps(args, nbk, pack, reduce_flat, stream, dist)

    # the same two kernels with packing overlapped: bucket b+1 packed on a second stream while b is reduced
    plans2 = grp.overlap_plans(table)
    side = torch.cuda.Stream()
    for _ in range(W_):
        grp.step_overlapped(plans2, hp, stream=stream, side_stream=side, flat_order=True)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(args.steps):
        grp.step_overlapped(plans2, hp, stream=stream, side_stream=side, flat_order=True)
    ev1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    ms_ov = dist.max(ev0.elapsed_time(ev1) / args.steps)

    value = nranks * L.T / (ms_step / 1e3)
    gbs = lambda byts, ms: byts * args.steps / (ms / 1e3) / 1e9
    direct_gbs, pack_gbs, fused_gbs = gbs(fused_bytes, t_direct), gbs(pack_bytes, t_pack), gbs(fused_bytes, t_fused)
    launches_per_step = max(1, round(launches / args.steps))
    kname = "rs_direct_bf16_w16" if wl.world == 16 else "rs_direct"
    tr = profiled_traffic(kname)
    elems_per_launch = L.P / launches_per_step
    roofline = {"bound": "hbm", "achieved": round(direct_gbs, 1), "peak": peak, "unit": "GB/s",
                "frac": round(direct_gbs / peak, 4),
                "traffic": round(tr["dram_bytes_per_element"] * elems_per_launch) if tr else None,
                "kernel": kname, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy)"
                if peak_kind == "measured" else "fallback 6.8 TB/s",
                "algorithmic_bytes_per_launch": round(fused_bytes / launches_per_step)}
    pb_gbs = gbs(fused_bytes, t_pb)
    kernels = {
        "rs_direct": {"ms_per_step": round(t_direct / args.steps, 4), "GB_per_s": round(direct_gbs, 1),
                      "frac_of_peak": round(direct_gbs / peak, 4), "bytes_per_param": 2 * wl.world + 26,
                      "launches_per_step": launches_per_step},
        "rs_direct_graph": {"ms_per_step": round(graph_ms, 4) if isinstance(graph_ms, float) else graph_ms,
                            "how": "the same step captured once in a CUDA graph, replayed"},
        "rs_direct_per_bucket": {"ms_per_step": round(ms_pb, 4), "params_per_s": round(nranks * L.T / (ms_pb / 1e3)),
                                 "GB_per_s": round(pb_gbs, 1), "frac_of_peak": round(pb_gbs / peak, 4),
                                 "launches_per_step": round(launches_pb / args.steps)},
    }
    two_kernel = {
        "ms_per_step": round(ms_two, 4), "params_per_s": round(nranks * L.T / (ms_two / 1e3)),
        "launches_per_step": round(launches_two / args.steps),
        "bucket_pack": {"ms_per_step": round(t_pack / args.steps, 4), "GB_per_s": round(pack_gbs, 1),
                        "frac_of_peak": round(pack_gbs / peak, 4), "bytes_per_param": 4 * wl.world,
                        "traffic_per_replica_element": (profiled_traffic("bucket_pack_bf16_w16") or {}).get(
                            "dram_bytes_per_element") if wl.world == 16 else None},
        "rs_adam_fused": {"ms_per_step": round(t_fused / args.steps, 4), "GB_per_s": round(fused_gbs, 1),
                          "frac_of_peak": round(fused_gbs / peak, 4), "bytes_per_param": 2 * wl.world + 26,
                          "traffic_per_element": (profiled_traffic("rs_adam_fused_bf16_w16") or {}).get(
                              "dram_bytes_per_element") if wl.world == 16 else None},
        "reduced_in_flat_order": {
            "ms_per_step": round(ms_two_f, 4), "params_per_s": round(nranks * L.T / (ms_two_f / 1e3)),
            "reduce_ms_per_step": round(t_red_f / args.steps, 4),
            "reduce_frac_of_peak": round(gbs(fused_bytes, t_red_f) / peak, 4),
            "how": "the same packed buckets, each reduced by zr_step_direct over a plan whose gradients are the "
                   "bucket buffers' param slices (DPGroup.reduce_packed)"},
        "overlapped": {"ms_per_step": round(ms_ov, 4), "params_per_s": round(nranks * L.T / (ms_ov / 1e3)),
                       "GB_per_s": round(gbs(pack_bytes + fused_bytes, ms_ov * args.steps), 1),
                       "how": "pack of bucket b+1 on a second stream while bucket b is reduced in flat order "
                              "(DPGroup.reduce_packed); two bucket buffer sets, ordered by events"},
    }

    # the unfused steps, one kernel each: the reduce-scatter and the all-reduce reference path
    # over every bucket of one contiguous gradient buffer per rank (the buckets back to back in
    # bucket order, filled once by the pack), AdamW over the partitions and the gather-cast
    from zero_partition_aware_gb300 import zr as _zr
    grads = grp.grad_shards()
    starts = [0]
    for b in range(nbk):
        starts.append(starts[-1] + L.bucket(b)[1])
    torch.cuda.empty_cache()
    free = torch.cuda.mem_get_info(torch.device(device))[0]
    if wl.world * starts[-1] * (grp.buckets[0].element_size() if grp.buckets else 2) * 3 > 0.9 * free:
        return_unfused = {"skipped": "the contiguous gradient buffers and the all-reduce outputs would not fit "
                                     f"({wl.world} ranks x {starts[-1]} elements)"}
    else:
        return_unfused = None
    gbuf = [torch.empty(starts[-1] if return_unfused is None else 1, dtype=grp.grad_dtype, device=device)
            for _ in range(wl.world)]
    if return_unfused is None:
        for b in range(nbk):
            _zr.zr_bucket_pack(L, b, table, [t[starts[b]:starts[b + 1]] for t in gbuf], dtype=grp.zr_dtype,
                               stream=stream)
    p_gbuf = _zr.PtrArray(gbuf)
    ar_out = [torch.empty(starts[-1] if return_unfused is None else 1, dtype=torch.float32, device=device)
              for _ in range(wl.world)]
    p_ar = _zr.PtrArray(ar_out)
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def unfused_step(timed):
        e = [ev() for _ in range(6)]
        e[0].record(stream)
        _zr.zr_reduce_scatter_avg_range(L, 0, nbk, p_gbuf, grp.scale, grp._p_grad, dtype=grp.zr_dtype, stream=stream)
        e[1].record(stream)
        _zr.zr_allreduce_avg_range(L, 0, nbk, p_gbuf, grp.scale, p_ar, dtype=grp.zr_dtype, stream=stream)
        e[2].record(stream)
        _zr.zr_adam_shard_step(L, -1, grp._p_master, grp._p_m, grp._p_v, grp._p_grad, hp, stream=stream)
        e[3].record(stream)
        _zr.zr_gather_cast_bf16(L, grp._p_master, grp.param, stream=stream)
        e[4].record(stream)
        _zr.zr_rs_adam_fused_range(L, 0, nbk, p_gbuf, grp.scale, grp._p_master, grp._p_m, grp._p_v, hp, grp.param,
                                   dtype=grp.zr_dtype, stream=stream)
        e[5].record(stream)
        timed += [("rs", e[0], e[1]), ("ar", e[1], e[2]), ("adam", e[2], e[3]), ("cast", e[3], e[4]),
                  ("fused_range", e[4], e[5])]

    def per_bucket_rs(timed):  # the per-bucket calls over the same buffer, for comparison
        for b in range(nbk):
            x = [t[starts[b]:starts[b + 1]] for t in gbuf]
            e = [ev() for _ in range(3)]
            e[0].record(stream)
            _zr.zr_reduce_scatter_avg(L, b, x, grp.scale, grp._p_grad, dtype=grp.zr_dtype, stream=stream)
            e[1].record(stream)
            _zr.zr_allreduce_avg(L, b, x, grp.scale, [t[starts[b]:starts[b + 1]] for t in ar_out],
                                 dtype=grp.zr_dtype, stream=stream)
            e[2].record(stream)
            timed += [("rs_pb", e[0], e[1]), ("ar_pb", e[1], e[2])]

    marks = []
    if return_unfused is None:
        for _ in range(W_):
            unfused_step([])
            per_bucket_rs([])
        torch.cuda.synchronize()
        for _ in range(args.steps):
            unfused_step(marks)
        for _ in range(args.steps):
            per_bucket_rs(marks)
        torch.cuda.synchronize()
    if return_unfused is None:
        tsum = {k: 0.0 for k in ("rs", "ar", "adam", "cast", "fused_range", "rs_pb", "ar_pb")}
        for k, a, b_ in marks:
            tsum[k] += a.elapsed_time(b_)
        unfused = {}
        w16 = wl.world == 16
        traffic_of = {"rs": ["reduce_scatter_range_bf16_w16"], "adam": ["adam_shard_w16"],
                      "ar": ["allreduce_pass_bf16_w16", "allreduce_bcast_w16"],
                      "fused_range": ["rs_adam_fused_bf16_w16"]}
        for k, name, bpp in (("rs", "reduce_scatter_avg", 2 * wl.world + 4), ("adam", "adam_shard_step", 28),
                             ("cast", "gather_cast_bf16", 6), ("ar", "allreduce_avg", 6 * wl.world),
                             ("fused_range", "rs_adam_fused_range", 2 * wl.world + 26),
                             ("rs_pb", "reduce_scatter_avg_per_bucket", 2 * wl.world + 4),
                             ("ar_pb", "allreduce_avg_per_bucket", 6 * wl.world)):
            g_ = gbs(L.P * bpp, tsum[k])
            unfused[name] = {"ms_per_step": round(tsum[k] / args.steps, 4), "GB_per_s": round(g_, 1),
                             "frac_of_peak": round(g_ / peak, 4), "bytes_per_param": bpp}
            if w16 and k in traffic_of:
                trs = [profiled_traffic(t) for t in traffic_of[k]]
                unfused[name]["traffic_per_element"] = (round(sum(t["dram_bytes_per_element"] for t in trs), 3)
                                                        if all(trs) else None)
    else:
        unfused = dict(return_unfused)
    unfused["how"] = ("reduce_scatter_avg, allreduce_avg and rs_adam_fused_range: the grouped calls "
                      "(zr_reduce_scatter_avg_range, zr_allreduce_avg_range, zr_rs_adam_fused_range) over one "
                      "contiguous buffer per rank holding every bucket; *_per_bucket: one zr_reduce_scatter_avg / "
                      "zr_allreduce_avg call per bucket of the same buffer")
    del ar_out, p_ar, gbuf, p_gbuf
    torch.cuda.empty_cache()

    clipped = None
    if not args.no_clipped:
        # the step with the global gradient check before the update (two passes)
        grp.grad_shards()
        for _ in range(W_):
            grp.step_direct_clipped(dplan, hp, args.max_norm, stream=stream)
        torch.cuda.synchronize()
        ms_c, t_norm, t_fin, t_clip, launches_c, outcome = timed_clipped(args, grp, dplan, hp, stream, dist)
        norm_bytes = L.P * (2 * wl.world + 4)
        clip_bytes = L.P * 30
        tr_norm = profiled_traffic("rs_direct_norm_bf16_w16" if wl.world == 16 else "rs_direct_norm")
        tr_clip = profiled_traffic("adam_clip_w16" if wl.world == 16 else "adam_clip")
        clipped = {
            "ms_per_step": round(ms_c, 4), "params_per_s": round(nranks * L.T / (ms_c / 1e3)),
            "max_norm": args.max_norm, "launches_per_step": round(launches_c / args.steps),
            "outcome": {"norm": outcome["norm"], "coef": outcome["coef"], "skip": outcome["skip"]},
            "rs_direct_norm": {"ms_per_step": round(t_norm / args.steps, 4),
                               "GB_per_s": round(gbs(norm_bytes, t_norm), 1),
                               "frac_of_peak": round(gbs(norm_bytes, t_norm) / peak, 4),
                               "bytes_per_param": 2 * wl.world + 4,
                               "traffic_per_element": tr_norm["dram_bytes_per_element"] if tr_norm else None},
            "grad_check_finalize": {"ms_per_step": round(t_fin / args.steps, 4)},
            "adam_clip_step": {"ms_per_step": round(t_clip / args.steps, 4),
                               "GB_per_s": round(gbs(clip_bytes, t_clip), 1),
                               "frac_of_peak": round(gbs(clip_bytes, t_clip) / peak, 4), "bytes_per_param": 30,
                               "traffic_per_element": tr_clip["dram_bytes_per_element"] if tr_clip else None},
        }

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, wl, grp, arenas, dplan, hp, stream, nranks, dist)

    out = {"metric": METRIC, "value": round(value), "unit": UNIT, "n_gpus": nranks, "steps": args.steps,
           "warmup": W_, "ms_per_step": round(ms_step, 4), "ms_per_step_median": step_stats["median"],
           "ms_per_step_best": step_stats["best"], "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
           "config": {"workload": wl.name, "params": L.T, "padded": L.P, "world": wl.world,
                      "reduce_bucket_size": wl.bucket, "buckets": nbk, "grad_dtype": "bf16",
                      "grad_layout": "per-parameter tensors, 512-byte aligned starts",
                      "arrival": args.arrival,
                      "step": "zr_step_direct_range over every bucket (pack + reduce-scatter + AdamW + bf16 cast in "
                              "one pass; consecutive buckets share launches)",
                      "l2": "no flush: every bucket's working set (~1 GB) exceeds the 129 MB L2",
                      "parallelism": f"replicas only x{nranks}"},
           "roofline": roofline, "kernels": kernels, "two_kernel_step": two_kernel, "unfused_steps": unfused,
           "gpu_launches": int(launches), "clocks": clk}
    if clipped is not None:
        out["clipped_step"] = clipped
    if e2e is not None:
        out["e2e"] = e2e
    return out


def run_gpu_micro(args, rank, nranks, local, dist):
    """A workload whose gradients come from several micro-steps (the Llama 1.1B
    configuration: 4 bf16 micro-steps summed into an fp32 main_grad buffer per
    rank, laid out flat in bucket order, then the fused step). One step is
    the whole path: zr_grad_accumulate_first for micro-step 0, zr_grad_accumulate
    for the middle ones, and per bucket zr_rs_adam_fused_acc, which adds the
    last micro-step while it averages. The unfolded sequence (every micro-step
    accumulated, then zr_rs_adam_fused on the fp32 buffer) is timed beside it."""
    import torch
    from zero_partition_aware_gb300 import workloads as W
    from zero_partition_aware_gb300 import zr
    from zero_partition_aware_gb300.engine import DPGroup
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    wl = W_lookup(args)
    S_ = wl.micro_steps
    grp = DPGroup(list(wl.numel), wl.world, wl.bucket, grad_dtype=torch.float32, device=device,
                  allocate_buckets=False)
    L = grp.layout
    gen = W.generator(device, 0)
    master = torch.randn(L.T, generator=gen, device=device).mul_(wl.master_std)
    mb = []
    for _ in range(wl.world):
        row = []
        for _ in range(S_):
            g = torch.zeros(L.P, dtype=torch.bfloat16, device=device)
            g[: L.T].copy_(W.draw_grad(wl, L.T, gen, device))
            row.append(g)
        mb.append(row)
    m = W.draw_state(wl, L.T, gen, device)
    v = W.draw_state(wl, L.T, gen, device)
    grp.load_flat(master, m, v)
    del master, m, v
    main = [torch.zeros(L.P, dtype=torch.float32, device=device) for _ in range(wl.world)]
    main_views = grp.main_grad_views(main)
    last_views = grp.main_grad_views([row[-1] for row in mb])
    hp = W.AdamW(step=wl.adam.step)
    stream = torch.cuda.current_stream()
    nbk = L.n_buckets
    peak, peak_kind = measured_peaks()
    W_ = max(args.warmup, 3)

    def accumulate(upto):
        for k in range(wl.world):
            zr.zr_grad_accumulate_first(main[k], mb[k][0], stream=stream)
        for s_ in range(1, upto):
            for k in range(wl.world):
                zr.zr_grad_accumulate(main[k], mb[k][s_], stream=stream)

    def timed(acc_upto, tail):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        dist.barrier()
        torch.cuda.synchronize()
        n0 = zr.zr_launch_count()
        for k in range(args.steps):
            ev[k][0].record(stream)
            accumulate(acc_upto)
            ev[k][1].record(stream)
            tail()
            ev[k][2].record(stream)
        torch.cuda.synchronize()
        launches = zr.zr_launch_count() - n0
        dist.barrier()
        t_acc = sum(ev[k][0].elapsed_time(ev[k][1]) for k in range(args.steps))
        t_tail = sum(ev[k][1].elapsed_time(ev[k][2]) for k in range(args.steps))
        ms = dist.max(ev[0][0].elapsed_time(ev[-1][2]) / args.steps)
        return ms, t_acc, t_tail, launches

    folded = lambda: grp.step_in_place_acc(main_views, last_views, hp, stream=stream)
    unfolded = lambda: grp.step_in_place(main_views, hp, stream=stream)
    for _ in range(W_):
        accumulate(S_ - 1)
        folded()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ms, t_acc, t_fold, launches = timed(S_ - 1, folded)
    clk = clocks.stop()
    for _ in range(W_):
        accumulate(S_)
        unfolded()
    torch.cuda.synchronize()
    ms_u, t_acc_u, t_fused_u, launches_u = timed(S_, unfolded)

    N = wl.world
    gbs = lambda byts, t: byts * args.steps / (t / 1e3) / 1e9
    acc_bytes = L.P * N * (6 + 10 * (S_ - 2))      # first micro-step: read 2, write 4; the others read 6, write 4
    fold_bytes = L.P * (6 * N + 26)                 # N x (fp32 main + bf16 last) + p, m, v r/w + bf16 param
    acc_bytes_u = L.P * N * (6 + 10 * (S_ - 1))
    fused_bytes_u = L.P * (4 * N + 26)
    acc_gbs, fold_gbs = gbs(acc_bytes, t_acc), gbs(fold_bytes, t_fold)
    dominant = ("grad_accumulate", acc_gbs, acc_bytes) if t_acc >= t_fold else ("rs_adam_fused_acc", fold_gbs,
                                                                                fold_bytes)
    launches_acc = N * (S_ - 1)
    is_acc = dominant[0] == "grad_accumulate"
    tr = profiled_traffic("grad_accumulate_bf16" if is_acc else ("rs_adam_fused_acc_w8" if N == 8 else "none"))
    elems_per_launch = L.P if is_acc else L.P / nbk
    roofline = {"bound": "hbm", "achieved": round(dominant[1], 1), "peak": peak, "unit": "GB/s",
                "frac": round(dominant[1] / peak, 4),
                "traffic": round(tr["dram_bytes_per_element"] * elems_per_launch) if tr else None,
                "kernel": dominant[0],
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy)"
                if peak_kind == "measured" else "fallback 6.8 TB/s",
                "algorithmic_bytes_per_launch": round(dominant[2] / (launches_acc if dominant[0] == "grad_accumulate"
                                                                     else nbk))}
    out = {"metric": METRIC, "value": round(nranks * L.T / (ms / 1e3)), "unit": UNIT, "n_gpus": nranks,
           "steps": args.steps, "warmup": W_, "ms_per_step": round(ms, 4), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
           "config": {"workload": wl.name, "params": L.T, "padded": L.P, "world": N,
                      "reduce_bucket_size": wl.bucket, "buckets": nbk, "micro_steps": S_,
                      "grad_dtype": "bf16 micro-steps into fp32 main_grad (flat, bucket order)",
                      "step": "zr_grad_accumulate_first + zr_grad_accumulate for micro-steps 0..S-2, then per "
                              "bucket zr_rs_adam_fused_acc (last micro-step folded into the fused step)",
                      "l2": "no flush: every launch's working set exceeds the 129 MB L2",
                      "parallelism": f"replicas only x{nranks}"},
           "roofline": roofline,
           "kernels": {
               "grad_accumulate": {"ms_per_step": round(t_acc / args.steps, 4), "GB_per_s": round(acc_gbs, 1),
                                   "frac_of_peak": round(acc_gbs / peak, 4),
                                   "bytes_per_param": N * (6 + 10 * (S_ - 2)), "launches_per_step": launches_acc},
               "rs_adam_fused_acc": {"ms_per_step": round(t_fold / args.steps, 4), "GB_per_s": round(fold_gbs, 1),
                                     "frac_of_peak": round(fold_gbs / peak, 4), "bytes_per_param": 6 * N + 26,
                                     "launches_per_step": nbk}},
           "unfolded_step": {
               "ms_per_step": round(ms_u, 4), "params_per_s": round(nranks * L.T / (ms_u / 1e3)),
               "grad_accumulate": {"ms_per_step": round(t_acc_u / args.steps, 4),
                                   "GB_per_s": round(gbs(acc_bytes_u, t_acc_u), 1),
                                   "bytes_per_param": N * (6 + 10 * (S_ - 1))},
               "rs_adam_fused": {"ms_per_step": round(t_fused_u / args.steps, 4),
                                 "GB_per_s": round(gbs(fused_bytes_u, t_fused_u), 1),
                                 "frac_of_peak": round(gbs(fused_bytes_u, t_fused_u) / peak, 4),
                                 "bytes_per_param": 4 * N + 26}},
           "gpu_launches": int(launches), "clocks": clk,
           "e2e": None, "e2e_note": "not run for micro-step workloads: 4 micro-steps of bf16 grads are 70 GB"}
    return out


def run_e2e(args, wl, grp, arenas, dplan, hp, stream, nranks, dist):
    """The same step through the public API with the gradients starting in pinned
    host memory and the bf16 parameters ending there, two ways:
    - pipelined copies: per step, H2D of every rank's gradients, the step, D2H of
      the full bf16 parameter buffer, which the engine pipelines over streams
      bucket by bucket (copies in for bucket b+1 and out for bucket b-1 while
      bucket b's step runs);
    - host-resident: the direct step over a plan whose gradient pointers are the
      pinned host tensors, writing the parameters into the pinned host buffer;
      the kernels move both over the host link.
    The reported value is the faster; both are in the record."""
    import torch
    from zero_partition_aware_gb300 import workloads as W
    L = grp.layout
    try:
        host = [torch.empty(a.numel(), dtype=a.dtype, pin_memory=True) for a in arenas]
    except RuntimeError as e:
        return {"value": None, "unit": UNIT, "error": f"pinned host allocation failed: {e}"}
    for h, a in zip(host, arenas):
        h.copy_(a)
    out_host = torch.empty(L.P, dtype=torch.bfloat16, pin_memory=True)
    # each bucket's params are contiguous in every rank's arena
    offs = W.arena_offsets(wl.numel, 256)
    lo = [None] * L.n_buckets
    hi = [0] * L.n_buckets
    for i, n in enumerate(wl.numel):
        b = L.param(i)[1]
        lo[b] = offs[i] if lo[b] is None else lo[b]
        hi[b] = offs[i] + n
    h2d_pairs = [[(h[lo[b]:hi[b]], a[lo[b]:hi[b]]) for h, a in zip(host, arenas)] for b in range(L.n_buckets)]
    h2d = sum(hs.numel() * hs.element_size() for pairs in h2d_pairs for hs, _ in pairs)  # the bytes copied
    d2h = out_host.numel() * out_host.element_size()
    cs, ds = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_step():
        grp.step_direct_from_host(dplan, hp, h2d_pairs, out_host, stream=stream, copy_stream=cs, d2h_stream=ds)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    k = max(2, min(args.steps, 5))
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    s.record(stream)
    for _ in range(k):
        e2e_step()
    e.record(stream)
    torch.cuda.synchronize()
    ms = dist.max(s.elapsed_time(e) / k)
    # the floor: the same host-to-device copies alone, on the copy stream
    cs.wait_stream(stream)
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record(cs)
    for _ in range(k):
        with torch.cuda.stream(cs):
            for pairs in h2d_pairs:
                for hs, dv in pairs:
                    dv.copy_(hs, non_blocking=True)
    e2.record(cs)
    torch.cuda.synchronize()
    ms_h2d = dist.max(s2.elapsed_time(e2) / k)
    # the parameter read-back alone, then both directions' copies at once (no compute)
    param = grp.param[: L.P]
    ds.wait_stream(stream)
    s3, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s3.record(ds)
    with torch.cuda.stream(ds):
        for _ in range(k):
            out_host.copy_(param, non_blocking=True)
    e3.record(ds)
    torch.cuda.synchronize()
    ms_d2h = dist.max(s3.elapsed_time(e3) / k)
    s4, e4 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s4.record(stream)
    cs.wait_stream(stream)
    ds.wait_stream(stream)
    for _ in range(k):
        with torch.cuda.stream(cs):
            for pairs in h2d_pairs:
                for hs, dv in pairs:
                    dv.copy_(hs, non_blocking=True)
        with torch.cuda.stream(ds):
            out_host.copy_(param, non_blocking=True)
    stream.wait_stream(cs)
    stream.wait_stream(ds)
    e4.record(stream)
    torch.cuda.synchronize()
    ms_both = dist.max(s4.elapsed_time(e4) / k)
    pipelined = {"ms_per_step": round(ms, 3), "params_per_s": round(nranks * L.T / (ms / 1e3)),
                 "h2d_only_ms_per_step": round(ms_h2d, 3), "h2d_only_GB_per_s": round(h2d / (ms_h2d / 1e3) / 1e9, 1),
                 "d2h_only_ms_per_step": round(ms_d2h, 3), "d2h_only_GB_per_s": round(d2h / (ms_d2h / 1e3) / 1e9, 1),
                 "copies_only_ms_per_step": round(ms_both, 3),
                 "how": "per bucket: H2D of its gradients, zr_step_direct, D2H of its bf16 params, on 3 streams"}
    # host-resident gradients: a direct plan over the pinned host tensors themselves;
    # the kernels read the gradients and write the bf16 params in place over the host link
    host_plan = grp.direct_plan(grp.grad_table([[h[o:o + n] for o, n in zip(offs, wl.numel)] for h in host]))

    def zc_step():
        grp.step_direct(host_plan, hp, stream=stream, param_out=out_host)

    for _ in range(2):
        zc_step()
    torch.cuda.synchronize()
    s5, e5 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    s5.record(stream)
    for _ in range(k):
        zc_step()
    e5.record(stream)
    torch.cuda.synchronize()
    ms_zc = dist.max(s5.elapsed_time(e5) / k)
    del host_plan, host
    zero_copy = {"ms_per_step": round(ms_zc, 3), "params_per_s": round(nranks * L.T / (ms_zc / 1e3)),
                 "how": "one zr_step_direct_range call over a direct plan whose gradient pointers are the pinned "
                        "host tensors, the bf16 params written to the pinned host buffer: the kernels move both "
                        "over the host link, no copy"}
    best = min(ms, ms_zc)
    return {"value": round(nranks * L.T / (best / 1e3)), "unit": UNIT, "ms_per_step": round(best, 3),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": k,
            "path": "host_resident" if ms_zc <= ms else "pipelined_copies",
            "host_resident": zero_copy, "pipelined_copies": pipelined}


# ----------------------------------------------------------------------------
# the CPU oracle (cpu_baseline leg and --impl reference)
# ----------------------------------------------------------------------------

def oracle_sample(wl, n_elems, seed=0, skip_larger=False):
    """A bounded sample of the workload on the host: the first bucket's leading
    params (at most n_elems elements; with skip_larger, params of more than
    n_elems elements are passed over) with their state, drawn on the CPU."""
    import torch
    import oracle
    from zero_partition_aware_gb300 import workloads as W
    numel = []
    tot = 0
    for n in wl.numel:
        if skip_larger and n > n_elems:
            continue
        if tot + n > n_elems and numel:
            break
        numel.append(int(n))
        tot += int(n)
    sub = W.replace(wl, numel=tuple(numel))
    lay = oracle.layout(numel, wl.world, wl.bucket)
    inp = W.draw_inputs(sub, "cpu", seed=seed)
    if wl.micro_steps > 1:  # the micro-steps' flat bf16 grads, accumulated inside the timed step
        grads = [[W.bf16_bits(g) for g in inp["grads"][k]] for k in range(wl.world)]
    else:
        grads = [oracle.params_from_flat(lay, W.bf16_bits(inp["grads"][k][0])) for k in range(wl.world)]
    p = oracle.shards_from_flat(lay, inp["master"].numpy())
    m = oracle.shards_from_flat(lay, inp["m"].numpy())
    v = oracle.shards_from_flat(lay, inp["v"].numpy())
    return lay, grads, p, m, v


def oracle_step(lay, grads, p, m, v, hp, scale, micro=False):
    import oracle
    param = np.zeros(lay.P, np.uint16)
    if micro:  # every micro-step into an fp32 main_grad per rank, then its buckets
        mains = []
        for row in grads:
            acc = np.zeros(lay.T, np.float32)
            for g in row:
                oracle.grad_accumulate(acc, g)
            mains.append(oracle.params_from_flat(lay, acc))
        grads = mains
    for b in range(lay.n_buckets):
        bucket = oracle.bucket_pack(lay, b, grads)
        oracle.rs_adam_fused(lay, b, bucket, scale, p, m, v, hp, param)
    return param


def cpu_baseline(wl, budget_s):
    """Time the oracle as it stands, single-threaded, on a bounded sample: the
    leading params of the workload (up to one bucket), re-run until about
    budget_s seconds of CPU work have been timed."""
    import oracle
    oracle.build()
    scale = float(np.float32(1.0 / wl.world))
    lay, grads, p, m, v = oracle_sample(wl, min(wl.bucket, 1 << 24))
    reps, dt = 0, 0.0
    while dt < budget_s and reps < 1000:
        t0 = time.perf_counter()
        oracle_step(lay, grads, p, m, v, wl.adam, scale, micro=wl.micro_steps > 1)
        dt += time.perf_counter() - t0
        reps += 1
    return {"value": round(reps * lay.T / dt), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"first {lay.n_params} params ({lay.T} elements) of {wl.name}, world {wl.world}: "
                      + (f"{wl.micro_steps} micro-step accumulations + " if wl.micro_steps > 1 else "")
                      + f"pack + fused step run {reps} times, {dt:.1f} s single-threaded",
            "seconds": round(dt, 2)}


def cpu_baseline_all_cores(wl, budget_s):
    """The oracle as it stands on every host core: one thread per core, each
    with its own copy of one bounded sample (leading params of at most
    2^24 / threads elements, or of the first bucket up to 2^20 if that is more;
    larger params passed over) and its own state,
    re-running pack + fused step over the same wall-clock window. The oracle
    is C called through ctypes, which releases the GIL for each call, so the
    threads run in parallel; no process is forked. Throughput = elements of
    all completed steps / the window."""
    import threading
    import oracle
    oracle.build()
    n_thr = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    scale = float(np.float32(1.0 / wl.world))
    cap = max(min(wl.bucket, 1 << 24) // n_thr, min(wl.bucket, 1 << 20))
    lay, grads, p, m, v = oracle_sample(wl, cap, skip_larger=True)
    copy = lambda x: [copy(y) for y in x] if isinstance(x, list) else x.copy()
    work = [(copy(grads), copy(p), copy(m), copy(v)) for _ in range(n_thr)]
    done = [0] * n_thr
    go = threading.Barrier(n_thr + 1)
    t_end = [0.0]

    def run(i):
        g, pp, mm, vv = work[i]
        go.wait()
        while time.perf_counter() < t_end[0]:
            oracle_step(lay, g, pp, mm, vv, wl.adam, scale, micro=wl.micro_steps > 1)
            done[i] += 1

    ths = [threading.Thread(target=run, args=(i,)) for i in range(n_thr)]
    for t in ths:
        t.start()
    t0 = time.perf_counter()
    t_end[0] = t0 + budget_s
    go.wait()
    for t in ths:
        t.join()
    dt = time.perf_counter() - t0
    return {"value": round(sum(done) * lay.T / dt), "unit": UNIT, "cores": n_thr, "kind": "oracle",
            "sample": f"{n_thr} threads, each its own copy of {lay.n_params} params ({lay.T} elements) of "
                      f"{wl.name} (leading params of at most {cap} elements), "
                      f"world {wl.world}: "
                      + (f"{wl.micro_steps} micro-step accumulations + " if wl.micro_steps > 1 else "")
                      + f"pack + fused step, {sum(done)} steps completed in {dt:.1f} s",
            "seconds": round(dt, 2)}


def run_reference(args):
    from zero_partition_aware_gb300 import workloads as W
    import oracle
    wl = W_lookup(args)
    oracle.build()
    scale = float(np.float32(1.0 / wl.world))
    # each step: a bounded sample (~2 s of single-threaded oracle work)
    lay, grads, p, m, v = oracle_sample(wl, 200_000)
    t0 = time.perf_counter()
    oracle_step(lay, grads, p, m, v, wl.adam, scale, micro=wl.micro_steps > 1)
    rate = lay.T / max(time.perf_counter() - t0, 1e-6)
    per_step = max(2.0, min(8.0, 150.0 / max(args.steps + args.warmup, 1)))
    lay, grads, p, m, v = oracle_sample(wl, int(min(max(rate * per_step, 200_000), 1 << 24)))
    for _ in range(args.warmup):
        oracle_step(lay, grads, p, m, v, wl.adam, scale, micro=wl.micro_steps > 1)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(lay, grads, p, m, v, wl.adam, scale, micro=wl.micro_steps > 1)
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    value = lay.T / dt
    sample = (f"first {lay.n_params} params ({lay.T} elements) of {wl.name}, world {wl.world}: "
              + (f"{wl.micro_steps} micro-step accumulations + " if wl.micro_steps > 1 else "")
              + "pack + fused step per timed step")
    return {"impl": "reference", "metric": METRIC, "value": round(value), "unit": UNIT, "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": wl.name, "params": lay.T, "world": wl.world,
                       "reduce_bucket_size": wl.bucket, "sample_of_params": wl.total},
            "cpu_baseline": {"value": round(value), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank, nranks, local = dist_env()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0
    from zero_partition_aware_gb300 import build
    dist = Dist(nranks)
    if rank == 0:
        build.build()
    dist.barrier()
    out = (run_gpu_micro if W_lookup(args).micro_steps > 1 else run_gpu)(args, rank, nranks, local, dist)
    if rank == 0:
        if nranks == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(W_lookup(args), args.cpu_seconds)
            out["cpu_baseline_all_cores"] = cpu_baseline_all_cores(W_lookup(args), args.cpu_seconds / 2)
        print(json.dumps(out), flush=True)
    dist.close()
    return 0


def W_lookup(args):
    """The workload named by --workload, with --world applied."""
    from zero_partition_aware_gb300 import workloads as W
    wl = W.WORKLOADS[args.workload]
    if args.world:
        wl = W.replace(wl, world=args.world)
    if args.bucket:
        wl = W.replace(wl, bucket=args.bucket)
    return wl


if __name__ == "__main__":
    sys.exit(main())

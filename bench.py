"""Benchmark of the FIFO data plane on one GB300 (replicas on N GPUs).

Timed step: one SIMPLE transfer of 1 GiB of bf16 N(0,1) values (seed 2)
through 16 channels, each a FIFO of 8 slots x 512 KiB in HBM.  `value` is
payload GB/s (whole job: all ranks' bytes / max-over-ranks time), with the
input resident in HBM.  The same JSON line carries the roofline of the
transfer kernel, an end-to-end figure through the C ABI with host buffers,
the CPU oracle's rate on a bounded sample of the same workload, and the other
rows of the data plane (zero copy, LL latency and size sweep, host-placed
FIFO against the concurrent pinned-memcpy ceiling, virtual ring allreduce).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

`--impl reference` times the CPU oracle (the slow, single-threaded protocol
simulation) on the same workload and metric, a bounded sample per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import re
import shutil
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "FIFO transfer GB/s and % of HBM roofline (SIMPLE, 1 GPU); LL 8 B latency µs"
GIB = 1 << 30
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["xp_p2p_tma.cu", "xp_device.cuh", "xp_internal.h"]


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(sources=KERNEL_SOURCES, root: str = ROOT) -> str:
    """Hash of a kernel's sources with comments and whitespace removed, so that
    only a change of code makes a committed ncu capture stale."""
    h = hashlib.sha256()
    for f in sources:
        src = open(os.path.join(root, "collective_transport_plane_gb300", "csrc", f)).read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(name: str = "p2p_tma_simple_1GiB_16ch", root: str = ROOT, field: str = "traffic_bytes_per_launch"):
    """DRAM bytes (per launch, or another field of the record) of a kernel
    from its committed ncu record (profiles/<name>.json), if the kernel's
    sources have not changed since it was captured; else None."""
    try:
        rec = json.load(open(os.path.join(root, "profiles", name + ".json")))
        current = kernel_source_hash(rec.get("sources", KERNEL_SOURCES), root)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_hash") != current or field not in rec:
        return None
    return int(rec[field])


def time_stats(ms_list):
    """Mean, best and median of per-launch times (ms)."""
    return {"ms_mean": statistics.mean(ms_list), "ms_best": min(ms_list), "ms_median": statistics.median(ms_list)}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        self.index = index
        if shutil.which("nvidia-smi"):
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(ms: float) -> float:
    """The slowest rank's time (replicas run in lock step between barriers)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, nbytes: int, steps: int, total_ms: float) -> float:
    """Payload of every rank's steps over the slowest rank's time, in GB/s."""
    return world * nbytes * steps / (total_ms * 1e-3) / 1e9


def time_events(torch, stream, fn, iters):
    """Per-iteration device times (ms) with CUDA events on `stream`."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    for a, b in evs:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


class OneCore:
    """Runs the enclosed code on one host core (the oracle is a
    single-threaded program); describes the host for the JSON line."""

    def __enter__(self):
        self.saved = os.sched_getaffinity(0) if hasattr(os, "sched_getaffinity") else None
        if self.saved:
            os.sched_setaffinity(0, {min(self.saved)})
        return self

    def __exit__(self, *exc):
        if self.saved:
            os.sched_setaffinity(0, self.saved)
        return False

    @staticmethod
    def host():
        return f"pinned to 1 of {os.cpu_count()} {platform.machine()} host cores"


def cpu_oracle_rate(budget_s: float):
    """The oracle on the 1 GiB multi-channel workload: whole channels (64 MiB
    each) in order until the budget is used; returns (GB/s, sample text)."""
    import oracle
    w = workloads.SIMPLE_MULTI
    src = workloads.normal_bf16_bits(w["nelems"], w["seed"]).view(np.uint8)
    per = len(src) // w["nchannels"]
    with OneCore():
        t0 = time.perf_counter()
        moved, nch = 0, 0
        while time.perf_counter() - t0 < budget_s and nch < 4096:
            c = nch % w["nchannels"]
            piece = src[c * per:(c + 1) * per]
            dst, _, _ = oracle.simple_transfer(piece, 1, w["nslots"], w["slot_bytes"], seed=nch)
            if not np.array_equal(dst, piece):
                raise RuntimeError("oracle transfer mismatch")
            moved += len(piece)
            nch += 1
        dt = time.perf_counter() - t0
    return moved / dt / 1e9, (f"{nch} channel(s) x 64 MiB of the 1 GiB bf16 workload, 8 x 512 KiB slots, "
                              f"slot-granular seeded interleaving ({dt:.1f} s, {OneCore.host()})")


def reference_arm(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    w = workloads.SIMPLE_MULTI
    src = workloads.normal_bf16_bits(w["nelems"], w["seed"]).view(np.uint8)
    per = len(src) // w["nchannels"]
    pin = OneCore().__enter__()
    # calibrate one channel, then size each step to fit ~90 s overall
    t0 = time.perf_counter()
    oracle.simple_transfer(src[:per // 8], 1, w["nslots"], w["slot_bytes"], seed=0)
    rate = (per // 8) / (time.perf_counter() - t0)
    budget = 90.0 / max(1, args.steps + args.warmup)
    nbytes = int(min(len(src), max(w["slot_bytes"], rate * budget)) // w["slot_bytes"] * w["slot_bytes"])
    sample = src[:nbytes]
    for i in range(args.warmup):
        oracle.simple_transfer(sample, w["nchannels"], w["nslots"], w["slot_bytes"], seed=i)
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        dst, _, _ = oracle.simple_transfer(sample, w["nchannels"], w["nslots"], w["slot_bytes"], seed=1000 + i)
        times.append(time.perf_counter() - t0)
        if not np.array_equal(dst, sample):
            raise RuntimeError("oracle transfer mismatch")
    pin.__exit__(None, None, None)
    t = sum(times)
    value = nbytes * args.steps / t / 1e9
    desc = (f"first {nbytes} bytes of the 1 GiB bf16 workload per step, 16 channels of 8 x 512 KiB, "
            f"slot-granular seeded interleaving, {OneCore.host()}")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {"workload": "SIMPLE multi-channel 1 GiB bf16, 16 channels x 8 slots x 512 KiB (CPU oracle sample)",
                   "nchannels": 16, "nslots": 8, "slot_bytes": 512 << 10},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--lanes", type=int, default=9, help="sender CTAs per channel")
    ap.add_argument("--rlanes", type=int, default=10, help="receiver CTAs per channel")
    ap.add_argument("--no-rows", action="store_true", help="time the step only")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--mib", type=int, default=0,
                    help="profiling only: move the first MiB of the workload instead of 1 GiB")
    ap.add_argument("--rows", default="",
                    help="profiling only: run just these comma-separated row groups (" + ",".join(ROW_GROUPS) +
                         ") after the step, without the end-to-end and CPU legs")
    ap.add_argument("--mode", default="simple", choices=["simple", "zero_copy", "posted_copy", "posted_direct", "ll128"],
                    help="profiling only: the transfer the timed step runs (the headline is simple)")
    ap.add_argument("--ring-mib", type=int, default=0,
                    help="profiling only: MiB per rank of the ring row instead of 256")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        return reference_arm(args)

    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    from collective_transport_plane_gb300 import build
    if rank == 0:
        build.build()
    if world > 1:
        dist.barrier()
    import collective_transport_plane_gb300.xp as xp

    hbm_peak, peak_kind = peaks()
    w = workloads.SIMPLE_MULTI
    src_np = workloads.normal_bf16_bits((args.mib << 19) if args.mib else w["nelems"], w["seed"])
    nbytes = src_np.nbytes
    src = torch.from_numpy(src_np).to("cuda")
    dst = torch.empty_like(src)
    stream = torch.cuda.Stream()
    if args.mode == "ll128":
        fifo = xp.xp_fifo_create(w["nchannels"], w["nslots"], w["slot_bytes"], xp.XP_PROTO_LL128)
        xp.xp_fifo_set_lanes(fifo, min(args.lanes, 8))
        xp.xp_fifo_set_recv_lanes(fifo, min(args.rlanes, 8))
    else:
        fifo = xp.xp_fifo_create(w["nchannels"], w["nslots"], w["slot_bytes"])
        xp.xp_fifo_set_lanes(fifo, args.lanes)
        xp.xp_fifo_set_recv_lanes(fifo, args.rlanes)

    if args.mode in ("simple", "ll128"):
        def step():
            xp.xp_send_recv(fifo, src, dst, nbytes, stream)
    elif args.mode == "zero_copy":
        def step():
            xp.xp_send_recv_zero_copy(fifo, src, dst, nbytes, stream)
    else:
        direct = args.mode == "posted_direct"

        def step():
            xp.xp_send_recv_posted(fifo, src, dst, nbytes, direct, stream)
    per_byte = {"zero_copy": 2, "posted_direct": 2, "ll128": 2 + 2 * 128 / 120}.get(args.mode, 4)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    st, rep = xp.xp_fifo_status(fifo, True)
    if st != xp.XP_OK:
        raise RuntimeError(f"warm-up transfer failed: status {st}")
    if not torch.equal(dst, src):
        raise RuntimeError("warm-up transfer is not byte-exact")

    # dst is poisoned before the timed region and compared after it, so the
    # check covers the timed transfers themselves
    dst.view(torch.uint8).fill_(0x7f)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    per = time_events(torch, stream, step, args.steps)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    st, rep = xp.xp_fifo_status(fifo, True)
    if st != xp.XP_OK:
        raise RuntimeError(f"timed transfer failed: status {st}")
    exact = bool(torch.equal(dst, src))
    if not exact:
        raise RuntimeError("timed transfers are not byte-exact")
    total_ms = max_over_ranks(sum(per))
    ms_step = total_ms / args.steps
    value = whole_job_gbs(world, nbytes, args.steps, total_ms)
    ts = time_stats(per)
    avg_launch_ms = ts["ms_mean"]
    achieved = per_byte * nbytes / (avg_launch_ms * 1e-3) / 1e9
    traffic = profiled_traffic() if args.mode == "simple" else None
    # the reachable floor of any transfer: src read once, dst written once
    copy_floor = 2 * nbytes / (avg_launch_ms * 1e-3) / 1e9

    out = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {"workload": "SIMPLE multi-channel: 1 GiB bf16 N(0,1) seed 2, 16 channels x 8 slots x 512 KiB, FIFO in HBM",
                   "nchannels": w["nchannels"], "nslots": w["nslots"], "slot_bytes": w["slot_bytes"],
                   "sender_ctas_per_channel": min(args.lanes, 8) if args.mode == "ll128" else args.lanes,
                   "receiver_ctas_per_channel": min(args.rlanes, 8) if args.mode == "ll128" else args.rlanes,
                   "payload_bytes": nbytes, "parallelism": f"replicas{world}",
                   "l2": "inputs (1 GiB) larger than L2; the 64 MiB FIFO itself is L2-resident by design"},
        "gpu_launches": args.steps,
        "ms_mean": ts["ms_mean"], "ms_best": ts["ms_best"], "ms_median": ts["ms_median"],
        "gbs_best": nbytes / (ts["ms_best"] * 1e-3) / 1e9, "gbs_median": nbytes / (ts["ms_median"] * 1e-3) / 1e9,
        "exact": exact,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": traffic,
                     "frac_copy_floor": copy_floor / hbm_peak,
                     "frac_dram": (traffic / (avg_launch_ms * 1e-3) / 1e9 / hbm_peak) if traffic else None,
                     "note": ("frac counts the algorithmic bytes of the path; the FIFO is L2-resident by design, "
                              "so it is an accounting, not a bound, and may exceed 1. frac_copy_floor counts "
                              "only the src read and dst write every transfer must make (2 bytes per payload "
                              "byte); frac_dram counts the DRAM bytes ncu measured for this kernel source"),
                     "peak_kind": f"{peak_kind} HBM copy (burst)",
                     "accounting": {4: "4 bytes per payload byte: src read, slot write, slot read, dst write",
                                    2: "2 bytes per payload byte: src read, dst write"}.get(
                                        per_byte, "2 + 2 x 128/120 bytes per payload byte: src read, dst write, "
                                                  "and 128-byte lines of 120 payload bytes written and read")},
        "clocks": clk,
    }

    if args.mib:
        out["config"]["workload"] += f" (profiling case: first {args.mib} MiB)"
    if args.mode != "simple":
        out["config"]["workload"] += f" (profiling case: {args.mode} transfer)"
    if rank == 0 and args.rows:
        out["rows"] = rows(torch, xp, hbm_peak, set(args.rows.split(",")), args.ring_mib)
    elif rank == 0 and not args.no_rows:
        out["e2e"] = e2e_row(torch, xp, fifo, src_np, stream)
        out["rows"] = rows(torch, xp, hbm_peak)
        rate, desc = cpu_oracle_rate(args.cpu_budget)
        out["cpu_baseline"] = {"value": rate, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc}
        out["ll_8B_latency_us"] = out["rows"]["ll"]["pingpong_one_way_us"]
    xp.xp_fifo_destroy(fifo)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def e2e_row(torch, xp, fifo, src_np, stream, iters=10, warmup=3, chunk=64 << 20):
    """Same transfer from pinned host memory to pinned host memory through the
    C ABI (xp_send_recv_staged): host -> device copies, the FIFO transfers and
    device -> host copies of 64 MiB chunks, overlapped on three streams, all
    inside the timed region."""
    n = src_np.nbytes
    h_src = torch.from_numpy(src_np).pin_memory()
    h_dst = torch.empty_like(h_src).pin_memory()
    d_src = torch.empty(h_src.shape, dtype=h_src.dtype, device="cuda")
    d_dst = torch.empty_like(d_src)

    def one():
        xp.xp_send_recv_staged(fifo, h_src, h_dst, d_src, d_dst, n, chunk, stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            one()
        torch.cuda.synchronize()
        t = time_events(torch, stream, one, iters)
    if not torch.equal(h_dst, h_src):
        raise RuntimeError("end-to-end transfer is not byte-exact")
    ms = sum(t) / iters
    return {"value": n / (ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": n, "d2h_bytes_per_step": n,
            "ms_per_step": ms, "ms_min": min(t), "ms_max": max(t), "steps": iters, "warmup": warmup,
            "api": "xp_send_recv_staged", "chunk_bytes": chunk}


ROW_GROUPS = ("hbm", "zero_copy", "simple_lanes1", "posted", "ce", "loopback", "ll", "ll128", "host_fifo", "ce_host",
              "ring")


def rows(torch, xp, hbm_peak, only=None, ring_mib=0):
    s = torch.cuda.Stream()
    res = {}

    def want(name):
        return only is None or name in only

    # HBM copy ceiling, re-measured in this run (read + write bytes)
    if want("hbm"):
        a = torch.empty(GIB // 2, dtype=torch.bfloat16, device="cuda")
        b = torch.empty_like(a)
        with torch.cuda.stream(s):
            t = time_events(torch, s, lambda: b.copy_(a), 10)
        res["hbm_copy_gbs_this_run"] = 2 * GIB / (min(t) * 1e-3) / 1e9
        del a, b

    w = workloads.SIMPLE_MULTI
    if want("zero_copy") or want("simple_lanes1") or want("posted") or want("ce"):
        src = torch.from_numpy(workloads.normal_bf16_bits(w["nelems"], w["seed"])).to("cuda")
        dst = torch.empty_like(src)
        n = src.numel() * 2

    if want("zero_copy"):
        # zero copy, 1 GiB through the same geometry
        zc = {}
        for lanes in (7, 8):
            f = xp.xp_fifo_create(w["nchannels"], w["nslots"], w["slot_bytes"])
            xp.xp_fifo_set_lanes(f, lanes)
            with torch.cuda.stream(s):
                for _ in range(5):
                    xp.xp_send_recv_zero_copy(f, src, dst, n, s)
                t = time_events(torch, s, lambda: xp.xp_send_recv_zero_copy(f, src, dst, n, s), 50)
            st, _ = xp.xp_fifo_status(f, True)
            ok = st == xp.XP_OK and torch.equal(dst, src)
            ms = statistics.median(t)
            zc[f"lanes{lanes}"] = {"gbs": n / (ms * 1e-3) / 1e9, "ms": ms, "ms_best": min(t), "ms_median": ms, "frac_of_hbm": 2 * n / (ms * 1e-3) / 1e9 / hbm_peak,
                                   "exact": bool(ok)}
            xp.xp_fifo_destroy(f)
        res["zero_copy"] = zc

    if want("simple_lanes1"):
        # SIMPLE with one sender CTA and one receiver CTA per channel (lanes 1)
        f = xp.xp_fifo_create(w["nchannels"], w["nslots"], w["slot_bytes"])
        with torch.cuda.stream(s):
            for _ in range(3):
                xp.xp_send_recv(f, src, dst, n, s)
            t = time_events(torch, s, lambda: xp.xp_send_recv(f, src, dst, n, s), 20)
        ms = statistics.median(t)
        res["simple_lanes1"] = {"gbs": n / (ms * 1e-3) / 1e9, "ms": ms, "ms_best": min(t), "ms_median": ms, "frac_of_hbm": 4 * n / (ms * 1e-3) / 1e9 / hbm_peak}
        xp.xp_fifo_destroy(f)

    if want("posted"):
        # receiver-driven credit (posts {addr, size, idx}): copy mode through the
        # staging slots (4 bytes of HBM traffic per payload byte) and direct
        # mode into dst (2 bytes per payload byte)
        posted = {}
        for direct, lanes, rl in ((False, 9, 9), (True, 6, None)):
            f = xp.xp_fifo_create(w["nchannels"], w["nslots"], w["slot_bytes"])
            xp.xp_fifo_set_lanes(f, lanes)
            if rl:
                xp.xp_fifo_set_recv_lanes(f, rl)
            dst.zero_()
            with torch.cuda.stream(s):
                for _ in range(5):
                    xp.xp_send_recv_posted(f, src, dst, n, direct, s)
                t = time_events(torch, s, lambda: xp.xp_send_recv_posted(f, src, dst, n, direct, s), 50)
            st, _ = xp.xp_fifo_status(f, True)
            ms = statistics.median(t)
            per = 2 if direct else 4
            posted["direct" if direct else "copy"] = {
                "lanes": lanes, "recv_lanes": rl or 1, "gbs": n / (ms * 1e-3) / 1e9, "ms": ms, "ms_best": min(t), "ms_median": ms,
                "frac_of_hbm": per * n / (ms * 1e-3) / 1e9 / hbm_peak, "exact": bool(st == xp.XP_OK and torch.equal(dst, src))}
            xp.xp_fifo_destroy(f)
        res["posted"] = posted
    if want("ce"):
        # proxy (copy-engine) mode, one hop: sender CTAs -> send ring, the
        # library's host pump copies every slot-step with cudaMemcpyAsync,
        # receiver CTAs drain the FIFO's slots.  Ceiling: one plain
        # cudaMemcpyAsync of the whole buffer, device to device.
        ce = {}
        for lanes in (2, 4):
            f = xp.xp_fifo_create(w["nchannels"], w["nslots"], w["slot_bytes"])
            xp.xp_fifo_set_lanes(f, lanes)
            xp.xp_fifo_enable_ce(f)
            dst.zero_()
            with torch.cuda.stream(s):
                for _ in range(3):
                    xp.xp_send_recv_ce(f, src, dst, n, s)
                t = time_events(torch, s, lambda: xp.xp_send_recv_ce(f, src, dst, n, s), 10)
            st, _ = xp.xp_fifo_status(f, True)
            ms = statistics.median(t)
            ce[f"lanes{lanes}"] = {"gbs": n / (ms * 1e-3) / 1e9, "ms": ms, "ms_best": min(t), "ms_median": ms,
                                   "exact": bool(st == xp.XP_OK and torch.equal(dst, src))}
            xp.xp_fifo_destroy(f)
        with torch.cuda.stream(s):
            t = time_events(torch, s, lambda: dst.copy_(src), 10)
        ceiling = n / (min(t) * 1e-3) / 1e9
        best = max(v["gbs"] for v in ce.values())
        res["ce_device"] = {"by_lanes": ce, "ceiling_one_memcpy_gbs": ceiling, "frac_of_ceiling": best / ceiling,
                            "slot_steps_per_op": n // w["slot_bytes"]}

    if want("zero_copy") or want("simple_lanes1") or want("posted") or want("ce"):
        del src, dst

    if want("loopback"):
        # SIMPLE loopback: 1 MiB, one sender CTA -> one receiver CTA, 8 x 64 KiB
        wl = workloads.SIMPLE_LOOPBACK
        src = torch.from_numpy(workloads.uniform_bytes(wl["nbytes"], wl["seed"])).to("cuda")
        dst = torch.empty_like(src)
        # (512 KiB of slots: by the FIFO's automatic choice its receivers do
        # not drop read lines from L2)
        f = xp.xp_fifo_create(1, wl["nslots"], wl["slot_bytes"])
        with torch.cuda.stream(s):
            for _ in range(10):
                xp.xp_send_recv(f, src, dst, wl["nbytes"], s)
            dst.zero_()
            t = time_events(torch, s, lambda: xp.xp_send_recv(f, src, dst, wl["nbytes"], s), 200)
            st, _ = xp.xp_fifo_status(f, True)
            ok = st == xp.XP_OK and torch.equal(dst, src)
            # device time of one transfer: the sender's start to the receiver's last head
            dev = []
            for _ in range(20):
                xp.xp_send_recv(f, src, dst, wl["nbytes"], s)
                s.synchronize()
                cs = xp.xp_fifo_stats(f, 0)
                dev.append((cs.t_end_ns - cs.t_start_ns) / 1e3)
        ms = statistics.median(t)
        res["simple_loopback_1MiB"] = {"us": ms * 1e3, "us_best": min(t) * 1e3, "us_median": ms * 1e3,
                                       "device_us_median": statistics.median(dev), "gbs": wl["nbytes"] / (ms * 1e-3) / 1e9,
                                       "line_drops": bool(xp.xp_fifo_describe(f, 0).discard), "exact": bool(ok)}
        xp.xp_fifo_destroy(f)

    if want("ll"):
        # LL: size sweep through one FIFO, and the device-side ping-pong
        wl = workloads.LL_SWEEP
        f = xp.xp_fifo_create(1, wl["nslots"], wl["slot_bytes"], xp.XP_PROTO_LL)
        sweep, best = {}, {}
        for size in wl["sizes"]:
            words = torch.from_numpy(workloads.uniform_u32(size // 4, wl["seed"])).to("cuda")
            out_t = torch.empty_like(words)
            with torch.cuda.stream(s):
                for _ in range(10):
                    xp.xp_send_recv(f, words, out_t, size, s)
                t = time_events(torch, s, lambda: xp.xp_send_recv(f, words, out_t, size, s), 100)
            sweep[str(size)] = statistics.median(t) * 1e3
            best[str(size)] = min(t) * 1e3
        st, _ = xp.xp_fifo_status(f, True)
        ab = xp.xp_fifo_create(1, wl["nslots"], wl["slot_bytes"], xp.XP_PROTO_LL)
        ns = xp.xp_ll_pingpong(f, ab, 20000, s)
        xp.xp_fifo_destroy(ab)
        xp.xp_fifo_destroy(f)
        sizes = np.array(wl["sizes"], float)
        us = np.array([sweep[str(x)] for x in wl["sizes"]])
        beta, alpha = np.polyfit(sizes, us, 1)          # us = alpha + beta * bytes
        res["ll"] = {"us_per_message_with_launch": sweep, "us_best_with_launch": best, "pingpong_one_way_us": ns / 2 / 20000 / 1e3,
                     "alpha_us": float(alpha), "beta_gbs": float(1e-3 / beta) if beta > 0 else None, "status": st}

    if want("ll128"):
        # LL128 (128-byte lines: 120 payload bytes and a flag word): the LL size
        # sweep through one FIFO of 8 x 32 KiB of lines, and 1 GiB through
        # 16 channels of 8 x 512 KiB (HBM bytes per payload byte: src read
        # and dst write, plus 128/120 for each of the slot write and read)
        wl = workloads.LL_SWEEP
        f = xp.xp_fifo_create(1, wl["nslots"], wl["slot_bytes"], xp.XP_PROTO_LL128)
        sweep = {}
        for size in wl["sizes"]:
            words = torch.from_numpy(workloads.uniform_u32(size // 4, wl["seed"])).to("cuda")
            out_t = torch.empty_like(words)
            with torch.cuda.stream(s):
                for _ in range(10):
                    xp.xp_send_recv(f, words, out_t, size, s)
                t = time_events(torch, s, lambda: xp.xp_send_recv(f, words, out_t, size, s), 100)
            sweep[str(size)] = statistics.median(t) * 1e3
        st, _ = xp.xp_fifo_status(f, True)
        xp.xp_fifo_destroy(f)
        src = torch.from_numpy(workloads.normal_bf16_bits(w["nelems"], w["seed"])).to("cuda")
        dst = torch.empty_like(src)
        n = src.numel() * 2
        multi = {}
        # sender:receiver CTAs per channel; 4:5 fills 144 of the 152 SMs (the
        # receivers are the slower side)
        for lanes, rlanes in ((1, 1), (2, 2), (4, 4), (4, 5)):
            f = xp.xp_fifo_create(w["nchannels"], w["nslots"], w["slot_bytes"], xp.XP_PROTO_LL128)
            xp.xp_fifo_set_lanes(f, lanes)
            xp.xp_fifo_set_recv_lanes(f, rlanes)
            dst.zero_()
            with torch.cuda.stream(s):
                for _ in range(3):
                    xp.xp_send_recv(f, src, dst, n, s)
                t = time_events(torch, s, lambda: xp.xp_send_recv(f, src, dst, n, s), 10)
            st2, _ = xp.xp_fifo_status(f, True)
            ms = statistics.median(t)
            multi[f"lanes{lanes}" if lanes == rlanes else f"lanes{lanes}_recv{rlanes}"] = {
                                      "gbs": n / (ms * 1e-3) / 1e9, "ms": ms, "ms_best": min(t), "ms_median": ms,
                                      "frac_of_hbm": (2 + 2 * 128 / 120) * n / (ms * 1e-3) / 1e9 / hbm_peak,
                                      "exact": bool(st2 == xp.XP_OK and torch.equal(dst, src))}
            if (lanes, rlanes) == (4, 5):
                # DRAM bytes of one launch from the committed ncu record of this configuration
                dram = profiled_traffic("ll128_1GiB_16ch")
                key = f"lanes{lanes}_recv{rlanes}"
                multi[key]["dram_bytes_per_launch_ncu"] = dram
                multi[key]["frac_dram"] = dram / (ms * 1e-3) / 1e9 / hbm_peak if dram else None
            xp.xp_fifo_destroy(f)
        res["ll128"] = {"us_per_message_with_launch": sweep, "sweep_status": st, "multi_1GiB_16ch": multi}
        del src, dst

    if want("host_fifo"):
        # host-placed FIFO: 256 MiB fp32, 8 channels x 8 x 1 MiB in pinned host memory
        wh = workloads.HOST_FIFO
        src = torch.from_numpy(workloads.uniform_f32(wh["nelems"], wh["seed"])).to("cuda")
        dst = torch.empty_like(src)
        n = src.numel() * 4
        host = {}
        for lanes in (1, 2, 4):
            f = xp.xp_fifo_create(wh["nchannels"], wh["nslots"], wh["slot_bytes"], xp.XP_PROTO_SIMPLE,
                                  xp.XP_PLACE_HOST_MAPPED)
            xp.xp_fifo_set_lanes(f, lanes)
            with torch.cuda.stream(s):
                for _ in range(3):
                    xp.xp_send_recv(f, src, dst, n, s)
                t = time_events(torch, s, lambda: xp.xp_send_recv(f, src, dst, n, s), 10)
            st, _ = xp.xp_fifo_status(f, True)
            ms = statistics.median(t)
            host[f"lanes{lanes}"] = {"gbs": n / (ms * 1e-3) / 1e9, "ms": ms, "ms_best": min(t), "ms_median": ms, "exact": bool(st == 0 and torch.equal(dst, src))}
            xp.xp_fifo_destroy(f)
        # ceiling: concurrent pinned cudaMemcpyAsync D2H || H2D of the same size
        hp = torch.empty(n, dtype=torch.uint8).pin_memory()
        hq = torch.empty(n, dtype=torch.uint8).pin_memory()
        d1 = torch.empty(n, dtype=torch.uint8, device="cuda")
        d2 = torch.empty(n, dtype=torch.uint8, device="cuda")
        s2 = torch.cuda.Stream()
        best = 1e30
        for i in range(6):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            s2.wait_event(e0)
            with torch.cuda.stream(s):
                d1.copy_(hp, non_blocking=True)
            with torch.cuda.stream(s2):
                hq.copy_(d2, non_blocking=True)
            s.wait_stream(s2)
            e1.record(s)
            torch.cuda.synchronize()
            if i >= 1:
                best = min(best, e0.elapsed_time(e1))
        ceiling = n / (best * 1e-3) / 1e9
        top = max(v["gbs"] for v in host.values())
        res["host_fifo"] = {"by_lanes": host, "ceiling_concurrent_memcpy_gbs": ceiling, "frac_of_ceiling": top / ceiling}
        del hp, hq, d1, d2

    if want("ce_host"):
        wh = workloads.HOST_FIFO
        if not want("host_fifo"):
            src = torch.from_numpy(workloads.uniform_f32(wh["nelems"], wh["seed"])).to("cuda")
            dst = torch.empty_like(src)
            n = src.numel() * 4
            ceiling = None
        # the same FIFO in proxy mode (shm useMemcpy style): the pump's copy
        # engines move each slot-step device -> host FIFO -> device
        f = xp.xp_fifo_create(wh["nchannels"], wh["nslots"], wh["slot_bytes"], xp.XP_PROTO_SIMPLE,
                              xp.XP_PLACE_HOST_MAPPED)
        xp.xp_fifo_set_lanes(f, 2)
        xp.xp_fifo_enable_ce(f)
        dst.zero_()
        with torch.cuda.stream(s):
            for _ in range(3):
                xp.xp_send_recv_ce(f, src, dst, n, s)
            t = time_events(torch, s, lambda: xp.xp_send_recv_ce(f, src, dst, n, s), 10)
        st, _ = xp.xp_fifo_status(f, True)
        ms = statistics.median(t)
        res["ce_host_2hops"] = {"gbs": n / (ms * 1e-3) / 1e9, "ms": ms, "ms_best": min(t), "ms_median": ms,
                                "frac_of_ceiling": n / (ms * 1e-3) / 1e9 / ceiling if ceiling else None,
                                "exact": bool(st == 0 and torch.equal(dst, src))}
        xp.xp_fifo_destroy(f)

    if want("host_fifo") or want("ce_host"):
        del src, dst

    if want("ring"):
        # virtual ring allreduce: 8 ranks x 256 MiB fp32, 8 channels x 8 x 512 KiB
        wr = workloads.RING
        nel = (ring_mib << 18) if ring_mib else wr["nelems"]
        xs = [torch.from_numpy(x).to("cuda") for x in workloads.ring_inputs(wr["nranks"], nel, "f32", wr["seed_base"])]
        ys = [torch.empty_like(x) for x in xs]
        ring = {}
        # lanes 1: every channel in one launch; 0: the library's choice (channels
        # in groups of 2 whose live FIFO data stays in L2, 8 lanes, one
        # cooperative grid of 128 CTAs per group)
        for lanes in (1, 0):
            r = xp.xp_ring_create(wr["nranks"], wr["nchannels"], wr["nslots"], wr["slot_bytes"])
            try:
                xp.xp_ring_set_lanes(r, lanes)
                with torch.cuda.stream(s):
                    for _ in range(3):
                        xp.xp_ring_allreduce_virtual(r, xs, ys, nel, xp.XP_F32, s)
                    t = time_events(torch, s, lambda: xp.xp_ring_allreduce_virtual(r, xs, ys, nel, xp.XP_F32, s), 10)
            except xp.XpError as e:
                ring["lanes_auto" if lanes == 0 else f"lanes{lanes}"] = {"error": str(e)}
                xp.xp_ring_destroy(r)
                continue
            st, _ = xp.xp_ring_status(r, True)
            ms = statistics.median(t)
            n = nel * 4
            P = wr["nranks"]
            alg = (6 * P - 4) * n
            ideal = 2 * P * n   # every rank reads its input once and writes its output once
            ring["lanes_auto" if lanes == 0 else f"lanes{lanes}"] = {
                "ms": ms, "ms_best": min(t), "ms_median": ms, "algbw_gbs": n / (ms * 1e-3) / 1e9,
                "hbm_gbs": alg / (ms * 1e-3) / 1e9, "frac_of_hbm": alg / (ms * 1e-3) / 1e9 / hbm_peak,
                "frac_of_ideal_2Pn": ideal / (ms * 1e-3) / 1e9 / hbm_peak,
                "note": "frac_of_hbm counts the (6P-4)n bytes every slot write and read would move through DRAM; "
                        "FIFO lines that stay in L2 let it exceed 1, frac_of_ideal_2Pn is the bound",
                "ranks_agree": bool(all(torch.equal(ys[0], y) for y in ys[1:])), "status": st}
            if lanes == 0 and not ring_mib:
                # DRAM bytes of one op from the committed ncu record of this configuration
                dram = profiled_traffic("ring_tma_8ranks_f32", field="traffic_bytes_per_op")
                ring["lanes_auto"]["dram_bytes_per_op_ncu"] = dram
                ring["lanes_auto"]["frac_dram"] = dram / (ms * 1e-3) / 1e9 / hbm_peak if dram else None
            xp.xp_ring_destroy(r)
        res["ring_f32"] = ring

    return res


if __name__ == "__main__":
    sys.exit(main())

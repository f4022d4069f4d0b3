"""Benchmark: sparse-MLA NVFP4 decode step on GB300.

One step = the whole hot path on one batch: the NVFP4 cache write of the
step's new tokens (one per session), then the sparse MLA decode over the
paged pool (index resolution, gather, in-SMEM dequantization, QK^T and PV on
tcgen05, online softmax, split-K merge).  Workload: the long-context
configuration -- 64 sessions x 204,800 tokens (4.6 GB pool of 352-byte rows),
H = 64, top-k 2048 (1024 from the most recent 4096 positions, 1024 uniform
over the rest), page size 64 -- synthetic, seeded, built on the device.

Timing: W warm-up steps, then K steps, each bracketed by CUDA events on the
launching stream, with a 256 MiB write between steps to flush L2 (outside the
events); barrier + synchronize around the timed loop; max over ranks.
value = gathered-KV bytes of all ranks / max step time (GB/s).  The decode
kernel alone (the roofline's kernel) is timed in a second loop, with an
event the library records right after the decode kernel.  e2e repeats the
step through the library's host-buffer C-ABI entry point (kv4_host_pipe_step)
from pinned host buffers (inputs in, out/lse back, copies inside the timed
region).

--impl reference times the CPU oracle (single-threaded C++, the method's
plain definition) on a bounded sample of the same workload.
Multi-GPU: torchrun, one process per GPU, each rank its own 64 sessions
(independent requests; no collective on the data path): weak scaling.
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
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from bit_kv_cache_nvfp4_gb300 import workloads as wl  # noqa: E402

METRIC = ("sparse-MLA NVFP4 decode µs/step and gathered-KV GB/s "
          "(% of GB300 HBM peak)")
CONFIG_NAME = "long"
WORKLOAD_DESC = ("long-context sparse-MLA decode step: 64 sessions x 204,800 tokens, H=64, "
                 "top-k 2048 (1024 recent + 1024 uniform), page 64, NVFP4 352-B rows; "
                 "cache write of 64 new tokens + decode")
FLUSH_BYTES = 256 << 20


def algorithmic_bytes(w: wl.Workload, valid_keys: int) -> int:
    """Bytes a perfect decode must move: the selected rows, the index and
    page-table words, q, out and lse (one page-table word per key is an upper
    bound)."""
    n_q = w.B * w.Sq
    return valid_keys * 352 + n_q * w.K * 4 * 2 + n_q * w.H * (1152 + 1024 + 4)


def valid_key_count(w: wl.Workload) -> int:
    n = 0
    for b in range(w.B):
        for s in range(w.Sq):
            L_eff = int(w.seq_lens[b]) - (w.Sq - 1 - s)
            row = w.topk[b, s]
            n += int(((row >= 0) & (row < L_eff)).sum())
    return n


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


DECODE_SOURCES = ("bit_kv_cache_nvfp4_gb300/csrc/kv4_sparse_mla_decode.cu",
                  "bit_kv_cache_nvfp4_gb300/csrc/kv4_device.cuh")


def _code_only(text: str) -> str:
    """C++ source without comments and blank lines, each line stripped: a
    change to comments alone leaves the compiled kernel as it was."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.strip() for line in text.splitlines() if line.strip())


def decode_source_hash() -> str:
    """Hash of the decode kernel's code (comments excluded), which the
    committed DRAM-traffic capture records."""
    import hashlib
    h = hashlib.sha256()
    for rel in DECODE_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic_bytes(sessions: int):
    """DRAM bytes (read + write) per decode launch from the committed ncu
    summary, scaled from the captured session count to `sessions` (the
    traffic is per key row, so it grows in proportion); None when the
    summary is missing or was taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", "decode_long_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("source_hash") != decode_source_hash():
            return None
        return float(d["dram_bytes_per_launch"]) * sessions / float(d["sessions"])
    except Exception:
        return None


class ClockSampler:
    """SM clock and throttle reasons sampled every few ms during the timed
    region, read through NVML (libnvidia-ml, read-only queries) in a
    background thread; nvidia-smi is the fallback."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int, period_s: float = 0.002):
        self.index = device_index
        self.period = period_s
        self.samples = []        # (sm_mhz, max_mhz, reasons bitmask)
        self._stop = None
        self._thread = None
        self._nvml = None
        self._handle = None

    def _open_nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        handle = ctypes.c_void_p()
        bus = None
        try:
            props = torch.cuda.get_device_properties(self.index)
            bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
        except Exception:
            bus = None
        if bus is None or lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(handle)):
            if lib.nvmlDeviceGetHandleByIndex_v2(self.index, ctypes.byref(handle)) != 0:
                raise RuntimeError("no NVML handle")
        self._nvml, self._handle = lib, handle

    def _poll(self):
        import ctypes
        lib, h = self._nvml, self._handle
        clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            ok = (lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and
                  lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0)
            if lib.nvmlDeviceGetCurrentClocksThrottleReasons(h, ctypes.byref(rs)) != 0:
                rs.value = 0
            if ok:
                self.samples.append((clk.value, mx.value, rs.value))
            time.sleep(self.period)

    def __enter__(self):
        import threading
        try:
            self._open_nvml()
            self._stop = threading.Event()
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
        except Exception:
            self._thread = None
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
        if not self.samples:
            self._nvidia_smi_once()

    def _nvidia_smi_once(self):
        q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.sw_power_cap,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown")
        try:
            out = subprocess.run(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                  "--format=csv,noheader,nounits"], capture_output=True,
                                 text=True, timeout=20).stdout
            p = [x.strip() for x in out.strip().split(",")]
            bits = 0
            for flag, val in zip((0x4, 0x8, 0x20, 0x40), p[2:6]):
                if val.lower() == "active":
                    bits |= flag
            self.samples.append((float(p[0]), float(p[1]), bits))
            self.source = "nvidia-smi (after the timed region)"
        except Exception:
            pass

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [s[0] for s in self.samples]
        bits = 0
        for s in self.samples:
            bits |= s[2]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(s[1] for s in self.samples),
                "sm_mhz_min": min(sm), "reasons": [n for b, n in self.REASONS.items() if bits & b],
                "samples": len(sm), "source": getattr(self, "source", "nvml")}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_over_ranks(t_ms: float, nbytes: float, device=None):
    """(max step time over ranks, sum of bytes over ranks); the identity
    without an initialized process group."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(t_ms), float(nbytes)
    t = torch.tensor([float(t_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    b = torch.tensor([float(nbytes)], dtype=torch.float64, device=device)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), float(b.item())


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.machine()


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample
# ---------------------------------------------------------------------------
def oracle_sample(w: wl.Workload, requests, repeats: int = 1):
    """Time the oracle's step (cache write of the requests' new tokens +
    decode) on `requests`; returns (seconds per repeat, gathered bytes)."""
    import oracle
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    qids = [(b, s) for b in requests for s in range(w.Sq)]
    pt_c, pages, ns = wl.compact_pool_plan(w, qids)
    ids, cslots = wl.compact_pool_tokens(w, pages, qids)
    lat, rope = wl.token_rows(w, ids)
    pool = np.zeros((max(ns, 64), 352), dtype=np.uint8)
    oracle.quantize_write(bits(lat), bits(rope), cslots.numpy(), pool)
    q = bits(wl.queries(w))
    nl, nr, nslots = wl.newest_tokens(w)
    sel = torch.tensor([b * w.Sq + s for b in requests for s in range(w.Sq)])
    nl, nr = bits(nl[sel]), bits(nr[sel])
    # the new tokens go to scratch rows past the compact pool (same work, no overlap)
    scratch = np.zeros((len(sel), 352), dtype=np.uint8)
    new_slots = np.arange(len(sel), dtype=np.int64)
    per_req = [(np.ascontiguousarray(q[b:b + 1]), np.ascontiguousarray(pt_c[b:b + 1].numpy()),
                np.ascontiguousarray(w.topk[b:b + 1].numpy()),
                np.ascontiguousarray(w.seq_lens[b:b + 1].numpy())) for b in requests]
    t0 = time.perf_counter()
    for _ in range(repeats):
        oracle.quantize_write(nl, nr, new_slots, scratch)
        for qb, ptb, tb, lb in per_req:
            oracle.sparse_mla_decode(qb, pool, ptb, tb, lb, w.sm_scale)
    dt = (time.perf_counter() - t0) / repeats
    valid = 0
    for b in requests:
        for s in range(w.Sq):
            L_eff = int(w.seq_lens[b]) - (w.Sq - 1 - s)
            row = w.topk[b, s]
            valid += int(((row >= 0) & (row < L_eff)).sum())
    return dt, valid * 352


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = wl.make_workload(CONFIG_NAME, seed=0, sessions=args.sessions)
    reqs = list(range(4))                       # bounded per-step sample
    for _ in range(args.warmup):
        oracle_sample(w, reqs)
    times = []
    gathered = 0
    for _ in range(args.steps):
        dt, gathered = oracle_sample(w, reqs)
        times.append(dt)
    t = sum(times) / len(times)
    gbs = gathered / t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC, "sample": f"{len(reqs)} of {w.B} sessions per step"},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{len(reqs)} sessions (new-token write + decode) per step",
                         "cpu": cpu_model()},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def build_pool(w: wl.Workload, dev) -> torch.Tensor:
    import bit_kv_cache_nvfp4_gb300 as kv
    pool = torch.zeros((w.num_slots, 352), dtype=torch.uint8, device=dev)
    for lat, rope, slots in wl.iter_pool_chunks(w, chunk=1 << 18, device=dev):
        kv.quantize_write(lat, rope, slots, pool)
    torch.cuda.synchronize(dev)
    return pool


def run_gpu(args):
    import bit_kv_cache_nvfp4_gb300 as kv
    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device for the GPU arm")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    w = wl.make_workload(CONFIG_NAME, seed=rank, sessions=args.sessions)
    pool = build_pool(w, dev)
    q = wl.queries(w, dev)
    pt, topk, lens = w.page_table.to(dev), w.topk.to(dev), w.seq_lens.to(dev)
    new_lat, new_rope, new_slots = wl.newest_tokens(w, dev)
    splits, ws_bytes = kv.decode_plan(w.B, w.Sq, w.H, w.K, args.splits)
    out = torch.empty((w.B, w.Sq, w.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.Sq, w.H), dtype=torch.float32, device=dev)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        # the cache write of the step's new tokens, then the decode (one call;
        # the decode's prologue overlaps the write)
        kv.quantize_write_and_decode(new_lat, new_rope, new_slots, pool, q, pt, topk, lens,
                                     w.sm_scale, out=out, lse=lse, workspace=ws, dev_err=err,
                                     force_splits=args.splits)

    valid = valid_key_count(w)
    kv_bytes = valid * 352
    alg_bytes = algorithmic_bytes(w, valid)
    flops = 2.0 * w.H * valid * (576 + 512)
    # cache write + decode, + the merge kernel when the split-K partials go
    # through the workspace (a unit split in two merges inside its cluster)
    launches_per_step = 2 + (1 if ws_bytes > 0 else 0)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    assert int(err.item()) == 0, f"device error flags {int(err.item())}"

    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    # The step's kernels run back to back (the decode may start while the
    # cache write finishes), so no event sits between them.
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            flush.zero_()
            e0[i].record(stream)
            step()
            e1[i].record(stream)
        torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    step_ms = [a.elapsed_time(b) for a, b in zip(e0, e1)]
    t_ms = sum(step_ms) / len(step_ms)
    assert int(err.item()) == 0, f"device error flags {int(err.item())}"

    # The decode kernel alone (for the roofline): a second loop on the same
    # inputs, the library recording an event right after the decode kernel
    # (before a merge kernel, if any).
    d0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    d1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for e in d1:                 # create the events the library will record
        e.record(stream)
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        flush.zero_()
        d0[i].record(stream)
        kv.set_timing_event(d1[i])
        kv.sparse_mla_decode(q, pool, pt, topk, lens, w.sm_scale, out=out, lse=lse, workspace=ws,
                             dev_err=err, force_splits=args.splits)
    kv.set_timing_event(None)
    torch.cuda.synchronize(dev)
    dec_ms = [a.elapsed_time(b) for a, b in zip(d0, d1)]
    dec_ms_avg = sum(dec_ms) / len(dec_ms)
    assert int(err.item()) == 0, f"device error flags {int(err.item())}"

    max_ms, tot_bytes = reduce_over_ranks(t_ms, kv_bytes, dev if world > 1 else None)
    value = tot_bytes / (max_ms * 1e-3) / 1e9

    # end to end through the public API, host buffers in and out; whole job:
    # the slowest rank's step time, every rank's bytes
    e2e = run_e2e(kv, w, dev, pool, pt, flush, args)
    if world > 1:
        e2e_ms, e2e_bytes = reduce_over_ranks(e2e["ms_per_step"], kv_bytes, dev)
        e2e.update({"value": e2e_bytes / (e2e_ms * 1e-3) / 1e9, "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": e2e["h2d_bytes_per_step"] * world,
                    "d2h_bytes_per_step": e2e["d2h_bytes_per_step"] * world})
    cache_write = run_cache_write(kv, dev, flush, args)
    per_config = None
    if rank == 0 and not args.skip_per_config:
        per_config = run_per_config(kv, dev, flush, args, long_inputs=(w, pool))
    latent = fp8 = dcp = None
    if not args.skip_variants:
        scratch = run_scratch_path(kv, w, dev, pool, q, pt, topk, lens, flush, args)
        del pool
        torch.cuda.empty_cache()
        latent = run_latent_rows(kv, w, dev, q, pt, topk, lens, flush, err, args, valid)
        fp8 = run_fp8_rows(kv, w, dev, q, pt, topk, lens, flush, args)
        fp8.update(scratch)
        fp8["nvfp4_decode_us"] = dec_ms_avg * 1e3
        fp8["nvfp4_vs_scratch_path"] = fp8["scratch_path_us"] / (dec_ms_avg * 1e3)
        fp8["nvfp4_vs_fp8_rows"] = fp8["fp8_rows_decode_us"] / (dec_ms_avg * 1e3)
        if rank == 0:
            dcp = run_dcp(kv, w, dev, q, pt, topk, lens, flush)

    peak_gbs, peak_tflops, peak_kind = measured_peaks()
    achieved_gbs = alg_bytes / (dec_ms_avg * 1e-3) / 1e9
    achieved_tflops = flops / (dec_ms_avg * 1e-3) / 1e12
    # The bound is the resource whose ideal time is longer: at 64 heads a key
    # row carries 2*64*1088 flops for 352 bytes (~400 flop/B), above the
    # ridge point of the measured peaks, so the tensor pipe bounds the decode.
    t_hbm, t_tensor = alg_bytes / (peak_gbs * 1e9), flops / (peak_tflops * 1e12)
    if t_tensor >= t_hbm:
        roof = {"bound": "tensor", "achieved": achieved_tflops, "peak": peak_tflops,
                "unit": "TFLOP/s", "frac": achieved_tflops / peak_tflops}
    else:
        roof = {"bound": "hbm", "achieved": achieved_gbs, "peak": peak_gbs, "unit": "GB/s",
                "frac": achieved_gbs / peak_gbs}
    roof.update({
        "traffic": ncu_traffic_bytes(w.B),
        "peak_source": (f"{peak_kind}: MEASURED_PEAKS.json bf16_tflops (burst; f16 operands run "
                        f"at the bf16 rate) and hbm_gbs") if peak_kind == "measured"
                       else "fallback: 1900 TFLOP/s bf16, 6800 GB/s",
        "kernel": "decode_kernel<64> (merge excluded)",
        "ideal_us": {"hbm": t_hbm * 1e6, "tensor": t_tensor * 1e6},
        "hbm": {"achieved": achieved_gbs, "peak": peak_gbs, "unit": "GB/s",
                "frac": achieved_gbs / peak_gbs},
        "tensor": {"achieved": achieved_tflops, "peak": peak_tflops, "unit": "TFLOP/s",
                   "frac": achieved_tflops / peak_tflops},
    })
    cpu = None
    if rank == 0 and not args.skip_cpu:
        reqs = list(range(min(w.B, args.cpu_sessions)))
        # repeat the sample until about 10 s of CPU work (at most 4 passes)
        runs = []
        while not runs or (sum(runs) < 10.0 and len(runs) < 4):
            dt, gathered = oracle_sample(w, reqs)
            runs.append(dt)
        dt = sum(runs) / len(runs)
        cpu = {"value": gathered / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{len(reqs)} of {w.B} sessions (new-token cache write + decode) x "
                         f"{len(runs)} passes, {sum(runs):.1f} s total", "cpu": cpu_model()}
    if world > 1:
        torch.distributed.barrier()
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": max_ms,
            "us_per_step": max_ms * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": WORKLOAD_DESC, "B": w.B, "Sq": w.Sq, "H": w.H, "K": w.K,
                       "seq_len": int(w.seq_lens[0]), "pool_bytes": w.num_slots * 352,
                       "splits": splits, "l2": "flushed between timed steps (256 MiB write)",
                       "parallelism": (f"{world} independent ranks (sessions sharded)" if world > 1
                                       else "1 GPU")},
            "kv_bytes_per_step": kv_bytes * world, "algorithmic_bytes_per_step": alg_bytes * world,
            "decode_kernel_us": dec_ms_avg * 1e3,
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "latent_rows_288B": latent,
            "fp8_comparison": fp8,
            "dcp": dcp,
            "cache_write_1M_tokens": cache_write,
            "per_config": per_config,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks.summary(),
            "wall_s_timed_loop": wall,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def _time_loop(fn, flush, stream, steps, warmup):
    """Average device time of fn() over `steps` calls, L2 flushed before each."""
    for _ in range(warmup):
        flush.zero_()
        fn()
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        e0[i].record(stream)
        fn()
        e1[i].record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in zip(e0, e1)) / steps


def graph_time_us(fn, flush, trials: int = 7, replays: int = 200):
    """Device time of one fn() call, in the timing form of the pages'
    graph-timed microbenchmarks: fn is captured in a CUDA graph and replayed
    `replays` times back to back between two events; the median over
    `trials` of the mean per replay.  Returns (cold, hot) microseconds: hot
    replays fn alone (its inputs stay in L2 from one replay to the next);
    cold replays [256 MiB L2 flush, fn] and subtracts the flush alone."""
    stream = torch.cuda.current_stream()

    def capture(body):
        for _ in range(2):                       # warm-up outside the capture
            body()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            body()
        return g

    def timed(g):
        meds = []
        for _ in range(trials):
            g.replay()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(replays):
                g.replay()
            b.record(stream)
            b.synchronize()
            meds.append(a.elapsed_time(b) * 1e3 / replays)
        return statistics.median(meds)

    def flushed():
        flush.zero_()
        fn()

    hot = timed(capture(fn))
    cold = timed(capture(flushed)) - timed(capture(flush.zero_))
    return cold, hot


PER_CONFIG_BOUND = {"tiny": "latency", "decode": "hbm ~ tensor", "long": "hbm ~ tensor (ridge)",
                    "specverify": "tensor", "splitk": "latency and SM fill"}


def run_per_config(kv, dev, flush, args, long_inputs=None):
    """Every configuration of the pages' workloads, each as one decode step
    (the cache write of the step's new tokens, then the decode), timed with
    CUDA-graph replays (cold and hot L2; graph_time_us), with the decode
    kernel alone, gathered-KV GB/s, both roofline fractions, and the oracle
    on one core on a bounded sample of the same workload."""
    peak_gbs, peak_tflops, _ = measured_peaks()
    res = {}
    for name in wl.CONFIG_NAMES:
        if name == "long" and long_inputs is not None:
            w, pool = long_inputs
        else:
            w = wl.make_workload(name, seed=0)
            pool = build_pool(w, dev)
        q = wl.queries(w, dev)
        pt, topk, lens = w.page_table.to(dev), w.topk.to(dev), w.seq_lens.to(dev)
        nl, nr, ns = wl.newest_tokens(w, dev)
        splits, ws_bytes = kv.decode_plan(w.B, w.Sq, w.H, w.K)
        out = torch.empty((w.B, w.Sq, w.H, 512), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((w.B, w.Sq, w.H), dtype=torch.float32, device=dev)
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)

        def step():
            kv.quantize_write_and_decode(nl, nr, ns, pool, q, pt, topk, lens, w.sm_scale,
                                         out=out, lse=lse, workspace=ws)

        def decode():
            kv.sparse_mla_decode(q, pool, pt, topk, lens, w.sm_scale, out=out, lse=lse,
                                 workspace=ws)

        step_cold, step_hot = graph_time_us(step, flush)
        dec_cold, dec_hot = graph_time_us(decode, flush)
        valid = valid_key_count(w)
        alg = algorithmic_bytes(w, valid)
        flops = 2.0 * w.H * valid * (576 + 512)
        t_hbm, t_tensor = alg / (peak_gbs * 1e3), flops / (peak_tflops * 1e6)   # us
        reqs = [0]
        runs = [oracle_sample(w, reqs)[0] for _ in range(3 if w.H * w.Sq <= 64 else 1)]
        o_s = statistics.median(runs)
        res[name] = {
            "B": w.B, "Sq": w.Sq, "H": w.H, "K": w.K, "splits": splits,
            "step_us_cold": step_cold, "step_us_hot": step_hot,
            "decode_us_cold": dec_cold, "decode_us_hot": dec_hot,
            "kv_gbs_cold": valid * 352 / (step_cold * 1e-6) / 1e9,
            "algorithmic_bytes": alg, "flops": flops,
            "bound_per_pages_table": PER_CONFIG_BOUND[name],
            "ideal_us": {"hbm": t_hbm, "tensor": t_tensor},
            "decode_hbm_frac": t_hbm / dec_cold, "decode_tensor_frac": t_tensor / dec_cold,
            "oracle_1core_ms_per_request": o_s * 1e3,
            "oracle_1core_ms_per_step_est": o_s * 1e3 * w.B,
        }
        del pool, q, pt, topk, lens, out, lse, ws
        torch.cuda.empty_cache()
    return res


def run_scratch_path(kv, w, dev, pool, q, pt, topk, lens, flush, args):
    """The comparison path of the README's kv4mla bullet: copy the selected
    NVFP4 rows into an FP8 scratch buffer in HBM (dequantize, cast to E4M3),
    then run the decode over the scratch rows."""
    scratch = kv.fp8_scratch(pool, pt, topk, lens)
    s_pt, s_topk, s_lens = kv.scratch_index(topk, lens)
    qs = q.reshape(w.B * w.Sq, 1, w.H, 576).contiguous()
    out = torch.empty((w.B * w.Sq, 1, w.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B * w.Sq, 1, w.H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def convert():
        kv.fp8_scratch(pool, pt, topk, lens, scratch=scratch)

    def path():
        convert()
        kv.sparse_mla_decode_fp8(qs, scratch, s_pt, s_topk, s_lens, w.sm_scale, out=out, lse=lse)

    t_conv = _time_loop(convert, flush, stream, args.steps, args.warmup)
    t_path = _time_loop(path, flush, stream, args.steps, args.warmup)
    return {"scratch_bytes": scratch.numel(), "scratch_convert_us": t_conv * 1e3,
            "scratch_path_us": t_path * 1e3}


def run_fp8_rows(kv, w, dev, q, pt, topk, lens, flush, args):
    """The decode over a pool of 576-byte FP8 rows (the row the NVFP4 row
    replaces), same workload and indices."""
    pool = torch.zeros((w.num_slots, 576), dtype=torch.uint8, device=dev)
    for lat, rope, slots in wl.iter_pool_chunks(w, chunk=1 << 18, device=dev):
        kv.quantize_write_fp8(lat, rope, slots, pool)
    out = torch.empty((w.B, w.Sq, w.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.Sq, w.H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    t = _time_loop(lambda: kv.sparse_mla_decode_fp8(q, pool, pt, topk, lens, w.sm_scale,
                                                    out=out, lse=lse),
                   flush, stream, args.steps, args.warmup)
    del pool
    torch.cuda.empty_cache()
    return {"fp8_pool_bytes": w.num_slots * 576, "fp8_rows_decode_us": t * 1e3,
            "note": "decode-only device times (cluster merge or merge kernel included); "
                    "scratch_path = scratch copy + FP8 decode over it"}


def run_cache_write(kv, dev, flush, args):
    """Throughput of the cache write alone on 1,048,576 tokens (N(0,1)
    latent and rope), with amax/6 scales and with MSE-searched scales.
    Bytes = the bf16 input read (1152 B) + the row written (352 B) per token."""
    n = 1 << 20
    lat, rope = wl.sweep_rows("normal", 0, 0, n, device=dev)
    slots = torch.arange(n, dtype=torch.int64, device=dev)
    pool = torch.empty((n, 352), dtype=torch.uint8, device=dev)
    res = {}
    for name, fn in (("amax", kv.quantize_write), ("mse", kv.quantize_write_mse)):
        for _ in range(3):
            fn(lat, rope, slots, pool)
        ts = []
        for _ in range(10):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn(lat, rope, slots, pool)
            b.record()
            b.synchronize()
            ts.append(a.elapsed_time(b))
        t = sorted(ts)[len(ts) // 2] * 1e-3
        res[name] = {"us": t * 1e6, "gbs": n * (1152 + 352) / t / 1e9}
    del lat, rope, slots, pool
    return res


def run_latent_rows(kv, w, dev, q, pt, topk, lens, flush, err, args, valid):
    """The same step on 288-byte latent-only rows (no rope; QK over the 512
    latent columns): cache write of the new tokens + decode, timed like the
    main step, and the decode kernel alone."""
    pool = torch.zeros((w.num_slots, 288), dtype=torch.uint8, device=dev)
    for lat, _rope, slots in wl.iter_pool_chunks(w, chunk=1 << 18, device=dev):
        kv.quantize_write_latent(lat, slots, pool)
    new_lat, _new_rope, new_slots = wl.newest_tokens(w, dev)
    q512 = q[..., :512].contiguous()
    splits, ws_bytes = kv.decode_plan_latent(w.B, w.Sq, w.H, w.K, args.splits)
    out = torch.empty((w.B, w.Sq, w.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.Sq, w.H), dtype=torch.float32, device=dev)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kv.quantize_write_latent(new_lat, new_slots, pool, err)
        kv.sparse_mla_decode_latent(q512, pool, pt, topk, lens, w.sm_scale, out=out, lse=lse,
                                    workspace=ws, dev_err=err, force_splits=args.splits)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        e0[i].record(stream)
        step()
        e1[i].record(stream)
    d0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    d1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for e in d1:
        e.record(stream)
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        flush.zero_()
        d0[i].record(stream)
        kv.set_timing_event(d1[i])
        kv.sparse_mla_decode_latent(q512, pool, pt, topk, lens, w.sm_scale, out=out, lse=lse,
                                    workspace=ws, dev_err=err, force_splits=args.splits)
    kv.set_timing_event(None)
    torch.cuda.synchronize(dev)
    assert int(err.item()) == 0, f"device error flags {int(err.item())}"
    t_ms = sum(a.elapsed_time(b) for a, b in zip(e0, e1)) / args.steps
    d_ms = sum(a.elapsed_time(b) for a, b in zip(d0, d1)) / args.steps
    n_q = w.B * w.Sq
    alg = valid * 288 + n_q * w.K * 4 * 2 + n_q * w.H * (1024 + 1024 + 4)
    flops = 2.0 * w.H * valid * (512 + 512)
    del pool
    return {"row_bytes": 288, "us_per_step": t_ms * 1e3,
            "kv_gbs": valid * 288 / (t_ms * 1e-3) / 1e9, "splits": splits,
            "decode_kernel_us": d_ms * 1e3,
            "decode_tflops": flops / (d_ms * 1e-3) / 1e12,
            "decode_algorithmic_gbs": alg / (d_ms * 1e-3) / 1e9,
            "note": "QK over the 512 latent columns, PV over the same 512; same workload"}


def run_dcp(kv, w, dev, q, pt, topk, lens, flush, worlds=(2, 8)):
    """Decode-context parallelism (README "Parallelism and disaggregation")
    on the long workload, its R ranks emulated one after another on this GPU,
    each with a pool of only its own pages and its page table over that pool
    (kept by the rank, as its pool is: built once here).  Per rank, one step
    is its top-k by page ownership and its fp32 partial decode; timed with
    CUDA-graph replays (cold L2) both with the masked full lists and with the
    rank's keys compacted to the front of its lists and a decode walking only
    those.  The log-sum-exp merge of the R partials is timed too.  The
    all-gather between ranks is not (one GPU)."""
    res = {}
    for R in worlds:
        o_parts = torch.empty((R, w.B, w.Sq, w.H, 512), dtype=torch.float32, device=dev)
        l_parts = torch.empty((R, w.B, w.Sq, w.H), dtype=torch.float32, device=dev)
        masked, compacted, pool_bytes = [], [], 0
        splits, wsb = kv.decode_plan(w.B, w.Sq, w.H, w.K)
        ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
        for r in range(R):
            n_pages = kv.dcp_local_pages(w.num_slots // 64, R, r)
            pool = torch.zeros((n_pages * 64, 352), dtype=torch.uint8, device=dev)
            for lat, rope, slots in wl.iter_pool_chunks(w, chunk=1 << 18, device=dev):
                kv.quantize_write(lat, rope, kv.dcp_local_slots(slots, R, r), pool)
            pool_bytes = max(pool_bytes, pool.numel())
            ptl = kv.dcp_local_page_table(pt, R, r)

            def step_masked(r=r, pool=pool, ptl=ptl):
                mine = kv.dcp_mask_topk(topk, pt, lens, R, r)
                kv.sparse_mla_decode_partial(q, pool, ptl, mine, lens, w.sm_scale,
                                             out=o_parts[r], lse=l_parts[r], workspace=ws)

            def step_compacted(r=r, pool=pool, ptl=ptl):
                mine, count = kv.dcp_compact_topk(topk, pt, lens, R, r)
                kv.sparse_mla_decode_partial(q, pool, ptl, mine, lens, w.sm_scale,
                                             out=o_parts[r], lse=l_parts[r], workspace=ws,
                                             k_count=count)

            masked.append(graph_time_us(step_masked, flush)[0])
            compacted.append(graph_time_us(step_compacted, flush)[0])
            del pool, ptl
            torch.cuda.empty_cache()
        merge_cold, _ = graph_time_us(lambda: kv.merge_partials(o_parts, l_parts), flush)
        res[f"R={R}"] = {
            "rank_step_us_max": {"masked": max(masked), "compacted": max(compacted)},
            "rank_step_us_mean": {"masked": sum(masked) / R, "compacted": sum(compacted) / R},
            "merge_us": merge_cold,
            "rank_pool_bytes": pool_bytes,
            "partials_bytes_per_rank": o_parts[0].numel() * 4 + l_parts[0].numel() * 4,
        }
        del o_parts, l_parts
    res["note"] = ("ranks emulated one after another on one GPU; cold-L2 graph replays; the "
                   "all-gather of the fp32 partials is not measured")
    return res


def run_e2e(kv, w, dev, pool, pt, flush, args, variants: int = 4):
    """The same step through the library's host-buffer C-ABI entry point
    (kv4_host_pipe_step, via HostPipe), as a serving loop runs it: every step
    copies its inputs (q, the top-k list, seq_lens, the new tokens and their
    slots) from pinned host memory into device staging and its result (out,
    lse) back into pinned host memory; the library keeps two steps in flight
    (inputs of step i+1 and the result of step i-1 move on two copy streams
    while step i computes).  The timed region spans all K steps, copies
    included.  L2 stays cold without a flush: consecutive steps rotate over
    `variants` top-k sets (the same positions shifted, so the same counts and
    structure) whose rows together exceed L2."""
    K = args.steps
    L = w.seq_lens.to(torch.int64).view(-1, 1, 1)
    q_h = wl.queries(w).pin_memory()
    topk_h = [((w.topk.to(torch.int64) + 7919 * 64 * v) % L).to(torch.int32).pin_memory()
              for v in range(variants)]
    lens_h = w.seq_lens.clone().pin_memory()
    nl, nr, ns = wl.newest_tokens(w)
    nl_h, nr_h, ns_h = nl.pin_memory(), nr.pin_memory(), ns.pin_memory()
    out_h = [torch.empty((w.B, w.Sq, w.H, 512), dtype=torch.bfloat16).pin_memory()
             for _ in range(2)]
    lse_h = [torch.empty((w.B, w.Sq, w.H), dtype=torch.float32).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in (q_h, topk_h[0], lens_h, nl_h, nr_h, ns_h))
    d2h = out_h[0].numel() * out_h[0].element_size() + lse_h[0].numel() * lse_h[0].element_size()
    pipe = kv.HostPipe(w.B, w.Sq, w.H, w.K, ns_h.shape[0], dev)

    def run(n):
        for i in range(n):
            pipe.step(nl_h, nr_h, ns_h, pool, q_h, pt, topk_h[i % variants], lens_h, w.sm_scale,
                      out_h[i % 2], lse_h[i % 2])

    run(max(3, args.warmup))
    pipe.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(pipe.compute)
    pipe.copy_in.wait_event(a)             # the first input copy starts after `a`
    run(K)
    pipe.compute.wait_stream(pipe.copy_out)  # ... and the last result copy ends before `b`
    b.record(pipe.compute)
    b.synchronize()
    pipe.close()
    t = a.elapsed_time(b) / K
    valid = valid_key_count(w)
    return {"value": valid * 352 / (t * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": t,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "form": (f"kv4_host_pipe_step from pinned host buffers, {K} steps, two in flight "
                     f"(inputs of step i+1 and result of step i-1 copied while step i "
                     f"computes); L2 cold by rotating {variants} top-k sets")}


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--cpu-sessions", type=int, default=64)
    p.add_argument("--skip-cpu", action="store_true")
    p.add_argument("--sessions", type=int, default=64,
                   help="sessions of the long-context workload per rank (smaller: profiling)")
    p.add_argument("--skip-variants", action="store_true",
                   help="skip the 288-byte row and FP8 comparison measurements")
    p.add_argument("--skip-per-config", action="store_true",
                   help="skip the graph-timed measurement of every workload configuration")
    p.add_argument("--splits", type=int, default=0,
                   help="force the split-K count (0: the library's plan)")
    p.add_argument("--cache-write-only", action="store_true",
                   help="time only the 1M-token cache write (amax and MSE scales) and print it")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.cache_write_only:
        import bit_kv_cache_nvfp4_gb300 as kv
        dev = torch.device("cuda", dist_env()[2])
        torch.cuda.set_device(dev)
        flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        print(json.dumps({"cache_write_1M_tokens": run_cache_write(kv, dev, flush, args)}))
        return 0
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())

"""Attention forward throughput on GB300.

One step = one attention forward (one launch of the library's kernel) over a
whole synthetic workload, inputs resident in HBM.  Prints one JSON line with
the metric (TFLOP/s over structurally visible keys, 4*D FLOPs per visible
(query, key) pair), the roofline of the kernel against the measured dense BF16
peak, an end-to-end number through the public API with host buffers, the fp64
CPU oracle timed on a bounded sample, and the SM clocks seen while timing.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...     # the CPU oracle arm

Multi-GPU (torchrun, one process per GPU): every rank runs an independent
replica of the workload (the path has no exchange step), the timed region is
bracketed by barriers, and the slowest rank's time is used.
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from tiled_online_softmax_02_gb300.inputs import (DSA_WORKLOADS, EXTRA_WORKLOADS,  # noqa: E402
                                                  WORKLOADS, DsaWorkload, Workload, make_dsa_inputs,
                                                  make_inputs)

ALL_WORKLOADS = {**WORKLOADS, **EXTRA_WORKLOADS}

DEFAULT_WORKLOAD = "gqa_causal_bf16"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the
# dominant kernel from one ncu capture, keyed by workload (+splitkv: the
# attn_fwd_splitkv entry), with the hash of that kernel's sources at the time;
# reported as null once those sources change.
NCU_TRAFFIC = {
    "gqa_causal_bf16": {"bytes_per_launch": 127417600, "source_hash": "8b5647f515ca3d4a"},
    "window_softcap_bf16": {"bytes_per_launch": 397537536, "source_hash": "8b5647f515ca3d4a"},
    "ragged_kvcache_f16": {"bytes_per_launch": 48649472, "source_hash": "8b5647f515ca3d4a"},
    "dit_f32": {"bytes_per_launch": 57792000, "source_hash": "8808934b75c1e438"},
    "dit_f32+f32split": {"bytes_per_launch": 69517568, "source_hash": "297cd19ddfb9bc7b"},
    "decode_bf16": {"bytes_per_launch": 775977216, "source_hash": "9febafcf1e6362f3"},
    "decode_bf16+splitkv": {"bytes_per_launch": 777591040, "source_hash": "9febafcf1e6362f3"},
    "gqa_causal_bf16_d256": {"bytes_per_launch": 365990656, "source_hash": "c52d466f411cd530"},
    "gqa_causal_bf16_d384": {"bytes_per_launch": 884027136, "source_hash": "c52d466f411cd530"},
    "vae_f32_d384": {"bytes_per_launch": 18930944, "source_hash": "8808934b75c1e438"},
    # the DSA indexer: the tile score kernel (the selection kernel's traffic is in its profile)
    "dsa_prefill_bf16": {"bytes_per_launch": 139097088, "source_hash": "fda2993782a35635"},
    "dsa_decode_bf16": {"bytes_per_launch": 34638080, "source_hash": "fda2993782a35635"},
}


# ----------------------------------------------------------------- FLOP count
def visible_counts(w: Workload, total=None, past=None) -> np.ndarray:
    """Number of structurally visible keys per (b, qi): [B, Sq] int64.  The
    rule of the prefill kernel page (valid length, causal limit from
    past_lengths or the end of the valid keys, window lower bound)."""
    qi = np.arange(w.Sq, dtype=np.int64)
    out = np.zeros((w.B, w.Sq), dtype=np.int64)
    for b in range(w.B):
        lsk = int(total[b]) if total is not None else w.Sk
        base = int(past[b]) if past is not None else lsk - w.Sq
        cmax = base + qi
        lo = np.maximum(0, cmax + 1 - w.local_window) if w.local_window > 0 else np.zeros_like(qi)
        hi = np.full_like(qi, min(lsk, w.Sk))
        if w.causal:
            hi = np.minimum(hi, cmax + 1)
        out[b] = np.maximum(0, hi - lo)
    return out


def flops_of(w: Workload, x: dict) -> tuple[int, int]:
    """(FLOPs over visible keys, FLOPs excluding mask entries equal to -inf)."""
    tot = x["total_lengths"].numpy() if x["total_lengths"] is not None else None
    pst = x["past_lengths"].numpy() if x["past_lengths"] is not None else None
    cnt = visible_counts(w, tot, pst)
    flops = 4 * w.D * w.Hq * int(cnt.sum())
    excl = flops
    if x["mask"] is not None:
        m = x["mask"].numpy()
        ninf = 0
        qi = np.arange(w.Sq, dtype=np.int64)
        for b in range(w.B):
            lsk = int(tot[b]) if tot is not None else w.Sk
            base = int(pst[b]) if pst is not None else lsk - w.Sq
            cmax = base + qi
            lo = np.maximum(0, cmax + 1 - w.local_window) if w.local_window > 0 else np.zeros_like(qi)
            hi = np.full_like(qi, min(lsk, w.Sk))
            if w.causal:
                hi = np.minimum(hi, cmax + 1)
            hi = np.maximum(hi, lo)
            planes = [b] if w.mask_planes == w.B else (range(b * w.Hq, (b + 1) * w.Hq)
                                                       if w.mask_planes == w.B * w.Hq else [0])
            for pl in planes:
                c = np.concatenate([np.zeros((w.Sq, 1), np.int64),
                                    np.cumsum(np.isneginf(m[pl]), axis=1)], axis=1)
                n = c[qi, hi] - c[qi, lo]
                ninf += int(n.sum()) * (w.Hq if len(planes) == 1 else 1)
        excl = flops - 4 * w.D * ninf
    return flops, excl


def algorithmic_bytes(w: Workload, x: dict) -> int:
    """Bytes a launch must move at least: Q read and O written once, each kv
    head's visible key and value rows read once, and every mask entry that
    some visible (row, key) pair uses read once per plane."""
    es = 4 if w.dtype == "f32" else 2
    tot = x["total_lengths"].numpy() if x["total_lengths"] is not None else None
    pst = x["past_lengths"].numpy() if x["past_lengths"] is not None else None
    qi = np.arange(w.Sq, dtype=np.int64)
    nbytes = 2 * w.B * w.Hq * w.Sq * w.D * es
    for b in range(w.B):
        lsk = int(tot[b]) if tot is not None else w.Sk
        base = int(pst[b]) if pst is not None else lsk - w.Sq
        cmax = base + qi
        lo = np.maximum(0, cmax + 1 - w.local_window) if w.local_window > 0 else np.zeros_like(qi)
        hi = np.full_like(qi, min(lsk, w.Sk))
        if w.causal:
            hi = np.minimum(hi, cmax + 1)
        hi = np.maximum(hi, lo)
        if w.Sq:
            # union of the rows' visible key ranges (each is an interval)
            keys = int(hi.max()) - int(lo.min()) if hi.max() > lo.min() else 0
            nbytes += 2 * w.Hkv * keys * w.D * es
        if x["mask"] is not None:
            planes = 1 if w.mask_planes == w.B else (w.Hq if w.mask_planes == w.B * w.Hq else 0)
            nbytes += 4 * int((hi - lo).sum()) * planes
    if x["mask"] is not None and w.mask_planes == 1:
        nbytes += 4 * w.Sq * w.Sk
    return nbytes


# ------------------------------------------------------------------- helpers
def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# Sources of each kernel family (the kernel, its launcher and the headers it
# includes): an ncu traffic figure stays valid while these are unchanged.
KERNEL_SOURCES = {
    "tc": ("attn_tc.cuh", "attn_tc.cu", "attn_tc_bf16_d64.cu", "attn_tc_bf16_d128.cu",
           "attn_tc_f16_d64.cu", "attn_tc_f16_d128.cu", "device_common.cuh", "attn_internal.h"),
    "f32": ("attn_f32.cu", "device_common.cuh", "attn_internal.h"),
    "decode": ("attn_decode.cu", "attn_decode.h", "device_common.cuh", "attn_internal.h"),
    "f32tc": ("attn_f32tc.cu", "attn_lane1.cuh", "device_common.cuh", "attn_internal.h"),
    "lane16": ("attn_lane16.cu", "attn_lane1.cuh", "device_common.cuh", "attn_internal.h"),
    "dsa": ("dsa_select.cu", "dsa_internal.h", "device_common.cuh"),
}


def kernel_family(w: Workload, splitkv: bool = False, f32split: bool = False) -> str:
    if w.dtype == "f32":
        return "f32tc" if f32split else "f32"
    if w.D in (256, 384):
        return "lane16"
    return "decode" if w.group * w.Sq <= 32 else "tc"


def kernel_source_hash(family: str) -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tiled_online_softmax_02_gb300", "csrc")
    for name in KERNEL_SOURCES[family]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms while active
    (a timed region of a few hundred ms then gets several samples)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines: list[tuple[float, str]] = []
        self.t0 = self.t1 = None
        self._reader = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._reader = threading.Thread(target=self._read, daemon=True)
        self._reader.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, start: bool):
        if start:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._reader:
            self._reader.join(timeout=2)
        sm, mx, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if self.t0 is not None and not (self.t0 - 0.25 <= ts <= (self.t1 or ts) + 0.25):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            n += 1
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": n}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value over all ranks (the slowest rank's time)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(flops_per_step: float, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job TFLOP/s: every rank ran `steps` replicas of the workload."""
    return flops_per_step * steps * world / max_seconds / 1e12


def workload_config(w: Workload, flops: int, flops_excl: int, n: int) -> dict:
    cfg = {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Sk": w.Sk,
           "kv_capacity": w.kv_capacity, "D": w.D, "causal": bool(w.causal),
           "local_window": w.local_window, "softcap": w.softcap, "mask_planes": w.mask_planes,
           "ragged": w.ragged, "out_layout": ["head_major", "token_major"][w.out_layout],
           "seed": w.seed, "flops_per_step": flops, "parallelism": f"replicas x{n}",
           "l2": "flushed between timed steps outside the timed events: a 256 MiB write, then a "
                 "256 MiB read so no dirty line is left to be written back inside the next step"}
    if flops_excl != flops:
        cfg["flops_per_step_excluding_neg_inf_mask"] = flops_excl
    return cfg


# ------------------------------------------------------------- oracle (CPU)
def oracle_sample(w: Workload, x: dict, budget_s: float, seed: int = 3):
    """Times the fp64 oracle on seeded random rows of the workload for about
    budget_s seconds.  Returns (flops, seconds, threads, rows)."""
    import oracle
    threads = oracle.default_threads()
    tot = x["total_lengths"].numpy() if x["total_lengths"] is not None else None
    pst = x["past_lengths"].numpy() if x["past_lengths"] is not None else None
    cnt = visible_counts(w, tot, pst)
    rng = np.random.default_rng(seed)
    kw = dict(B=w.B, Hq=w.Hq, Hkv=w.Hkv, Sq=w.Sq, Sk=w.Sk, kv_capacity=w.kv_capacity, D=w.D,
              causal=w.causal, local_window=w.local_window, scale=w.softmax_scale,
              softcap=w.softcap, mask=x["mask"], mask_planes=w.mask_planes,
              total_lengths=x["total_lengths"], past_lengths=x["past_lengths"], nthreads=threads)
    qf, kf, vf = x["q"].float().numpy(), x["k"].float().numpy(), x["v"].float().numpy()

    def pick(n):
        return np.stack([rng.integers(0, w.B, n), rng.integers(0, w.Hq, n),
                         rng.integers(0, w.Sq, n)], axis=1).astype(np.int64)

    def run(rows):
        t = time.perf_counter()
        oracle.attn_rows(qf, kf, vf, rows, **kw)
        return time.perf_counter() - t, 4 * w.D * int(cnt[rows[:, 0], rows[:, 2]].sum())

    # grow a calibration sample until its timing means something, then size
    # the rest of the sample to the budget
    n, tot_s, tot_fl, tot_rows = 4 * threads, 0.0, 0, 0
    while True:
        dt, fl = run(pick(n))
        tot_s, tot_fl, tot_rows = tot_s + dt, tot_fl + fl, tot_rows + n
        if dt >= 0.5 or n >= 2_000_000 or tot_s + 4 * dt > budget_s:
            break
        n *= 4
    rate = tot_fl / max(tot_s, 1e-6)
    per_row = max(tot_fl / tot_rows, 1.0)
    left = budget_s - tot_s
    if left > 0.2:
        n2 = int(max(threads, min(5_000_000, left * rate / per_row)))
        dt, fl = run(pick(n2))
        tot_s, tot_fl, tot_rows = tot_s + dt, tot_fl + fl, tot_rows + n2
    return tot_fl, tot_s, threads, tot_rows


def reference_arm(args, world, rank):
    if rank != 0:
        return 0
    w = ALL_WORKLOADS[args.workload]
    x = make_inputs(w)
    flops, flops_excl = flops_of(w, x)
    # the whole arm (warm-up included) stays within about --ref-seconds
    per_step_budget = max(0.02, args.ref_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(w, x, per_step_budget, seed=11)
    tot_fl, tot_s, threads, rows = 0, 0.0, 0, 0
    for i in range(args.steps):
        fl, s, threads, r = oracle_sample(w, x, per_step_budget, seed=100 + i)
        tot_fl, tot_s, rows = tot_fl + fl, tot_s + s, rows + r
    value = tot_fl / tot_s / 1e12
    sample = (f"{rows} seeded random (b, h, qi) rows of {w.name}, oracle_attn_rows, "
              f"{args.steps} steps of ~{per_step_budget:.2f} s")
    line = {"metric": "attention fwd TFLOP/s (unmasked FLOPs)", "impl": "reference",
            "value": value, "unit": "TFLOP/s", "n_gpus": 0, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": tot_s * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, shaped like the pages' workloads)",
            # the same config as our arm at this world size (only rank 0 runs the oracle)
            "config": workload_config(w, flops, flops_excl, world),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm
def run_ours(args, world, rank, local):
    import tiled_online_softmax_02_gb300 as attn
    from tiled_online_softmax_02_gb300 import build as libbuild
    if not libbuild.up_to_date() and rank == 0:
        libbuild.build()
    barrier(world)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    attn.load_library()
    w = ALL_WORKLOADS[args.workload]
    x = make_inputs(w)
    flops, flops_excl = flops_of(w, x)
    abytes = algorithmic_bytes(w, x)
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    out = torch.empty((w.B, w.Hq, w.Sq, w.D) if w.out_layout == 0 else (w.B, w.Sq, w.Hq * w.D),
                      dtype=g["q"].dtype, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def evict_l2():
        # A write larger than L2 evicts it, but leaves it full of dirty lines
        # whose write-back would land inside the next timed launch; reading
        # another buffer larger than L2 writes them back here instead.
        flush.zero_()
        flush_rd.max()
    stream = torch.cuda.current_stream(dev)

    launches_per_step = 1
    # fp32 workloads run the tensor-core entry (attn_fwd_f32_split) for the
    # head dims it covers unless --f32-path exact asks for the CUDA-core kernel
    f32split = w.dtype == "f32" and args.f32_path == "split" and w.D in (64, 128)
    if f32split:
        lib = attn.load_library()
        ws_f32 = torch.empty(lib.attn_f32_split_workspace_bytes(w.B, w.Hkv, w.kv_capacity, w.D),
                             dtype=torch.uint8, device=dev)
        launches_per_step = 2  # the K / V split, then the attention kernel
    if args.splitkv:
        lib = attn.load_library()
        splits = args.splits or lib.attn_splitkv_num_splits(w.B, w.Hq, w.Hkv, w.Sq, w.Sk)
        need = lib.attn_splitkv_workspace_bytes(w.B, w.Hq, w.Sq, w.D, splits)
        ws_buf = torch.empty(max(need // 4, 4), dtype=torch.float32, device=dev)
        lse_buf = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
        launches_per_step = 2 if splits > 1 else 1

    def step():
        if args.splitkv:
            attn.attn_fwd_splitkv(g["q"], g["k"], g["v"], mask=g["mask"],
                                  total_lengths=g["total_lengths"], past_lengths=g["past_lengths"],
                                  causal=w.causal, local_window=w.local_window,
                                  scale=w.softmax_scale, softcap=w.softcap,
                                  out_layout=w.out_layout, seq_k=w.Sk, num_splits=splits,
                                  out=out, lse=lse_buf, workspace=ws_buf)
            return
        if f32split:
            attn.attn_fwd_f32_split(g["q"], g["k"], g["v"], mask=g["mask"],
                                    total_lengths=g["total_lengths"], past_lengths=g["past_lengths"],
                                    causal=w.causal, local_window=w.local_window,
                                    scale=w.softmax_scale, softcap=w.softcap,
                                    out_layout=w.out_layout, seq_k=w.Sk, out=out, workspace=ws_f32)
            return
        attn.attn_fwd(g["q"], g["k"], g["v"], mask=g["mask"], total_lengths=g["total_lengths"],
                      past_lengths=g["past_lengths"], causal=w.causal,
                      local_window=w.local_window, scale=w.softmax_scale, softcap=w.softcap,
                      out_layout=w.out_layout, seq_k=w.Sk, out=out)

    for _ in range(args.warmup):
        evict_l2()
        step()
    torch.cuda.synchronize()
    if attn.get_device_status() != attn.ATTN_OK:
        raise RuntimeError("kernel reported a timeout during warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local) if not args.no_clocks else None
    if clocks:
        clocks.start()
        time.sleep(0.6)  # let nvidia-smi come up before the timed region
    barrier(world)
    torch.cuda.synchronize()
    if clocks:
        clocks.mark(True)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        evict_l2()                    # outside the timed events
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    if clocks:
        clocks.mark(False)
    clock_info = clocks.stop() if clocks else None
    if attn.get_device_status() != attn.ATTN_OK:
        raise RuntimeError("kernel reported a timeout during the timed region")
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    kernel_s = sum(step_ms) / 1e3
    max_s = max_over_ranks(kernel_s, world, dev)
    value = replica_throughput(flops, args.steps, world, max_s)
    avg_launch_s = kernel_s / args.steps

    # end to end through the public API with pinned host buffers
    host = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)

    def e2e_step():
        if f32split:
            attn.attn_fwd_f32_split(host["q"], host["k"], host["v"], mask=host["mask"],
                                    total_lengths=host["total_lengths"],
                                    past_lengths=host["past_lengths"], causal=w.causal,
                                    local_window=w.local_window, scale=w.softmax_scale,
                                    softcap=w.softcap, out_layout=w.out_layout, seq_k=w.Sk,
                                    out=host_out, workspace=ws_f32)
            return
        attn.attn_fwd(host["q"], host["k"], host["v"], mask=host["mask"],
                      total_lengths=host["total_lengths"], past_lengths=host["past_lengths"],
                      causal=w.causal, local_window=w.local_window, scale=w.softmax_scale,
                      softcap=w.softcap, out_layout=w.out_layout, seq_k=w.Sk, out=host_out)
    for _ in range(2):
        e2e_step()
    # the bytes each step moves, as the library counted its copies (only the
    # cache rows and mask columns that can reach the output go up)
    h2d, d2h = attn.host_copy_bytes()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)
    e2e_value = replica_throughput(flops, args.e2e_steps, world, e2e_s)

    if rank != 0:
        return 0
    peaks, src = read_peaks()
    hbm_gbs = abytes / avg_launch_s / 1e9
    ridge = float(peaks["bf16_tflops"]) * 1e3 / float(peaks["hbm_gbs"])  # FLOP per byte
    if w.dtype != "f32" and flops / max(abytes, 1) < ridge:
        # below the ridge point HBM, not the tensor pipe, bounds the launch
        peak, bound = float(peaks["hbm_gbs"]), "hbm"
        src = f"{src} hbm_gbs"
    elif f32split:
        # bf16 tensor cores doing 4.5 MMAs per fp32 MMA (6 for QK^T, 3 for P.V)
        peak, bound = float(peaks["bf16_tflops"]) / 4.5, "tensor"
        src = f"{src} bf16_tflops (burst) / 4.5 bf16 MMAs per fp32 MMA (6 for QK^T, 3 for PV)"
    elif w.dtype == "f32":
        # fp32 FFMA on CUDA cores: SMs x 128 FMA/clk x 2 FLOP x max SM clock
        props = torch.cuda.get_device_properties(dev)
        mhz = float(peaks.get("sm_max_mhz", 2070.0))
        peak, bound, src = props.multi_processor_count * 128 * 2 * mhz * 1e6 / 1e12, "alu", \
            "derived: SMs x 128 FFMA/clk x 2 x max SM clock"
    else:
        peak, bound = float(peaks["bf16_tflops"]), "tensor"
        src = f"{src} bf16_tflops (burst)"
    achieved = flops / avg_launch_s / 1e12
    roof = hbm_gbs if bound == "hbm" else achieved
    traffic = None
    ent = NCU_TRAFFIC.get(w.name + ("+splitkv" if args.splitkv else "") + ("+f32split" if f32split else ""))
    if ent and ent.get("source_hash") == kernel_source_hash(kernel_family(w, args.splitkv, f32split)):
        traffic = ent["bytes_per_launch"]
    cpu = None
    if not args.no_cpu_baseline:
        fl, s, threads, rows = oracle_sample(w, x, args.cpu_seconds)
        cpu = {"value": fl / s / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{rows} seeded random (b, h, qi) rows of {w.name} ({fl / 1e9:.2f} GFLOP, "
                         f"{s:.1f} s), fp64 oracle_attn_rows"}
    line = {
        "metric": "attention fwd TFLOP/s (unmasked FLOPs)",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": max_s * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic (seeded, shaped like the pages' workloads)",
        "config": workload_config(w, flops, flops_excl, world),
        # the C-ABI entry timed (kept out of config, which both arms print alike)
        "entry": ("attn_fwd_splitkv" if args.splitkv else "attn_fwd_f32_split" if f32split else "attn_fwd"),
        **({"num_splits": splits} if args.splitkv else {}),
        "frac_of_peak": roof / peak,
        "roofline": {"bound": bound, "achieved": roof, "peak": peak,
                     "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
                     "frac": roof / peak, "traffic": traffic, "peak_source": src,
                     "algorithmic_bytes": abytes, "hbm_gbs": hbm_gbs,
                     "frac_of_sustained": (achieved / (float(peaks.get("bf16_tflops_sustained", peak))
                                                       / (4.5 if f32split else 1.0))
                                           if bound == "tensor" else None)},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": args.e2e_steps},
        "cpu_baseline": cpu,
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clock_info,
        "wall_s_timed_region": wall,
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------- DSA indexer workloads
DSA_METRIC = "DSA index select TFLOP/s (2*H*D per allowed cell)"


def dsa_allowed_counts(x: dict) -> np.ndarray:
    """Allowed keys per (b, s) row (bias above -1e30), [B, S]."""
    return (x["bias"].numpy()[:, 0] > np.float32(-1e30)).sum(-1)


def dsa_flops(w: DsaWorkload, cnt: np.ndarray) -> int:
    return 2 * w.H * w.D * int(cnt.sum())


def dsa_algorithmic_bytes(w: DsaWorkload) -> int:
    es = 4 if w.dtype == "f32" else 2
    rows = w.B * w.S
    return (rows * w.H * w.D * es + w.B * w.T * w.D * es + rows * w.H * es   # query, key, weights
            + rows * w.T * 4                                                # bias
            + 2 * rows * w.T * 4                                            # scores written, read back
            + rows * w.top_k * 8)                                           # indices


def dsa_config(w: DsaWorkload, flops: int, n: int) -> dict:
    return {"workload": w.name, "B": w.B, "S": w.S, "H": w.H, "D": w.D, "T": w.T, "top_k": w.top_k,
            "bias": w.bias, "scale": w.softmax_scale, "weights_scale": w.weights_scale,
            "seed": w.seed, "flops_per_step": flops, "parallelism": f"replicas x{n}",
            "entry": "dsa_index_select",
            "l2": "flushed between timed steps outside the timed events: a 256 MiB write, then a "
                  "256 MiB read"}


def dsa_oracle_sample(w: DsaWorkload, x: dict, budget_s: float, seed: int = 3):
    """Times the fp32 oracle (oracle_dsa_rows, one thread) on seeded random
    rows for about budget_s seconds.  Returns (flops, seconds, threads, rows)."""
    from oracle import dsa
    cnt = dsa_allowed_counts(x).reshape(-1)
    arrs = [np.ascontiguousarray(x[n].float().numpy()) for n in ("query", "key", "weights", "bias")]
    rng = np.random.default_rng(seed)
    rows_total = w.B * w.S

    def run(n):
        rows = rng.integers(0, rows_total, n)
        t = time.perf_counter()
        dsa.rows(*arrs, rows, top_k=w.top_k, scale=w.softmax_scale, weights_scale=w.weights_scale)
        return time.perf_counter() - t, 2 * w.H * w.D * int(cnt[rows].sum()), n

    n, tot_s, tot_fl, tot_rows = 1, 0.0, 0, 0
    while True:
        dt, fl, r = run(n)
        tot_s, tot_fl, tot_rows = tot_s + dt, tot_fl + fl, tot_rows + r
        if dt >= 0.5 or tot_s + 4 * dt > budget_s:
            break
        n *= 4
    left = budget_s - tot_s
    per_row_s = tot_s / max(tot_rows, 1)
    if left > 0.2 and per_row_s > 0:
        dt, fl, r = run(int(max(1, min(1_000_000, left / per_row_s))))
        tot_s, tot_fl, tot_rows = tot_s + dt, tot_fl + fl, tot_rows + r
    return tot_fl, tot_s, 1, tot_rows


def dsa_reference_arm(args, world, rank):
    if rank != 0:
        return 0
    w = DSA_WORKLOADS[args.workload]
    x = make_dsa_inputs(w)
    flops = dsa_flops(w, dsa_allowed_counts(x))
    per_step_budget = max(0.02, args.ref_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        dsa_oracle_sample(w, x, per_step_budget, seed=11)
    tot_fl, tot_s, rows = 0, 0.0, 0
    for i in range(args.steps):
        fl, s, threads, r = dsa_oracle_sample(w, x, per_step_budget, seed=100 + i)
        tot_fl, tot_s, rows = tot_fl + fl, tot_s + s, rows + r
    value = tot_fl / tot_s / 1e12
    sample = (f"{rows} seeded random (b, s) rows of {w.name}, oracle_dsa_rows, "
              f"{args.steps} steps of ~{per_step_budget:.2f} s")
    line = {"metric": DSA_METRIC, "impl": "reference", "value": value, "unit": "TFLOP/s", "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_s * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded)", "config": dsa_config(w, flops, world),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_dsa(args, world, rank, local):
    import tiled_online_softmax_02_gb300 as attn
    from tiled_online_softmax_02_gb300 import build as libbuild
    if not libbuild.up_to_date() and rank == 0:
        libbuild.build()
    barrier(world)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib = attn.load_library()
    w = DSA_WORKLOADS[args.workload]
    x = make_dsa_inputs(w)
    flops = dsa_flops(w, dsa_allowed_counts(x))
    abytes = dsa_algorithmic_bytes(w)
    names = ("query", "key", "weights", "bias")
    g = {n: x[n].to(dev) for n in names}
    out = torch.empty((w.B, 1, w.S, w.top_k), dtype=torch.int64, device=dev)
    ws = torch.empty(max(lib.dsa_index_select_workspace_bytes(w.B, w.S, w.T), 16), dtype=torch.uint8,
                     device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def evict_l2():
        flush.zero_()
        flush_rd.max()

    def step():
        attn.dsa_index_select(g["query"], g["key"], g["weights"], g["bias"], top_k=w.top_k,
                              scale=w.softmax_scale, weights_scale=w.weights_scale, out=out, workspace=ws)

    for _ in range(args.warmup):
        evict_l2()
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local) if not args.no_clocks else None
    if clocks:
        clocks.start()
        time.sleep(0.6)
    barrier(world)
    torch.cuda.synchronize()
    if clocks:
        clocks.mark(True)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        evict_l2()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    if clocks:
        clocks.mark(False)
    clock_info = clocks.stop() if clocks else None
    kernel_s = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / 1e3
    max_s = max_over_ranks(kernel_s, world, dev)
    value = replica_throughput(flops, args.steps, world, max_s)
    avg_step_s = kernel_s / args.steps

    # end to end through the public API with pinned host tensors
    host = {n: x[n].pin_memory() for n in names}
    host_out = torch.empty(out.shape, dtype=torch.int64, pin_memory=True)
    h2d = sum(int(v.numel() * v.element_size()) for v in host.values())
    d2h = int(host_out.numel() * host_out.element_size())

    def e2e_step():
        attn.dsa_index_select(host["query"], host["key"], host["weights"], host["bias"], top_k=w.top_k,
                              scale=w.softmax_scale, weights_scale=w.weights_scale, out=host_out,
                              workspace=ws)
    for _ in range(2):
        e2e_step()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)
    e2e_value = replica_throughput(flops, args.e2e_steps, world, e2e_s)
    if rank != 0:
        return 0

    # The score kernel is bound by fp32 arithmetic on the CUDA cores: each
    # multiply and add is its own instruction (the page fixes unfused fp32),
    # so the ceiling is one FLOP per lane per clock.  The step time (both
    # kernels of the call) is the denominator, so the fraction is a floor.
    peaks, _ = read_peaks()
    props = torch.cuda.get_device_properties(dev)
    mhz = float(peaks.get("sm_max_mhz", 2070.0))
    peak = props.multi_processor_count * 128 * mhz * 1e6 / 1e12
    achieved = flops / avg_step_s / 1e12
    traffic = None
    ent = NCU_TRAFFIC.get(w.name)
    if ent and ent.get("source_hash") == kernel_source_hash("dsa"):
        traffic = ent["bytes_per_launch"]
    cpu = None
    if not args.no_cpu_baseline:
        fl, s, threads, rows = dsa_oracle_sample(w, x, args.cpu_seconds)
        cpu = {"value": fl / s / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{rows} seeded random (b, s) rows of {w.name} ({fl / 1e9:.2f} GFLOP, {s:.1f} s), "
                         f"fp32 oracle_dsa_rows"}
    line = {
        "metric": DSA_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": max_s * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded)", "config": dsa_config(w, flops, world),
        "frac_of_peak": achieved / peak,
        "roofline": {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": "derived: SMs x 128 fp32 lanes x 1 unfused op/clk x max SM clock",
                     "kernel": "dsa_score_kernel + dsa_select_kernel (one call, timed together)",
                     "algorithmic_bytes": abytes, "hbm_gbs": abytes / avg_step_s / 1e9},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": args.e2e_steps},
        "cpu_baseline": cpu,
        "gpu_launches": args.steps * 2,
        "clocks": clock_info,
        "wall_s_timed_region": wall,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(ALL_WORKLOADS) + list(DSA_WORKLOADS),
                    default=DEFAULT_WORKLOAD)
    ap.add_argument("--splitkv", action="store_true",
                    help="time attn_fwd_splitkv (split count: --splits, else the library's choice)")
    ap.add_argument("--splits", type=int, default=0, help="split count for --splitkv (0: library)")
    ap.add_argument("--f32-path", choices=["split", "exact"], default="split",
                    help="fp32 workloads: the tensor-core entry attn_fwd_f32_split (D 64 / 128) or "
                         "the fp32-exact CUDA-core kernel of attn_fwd")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    world, rank, local = dist_setup()
    try:
        if args.workload in DSA_WORKLOADS:
            if args.impl == "reference":
                return dsa_reference_arm(args, world, rank)
            return run_dsa(args, world, rank, local)
        if args.impl == "reference":
            return reference_arm(args, world, rank)
        return run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())

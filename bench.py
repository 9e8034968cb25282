"""Benchmark of the exact-attention hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
  1. prefill: Llama-3-8B GQA layer, h=32, h_kv=8, d_h=128, T=8192, causal,
     bf16 Q/K/V ~ N(0,1) with Q and K x3 (widened logits);   [attn_prefill]
  2. paged decode: 64 rows with lengths U[1,16384] plus 2 empty rows, h=32,
     h_kv=8, d_h=128, bf16 KV in 16-token pages, shuffled physical pages,
     split count from attn_recommended_splits;              [attn_decode_paged
                                                            = split kernel + merge]
L2 is flushed (a 512 MiB write) before each prefill; the decode streams a
2.15 GB cache, far larger than L2.

Prints ONE JSON line. `value` is prefill attention TFLOP/s (algorithmic FLOPs
4*h*d_h*T(T+1)/2 over the prefill kernel's CUDA-event time, summed over all
ranks); the `decode` object carries paged-decode KV GB/s.
`--impl reference` times the float64 CPU oracle on a bounded sample instead.
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

import workloads as W  # noqa: E402

METRIC = "prefill attention TFLOP/s; paged decode KV GB/s (fraction of GB300 roofline)"
PREFILL = W.GQA_T8192_CAUSAL
DECODE = W.DECODE_PAGED_B64

# DRAM traffic per launch from one ncu capture of the kernel, valid only for
# the kernel source it was taken on (hash of its files).
KERNEL_FILES = {
    "prefill": ["online_softmax_attn_gb300/csrc/prefill_tc.cu", "online_softmax_attn_gb300/csrc/tc.cuh",
                "online_softmax_attn_gb300/csrc/common.cuh", "online_softmax_attn_gb300/csrc/pdl.cuh"],
    "decode": ["online_softmax_attn_gb300/csrc/decode.cu", "online_softmax_attn_gb300/csrc/common.cuh",
               "online_softmax_attn_gb300/csrc/pdl.cuh"],
}
KERNEL_FILES["prefill_paged"] = KERNEL_FILES["prefill"]
KERNEL_FILES["prefill_T2048"] = KERNEL_FILES["prefill"]
KERNEL_FILES["merge_pair"] = ["online_softmax_attn_gb300/csrc/merge.cu", "online_softmax_attn_gb300/csrc/common.cuh",
                              "online_softmax_attn_gb300/csrc/pdl.cuh"]
NCU_TRAFFIC = {
    # kind: (dram read + write bytes per launch, sha256[:16] of the kernel's files)
    # prefill_bf16_kernel, causal T=8192 layer, full-size capture: 102.5 MB read
    # (compulsory Q, K, fp16 V) + 30.6 MB of the 67.1 MB output written back by exit
    "prefill": (133.14e6, "b157eca97be5ddc7"),
    # prefill_bf16_kernel, causal T=2048 layer, full-size capture: the compulsory
    # 25.3 MB read; the 16.8 MB output is still in L2 when the kernel exits
    "prefill_T2048": (25.26e6, "b157eca97be5ddc7"),
    # prefill_bf16_kernel (paged), 8 rows x 1024 queries over 8192 keys, full-size capture
    "prefill_paged": (473.54e6, "b157eca97be5ddc7"),
    # decode_split_kernel: a 16-row capture (304.0 MB for 299.5 MB algorithmic) scaled by
    # the KV bytes to the 66-row batch
    "decode": (2.1520e9, "61652ac3d8eae098"),
    # merge_pair_kernel, 262144 rows x 128 bf16, full-size capture: reads are the compulsory
    # 136.3 MB, writes 37.4 MB of the 68.2 MB output (the rest still in L2 at exit)
    "merge_pair": (173.71e6, "b69c2e0580ea7eaf"),
}


def src_hash(kind: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_FILES[kind]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(kind: str):
    rec = NCU_TRAFFIC.get(kind)
    if rec is None or rec[1] != src_hash(kind):
        return None
    return rec[0]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], "measured"
    return 6800.0, 1900.0, "fallback"


def prefill_flops(shape) -> float:
    T = shape.T
    pairs = T * (T + 1) / 2 if shape.causal else T * T
    return 4.0 * shape.h * shape.d_h * pairs


def decode_bytes(lens, shape) -> int:
    """Algorithmic decode bytes: K and V of every attended key, q, o, and the
    block-table entries of the attended pages (partials are overhead)."""
    kv = 2 * sum(lens) * shape.h_kv * shape.d_h * 2
    qo = 2 * len(lens) * shape.h * shape.d_h * 2
    bt = sum((s + 15) // 16 for s in lens) * 4
    return kv + qo + bt


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, out_dir: str | None = None):
        self.index = index
        self.proc = None
        self.path = os.path.join(out_dir or tempfile.gettempdir(), f"attn_bench_clocks_rank{index}.csv")

    def _gpu_id(self):
        """nvidia-smi index of this rank's GPU (None: the only one visible)."""
        try:
            n = len(subprocess.run(["nvidia-smi", "-L"], capture_output=True, text=True,
                                   timeout=30).stdout.strip().splitlines())
        except (OSError, subprocess.SubprocessError):
            return None
        if n <= 1:
            return None
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            ids = [x.strip() for x in vis.split(",") if x.strip()]
            if self.index < len(ids):
                return ids[self.index]
        return str(self.index)

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            gid = self._gpu_id()
            cmd = ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "50"]
            if gid is not None:
                cmd.insert(1, f"--id={gid}")
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.fh, stderr=subprocess.DEVNULL)
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
        self.fh.close()
        sm, mx, reasons = [], None, set()
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for name, col in (("hw_slowdown", 5), ("hw_thermal_slowdown", 6),
                                  ("sw_thermal_slowdown", 7), ("sw_power_cap", 8)):
                    if parts[col].lower().startswith("active"):
                        reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


class NvmlClockSampler:
    """SM clock, power and clock-event reasons of this process's GPU, read
    through NVML (read-only queries) every ``period_s`` on a background thread
    while the timed region runs. NVML identifies the GPU by its UUID."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown"}

    def __init__(self, dev, period_s: float = 0.002):
        import ctypes
        import threading

        self.period = period_s
        self.samples = []
        self._stop = threading.Event()
        self._thread = None
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib, self.ct = lib, ctypes
        self.h = ctypes.c_void_p()
        uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
        if uuid is None or lib.nvmlDeviceGetHandleByUUID(f"GPU-{uuid}".encode(),
                                                         ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle for this GPU")
        mx = ctypes.c_uint()
        lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))  # 1 = SM clock
        self.max_mhz = float(mx.value)
        self._reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def _loop(self):
        ct, lib = self.ct, self.lib
        c, r, pw = ct.c_uint(), ct.c_ulonglong(), ct.c_uint()
        while not self._stop.is_set():
            if lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(c)) == 0:
                self._reasons(self.h, ct.byref(r))
                lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(pw))
                self.samples.append((float(c.value), int(r.value), pw.value / 1000.0))
            self._stop.wait(self.period)

    def start(self):
        import threading

        self._thread = threading.Thread(target=self._loop, daemon=True)
        self._thread.start()

    def stop(self):
        self._stop.set()
        if self._thread is not None:
            self._thread.join(timeout=5)
        if not self.samples:
            return None
        reasons = sorted({name for _, r, _ in self.samples for bit, name in self.REASONS.items()
                          if r & bit})
        return {"sm_mhz": statistics.median(c for c, _, _ in self.samples),
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(self.samples),
                "power_w_max": max(p for _, _, p in self.samples), "via": "nvml"}


def make_clock_sampler(dev, local, out_dir):
    try:
        return NvmlClockSampler(dev)
    except (OSError, AttributeError):
        return ClockSampler(local, out_dir)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ---------------------------------------------------------------------------
# CPU oracle legs (float64, host cores)
# ---------------------------------------------------------------------------

def oracle_prefill_sample(q, k, v, rows_per_call: int, seed: int):
    """Oracle on a bounded sample: `rows_per_call` causal rows of one head near
    the end of the sequence (the costliest rows). Returns (seconds, FLOPs)."""
    import oracle

    rng = np.random.default_rng(seed)
    hq = int(rng.integers(0, PREFILL.h))
    r0 = PREFILL.T - rows_per_call - int(rng.integers(0, 64))
    rows = list(range(r0, r0 + rows_per_call))
    t0 = time.perf_counter()
    oracle.attention_rows_ref(q, k, v, PREFILL.scale, True, [hq] * len(rows), rows)
    dt = time.perf_counter() - t0
    flops = sum(4.0 * PREFILL.d_h * (r + 1) for r in rows)
    return dt, flops


def oracle_decode_sample(q, kc, vc, table, seq, rows):
    import oracle

    t0 = time.perf_counter()
    oracle.decode_paged_ref(q, kc, vc, table, seq, DECODE.scale, rows=rows)
    dt = time.perf_counter() - t0
    lens = seq.tolist()
    return dt, decode_bytes([lens[r] for r in rows], DECODE)


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, world, rank):
    """--impl reference: the float64 CPU oracle on bounded samples, rank 0 only."""
    if rank != 0:
        return
    torch.set_num_threads(cpu_cores())
    q, k, v = W.prefill_inputs(PREFILL, 0)
    rows_per_step = 64
    for i in range(args.warmup):
        oracle_prefill_sample(q, k, v, rows_per_step, seed=1000 + i)
    tot_t, tot_f = 0.0, 0.0
    for i in range(args.steps):
        dt, fl = oracle_prefill_sample(q, k, v, rows_per_step, seed=i)
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "float64 CPU oracle (materialised safe softmax) on a bounded sample of "
                               "the causal GQA T=8192 prefill: per step 64 query rows of one head "
                               "near the end of the sequence", "prefill": PREFILL.name},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"{rows_per_step} causal rows x {args.steps} steps of one head at T=8192"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def g4(x):
    return None if x is None else float(f"{x:.4g}")


def bench_line(*, world, steps, warmup, value, dec_value, dec_frac, step_ms, S, pre_achieved,
               tc_peak, traffic, e2e, cpu, cpu_rows_n, launches, clk, dec_avg, dec_e2e=None,
               det=None, adaptive=None, prefill_2048=None, prefill_paged=None, merge_pair=None,
               mixed=None, decode_b1=None) -> dict:
    """The one JSON line rank 0 prints: the step's prefill and decode figures,
    the roofline of the prefill kernel, e2e, the CPU baseline and clocks, and
    the measurements outside the step as a compact ``x`` object (the line
    stays short enough for a log tail to hold it whole)."""
    extras = {"decode_ms": g4(dec_avg)}
    if dec_e2e:
        extras["decode_e2e_gbs"] = g4(dec_e2e["value"])
    if det:
        extras["det_gbs"] = g4(det["value"])
    if adaptive:
        extras["adaptive_gbs"] = g4(adaptive["value"])
    if prefill_2048:
        extras["t2048_tflops"] = g4(prefill_2048["value"])
        extras["t2048_frac"] = g4(prefill_2048["roofline"]["frac"])
    if prefill_paged:
        extras["paged_prefill_tflops"] = g4(prefill_paged["value"])
        extras["paged_prefill_frac"] = g4(prefill_paged["roofline"]["frac"])
    if merge_pair:
        extras["merge_pair_gbs"] = g4(merge_pair["value"])
    if mixed:
        extras["mixed_prefill_tflops"] = g4(mixed["prefill_tflops"])
        extras["mixed_decode_gbs"] = g4(mixed["decode_rows_gbs"])
        extras["mixed_decode_alone_gbs"] = g4(mixed["decode_alone_gbs"])
    if decode_b1:
        for key, short in ((W.DECODE_S32K.name, "b1_h32"), (W.DECODE_70B_TP8.name, "b1_70b_tp8")):
            if key in decode_b1:
                extras[f"{short}_us"] = g4(decode_b1[key]["us_per_call"])
                extras[f"{short}_frac"] = g4(decode_b1[key]["frac_of_hbm"])
    return {
        "metric": METRIC,
        "value": g4(value),
        "unit": "TFLOP/s",
        "decode_gbs": g4(dec_value),
        "decode_frac": g4(dec_frac),
        "n_gpus": world,
        "steps": steps,
        "warmup": warmup,
        "ms_per_step": g4(step_ms),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": "causal GQA prefill T8192 h32 kv8 d128 + paged decode 66 rows",
            "decode_splits": S,
            "l2": "flush 512MiB; decode KV 2.1GB>L2",
            "parallelism": f"replicas x{world}",
        },
        "roofline": {"bound": "tensor", "achieved": g4(pre_achieved), "peak": tc_peak, "unit": "TFLOP/s",
                     "frac": g4(pre_achieved / tc_peak), "traffic": traffic},
        "e2e": None if e2e is None else {k: (g4(v) if isinstance(v, float) else v)
                                         for k, v in e2e.items() if k != "ms"},
        "cpu_baseline": None if cpu is None else {
            "value": g4(cpu["value"]), "unit": cpu["unit"], "cores": cpu["cores"], "kind": "oracle",
            "sample": f"{cpu_rows_n}x64 rows of one T8192 head"},
        "gpu_launches": launches,
        "clocks": None if clk is None else {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"],
                                            "reasons": clk["reasons"], "samples": clk["samples"]},
        "x": extras,
    }


def run_gpu(args, world, rank, local):
    import online_softmax_attn_gb300 as attn
    from online_softmax_attn_gb300 import build as attn_build

    attn_build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    hbm_peak, tc_peak, peak_kind = peaks()
    stream = torch.cuda.current_stream()
    if args.only == "prefill_paged":
        # The paged chunked-prefill measurement alone (profiler captures).
        flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
        res = measure_prefill_paged(dev, flush, tc_peak, peak_kind, iters=max(1, args.steps))
        if rank == 0:
            print(json.dumps({"only": "prefill_paged", "prefill_paged": res}), flush=True)
        return
    if args.only == "decode_batch1":
        # The batch-1 decode measurements alone (profiler captures).
        res = measure_decode_batch1(dev, hbm_peak, peak_kind)
        if rank == 0:
            print(json.dumps({"only": "decode_batch1", "decode_batch1": res}), flush=True)
        return
    if args.only == "prefill_t2048":
        # The T=2048 layer's measurement alone (profiler captures).
        flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
        res = measure_prefill_t2048(dev, flush, tc_peak, peak_kind, iters=max(1, args.steps))
        if rank == 0:
            print(json.dumps({"only": "prefill_t2048", "prefill_T2048": res}), flush=True)
        return
    if args.only == "mixed":
        flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
        res = measure_mixed(dev, flush, hbm_peak, tc_peak, peak_kind)
        if rank == 0:
            print(json.dumps({"only": "mixed", "mixed": res}), flush=True)
        return
    if args.only == "merge_pair":
        # The pairwise merge measurement alone (profiler captures).
        flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
        res = measure_merge_pair(dev, flush, hbm_peak, peak_kind, iters=max(1, args.steps))
        if rank == 0:
            print(json.dumps({"only": "merge_pair", "merge_pair": res}), flush=True)
        return

    # ---- inputs, resident in HBM before the timed region ----
    q, k, v = W.prefill_inputs(PREFILL, seed=rank, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((PREFILL.h, PREFILL.T), dtype=torch.float32, device=dev)
    pws = torch.empty(attn.attn_prefill_workspace_bytes(PREFILL.T, PREFILL.h_kv, PREFILL.d_h),
                      dtype=torch.uint8, device=dev)
    lens = W.decode_seq_lens(DECODE, seed=rank)
    if args.decode_rows:
        lens = lens[:args.decode_rows]  # smaller batch, for profiler captures only
    dq, kc, vc, table, seq = W.decode_inputs(DECODE, seed=rank, device=dev, seq_lens=lens)
    table, seq = table.to(dev), seq.to(dev)
    B = len(lens)
    S = attn.attn_recommended_splits_ragged(B, DECODE.h_kv, max(lens), sum(lens))
    ws = torch.empty(attn.attn_decode_workspace_bytes(B, DECODE.h, S, DECODE.d_h), dtype=torch.uint8, device=dev)
    do = torch.empty_like(dq)
    dlse = torch.empty((B, DECODE.h), dtype=torch.float32, device=dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)

    do_pre = args.only in (None, "prefill")
    do_dec = args.only in (None, "decode")

    def step(ev):
        flush.fill_(1)
        ev[0].record(stream)
        if do_pre:
            attn.attn_prefill(q, k, v, True, PREFILL.scale, o=o, lse=lse, workspace=pws)
        ev[1].record(stream)
        if do_dec:
            attn.attn_decode_paged(dq, kc, vc, table, seq, S, DECODE.scale, workspace=ws, o=do, lse=dlse)
        ev[2].record(stream)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for _ in range(args.warmup):
        step([torch.cuda.Event(enable_timing=True) for _ in range(3)])
    torch.cuda.synchronize()
    if attn.attn_get_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    clocks = make_clock_sampler(dev, local, args.clocks_dir)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()

    total_ms = t_start.elapsed_time(t_end)
    pre_ms = [evs[i][0].elapsed_time(evs[i][1]) for i in range(args.steps)]
    dec_ms = [evs[i][1].elapsed_time(evs[i][2]) for i in range(args.steps)]
    pre_avg = max_over_ranks(sum(pre_ms) / len(pre_ms), world)
    dec_avg = max_over_ranks(sum(dec_ms) / len(dec_ms), world)
    step_ms = max_over_ranks(total_ms / args.steps, world)
    err = attn.attn_get_device_error()
    if err:
        raise RuntimeError(f"device error bits {err:#x} during the timed region")

    pf = prefill_flops(PREFILL)
    db = decode_bytes(lens, DECODE)
    value = world * pf / (pre_avg * 1e-3) / 1e12
    dec_value = world * db / (dec_avg * 1e-3) / 1e9
    pre_achieved = pf / (pre_avg * 1e-3) / 1e12
    dec_achieved = db / (dec_avg * 1e-3) / 1e9

    if args.only in ("prefill", "decode"):
        # One half of the step alone (profiler captures): not a bench line.
        if rank == 0:
            half = ({"prefill_tflops": value, "prefill_ms": pre_avg} if args.only == "prefill" else
                    {"decode_gbs": dec_value, "decode_ms": dec_avg, "decode_frac": dec_achieved / hbm_peak,
                     "rows": B, "num_splits": S})
            print(json.dumps({"only": args.only, **half}), flush=True)
        return

    # ---- end to end through the public API, host buffers ----
    e2e = None
    dec_e2e = None
    if not args.no_e2e:
        hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
        ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        hdq = dq.cpu().pin_memory()
        htab, hseq = table.cpu().pin_memory(), seq.cpu().pin_memory()
        hdo = torch.empty(do.shape, dtype=do.dtype).pin_memory()
        hdl = torch.empty(dlse.shape, dtype=dlse.dtype).pin_memory()
        ddq, dtab, dseq = torch.empty_like(dq), torch.empty_like(table), torch.empty_like(seq)

        # Host-buffer entry point: the copies in and out run inside the call,
        # pipelined over groups of KV heads against the attention.
        hscratch = torch.empty(attn.attn_prefill_host_scratch_bytes(PREFILL.T, PREFILL.h, PREFILL.h_kv,
                                                                    PREFILL.d_h), dtype=torch.uint8, device=dev)

        def e2e_prefill():
            attn.attn_prefill_host(hq, hk, hv, True, PREFILL.scale, o=ho, lse=hl, scratch=hscratch)

        def e2e_decode():
            ddq.copy_(hdq, non_blocking=True)
            dtab.copy_(htab, non_blocking=True)
            dseq.copy_(hseq, non_blocking=True)
            attn.attn_decode_paged(ddq, kc, vc, dtab, dseq, S, DECODE.scale, workspace=ws, o=do, lse=dlse)
            hdo.copy_(do, non_blocking=True)
            hdl.copy_(dlse, non_blocking=True)

        n_e2e = max(3, min(args.steps, 20))
        for fn, name in ((e2e_prefill, "p"), (e2e_decode, "d")):
            for _ in range(2):
                flush.fill_(1)
                fn()
            torch.cuda.synchronize()
            ms = []
            for _ in range(n_e2e):
                flush.fill_(1)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                b.synchronize()
                ms.append(a.elapsed_time(b))
            avg = max_over_ranks(sum(ms) / len(ms), world)
            if name == "p":
                e2e = {"value": world * pf / (avg * 1e-3) / 1e12, "unit": "TFLOP/s",
                       "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in (hq, hk, hv)),
                       "d2h_bytes_per_step": ho.numel() * ho.element_size() + hl.numel() * hl.element_size(),
                       "ms": avg}
            else:
                dec_e2e = {"value": world * db / (avg * 1e-3) / 1e9, "unit": "GB/s",
                           "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in (hdq, htab, hseq)),
                           "d2h_bytes_per_step": hdo.numel() * hdo.element_size() + hdl.numel() * hdl.element_size(),
                           "ms": avg}

    # ---- deterministic decode (fixed 2048-key splits) on the same batch, outside the step ----
    det = None
    if args.only is None and not args.no_extras:
        pps = 128
        det_splits = -(-table.shape[1] // pps)
        det_ws = torch.empty(attn.attn_decode_workspace_bytes(B, DECODE.h, det_splits, DECODE.d_h),
                             dtype=torch.uint8, device=dev)
        for _ in range(3):
            attn.attn_decode_paged_deterministic(dq, kc, vc, table, seq, pps, DECODE.scale,
                                                 workspace=det_ws, o=do, lse=dlse)
        dms = []
        for _ in range(20):
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(stream)
            attn.attn_decode_paged_deterministic(dq, kc, vc, table, seq, pps, DECODE.scale,
                                                 workspace=det_ws, o=do, lse=dlse)
            b_.record(stream)
            b_.synchronize()
            dms.append(a_.elapsed_time(b_))
        dt = statistics.median(dms)
        det = {"value": db / (dt * 1e-3) / 1e9, "unit": "GB/s", "ms": dt, "pages_per_split": pps,
               "num_splits": det_splits, "frac_of_hbm": db / (dt * 1e-3) / 1e9 / hbm_peak}

    # ---- adaptive decode (split count planned on the device, grid of 32), outside the step ----
    adaptive = None
    if args.only is None and not args.no_extras:
        amax = 32
        ad_ws = torch.empty(attn.attn_decode_adaptive_workspace_bytes(B, DECODE.h, amax, DECODE.d_h),
                            dtype=torch.uint8, device=dev)
        for _ in range(3):
            attn.attn_decode_paged_adaptive(dq, kc, vc, table, seq, amax, DECODE.scale,
                                            workspace=ad_ws, o=do, lse=dlse)
        ams = []
        for _ in range(20):
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(stream)
            attn.attn_decode_paged_adaptive(dq, kc, vc, table, seq, amax, DECODE.scale,
                                            workspace=ad_ws, o=do, lse=dlse)
            b_.record(stream)
            b_.synchronize()
            ams.append(a_.elapsed_time(b_))
        at = statistics.median(ams)
        off = attn.attn_decode_workspace_bytes(B, DECODE.h, amax, DECODE.d_h)
        adaptive = {"value": db / (at * 1e-3) / 1e9, "unit": "GB/s", "ms": at, "max_splits": amax,
                    "device_pages_per_split": int(ad_ws[off:off + 4].view(torch.int32).item()),
                    "frac_of_hbm": db / (at * 1e-3) / 1e9 / hbm_peak}

    # ---- pairwise (O, LSE) merge (prefix / suffix combine), outside the step ----
    extras = args.only is None and not args.no_extras
    merge_pair = measure_merge_pair(dev, flush, hbm_peak, peak_kind) if extras else None
    decode_b1 = measure_decode_batch1(dev, hbm_peak, peak_kind) if extras else None
    prefill_2048 = measure_prefill_t2048(dev, flush, tc_peak, peak_kind) if extras else None
    prefill_paged = measure_prefill_paged(dev, flush, tc_peak, peak_kind) if extras else None
    mixed = measure_mixed(dev, flush, hbm_peak, tc_peak, peak_kind) if extras else None

    # ---- CPU oracle baseline (rank 0, N = 1 only) ----
    cpu = None
    dec_cpu = None
    cpu_rows_n = 0
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        torch.set_num_threads(cpu_cores())
        qc, kc_, vc_ = q.cpu(), k.cpu(), v.cpu()
        t_tot, f_tot, n = 0.0, 0.0, 0
        while t_tot < args.cpu_seconds / 2 and n < 200:
            dt, fl = oracle_prefill_sample(qc, kc_, vc_, 64, seed=n)
            t_tot += dt
            f_tot += fl
            n += 1
        cpu_rows_n = n
        cpu = {"value": f_tot / t_tot / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{n} x 64 causal query rows of one head at T=8192 (float64 materialised softmax)"}
        order = np.argsort(lens)
        rows = [int(order[len(order) // 2])]
        kcc, vcc, dqc, tabc, seqc = kc.cpu(), vc.cpu(), dq.cpu(), table.cpu(), seq.cpu()
        tt, bb, m = 0.0, 0, 0
        while tt < args.cpu_seconds / 2 and m < 64:
            dt, by = oracle_decode_sample(dqc, kcc, vcc, tabc, seqc, rows)
            tt += dt
            bb += by
            m += 1
        dec_cpu = {"value": bb / tt / 1e9, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
                   "sample": f"{m} x one median-length row of the paged batch (float64)"}

    if rank != 0:
        return
    detail = {
        "prefill": {"ms": pre_avg, "flops": pf, "T": PREFILL.T, "h": PREFILL.h, "h_kv": PREFILL.h_kv,
                    "d_h": PREFILL.d_h, "causal": True, "e2e": e2e, "cpu_baseline": cpu},
        "decode": {"value": dec_value, "unit": "GB/s", "ms": dec_avg, "B": B, "num_splits": S,
                   "kv_tokens": sum(lens), "bytes": db, "traffic": traffic_for("decode"),
                   "e2e": dec_e2e, "cpu_baseline": dec_cpu, "deterministic": det,
                   "adaptive": adaptive},
        "merge_pair": merge_pair, "decode_batch1": decode_b1, "prefill_T2048": prefill_2048,
        "prefill_paged": prefill_paged, "mixed": mixed, "clocks": clk,
    }
    # The full record goes to stderr; stdout carries one short line.
    print("bench detail: " + json.dumps(detail), file=sys.stderr, flush=True)

    line = bench_line(
        world=world, steps=args.steps, warmup=args.warmup, value=value, dec_value=dec_value,
        dec_frac=dec_achieved / hbm_peak, step_ms=step_ms, S=S, pre_achieved=pre_achieved,
        tc_peak=tc_peak, traffic=traffic_for("prefill"), e2e=e2e, cpu=cpu, cpu_rows_n=cpu_rows_n,
        # prefill: V-to-fp16 pass + attention kernel; decode: split kernel + merge
        launches=(2 * int(do_pre) + 2 * int(do_dec)) * args.steps, clk=clk, dec_avg=dec_avg,
        dec_e2e=dec_e2e, det=det, adaptive=adaptive, prefill_2048=prefill_2048,
        prefill_paged=prefill_paged, merge_pair=merge_pair, mixed=mixed, decode_b1=decode_b1)
    print(json.dumps(line), flush=True)


def measure_prefill_paged(dev, flush, tc_peak, peak_kind, iters=10):
    """Chunked prefill over a paged cache: 8 rows, each with its last 1024
    positions as new queries over an 8192-key context (h=32, h_kv=8, d_h=128,
    Q and K x3 as in the main prefill workload). TFLOP/s of allowed pairs,
    L2 flushed before each call; the time includes the fp16 V copy."""
    import online_softmax_attn_gb300 as attn

    B, qn, ctx = 8, 1024, PREFILL.T
    h, h_kv, d = PREFILL.h, PREFILL.h_kv, PREFILL.d_h
    table, nblk = W.paged_layout([ctx] * B, seed=11)
    q = W.normal((B * qn, h, d), 31, torch.bfloat16, dev, PREFILL.qk_mult)
    kc = W.normal((nblk, W.PAGE_SIZE, h_kv, d), 32, torch.bfloat16, dev, PREFILL.qk_mult)
    vc = W.normal((nblk, W.PAGE_SIZE, h_kv, d), 33, torch.bfloat16, dev)
    cu = torch.arange(0, (B + 1) * qn, qn, dtype=torch.int32, device=dev)
    seq = torch.full((B,), ctx, dtype=torch.int32, device=dev)
    table = table.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((B * qn, h), dtype=torch.float32, device=dev)
    # The workspace with room for the fp16 V copy (the pre-pass that fills it
    # runs inside every timed call).
    ws = torch.empty(attn.attn_prefill_paged_workspace_bytes(B, table.shape[1], h_kv, d, v16=True),
                     dtype=torch.uint8, device=dev)
    call = lambda: attn.attn_prefill_paged(q, kc, vc, table, cu, seq, qn, True, PREFILL.scale,
                                           workspace=ws, o=o, lse=lse)
    for _ in range(3):
        call()
    ms = []
    for _ in range(iters):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        b.record()
        b.synchronize()
        ms.append(a.elapsed_time(b))
    t = statistics.median(ms)
    pairs = B * sum(ctx - qn + i + 1 for i in range(qn))
    flops = 4.0 * h * d * pairs
    tf = flops / (t * 1e-3) / 1e12
    return {"value": tf, "unit": "TFLOP/s", "ms": t, "rows": B, "queries_per_row": qn, "context": ctx,
            "flops": flops,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": tc_peak, "unit": "TFLOP/s",
                         "frac": tf / tc_peak, "traffic": traffic_for("prefill_paged"),
                         "kernel": "prefill_bf16_kernel (paged)",
                         "peak_source": f"{peak_kind} bf16 burst"}}


def measure_mixed(dev, flush, hbm_peak, tc_peak, peak_kind, iters=10):
    """A mixed serving step through attn_prefill_paged: 4 chunked-prefill rows
    (the last 1024 of 8192 positions each, causal) and 64 decode rows over
    seeded lengths U[4096, 16384], h=32, h_kv=8, d_h=128, bf16, the decode
    rows routed to the split-KV decode (at most 32 splits). Timed with events
    after an L2 flush: the mixed call, the 4 prefill rows alone, and
    attn_decode_paged on the 64 decode rows alone. The decode rows' GB/s is
    their KV bytes over (mixed - prefill alone)."""
    import online_softmax_attn_gb300 as attn

    h, h_kv, d, P = PREFILL.h, PREFILL.h_kv, PREFILL.d_h, W.PAGE_SIZE
    n_pre, qn, ctx = 4, 1024, PREFILL.T
    g = torch.Generator().manual_seed(41)
    dec_lens = torch.randint(4096, 16385, (64,), generator=g).tolist()
    lens = [ctx] * n_pre + dec_lens
    q_lens = [qn] * n_pre + [1] * 64
    table, nblk = W.paged_layout(lens, seed=43)
    kc = W.normal((nblk, P, h_kv, d), 44, torch.bfloat16, dev)
    vc = W.normal((nblk, P, h_kv, d), 45, torch.bfloat16, dev)
    total_q = sum(q_lens)
    q = W.normal((total_q, h, d), 46, torch.bfloat16, dev)
    cu = torch.tensor([0] + list(np.cumsum(q_lens)), dtype=torch.int32, device=dev)
    seq = torch.tensor(lens, dtype=torch.int32, device=dev)
    table = table.to(dev)
    B, mb = len(lens), table.shape[1]
    o = torch.empty_like(q)
    lse = torch.empty((total_q, h), dtype=torch.float32, device=dev)
    dsplit = 32
    ws = torch.empty(attn.attn_prefill_paged_decode_workspace_bytes(B, h, dsplit, d) +
                     attn.attn_prefill_paged_workspace_bytes(B, mb, h_kv, d, v16=True),
                     dtype=torch.uint8, device=dev)
    # the prefill rows alone
    pq = q[:n_pre * qn]
    po, pl = torch.empty_like(pq), torch.empty((n_pre * qn, h), dtype=torch.float32, device=dev)
    pws = torch.empty(attn.attn_prefill_paged_workspace_bytes(n_pre, mb, h_kv, d, v16=True),
                      dtype=torch.uint8, device=dev)
    pcu, pseq, ptab = cu[:n_pre + 1].contiguous(), seq[:n_pre].contiguous(), table[:n_pre].contiguous()
    # the decode rows alone
    dq = q[n_pre * qn:].contiguous()
    dseq, dtab = seq[n_pre:].contiguous(), table[n_pre:].contiguous()
    S = attn.attn_recommended_splits_ragged(64, h_kv, max(dec_lens), sum(dec_lens))
    dws = torch.empty(attn.attn_decode_workspace_bytes(64, h, S, d), dtype=torch.uint8, device=dev)
    do, dl = torch.empty_like(dq), torch.empty((64, h), dtype=torch.float32, device=dev)
    calls = {
        "mixed": lambda: attn.attn_prefill_paged(q, kc, vc, table, cu, seq, qn, True, PREFILL.scale,
                                                 workspace=ws, o=o, lse=lse, decode_splits=dsplit),
        "prefill": lambda: attn.attn_prefill_paged(pq, kc, vc, ptab, pcu, pseq, qn, True, PREFILL.scale,
                                                   workspace=pws, o=po, lse=pl),
        "decode": lambda: attn.attn_decode_paged(dq, kc, vc, dtab, dseq, S, PREFILL.scale,
                                                 workspace=dws, o=do, lse=dl),
    }
    t = {}
    for name, fn in calls.items():
        for _ in range(3):
            fn()
        ms = []
        for _ in range(iters):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            ms.append(a.elapsed_time(b))
        t[name] = statistics.median(ms)
    pairs = n_pre * sum(ctx - qn + i + 1 for i in range(qn))
    pf = 4.0 * h * d * pairs
    db = decode_bytes(dec_lens, DECODE)
    dec_ms = max(t["mixed"] - t["prefill"], 1e-6)
    return {"ms": t["mixed"], "prefill_alone_ms": t["prefill"], "decode_alone_ms": t["decode"],
            "prefill_tflops": pf / (t["prefill"] * 1e-3) / 1e12,
            "decode_rows_gbs": db / (dec_ms * 1e-3) / 1e9,
            "decode_alone_gbs": db / (t["decode"] * 1e-3) / 1e9, "decode_alone_splits": S,
            "rows": {"prefill": f"{n_pre} x {qn} queries over {ctx} keys", "decode": "64 x U[4096, 16384]"},
            "hbm_peak": hbm_peak, "tc_peak": tc_peak, "peak_source": peak_kind}


def measure_prefill_t2048(dev, flush, tc_peak, peak_kind, iters=15):
    """The T=2048 causal GQA layer (h=32, h_kv=8, d_h=128, bf16 N(0,1)): a
    call is ~40 us, so it is timed two ways -- an event pair around one call
    after an L2 flush, and a CUDA graph of back-to-back calls whose inputs
    rotate over copies larger than three times L2."""
    import online_softmax_attn_gb300 as attn

    sh = W.GQA_T2048_CAUSAL
    q, k, v = W.prefill_inputs(sh, 0, device=dev)
    flops = prefill_flops(sh)
    ws = torch.empty(attn.attn_prefill_workspace_bytes(sh.T, sh.h_kv, sh.d_h), dtype=torch.uint8,
                     device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((sh.h, sh.T), dtype=torch.float32, device=dev)
    for _ in range(3):
        attn.attn_prefill(q, k, v, True, sh.scale, o=o, lse=lse, workspace=ws)
    ms = []
    for _ in range(iters):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        attn.attn_prefill(q, k, v, True, sh.scale, o=o, lse=lse, workspace=ws)
        b.record()
        b.synchronize()
        ms.append(a.elapsed_time(b))
    t_ev = statistics.median(ms)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per = (q.numel() + k.numel() + v.numel()) * q.element_size() * 2  # inputs and output
    copies = max(2, -(-3 * l2 // per))
    sets = [(q.clone(), k.clone(), v.clone(), torch.empty_like(o), torch.empty_like(lse))
            for _ in range(copies)]
    n = 4 * copies

    def calls():
        for i in range(n):
            q_, k_, v_, o_, l_ = sets[i % copies]
            attn.attn_prefill(q_, k_, v_, True, sh.scale, o=o_, lse=l_, workspace=ws)

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        calls()
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            calls()
    graph.replay()
    torch.cuda.synchronize(dev)
    gms = []
    for _ in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        graph.replay()
        b.record()
        b.synchronize()
        gms.append(a.elapsed_time(b) / n)
    t_g = statistics.median(gms)
    tf = flops / (t_g * 1e-3) / 1e12
    return {"value": tf, "unit": "TFLOP/s", "us_per_call": t_g * 1e3, "flops": flops,
            "timing": f"CUDA graph of {n} calls", "event_single_call_us": t_ev * 1e3,
            "event_single_call_tflops": flops / (t_ev * 1e-3) / 1e12,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": tc_peak, "unit": "TFLOP/s",
                         "frac": tf / tc_peak, "traffic": traffic_for("prefill_T2048"),
                         "kernel": "prefill_bf16_kernel",
                         "peak_source": f"{peak_kind} bf16 burst"}}


def measure_decode_batch1(dev, hbm_peak, peak_kind):
    """Batch-1 decode (one query token per call) over a contiguous 32768-key
    cache: h=32 / h_kv=8 at 16 splits, and the 70B tensor-parallel shard
    h=8 / h_kv=1 at 132 splits. A single call is a few microseconds, so each
    is timed as a CUDA graph of back-to-back calls whose KV caches rotate over
    copies larger than twice L2 (every call reads its cache from HBM)."""
    import online_softmax_attn_gb300 as attn

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    out = {}
    for shape, splits in ((W.DECODE_S32K, 16), (W.DECODE_70B_TP8, 132)):
        q, kc, vc, tab, seq = W.decode_inputs(shape, 0, device=dev, contiguous=True)
        tab, seq = tab.to(dev), seq.to(dev)
        lens = seq.tolist()
        nbytes = decode_bytes(lens, shape)
        kv = kc.numel() * kc.element_size() * 2
        copies = max(2, -(-2 * l2 // kv))
        caches = [(kc.clone(), vc.clone()) for _ in range(copies)]
        ws = torch.empty(max(attn.attn_decode_workspace_bytes(1, shape.h, splits, shape.d_h), 256),
                         dtype=torch.uint8, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((1, shape.h), dtype=torch.float32, device=dev)
        n = 4 * copies

        def calls():
            for i in range(n):
                k_, v_ = caches[i % copies]
                attn.attn_decode_paged(q, k_, v_, tab, seq, splits, shape.scale, workspace=ws, o=o, lse=lse)

        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            calls()  # warm-up outside the capture
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                calls()
        graph.replay()
        torch.cuda.synchronize(dev)
        ms = []
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            graph.replay()
            b.record()
            b.synchronize()
            ms.append(a.elapsed_time(b) / n)
        t = statistics.median(ms)
        gbs = nbytes / (t * 1e-3) / 1e9
        out[shape.name] = {"us_per_call": t * 1e3, "value": gbs, "unit": "GB/s", "num_splits": splits,
                           "kv_bytes": nbytes, "frac_of_hbm": gbs / hbm_peak,
                           "peak_source": f"{peak_kind} copy bandwidth", "timing": f"CUDA graph of {n} calls"}
        del caches, graph
    return out


def measure_merge_pair(dev, flush, hbm_peak, peak_kind, iters=20):
    """Pairwise (O, LSE) merge of two prefill-shaped results (32 heads x 8192
    tokens, d_h 128, bf16 in and out): the prefix / suffix combine. HBM-bound;
    204 MB per call. A single call is ~35 us, so the host's launch time would
    show in an event pair around one call: the calls are timed as a CUDA graph
    of back-to-back calls alternating between two input sets (268 MB of
    inputs, twice L2), so every call reads its inputs from HBM. `flush` is
    unused (kept for the common signature)."""
    import online_softmax_attn_gb300 as attn

    rows, d = PREFILL.h * PREFILL.T, PREFILL.d_h
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    sets = []
    for _ in range(2):
        oa = torch.randn(rows, d, generator=g, device=dev).to(torch.bfloat16)
        ob = torch.randn(rows, d, generator=g, device=dev).to(torch.bfloat16)
        la = torch.randn(rows, generator=g, device=dev) * 20
        lb = torch.randn(rows, generator=g, device=dev) * 20
        sets.append((oa, la, ob, lb))
    o = torch.empty_like(sets[0][0])
    lse = torch.empty_like(sets[0][1])
    n = 10

    def calls():
        for i in range(n):
            oa, la, ob, lb = sets[i % 2]
            attn.attn_merge_lse_pair(oa, la, ob, lb, o=o, lse=lse)

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        calls()  # warm-up outside the capture
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            calls()
    graph.replay()
    torch.cuda.synchronize(dev)
    ms = []
    for _ in range(max(3, iters)):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        graph.replay()
        b.record()
        b.synchronize()
        ms.append(a.elapsed_time(b) / n)
    t = statistics.median(ms)
    nbytes = rows * (2 * d * 2 + 2 * 4 + d * 2 + 4)
    gbs = nbytes / (t * 1e-3) / 1e9
    return {"value": gbs, "unit": "GB/s", "ms": t, "rows": rows, "d_h": d, "bytes": nbytes,
            "timing": f"CUDA graph of {n} calls",
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": gbs / hbm_peak, "traffic": traffic_for("merge_pair"),
                         "kernel": "merge_pair_kernel", "peak_source": f"{peak_kind} copy bandwidth"}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=16.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--clocks-dir", default=None,
                    help="where to keep the raw nvidia-smi clock samples (default: the temp directory)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the measurements outside the step (deterministic / adaptive decode, "
                         "pair merge, paged prefill), e.g. for a launch list of the step alone")
    ap.add_argument("--only", choices=["prefill", "decode", "prefill_paged", "merge_pair", "decode_batch1",
                                       "mixed", "prefill_t2048"],
                    default=None,
                    help="run one half of the step, or the paged prefill or pair merge measurement "
                         "alone (profiler captures; not a bench line)")
    ap.add_argument("--decode-rows", type=int, default=0,
                    help="truncate the decode batch (profiler captures; not a bench line)")
    args = ap.parse_args()
    if args.only or args.decode_rows:
        args.no_e2e = True
        args.no_cpu_baseline = True
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_gpu(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python3
"""Decode-attention benchmark: tokens/s and achieved HBM GB/s on one GB300.

A step is one fa_decode_run over one resident batch: the split-KV decode
kernel plus the merge kernel of split requests.  The plan (host work list,
one host-to-device copy) is amortised per batch, as the plan/run split
intends; it is timed separately and it is inside the end-to-end number.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--no-cpu-baseline]

Prints one JSON line (rank 0).  Workloads are the seeded synthetic batches of
paged_kv_decode_fa_gb300.workloads; the default is the largest one, the
heterogeneous ragged batch (B=450, 32 qo / 8 kv heads, head_dim 128, bf16,
lengths log-uniform in [256, 64000], 21.5 GB of KV).  The other decode
workloads are measured in the same run and reported under "other_workloads",
each with its own algorithmic bytes, kernel time and roofline fraction.  With
--impl reference the float64 CPU oracle is timed instead, on the host cores,
over bounded samples of the same workload.  Under torchrun (N > 1) each rank
runs an independent replica of the workload on its own GPU (the path has no
exchange step); value is the tokens of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_decode_fa_gb300 import workloads as W  # noqa: E402

METRIC = "decode attention tokens/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
DTYPE_NAMES = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16",
               torch.float8_e4m3fn: "e4m3"}
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ helpers

def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def algorithmic_bytes(b: W.DecodeBatch) -> int:
    """Bytes any decode implementation must move for this batch: K and V of
    every valid token and kv head, the page ids, q, o and lse."""
    kv_es = b.paged_kv.element_size()
    q_es = b.q.element_size()
    kv = b.total_tokens * b.num_kv_heads * 2 * b.head_dim * kv_es
    if "k_scales" in b.extra:          # one fp32 K and one V scale per token and kv head
        kv += b.total_tokens * b.num_kv_heads * 2 * 4
    idx = int(b.indptr[-1]) * 4
    qo = 2 * b.q.numel() * q_es                     # q read, o written (any q layout)
    lse = b.q.numel() // b.head_dim * 4
    if "qo_indptr" in b.extra:                       # a ragged plan's row boundaries
        idx += (b.batch + 1) * 4
    return int(kv + idx + qo + lse)


def query_rows(b: W.DecodeBatch) -> int:
    """Query tokens of one step: B, B * q_len, or the ragged rows."""
    return b.q.numel() // (b.num_qo_heads * b.head_dim)


def read_bf16_peak():
    """Dense bf16 tensor TFLOP/s of this GPU: the measured burst figure (the
    prefix kernel is timed alone, within a short step), else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            v = json.load(f).get("bf16_tflops")
        if v:
            return float(v), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except (OSError, ValueError):
        pass
    return 1900.0, "fallback (1.9 PFLOP/s bf16 burst, one earlier GB300 measurement)"


# Sources that are not part of the decode kernels or their launch: the
# cascade's own kernels, the no-allocation entry point, fa_merge_states.
NOT_DECODE_SOURCES = ("cascade.cu", "cascade_tc.cuh", "static_scratch.cu", "merge.cu")


def kernel_source_hash(workload: str = "gqa_uniform") -> str:
    """Hash of the code a workload's kernels are built and launched from,
    comments and layout left out (a profile summary is current while this
    hash matches: a changed comment changes no kernel)."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_decode_fa_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        if not fn.endswith((".cu", ".cuh", ".h", ".cpp")):
            continue
        if workload != "cascade" and fn in NOT_DECODE_SOURCES:
            continue
        with open(os.path.join(csrc, fn), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        text = " ".join(text.split())
        h.update(fn.encode() + text.encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the workload's dominant kernel from the
    committed ncu figures (profiles/traffic.json), if they were taken on the
    current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        entry = json.load(f).get("workloads", {}).get(workload)
    if not entry or entry.get("kernel_source_hash") != kernel_source_hash(workload):
        return None
    return float(entry["traffic_bytes_per_launch"])


class ClockSampler:
    """SM clock and clock-event-reason samples while running: read through
    NVML (ctypes, read-only queries) every 2 ms, else from an nvidia-smi
    stream every 50 ms."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits: sw power cap, hw slowdown, sw thermal, hw thermal
    _BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
             "hw_thermal_slowdown": 0x40}

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None
        self.stop_flag = threading.Event()
        self.source = None

    def _nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(h)) != 0:
            return None
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        mhz, mx, mem, mask = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()

        def read():
            # clock types: 1 = SM, 2 = memory
            if (lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) != 0 or
                    lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) != 0 or
                    reasons(h, ctypes.byref(mask)) != 0):
                return None
            mem_mhz = str(mem.value) if lib.nvmlDeviceGetClockInfo(h, 2, ctypes.byref(mem)) == 0 \
                else ""
            flags = ["Active" if mask.value & b else "Not Active" for b in
                     (self._BITS["hw_slowdown"], self._BITS["hw_thermal_slowdown"],
                      self._BITS["sw_thermal_slowdown"], self._BITS["sw_power_cap"])]
            return ", ".join([str(self.gpu), str(mhz.value), str(mx.value), "", mem_mhz] + flags)
        return read if read() is not None else None

    def start(self):
        try:
            read = self._nvml()
        except (OSError, AttributeError):
            read = None
        if read is not None:
            self.source = "nvml, 2 ms"

            def loop():
                while not self.stop_flag.is_set():
                    line = read()
                    if line is not None:
                        self.samples.append((time.perf_counter(), line))
                    time.sleep(0.002)
            self.thread = threading.Thread(target=loop, daemon=True)
            self.thread.start()
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.source = "nvidia-smi, 50 ms"
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.perf_counter(), line.strip()))

    def stop(self):
        self.stop_flag.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        rows = []
        for t, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                row = (t, float(parts[1]), float(parts[2]), parts[5:9])
            except ValueError:
                continue
            try:  # memory clock (NVML samples only)
                row += (float(parts[4]),)
            except ValueError:
                pass
            rows.append(row)
        # samples inside the region (nvidia-smi's 50 ms stream: within one
        # interval of it)
        margin = 0.005 if self.source and self.source.startswith("nvml") else 0.05
        window = [r for r in rows if t0 - margin <= r[0] <= t1 + margin]
        which = "timed"
        if not window:
            window, which = rows, "warmup+timed"
        if not window:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in window for i, v in enumerate(r[3])
                          if v.lower() == "active"})
        out = {"sm_mhz": statistics.median(r[1] for r in window),
               "sm_max_mhz": max(r[2] for r in window), "reasons": reasons,
               "samples": len(window), "window": which, "source": self.source}
        mem = [r[4] for r in window if len(r) > 4]
        if mem:
            out["mem_mhz"] = statistics.median(mem)
        return out


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, units_per_rank_step: int, steps: int, elapsed_s: float) -> float:
    """Units per second of the whole job: every rank processes the same units
    per step (weak scaling), elapsed_s is the slowest rank's time."""
    return world * units_per_rank_step * steps / elapsed_s


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ oracle timing

def oracle_timing(b: W.DecodeBatch, target_s: float, max_requests: int | None = None):
    """Time the float64 oracle on a sample of whole requests of b sized to take
    about target_s seconds on all host cores.  Returns (requests, seconds,
    tokens, threads, description, algorithmic bytes of the sample)."""
    import oracle
    from tests.helpers import oracle_decode, sub_batch  # test-side marshalling
    order = list(np.random.default_rng(0).permutation(b.batch))
    one = sub_batch(b, order[:1])
    t = time.perf_counter()
    oracle_decode(one)
    t1 = max(time.perf_counter() - t, 1e-4)
    n = int(max(1, min(b.batch if max_requests is None else max_requests, target_s / t1)))
    sb = sub_batch(b, order[:n])
    t = time.perf_counter()
    oracle_decode(sb)
    dt = time.perf_counter() - t
    threads = oracle.max_threads()
    desc = (f"{n} of {b.batch} requests ({int(sb.lengths.sum())} KV tokens), seeded random "
            f"choice, float64 C oracle, OpenMP {threads} threads")
    return query_rows(sb), dt, int(sb.lengths.sum()), threads, desc, algorithmic_bytes(sb)


# ------------------------------------------------------------------ arms

def bench_reference(args, world, rank):
    """The oracle as the reference arm: K timed steps, each a bounded sample."""
    if rank != 0:
        return None
    # inputs drawn where the timed arm draws them (the same values); only
    # the sampled requests are copied to the host for the oracle
    b = W.make_config_batch(args.workload,
                            device="cuda" if torch.cuda.is_available() else "cpu")
    import oracle
    from tests.helpers import oracle_decode, sub_batch
    budget = 150.0
    order = list(np.random.default_rng(0).permutation(b.batch))
    one = sub_batch(b, order[:1])
    t = time.perf_counter()
    oracle_decode(one)
    t1 = max(time.perf_counter() - t, 1e-4)
    per_step = budget / max(1, args.steps + args.warmup)
    n = int(max(1, min(b.batch, per_step / t1)))
    sb = sub_batch(b, order[:n])
    for _ in range(args.warmup):
        oracle_decode(sb)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_decode(sb)
    dt = time.perf_counter() - t
    value = query_rows(sb) * args.steps / dt
    threads = oracle.max_threads()
    cfg = W.CONFIGS[args.workload]
    desc = f"{n} of {b.batch} requests per step, float64 C oracle, OpenMP {threads} threads"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(cfg, b),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def config_dict(cfg: W.DecodeConfig, b: W.DecodeBatch) -> dict:
    kv_bytes = int(b.total_tokens * cfg.num_kv_heads * 2 * cfg.head_dim *
                   b.paged_kv.element_size())
    return {"workload": cfg.name, "batch": b.batch, "num_qo_heads": cfg.num_qo_heads,
            "num_kv_heads": cfg.num_kv_heads, "head_dim": cfg.head_dim,
            "page_size": cfg.page_size, "q_len": cfg.q_len, "q_dtype": DTYPE_NAMES[cfg.q_dtype],
            "kv_dtype": DTYPE_NAMES[cfg.kv_dtype],
            "kv_tokens": b.total_tokens, "mean_seq_len": round(b.total_tokens / max(1, b.batch), 1),
            "query_tokens": query_rows(b),
            "kv_bytes": kv_bytes,
            "l2": ("inputs larger than L2 (129 MB): the KV read each step exceeds it"
                   if kv_bytes > 129e6 else
                   f"L2-resident ({kv_bytes / 1e6:.1f} MB of KV): a launch-bound correctness "
                   "case; its HBM fraction is not a bandwidth figure"),
            "parallelism": "replicas (one independent batch per GPU)",
            "softmax": ("unified max against a static Cauchy-Schwarz logit bound"
                        if cfg.name == "gqa_unified_max" else "online (running max)")}


def cascade_bytes(b: W.DecodeBatch) -> int:
    """Algorithmic bytes of a cascade batch: the shared prefix once, every
    request's own tokens, page ids, q, o and lse."""
    es = b.paged_kv.element_size()
    npre = b.extra["prefix_pages"]
    own_tokens = int(b.lengths.sum()) - b.batch * npre * b.page_size
    kv = (npre * b.page_size + own_tokens) * b.num_kv_heads * 2 * b.head_dim * es
    idx = (int(b.indptr[-1]) - (b.batch - 1) * npre) * 4
    qo = 2 * b.batch * b.num_qo_heads * b.head_dim * b.q.element_size()
    return int(kv + idx + qo + b.batch * b.num_qo_heads * 4)


def bench_cascade(args, world, rank, local, b, cfg, dev):
    """Cascade decode of a shared-prefix batch, next to plain decode of the
    same batch (which reads the prefix once per request)."""
    import paged_kv_decode_fa_gb300 as fa
    stream = torch.cuda.current_stream(dev)
    pre, ip, idx, last = W.cascade_parts(b)
    t = time.perf_counter()
    p = fa.cascade_plan(pre, ip, idx, last, b.num_qo_heads, b.num_kv_heads, b.head_dim,
                        b.page_size, q_data_type=b.q.dtype)
    torch.cuda.synchronize(dev)
    plan_ms = (time.perf_counter() - t) * 1e3
    o = torch.empty_like(b.q)
    lse = torch.empty((b.batch, b.num_qo_heads), dtype=torch.float32, device=dev)
    plain = fa.plan(b.indptr, b.indices, b.last_page_len, b.num_qo_heads, b.num_kv_heads,
                    b.head_dim, b.page_size, q_data_type=b.q.dtype)

    def timed(fn, steps):
        for _ in range(args.warmup):
            fn()
        barrier(world)
        torch.cuda.synchronize(dev)
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        z.record(stream)
        torch.cuda.synchronize(dev)
        return max_over_ranks(a.elapsed_time(z) / 1e3, world, dev)

    # the production step: the prefix kernel on the plan's side stream,
    # alongside the suffix decode
    clocks = ClockSampler(local).start()
    time.sleep(0.3)
    t0 = time.perf_counter()
    elapsed_s = timed(lambda: p.run(b.q, b.paged_kv, out=o, lse=lse), args.steps)
    t1 = time.perf_counter()
    clocks.stop()
    # the prefix kernel alone: events around it in every step of a second
    # loop (a timed run keeps the kernel alone on the GPU, after the suffix
    # decode); recorded once by torch first so that they exist
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, z in evs:
        a.record(stream)
        z.record(stream)
    step_no = [0]

    def serial_step():
        i = step_no[0]
        step_no[0] += 1
        if i >= args.warmup:
            p.set_timing_events(*evs[i - args.warmup])
        p.run(b.q, b.paged_kv, out=o, lse=lse)

    serial_s = timed(serial_step, args.steps)
    p.set_timing_events(None, None)
    prefix_s = statistics.mean(a.elapsed_time(z) for a, z in evs) / 1e3
    if p.check() != 0:
        raise RuntimeError("device check flagged the cascade batch")
    plain_s = timed(lambda: plain.run(b.q, b.paged_kv, out=o, lse=lse), args.steps)
    # end to end: upload q, plan, run, read o and lse back
    q_h = b.q.cpu().pin_memory()
    q_d = torch.empty_like(b.q)
    o_h = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    ws = torch.empty(fa.library().fa_cascade_workspace_size(b.batch, b.num_qo_heads,
                                                            b.num_kv_heads, b.head_dim),
                     dtype=torch.uint8, device=dev)
    e2e_steps = max(1, min(args.steps, 200))

    def e2e_step():
        q_d.copy_(q_h, non_blocking=True)
        pe = fa.cascade_plan(pre, ip, idx, last, b.num_qo_heads, b.num_kv_heads, b.head_dim,
                             b.page_size, q_data_type=b.q.dtype, workspace=ws)
        pe.run(q_d, b.paged_kv, out=o, lse=lse)
        o_h.copy_(o, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)
        return pe

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize(dev)
    te = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    torch.cuda.synchronize(dev)
    e2e_s = max_over_ranks(time.perf_counter() - te, world, dev)
    alg = cascade_bytes(b)
    peak, peak_kind = read_peaks()
    step_s = elapsed_s / args.steps
    # the prefix kernel is a dense contraction: QK^T and P.V over the shared
    # tokens for every query head of the batch, 2 flops per multiply-add
    prefix_tokens = b.extra["prefix_pages"] * b.page_size
    prefix_flops = 2 * 2 * b.batch * b.num_qo_heads * prefix_tokens * b.head_dim
    prefix_bytes = prefix_tokens * b.num_kv_heads * 2 * b.head_dim * b.paged_kv.element_size()
    tflops_peak, tflops_kind = read_bf16_peak()
    return {
        "metric": METRIC, "value": whole_job_rate(world, b.batch, args.steps, elapsed_s), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE_NAMES[cfg.kv_dtype], "data": "synthetic",
        "config": dict(config_dict(cfg, b), prefix_pages=b.extra["prefix_pages"]),
        "hbm_gbs": alg / step_s / 1e9, "hbm_frac_of_peak": alg / step_s / 1e9 / peak,
        "peak_kind": peak_kind, "plan_ms": plan_ms,
        "serial_ms_per_step": serial_s / args.steps * 1e3,
        "plain_decode_ms_per_step": plain_s / args.steps * 1e3,
        "speedup_vs_plain_decode": plain_s / elapsed_s,
        "roofline": {"bound": "tensor", "achieved": prefix_flops / prefix_s / 1e12,
                     "peak": tflops_peak, "unit": "TFLOP/s",
                     "frac": prefix_flops / prefix_s / 1e12 / tflops_peak,
                     "traffic": profiled_traffic("cascade"),
                     "kernel": ("fa_prefix_kernel (mma.sync bf16)"
                                if os.environ.get("FADECODE_CASCADE") == "mma"
                                else "fa_prefix_tc_kernel (tcgen05 bf16, TMEM accumulators)"), "peak_kind": tflops_kind,
                     "flops_per_launch": prefix_flops,
                     "prefix_kernel_us": prefix_s * 1e6,
                     "prefix_hbm_gbs": prefix_bytes / prefix_s / 1e9},
        "e2e": {"value": whole_job_rate(world, b.batch, e2e_steps, e2e_s), "unit": "tokens/s",
                "h2d_bytes_per_step": int(q_h.numel() * q_h.element_size()),
                "d2h_bytes_per_step": int(o_h.numel() * o_h.element_size() + lse_h.numel() * 4),
                "steps": e2e_steps, "includes": "H2D q, cascade plan, run, D2H o + lse"},
        "gpu_launches": args.steps * 3,
        "clocks": clocks.summary(t0, t1),
    }


def plan_batch(fa, b: W.DecodeBatch, idx=None, ws=None):
    """Plan a decode batch (multi-token plans for q_len > 1, ragged-q plans
    for a per-request number of query tokens)."""
    idx = b.indices if idx is None else idx
    if "qo_indptr" in b.extra:
        return fa.plan_ragged_q(b.indptr.numpy(), idx, b.last_page_len.numpy(),
                                b.extra["qo_indptr"], b.num_qo_heads, b.num_kv_heads, b.head_dim,
                                b.page_size, q_data_type=b.q.dtype, kv_data_type=b.paged_kv.dtype,
                                workspace=ws)
    if b.q_len > 1:
        return fa.plan_multi_token(b.indptr.numpy(), idx, b.last_page_len.numpy(), b.q_len,
                                   b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size,
                                   q_data_type=b.q.dtype, kv_data_type=b.paged_kv.dtype,
                                   workspace=ws)
    return fa.plan(b.indptr.numpy(), idx, b.last_page_len.numpy(), b.num_qo_heads,
                   b.num_kv_heads, b.head_dim, b.page_size, q_data_type=b.q.dtype,
                   kv_data_type=b.paged_kv.dtype, workspace=ws)


def launches_per_run(p) -> int:
    """Kernel launches one run of a plan makes: one decode launch per bucket
    (one, or up to four for a ragged plan), and with the separate merge
    kernel one more after each decode launch that has split requests to
    fold."""
    info = p.info
    nb = info.get("num_buckets", 1)
    n = nb
    if info["num_merge_units"] > 0 and not info["fused_merge"]:
        cta, seg, _ = p.work()
        first = list(info["bucket_first_cta"][:nb]) + [info["num_ctas"]]
        for b in range(nb):
            n += int((seg[cta[first[b]]:cta[first[b + 1]], 6] >= 0).any())
    return n


def workspace_bytes(fa, b: W.DecodeBatch) -> int:
    """Workspace bound of the batch's plan kind."""
    G = b.num_qo_heads // b.num_kv_heads
    if "qo_indptr" in b.extra or G * b.q_len > 8:
        return int(fa.library().fa_decode_workspace_size_ragged_q(
            b.batch, b.num_qo_heads, b.num_kv_heads, b.head_dim))
    return fa.workspace_size(b.batch, b.num_qo_heads * b.q_len, b.num_kv_heads, b.head_dim)


def step_fn(name: str, b: W.DecodeBatch, um_bound):
    """The production run call of a workload: plan.run, the per-token-scale
    run, or the unified-max run against a static bound."""
    token_scales = "k_scales" in b.extra

    def run_step(plan, q, out, lse_out):
        if um_bound is not None:
            return plan.run_unified_max(q, b.paged_kv, um_bound, out=out, lse=lse_out)
        if token_scales:
            return plan.run_token_scales(q, b.paged_kv, b.extra["k_scales"], b.extra["v_scales"],
                                         out=out, lse=lse_out)
        return plan.run(q, b.paged_kv, k_scale=b.k_scale, v_scale=b.v_scale, out=out,
                        lse=lse_out)
    return run_step


# Decode workloads measured beside the headline one, in the same run.
OTHER_WORKLOADS = ("tiny", "gqa_uniform", "long_split", "fp8_kv", "fp8_kv_token_scales",
                   "spec_decode", "spec_decode_ragged", "gqa_unified_max", "cascade")


def measure_other(args, world, dev, name: str) -> dict:
    """One more decode workload: at least 100 timed steps after at least 10
    warm-ups (a region of a few 0.1 ms launches is too short to time well),
    the region's events over its launches as the kernel time, the workload's
    own algorithmic bytes, roofline fraction and (current) ncu traffic."""
    steps, warmup = max(args.steps, 100), max(args.warmup, 10)
    import paged_kv_decode_fa_gb300 as fa
    cfg = W.CONFIGS[name]
    b = W.make_config_batch(name, device=dev)
    if name == "cascade":
        sub = argparse.Namespace(**dict(vars(args), steps=steps, warmup=warmup))
        r = bench_cascade(sub, world, 0, dev.index, b, cfg, dev)
        keep = ("config", "value", "unit", "ms_per_step", "hbm_gbs", "hbm_frac_of_peak",
                "serial_ms_per_step", "plain_decode_ms_per_step", "speedup_vs_plain_decode",
                "roofline", "e2e", "steps", "warmup", "gpu_launches", "clocks")
        del b
        torch.cuda.empty_cache()
        return {k: r[k] for k in keep}
    stream = torch.cuda.current_stream(dev)
    p = plan_batch(fa, b)
    info = p.info
    o = torch.empty_like(b.q)
    lse = torch.empty(tuple(b.q.shape[:-1]), dtype=torch.float32, device=dev)
    um_bound = W.cauchy_schwarz_bound(b) if name == "gqa_unified_max" else None
    run_step = step_fn(name, b, um_bound)
    for _ in range(warmup):
        run_step(p, b.q, o, lse)
    torch.cuda.synchronize(dev)
    if p.check() != 0:
        raise RuntimeError(f"device check flagged the {name} batch")
    launches = launches_per_run(p)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index).start()
    time.sleep(0.05)
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    start.record(stream)
    for _ in range(steps):
        run_step(p, b.q, o, lse)
    end.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.perf_counter()
    clocks.stop()
    elapsed_s = max_over_ranks(start.elapsed_time(end) / 1e3, world, dev)
    step_s = elapsed_s / steps
    alg = algorithmic_bytes(b)
    peak, _ = read_peaks()
    res = {
        "config": config_dict(cfg, b),
        "value": whole_job_rate(world, query_rows(b), steps, elapsed_s),
        "unit": "tokens/s", "ms_per_step": step_s * 1e3,
        "kv_tokens_per_s": world * b.total_tokens * steps / elapsed_s,
        "hbm_gbs": alg / step_s / 1e9,
        "roofline": {"bound": "hbm", "achieved": alg / step_s / 1e9, "peak": peak,
                     "unit": "GB/s", "frac": alg / step_s / 1e9 / peak,
                     "traffic": profiled_traffic(name),
                     "kernel": ("fa_decode_mma_kernel" if info["tensor_cores"]
                                else "fa_decode_split_kernel"),
                     "algorithmic_bytes_per_launch": alg, "duration_us": step_s * 1e6,
                     "duration_from": ("timed-region events / launches" if launches == 1 else
                                       f"timed-region events / steps ({launches} launches a "
                                       "step: decode buckets and merge kernels)")},
        "steps": steps, "warmup": warmup, "gpu_launches": steps * launches,
        "clocks": clocks.summary(t0, t1),
    }
    if um_bound is not None:
        res["unified_max"] = {"bound": um_bound, "fallbacks": p.unified_max_fallbacks()}
    del p, b, o, lse
    torch.cuda.empty_cache()
    return res


def bench_ours(args, world, rank, local):
    import paged_kv_decode_fa_gb300 as fa
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = W.CONFIGS[args.workload]
    b = W.make_config_batch(args.workload, device=dev, max_requests=args.max_requests)
    if "prefix_pages" in b.extra:
        return bench_cascade(args, world, rank, local, b, cfg, dev)
    stream = torch.cuda.current_stream(dev)

    # plan (amortised), timed on the host including its upload: the first
    # plan of the process (occupancy queries, staging buffers) and the
    # median of later plans of the same batch
    torch.cuda.synchronize(dev)
    t = time.perf_counter()
    p = plan_batch(fa, b)
    torch.cuda.synchronize(dev)
    plan_ms = (time.perf_counter() - t) * 1e3
    info = p.info
    ws_warm = torch.empty(workspace_bytes(fa, b), dtype=torch.uint8, device=dev)
    warm = []
    for _ in range(50):
        t = time.perf_counter()
        pw = plan_batch(fa, b, ws=ws_warm)
        torch.cuda.synchronize(dev)
        warm.append((time.perf_counter() - t) * 1e3)
        del pw
    plan_ms_warm = statistics.median(warm)
    del ws_warm
    o = torch.empty_like(b.q)
    lse = torch.empty(tuple(b.q.shape[:-1]), dtype=torch.float32, device=dev)
    # unified max: a static logit bound, fixed before the timed region the
    # way an offline profile of the model would fix it
    um_bound = W.cauchy_schwarz_bound(b) if args.workload == "gqa_unified_max" else None
    run_step_fn = step_fn(args.workload, b, um_bound)

    def run_step(plan, q, out=o, lse_out=lse):
        return run_step_fn(plan, q, out, lse_out)

    def make_plan(idx, ws=None):
        return plan_batch(fa, b, idx, ws)

    for _ in range(args.warmup):
        run_step(p, b.q)
    torch.cuda.synchronize(dev)
    if p.check() != 0:
        raise RuntimeError("device check flagged the benchmark batch")
    if um_bound is not None:
        p.unified_max_fallbacks()  # clear the warm-up count

    launches_per_step = launches_per_run(p)
    # The timed region: the production step back to back, nothing recorded
    # between launches (an event pair around every launch adds its own
    # records between the kernels).
    clocks = ClockSampler(local).start()
    time.sleep(0.3)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    start.record(stream)
    for _ in range(args.steps):
        run_step(p, b.q)
    end.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.perf_counter()
    barrier(world)
    clocks.stop()
    um_fallbacks = p.unified_max_fallbacks() if um_bound is not None else None
    elapsed_s = start.elapsed_time(end) / 1e3
    elapsed_s = max_over_ranks(elapsed_s, world, dev)
    # The decode kernel alone: a second loop of the same length with the
    # library recording events around the kernel of every step (torch
    # creates an event at its first record, so each is recorded once first).
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, z in evs:
        a.record(stream)
        z.record(stream)
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        p.set_timing_events(*evs[i])
        run_step(p, b.q)
    torch.cuda.synchronize(dev)
    p.set_timing_events(None, None)
    kern_ms = [a.elapsed_time(z) for a, z in evs]
    kern_avg_s = statistics.mean(kern_ms) / 1e3
    kern_med_s = statistics.median(kern_ms) / 1e3
    # the dominant kernel's average duration inside the timed region: the
    # region's events over its launches when a step is that one launch, else
    # the per-launch events of the second loop
    if launches_per_step == 1:
        kern_region_s, duration_from = elapsed_s / args.steps, "timed-region events / launches"
    else:
        kern_region_s, duration_from = kern_avg_s, "events around each decode launch"

    # End to end through the public API with host buffers.  Every step plans
    # the batch and decodes it with q, the page ids, o and lse in page-locked
    # host memory: the kernels read q and the page ids and write o and lse
    # over the CPU-GPU link (NVLink-C2C on a GB300 node), so the step's
    # host-to-device and device-to-host traffic happens inside the timed
    # kernels and no staging copy is issued.  For comparison, the same step
    # with explicit pinned copies to and from device buffers on one stream.
    q_h = b.q.cpu().pin_memory()
    idx_h = b.indices.cpu().pin_memory()
    o_h = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    q_d = torch.empty_like(b.q)
    idx_d = torch.empty_like(b.indices)
    ws = torch.empty(workspace_bytes(fa, b), dtype=torch.uint8, device=dev)

    def e2e_step():
        pe = make_plan(idx_h, ws)
        run_step(pe, q_h, o_h, lse_h)
        return pe

    def staged_step():
        q_d.copy_(q_h, non_blocking=True)
        idx_d.copy_(idx_h, non_blocking=True)
        pe = make_plan(idx_d, ws)
        run_step(pe, q_d)
        o_h.copy_(o, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)
        return pe

    e2e_steps = max(1, min(args.steps, 200))

    def timed_e2e(step_fn):
        for _ in range(max(3, args.warmup)):
            step_fn()
        torch.cuda.synchronize(dev)
        barrier(world)
        te = time.perf_counter()
        for _ in range(e2e_steps):
            pe = step_fn()
        torch.cuda.synchronize(dev)
        return max_over_ranks(time.perf_counter() - te, world, dev), pe

    staged_s, _ = timed_e2e(staged_step)
    assert torch.equal(o_h, o.cpu()), "staged end-to-end output differs from the device run"
    o_h.zero_()
    e2e_s, pe = timed_e2e(e2e_step)
    assert torch.equal(o_h, o.cpu()), "end-to-end output differs from the device run"
    upload = pe.info["plan_upload_bytes"]
    h2d = q_h.numel() * q_h.element_size() + idx_h.numel() * 4 + upload
    d2h = o_h.numel() * o_h.element_size() + lse_h.numel() * 4

    alg = algorithmic_bytes(b)
    peak, peak_kind = read_peaks()
    step_s = elapsed_s / args.steps
    value = whole_job_rate(world, query_rows(b), args.steps, elapsed_s)
    achieved = alg / kern_region_s / 1e9
    traffic = profiled_traffic(args.workload) if args.max_requests is None else None
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": DTYPE_NAMES[cfg.kv_dtype] if cfg.kv_dtype != torch.float8_e4m3fn else "e4m3",
        "data": "synthetic", "config": config_dict(cfg, b),
        "kv_tokens_per_s": world * b.total_tokens * args.steps / elapsed_s,
        "hbm_gbs": alg / step_s / 1e9,
        "hbm_frac_of_peak": alg / step_s / 1e9 / peak,
        "hbm_frac_of_nominal_7900": alg / step_s / 1e9 / 7900.0,
        "peak_kind": peak_kind,
        "plan_ms": plan_ms,
        "plan_ms_warm": plan_ms_warm,
        "decode_kernel_us": {"mean": kern_avg_s * 1e6, "median": kern_med_s * 1e6,
                             "measured": "events around each launch, second loop"},
        "plan": {k: info[k] for k in ("num_ctas", "ctas_per_sm", "num_segments",
                                      "num_merge_units", "num_partial_slots", "stages",
                                      "threads_per_cta", "smem_bytes_per_cta",
                                      "tensor_cores", "fused_merge")},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": ("fa_decode_mma_kernel" if info["tensor_cores"]
                                else "fa_decode_split_kernel"),
                     "algorithmic_bytes_per_launch": alg,
                     "duration_us": kern_region_s * 1e6, "duration_from": duration_from},
        "e2e": {"value": whole_job_rate(world, query_rows(b), e2e_steps, e2e_s), "unit": "tokens/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "steps": e2e_steps,
                "includes": "plan (work-list upload) and run every step; q and page ids read, "
                            "o and lse written by the kernels in page-locked host memory",
                "staged_copies": {
                    "value": whole_job_rate(world, query_rows(b), e2e_steps, staged_s),
                    "includes": "pinned H2D q + page ids, plan, run, D2H o + lse on one stream"}},
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clocks.summary(t0, t1),
    }
    if um_bound is not None:
        out["unified_max"] = {"bound": um_bound, "fallbacks_in_timed_steps": um_fallbacks}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n, dt, toks, threads, desc, nbytes = oracle_timing(b, target_s=args.cpu_seconds)
        out["cpu_baseline"] = {"value": n / dt, "unit": "tokens/s", "cores": threads,
                               "kind": "oracle", "sample": desc,
                               "kv_tokens_per_s": toks / dt, "gbs": nbytes / dt / 1e9}
    if not args.no_others and args.max_requests is None:
        # the headline batch's memory is released first: every workload
        # holds its own batch while it is measured (each in its own timed
        # region; gpu_launches above counts the headline's region only)
        del b, p, pe, o, lse, q_h, idx_h, o_h, lse_h, q_d, idx_d, ws
        torch.cuda.empty_cache()
        out["other_workloads"] = {name: measure_other(args, world, dev, name)
                                  for name in OTHER_WORKLOADS if name != args.workload}
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=15)
    ap.add_argument("--workload", default="ragged", choices=list(W.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-others", action="store_true",
                    help="measure only --workload (not the other decode workloads)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--max-requests", type=int, default=None,
                    help="keep only the first N requests of the workload (profiler captures "
                         "that must fit a few GB; not a bench line)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        res = bench_reference(args, world, rank)
    else:
        res = bench_ours(args, world, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

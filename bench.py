#!/usr/bin/env python3
"""Benchmark of the sparse MoE FFN forward pass on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one moe_forward call (router, dispatch, expert GEMMs, combine) over
one batch of seeded synthetic input already resident in HBM; L2 is flushed
(a 256 MiB write) before every step, outside the step's CUDA events.  The
headline workload is the Mixtral-sized prefill (T = 16384, the largest
single-GPU configuration with a tensor-core roof).  Rank 0 prints one JSON
line; with one GPU it also carries a ``per_config`` block that measures every
other layer configuration of the pages (MoELayer, Mixtral decode, DeepSeek
prefill / decode, Switch capacity) the same way.  Under torchrun (N > 1)
every rank runs an independent replica on its own batch (weak scaling) and
the slowest rank's time counts.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_workloads as wl  # noqa: E402

DEFAULT_WORKLOAD = "mixtral_prefill"
# every layer configuration of the pages, measured in the same run (the
# headline is one of them), and the Mixtral-sized decode with E4M3 expert
# weights
# (in an order that lets consecutive workloads with the same layer share
# their device weights)
PER_CONFIG = ("mixtral_prefill", "mixtral_decode", "moelayer", "switch_capacity",
              "deepseek_prefill", "deepseek_decode", "mixtral_decode_fp8")
METRIC = "MoE-layer fwd tokens/s; % of bf16 TC peak (prefill) or HBM BW (decode)"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
# timed region of each per-config measurement: at least this long, so that
# the clock sampler sees it
PER_CONFIG_MIN_S = 0.4
CLOCK_INTERVAL_S = 0.005


# ---------------------------------------------------------------------------
# helpers shared by both arms (host logic, testable on CPU)

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_max(value: float, world: int, device=None) -> float:
    """Maximum of a per-rank float over all ranks (identity when world == 1)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(tokens_per_rank: int, world: int, ms_per_step_max: float) -> float:
    """Whole-job throughput: tokens every rank processed per step / slowest rank's step time."""
    return tokens_per_rank * world / (ms_per_step_max * 1e-3)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def code_without_comments(src: str) -> str:
    """C++ source without its comments and blank lines (the kernels' code)."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(l.rstrip() for l in src.splitlines() if l.strip())


def kernel_source_hash() -> str:
    """Hash of the FFN kernels' code (comments excluded): DRAM traffic taken
    on other code is not reported."""
    h = hashlib.sha256()
    for f in ("gemm_tc.cu", "decode_tc.cu", "common.cuh", "kernels.cuh"):
        with open(os.path.join(ROOT, "sparse_mixture_experts_72_b300", "csrc", f),
                  encoding="utf-8") as fh:
            h.update(code_without_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def committed_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; otherwise None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(workload, {}).get(kernel)
        if e and e.get("src_sha") == kernel_source_hash():
            return float(e["dram_bytes_per_launch"])
    except (ValueError, KeyError, TypeError):
        return None
    return None


# clock-event reason bits of NVML (nvmlClocksEventReason*)
_REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}


def summarise_clocks(samples, source: str) -> dict:
    """samples: [(sm_mhz, sm_max_mhz, power_w, reasons_bitmask)] -> the line's clocks block."""
    sm = [s[0] for s in samples]
    reasons = sorted({n for s in samples for n, b in _REASON_BITS.items() if s[3] & b})
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(s[1] for s in samples) if samples else None,
            "sm_mhz_min": min(sm) if sm else None,
            "power_w_max": max(s[2] for s in samples) if samples else None,
            "reasons": reasons, "samples": len(sm), "source": source}


class _Nvml:
    """The few read-only NVML queries the clock sampler needs, through ctypes
    on the driver's libnvidia-ml (no Python NVML package required)."""
    CLOCK_SM = 1

    class PciInfo(__import__("ctypes").Structure):
        import ctypes as _c
        _fields_ = [("busIdLegacy", _c.c_char * 16), ("domain", _c.c_uint), ("bus", _c.c_uint),
                    ("device", _c.c_uint), ("pciDeviceId", _c.c_uint),
                    ("pciSubSystemId", _c.c_uint), ("busId", _c.c_char * 32)]

    def __init__(self):
        import ctypes as c
        self.c = c
        self.lib = c.CDLL("libnvidia-ml.so.1")
        self._ok(self.lib.nvmlInit_v2())

    def _ok(self, r):
        if r != 0:
            raise RuntimeError(f"NVML error {r}")

    def handle_by_pci(self, domain, bus, device):
        c = self.c
        n = c.c_uint(0)
        self._ok(self.lib.nvmlDeviceGetCount_v2(c.byref(n)))
        for i in range(n.value):
            h = c.c_void_p()
            self._ok(self.lib.nvmlDeviceGetHandleByIndex_v2(c.c_uint(i), c.byref(h)))
            pci = self.PciInfo()
            self._ok(self.lib.nvmlDeviceGetPciInfo_v3(h, c.byref(pci)))
            if (pci.domain, pci.bus, pci.device) == (domain, bus, device):
                return h
        raise RuntimeError(f"no NVML device at PCI {(domain, bus, device)}")

    def sm_clock(self, h):
        v = self.c.c_uint(0)
        self._ok(self.lib.nvmlDeviceGetClockInfo(h, self.CLOCK_SM, self.c.byref(v)))
        return v.value

    def sm_max_clock(self, h):
        v = self.c.c_uint(0)
        self._ok(self.lib.nvmlDeviceGetMaxClockInfo(h, self.CLOCK_SM, self.c.byref(v)))
        return v.value

    def power_w(self, h):
        v = self.c.c_uint(0)
        self._ok(self.lib.nvmlDeviceGetPowerUsage(h, self.c.byref(v)))
        return v.value / 1000.0

    def reasons(self, h):
        v = self.c.c_ulonglong(0)
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self._ok(fn(h, self.c.byref(v)))
        return v.value


class ClockSampler:
    """SM clock, power and clock-event reasons of this process's GPU, sampled
    every CLOCK_INTERVAL_S by a thread through NVML (read-only queries) while
    the timed region runs; nvidia-smi is the fallback.  The GPU is found by
    its PCI bus id, so CUDA_VISIBLE_DEVICES remapping does not matter."""

    def __init__(self, device, out_dir: str):
        self.samples, self._stop, self.proc, self.thread = [], threading.Event(), None, None
        self.source = "nvml"
        self.handle = None
        self.error = None
        try:
            import torch
            pr = torch.cuda.get_device_properties(device)
            self.nv = _Nvml()
            self.handle = self.nv.handle_by_pci(pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
            self.smax = float(self.nv.sm_max_clock(self.handle))
            self.thread = threading.Thread(target=self._loop, daemon=True)
            self.thread.start()
        except Exception as e:  # noqa: BLE001
            self.handle = None
            self.error = f"{type(e).__name__}: {e}"[:200]
            self._start_smi(device, out_dir)

    def _loop(self):
        nv, h = self.nv, self.handle
        while not self._stop.is_set():
            try:
                self.samples.append((float(nv.sm_clock(h)), self.smax, nv.power_w(h),
                                     int(nv.reasons(h))))
            except Exception:  # noqa: BLE001 - a failed query is a missing sample
                pass
            time.sleep(CLOCK_INTERVAL_S)

    def _start_smi(self, device, out_dir):
        self.source = "nvidia-smi"
        fields = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active")
        self.path = os.path.join(out_dir, "clocks.csv")
        os.makedirs(out_dir, exist_ok=True)
        try:
            idx = device.index or 0
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={idx}", f"--query-gpu={fields}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.thread is not None:
            self._stop.set()
            self.thread.join(timeout=5)
            return summarise_clocks(self.samples, "nvml")
        fallback = self._stop_smi()
        if self.error:
            fallback["nvml_error"] = self.error
        return fallback

    def _stop_smi(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock source"],
                    "samples": 0, "source": "none"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        samples = []
        with open(self.path) as f:
            for line in f:
                p = [s.strip() for s in line.split(",")]
                try:
                    samples.append((float(p[0]), float(p[1]), float(p[2]), int(p[3], 16)))
                except (ValueError, IndexError):
                    continue
        return summarise_clocks(samples, "nvidia-smi")


def algorithmic_work(w: wl.Workload, counts: np.ndarray, R: int):
    """FLOPs and bytes the expert-FFN launch must do at minimum (routed
    experts and the shared expert, which is a group of the same launch).

    Per kept row: 2*H*F FLOPs in each Linear (two, or three for SwiGLU's
    gate, up and down).  Bytes: the weight
    matrices of every expert that received a row (F*H weights of 2 bytes
    (bf16) or 1 byte (E4M3) plus 4 bytes per row scale), the token rows
    read (R*H bf16) and the weighted rows written (R*H bf16); for the shared
    expert its weights and T rows in and out; the hidden activations between
    the two Linears are the implementation's own round trip and are not
    counted."""
    hit = int((np.asarray(counts) > 0).sum())
    m = 3 if w.activation == "swiglu" else 2   # weight matrices per expert (gate, up, down)
    fp8 = w.weight_dtype == "e4m3"
    wb = 1.0 if fp8 else 2.0                  # bytes per weight

    def mats(F):                               # weight (+ scale) bytes of one expert
        scales = 4.0 * ((m - 1) * F + w.H) if fp8 else 0.0
        return wb * m * F * w.H + scales
    flops = 2.0 * m * R * w.H * w.F
    nbytes = hit * mats(w.F) + 2.0 * 2 * R * w.H
    if w.F_shared:
        # the shared expert is one more group of the same launch: all T rows
        flops += 2.0 * m * w.T * w.H * w.F_shared
        nbytes += mats(w.F_shared) + 2.0 * 2 * w.T * w.H
    work = dict(flops=flops, bytes=nbytes)
    # the token-row launch and the operand-swapped decode launch do the same work
    return {"expert_ffn": work, "expert_ffn_decode": dict(work)}


def forward_work(w: wl.Workload, counts: np.ndarray, R: int) -> dict:
    """FLOPs and bytes of the whole forward pass at minimum: the gate GEMM
    (2*T*N*H), both (SwiGLU: three) Linears of every kept row and of the
    shared expert; the weights of every expert hit, the shared expert and
    W_g (fp32) read once, x read once and out written once.  Intermediate
    tensors (logits, the permuted rows, Hid, the weighted rows) are the
    implementation's own and are not counted."""
    m = 3 if w.activation == "swiglu" else 2
    fp8 = w.weight_dtype == "e4m3"
    wb = 1.0 if fp8 else 2.0
    hit = int((np.asarray(counts) > 0).sum())

    def mats(F):
        return wb * m * F * w.H + (4.0 * ((m - 1) * F + w.H) if fp8 else 0.0)
    flops = 2.0 * w.T * w.N * w.H + 2.0 * m * R * w.H * w.F
    nbytes = hit * mats(w.F) + 4.0 * w.N * w.H + 2.0 * 2 * w.T * w.H
    if w.F_shared:
        flops += 2.0 * m * w.T * w.H * w.F_shared
        nbytes += mats(w.F_shared)
    return {"flops": flops, "bytes": nbytes}


def roofline_fraction(flops: float, nbytes: float, seconds: float, peaks: dict,
                      tc_key: str = "bf16_tflops") -> dict:
    """Fraction of the slower roof: t_roof / t, t_roof = max(FLOPs / tensor peak,
    bytes / HBM peak)."""
    t_tc = flops / (peaks[tc_key] * 1e12)
    t_bw = nbytes / (peaks["hbm_gbs"] * 1e9)
    bound = "tensor" if t_tc >= t_bw else "hbm"
    return {"bound": bound, "frac": max(t_tc, t_bw) / seconds if seconds > 0 else None,
            "tflops": flops / seconds / 1e12 if seconds > 0 else None,
            "gbs": nbytes / seconds / 1e9 if seconds > 0 else None}


def bench_config(w: wl.Workload, world: int) -> dict:
    """The workload description both arms print (shapes, options, protocol)."""
    return {"workload": w.name, "T": w.T, "H": w.H, "F": w.F, "N": w.N, "k": w.k,
            "capacity_factor": w.capacity_factor, "F_shared": w.F_shared,
            "routing": w.routing, "activation": w.activation,
            "expert_weights": w.weight_dtype,
            "l2": "flushed before every step (256 MiB write, outside the step's events)",
            "launch": "CUDA graph replay of moe_forward; per-launch times from replays of a copy "
                      "with an event node before each launch, interleaved with the timed steps",
            "parallelism": f"replicas x{world}"}


def per_config_steps(est_ms: float, k_min: int, min_s: float = PER_CONFIG_MIN_S,
                     k_max: int = 4000) -> int:
    """Steps of a per-config measurement: at least k_min, and enough for a
    timed region of min_s at the estimated step time."""
    want = int(math.ceil(min_s * 1e3 / max(est_ms, 1e-3)))
    return max(k_min, min(k_max, want))


# ---------------------------------------------------------------------------
# oracle arm (CPU baseline and --impl reference)

def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:  # noqa: BLE001
        return 1


def host_cores() -> int:
    """CPUs this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def split_rows(S: int, parts: int):
    """[start, stop) of `parts` contiguous near-equal slices of range(S) (empty ones dropped)."""
    b = np.linspace(0, S, parts + 1).round().astype(int)
    return [(int(b[i]), int(b[i + 1])) for i in range(parts) if b[i + 1] > b[i]]


def oracle_timing_all_cores(w: wl.Workload, steps: int, warmup: int, budget_s: float):
    """oracle_timing in a child process that never touches CUDA, with one
    BLAS thread per process (set before numpy loads) and a pool of worker
    processes, one per host core, forked from it after the weights are
    drawn (so they share them).  Returns (tokens/s, sample tokens, desc,
    workers)."""
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[v] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    code = ("import json, sys; sys.path.insert(0, %r); import bench, moe_workloads as wl; "
            "w = wl.get_workload(%r); r = bench.oracle_timing(w, %d, %d, %r, bench.host_cores()); "
            "print(json.dumps(list(r)))" % (ROOT, w.name, steps, warmup, float(budget_s)))
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         check=True, cwd=ROOT)
    tps, S, desc, workers = json.loads(out.stdout.strip().splitlines()[-1])
    return tps, S, desc, workers


def oracle_step(w: wl.Workload, x_bits, router, getter, shared, rows: slice):
    """One oracle forward over the token rows `rows` (a sub-batch of the
    workload).  Without a capacity limit the rows are routed exactly as in
    the full batch; with one, capacity couples all tokens, so the whole
    batch is routed and dispatched and the experts are evaluated for `rows`."""
    from oracle import moe_oracle as O
    Wg, bg, sel = router
    kw = dict(routing=w.routing, activation=w.activation, min_capacity=w.min_capacity,
              drop_order=w.drop_order)
    if w.capacity_factor > 0:
        xs = wl.bf16_bits_to_f64(x_bits)
        return O.forward(xs, Wg, bg, sel, w.k, w.capacity_factor, w.aux_alpha, getter, shared,
                         tokens=np.arange(rows.start, rows.stop), **kw)
    xs = wl.bf16_bits_to_f64(x_bits[rows])
    return O.forward(xs, Wg, bg, sel, w.k, w.capacity_factor, w.aux_alpha, getter, shared, **kw)


_POOL_STATE = {}


def _pool_slice(span):
    """Worker body: the oracle over rows [span) of the batch held in _POOL_STATE."""
    st = _POOL_STATE
    oracle_step(st["w"], st["x_bits"], st["router"], st["getter"], st["shared"],
                slice(span[0], span[1]))
    return span[1] - span[0]


def oracle_inputs(w: wl.Workload, seed: int = 0):
    """x bits, router and float64 expert weights (all drawn now) for the oracle."""
    from oracle import moe_oracle as O
    x_bits = wl.gen_x(w, seed)
    router = wl.gen_router(w, seed)
    if w.weight_dtype == "e4m3":
        cache = {}

        def getter(e):
            if e not in cache:
                q1, s1, b1, q2, s2, b2 = wl.gen_expert_e4m3(w, seed, e)
                cache[e] = (O.dequantize_rows(q1, s1),
                            None if b1 is None else wl.bf16_bits_to_f64(b1),
                            O.dequantize_rows(q2, s2),
                            None if b2 is None else wl.bf16_bits_to_f64(b2))
            return cache[e]
        sh = wl.gen_shared_e4m3(w, seed)
        shared = None if sh is None else (
            O.dequantize_rows(sh[0], sh[1]), None if sh[2] is None else wl.bf16_bits_to_f64(sh[2]),
            O.dequantize_rows(sh[3], sh[4]), None if sh[5] is None else wl.bf16_bits_to_f64(sh[5]))
    else:
        getter = wl.expert_getter_f64(w, seed)
        shared = wl.shared_f64(w, seed)
    # draw and widen every expert before timing (threads: the draws release the GIL)
    wl._pool_map(getter, range(w.N), None)
    return x_bits, router, getter, shared


def oracle_timing(w: wl.Workload, steps: int, warmup: int, budget_s: float, workers: int = 1,
                  seed: int = 0):
    """Times the oracle on bounded token samples with `workers` processes
    (forked after the inputs are drawn; each computes a contiguous slice of
    the sample).  Returns (tokens/s, sample tokens, desc, workers used)."""
    x_bits, router, getter, shared = oracle_inputs(w, seed)
    _POOL_STATE.update(w=w, x_bits=x_bits, router=router, getter=getter, shared=shared)
    # size the sample so that warmup + steps fit in the budget
    probe = min(w.T, 32)
    t0 = time.perf_counter()
    _pool_slice((0, probe))
    per_tok = (time.perf_counter() - t0) / probe
    total_steps = max(1, steps + warmup)
    per_step = budget_s / total_steps
    S = int(max(8, min(w.T, workers * per_step / max(per_tok, 1e-9))))
    workers = max(1, min(workers, S))
    pool = None
    if workers > 1:
        import multiprocessing as mp
        pool = mp.get_context("fork").Pool(workers)

    def one_step(s0):
        spans = [(s0 + a, s0 + b) for a, b in split_rows(S, workers)]
        t = time.perf_counter()
        n = sum(pool.map(_pool_slice, spans, chunksize=1)) if pool else _pool_slice(spans[0])
        assert n == S
        return time.perf_counter() - t
    try:
        for i in range(warmup):
            one_step(0)
        times = [one_step((i * S) % max(1, w.T - S + 1)) for i in range(steps)]
    finally:
        if pool:
            pool.close()
            pool.join()
    tps = S / statistics.median(times)
    desc = (f"oracle forward over {S}-token slices of the {w.name} batch (T={w.T}), "
            f"{steps} timed slices, each split over {workers} worker processes with one "
            f"BLAS thread each, float64 numpy on host")
    return tps, S, desc, workers


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w = wl.get_workload(args.workload)
    budget = 150.0
    tps, S, desc, cores = oracle_timing_all_cores(w, args.steps, args.warmup, budget)
    line = {"metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": S / tps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": bench_config(w, args.gpus),
            "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# CUDA arm

def measure(m, w, d, device, steps: int, warmup: int, world: int, flush, peaks, clocks_dir,
            min_s: float = 0.0):
    """Times `steps` graph replays of moe_forward on the inputs `d` (with
    min_s > 0: at least min_s of them, the step count raised from a warm-up
    estimate).  Returns a dict of results (ms_per_step is this rank's)."""
    import torch
    cfg = m.MoEConfig(**w.config_kwargs())
    weights = m.MoEWeights(**{k: d[k] for k in wl.WEIGHT_KEYS})
    x = d["x"]
    ws = m.make_workspace(cfg, device)
    outs = m.alloc_outputs(cfg, device)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=device)
    n_launch = m.moe_forward_num_launches(cfg)
    W = max(warmup, 3)
    for _ in range(W):
        flush.zero_()
        m.moe_forward(cfg, weights, x, out=out, outputs=outs, ws=ws)
    torch.cuda.synchronize()
    if m.moe_workspace_status(ws) != 0:
        raise RuntimeError(f"{w.name}: device status after warm-up is not OK")
    fwd = m.MoEForwardGraph(cfg, weights, x, out, outputs=outs, ws=ws)
    trace_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_launch + 1)]
    fwd_traced = m.MoEForwardGraph(cfg, weights, x, out, outputs=outs, ws=ws,
                                   trace_events=trace_ev)
    counts = outs["counts"].cpu().numpy()
    R = int(outs["offsets"][-1].item())
    names = m.moe_forward_launch_names(cfg)
    K = steps
    if min_s > 0:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(3):
            fwd.replay()
        e1.record()
        torch.cuda.synchronize()
        K = per_config_steps(e0.elapsed_time(e1) / 3, steps, min_s)
    # per-launch device times: a traced replay after every trace_every-th
    # step (not a step: its own events are not in the step times)
    trace_every = max(1, K // 5)
    traced_after = set(range(0, K, trace_every))
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    per = {n: [] for n in names}

    clocks = ClockSampler(device, clocks_dir)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for i in range(K):
        flush.zero_()
        ev_s[i].record()
        fwd.replay()
        ev_e[i].record()
        if i in traced_after:
            flush.zero_()
            fwd_traced.replay()
            torch.cuda.synchronize()  # read this replay's stamps before the next overwrites them
            for j, n in enumerate(names):
                per[n].append(trace_ev[j].elapsed_time(trace_ev[j + 1]))
    torch.cuda.synchronize()
    wall_s = time.perf_counter() - t_wall
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    if m.moe_workspace_status(ws) != 0:
        raise RuntimeError(f"{w.name}: device status after the timed steps is not OK")

    step_ms = [ev_s[i].elapsed_time(ev_e[i]) for i in range(K)]
    ms_local = float(np.mean(step_ms))
    per_ms = {n: float(np.mean(v)) for n, v in per.items()}
    work = algorithmic_work(w, counts, R)
    fw = forward_work(w, counts, R)
    gemms = [n for n in names if "_ffn" in n]
    dom = max(gemms, key=lambda n: per_ms[n]) if gemms else max(per_ms, key=per_ms.get)
    res = dict(cfg=cfg, weights=weights, ws=ws, outs=outs, out=out, x=x, names=names,
               n_launch=n_launch, K=K, W=W, n_traced=len(traced_after), ms_local=ms_local,
               step_ms_min=float(np.min(step_ms)), step_ms_max=float(np.max(step_ms)),
               per_ms=per_ms, counts=counts, R=R, work=work, fw=fw, dom=dom, clocks=clk,
               wall_s=wall_s)
    return res


def kernel_roofline(w, res, peaks, peak_src):
    """The roofline object of the dominant launch (an expert-FFN launch)."""
    dom = res["dom"]
    t_dom = res["per_ms"][dom] * 1e-3
    wk = res["work"].get(dom)
    if wk is None or t_dom <= 0:
        return None
    t_tc = wk["flops"] / (peaks["bf16_tflops"] * 1e12)
    t_bw = wk["bytes"] / (peaks["hbm_gbs"] * 1e9)
    if t_tc >= t_bw:
        ach = wk["flops"] / t_dom / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"]}
    else:
        ach = wk["bytes"] / t_dom / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"]}
    roof["traffic"] = committed_traffic(w.name, dom)
    roof["algorithmic"] = wk["bytes"] if roof["bound"] == "hbm" else wk["flops"]
    roof["kernel"] = ("decode_ffn_kernel" if dom.endswith("_decode") else "grouped_gemm_kernel") + \
        f" ({dom})"
    roof["launch_ms"] = res["per_ms"][dom]
    roof["peak_source"] = f"{peak_src} ({'burst' if roof['bound'] == 'tensor' else 'copy'})"
    return roof


def forward_roofline(res, ms, peaks, peak_src):
    """Whole-step fraction of the slower roof, against the burst and the
    sustained tensor peak."""
    fw = res["fw"]
    s = ms * 1e-3
    burst = roofline_fraction(fw["flops"], fw["bytes"], s, peaks, "bf16_tflops")
    sus = roofline_fraction(fw["flops"], fw["bytes"], s, peaks,
                            "bf16_tflops_sustained" if "bf16_tflops_sustained" in peaks
                            else "bf16_tflops")
    return {"bound": burst["bound"], "frac": burst["frac"], "frac_sustained_peak": sus["frac"],
            "flops": fw["flops"], "bytes": fw["bytes"], "tflops": burst["tflops"],
            "gbs": burst["gbs"], "peak_source": peak_src}


def config_entry(w, res, ms, peaks, peak_src):
    roof = kernel_roofline(w, res, peaks, peak_src)
    return {"T": w.T, "ms_per_step": ms, "tokens_per_s": w.T / (ms * 1e-3),
            "steps": res["K"], "step_ms_min": res["step_ms_min"], "step_ms_max": res["step_ms_max"],
            "kept_rows": res["R"], "experts_hit": int((res["counts"] > 0).sum()),
            "ffn": None if roof is None else {k: roof[k] for k in
                                              ("bound", "achieved", "unit", "frac", "launch_ms",
                                               "traffic")},
            "forward": forward_roofline(res, ms, peaks, peak_src),
            "launch_ms": res["per_ms"], "clocks": res["clocks"]}


def e2e_measure(m, w, res, x_bits_host, K, world, device):
    """End to end through the C ABI with host buffers (moe_forward_host: H2D
    of x from pinned memory, the forward, D2H of out), pipelined over three
    streams (input copies, layers, output copies) and three buffer sets, so
    batch i+1's input copy and batch i-1's output copy overlap batch i's
    layer.  No flush here: the batches alternate between two weight
    replicas, so each step's weights were last read two steps earlier with
    the other replica's weights (2x the expert bytes) read in between."""
    import torch
    cfg, weights, ws, x, out = res["cfg"], res["weights"], res["ws"], res["x"], res["out"]
    wrep = [weights, m.MoEWeights(**{k: (None if v is None else v.clone())
                                     for k, v in weights.__dict__.items()})]
    SL = 3
    x_pin = [torch.from_numpy(np.ascontiguousarray(x_bits_host).view(np.int16)).pin_memory()
             .view(torch.bfloat16) for _ in range(SL)]
    out_pin = [torch.empty((w.T, w.H), dtype=torch.bfloat16).pin_memory() for _ in range(SL)]
    x_st = [torch.empty_like(x) for _ in range(SL)]
    out_st = [torch.empty_like(out) for _ in range(SL)]
    h2d_s, k_s, d2h_s = (torch.cuda.Stream(device) for _ in range(3))
    done = [torch.cuda.Event() for _ in range(SL)]
    wcs = [wr.c(cfg) for wr in wrep]

    def e2e_step(i):
        b = i % SL
        h2d_s.wait_event(done[b])   # slot b's previous output copy has finished
        m.moe_forward_host(cfg, None, x_pin[b], out_pin[b], x_st[b], out_st[b], ws=ws,
                           h2d_stream=h2d_s, compute_stream=k_s, d2h_stream=d2h_s,
                           weights_c=wcs[i % 2])
        done[b].record(d2h_s)

    E = max(20, min(K, 200))
    torch.cuda.synchronize()
    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize()
    if m.moe_workspace_status(ws) != 0:
        raise RuntimeError("device status after the end-to-end warm-up is not OK")
    cur = torch.cuda.current_stream(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for s_ in (h2d_s, k_s, d2h_s):
        s_.wait_stream(cur)
    for i in range(E):
        e2e_step(i)
    for s_ in (h2d_s, k_s, d2h_s):
        cur.wait_stream(s_)
    e1.record(cur)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1) / E, world, device)
    if not all(torch.equal(out_pin[0].view(torch.int16), o.view(torch.int16)) for o in out_pin):
        raise RuntimeError("the end-to-end batches disagree")
    del wrep
    return {"value": aggregate(w.T, world, e2e_ms), "unit": "tokens/s",
            "h2d_bytes_per_step": int(x_pin[0].numel() * 2),
            "d2h_bytes_per_step": int(out_pin[0].numel() * 2),
            "ms_per_step": e2e_ms, "steps": E,
            "how": "moe_forward_host (C ABI, pinned host buffers) pipelined on H2D, compute "
                   "and D2H streams with three buffer sets; two weight replicas alternate"}


def run_ours(args):
    import torch
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    device = torch.device("cuda", local_rank if world > 1 else 0)
    torch.cuda.set_device(device)

    import sparse_mixture_experts_72_b300 as m

    peaks, peak_src = load_peaks()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    w = wl.get_workload(args.workload)
    # replicas share the weights; each rank draws its own batch
    d = wl.to_device(w, seed=0, device=device, x_seed=None if rank == 0 else 1000 + rank)
    res = measure(m, w, d, device, args.steps, args.warmup, world, flush, peaks, args.clocks_dir)
    K = res["K"]
    ms_max = reduce_max(res["ms_local"], world, device)
    value = aggregate(w.T, world, ms_max)
    roof = kernel_roofline(w, res, peaks, peak_src)
    fwd_roof = forward_roofline(res, ms_max, peaks, peak_src)
    e2e = None if args.no_e2e else e2e_measure(m, w, res, d["x_bits"], K, world, device)
    launches = (K + res["n_traced"]) * sum(1 for n in res["names"] if "memset" not in n)
    headline_entry = config_entry(w, res, ms_max, peaks, peak_src)

    per_config = None
    if world == 1 and not args.no_per_config:
        per_config = {w.name: headline_entry}
        cache = {w.name: d}
        del res
        for name in PER_CONFIG:
            if name in per_config:
                continue
            wc = wl.get_workload(name)
            # reuse the device weights of a workload with the same layer
            src = next((cache[n] for n in cache if wl.same_weights(wl.get_workload(n), wc)), None)
            for n in list(cache):
                if cache[n] is not src:
                    del cache[n]
            torch.cuda.empty_cache()
            dc = wl.to_device(wc, seed=0, device=device, reuse=src)
            cache = {name: dc}
            rc = measure(m, wc, dc, device, args.steps, args.warmup, 1, flush, peaks,
                         args.clocks_dir, min_s=PER_CONFIG_MIN_S)
            per_config[name] = config_entry(wc, rc, rc["ms_local"], peaks, peak_src)
            del rc
        cache.clear()
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tps, S, desc, cores = oracle_timing_all_cores(w, steps=3, warmup=1, budget_s=24.0)
        cpu = {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": desc, "host_cores": host_cores()}

    if rank == 0:
        hr = headline_entry
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
                "steps": K, "warmup": max(args.warmup, 3), "ms_per_step": ms_max,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic",
                "config": bench_config(w, world),
                "work": {"kept_rows": hr["kept_rows"], "experts_hit": hr["experts_hit"]},
                "roofline": roof, "forward_roofline": fwd_roof,
                "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": int(launches),
                "clocks": hr["clocks"],
                "launch_ms": hr["launch_ms"],
                "step_ms": {"mean": ms_max, "min": hr["step_ms_min"], "max": hr["step_ms_max"]},
                "per_config": per_config}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(wl.WORKLOADS) + sorted(wl.TEST_WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="measure only the headline workload")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end (host buffers) leg, e.g. under a profiler")
    ap.add_argument("--clocks-dir", default=os.path.join(tempfile.gettempdir(), "moe_bench"),
                    help="where nvidia-smi clock samples go if NVML is unavailable")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())

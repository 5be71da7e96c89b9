#!/usr/bin/env python3
"""Benchmark of the sparse MoE FFN forward pass on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one moe_forward call (router, dispatch, expert GEMMs, combine) over
one batch of seeded synthetic input already resident in HBM; L2 is flushed
(a 256 MiB write) between timed steps, outside the timed events.  Prints one
JSON line on rank 0.  Under torchrun (N > 1) every rank runs an independent
replica on its own batch (weak scaling) and the slowest rank's time counts.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_workloads as wl  # noqa: E402

DEFAULT_WORKLOAD = "moelayer"
METRIC = "MoE-layer fwd tokens/s; % of bf16 TC peak (prefill) or HBM BW (decode)"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


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


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("gemm_tc.cu", "common.cuh", "kernels.cuh"):
        with open(os.path.join(ROOT, "sparse_mixture_experts_72_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
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


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, out_dir: str, interval_ms: int = 50):
        self.proc = None
        self.path = os.path.join(out_dir, f"clocks_rank{gpu_index}.csv")
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms", str(interval_ms)],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def algorithmic_work(w: wl.Workload, counts: np.ndarray, R: int):
    """FLOPs and bytes each expert-FFN launch must do at minimum.

    Per kept row: 2*H*F FLOPs in each Linear (two, or three for SwiGLU's
    gate, up and down).  Bytes: the weight
    matrices of every expert that received a row (F*H weights of 2 bytes
    (bf16) or 1 byte (E4M3) plus 4 bytes per row scale), the token rows
    read (R*H bf16) and the weighted rows written (R*H bf16); the hidden
    activations between the two Linears are the implementation's own round
    trip and are not counted."""
    hit = int((np.asarray(counts) > 0).sum())
    m = 3 if w.activation == "swiglu" else 2   # weight matrices per expert (gate, up, down)
    fp8 = w.weight_dtype == "e4m3"
    wb = 1.0 if fp8 else 2.0                  # bytes per weight

    def mats(F):                               # weight (+ scale) bytes of one expert
        scales = 4.0 * ((m - 1) * F + w.H) if fp8 else 0.0
        return wb * m * F * w.H + scales
    out = {"expert_ffn": dict(flops=2.0 * m * R * w.H * w.F,
                              bytes=hit * mats(w.F) + 2.0 * 2 * R * w.H)}
    if w.F_shared:
        Fs = w.F_shared
        out["shared_ffn"] = dict(flops=2.0 * m * w.T * w.H * Fs,
                                 bytes=mats(Fs) + 2.0 * 2 * w.T * w.H)
    return out


def bench_config(w: wl.Workload, world: int) -> dict:
    """The workload description both arms print (shapes, options, protocol)."""
    return {"workload": w.name, "T": w.T, "H": w.H, "F": w.F, "N": w.N, "k": w.k,
            "capacity_factor": w.capacity_factor, "F_shared": w.F_shared,
            "routing": w.routing, "activation": w.activation,
            "expert_weights": w.weight_dtype,
            "l2": "flushed between steps (256 MiB write, untimed)",
            "launch": "CUDA graph replay of moe_forward; every 10th step replays a copy with an "
                      "event node before each launch",
            "parallelism": f"replicas x{world}"}


def launch_names(w: wl.Workload, has_rows: bool):
    """Names of the launches moe_forward makes, in order (the status clear is
    folded into the tensor-core router's first kernel, the scan into the
    rank launch's last block, and the dispatch scatter also gathers the
    expert rows)."""
    names = []
    tc_router = w.N <= 256
    if not (tc_router and w.T > 0):
        names += ["status_memset"]
    if tc_router:  # tensor-core router: W_g split + fused router
        names += ["router_split", "router_tc"] if w.T > 0 else ["router_pmean"]
    else:
        names += ["router_logits", "router_select", "router_pmean"] if w.T > 0 else ["router_pmean"]
    if w.routing == "expert":
        names += ["expert_choice"]
        if has_rows:
            names += ["gather_rows"]
    elif w.T * w.k > 0:
        names += ["permute_rank_scan", "scatter_gather"]
    else:
        names += ["permute_scan"]
    if has_rows:
        names += ["expert_ffn"]   # both Linears of every expert in one launch
    if w.F_shared:
        names += ["shared_ffn"]
    if w.T > 0:
        names += ["combine"]
    return names


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


def oracle_timing_all_cores(w: wl.Workload, steps: int, warmup: int, budget_s: float):
    """oracle_timing in a child process whose BLAS may use every host core
    (thread-count variables set before numpy loads: a BLAS started with one
    thread cannot grow later).  Returns (tokens/s, sample tokens, desc, threads)."""
    n = host_cores()
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[v] = str(n)
    code = ("import json, sys; sys.path.insert(0, %r); import bench, moe_workloads as wl; "
            "w = wl.get_workload(%r); r = bench.oracle_timing(w, %d, %d, %r); "
            "print(json.dumps([r[0], r[1], r[2], bench.blas_threads()]))"
            % (ROOT, w.name, steps, warmup, float(budget_s)))
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         check=True, cwd=ROOT)
    tps, S, desc, threads = json.loads(out.stdout.strip().splitlines()[-1])
    return tps, S, desc, threads


def oracle_step(w: wl.Workload, x_bits, router, getter, shared, rows: slice):
    """One oracle forward over the token rows `rows` (a sub-batch of the
    workload: with no capacity limit the rows are routed exactly as in the
    full batch)."""
    from oracle import moe_oracle as O
    Wg, bg, sel = router
    xs = wl.bf16_bits_to_f64(x_bits[rows])
    return O.forward(xs, Wg, bg, sel, w.k, w.capacity_factor, w.aux_alpha, getter, shared,
                     routing=w.routing, activation=w.activation, min_capacity=w.min_capacity,
                     drop_order=w.drop_order)


def oracle_timing(w: wl.Workload, steps: int, warmup: int, budget_s: float, seed: int = 0):
    """Times the oracle on bounded token samples; returns (tokens/s, sample tokens, desc)."""
    x_bits = wl.gen_x(w, seed)
    router = wl.gen_router(w, seed)
    if w.weight_dtype == "e4m3":
        from oracle import moe_oracle as O
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
    for e in range(w.N):
        getter(e)  # draw and widen the weights before timing
    # size the sample so that warmup + steps fit in the budget
    probe = min(w.T, 64)
    t0 = time.perf_counter()
    oracle_step(w, x_bits, router, getter, shared, slice(0, probe))
    per_tok = (time.perf_counter() - t0) / probe
    total_steps = max(1, steps + warmup)
    S = int(max(8, min(w.T, budget_s / total_steps / max(per_tok, 1e-9))))
    if w.capacity_factor > 0:
        S = w.T  # capacity couples tokens: only the whole batch is exact
    for i in range(warmup):
        oracle_step(w, x_bits, router, getter, shared, slice(0, S))
    times = []
    for i in range(steps):
        s0 = (i * S) % max(1, w.T - S + 1)
        t0 = time.perf_counter()
        oracle_step(w, x_bits, router, getter, shared, slice(s0, s0 + S))
        times.append(time.perf_counter() - t0)
    tps = S / statistics.median(times)
    desc = (f"oracle forward over {S}-token slices of the {w.name} batch "
            f"(T={w.T}), {steps} timed slices, float64 numpy on host")
    return tps, S, desc


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

    w = wl.get_workload(args.workload)
    cfg = m.MoEConfig(**w.config_kwargs())
    # replicas share the weights; each rank draws its own batch
    d = wl.to_device(w, seed=0, device=device, x_seed=None if rank == 0 else 1000 + rank)
    weights = m.MoEWeights(**{k: d[k] for k in wl.WEIGHT_KEYS})
    x_bits_host, x = d["x_bits"], d["x"]
    ws = m.make_workspace(cfg, device)
    outs = m.alloc_outputs(cfg, device)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    n_launch = m.moe_forward_num_launches(cfg)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        m.moe_forward(cfg, weights, x, out=out, outputs=outs, ws=ws)
    torch.cuda.synchronize()
    if m.moe_workspace_status(ws) != 0:
        raise RuntimeError("device status after warm-up is not OK")
    # the timed steps replay the whole forward as one CUDA graph; every
    # TRACE_EVERY-th step replays a copy of it that also records an event
    # before each launch (device timestamps, no host gaps)
    fwd = m.MoEForwardGraph(cfg, weights, x, out, outputs=outs, ws=ws)
    trace_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_launch + 1)]
    fwd_traced = m.MoEForwardGraph(cfg, weights, x, out, outputs=outs, ws=ws,
                                   trace_events=trace_ev)
    counts = outs["counts"].cpu().numpy()
    R = int(outs["offsets"][-1].item())
    names = launch_names(w, m.moe_max_rows(cfg) > 0)
    assert len(names) == n_launch, (names, n_launch)

    K = args.steps
    TRACE_EVERY = 10
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    traced_steps = set(range(0, K, TRACE_EVERY))
    per = {n: [] for n in names}

    clocks = ClockSampler(device.index or 0, args.clocks_dir)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for i in range(K):
        flush.zero_()
        ev_s[i].record()
        if i in traced_steps:
            fwd_traced.replay()
            ev_e[i].record()
            torch.cuda.synchronize()  # read this replay's stamps before the next overwrites them
            for j, n in enumerate(names):
                per[n].append(trace_ev[j].elapsed_time(trace_ev[j + 1]))
        else:
            fwd.replay()
            ev_e[i].record()
    torch.cuda.synchronize()
    wall_s = time.perf_counter() - t_wall
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    if m.moe_workspace_status(ws) != 0:
        raise RuntimeError("device status after the timed steps is not OK")

    step_ms = [ev_s[i].elapsed_time(ev_e[i]) for i in range(K)]
    ms_local = float(np.mean(step_ms))
    graph_ms = float(np.mean([t for i, t in enumerate(step_ms) if i not in traced_steps] or step_ms))
    traced_ms = float(np.mean([step_ms[i] for i in traced_steps]))
    ms_max = reduce_max(ms_local, world, device)
    value = aggregate(w.T, world, ms_max)

    # per-launch device times from the traced replays
    per_ms = {n: float(np.mean(v)) for n, v in per.items()}

    peaks, peak_src = load_peaks()
    work = algorithmic_work(w, counts, R)
    gemms = [n for n in names if n.endswith("_ffn")]
    dom = max(gemms, key=lambda n: per_ms[n]) if gemms else max(per_ms, key=per_ms.get)
    t_dom = per_ms[dom] * 1e-3
    wk = work.get(dom)
    roof = None
    if wk is not None and t_dom > 0:
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
        roof["kernel"] = f"grouped_gemm_kernel ({dom})"
        roof["launch_ms"] = per_ms[dom]
        roof["peak_source"] = f"{peak_src} (burst)"

    # End to end through the C ABI with host buffers (moe_forward_host: H2D
    # of x from pinned memory, the forward, D2H of out), pipelined over three
    # streams (input copies, layers, output copies) and three buffer sets,
    # so batch i+1's input copy and batch i-1's output copy overlap batch i's
    # layer.  No flush here: the batches alternate between two weight
    # replicas, so each step's weights were last read two steps earlier with
    # the other replica's weights (2x the expert bytes) read in between.
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
    e2e = {"value": aggregate(w.T, world, e2e_ms), "unit": "tokens/s",
           "h2d_bytes_per_step": int(x_pin[0].numel() * 2),
           "d2h_bytes_per_step": int(out_pin[0].numel() * 2),
           "ms_per_step": e2e_ms,
           "how": "moe_forward_host (C ABI, pinned host buffers) pipelined on H2D, compute "
                  "and D2H streams with three buffer sets; two weight replicas alternate"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tps, S, desc, cores = oracle_timing_all_cores(w, steps=3, warmup=1, budget_s=20.0)
        cpu = {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": desc}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
                "steps": K, "warmup": max(args.warmup, 3), "ms_per_step": ms_max,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic",
                "config": bench_config(w, world),
                "work": {"kept_rows": R, "experts_hit": int((counts > 0).sum())},
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": int(K * sum(1 for n in names if "memset" not in n)),
                "step_ms": {"graph_replay": graph_ms, "graph_replay_traced": traced_ms,
                            "traced_steps": len(traced_steps)},
                "clocks": clk,
                "launch_ms": per_ms,
                "wall_s_timed_region": wall_s}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(wl.WORKLOADS) + sorted(wl.TEST_WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clocks-dir", default=os.path.join(tempfile.gettempdir(), "moe_bench"),
                    help="where the nvidia-smi clock samples of the timed region are kept")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())

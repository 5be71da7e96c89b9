"""Host logic of bench.py: the multi-rank reduction (two gloo ranks on CPU),
the aggregate throughput and the algorithmic work counts."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
import moe_workloads as wl


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, wsz, lr = bench.dist_env()
    ms = 1.0 + rank  # rank 1 is the slower one
    mx = bench.reduce_max(ms, wsz)
    q.put((r, wsz, lr, mx, bench.aggregate(4096, wsz, mx)))
    dist.destroy_process_group()


def test_two_rank_max_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1]
    for r, wsz, lr, mx, agg in res:
        assert wsz == 2 and lr == r and mx == 2.0
        assert agg == pytest.approx(2 * 4096 / 2e-3)


def test_single_rank_identity():
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.aggregate(100, 1, 1.0) == pytest.approx(1e5)


def test_algorithmic_work_counts():
    w = wl.WORKLOADS["moelayer"]
    counts = np.full(w.N, w.T * w.k // w.N)
    work = bench.algorithmic_work(w, counts, w.T * w.k)
    # both Linears of all 8192 kept rows; both weight matrices of the 8 experts
    assert work["expert_ffn"]["flops"] == 4 * 8192 * 1024 * 4096
    assert work["expert_ffn"]["bytes"] == 2 * (2 * 8 * 4096 * 1024 + 2 * 8192 * 1024)
    d = wl.WORKLOADS["deepseek_prefill"]
    wk = bench.algorithmic_work(d, np.ones(d.N), d.T * d.k)
    assert "shared_ffn" in wk and wk["shared_ffn"]["flops"] == 4 * d.T * d.F_shared * d.H
    # SwiGLU: gate, up and down matrices
    s = wl.WORKLOADS["mixtral_swiglu_decode"]
    ws = bench.algorithmic_work(s, np.full(s.N, 16), 128)
    assert ws["expert_ffn"]["flops"] == 6 * 128 * s.H * s.F
    assert ws["expert_ffn"]["bytes"] == 2 * 3 * 8 * s.F * s.H + 2 * 2 * 128 * s.H
    # E4M3 weights: one byte per weight plus one fp32 scale per matrix row
    # (W1: F rows, W2: H rows); activations stay bf16
    f = wl.WORKLOADS["mixtral_decode_fp8"]
    wf = bench.algorithmic_work(f, np.array([16] * 7 + [0]), 112)
    assert wf["expert_ffn"]["flops"] == 4 * 112 * f.H * f.F
    assert wf["expert_ffn"]["bytes"] == 7 * (2 * f.F * f.H + 4 * (f.F + f.H)) + 2 * 2 * 112 * f.H


def test_peaks_and_traffic_lookup():
    peaks, src = bench.load_peaks()
    assert peaks["hbm_gbs"] > 0 and peaks["bf16_tflops"] > 0
    assert bench.committed_traffic("no_such_workload", "expert_ffn") is None

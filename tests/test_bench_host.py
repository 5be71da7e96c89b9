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
    # the shared expert is part of the expert-FFN launch
    assert wk["expert_ffn"]["flops"] == 4 * d.T * d.k * d.F * d.H + 4 * d.T * d.F_shared * d.H
    assert wk["expert_ffn"]["bytes"] == (d.N * 2 * 2 * d.F * d.H + 2 * 2 * d.T * d.k * d.H +
                                         2 * 2 * d.F_shared * d.H + 2 * 2 * d.T * d.H)
    assert wk["expert_ffn_decode"] == wk["expert_ffn"]
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


def test_forward_work_counts():
    """Whole-forward work: gate GEMM + both Linears of every kept row; every
    hit expert's weights, W_g (fp32), x and out once."""
    w = wl.WORKLOADS["moelayer"]
    counts = np.full(w.N, w.T * w.k // w.N)
    fw = bench.forward_work(w, counts, w.T * w.k)
    assert fw["flops"] == 2 * 4096 * 8 * 1024 + 4 * 8192 * 1024 * 4096
    assert fw["bytes"] == 8 * 2 * 2 * 4096 * 1024 + 4 * 8 * 1024 + 2 * 2 * 4096 * 1024
    d = wl.WORKLOADS["deepseek_decode"]
    cd = np.zeros(d.N)
    cd[:200] = 1
    fd = bench.forward_work(d, cd, 200)
    # 200 routed experts hit plus the shared one
    assert fd["bytes"] == 201 * 2 * 2 * d.F * d.H + 4 * d.N * d.H + 2 * 2 * d.T * d.H


def test_roofline_fraction_takes_the_slower_roof():
    peaks = {"bf16_tflops": 1000.0, "hbm_gbs": 1000.0}
    # 1e12 FLOP -> 1 ms at the tensor peak; 0.5e9 B -> 0.5 ms: tensor-bound
    r = bench.roofline_fraction(1e12, 0.5e9, 2e-3, peaks)
    assert r["bound"] == "tensor" and r["frac"] == pytest.approx(0.5)
    r = bench.roofline_fraction(1e9, 4e9, 5e-3, peaks)
    assert r["bound"] == "hbm" and r["frac"] == pytest.approx(0.8)
    assert r["gbs"] == pytest.approx(800.0)


def test_per_config_steps_and_row_split():
    assert bench.per_config_steps(0.16, 20, 0.4) == 2500
    assert bench.per_config_steps(10.0, 20, 0.4) == 40
    assert bench.per_config_steps(100.0, 20, 0.4) == 20
    assert bench.per_config_steps(1e-6, 20, 0.4, k_max=4000) == 4000
    for S, parts in ((10, 3), (7, 8), (1000, 64)):
        spans = bench.split_rows(S, parts)
        assert spans[0][0] == 0 and spans[-1][1] == S
        assert all(a < b for a, b in spans)
        assert all(spans[i][1] == spans[i + 1][0] for i in range(len(spans) - 1))


def test_clock_summary_decodes_reasons():
    s = [(2032.0, 2032.0, 900.0, 0x0), (1900.0, 2032.0, 1100.0, 0x4), (1800.0, 2032.0, 1000.0, 0x4)]
    c = bench.summarise_clocks(s, "nvml")
    assert c["samples"] == 3 and c["sm_mhz"] == 1900.0 and c["sm_max_mhz"] == 2032.0
    assert c["reasons"] == ["sw_power_cap"]
    c2 = bench.summarise_clocks([(1000.0, 2032.0, 500.0, 0x8 | 0x40)], "nvml")
    assert c2["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]


def test_weight_reuse_between_workloads():
    W = wl.WORKLOADS
    assert wl.same_weights(W["mixtral_prefill"], W["mixtral_decode"])
    assert wl.same_weights(W["deepseek_prefill"], W["deepseek_decode"])
    assert not wl.same_weights(W["mixtral_prefill"], W["mixtral_decode_fp8"])
    assert not wl.same_weights(W["moelayer"], W["mixtral_prefill"])
    t = wl.get_workload("tiny")
    d0 = wl.to_device(t, 0, "cpu")
    d1 = wl.to_device(t.with_tokens(16), 0, "cpu", reuse=d0)
    assert d1["W1"] is d0["W1"] and d1["Wg"] is d0["Wg"]
    assert d1["x"].shape == (16, t.H)
    assert np.array_equal(d1["x_bits"], wl.gen_x(t.with_tokens(16), 0))


def test_bench_defaults_to_the_largest_prefill_config():
    assert bench.DEFAULT_WORKLOAD == "mixtral_prefill"
    assert set(bench.PER_CONFIG) == {"moelayer", "mixtral_prefill", "mixtral_decode",
                                     "deepseek_prefill", "deepseek_decode", "switch_capacity",
                                     "mixtral_decode_fp8"}


def test_traffic_hash_ignores_comments_only():
    src = "// a\nint f(int x) {  // b\n  /* c\n d */ return x + 1;\n}\n"
    same = "int f(int x) {\n   return x + 1;\n}\n// other words\n"
    other = "int f(int x) {\n  return x + 2;\n}\n"
    c = bench.code_without_comments
    assert c(src) == c(same)
    assert c(src) != c(other)
    assert "a" not in c(src).split() and "return x + 1;" in c(src)

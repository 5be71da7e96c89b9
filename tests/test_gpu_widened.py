"""GPU-vs-oracle parity of the widened rows: SiLU and SwiGLU experts,
expert-choice routing, slot-major drops, min_capacity, FP8 (E4M3) expert
weights, the router z-loss and logits outputs, and the auxiliary-loss-free
bias step.  Stages are also run
on the oracle's own upstream results (bit-exact integer dispatch); the whole
layer is compared element by element on small cases and on sampled tokens at
the benchmark sizes."""
import numpy as np
import pytest
import torch

import moe_workloads as wl
from oracle import moe_oracle as O
from tests import _helpers as h

pytestmark = pytest.mark.gpu

SMALL = ["small_silu", "small_swiglu", "swiglu_pairs", "small_expert_choice",
         "expert_choice_ragged", "expert_choice_all", "many_experts_choice",
         "slot_major_capacity", "min_capacity", "small_fp8", "fp8_pairs", "swiglu_fp8",
         "fp8_decode_small", "fp8_capacity_small"]
FULL_EXACT = ["mixtral_swiglu_decode", "mixtral_decode_fp8"]
FULL_SAMPLED = ["moelayer_expert_choice", "mixtral_swiglu_prefill", "mixtral_prefill_fp8"]
# logit gap under which the fp32 router and the float64 oracle may order two
# tokens of one expert's column differently (far above fp32 rounding of the
# logits, far below the gaps of distinct random logits)
EC_SLACK = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_mixture_experts_72_b300 as m
    return m


_CACHE = {}


def _case(name, tokens=None):
    key = (name, None if tokens is None else len(tokens))
    if key in _CACHE:
        return _CACHE[key]
    _CACHE.clear()
    torch.cuda.empty_cache()
    w = wl.get_workload(name)
    x_bits, weights, router = h.upload(w)
    ref = h.oracle_forward(w, x_bits, router, tokens=tokens)
    val = (w, h.config_of(w), x_bits, h.bf16_dev(x_bits), weights, router, ref)
    _CACHE[key] = val
    return val


def _i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()


def _check_expert_choice(w, ref, perm_g, offsets_g):
    """Each expert's token set equals the oracle's, except where its C-th and
    (C+1)-th logits are within EC_SLACK; there the GPU's set must still be a
    top-C of the oracle's logits up to that slack.  Returns the experts whose
    sets differ."""
    N = w.N
    C = int(ref["offsets"][1] - ref["offsets"][0]) if N > 0 else 0
    assert np.array_equal(offsets_g, ref["offsets"])
    l = ref["logits"]
    differ = []
    for e in range(N):
        a_g = perm_g[e * C:(e + 1) * C]
        a_r = ref["perm"][e * C:(e + 1) * C]
        assert np.all(a_g % N == e)
        tg = a_g // N
        assert np.all(np.diff(tg) > 0), "rows of an expert must be in token order"
        if np.array_equal(a_g, a_r):
            continue
        assert ref["ec_margin"][e] < EC_SLACK, f"expert {e} differs without a near tie"
        rest = np.setdiff1d(np.arange(w.T), tg)
        if rest.size:
            assert l[tg, e].min() >= l[rest, e].max() - EC_SLACK
        differ.append(e)
    return differ


def _check_forward(m, name, tokens=None):
    w, cfg, xb, x, W, router, ref = _case(name, tokens)
    outs = m.alloc_outputs(cfg, "cuda", want_probs=True, want_logits=True)
    ws = m.make_workspace(cfg)
    out = m.moe_forward(cfg, W, x, outputs=outs, ws=ws)
    assert m.moe_workspace_status(ws) == 0
    np.testing.assert_allclose(outs["probs"].cpu().numpy(), ref["probs"], rtol=0, atol=h.PROB_ATOL)
    np.testing.assert_allclose(outs["p_mean"].cpu().numpy(), ref["p"], rtol=0, atol=h.PROB_ATOL)
    lg = outs["logits"].cpu().numpy()
    np.testing.assert_allclose(lg, ref["logits"], rtol=1e-5, atol=1e-5)
    h.laux_close(float(outs["l_aux"].item()), ref["l_aux"])
    z = float(outs["z_loss"].item())
    assert abs(z - ref["z_loss"]) <= 1e-5 * abs(ref["z_loss"]) + 1e-12, (z, ref["z_loss"])
    toks = np.arange(w.T) if tokens is None else np.asarray(tokens)
    got = h.bf16_host(out[torch.from_numpy(toks).cuda()])
    if w.routing == "expert":
        differ = _check_expert_choice(w, ref, outs["perm"].cpu().numpy(),
                                      outs["offsets"].cpu().numpy())
        inv_g = outs["inv"].cpu().numpy().reshape(w.T, w.N)
        same = ((inv_g >= 0) == (ref["inv"].reshape(w.T, w.N) >= 0)).all(1)
        assert same.mean() > 0.99 if not differ else same.mean() > 0.9
        if not differ:
            assert np.array_equal(outs["inv"].cpu().numpy(), ref["inv"])
        keep = same[toks]
    else:
        diff = h.check_routing(ref, outs["topk_idx"].cpu().numpy(), outs["topk_w"].cpu().numpy(),
                               w.k)
        keep = np.ones(toks.size, bool)
        if not diff:
            R = int(ref["offsets"][-1])
            assert np.array_equal(outs["offsets"].cpu().numpy(), ref["offsets"])
            assert np.array_equal(outs["perm"].cpu().numpy()[:R], ref["perm"])
            assert np.array_equal(outs["inv"].cpu().numpy(), ref["inv"])
        else:
            inv_g = outs["inv"].cpu().numpy().reshape(w.T, w.k)
            same = (outs["topk_idx"].cpu().numpy() == ref["idx"]).all(1) & \
                ((inv_g >= 0) == (ref["inv"].reshape(w.T, w.k) >= 0)).all(1)
            assert same.mean() > 0.99
            keep = same[toks]
    h.assert_close_out(got[keep], ref["out"][keep])
    return toks[keep]


@pytest.mark.parametrize("name", SMALL + FULL_EXACT)
def test_forward(name, _lib):
    _check_forward(_lib, name)


@pytest.mark.parametrize("name", FULL_SAMPLED)
def test_forward_full_size_sampled(name, _lib):
    """Random tokens plus the owners of the first and last row of every row
    tile of every expert: each M-tile of the expert GEMMs is checked."""
    w = wl.get_workload(name)
    tokens, offsets, perm = h.tile_tokens(w, wl.gen_x(w, 0), wl.gen_router(w, 0), n_random=40)
    checked = _check_forward(_lib, name, tokens=tokens)
    h.assert_tiles_covered(offsets, perm, w.N if w.routing == "expert" else w.k, checked)


@pytest.mark.parametrize("name", ["small_expert_choice", "expert_choice_ragged",
                                  "expert_choice_all", "many_experts_choice"])
def test_expert_choice_stage_bit_exact(name, _lib):
    """The dispatch alone on the oracle's logits rounded to fp32: the oracle
    selects on the same values, so the result must match bit for bit."""
    m = _lib
    w, cfg, xb, x, W, router, ref = _case(name)
    l32 = ref["logits"].astype(np.float32)
    want = O.expert_choice(l32.astype(np.float64), O.capacity(w.T, w.N, w.capacity_factor,
                                                              w.min_capacity))
    p32 = torch.from_numpy(ref["p"].astype(np.float32)).cuda()
    d = m.moe_expert_choice(cfg, torch.from_numpy(l32).cuda(), p32)
    torch.cuda.synchronize()
    assert np.array_equal(d["counts"].cpu().numpy(), want["counts"])
    assert np.array_equal(d["offsets"].cpu().numpy(), want["offsets"])
    assert np.array_equal(d["perm"].cpu().numpy(), want["perm"])
    assert np.array_equal(d["inv"].cpu().numpy(), want["inv"])
    np.testing.assert_allclose(d["f"].cpu().numpy(), 1.0 / w.N, rtol=1e-7)
    h.laux_close(float(d["l_aux"].item()), float(w.aux_alpha * np.sum(ref["p"])))


def test_expert_choice_ties_take_lower_tokens(_lib):
    """Integer-valued logits with many equal entries: the lower tokens win."""
    m = _lib
    rng = np.random.default_rng(5)
    T, N = 500, 8
    l = rng.integers(-3, 4, size=(T, N)).astype(np.float32)
    cfg = m.MoEConfig(T=T, H=64, F=64, N=N, k=1, capacity_factor=1.3, routing="expert")
    C = O.capacity(T, N, 1.3)
    want = O.expert_choice(l.astype(np.float64), C)
    d = m.moe_expert_choice(cfg, torch.from_numpy(l).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(d["perm"].cpu().numpy(), want["perm"])
    assert np.array_equal(d["inv"].cpu().numpy(), want["inv"])


@pytest.mark.parametrize("name", ["slot_major_capacity", "min_capacity"])
def test_permute_stage_bit_exact(name, _lib):
    m = _lib
    w, cfg, xb, x, W, router, ref = _case(name)
    assert m.moe_capacity(cfg) == O.capacity(w.T, w.N, w.capacity_factor, w.min_capacity)
    d = m.moe_permute(cfg, _i32(ref["idx"]), torch.from_numpy(ref["p"].astype(np.float32)).cuda())
    torch.cuda.synchronize()
    R = int(ref["offsets"][-1])
    assert np.array_equal(d["counts"].cpu().numpy(), ref["counts"])
    assert np.array_equal(d["offsets"].cpu().numpy(), ref["offsets"])
    assert np.array_equal(d["perm"].cpu().numpy()[:R], ref["perm"])
    assert np.array_equal(d["inv"].cpu().numpy(), ref["inv"])


@pytest.mark.parametrize("name", ["tiny", "small_shared", "wide_router", "many_experts"])
def test_route_logits_and_z_loss(name, _lib):
    m = _lib
    w, cfg, xb, x, W, router, ref = _case(name)
    idx, tw, probs, p_mean, logits, z = m.moe_route(cfg, x, W.Wg, W.bg, W.sel_bias,
                                                    want_probs=True, want_logits=True,
                                                    want_z=True)
    torch.cuda.synchronize()
    h.check_routing(ref, idx.cpu().numpy(), tw.cpu().numpy(), w.k)
    np.testing.assert_allclose(logits.cpu().numpy(), ref["logits"], rtol=1e-5, atol=1e-5)
    zr = O.z_loss(ref["logits"])
    assert abs(float(z.item()) - zr) <= 1e-5 * abs(zr), (float(z.item()), zr)


def test_update_sel_bias_matches_oracle(_lib):
    m = _lib
    rng = np.random.default_rng(9)
    N = 300
    counts = rng.integers(0, 50, size=N).astype(np.int32)
    counts[:5] = int(round(counts.mean()))  # some may sit exactly at the mean
    b0 = rng.uniform(-0.1, 0.1, size=N).astype(np.float32)
    cfg = m.MoEConfig(T=64, H=64, F=64, N=N, k=2)
    b = torch.from_numpy(b0.copy()).cuda()
    m.moe_update_sel_bias(cfg, _i32(counts), b, 0.001)
    torch.cuda.synchronize()
    step = np.sign(counts.astype(np.int64) * N - counts.astype(np.int64).sum()).astype(np.float32)
    want = b0 + np.float32(0.001) * step  # float32 arithmetic, as the kernel
    assert np.array_equal(b.cpu().numpy(), want)
    # and the step is the oracle's rule
    np.testing.assert_allclose(O.update_sel_bias(b0, counts, 0.001), want, rtol=0, atol=1e-7)


def test_widened_launch_counts_and_trace(_lib):
    m = _lib
    for name in ["small_expert_choice", "small_swiglu", "slot_major_capacity"]:
        w, cfg, xb, x, W, router, ref = _case(name)
        n = m.moe_forward_num_launches(cfg)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        m.moe_forward(cfg, W, x, trace_events=ev)
        torch.cuda.synchronize()
        assert all(ev[i].elapsed_time(ev[i + 1]) >= 0 for i in range(n))


def test_fp8_group_above_bound_is_reported(_lib):
    """FP8 launches of the token-row kernel with groups below 128 rows copy at
    most the rows one expert can hold (here T = 100, so 112); offsets that
    give an expert 200 rows (more than a token-choice dispatch can) must be
    reported in the status word, not computed silently.  A dispatch within
    the bound leaves the word 0.  (100 rows per expert on average: not the
    operand-swapped decode kernel, which takes any row count.)"""
    m = _lib
    T, H, F = 100, 64, 64
    cfg = m.MoEConfig(T=T, H=H, F=F, N=2, k=2, weight_dtype="e4m3")
    assert "expert_ffn" in m.moe_forward_launch_names(cfg)
    dev = "cuda"
    g = torch.Generator().manual_seed(3)
    codes = lambda *s: torch.randint(0, 0x7E, s, generator=g, dtype=torch.uint8).to(dev)
    weights = m.MoEWeights(Wg=torch.zeros((2, H), device=dev), W1=codes(2, F, H),
                           W2=codes(2, H, F), s1=torch.full((2, F), 1e-3, device=dev),
                           s2=torch.full((2, H), 1e-3, device=dev))
    x = torch.randn((T, H), generator=g).to(torch.bfloat16).to(dev)
    perm = torch.arange(T * 2, dtype=torch.int32, device=dev)
    topk_w = torch.full((T, 2), 0.5, dtype=torch.float32, device=dev)
    ws = m.make_workspace(cfg, dev)
    ok_offsets = torch.tensor([0, T, 2 * T], dtype=torch.int32, device=dev)
    m.moe_expert_ffn(cfg, x, perm, ok_offsets, topk_w, weights, ws=ws)
    assert m.moe_workspace_status(ws) == 0
    bad_offsets = torch.tensor([0, 2 * T, 2 * T], dtype=torch.int32, device=dev)
    m.moe_expert_ffn(cfg, x, perm, bad_offsets, topk_w, weights, ws=ws)
    assert m.moe_workspace_status(ws) == 1   # MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("weight_dtype", ["bf16", "e4m3"])
def test_decode_kernel_takes_any_group_size(weight_dtype, _lib):
    """The operand-swapped decode kernel computes groups of any size, in token
    chunks: offsets that give one expert every row (80, more than a
    token-choice dispatch can, so several chunks) and the other none match
    the oracle row by row."""
    m = _lib
    T, H, F, N = 40, 64, 96, 2
    cfg = m.MoEConfig(T=T, H=H, F=F, N=N, k=2, weight_dtype=weight_dtype)
    assert "expert_ffn_decode" in m.moe_forward_launch_names(cfg)
    dev = "cuda"
    rng = np.random.default_rng(5)
    if weight_dtype == "e4m3":
        c1 = rng.integers(0, 0x7E, (N, F, H), dtype=np.uint8) | (rng.integers(0, 2, (N, F, H), dtype=np.uint8) << 7)
        c2 = rng.integers(0, 0x7E, (N, H, F), dtype=np.uint8) | (rng.integers(0, 2, (N, H, F), dtype=np.uint8) << 7)
        s1 = np.full((N, F), 2e-3, np.float32)
        s2 = np.full((N, H), 2e-3, np.float32)
        W1f = np.stack([O.dequantize_rows(c1[e], s1[e]) for e in range(N)])
        W2f = np.stack([O.dequantize_rows(c2[e], s2[e]) for e in range(N)])
        weights = m.MoEWeights(Wg=torch.zeros((N, H), device=dev),
                               W1=torch.from_numpy(c1).to(dev), W2=torch.from_numpy(c2).to(dev),
                               s1=torch.from_numpy(s1).to(dev), s2=torch.from_numpy(s2).to(dev))
    else:
        W1b = wl.f32_to_bf16_bits(rng.standard_normal((N, F, H)).astype(np.float32) / 8)
        W2b = wl.f32_to_bf16_bits(rng.standard_normal((N, H, F)).astype(np.float32) / 10)
        W1f, W2f = wl.bf16_bits_to_f64(W1b), wl.bf16_bits_to_f64(W2b)
        weights = m.MoEWeights(Wg=torch.zeros((N, H), device=dev),
                               W1=h.bf16_dev(W1b), W2=h.bf16_dev(W2b))
    xb = wl.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    x = h.bf16_dev(xb)
    perm = torch.arange(T * 2, dtype=torch.int32, device=dev)   # row r <- assignment r
    w_np = rng.random((T, 2)).astype(np.float32)
    topk_w = torch.from_numpy(w_np).to(dev)
    offsets = torch.tensor([0, 2 * T, 2 * T], dtype=torch.int32, device=dev)
    ws = m.make_workspace(cfg, dev)
    y, _ = m.moe_expert_ffn(cfg, x, perm, offsets, topk_w, weights, ws=ws)
    assert m.moe_workspace_status(ws) == 0
    a = np.arange(2 * T)
    xs = wl.bf16_bits_to_f64(xb)[a // 2]
    want = w_np.reshape(-1)[a][:, None] * O.expert_ffn(xs, W1f[0], None, W2f[0], None)
    h.assert_close_out(h.bf16_host(y[:2 * T]), want, "rows of the one expert")

"""moe_permute_static: the dispatch step without a workspace.

Some callers cannot allocate device memory at the point where they run the
layer - a plugin inside an inference engine that owns all GPU memory and
forbids allocation on its execution path, or a service that reserves every
byte at start-up so no request can fail on an allocation.  moe_permute_static
serves them: it takes only inputs and outputs and keeps its scratch in a
fixed device array inside the library.

This test calls it through the C ABI twice in a row: first at the array's
size limit (256 experts), then a smaller case with another expert count, so
the second call reads histograms laid out with a different stride over the
first call's leftovers.  Each result is checked against the CPU oracle's
dispatch (bit-exact integers, L_aux within 1e-5 relative) and against
moe_permute, the workspace version.  It lives in a file of its own that
pytest collects last.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu


def _idx(T, N, k, seed):
    """Seeded top-k index sets (distinct experts per token, skewed load)."""
    rng = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, N + 1) ** 1.1
    p /= p.sum()
    keys = rng.random((T, N)) ** (1.0 / p)[None, :]   # weighted sampling without replacement
    return np.argsort(-keys, axis=1, kind="stable")[:, :k].astype(np.int32)


def _run(lib, cfg, fn, idx, p_mean, ws=None):
    from sparse_mixture_experts_72_b300 import _lib
    T, N, k = cfg.T, cfg.N, cfg.k
    R = int(lib.moe_max_rows(C.byref(cfg)))
    o = dict(counts=torch.full((N,), -7, dtype=torch.int32, device="cuda"),
             offsets=torch.full((N + 1,), -7, dtype=torch.int32, device="cuda"),
             perm=torch.full((max(R, 1),), -7, dtype=torch.int32, device="cuda"),
             inv=torch.full((T * k,), -7, dtype=torch.int32, device="cuda"),
             f=torch.full((N,), -7.0, dtype=torch.float32, device="cuda"),
             l_aux=torch.full((1,), -7.0, dtype=torch.float32, device="cuda"))
    ptr = lambda t: C.c_void_p(t.data_ptr())
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = [C.byref(cfg), ptr(idx), ptr(p_mean), ptr(o["counts"]), ptr(o["offsets"]),
            ptr(o["perm"]), ptr(o["inv"]), ptr(o["f"]), ptr(o["l_aux"])]
    if ws is None:
        st = fn(*args, stream)
    else:
        st = fn(*args, ptr(ws), C.c_size_t(ws.numel()), stream)
    assert st == _lib.MOE_OK, _lib.STATUS_NAMES.get(st, st)
    torch.cuda.synchronize()
    R_kept = int(o["offsets"][-1].item())
    return {n: t.cpu().numpy() for n, t in o.items()}, R_kept


def test_static_scratch_matches_workspace_version_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mixture_experts_72_b300 import _lib
    lib = _lib.load()
    cases = [
        # (T, N, k, capacity_factor): the size limit, then a smaller
        # capacity-limited case with fewer experts
        (_lib.MOE_STATIC_MAX_ASSIGNMENTS // 8, _lib.MOE_STATIC_MAX_EXPERTS, 8, 1.25),
        (1000, 8, 2, 1.0),
    ]
    for i, (T, N, k, cf) in enumerate(cases):
        cfg = _lib.MoeConfig(T=T, H=64, F=64, N=N, k=k, capacity_factor=cf, F_shared=0,
                             aux_alpha=0.01)
        idx = torch.from_numpy(_idx(T, N, k, seed=i)).cuda()
        p_mean = torch.from_numpy(np.random.default_rng(10 + i).dirichlet(np.ones(N))
                                  .astype(np.float32)).cuda()
        ws = torch.empty(int(lib.moe_workspace_size(C.byref(cfg))), dtype=torch.uint8,
                         device="cuda")
        got, R = _run(lib, cfg, lib.moe_permute_static, idx, p_mean)
        want, R_w = _run(lib, cfg, lib.moe_permute, idx, p_mean, ws)
        assert R == R_w
        # the oracle's dispatch of the same indices
        idx_h = idx.cpu().numpy()
        ref = O.permute(idx_h, N, O.capacity(T, N, cf))
        for name in ("counts", "offsets", "inv"):
            assert np.array_equal(got[name], ref[name]), name
        assert np.array_equal(got["perm"][:R], ref["perm"])
        P = np.tile(p_mean.cpu().numpy().astype(np.float64), (T, 1))   # column means = p_mean
        lb = O.load_balance(P, ref["counts"], k, 0.01)
        np.testing.assert_allclose(got["f"], lb["f"], rtol=1e-6, atol=0)
        assert abs(got["l_aux"][0] - lb["l_aux"]) <= 1e-5 * abs(lb["l_aux"])
        for name in ("counts", "offsets", "inv"):
            assert np.array_equal(got[name], want[name]), name
        assert np.array_equal(got["perm"][:R], want["perm"][:R])
        np.testing.assert_allclose(got["f"], want["f"], rtol=1e-6, atol=0)
        assert abs(got["l_aux"][0] - want["l_aux"][0]) <= 1e-5 * abs(want["l_aux"][0])
        assert got["counts"].sum() == T * k


def test_static_rejects_sizes_beyond_its_array():
    from sparse_mixture_experts_72_b300 import _lib
    lib = _lib.load()
    too_many = _lib.MoeConfig(T=_lib.MOE_STATIC_MAX_ASSIGNMENTS + 1, H=64, F=64, N=8, k=1,
                              capacity_factor=0.0, F_shared=0, aux_alpha=0.01)
    wide = _lib.MoeConfig(T=16, H=64, F=64, N=_lib.MOE_STATIC_MAX_EXPERTS + 1, k=1,
                          capacity_factor=0.0, F_shared=0, aux_alpha=0.01)
    fake = C.c_void_p(0x10000)  # rejected on the host before any use
    for cfg in (too_many, wide):
        st = lib.moe_permute_static(C.byref(cfg), fake, fake, fake, fake, fake, fake, fake, fake,
                                    None)
        assert st == 2  # MOE_ERR_UNSUPPORTED

"""Failure detection on the GPU without a fault: a GEMM launch whose TMA
producer is silenced (the library's failure-injection hook) must give up on
its bounded waits, record MOE_ERR_TIMEOUT in the workspace status word and
return, leaving the CUDA context usable; the next call must clear the word
and produce the oracle's result again."""
import time

import numpy as np
import pytest
import torch

import moe_workloads as wl
from tests import _helpers as h

pytestmark = pytest.mark.gpu

MOE_ERR_TIMEOUT = 5


@pytest.fixture(scope="module")
def m():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_mixture_experts_72_b300 as lib
    return lib


@pytest.mark.parametrize("name", ["small_shared", "moelayer"])
def test_silenced_producer_times_out_and_context_survives(m, name):
    # small_shared runs one-CTA tiles, moelayer CTA-pair tiles
    w = wl.get_workload(name)
    x_bits, W, router = h.upload(w)
    tok = h.sample_tokens(w.T, 16)
    ref = h.oracle_forward(w, x_bits, router, tokens=tok)
    cfg = h.config_of(w)
    x = h.bf16_dev(x_bits)
    ws = m.make_workspace(cfg)
    outs = m.alloc_outputs(cfg, "cuda")
    m.moe_forward(cfg, W, x, outputs=outs, ws=ws)   # routing and dispatch on the GPU
    assert m.moe_workspace_status(ws) == 0

    m.moe_debug_suppress_gemm_producer(1)           # the first expert GEMM hears nothing
    t0 = time.monotonic()
    m.moe_expert_ffn(cfg, x, outs["perm"], outs["offsets"], outs["topk_w"], W, ws=ws)
    status = m.moe_workspace_status(ws)
    waited = time.monotonic() - t0
    assert status == MOE_ERR_TIMEOUT
    assert waited < 60.0

    # the context still works, the status word is cleared by the next call,
    # and the hook has been consumed
    out = m.moe_forward(cfg, W, x, outputs=outs, ws=ws)
    assert m.moe_workspace_status(ws) == 0
    idx = outs["topk_idx"].cpu().numpy()
    h.check_routing(ref, idx, outs["topk_w"].cpu().numpy(), w.k)
    same = (idx[tok] == ref["idx"][tok]).all(1)      # near-tie tokens may differ
    assert same.mean() > 0.9
    got = h.bf16_host(out[torch.from_numpy(tok).cuda()])
    h.assert_close_out(got[same], ref["out"][same])

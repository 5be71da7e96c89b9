"""Sparse Mixture-of-Experts FFN forward pass on B300 (sm_103a).

Thin Python binding over the C ABI in include/moe.h: the functions below
have the C entry points' names, check tensor dtypes/devices/shapes, pass
raw device pointers and the current CUDA stream, and raise ``MoeError`` on a
non-OK status.  Every step of the layer runs in the library's CUDA kernels;
PyTorch only provides device memory and streams.  Importing the package
fails if the library has not been built.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

from . import _lib
from ._lib import MOE_TRACE_MAX_EVENTS, MoeError, check

_L = _lib.load()

__all__ = ["MoEConfig", "MoEWeights", "MoeError", "moe_workspace_size", "moe_max_rows",
           "moe_capacity", "moe_forward_num_launches", "moe_forward_launch_names", "moe_route",
           "moe_permute",
           "moe_permute_static",
           "moe_expert_ffn", "moe_combine", "moe_forward", "moe_workspace_status",
           "moe_debug_suppress_gemm_producer", "moe_expert_choice", "moe_update_sel_bias",
           "moe_forward_host",
           "MoEForwardGraph", "alloc_outputs",
           "make_workspace", "library_path", "MOE_TRACE_MAX_EVENTS"]


def library_path() -> str:
    return _lib.LIB_PATH


@dataclass(frozen=True)
class MoEConfig:
    T: int
    H: int
    F: int
    N: int
    k: int
    capacity_factor: float = 0.0
    F_shared: int = 0
    aux_alpha: float = 0.01
    routing: str = "token"       # "token" (top-k per token) | "expert" (top-C per expert)
    activation: str = "gelu"     # "gelu" | "silu" | "swiglu" (W1 [N, 2F, H])
    min_capacity: int = 0
    drop_order: str = "token"    # "token" | "slot"
    weight_dtype: str = "bf16"   # expert weights: "bf16" | "e4m3" (codes + fp32 row scales)

    def c(self) -> _lib.MoeConfig:
        return _lib.MoeConfig(self.T, self.H, self.F, self.N, self.k,
                              float(self.capacity_factor), self.F_shared, float(self.aux_alpha),
                              _lib.ROUTING[self.routing], _lib.ACTIVATION[self.activation],
                              int(self.min_capacity), _lib.DROP_ORDER[self.drop_order],
                              _lib.WEIGHT_DTYPE[self.weight_dtype])

    @property
    def slots(self) -> int:
        """Assignments per token: k, or N for expert choice (a = t * slots + j)."""
        return self.N if self.routing == "expert" else self.k

    @property
    def w1_rows(self) -> int:
        return 2 * self.F if self.activation == "swiglu" else self.F


@dataclass
class MoEWeights:
    """Layer parameters.  The expert matrices W1, W2, W1s, W2s are bf16, or
    with ``weight_dtype="e4m3"`` E4M3 codes (uint8 or torch.float8_e4m3fn)
    with one fp32 scale per row in s1, s2, s1s, s2s."""
    Wg: torch.Tensor                     # [N, H] fp32
    W1: torch.Tensor                     # [N, F, H] bf16
    W2: torch.Tensor                     # [N, H, F] bf16
    bg: Optional[torch.Tensor] = None    # [N] fp32
    sel_bias: Optional[torch.Tensor] = None  # [N] fp32
    b1: Optional[torch.Tensor] = None    # [N, F] bf16
    b2: Optional[torch.Tensor] = None    # [N, H] bf16
    W1s: Optional[torch.Tensor] = None   # [Fs, H] bf16
    b1s: Optional[torch.Tensor] = None   # [Fs] bf16
    W2s: Optional[torch.Tensor] = None   # [H, Fs] bf16
    b2s: Optional[torch.Tensor] = None   # [H] bf16
    s1: Optional[torch.Tensor] = None    # e4m3: [N, F] ([N, 2F] SwiGLU) fp32 row scales of W1
    s2: Optional[torch.Tensor] = None    # e4m3: [N, H] fp32 row scales of W2
    s1s: Optional[torch.Tensor] = None   # e4m3: [Fs] ([2Fs]) fp32 row scales of W1s
    s2s: Optional[torch.Tensor] = None   # e4m3: [H] fp32 row scales of W2s

    def c(self, cfg: MoEConfig) -> _lib.MoeWeights:
        N, H, F, Fs = cfg.N, cfg.H, cfg.F, cfg.F_shared
        g = 2 if cfg.activation == "swiglu" else 1   # SwiGLU: gate and up rows
        fp8 = cfg.weight_dtype == "e4m3"
        wt = (torch.uint8, torch.float8_e4m3fn) if fp8 else torch.bfloat16
        no_scale = not fp8
        return _lib.MoeWeights(
            _p(self.Wg, torch.float32, (N, H), "Wg"),
            _p(self.bg, torch.float32, (N,), "bg", True),
            _p(self.sel_bias, torch.float32, (N,), "sel_bias", True),
            _p(self.W1, wt, (N, g * F, H), "W1"),
            _p(self.b1, torch.bfloat16, (N, g * F), "b1", True),
            _p(self.W2, wt, (N, H, F), "W2"),
            _p(self.b2, torch.bfloat16, (N, H), "b2", True),
            _p(self.W1s, wt, (g * Fs, H), "W1s", Fs == 0),
            _p(self.b1s, torch.bfloat16, (g * Fs,), "b1s", True),
            _p(self.W2s, wt, (H, Fs), "W2s", Fs == 0),
            _p(self.b2s, torch.bfloat16, (H,), "b2s", True),
            _p(None if no_scale else self.s1, torch.float32, (N, g * F), "s1", no_scale),
            _p(None if no_scale else self.s2, torch.float32, (N, H), "s2", no_scale),
            _p(None if no_scale else self.s1s, torch.float32, (g * Fs,), "s1s",
               no_scale or Fs == 0),
            _p(None if no_scale else self.s2s, torch.float32, (H,), "s2s", no_scale or Fs == 0))


def _p(t: Optional[torch.Tensor], dtype, shape, name, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    allowed = dtype if isinstance(dtype, tuple) else (dtype,)
    if t.dtype not in allowed:
        raise TypeError(f"{name} must be {' or '.join(map(str, allowed))}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return C.c_void_p(t.data_ptr()) if t.numel() > 0 else None


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def moe_workspace_size(cfg: MoEConfig) -> int:
    return int(_L.moe_workspace_size(C.byref(cfg.c())))


def moe_max_rows(cfg: MoEConfig) -> int:
    return int(_L.moe_max_rows(C.byref(cfg.c())))


def moe_capacity(cfg: MoEConfig) -> Optional[int]:
    v = int(_L.moe_capacity(C.byref(cfg.c())))
    return None if v < 0 else v


def moe_forward_num_launches(cfg: MoEConfig) -> int:
    return int(_L.moe_forward_num_launches(C.byref(cfg.c())))


def moe_forward_launch_names(cfg: MoEConfig) -> list:
    """Names of the launches moe_forward makes, in order (one per trace interval)."""
    c = cfg.c()
    n = moe_forward_num_launches(cfg)
    return [_L.moe_forward_launch_name(C.byref(c), i).decode() for i in range(n)]


def make_workspace(cfg: MoEConfig, device=None) -> torch.Tensor:
    n = moe_workspace_size(cfg)
    if n == 0:
        raise ValueError(f"invalid configuration {cfg}")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def _ws(cfg, ws, device):
    if ws is None:
        ws = make_workspace(cfg, device)
    return ws, C.c_void_p(ws.data_ptr()), C.c_size_t(ws.numel())


def moe_route(cfg: MoEConfig, x, Wg, bg=None, sel_bias=None, *, want_probs=False,
              want_logits=False, want_z=False, ws=None, stream=None):
    """Returns (topk_idx int32 [T,k], topk_w fp32 [T,k], probs fp32 [T,N] or None, p_mean [N]);
    with want_logits / want_z also logits fp32 [T,N] and z_loss fp32 [1] (in that order).
    For expert choice topk_idx and topk_w are None."""
    dev = x.device
    T, N, k = cfg.T, cfg.N, cfg.k
    ec = cfg.routing == "expert"
    idx = None if ec else torch.empty((T, k), dtype=torch.int32, device=dev)
    w = None if ec else torch.empty((T, k), dtype=torch.float32, device=dev)
    probs = torch.empty((T, N), dtype=torch.float32, device=dev) if want_probs else None
    logits = torch.empty((T, N), dtype=torch.float32, device=dev) if want_logits else None
    z = torch.empty(1, dtype=torch.float32, device=dev) if want_z else None
    p_mean = torch.empty(N, dtype=torch.float32, device=dev)
    ws, wsp, wsn = _ws(cfg, ws, dev)
    st = _L.moe_route(C.byref(cfg.c()), _p(x, torch.bfloat16, (T, cfg.H), "x", T == 0),
                      _p(Wg, torch.float32, (N, cfg.H), "Wg"),
                      _p(bg, torch.float32, (N,), "bg", True),
                      _p(sel_bias, torch.float32, (N,), "sel_bias", True),
                      _p(idx, torch.int32, None, "idx", True), _p(w, torch.float32, None, "w", True),
                      _p(probs, torch.float32, None, "probs", True),
                      _p(logits, torch.float32, None, "logits", True),
                      _p(p_mean, torch.float32, None, "p_mean"),
                      _p(z, torch.float32, None, "z_loss", True), wsp, wsn, _stream(stream))
    check(st, "moe_route")
    res = (idx, w, probs, p_mean)
    if want_logits:
        res += (logits,)
    if want_z:
        res += (z,)
    return res


def moe_expert_choice(cfg: MoEConfig, logits, p_mean=None, *, stream=None) -> dict:
    """Expert-choice dispatch.  Returns dict(counts, offsets, perm, inv [T*N], f, l_aux)."""
    dev = logits.device
    T, N = cfg.T, cfg.N
    R = moe_max_rows(cfg)
    out = dict(counts=torch.empty(N, dtype=torch.int32, device=dev),
               offsets=torch.empty(N + 1, dtype=torch.int32, device=dev),
               perm=torch.empty(max(R, 0), dtype=torch.int32, device=dev),
               inv=torch.empty(T * N, dtype=torch.int32, device=dev),
               f=torch.empty(N, dtype=torch.float32, device=dev),
               l_aux=torch.empty(1, dtype=torch.float32, device=dev) if p_mean is not None else None)
    st = _L.moe_expert_choice(C.byref(cfg.c()), _p(logits, torch.float32, (T, N), "logits", True),
                              _p(p_mean, torch.float32, (N,), "p_mean", True),
                              _p(out["counts"], torch.int32, None, "counts"),
                              _p(out["offsets"], torch.int32, None, "offsets"),
                              _p(out["perm"], torch.int32, None, "perm", True),
                              _p(out["inv"], torch.int32, None, "inv", True),
                              _p(out["f"], torch.float32, None, "f"),
                              _p(out["l_aux"], torch.float32, None, "l_aux", True),
                              _stream(stream))
    check(st, "moe_expert_choice")
    return out


def moe_update_sel_bias(cfg: MoEConfig, counts, sel_bias, gamma: float, *, stream=None):
    """In place: sel_bias[e] += gamma * sign(counts[e] - mean(counts))."""
    st = _L.moe_update_sel_bias(C.byref(cfg.c()), _p(counts, torch.int32, (cfg.N,), "counts"),
                                _p(sel_bias, torch.float32, (cfg.N,), "sel_bias"),
                                C.c_float(gamma), _stream(stream))
    check(st, "moe_update_sel_bias")
    return sel_bias


def moe_permute(cfg: MoEConfig, topk_idx, p_mean=None, *, ws=None, stream=None) -> dict:
    """Returns dict(counts, offsets, perm, inv, f, l_aux) as device tensors."""
    dev = topk_idx.device
    T, N, k = cfg.T, cfg.N, cfg.k
    R = moe_max_rows(cfg)
    out = dict(counts=torch.empty(N, dtype=torch.int32, device=dev),
               offsets=torch.empty(N + 1, dtype=torch.int32, device=dev),
               perm=torch.empty(max(R, 0), dtype=torch.int32, device=dev),
               inv=torch.empty(T * k, dtype=torch.int32, device=dev),
               f=torch.empty(N, dtype=torch.float32, device=dev),
               l_aux=torch.empty(1, dtype=torch.float32, device=dev) if p_mean is not None else None)
    ws, wsp, wsn = _ws(cfg, ws, dev)
    st = _L.moe_permute(C.byref(cfg.c()), _p(topk_idx, torch.int32, (T, k), "topk_idx", T == 0),
                        _p(p_mean, torch.float32, (N,), "p_mean", True),
                        _p(out["counts"], torch.int32, None, "counts"),
                        _p(out["offsets"], torch.int32, None, "offsets"),
                        _p(out["perm"], torch.int32, None, "perm", True),
                        _p(out["inv"], torch.int32, None, "inv", True),
                        _p(out["f"], torch.float32, None, "f"),
                        _p(out["l_aux"], torch.float32, None, "l_aux", True),
                        wsp, wsn, _stream(stream))
    check(st, "moe_permute")
    return out


def moe_permute_static(cfg: MoEConfig, topk_idx, p_mean=None, *, stream=None) -> dict:
    """moe_permute without a workspace, for callers that cannot allocate:
    the scratch is a fixed device array inside the library (T*k <= 65536,
    N <= 256).  Calls share that array, so calls that overlap on the GPU race.
    Make the first call on a device before any stream capture.  (This
    binding allocates its output tensors; a caller that cannot allocate
    calls the C entry point with its own buffers.)"""
    dev = topk_idx.device
    T, N, k = cfg.T, cfg.N, cfg.k
    R = moe_max_rows(cfg)
    out = dict(counts=torch.empty(N, dtype=torch.int32, device=dev),
               offsets=torch.empty(N + 1, dtype=torch.int32, device=dev),
               perm=torch.empty(max(R, 0), dtype=torch.int32, device=dev),
               inv=torch.empty(T * k, dtype=torch.int32, device=dev),
               f=torch.empty(N, dtype=torch.float32, device=dev),
               l_aux=torch.empty(1, dtype=torch.float32, device=dev) if p_mean is not None else None)
    st = _L.moe_permute_static(C.byref(cfg.c()),
                               _p(topk_idx, torch.int32, (T, k), "topk_idx", T == 0),
                               _p(p_mean, torch.float32, (N,), "p_mean", True),
                               _p(out["counts"], torch.int32, None, "counts"),
                               _p(out["offsets"], torch.int32, None, "offsets"),
                               _p(out["perm"], torch.int32, None, "perm", True),
                               _p(out["inv"], torch.int32, None, "inv", True),
                               _p(out["f"], torch.float32, None, "f"),
                               _p(out["l_aux"], torch.float32, None, "l_aux", True),
                               _stream(stream))
    check(st, "moe_permute_static")
    return out


def moe_expert_ffn(cfg: MoEConfig, x, perm, offsets, topk_w, weights: MoEWeights, *, ws=None,
                   stream=None):
    """Returns (y bf16 [max_rows, H] (first offsets[N] rows valid), y_shared bf16 [T, H] or None)."""
    dev = x.device
    R = moe_max_rows(cfg)
    y = torch.empty((max(R, 0), cfg.H), dtype=torch.bfloat16, device=dev)
    ys = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev) if cfg.F_shared > 0 else None
    ws, wsp, wsn = _ws(cfg, ws, dev)
    wc = weights.c(cfg)
    st = _L.moe_expert_ffn(C.byref(cfg.c()), _p(x, torch.bfloat16, (cfg.T, cfg.H), "x", True),
                           _p(perm, torch.int32, None, "perm", True),
                           _p(offsets, torch.int32, (cfg.N + 1,), "offsets"),
                           _p(topk_w, torch.float32, (cfg.T, cfg.slots), "topk_w", True),
                           C.byref(wc), _p(y, torch.bfloat16, None, "y", True),
                           _p(ys, torch.bfloat16, None, "y_shared", True), wsp, wsn,
                           _stream(stream))
    check(st, "moe_expert_ffn")
    return y, ys


def moe_combine(cfg: MoEConfig, y, inv, y_shared=None, *, stream=None):
    dev = inv.device
    out = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev)
    st = _L.moe_combine(C.byref(cfg.c()), _p(y, torch.bfloat16, None, "y", True),
                        _p(inv, torch.int32, (cfg.T * cfg.slots,), "inv", True),
                        _p(y_shared, torch.bfloat16, (cfg.T, cfg.H), "y_shared", True),
                        _p(out, torch.bfloat16, None, "out", True), _stream(stream))
    check(st, "moe_combine")
    return out


_OUT_FIELDS = ("topk_idx", "topk_w", "probs", "p_mean", "counts", "offsets", "perm", "inv", "f",
               "l_aux", "z_loss", "logits")


def alloc_outputs(cfg: MoEConfig, device, want_probs=False, want_logits=False) -> dict:
    T, N, k = cfg.T, cfg.N, cfg.k
    i32, f32 = torch.int32, torch.float32
    ec = cfg.routing == "expert"
    return dict(topk_idx=None if ec else torch.empty((T, k), dtype=i32, device=device),
                topk_w=None if ec else torch.empty((T, k), dtype=f32, device=device),
                probs=torch.empty((T, N), dtype=f32, device=device) if want_probs else None,
                p_mean=torch.empty(N, dtype=f32, device=device),
                counts=torch.empty(N, dtype=i32, device=device),
                offsets=torch.empty(N + 1, dtype=i32, device=device),
                perm=torch.empty(max(moe_max_rows(cfg), 0), dtype=i32, device=device),
                inv=torch.empty(T * cfg.slots, dtype=i32, device=device),
                f=torch.empty(N, dtype=f32, device=device),
                l_aux=torch.empty(1, dtype=f32, device=device),
                z_loss=torch.empty(1, dtype=f32, device=device),
                logits=torch.empty((T, N), dtype=f32, device=device) if want_logits else None)


def moe_forward(cfg: MoEConfig, weights: MoEWeights, x, *, out=None, outputs: Optional[dict] = None,
                ws=None, stream=None, trace_events: Optional[Sequence] = None,
                weights_c=None):
    """The whole layer.  ``outputs`` (from ``alloc_outputs``) receives the
    intermediate results; ``trace_events`` is a list of torch.cuda.Event
    (enable_timing=True) recorded around each launch."""
    dev = x.device
    if out is None:
        out = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev)
    oc = None
    if outputs is not None:
        oc = _lib.MoeOutputs(*[(C.c_void_p(outputs[n].data_ptr())
                                if outputs.get(n) is not None and outputs[n].numel() > 0 else None)
                               for n in _OUT_FIELDS])
    ws, wsp, wsn = _ws(cfg, ws, dev)
    wc = weights_c if weights_c is not None else weights.c(cfg)
    ev = None
    if trace_events is not None:
        if len(trace_events) > MOE_TRACE_MAX_EVENTS:
            raise ValueError("too many trace events")
        handles = []
        for e in trace_events:
            if not e.cuda_event:
                e.record()  # torch creates its events lazily, on first record
            handles.append(e.cuda_event)
        handles += [None] * (MOE_TRACE_MAX_EVENTS - len(handles))
        ev = (C.c_void_p * MOE_TRACE_MAX_EVENTS)(*handles)
    st = _L.moe_forward(C.byref(cfg.c()), C.byref(wc),
                        _p(x, torch.bfloat16, (cfg.T, cfg.H), "x", True),
                        _p(out, torch.bfloat16, (cfg.T, cfg.H), "out", True),
                        C.byref(oc) if oc is not None else None, wsp, wsn, _stream(stream), ev)
    check(st, "moe_forward")
    return out


def moe_forward_host(cfg: MoEConfig, weights: MoEWeights, x_host, out_host, x_dev, out_dev, *,
                     outputs: Optional[dict] = None, ws=None, h2d_stream=None,
                     compute_stream=None, d2h_stream=None, weights_c=None):
    """The whole layer on a batch in host memory: H2D of x_host into x_dev
    (h2d_stream), the forward (compute_stream), D2H of out_dev into out_host
    (d2h_stream); the streams default to the current one.  Pin x_host /
    out_host for asynchronous copies.  Returns out_host."""
    for t, n in ((x_host, "x_host"), (out_host, "out_host")):
        if t.is_cuda or t.dtype != torch.bfloat16 or tuple(t.shape) != (cfg.T, cfg.H) or \
                not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous host bf16 tensor of shape {(cfg.T, cfg.H)}")
    oc = None
    if outputs is not None:
        oc = _lib.MoeOutputs(*[(C.c_void_p(outputs[n].data_ptr())
                                if outputs.get(n) is not None and outputs[n].numel() > 0 else None)
                               for n in _OUT_FIELDS])
    ws, wsp, wsn = _ws(cfg, ws, x_dev.device)
    wc = weights_c if weights_c is not None else weights.c(cfg)
    hp = lambda t: C.c_void_p(t.data_ptr()) if t.numel() > 0 else None  # noqa: E731
    st = _L.moe_forward_host(C.byref(cfg.c()), C.byref(wc), hp(x_host),
                             _p(x_dev, torch.bfloat16, (cfg.T, cfg.H), "x_dev", True),
                             _p(out_dev, torch.bfloat16, (cfg.T, cfg.H), "out_dev", True),
                             hp(out_host), C.byref(oc) if oc is not None else None, wsp, wsn,
                             _stream(h2d_stream), _stream(compute_stream),
                             _stream(d2h_stream))
    check(st, "moe_forward_host")
    return out_host


class MoEForwardGraph:
    """One moe_forward over fixed buffers, captured into a CUDA graph.

    The launch sequence, its kernel arguments (including the TMA tensor
    maps) and the buffers are frozen at capture; replay() re-runs the whole
    layer with one graph launch, reading whatever x holds at that time and
    writing out / outputs / ws in place.  A warm-up call before the capture
    sets kernel attributes and fills the library's per-device caches."""

    def __init__(self, cfg: MoEConfig, weights: MoEWeights, x, out, outputs=None, ws=None,
                 trace_events=None):
        self.cfg, self.x, self.out, self.outputs = cfg, x, out, outputs
        self.ws = ws if ws is not None else make_workspace(cfg, x.device)
        self.weights_c = weights.c(cfg)
        self._run()
        torch.cuda.synchronize()
        if trace_events is not None:
            for e in trace_events:  # create the lazily made torch events outside the capture
                e.record()
            torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            # with trace_events the graph also carries one event-record node
            # before each launch and one after the last
            self._run(trace_events)
        torch.cuda.synchronize()

    def _run(self, trace_events=None):
        moe_forward(self.cfg, None, self.x, out=self.out, outputs=self.outputs, ws=self.ws,
                    weights_c=self.weights_c, trace_events=trace_events)

    def replay(self):
        self.graph.replay()

    def run_eager(self, trace_events=None):
        """The same forward launched directly (optionally with per-launch events)."""
        self._run(trace_events)


def moe_debug_suppress_gemm_producer(launches: int) -> None:
    """Failure injection for tests: the next `launches` expert-GEMM launches
    run with their TMA producer silent, so their bounded waits run out and
    the call records MOE_ERR_TIMEOUT in the workspace status word."""
    check(_L.moe_debug_suppress_gemm_producer(int(launches)), "moe_debug_suppress_gemm_producer")


def moe_workspace_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns the status word (0 = MOE_OK)."""
    return int(_L.moe_workspace_status(C.c_void_p(ws.data_ptr()), _stream(stream)))

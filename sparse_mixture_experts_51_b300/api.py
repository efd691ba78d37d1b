"""PyTorch-facing binding of the C ABI (include/moe_b300.h).

Argument marshalling only: every step of the layer runs in the CUDA library.
PyTorch provides device memory (output and workspace tensors) and the
current CUDA stream.  Names mirror the C entry points: ``route``,
``dispatch``, ``expert_ffn``, ``combine``, ``forward``.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _lib
from ._lib import (MOE_ACT_GELU, MOE_ACT_SWIGLU, MOE_BF16, MOE_F32, MOE_ROUTE_EXPERT_CHOICE, MOE_ROUTE_TOKEN_CHOICE,
                   MoeError, MoeShape, MoeShared)

ACTS = {"gelu": MOE_ACT_GELU, "swiglu": MOE_ACT_SWIGLU, MOE_ACT_GELU: MOE_ACT_GELU, MOE_ACT_SWIGLU: MOE_ACT_SWIGLU}


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return MOE_BF16
    if dt == torch.float32:
        return MOE_F32
    raise TypeError(f"unsupported dtype {dt} (bf16 or fp32)")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor arguments must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


ROUTINGS = {"token": MOE_ROUTE_TOKEN_CHOICE, "expert": MOE_ROUTE_EXPERT_CHOICE,
            MOE_ROUTE_TOKEN_CHOICE: MOE_ROUTE_TOKEN_CHOICE, MOE_ROUTE_EXPERT_CHOICE: MOE_ROUTE_EXPERT_CHOICE}


GATES = {"renorm": 0, "raw": 1, 0: 0, 1: 1}
OVERFLOWS = {"drop": 0, "reroute": 1, 0: 0, 1: 1}


def shape_of(T: int, d: int, E: int, k: int, d_ff: int, dtype: torch.dtype, act, d_ff_shared: int = 0,
             routing="token", gates="renorm", overflow="drop") -> MoeShape:
    return MoeShape(T=int(T), d=int(d), E=int(E), k=int(k), d_ff=int(d_ff), dtype=_dtype_code(dtype),
                    act=ACTS[act], d_ff_shared=int(d_ff_shared), routing=ROUTINGS[routing], gates=GATES[gates],
                    overflow=OVERFLOWS[overflow])


def shared_weights(W1s, W2s, W3s=None, b1s=None, b2s=None) -> MoeShared:
    """moe_shared_t over device tensors (keep the tensors alive while it is used).
    W1s, W3s [d_ff_shared, d]; W2s [d, d_ff_shared]; b1s [d_ff_shared]; b2s [d]."""
    for t in (W1s, W2s, W3s, b1s, b2s):
        if t is not None and not t.is_contiguous():
            raise ValueError("shared-expert weights must be contiguous")
    return MoeShared(W1s=_ptr(W1s), W3s=_ptr(W3s), W2s=_ptr(W2s), b1s=_ptr(b1s), b2s=_ptr(b2s))


def capacity(T: int, k: int, E: int, capacity_factor: float) -> int:
    c = _lib.load().moe_capacity(int(T), int(k), int(E), float(capacity_factor))
    if c < 0:
        raise ValueError("invalid capacity arguments")
    return c


def max_rows(shape: MoeShape, C: int) -> int:
    return int(_lib.load().moe_max_rows(ctypes.byref(shape), int(C)))


def workspace_size(shape: MoeShape, C: int) -> int:
    n = ctypes.c_size_t(0)
    _lib.check(_lib.load().moe_workspace_size(ctypes.byref(shape), int(C), ctypes.byref(n)), "moe_workspace_size")
    return int(n.value)


def new_workspace(shape: MoeShape, C: int, device=None) -> torch.Tensor:
    """Zero-filled workspace (the library expects zeros at first use)."""
    n = workspace_size(shape, C)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def get_device_error(ws: torch.Tensor, stream=None) -> int:
    """Synchronise, read and clear the workspace error word; returns the status code."""
    return int(_lib.load().moe_get_device_error(_ptr(ws), _stream(stream)))


def route(x: torch.Tensor, W_g: torch.Tensor, k: int, b_g=None, W_noise=None, eps=None,
          want_logits: bool = False, stats: Optional[torch.Tensor] = None, stream=None, gates="renorm"):
    """Router logits + exact top-k + gates (renormalised, or "raw" routing
    probabilities).  Returns (idx int32 [T,k], w fp32 [T,k], logits or None)."""
    T, d = x.shape
    E = W_g.shape[1]
    shape = shape_of(T, d, E, k, 64, x.dtype, MOE_ACT_GELU, gates=gates)
    idx = torch.empty(T, k, dtype=torch.int32, device=x.device)
    w = torch.empty(T, k, dtype=torch.float32, device=x.device)
    logits = torch.empty(T, E, dtype=torch.float32, device=x.device) if want_logits else None
    st = _lib.load().moe_route(ctypes.byref(shape), _ptr(x), _ptr(W_g), _ptr(b_g), _ptr(W_noise), _ptr(eps),
                               _ptr(idx), _ptr(w), _ptr(logits), _ptr(stats), _stream(stream))
    _lib.check(st, "moe_route")
    return idx, w, logits


def route_expert_choice(x: torch.Tensor, W_g: torch.Tensor, k: int, C: int, b_g=None, W_noise=None, eps=None,
                        want_logits: bool = False, ws: Optional[torch.Tensor] = None, stream=None) -> dict:
    """Expert-choice routing: expert e takes its min(C, T) highest-scoring tokens.
    Returns sel int32 [E, C'] (ascending token ids), gates fp32 [E, C'],
    dropped int64 [1] (tokens no expert chose) and logits (or None)."""
    T, d = x.shape
    E = W_g.shape[1]
    shape = shape_of(T, d, E, k, 64, x.dtype, MOE_ACT_GELU, routing="expert")
    dev = x.device
    if ws is None:
        ws = new_workspace(shape, C, dev)
    Cp = min(int(C), T)
    out = dict(sel=torch.empty(E, Cp, dtype=torch.int32, device=dev),
               gates=torch.empty(E, Cp, dtype=torch.float32, device=dev),
               dropped=torch.empty(1, dtype=torch.int64, device=dev),
               logits=torch.empty(T, E, dtype=torch.float32, device=dev) if want_logits else None)
    st = _lib.load().moe_route_expert_choice(ctypes.byref(shape), int(C), _ptr(x), _ptr(W_g), _ptr(b_g),
                                             _ptr(W_noise), _ptr(eps), _ptr(out["sel"]), _ptr(out["gates"]),
                                             _ptr(out["logits"]), _ptr(out["dropped"]), _ptr(ws), ws.numel(),
                                             _stream(stream))
    _lib.check(st, "moe_route_expert_choice")
    out["ws"] = ws
    return out


def dispatch(idx: torch.Tensor, x: torch.Tensor, E: int, C: int, d_ff: int = 64, act=MOE_ACT_GELU,
             ws: Optional[torch.Tensor] = None, want_row_token: bool = False, stream=None) -> dict:
    """Capacity-limited dispatch + gather.  Returns pos, counts, offsets, dropped, x_perm (and row_token)."""
    T, d = x.shape
    k = idx.shape[1]
    shape = shape_of(T, d, E, k, d_ff, x.dtype, act)
    R = max_rows(shape, C)
    dev = x.device
    if ws is None:
        ws = new_workspace(shape, C, dev)
    out = dict(pos=torch.empty(T, k, dtype=torch.int32, device=dev),
               counts=torch.empty(E, dtype=torch.int32, device=dev),
               offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
               dropped=torch.empty(1, dtype=torch.int64, device=dev),
               x_perm=torch.empty(max(R, 1), d, dtype=x.dtype, device=dev),
               row_token=torch.full((max(R, 1),), -1, dtype=torch.int32, device=dev) if want_row_token else None)
    st = _lib.load().moe_dispatch(ctypes.byref(shape), int(C), _ptr(idx), _ptr(x), _ptr(out["pos"]),
                                  _ptr(out["counts"]), _ptr(out["offsets"]), _ptr(out["dropped"]),
                                  _ptr(out["x_perm"]), _ptr(out["row_token"]), _ptr(ws), ws.numel(),
                                  _stream(stream))
    _lib.check(st, "moe_dispatch")
    out["ws"] = ws
    return out


STATS_SUMMARY = ("aux_loss", "entropy", "load_cv", "kept_cv", "utilisation", "overflow")


def routing_stats(logits: torch.Tensor, idx: torch.Tensor, counts: torch.Tensor, dropped: torch.Tensor,
                  ws: Optional[torch.Tensor] = None, stream=None) -> dict:
    """Routing diagnostics and the auxiliary load-balancing loss of one batch.

    Returns device tensors: f [E] fp64 (routed load over T*k, before the
    capacity cut), P [E] fp64 (mean full-softmax probability) and summary [6]
    fp64 in the order of STATS_SUMMARY.  ``ws`` is any workspace of the same
    T, k and E (a fresh one is made if None)."""
    T, E = logits.shape
    k = idx.shape[1]
    shape = shape_of(T, 64, E, k, 64, torch.float32, MOE_ACT_GELU)
    dev = logits.device
    if ws is None:
        ws = new_workspace(shape, 0, dev)
    out = dict(f=torch.empty(E, dtype=torch.float64, device=dev), P=torch.empty(E, dtype=torch.float64, device=dev),
               summary=torch.empty(len(STATS_SUMMARY), dtype=torch.float64, device=dev))
    st = _lib.load().moe_routing_stats(ctypes.byref(shape), _ptr(logits), _ptr(idx), _ptr(counts), _ptr(dropped),
                                       _ptr(out["f"]), _ptr(out["P"]), _ptr(out["summary"]), _ptr(ws), ws.numel(),
                                       _stream(stream))
    _lib.check(st, "moe_routing_stats")
    return out


def stats_summary(stats: dict) -> dict:
    """The summary tensor of routing_stats as named Python floats (synchronises)."""
    return dict(zip(STATS_SUMMARY, stats["summary"].tolist()))


def expert_ffn(x_perm: torch.Tensor, offsets: torch.Tensor, W1: torch.Tensor, W2: torch.Tensor, T: int, k: int,
               C: int, act, W3=None, b1=None, b2=None, ws: Optional[torch.Tensor] = None, stream=None):
    """Every expert's FFN over its rows of x_perm.  Returns y_perm fp32 [max_rows, d]."""
    E, F, d = W1.shape
    shape = shape_of(T, d, E, k, F, W1.dtype, act)
    R = max_rows(shape, C)
    if ws is None:
        ws = new_workspace(shape, C, x_perm.device)
    y = torch.zeros(max(R, 1), d, dtype=torch.float32, device=x_perm.device)
    st = _lib.load().moe_expert_ffn(ctypes.byref(shape), int(C), _ptr(x_perm), _ptr(offsets), _ptr(W1), _ptr(W3),
                                    _ptr(W2), _ptr(b1), _ptr(b2), _ptr(y), _ptr(ws), ws.numel(), _stream(stream))
    _lib.check(st, "moe_expert_ffn")
    return y


def shared_ffn(x: torch.Tensor, W1s: torch.Tensor, W2s: torch.Tensor, act, W3s=None, b1s=None, b2s=None,
               ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The shared experts (one dense FFN of width d_ff_shared) on every token.
    Returns y_shared fp32 [T, d]."""
    T, d = x.shape
    Fs = W1s.shape[0]
    shape = shape_of(T, d, 1, 1, 64, x.dtype, act, d_ff_shared=Fs)
    if ws is None:
        ws = new_workspace(shape, 0, x.device)
    y = torch.empty(T, d, dtype=torch.float32, device=x.device)
    sh = shared_weights(W1s, W2s, W3s, b1s, b2s)
    st = _lib.load().moe_shared_ffn(ctypes.byref(shape), _ptr(x), ctypes.addressof(sh), _ptr(y), _ptr(ws),
                                    ws.numel(), _stream(stream))
    _lib.check(st, "moe_shared_ffn")
    return y


def combine(y_perm, idx, w, pos, offsets, residual, E: int, C: int, out_dtype, d_ff: int = 64,
            want_moe: bool = False, y_shared: Optional[torch.Tensor] = None, stream=None):
    """out = residual + sum of kept w * y rows (+ y_shared).  Returns (out, moe_out or None)."""
    T, k = idx.shape
    d = y_perm.shape[1]
    shape = shape_of(T, d, E, k, d_ff, out_dtype, MOE_ACT_GELU)
    out = torch.empty(T, d, dtype=out_dtype, device=idx.device)
    moe = torch.empty(T, d, dtype=torch.float32, device=idx.device) if want_moe else None
    st = _lib.load().moe_combine(ctypes.byref(shape), int(C), _ptr(y_perm), _ptr(idx), _ptr(w), _ptr(pos),
                                 _ptr(offsets), _ptr(residual), _ptr(y_shared), _ptr(out), _ptr(moe),
                                 _stream(stream))
    _lib.check(st, "moe_combine")
    return out, moe


class MoELayer:
    """One sparse MoE layer with resident weights and a reusable workspace.

    ``layer(x, eps=None)`` runs the whole forward pass (moe_forward) on the
    current stream and returns the output tensor; ``layer.last`` keeps the
    routing outputs of the call (idx, w, pos, counts, offsets, dropped, and
    the router logits) when ``keep_routing`` is set, and
    ``layer.routing_stats()`` turns them into the routing diagnostics and the
    auxiliary load-balancing loss.  ``W1s``/``W2s`` (and ``W3s``, ``b1s``,
    ``b2s``) add shared experts: one dense FFN of width ``W1s.shape[0]`` that
    every token passes through, added in the combine.
    """

    def __init__(self, W_g, W1, W2, k: int, act, W3=None, b_g=None, W_noise=None, b1=None, b2=None,
                 capacity_factor: Optional[float] = None, C: Optional[int] = None, keep_routing: bool = True,
                 want_moe: bool = False, W1s=None, W2s=None, W3s=None, b1s=None, b2s=None, routing="token",
                 gates="renorm", overflow="drop"):
        if (capacity_factor is None) == (C is None):
            raise ValueError("give exactly one of capacity_factor and C")
        if (W1s is None) != (W2s is None):
            raise ValueError("shared experts need both W1s and W2s")
        self.W_g, self.W1, self.W2, self.W3 = W_g, W1, W2, W3
        self.b_g, self.W_noise, self.b1, self.b2 = b_g, W_noise, b1, b2
        self.k, self.act = int(k), ACTS[act]
        self.E, self.F, self.d = W1.shape
        self.dtype = W1.dtype
        self.Fs = 0 if W1s is None else int(W1s.shape[0])
        self.routing = ROUTINGS[routing]
        self.gates, self.overflow = GATES[gates], OVERFLOWS[overflow]
        self._shared_t = (W1s, W2s, W3s, b1s, b2s)
        self._shared = shared_weights(W1s, W2s, W3s, b1s, b2s) if W1s is not None else None
        self.capacity_factor, self.C_fixed = capacity_factor, C
        self.keep_routing, self.want_moe = keep_routing, want_moe
        self._ws = {}
        self.last = None

    def capture(self, x: torch.Tensor, eps: Optional[torch.Tensor] = None,
                out: Optional[torch.Tensor] = None) -> "CapturedForward":
        """Capture this layer's forward over the device buffers x (and eps)
        into a CUDA graph.  The routing outputs of replays are not kept."""
        if out is None:
            out = torch.empty(x.shape[0], self.d, dtype=x.dtype, device=x.device)
        keep = self.keep_routing
        self.keep_routing = False
        try:
            return _capture(self, x, eps, out)
        finally:
            self.keep_routing = keep

    def capacity(self, T: int) -> int:
        return self.C_fixed if self.C_fixed is not None else capacity(T, self.k, self.E, self.capacity_factor)

    def workspace(self, T: int) -> torch.Tensor:
        C = self.capacity(T)
        key = (T, C)
        if key not in self._ws:
            shape = shape_of(T, self.d, self.E, self.k, self.F, self.dtype, self.act, self.Fs, self.routing,
                             self.gates, self.overflow)
            self._ws[key] = new_workspace(shape, C, self.W1.device)
        return self._ws[key]

    def __call__(self, x: torch.Tensor, eps: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                 stats: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        T = x.shape[0]
        C = self.capacity(T)
        shape = shape_of(T, self.d, self.E, self.k, self.F, x.dtype, self.act, self.Fs, self.routing, self.gates,
                         self.overflow)
        ws = self.workspace(T)
        dev = x.device
        if out is None:
            out = torch.empty(T, self.d, dtype=x.dtype, device=dev)
        moe = torch.empty(T, self.d, dtype=torch.float32, device=dev) if self.want_moe else None
        r = None
        if self.keep_routing:
            r = dict(idx=torch.empty(T, self.k, dtype=torch.int32, device=dev),
                     w=torch.empty(T, self.k, dtype=torch.float32, device=dev),
                     pos=torch.empty(T, self.k, dtype=torch.int32, device=dev),
                     counts=torch.empty(self.E, dtype=torch.int32, device=dev),
                     offsets=torch.empty(self.E + 1, dtype=torch.int32, device=dev),
                     dropped=torch.empty(1, dtype=torch.int64, device=dev),
                     logits=torch.empty(T, self.E, dtype=torch.float32, device=dev))
        if r is not None and self.routing == MOE_ROUTE_EXPERT_CHOICE:
            # the token-choice tables do not exist with expert choice
            r["idx"] = r["w"] = r["pos"] = None
        g = (lambda n: _ptr(r[n])) if r is not None else (lambda n: None)
        st = _lib.load().moe_forward(
            ctypes.byref(shape), float(self.capacity_factor or 0.0), int(C if self.C_fixed is not None else -1),
            _ptr(x), _ptr(self.W_g), _ptr(self.b_g), _ptr(self.W_noise), _ptr(eps), _ptr(self.W1), _ptr(self.W3),
            _ptr(self.W2), _ptr(self.b1), _ptr(self.b2),
            ctypes.addressof(self._shared) if self._shared is not None else None, _ptr(out), _ptr(moe),
            g("idx"), g("w"), g("pos"),
            g("counts"), g("offsets"), g("dropped"), _ptr(stats), g("logits"), _ptr(ws), ws.numel(),
            _stream(stream))
        _lib.check(st, "moe_forward")
        if r is not None:
            r["C"] = C
            r["moe"] = moe
            r["ws"] = ws
        self.last = r
        return out

    def routing_stats(self, stream=None) -> dict:
        """Routing diagnostics of the last call (see routing_stats); needs keep_routing
        and token-choice routing."""
        r = self.last
        if r is None:
            raise RuntimeError("no routing outputs kept: call the layer with keep_routing=True first")
        if self.routing != MOE_ROUTE_TOKEN_CHOICE:
            raise ValueError("routing_stats needs a top-k table: token-choice routing only")
        return routing_stats(r["logits"], r["idx"], r["counts"], r["dropped"], ws=r["ws"], stream=stream)


class CapturedForward:
    """A CUDA graph of one MoELayer forward over fixed device buffers.

    ``replay()`` re-runs the captured forward on whatever the static input
    buffers (``x``, ``eps``) hold at that moment and writes ``out``; all
    launches of the layer go to the GPU as one graph launch.  Build it with
    ``MoELayer.capture``."""

    def __init__(self, graph, x, eps, out):
        self.graph, self.x, self.eps, self.out = graph, x, eps, out

    def replay(self):
        self.graph.replay()
        return self.out


def _capture(layer, x, eps, out):
    # one eager call first: per-device set-up (attribute queries, launch
    # limits) happens outside the capture
    layer(x, eps=eps, out=out)
    torch.cuda.synchronize(x.device)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer(x, eps=eps, out=out)
    return CapturedForward(graph, x, eps, out)


def forward(x, W_g, k: int, act, W1, W2, W3=None, b_g=None, W_noise=None, eps=None, b1=None, b2=None,
            capacity_factor: Optional[float] = None, C: Optional[int] = None, want_moe: bool = False,
            stats: Optional[torch.Tensor] = None, stream=None, W1s=None, W2s=None, W3s=None, b1s=None, b2s=None,
            routing="token", gates="renorm", overflow="drop"):
    """One-shot whole-layer forward.  Returns (out, routing dict incl. 'moe' when want_moe)."""
    if C is None and capacity_factor is None:
        raise ValueError("give capacity_factor or C")
    if C is not None:
        capacity_factor = None
    layer = MoELayer(W_g, W1, W2, k, act, W3=W3, b_g=b_g, W_noise=W_noise, b1=b1, b2=b2,
                     capacity_factor=capacity_factor, C=C, keep_routing=True, want_moe=want_moe,
                     W1s=W1s, W2s=W2s, W3s=W3s, b1s=b1s, b2s=b2s, routing=routing, gates=gates, overflow=overflow)
    out = layer(x, eps=eps, stats=stats, stream=stream)
    return out, layer.last


__all__ = ["capacity", "max_rows", "workspace_size", "new_workspace", "get_device_error", "route", "dispatch",
           "route_expert_choice", "expert_ffn", "shared_ffn", "shared_weights", "combine", "forward", "routing_stats", "stats_summary", "STATS_SUMMARY", "MoELayer",
           "CapturedForward", "MoeError", "shape_of"]

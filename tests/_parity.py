"""Helpers for the GPU parity tests: run the CUDA library and the fp64 oracle
on the same seeded inputs and compare.  The oracle sees the stored input
values widened to fp64; nothing it consumes comes from the CUDA path except,
where a test says so, the GPU's own top-k table fed to later oracle steps."""
from __future__ import annotations

import numpy as np
import torch

from oracle import moe_oracle as O
from sparse_mixture_experts_51_b300 import api
from sparse_mixture_experts_51_b300 import workloads as W


class F64Experts:
    """Lazy fp64 view of a [E, ...] weight tensor: W[e] -> float64 numpy."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, e):
        return W.as_f64_numpy(self.t[e])


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def to_gpu(inp: dict, dev="cuda") -> dict:
    return {k: (None if v is None else v.to(dev).contiguous()) for k, v in inp.items()}


def shared_args(g: dict) -> dict:
    """The library's form of the shared experts in ``g`` (one FFN of width
    S*F_s; b2 of the wide FFN = the sum of the experts' b2), or no shared
    experts."""
    sw = W.shared_wide(g)
    if sw["W1s"] is None:
        return {}
    b2 = None if sw["b2s_rows"] is None else sw["b2s_rows"].sum(dim=0).contiguous()
    return dict(W1s=sw["W1s"], W2s=sw["W2s"], W3s=sw["W3s"], b1s=sw["b1s"], b2s=b2)


def gpu_forward(w: W.Workload, g: dict, C=None, want_moe=True, gates="renorm", overflow="drop"):
    stats = torch.zeros(2, dtype=torch.int64, device="cuda")
    act = "swiglu" if w.act == W.ACT_SWIGLU else "gelu"
    out, r = api.forward(g["x"], g["W_g"], w.k, act, g["W1"], g["W2"], W3=g["W3"], b_g=g["b_g"],
                         W_noise=g["W_noise"], eps=g["eps"], b1=g["b1"], b2=g["b2"],
                         capacity_factor=None if C is not None else w.capacity_factor, C=C,
                         want_moe=want_moe, stats=stats, gates=gates, overflow=overflow, **shared_args(g))
    torch.cuda.synchronize()
    res = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in r.items()}
    res["out"] = out.cpu()
    res["stats"] = stats.cpu()
    return res


def oracle_shared(inp: dict):
    """The shared experts of ``inp`` per expert, widened to fp64, or None."""
    if inp.get("W1s") is None:
        return None
    f = W.as_f64_numpy
    return dict(W1s=f(inp["W1s"]), W2s=f(inp["W2s"]), W3s=f(inp["W3s"]), b1s=f(inp.get("b1s")),
                b2s=f(inp.get("b2s")))


def oracle_forward(w: W.Workload, inp: dict, C=None, tokens=None, idx_override=None, gates="renorm",
                   overflow="drop"):
    f = W.as_f64_numpy
    return O.forward(f(inp["x"]), f(inp["W_g"]), w.k, w.act, F64Experts(inp["W1"]), F64Experts(inp["W2"]),
                     W3=None if inp["W3"] is None else F64Experts(inp["W3"]),
                     b1=None if inp["b1"] is None else F64Experts(inp["b1"]),
                     b2=None if inp["b2"] is None else F64Experts(inp["b2"]),
                     b_g=f(inp["b_g"]), W_noise=f(inp["W_noise"]), eps=f(inp["eps"]),
                     capacity_factor=w.capacity_factor if C is None else None, C=C, tokens=tokens,
                     idx_override=idx_override, shared=oracle_shared(inp), gate_mode=gates, overflow=overflow)


def tolerance(w: W.Workload) -> float:
    """Relative L2 bound on the layer output: 1e-5 for fp32 layers, 1e-2 for bf16 layers
    (bf16 operands and hidden activation, fp32 accumulation)."""
    return 1e-5 if w.dtype == torch.float32 else 1e-2


def check_layer(w: W.Workload, inp: dict, gpu: dict, ref: dict, tokens=None):
    """Routing, slots and drops bit-exact; gates and outputs within tolerance."""
    T = w.T
    np.testing.assert_array_equal(gpu["idx"].numpy(), ref["idx"], err_msg="top-k indices")
    np.testing.assert_array_equal(gpu["pos"].numpy(), ref["pos"], err_msg="slots")
    np.testing.assert_array_equal(gpu["counts"].numpy(), ref["counts"], err_msg="counts")
    np.testing.assert_array_equal(gpu["offsets"].numpy(), ref["offsets"], err_msg="offsets")
    assert int(gpu["dropped"][0]) == ref["dropped"], "drop count"
    gate_tol = 1e-6 if w.dtype == torch.float32 else 1e-4
    np.testing.assert_allclose(gpu["w"].numpy(), ref["w"], rtol=0, atol=gate_tol, err_msg="gates")
    toks = np.arange(T) if tokens is None else np.asarray(tokens)
    tol = tolerance(w)
    if T == 0:
        return
    if gpu.get("moe") is not None:
        e_moe = rel_l2(gpu["moe"].numpy()[toks], ref["moe"])
        assert e_moe <= tol, f"moe rel-L2 {e_moe:.3e} > {tol}"
    e_out = rel_l2(gpu["out"].float().numpy()[toks], ref["out"])
    assert e_out <= tol, f"out rel-L2 {e_out:.3e} > {tol}"

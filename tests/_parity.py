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


def row_rel_l2(a, b) -> np.ndarray:
    """Relative L2 error of every row of ``a`` against ``b`` (one token's
    output vector per row); rows whose reference is zero give 0 if ``a``'s
    row is exactly zero and inf otherwise."""
    a = np.asarray(a, dtype=np.float64).reshape(len(b), -1)
    b = np.asarray(b, dtype=np.float64).reshape(len(b), -1)
    num = np.linalg.norm(a - b, axis=1)
    den = np.linalg.norm(b, axis=1)
    out = np.zeros(len(b))
    nz = den > 0
    out[nz] = num[nz] / den[nz]
    out[~nz] = np.where(num[~nz] == 0, 0.0, np.inf)
    return out


def check_rows(what: str, a, b, tol: float, labels=None) -> float:
    """Every row of ``a`` within relative L2 ``tol`` of the same row of ``b``
    (and exactly zero where ``b``'s row is zero); returns the largest row error."""
    if len(b) == 0:
        return 0.0
    e = row_rel_l2(a, b)
    i = int(np.argmax(e))
    lab = i if labels is None else labels[i]
    assert e[i] <= tol, f"{what}: row {lab} rel-L2 {e[i]:.3e} > {tol} (median {np.median(e):.2e})"
    return float(e[i])


def segment_edge_rows(offsets, head: int = 4, tail: int = 32) -> np.ndarray:
    """Grouped rows where the expert GEMMs take their edge paths: the first
    ``head`` and the last ``tail`` rows of every expert's segment (the
    epilogue warp that holds a segment's end stores its rows directly), and
    the first row of every 32-row epilogue group of each segment's last
    128-row tile and of its last 256-row tile (a 256-row tile with at most
    128 valid rows issues only its first M half)."""
    offsets = np.asarray(offsets, dtype=np.int64)
    rows = set()
    for e in range(len(offsets) - 1):
        a, b = int(offsets[e]), int(offsets[e + 1])
        n = b - a
        if n <= 0:
            continue
        rows.update(range(a, min(b, a + head)))
        rows.update(range(max(a, b - tail), b))
        for tile in (128, 256):
            rows.update(range(a + (n - 1) // tile * tile, b, 32))
    return np.array(sorted(rows), dtype=np.int64)


def edge_tokens(idx, pos, offsets, **kw) -> list:
    """Tokens whose kept assignments land on ``segment_edge_rows`` of the
    token-choice grouped layout (row = offsets[idx[t,r]] + pos[t,r])."""
    idx = np.asarray(idx, dtype=np.int64)
    pos = np.asarray(pos, dtype=np.int64)
    offsets = np.asarray(offsets, dtype=np.int64)
    kept = pos >= 0
    rows = np.where(kept, offsets[np.clip(idx, 0, len(offsets) - 2)] + pos, -1)
    want = np.zeros(int(offsets[-1]) + 1, dtype=bool)
    want[segment_edge_rows(offsets, **kw)] = True
    hit = kept & want[np.where(kept, rows, len(want) - 1)]
    return sorted(set(np.nonzero(hit.any(axis=1))[0].tolist()))


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


def row_tolerance(w: W.Workload) -> float:
    """Relative L2 bound on each token's output row: the layer tolerance
    applied token by token.  For bf16 layers the row error is set by the bf16
    rounding of the hidden activation (relative spacing 2^-8, errors spread
    uniformly, so about 2^-8/sqrt(3) = 2.3e-3 per row after the fp32 down
    projection mixes them), plus the bf16 output rounding of ``out`` (at most
    2^-8 of the row, element by element); fp32 layers see only fp32
    accumulation (~1e-7)."""
    return tolerance(w)


def check_layer(w: W.Workload, inp: dict, gpu: dict, ref: dict, tokens=None):
    """Routing, slots and drops bit-exact; gates within tolerance; outputs
    within tolerance as a whole and token by token (every row of the weighted
    expert sum and of the layer output)."""
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
    rtol = row_tolerance(w)
    if gpu.get("moe") is not None:
        e_moe = rel_l2(gpu["moe"].numpy()[toks], ref["moe"])
        assert e_moe <= tol, f"moe rel-L2 {e_moe:.3e} > {tol}"
        check_rows("moe", gpu["moe"].numpy()[toks], ref["moe"], rtol, labels=toks)
    e_out = rel_l2(gpu["out"].float().numpy()[toks], ref["out"])
    assert e_out <= tol, f"out rel-L2 {e_out:.3e} > {tol}"
    check_rows("out", gpu["out"].float().numpy()[toks], ref["out"], rtol, labels=toks)

"""Seeded synthetic workloads for the sparse MoE layer forward.

This module only draws random numbers and builds tensors of the right
shapes and dtypes.  It holds none of the layer's arithmetic (no routing,
no dispatch, no expert math), so both the CUDA path and the CPU oracle can
take their inputs from it without sharing any of the method.

Shapes follow the five layer configurations this library is measured on:

  tiny_fp32       T=64    d=32   E=4  k=2 GELU   F=64    cf=1.25  fp32
  bf16_t4096      T=4096  d=1024 E=8  k=2 SwiGLU F=4096  cf=1.25  bf16
  mixtral_t16384  T=16384 d=4096 E=8  k=2 SwiGLU F=14336 no-drop  bf16
  switch_top1     T=32768 d=768  E=64 k=1 GELU   F=3072  cf=1.0   bf16,
                  Zipf router bias and noisy gating
  decode_t128     T=128   d=2048 E=64 k=6 SwiGLU F=1408  cf=2.0   bf16
and two layers for the next-step extensions:
  shared_t4096    T=4096  d=2048 E=64 k=6 SwiGLU F=1408  cf=1.25  bf16,
                  plus 2 shared experts of width 1408
  ec_t4096        bf16_t4096's layer and tokens with expert-choice routing

Value recipe (all draws fp32 standard normal from one CPU torch.Generator
seeded per workload, scaled, then cast to the storage dtype):
  x ~ N(0,1); W_g ~ N(0, 1/d); W1, W3 ~ N(0, 1/d); W2 ~ N(0, 1/F)
  (tiny_fp32 takes "N(0, 1/d)" literally for every weight, W2 included);
  biases zero (tiny_fp32 carries explicit zero b1/b2; the others have none);
  switch_top1: b_g[e] = 2*ln(1/(e+1)), W_noise ~ N(0, 1/d), eps ~ N(0,1)[T,E];
  shared experts: W1s, W3s ~ N(0, 1/d) [S,F_s,d]; W2s ~ N(0, 1/F_s) [S,d,F_s].
The draw order is fixed: x, W_g, W_noise, eps, W1, W3, W2, W1s, W3s, W2s.

Layouts (row-major, nn.Linear style, K contiguous):
  x [T,d]; W_g [d,E] fp32; b_g [E] fp32; W_noise [d,E] fp32; eps [T,E] fp32;
  W1, W3 [E,F,d]; W2 [E,d,F]; b1 [E,F] fp32; b2 [E,d] fp32.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

ACT_GELU = 0
ACT_SWIGLU = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    k: int
    F: int
    act: int                 # ACT_GELU or ACT_SWIGLU
    capacity_factor: float
    dtype: torch.dtype       # storage/compute dtype of x, expert weights, out
    seed: int
    noisy: bool = False      # noisy gating with supplied eps and W_noise
    zipf_bias: bool = False  # router bias b_e = 2 ln(1/(e+1))
    expert_bias: bool = False  # explicit (zero) b1/b2 tensors
    weight_std_literal_d: bool = False  # every weight ~N(0,1/d)
    n_shared: int = 0        # shared experts (every token, weight 1)
    F_shared: int = 0        # hidden width of each shared expert
    routing: str = "token"   # "token" (top-k per token) or "expert" (top-C tokens per expert)

    @property
    def dtype_name(self) -> str:
        return {torch.float32: "f32", torch.bfloat16: "bf16"}[self.dtype]

    def scaled(self, T: int, seed: Optional[int] = None) -> "Workload":
        """Same layer with a different token count (used for small parity cases)."""
        return dataclasses.replace(self, T=T, seed=self.seed if seed is None else seed,
                                   name=f"{self.name}@T{T}")

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", T=64, d=32, E=4, k=2, F=64, act=ACT_GELU,
                          capacity_factor=1.25, dtype=torch.float32, seed=0,
                          expert_bias=True, weight_std_literal_d=True),
    "bf16_t4096": Workload("bf16_t4096", T=4096, d=1024, E=8, k=2, F=4096, act=ACT_SWIGLU,
                           capacity_factor=1.25, dtype=torch.bfloat16, seed=1),
    # no-drop: capacity factor E/k makes C = T
    "mixtral_t16384": Workload("mixtral_t16384", T=16384, d=4096, E=8, k=2, F=14336,
                               act=ACT_SWIGLU, capacity_factor=4.0, dtype=torch.bfloat16,
                               seed=3),
    "switch_top1": Workload("switch_top1", T=32768, d=768, E=64, k=1, F=3072, act=ACT_GELU,
                            capacity_factor=1.0, dtype=torch.bfloat16, seed=4,
                            noisy=True, zipf_bias=True),
    "decode_t128": Workload("decode_t128", T=128, d=2048, E=64, k=6, F=1408, act=ACT_SWIGLU,
                            capacity_factor=2.0, dtype=torch.bfloat16, seed=5),
    # fine-grained routed experts plus two always-on shared experts of the
    # same width (the DeepSeek-MoE layout, at a prefill-sized batch)
    "shared_t4096": Workload("shared_t4096", T=4096, d=2048, E=64, k=6, F=1408, act=ACT_SWIGLU,
                             capacity_factor=1.25, dtype=torch.bfloat16, seed=6, n_shared=2, F_shared=1408),
    # the bench layer and tokens with expert-choice routing at the same capacity (1280 tokens per expert)
    "ec_t4096": Workload("ec_t4096", T=4096, d=1024, E=8, k=2, F=4096, act=ACT_SWIGLU,
                         capacity_factor=1.25, dtype=torch.bfloat16, seed=1, routing="expert"),
}
ORDER = ["tiny_fp32", "bf16_t4096", "mixtral_t16384", "switch_top1", "decode_t128"]


def _normal(g: torch.Generator, shape, std: float) -> torch.Tensor:
    t = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def make_inputs(w: Workload) -> dict:
    """Draw every input tensor of workload ``w`` on the CPU.

    Returns a dict of CPU tensors: x, W_g, b_g (or None), W_noise (or None),
    eps (or None), W1, W3 (or None), W2, b1 (or None), b2 (or None).
    Expert weights and x are in ``w.dtype``; router tensors are fp32.
    """
    g = torch.Generator().manual_seed(w.seed)
    T, d, E, F = w.T, w.d, w.E, w.F
    std_d = 1.0 / math.sqrt(d)
    std_f = std_d if w.weight_std_literal_d else 1.0 / math.sqrt(F)
    x = _normal(g, (T, d), 1.0)
    W_g = _normal(g, (d, E), std_d)
    b_g = None
    if w.zipf_bias:
        b_g = torch.tensor([2.0 * math.log(1.0 / (e + 1)) for e in range(E)], dtype=torch.float32)
    W_noise = eps = None
    if w.noisy:
        W_noise = _normal(g, (d, E), std_d)
        eps = _normal(g, (T, E), 1.0)
    W1 = _normal(g, (E, F, d), std_d)
    W3 = _normal(g, (E, F, d), std_d) if w.act == ACT_SWIGLU else None
    W2 = _normal(g, (E, d, F), std_f)
    b1 = b2 = None
    if w.expert_bias:
        b1 = torch.zeros(E, F, dtype=torch.float32)
        b2 = torch.zeros(E, d, dtype=torch.float32)
    cast = (lambda t: t) if w.dtype == torch.float32 else (lambda t: t.to(w.dtype))
    out = dict(x=cast(x), W_g=W_g, b_g=b_g, W_noise=W_noise, eps=eps,
               W1=cast(W1), W3=None if W3 is None else cast(W3), W2=cast(W2),
               b1=b1, b2=b2, W1s=None, W3s=None, W2s=None, b1s=None, b2s=None)
    if w.n_shared > 0:
        # drawn after every routed tensor, so the routed inputs do not depend on them
        S, Fs = w.n_shared, w.F_shared
        out["W1s"] = cast(_normal(g, (S, Fs, d), std_d))
        out["W3s"] = cast(_normal(g, (S, Fs, d), std_d)) if w.act == ACT_SWIGLU else None
        out["W2s"] = cast(_normal(g, (S, d, Fs), 1.0 / math.sqrt(Fs)))
        if w.expert_bias:
            out["b1s"] = torch.zeros(S, Fs, dtype=torch.float32) if w.act == ACT_GELU else None
            out["b2s"] = torch.zeros(S, d, dtype=torch.float32)
    return out


def shared_wide(inp: dict) -> dict:
    """The shared experts of ``inp`` (per expert: W1s, W3s [S,F_s,d], W2s
    [S,d,F_s], b1s [S,F_s], b2s [S,d]) laid out as the one FFN of width S*F_s
    that the library takes: W1s/W3s rows stacked, W2s columns stacked, b1s
    concatenated; b2s becomes the list of per-expert rows to be summed by the
    caller (returned stacked as [S,d]).  Pure layout: no arithmetic."""
    if inp.get("W1s") is None:
        return dict(W1s=None, W3s=None, W2s=None, b1s=None, b2s_rows=None)
    W1s, W3s, W2s = inp["W1s"], inp["W3s"], inp["W2s"]
    S, Fs, d = W1s.shape
    return dict(W1s=W1s.reshape(S * Fs, d).contiguous(),
                W3s=None if W3s is None else W3s.reshape(S * Fs, d).contiguous(),
                W2s=torch.cat(list(W2s), dim=1).contiguous(),
                b1s=None if inp.get("b1s") is None else inp["b1s"].reshape(S * Fs).contiguous(),
                b2s_rows=inp.get("b2s"))


def make_tokens(w: Workload, seed: int) -> tuple:
    """A fresh token batch (and noise, when the workload is noisy) for the same layer.

    Used by timing loops that stream new inputs each step; weights are not redrawn.
    """
    g = torch.Generator().manual_seed(seed)
    x = _normal(g, (w.T, w.d), 1.0)
    eps = _normal(g, (w.T, w.E), 1.0) if w.noisy else None
    if w.dtype != torch.float32:
        x = x.to(w.dtype)
    return x, eps


def make_routing_tables(T: int, E: int, k: int, seed: int, logit_std: float = 2.0) -> dict:
    """Arbitrary routing tables of the shapes the routing-statistics call takes.

    logits [T,E] fp32 ~ N(0, logit_std^2); idx [T,k] int32 uniform in [0,E)
    (any ids, not necessarily the top-k of the logits); counts [E] int32
    uniform in [0, k*T/E + 1]; dropped [1] int64 uniform in [0, T*k]."""
    g = torch.Generator().manual_seed(seed)
    logits = _normal(g, (T, E), logit_std)
    idx = torch.randint(0, E, (T, k), generator=g, dtype=torch.int64).to(torch.int32)
    counts = torch.randint(0, k * T // E + 2, (E,), generator=g, dtype=torch.int64).to(torch.int32)
    dropped = torch.randint(0, T * k + 1, (1,), generator=g, dtype=torch.int64)
    return dict(logits=logits, idx=idx, counts=counts, dropped=dropped)


def as_f64_numpy(t: Optional[torch.Tensor]):
    """Widen a stored tensor (fp32 or bf16) to a float64 numpy array, exactly."""
    if t is None:
        return None
    return t.detach().to("cpu").to(torch.float64).numpy()

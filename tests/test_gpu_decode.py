"""The fused expert FFN of decode-sized batches (T <= 128 tokens, enough
assignments that every expert is expected to be active): moe_forward runs
both expert GEMMs as one kernel whose first phase covers every token of
every expert without waiting for the routing, and scatters the kept rows
in the second.  Each output row depends only on its own input row, so the
layer must equal, bit for bit, the step-by-step path (moe_route ->
moe_dispatch -> moe_expert_ffn -> moe_combine), whose grouped GEMMs run on
the kept rows only; and it must match the fp64 oracle like every layer."""
import numpy as np
import pytest
import torch

from sparse_mixture_experts_51_b300 import api
from sparse_mixture_experts_51_b300 import workloads as W

from _parity import check_layer, gpu_forward, oracle_forward, to_gpu

pytestmark = pytest.mark.gpu

CASES = [
    W.WORKLOADS["decode_t128"],
    # fewer tokens than the 128-row tile (the token matrix is read with zero-filled rows past T)
    W.Workload("dec_t77", T=77, d=512, E=64, k=6, F=1408, act=W.ACT_SWIGLU, capacity_factor=2.0,
               dtype=torch.bfloat16, seed=81),
    # tight capacity: many dropped assignments are computed in phase 1 but never stored
    W.Workload("dec_drops", T=128, d=256, E=16, k=4, F=384, act=W.ACT_SWIGLU, capacity_factor=0.6,
               dtype=torch.bfloat16, seed=82),
    # GELU experts (256-column phase-1 tiles), F not a multiple of 256
    W.Workload("dec_gelu", T=100, d=192, E=16, k=2, F=320, act=W.ACT_GELU, capacity_factor=1.5,
               dtype=torch.bfloat16, seed=83),
    # a Zipf-skewed noisy router: some experts may stay empty (their phase-2 tiles are skipped)
    W.Workload("dec_skewed", T=96, d=128, E=16, k=2, F=128, act=W.ACT_SWIGLU, capacity_factor=1.0,
               dtype=torch.bfloat16, seed=84, noisy=True, zipf_bias=True),
]


def _step_by_step(w, g, C, gates, overflow):
    act = "swiglu" if w.act == W.ACT_SWIGLU else "gelu"
    idx, wt, _ = api.route(g["x"], g["W_g"], w.k, b_g=g["b_g"], W_noise=g["W_noise"], eps=g["eps"], gates=gates)
    d = api.dispatch(idx, g["x"], w.E, C, d_ff=w.F, act=act)
    y = api.expert_ffn(d["x_perm"], d["offsets"], g["W1"], g["W2"], w.T, w.k, C, act, W3=g["W3"], b1=g["b1"],
                       b2=g["b2"])
    out, moe = api.combine(y, idx, wt, d["pos"], d["offsets"], g["x"], w.E, C, w.dtype, d_ff=w.F, want_moe=True)
    torch.cuda.synchronize()
    return out, moe, idx, d


def _with_biases(w, inp, seed):
    gen = torch.Generator().manual_seed(seed)
    if w.act == W.ACT_GELU:
        inp["b1"] = torch.randn(w.E, w.F, generator=gen) * 0.3
    inp["b2"] = torch.randn(w.E, w.d, generator=gen) * 0.3
    return inp


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_decode_layer_equals_step_by_step_and_oracle(w):
    inp = W.make_inputs(w)
    if w.name == "dec_gelu":
        inp = _with_biases(w, inp, 85)
    g = to_gpu(inp)
    C = api.capacity(w.T, w.k, w.E, w.capacity_factor)
    gpu = gpu_forward(w, g)
    out_s, moe_s, idx_s, d_s = _step_by_step(w, g, C, "renorm", "drop")
    assert torch.equal(gpu["idx"], idx_s.cpu())
    assert torch.equal(gpu["pos"], d_s["pos"].cpu())
    assert torch.equal(gpu["out"], out_s.cpu()), "fused decode FFN differs from the grouped GEMMs"
    assert torch.equal(gpu["moe"], moe_s.cpu())
    ref = oracle_forward(w, inp)
    check_layer(w, inp, gpu, ref)
    if w.name == "dec_drops":
        assert ref["dropped"] > 0


def test_decode_layer_repeated_calls_and_graph_replay():
    """The fused kernel's tile ticket and counts reset themselves: back-to-back
    calls, and replays of a captured graph, give the same output bit for bit."""
    w = CASES[2]
    inp = W.make_inputs(w)
    g = to_gpu(inp)
    layer = api.MoELayer(g["W_g"], g["W1"], g["W2"], w.k, "swiglu", W3=g["W3"], capacity_factor=w.capacity_factor,
                         keep_routing=False)
    first = layer(g["x"]).clone()
    for _ in range(5):
        assert torch.equal(layer(g["x"]), first)
    cap = layer.capture(g["x"])
    for _ in range(3):
        assert torch.equal(cap.replay(), first)
    x2 = torch.randn(g["x"].shape, generator=torch.Generator().manual_seed(86)).to(torch.bfloat16).cuda()
    g["x"].copy_(x2)
    out2 = cap.replay().clone()
    torch.cuda.synchronize()
    assert torch.equal(out2, layer(x2))
    assert api.get_device_error(layer.workspace(w.T)) == 0


def test_decode_layer_with_rerouting():
    """Overflow re-routing on a decode-sized batch: the fused FFN reads the
    final tables (after the second dispatch pass)."""
    w = CASES[2]
    inp = W.make_inputs(w)
    g = to_gpu(inp)
    gpu = gpu_forward(w, g, overflow="reroute")
    ref = oracle_forward(w, inp, overflow="reroute")
    assert ref["rerouted"] > 0
    check_layer(w, inp, gpu, ref)


def test_decode_kernel_count():
    """router, dispatch and one kernel for both expert GEMMs and the combine: three launches."""
    from sparse_mixture_experts_51_b300 import _lib

    lib = _lib.load()
    w = W.WORKLOADS["decode_t128"]
    g = to_gpu(W.make_inputs(w))
    layer = api.MoELayer(g["W_g"], g["W1"], g["W2"], w.k, "swiglu", W3=g["W3"], capacity_factor=w.capacity_factor,
                         keep_routing=False)
    layer(g["x"])
    torch.cuda.synchronize()
    n0 = lib.moe_kernel_launches()
    layer(g["x"])
    torch.cuda.synchronize()
    assert lib.moe_kernel_launches() - n0 == 3


def test_decode_layer_with_shared_experts():
    """A decode-sized layer with a shared expert: the fused kernel's combine
    adds the shared experts' output after the routed ranks, as the standalone
    combine does."""
    from _parity import shared_args

    w = W.Workload("dec_shared", T=64, d=256, E=16, k=2, F=256, act=W.ACT_SWIGLU, capacity_factor=1.5,
                   dtype=torch.bfloat16, seed=87, n_shared=1, F_shared=256)
    inp = W.make_inputs(w)
    g = to_gpu(inp)
    gpu = gpu_forward(w, g)
    ref = oracle_forward(w, inp)
    check_layer(w, inp, gpu, ref)
    C = api.capacity(w.T, w.k, w.E, w.capacity_factor)
    idx, wt, _ = api.route(g["x"], g["W_g"], w.k)
    d = api.dispatch(idx, g["x"], w.E, C, d_ff=w.F, act="swiglu")
    y = api.expert_ffn(d["x_perm"], d["offsets"], g["W1"], g["W2"], w.T, w.k, C, "swiglu", W3=g["W3"])
    ys = api.shared_ffn(g["x"], act="swiglu", **shared_args(g))
    out, moe = api.combine(y, idx, wt, d["pos"], d["offsets"], g["x"], w.E, C, w.dtype, d_ff=w.F, want_moe=True,
                           y_shared=ys)
    torch.cuda.synchronize()
    assert torch.equal(gpu["out"], out.cpu())
    assert torch.equal(gpu["moe"], moe.cpu())

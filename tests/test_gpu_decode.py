"""The fused layer of decode-sized batches (T <= 128 tokens, enough
assignments that every expert is expected to be active): moe_forward runs
both expert GEMMs and the combine as one kernel whose first phase covers
every token of every expert, and scatters the kept rows in the second.

Self-routed layers (overflow drop, E or 2E logit columns a power of two up
to 256) also route and dispatch inside that kernel (its first tiles): the
whole layer is one launch.  Its top-k is exact, so idx, the slots, counts
and offsets equal the standalone router's and dispatch's bit for bit; its
fp32 logits are summed in another order, so the gates agree to rounding.
Given its own routing tables, each output row depends only on its own input
row: the layer equals, bit for bit, the step-by-step path (moe_dispatch ->
moe_expert_ffn -> moe_combine) run on those tables.  Every layer must also
match the fp64 oracle."""
import numpy as np
import pytest
import torch

from sparse_mixture_experts_51_b300 import api
from sparse_mixture_experts_51_b300 import workloads as W

from _parity import check_layer, gpu_forward, oracle_forward, to_gpu

pytestmark = pytest.mark.gpu

CASES = [
    W.WORKLOADS["decode_t128"],
    # fewer tokens than the 128-row tile (the token matrix is read with zero-filled
    # rows past T) and than a whole number of 4-token rank tiles
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
    # the widest logit table the rank tiles take: 128 experts with the noise projection (256 columns)
    W.Workload("dec_e128_noisy", T=128, d=256, E=128, k=4, F=128, act=W.ACT_SWIGLU, capacity_factor=1.5,
               dtype=torch.bfloat16, seed=88, noisy=True),
    # the smallest self-routed layer: 4 experts, top-4 (every token takes every expert), two rank
    # tiles the second of which holds one token, logit columns split 256 ways along d
    W.Workload("dec_tiny", T=5, d=64, E=4, k=4, F=64, act=W.ACT_SWIGLU, capacity_factor=1.0,
               dtype=torch.bfloat16, seed=90),
    # E = 48: not a power of two, so the router and the dispatch run as their own kernels
    W.Workload("dec_e48", T=96, d=256, E=48, k=4, F=256, act=W.ACT_SWIGLU, capacity_factor=1.25,
               dtype=torch.bfloat16, seed=89),
]


def _self_routed(w) -> bool:
    nc = 2 * w.E if w.noisy else w.E
    return 4 <= nc <= 256 and nc & (nc - 1) == 0 and w.E % 4 == 0


def _tail_by_step(w, g, idx, wt, C):
    """dispatch -> expert FFN -> combine on the given routing tables."""
    act = "swiglu" if w.act == W.ACT_SWIGLU else "gelu"
    d = api.dispatch(idx, g["x"], w.E, C, d_ff=w.F, act=act)
    y = api.expert_ffn(d["x_perm"], d["offsets"], g["W1"], g["W2"], w.T, w.k, C, act, W3=g["W3"], b1=g["b1"],
                       b2=g["b2"])
    out, moe = api.combine(y, idx, wt, d["pos"], d["offsets"], g["x"], w.E, C, w.dtype, d_ff=w.F, want_moe=True)
    torch.cuda.synchronize()
    return out, moe, d


def _with_biases(w, inp, seed):
    gen = torch.Generator().manual_seed(seed)
    if w.act == W.ACT_GELU:
        inp["b1"] = torch.randn(w.E, w.F, generator=gen) * 0.3
    inp["b2"] = torch.randn(w.E, w.d, generator=gen) * 0.3
    return inp


def _logit_bound(inp, H):
    """|fp32 logit - exact| allowed: 2e-5 ||x_t|| ||w_e|| (summation depth
    below 300 at fp32's 2^-24, with room), scaled by |eps| on the noise term."""
    x = W.as_f64_numpy(inp["x"])
    nx = np.linalg.norm(x, axis=1)[:, None]
    wg = np.linalg.norm(W.as_f64_numpy(inp["W_g"]), axis=0)[None, :]
    b = 2e-5 * nx * wg
    if inp.get("W_noise") is not None:
        wn = np.linalg.norm(W.as_f64_numpy(inp["W_noise"]), axis=0)[None, :]
        b = b + 2e-5 * nx * wn * np.abs(W.as_f64_numpy(inp["eps"])) + 1e-6 * np.abs(H)
    return b + 1e-6


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_decode_layer_equals_step_by_step_and_oracle(w):
    inp = W.make_inputs(w)
    if w.name == "dec_gelu":
        inp = _with_biases(w, inp, 85)
    g = to_gpu(inp)
    C = api.capacity(w.T, w.k, w.E, w.capacity_factor)
    gpu = gpu_forward(w, g)
    # the standalone router: the same exact top-k; gates to rounding
    idx_s, wt_s, _ = api.route(g["x"], g["W_g"], w.k, b_g=g["b_g"], W_noise=g["W_noise"], eps=g["eps"])
    torch.cuda.synchronize()
    assert torch.equal(gpu["idx"], idx_s.cpu())
    if _self_routed(w):
        np.testing.assert_allclose(gpu["w"].numpy(), wt_s.cpu().numpy(), rtol=0, atol=1e-5)
    else:
        assert torch.equal(gpu["w"], wt_s.cpu())
    # the tail on the layer's own tables, bit for bit
    out_s, moe_s, d_s = _tail_by_step(w, g, gpu["idx"].cuda(), gpu["w"].cuda(), C)
    assert torch.equal(gpu["pos"], d_s["pos"].cpu())
    assert torch.equal(gpu["counts"], d_s["counts"].cpu())
    assert torch.equal(gpu["offsets"], d_s["offsets"].cpu())
    assert torch.equal(gpu["out"], out_s.cpu()), "fused decode FFN differs from the grouped GEMMs"
    assert torch.equal(gpu["moe"], moe_s.cpu())
    ref = oracle_forward(w, inp)
    check_layer(w, inp, gpu, ref)
    err = np.abs(gpu["logits"].numpy().astype(np.float64) - ref["H"])
    assert (err <= _logit_bound(inp, ref["H"])).all(), f"logits off by {err.max():.3e}"
    if w.name == "dec_drops":
        assert ref["dropped"] > 0


@pytest.mark.parametrize("gates", ["renorm", "raw"])
def test_self_routed_gate_modes(gates):
    """Both gate definitions inside the fused kernel: softmax over the selected
    logits, or the full-softmax probabilities of the selected experts."""
    w = CASES[2]
    inp = W.make_inputs(w)
    g = to_gpu(inp)
    gpu = gpu_forward(w, g, gates=gates)
    ref = oracle_forward(w, inp, gates=gates)
    check_layer(w, inp, gpu, ref)


def test_decode_layer_repeated_calls_and_graph_replay():
    """The fused kernel's tile ticket and counts (routing counters included)
    reset themselves: back-to-back calls, and replays of a captured graph,
    give the same output bit for bit."""
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
    """Overflow re-routing on a decode-sized batch (router, dispatch passes,
    then the fused FFN reading the final tables)."""
    w = CASES[2]
    inp = W.make_inputs(w)
    g = to_gpu(inp)
    gpu = gpu_forward(w, g, overflow="reroute")
    ref = oracle_forward(w, inp, overflow="reroute")
    assert ref["rerouted"] > 0
    check_layer(w, inp, gpu, ref)


@pytest.mark.parametrize("name,launches", [("decode_t128", 1), ("dec_e48", 3)])
def test_decode_kernel_count(name, launches):
    """Self-routed: the whole layer is one launch.  Otherwise router, dispatch
    and one kernel for both expert GEMMs and the combine: three."""
    from sparse_mixture_experts_51_b300 import _lib

    lib = _lib.load()
    w = W.WORKLOADS.get(name) or next(c for c in CASES if c.name == name)
    g = to_gpu(W.make_inputs(w))
    layer = api.MoELayer(g["W_g"], g["W1"], g["W2"], w.k, "swiglu", W3=g["W3"], capacity_factor=w.capacity_factor,
                         keep_routing=False)
    layer(g["x"])
    torch.cuda.synchronize()
    n0 = lib.moe_kernel_launches()
    layer(g["x"])
    torch.cuda.synchronize()
    assert lib.moe_kernel_launches() - n0 == launches


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
    idx, wt = gpu["idx"].cuda(), gpu["w"].cuda()
    d = api.dispatch(idx, g["x"], w.E, C, d_ff=w.F, act="swiglu")
    y = api.expert_ffn(d["x_perm"], d["offsets"], g["W1"], g["W2"], w.T, w.k, C, "swiglu", W3=g["W3"])
    ys = api.shared_ffn(g["x"], act="swiglu", **shared_args(g))
    out, moe = api.combine(y, idx, wt, d["pos"], d["offsets"], g["x"], w.E, C, w.dtype, d_ff=w.F, want_moe=True,
                           y_shared=ys)
    torch.cuda.synchronize()
    assert torch.equal(gpu["out"], out.cpu())
    assert torch.equal(gpu["moe"], moe.cpu())


def test_self_routed_router_stats():
    """The rank tiles add their counters (tokens settled in fp64, near ties)
    to the caller's stats like the router kernels: called twice, they double."""
    w = CASES[0]
    g = to_gpu(W.make_inputs(w))
    stats = torch.zeros(2, dtype=torch.int64, device="cuda")
    layer = api.MoELayer(g["W_g"], g["W1"], g["W2"], w.k, "swiglu", W3=g["W3"], capacity_factor=w.capacity_factor,
                         keep_routing=False)
    layer(g["x"], stats=stats)
    torch.cuda.synchronize()
    once = stats.clone()
    layer(g["x"], stats=stats)
    torch.cuda.synchronize()
    assert torch.equal(stats, 2 * once)
    assert int(once[0]) <= w.T and int(once[1]) <= w.T

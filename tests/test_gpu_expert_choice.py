"""Expert-choice routing on the CUDA path against the fp64 oracle.

Bar: every expert's chosen token set bit-exact (the selection is made exact
by the router's error radii and the fp64 re-scoring of the undecided band),
counts / offsets / drop count exact; gates (router probabilities from fp32
logits) within 1e-5; the layer output and the expert sum within relative L2
1e-5 (fp32 layers) / 1e-2 (bf16 layers)."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_mixture_experts_51_b300 import api
from sparse_mixture_experts_51_b300 import workloads as W

from _parity import F64Experts, check_rows, oracle_shared, rel_l2, segment_edge_rows, shared_args, to_gpu, tolerance

pytestmark = pytest.mark.gpu

GATE_TOL = 1e-5


def _capacity(w, C):
    return C if C is not None else api.capacity(w.T, w.k, w.E, w.capacity_factor)


def oracle_ec(w, inp, C=None, tokens=None):
    f = W.as_f64_numpy
    return O.forward_expert_choice(
        f(inp["x"]), f(inp["W_g"]), w.act, F64Experts(inp["W1"]), F64Experts(inp["W2"]),
        W3=None if inp["W3"] is None else F64Experts(inp["W3"]),
        b1=None if inp["b1"] is None else F64Experts(inp["b1"]),
        b2=None if inp["b2"] is None else F64Experts(inp["b2"]),
        b_g=f(inp["b_g"]), W_noise=f(inp["W_noise"]), eps=f(inp["eps"]), C=_capacity(w, C), tokens=tokens,
        shared=oracle_shared(inp))


def gpu_ec(w, g, C=None):
    act = "swiglu" if w.act == W.ACT_SWIGLU else "gelu"
    Cc = _capacity(w, C)
    layer = api.MoELayer(g["W_g"], g["W1"], g["W2"], w.k, act, W3=g["W3"], b_g=g["b_g"], W_noise=g["W_noise"],
                         b1=g["b1"], b2=g["b2"], C=Cc, want_moe=True, routing="expert", **shared_args(g))
    out = layer(g["x"], eps=g["eps"])
    r = layer.last
    route = api.route_expert_choice(g["x"], g["W_g"], w.k, Cc, b_g=g["b_g"], W_noise=g["W_noise"], eps=g["eps"],
                                    want_logits=True)
    torch.cuda.synchronize()
    assert api.get_device_error(r["ws"]) == 0
    assert api.get_device_error(route["ws"]) == 0
    return dict(out=out.cpu(), moe=r["moe"].cpu(), counts=r["counts"].cpu(), offsets=r["offsets"].cpu(),
                dropped=r["dropped"].cpu(), sel=route["sel"].cpu(), gates=route["gates"].cpu(),
                dropped_route=route["dropped"].cpu(), C=Cc)


def check_ec(w, gpu, ref, tokens=None):
    T, E = w.T, w.E
    Cp = min(gpu["C"], T)
    np.testing.assert_array_equal(gpu["sel"].numpy(), ref["sel"], err_msg="chosen tokens")
    np.testing.assert_array_equal(gpu["counts"].numpy(), np.full(E, Cp), err_msg="counts")
    np.testing.assert_array_equal(gpu["offsets"].numpy(), np.arange(E + 1) * Cp, err_msg="offsets")
    assert int(gpu["dropped"][0]) == ref["dropped"] == int(gpu["dropped_route"][0])
    np.testing.assert_allclose(gpu["gates"].numpy(), ref["gates"], rtol=0, atol=GATE_TOL, err_msg="gates")
    toks = np.arange(T) if tokens is None else np.asarray(tokens)
    tol = tolerance(w)
    if T == 0:
        return
    e1 = rel_l2(gpu["moe"].numpy()[toks], ref["moe"])
    e2 = rel_l2(gpu["out"].float().numpy()[toks], ref["out"])
    assert e1 <= tol and e2 <= tol, (e1, e2)
    # token by token as well
    check_rows("moe", gpu["moe"].numpy()[toks], ref["moe"], tol, labels=toks)
    check_rows("out", gpu["out"].float().numpy()[toks], ref["out"], tol, labels=toks)


CASES = [
    W.WORKLOADS["tiny_fp32"],
    W.Workload("ec_swiglu", T=333, d=256, E=8, k=2, F=256, act=W.ACT_SWIGLU, capacity_factor=1.0,
               dtype=torch.bfloat16, seed=61),
    W.Workload("ec_noisy_zipf_top1", T=700, d=128, E=16, k=1, F=128, act=W.ACT_GELU, capacity_factor=1.0,
               dtype=torch.bfloat16, seed=62, noisy=True, zipf_bias=True),
    W.Workload("ec_fine_grained", T=77, d=512, E=64, k=6, F=128, act=W.ACT_SWIGLU, capacity_factor=2.0,
               dtype=torch.bfloat16, seed=63),
    W.Workload("ec_fp32_noisy", T=150, d=48, E=5, k=2, F=40, act=W.ACT_GELU, capacity_factor=0.8,
               dtype=torch.float32, seed=64, noisy=True, zipf_bias=True, expert_bias=True),
    W.Workload("ec_shared", T=300, d=128, E=8, k=2, F=128, act=W.ACT_SWIGLU, capacity_factor=1.0,
               dtype=torch.bfloat16, seed=65, n_shared=1, F_shared=256),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_expert_choice_layer(w):
    inp = W.make_inputs(w)
    gpu = gpu_ec(w, to_gpu(inp))
    ref = oracle_ec(w, inp)
    check_ec(w, gpu, ref)


def test_capacity_above_T_takes_every_token():
    w = CASES[1].with_(T=50, name="ec_all")
    inp = W.make_inputs(w)
    gpu = gpu_ec(w, to_gpu(inp), C=70)
    ref = oracle_ec(w, inp, C=70)
    assert ref["dropped"] == 0
    check_ec(w, gpu, ref)


def test_zero_capacity_and_empty_batch():
    w = CASES[1]
    inp = W.make_inputs(w)
    gpu = gpu_ec(w, to_gpu(inp), C=0)
    ref = oracle_ec(w, inp, C=0)
    assert ref["dropped"] == w.T
    check_ec(w, gpu, ref)
    we = w.with_(T=0, name="ec_empty")
    inp = W.make_inputs(we)
    gpu = gpu_ec(we, to_gpu(inp), C=5)
    assert int(gpu["dropped"][0]) == 0 and gpu["out"].shape == (0, we.d)


@pytest.mark.parametrize("T", [700, 3000])
def test_exact_ties_go_to_lower_token(T):
    """Integer tokens and router weights: integer scores with large groups of
    equal values at every expert's boundary (the undecided band holds them;
    T = 3000 makes it larger than one block's worth)."""
    w = W.Workload("ec_ties", T=T, d=64, E=4, k=1, F=64, act=W.ACT_GELU, capacity_factor=1.0,
                   dtype=torch.bfloat16, seed=66)
    inp = W.make_inputs(w)
    g = torch.Generator().manual_seed(67)
    x = torch.randint(-1, 2, (T, w.d), generator=g)
    if T > 1024:
        x[torch.arange(T) % 3 != 0] = 0  # two thirds of the tokens score exactly 0 for every expert
    inp["x"] = x.to(torch.bfloat16)
    inp["W_g"] = torch.randint(-1, 2, (w.d, w.E), generator=g).to(torch.float32)
    gpu = gpu_ec(w, to_gpu(inp))
    ref = oracle_ec(w, inp)
    check_ec(w, gpu, ref)


def test_full_size_bf16_t4096_expert_choice():
    """The bench layer (T=4096, d=1024, E=8, SwiGLU d_ff=4096) with expert choice
    at the same capacity (C = 1280 per expert), whole batch."""
    w = W.WORKLOADS["bf16_t4096"]
    inp = W.make_inputs(w)
    gpu = gpu_ec(w, to_gpu(inp))
    ref = oracle_ec(w, inp)
    check_ec(w, gpu, ref)


def test_full_size_switch_expert_choice_sampled():
    """The Switch-style layer (T=32768, E=64, noisy, Zipf bias) with expert
    choice: selections over the whole batch, outputs on a token sample."""
    w = W.WORKLOADS["switch_top1"]
    inp = W.make_inputs(w)
    gpu = gpu_ec(w, to_gpu(inp))
    toks = np.random.default_rng(9).choice(w.T, size=64, replace=False).tolist()
    # the tokens on the edge rows of every expert's segment (rows e*C' .. e*C'+C'-1 hold sel[e])
    Cp = min(gpu["C"], w.T)
    sel = gpu["sel"].numpy().reshape(-1)
    edges = segment_edge_rows(np.arange(w.E + 1) * Cp, head=2, tail=8)
    toks = np.array(sorted(set(toks + sel[edges].tolist())))
    ref = oracle_ec(w, inp, tokens=toks)
    check_ec(w, gpu, ref, tokens=toks)


def test_expert_choice_graph_replay():
    w = CASES[1]
    inp = W.make_inputs(w)
    g = to_gpu(inp)
    layer = api.MoELayer(g["W_g"], g["W1"], g["W2"], w.k, "swiglu", W3=g["W3"], capacity_factor=w.capacity_factor,
                         routing="expert")
    eager = layer(g["x"]).clone()
    cap = layer.capture(g["x"])
    cap.replay()
    torch.cuda.synchronize()
    assert torch.equal(cap.out, eager)

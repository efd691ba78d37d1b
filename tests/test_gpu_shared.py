"""Shared experts (every token through one dense FFN, weight 1, added in the
combine) on the CUDA path against the fp64 oracle.

Bar as for the routed layer: routing, slots and drops bit-exact, gates to
1e-6 (fp32) / 1e-4 (bf16), the layer output and the expert sum within
relative L2 1e-5 (fp32 layers) / 1e-2 (bf16 layers); the shared FFN alone
within the same relative L2 bounds."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_mixture_experts_51_b300 import api
from sparse_mixture_experts_51_b300 import workloads as W

from _parity import (check_layer, check_rows, edge_tokens, gpu_forward, oracle_forward, oracle_shared, rel_l2,
                     shared_args, to_gpu, tolerance)

pytestmark = pytest.mark.gpu

CASES = [
    # SwiGLU, two shared experts, drops, ragged token count
    W.Workload("swiglu_shared", T=333, d=256, E=8, k=2, F=256, act=W.ACT_SWIGLU, capacity_factor=1.0,
               dtype=torch.bfloat16, seed=51, n_shared=2, F_shared=128),
    # GELU, one shared expert with a ragged last N tile (320 = 256 + 64) and
    # 256-row tiles (T > 512)
    W.Workload("gelu_shared_wide", T=3000, d=128, E=4, k=2, F=192, act=W.ACT_GELU, capacity_factor=1.1,
               dtype=torch.bfloat16, seed=52, n_shared=1, F_shared=320),
    # fine-grained routed experts + shared experts, top-6
    W.Workload("fine_grained_shared", T=77, d=512, E=64, k=6, F=256, act=W.ACT_SWIGLU, capacity_factor=2.0,
               dtype=torch.bfloat16, seed=53, n_shared=2, F_shared=256),
    # fp32 layer (CUDA-core FFN), noisy routing, three shared experts of odd width
    W.Workload("fp32_shared", T=150, d=48, E=5, k=2, F=40, act=W.ACT_GELU, capacity_factor=1.0,
               dtype=torch.float32, seed=54, noisy=True, zipf_bias=True, n_shared=3, F_shared=24),
]


def _with_bias(w, inp, seed):
    """Nonzero shared-expert biases (b1s for GELU, b2s for both)."""
    g = torch.Generator().manual_seed(seed)
    S, Fs, d = w.n_shared, w.F_shared, w.d
    if w.act == W.ACT_GELU:
        inp["b1s"] = torch.randn(S, Fs, generator=g) * 0.5
    inp["b2s"] = torch.randn(S, d, generator=g) * 0.5
    return inp


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_layer_with_shared_experts(w):
    inp = _with_bias(w, W.make_inputs(w), w.seed + 100)
    gpu = gpu_forward(w, to_gpu(inp))
    ref = oracle_forward(w, inp)
    check_layer(w, inp, gpu, ref)


def test_zero_capacity_leaves_residual_plus_shared():
    w = CASES[0]
    inp = W.make_inputs(w)
    gpu = gpu_forward(w, to_gpu(inp), C=0)
    ref = oracle_forward(w, inp, C=0)
    assert ref["dropped"] == w.T * w.k
    check_layer(w, inp, gpu, ref)


@pytest.mark.parametrize("w", [CASES[0], CASES[1], CASES[3]], ids=lambda w: w.name)
def test_shared_ffn_alone(w):
    inp = _with_bias(w, W.make_inputs(w), w.seed + 200)
    g = to_gpu(inp)
    act = "swiglu" if w.act == W.ACT_SWIGLU else "gelu"
    y = api.shared_ffn(g["x"], act=act, **shared_args(g))
    torch.cuda.synchronize()
    sh = oracle_shared(inp)
    ref = O.shared_experts(W.as_f64_numpy(inp["x"]), w.act, sh["W1s"], sh["W2s"], sh["W3s"], sh["b1s"], sh["b2s"])
    err = rel_l2(y.cpu().numpy(), ref)
    assert err <= tolerance(w), err
    # every token's row, the dense group's last (partial) M tile included
    check_rows("shared", y.cpu().numpy(), ref, tolerance(w))


def test_step_by_step_combine_with_shared_matches_forward():
    """route -> dispatch -> expert_ffn -> shared_ffn -> combine(y_shared) gives
    the whole-layer forward's output bit for bit."""
    w = CASES[0]
    inp = W.make_inputs(w)
    g = to_gpu(inp)
    sa = shared_args(g)
    C = api.capacity(w.T, w.k, w.E, w.capacity_factor)
    idx, gates, _ = api.route(g["x"], g["W_g"], w.k)
    d = api.dispatch(idx, g["x"], w.E, C, d_ff=w.F, act="swiglu")
    y = api.expert_ffn(d["x_perm"], d["offsets"], g["W1"], g["W2"], w.T, w.k, C, "swiglu", W3=g["W3"])
    ys = api.shared_ffn(g["x"], act="swiglu", **sa)
    out, moe = api.combine(y, idx, gates, d["pos"], d["offsets"], g["x"], w.E, C, w.dtype, d_ff=w.F,
                           want_moe=True, y_shared=ys)
    full = gpu_forward(w, g)
    assert torch.equal(out.cpu(), full["out"])
    ref = oracle_forward(w, inp)
    assert rel_l2(moe.cpu().numpy(), ref["moe"]) <= tolerance(w)
    check_rows("moe", moe.cpu().numpy(), ref["moe"], tolerance(w))


def test_full_size_shared_layer_sampled():
    """The full shared_t4096 layer (T=4096, d=2048, 64 experts top-6 + two
    shared experts of width 1408): routing bit-exact over the whole batch,
    outputs on a token sample."""
    w = W.WORKLOADS["shared_t4096"]
    inp = W.make_inputs(w)
    gpu = gpu_forward(w, to_gpu(inp))
    rng = np.random.default_rng(7)
    toks = rng.choice(w.T, size=48, replace=False).tolist()
    # the tokens on each expert's segment edges (last 8 rows, partial tiles): 64 experts make this a large sample
    toks += edge_tokens(gpu["idx"].numpy(), gpu["pos"].numpy(), gpu["offsets"].numpy(), head=1, tail=8)
    toks = np.array(sorted(set(toks + list(range(w.T - 32, w.T)))))
    ref = oracle_forward(w, inp, tokens=toks)
    check_layer(w, inp, gpu, ref, tokens=toks)


def test_graph_replay_with_shared_experts():
    w = CASES[0]
    inp = W.make_inputs(w)
    g = to_gpu(inp)
    layer = api.MoELayer(g["W_g"], g["W1"], g["W2"], w.k, "swiglu", W3=g["W3"], capacity_factor=w.capacity_factor,
                         **shared_args(g))
    eager = layer(g["x"]).clone()
    cap = layer.capture(g["x"])
    cap.replay()
    torch.cuda.synchronize()
    assert torch.equal(cap.out, eager)

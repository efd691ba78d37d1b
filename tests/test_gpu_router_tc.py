"""The tensor-core filter router (wide logit tables of long bf16 batches,
T >= 16384, taken by the whole-layer forward) against the fp64 oracle and against the
CUDA-core router: the same exact top-k, rank order, backup rank and drops;
gates within 1e-4 of the oracle's; outputs within relative L2 1e-2."""
import numpy as np
import pytest
import torch

from sparse_mixture_experts_51_b300 import api
from sparse_mixture_experts_51_b300 import workloads as W

from _parity import check_layer, gpu_forward, oracle_forward, to_gpu

pytestmark = pytest.mark.gpu

CASES = [
    # Switch-like: noisy top-1, Zipf-biased router, 128 logit columns
    W.Workload("tc_noisy_top1", T=16384, d=256, E=64, k=1, F=64, act=W.ACT_GELU, capacity_factor=1.0,
               dtype=torch.bfloat16, seed=81, noisy=True, zipf_bias=True),
    # fine-grained top-6, 64 columns
    W.Workload("tc_top6", T=16384, d=256, E=64, k=6, F=64, act=W.ACT_SWIGLU, capacity_factor=1.25,
               dtype=torch.bfloat16, seed=82),
    # the widest table: 128 experts with noise (256 columns), top-2
    W.Workload("tc_e128_noisy", T=16400, d=128, E=128, k=2, F=64, act=W.ACT_GELU, capacity_factor=1.0,
               dtype=torch.bfloat16, seed=83, noisy=True),
    # 32 experts top-4 (32 columns), d not a multiple of 128
    W.Workload("tc_e32", T=16500, d=192, E=32, k=4, F=64, act=W.ACT_SWIGLU, capacity_factor=1.0,
               dtype=torch.bfloat16, seed=84, zipf_bias=True),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_tensor_core_router_layer(w):
    inp = W.make_inputs(w)
    g = to_gpu(inp)
    gpu = gpu_forward(w, g)
    ref = oracle_forward(w, inp)
    check_layer(w, inp, gpu, ref)
    # the CUDA-core router (moe_route, no workspace) selects the same experts
    idx, gates, _ = api.route(g["x"], g["W_g"], w.k, b_g=g["b_g"], W_noise=g["W_noise"], eps=g["eps"])
    torch.cuda.synchronize()
    np.testing.assert_array_equal(idx.cpu().numpy(), gpu["idx"].numpy())
    np.testing.assert_allclose(gates.cpu().numpy(), gpu["w"].numpy(), rtol=0, atol=1e-5)


def test_tensor_core_router_with_rerouting():
    """The backup (k+1)-th rank through the filter path."""
    w = CASES[3].with_(capacity_factor=0.8, name="tc_reroute")
    inp = W.make_inputs(w)
    gpu = gpu_forward(w, to_gpu(inp), overflow="reroute")
    ref = oracle_forward(w, inp, overflow="reroute")
    assert ref["rerouted"] > 0
    check_layer(w, inp, gpu, ref)


@pytest.mark.parametrize("k", [1, 2])
def test_tensor_core_router_exact_ties(k):
    """Integer tokens and router weights: many exactly equal logits; the
    lower expert index wins through the filter path too (top-1: tied experts
    are both candidates, so the single-candidate shortcut never takes them)."""
    w = W.Workload("tc_ties", T=16384, d=64, E=32, k=k, F=64, act=W.ACT_GELU, capacity_factor=2.0,
                   dtype=torch.bfloat16, seed=85)
    inp = W.make_inputs(w)
    g = torch.Generator().manual_seed(86)
    inp["x"] = torch.randint(-1, 2, (w.T, w.d), generator=g).to(torch.bfloat16)
    inp["W_g"] = torch.randint(-1, 2, (w.d, w.E), generator=g).to(torch.float32)
    gpu = gpu_forward(w, to_gpu(inp))
    ref = oracle_forward(w, inp)
    check_layer(w, inp, gpu, ref)

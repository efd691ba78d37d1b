"""Overflow variants on the CUDA path against the fp64 oracle: re-routing of
an over-capacity assignment to the token's backup (its (k+1)-th ranked)
expert, and un-renormalised (raw-p) gates.

Bar as for the default layer: final experts, slots, counts, offsets and the
drop count bit-exact (the backup's rank is settled as exactly as the
top-k), gates to 1e-6 (fp32) / 1e-4 (bf16), layer output and expert sum
within relative L2 1e-5 (fp32 layers) / 1e-2 (bf16 layers)."""
import numpy as np
import pytest
import torch

from sparse_mixture_experts_51_b300 import workloads as W

from _parity import check_layer, edge_tokens, gpu_forward, oracle_forward, to_gpu

pytestmark = pytest.mark.gpu

CASES = [
    # single-CTA dispatch passes, SwiGLU, Zipf-skewed router: the low-ranked experts have room
    W.Workload("rr_swiglu", T=333, d=256, E=8, k=2, F=256, act=W.ACT_SWIGLU, capacity_factor=0.8,
               dtype=torch.bfloat16, seed=71, zipf_bias=True),
    # Switch-style noisy top-1 with a Zipf bias: heavy overflow, many requests per backup
    W.Workload("rr_noisy_top1", T=700, d=128, E=16, k=1, F=128, act=W.ACT_GELU, capacity_factor=1.0,
               dtype=torch.bfloat16, seed=72, noisy=True, zipf_bias=True),
    # fine-grained top-6, tight capacity
    W.Workload("rr_fine_grained", T=150, d=512, E=64, k=6, F=128, act=W.ACT_SWIGLU, capacity_factor=0.7,
               dtype=torch.bfloat16, seed=73),
    # tiled dispatch passes (T*k > 8192) with the base counts of the second pass
    W.Workload("rr_multi_tile", T=5000, d=128, E=8, k=2, F=128, act=W.ACT_SWIGLU, capacity_factor=0.9,
               dtype=torch.bfloat16, seed=74, zipf_bias=True),
    # fp32 layer
    W.Workload("rr_fp32", T=150, d=48, E=5, k=2, F=40, act=W.ACT_GELU, capacity_factor=0.8,
               dtype=torch.float32, seed=75, noisy=True, zipf_bias=True),
]


def _run(w, gates="renorm", overflow="drop", C=None):
    inp = W.make_inputs(w)
    gpu = gpu_forward(w, to_gpu(inp), C=C, gates=gates, overflow=overflow)
    ref = oracle_forward(w, inp, C=C, gates=gates, overflow=overflow)
    check_layer(w, inp, gpu, ref)
    return gpu, ref


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_reroute(w):
    gpu, ref = _run(w, overflow="reroute")
    assert ref["rerouted"] > 0  # every case moves some assignments


@pytest.mark.parametrize("w", [CASES[0], CASES[1], CASES[4]], ids=lambda w: w.name)
def test_raw_gates(w):
    _run(w, gates="raw")


def test_raw_gates_with_reroute():
    _run(CASES[3], gates="raw", overflow="reroute")


def test_reroute_without_backups_when_k_equals_E():
    w = W.Workload("rr_k_eq_E", T=200, d=64, E=4, k=4, F=64, act=W.ACT_SWIGLU, capacity_factor=0.5,
                   dtype=torch.bfloat16, seed=76)
    gpu, ref = _run(w, overflow="reroute")
    assert ref["rerouted"] == 0 and ref["dropped"] > 0


def test_reroute_zero_capacity_drops_everything():
    gpu, ref = _run(CASES[0], overflow="reroute", C=0)
    assert ref["dropped"] == CASES[0].T * CASES[0].k


def test_full_size_switch_reroute_sampled():
    """The Switch-style layer (T=32768, E=64, noisy, Zipf bias, C=512) with
    re-routing: routing and the two dispatch passes over the whole batch
    bit-exact, outputs on a token sample."""
    w = W.WORKLOADS["switch_top1"]
    inp = W.make_inputs(w)
    gpu = gpu_forward(w, to_gpu(inp), overflow="reroute")
    toks = np.random.default_rng(11).choice(w.T, size=64, replace=False).tolist()
    toks = np.array(sorted(set(toks + edge_tokens(gpu["idx"].numpy(), gpu["pos"].numpy(), gpu["offsets"].numpy()))))
    ref = oracle_forward(w, inp, tokens=toks, overflow="reroute")
    assert ref["rerouted"] > 0
    check_layer(w, inp, gpu, ref, tokens=toks)

"""Parity of the routing diagnostics and the auxiliary load-balancing loss
(moe_routing_stats) with the fp64 oracle.

Bar: f (integer loads over T*k), utilisation and overflow bit-exact; the
load and kept-count imbalance (fp64 arithmetic on exact integers) within
1e-12 relative; P, the aux loss and the mean entropy within 2e-6 (P and aux
relative, entropy absolute): the kernel takes each token's softmax in fp32
(a few ulps, about 1e-7 relative per probability) and sums in fp64.  Where
the GPU's fp32 logits feed the kernel and the oracle uses fp64 logits, the
fp32 rounding of the logits adds up to ~1e-6 relative per probability, the
reason for 2e-6 instead of 1e-6."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_mixture_experts_51_b300 import api
from sparse_mixture_experts_51_b300 import workloads as W

from _parity import to_gpu

pytestmark = pytest.mark.gpu

SUMMARY = api.STATS_SUMMARY


def _check(gpu: dict, ref: dict, tol=2e-6):
    f = gpu["f"].cpu().numpy()
    P = gpu["P"].cpu().numpy()
    s = dict(zip(SUMMARY, gpu["summary"].cpu().tolist()))
    np.testing.assert_array_equal(f, ref["f"], err_msg="f")
    np.testing.assert_allclose(P, ref["P"], rtol=tol, atol=1e-12, err_msg="P")
    assert abs(s["aux_loss"] - ref["aux_loss"]) <= tol * max(1.0, abs(ref["aux_loss"])), (s, ref["aux_loss"])
    assert abs(s["entropy"] - ref["entropy"]) <= tol, (s["entropy"], ref["entropy"])
    for key in ("load_cv", "kept_cv"):
        assert abs(s[key] - ref[key]) <= 1e-12 * max(1.0, abs(ref[key])), (key, s[key], ref[key])
    assert s["utilisation"] == ref["utilisation"]
    assert s["overflow"] == ref["overflow"]


def _oracle_routing(w: W.Workload, inp: dict, C: int):
    f = W.as_f64_numpy
    H = O.logits(f(inp["x"]), f(inp["W_g"]), b_g=f(inp["b_g"]), W_noise=f(inp["W_noise"]), eps=f(inp["eps"]))
    idx = O.topk(H, w.k)
    disp = O.dispatch(idx, w.E, C)
    return H, idx, disp


LAYER_CASES = [
    W.WORKLOADS["tiny_fp32"],
    W.Workload("noisy_top1", T=700, d=128, E=16, k=1, F=128, act=W.ACT_GELU, capacity_factor=1.0,
               dtype=torch.bfloat16, seed=13, noisy=True, zipf_bias=True),
    W.Workload("fine_grained", T=77, d=512, E=64, k=6, F=128, act=W.ACT_SWIGLU, capacity_factor=2.0,
               dtype=torch.bfloat16, seed=14),
    W.Workload("fp32_noisy", T=150, d=48, E=5, k=2, F=40, act=W.ACT_GELU, capacity_factor=1.0,
               dtype=torch.float32, seed=16, noisy=True, zipf_bias=True),
    W.Workload("many_blocks", T=40000, d=64, E=8, k=2, F=64, act=W.ACT_SWIGLU, capacity_factor=0.9,
               dtype=torch.bfloat16, seed=18),
]


@pytest.mark.parametrize("w", LAYER_CASES, ids=lambda w: w.name)
def test_layer_routing_stats(w):
    """The layer's own logits, top-k table and dispatch counts feed the stats."""
    inp = W.make_inputs(w)
    g = to_gpu(inp)
    act = "swiglu" if w.act == W.ACT_SWIGLU else "gelu"
    layer = api.MoELayer(g["W_g"], g["W1"], g["W2"], w.k, act, W3=g["W3"], b_g=g["b_g"], W_noise=g["W_noise"],
                         b1=g["b1"], b2=g["b2"], capacity_factor=w.capacity_factor)
    layer(g["x"], eps=g["eps"])
    gpu = layer.routing_stats()
    torch.cuda.synchronize()
    assert api.get_device_error(layer.last["ws"]) == 0
    H, idx, disp = _oracle_routing(w, inp, layer.last["C"])
    np.testing.assert_array_equal(layer.last["idx"].cpu().numpy(), idx)
    ref = O.routing_stats(H, idx, disp["counts"], disp["dropped"])
    _check(gpu, ref)


FULL_ROUTERS = ["bf16_t4096", "mixtral_t16384", "switch_top1", "decode_t128"]


@pytest.mark.parametrize("name", FULL_ROUTERS)
def test_full_size_router_stats(name):
    """Full-size token batches: route + dispatch through the C ABI, then the stats.
    The expert width is irrelevant here and set small (the router inputs are
    drawn before the expert weights, so they are those of the full workload)."""
    w = W.WORKLOADS[name].with_(F=64)
    inp = W.make_inputs(w)
    g = to_gpu(inp)
    C = api.capacity(w.T, w.k, w.E, w.capacity_factor)
    idx, _, logits = api.route(g["x"], g["W_g"], w.k, b_g=g["b_g"], W_noise=g["W_noise"], eps=g["eps"],
                               want_logits=True)
    r = api.dispatch(idx, g["x"], w.E, C)
    gpu = api.routing_stats(logits, idx, r["counts"], r["dropped"], ws=r["ws"])
    torch.cuda.synchronize()
    assert api.get_device_error(r["ws"]) == 0
    H, idx_ref, disp = _oracle_routing(w, inp, C)
    np.testing.assert_array_equal(idx.cpu().numpy(), idx_ref)
    ref = O.routing_stats(H, idx_ref, disp["counts"], disp["dropped"])
    _check(gpu, ref)


TABLES = [
    (1001, 128, 16, 31),   # widest E and k, ragged token count
    (5, 1, 1, 32),         # one expert: P = 1, entropy 0, aux loss 1
    (100000, 3, 2, 33),    # every block of the grid busy, odd E
    (1, 7, 3, 34),         # one token
    (300, 33, 4, 35),      # E just above one warp
]


@pytest.mark.parametrize("T,E,k,seed", TABLES)
def test_stats_of_arbitrary_tables(T, E, k, seed):
    """Same fp32 logits on both sides (no router in between); any expert ids."""
    t = W.make_routing_tables(T, E, k, seed)
    g = to_gpu(t)
    gpu = api.routing_stats(g["logits"], g["idx"], g["counts"], g["dropped"])
    ref = O.routing_stats(W.as_f64_numpy(t["logits"]), t["idx"].numpy(), t["counts"].numpy(), int(t["dropped"][0]))
    _check(gpu, ref, tol=1e-6)
    if E == 1:
        s = api.stats_summary(gpu)
        assert s["aux_loss"] == 1.0 and s["entropy"] == 0.0


def test_empty_batch_gives_zeros():
    logits = torch.empty(0, 8, dtype=torch.float32, device="cuda")
    idx = torch.empty(0, 2, dtype=torch.int32, device="cuda")
    counts = torch.zeros(8, dtype=torch.int32, device="cuda")
    dropped = torch.zeros(1, dtype=torch.int64, device="cuda")
    gpu = api.routing_stats(logits, idx, counts, dropped)
    assert gpu["f"].abs().sum().item() == 0 and gpu["P"].abs().sum().item() == 0
    assert gpu["summary"].abs().sum().item() == 0


def test_repeat_calls_on_one_workspace_are_deterministic():
    """The last-block ticket resets itself: a second and third call on the same
    workspace (different inputs in between) give the oracle's values again,
    bit-identical to the first."""
    T, E, k = 20000, 16, 2
    a = to_gpu(W.make_routing_tables(T, E, k, 41))
    b = to_gpu(W.make_routing_tables(T, E, k, 42))
    shape = api.shape_of(T, 64, E, k, 64, torch.float32, 0)
    ws = api.new_workspace(shape, 0, "cuda")
    r1 = api.routing_stats(a["logits"], a["idx"], a["counts"], a["dropped"], ws=ws)
    r1 = {n: v.clone() for n, v in r1.items()}
    rb = api.routing_stats(b["logits"], b["idx"], b["counts"], b["dropped"], ws=ws)
    r2 = api.routing_stats(a["logits"], a["idx"], a["counts"], a["dropped"], ws=ws)
    torch.cuda.synchronize()
    for n in ("f", "P", "summary"):
        assert torch.equal(r1[n], r2[n]), n
    tb = {n: v.cpu() for n, v in b.items()}
    ref = O.routing_stats(W.as_f64_numpy(tb["logits"]), tb["idx"].numpy(), tb["counts"].numpy(),
                          int(tb["dropped"][0]))
    _check(rb, ref, tol=1e-6)


def test_out_of_range_expert_is_reported():
    t = W.make_routing_tables(500, 8, 2, 43)
    t["idx"][123, 1] = 8  # one id past the last expert
    g = to_gpu(t)
    shape = api.shape_of(500, 64, 8, 2, 64, torch.float32, 0)
    ws = api.new_workspace(shape, 0, "cuda")
    gpu = api.routing_stats(g["logits"], g["idx"], g["counts"], g["dropped"], ws=ws)
    assert api.get_device_error(ws) == 6  # MOE_ERR_BOUNDS
    # the bad assignment is counted in no load
    assert gpu["f"].sum().item() * 1000 == pytest.approx(999, abs=1e-9)
    assert api.get_device_error(ws) == 0

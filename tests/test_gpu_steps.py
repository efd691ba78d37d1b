"""Per-step parity through the separate C entry points (moe_route,
moe_dispatch, moe_expert_ffn, moe_combine) and the bounded-wait error path."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_mixture_experts_51_b300 import _lib, api
from sparse_mixture_experts_51_b300 import workloads as W

from _parity import F64Experts, check_rows, rel_l2, to_gpu

pytestmark = pytest.mark.gpu

CASES = [
    W.Workload("steps_swiglu", T=600, d=256, E=8, k=2, F=384, act=W.ACT_SWIGLU, capacity_factor=1.0,
               dtype=torch.bfloat16, seed=31),
    W.Workload("steps_noisy_gelu", T=900, d=192, E=32, k=1, F=256, act=W.ACT_GELU, capacity_factor=1.0,
               dtype=torch.bfloat16, seed=32, noisy=True, zipf_bias=True),
    W.Workload("steps_fp32", T=64, d=32, E=4, k=2, F=64, act=W.ACT_GELU, capacity_factor=1.25,
               dtype=torch.float32, seed=33, expert_bias=True),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_steps(w):
    inp = W.make_inputs(w)
    g = to_gpu(inp)
    f = W.as_f64_numpy
    C = O.capacity(w.T, w.k, w.E, w.capacity_factor)
    assert api.capacity(w.T, w.k, w.E, w.capacity_factor) == C

    # ---- route: exact top-k, gates, fp32 logits
    idx, gates, logits = api.route(g["x"], g["W_g"], w.k, b_g=g["b_g"], W_noise=g["W_noise"], eps=g["eps"],
                                   want_logits=True)
    H = O.logits(f(inp["x"]), f(inp["W_g"]), f(inp["b_g"]), f(inp["W_noise"]), f(inp["eps"]))
    ref_idx = O.topk(H, w.k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    np.testing.assert_allclose(gates.cpu().numpy(), O.gates(H, ref_idx), rtol=0, atol=1e-4)
    np.testing.assert_allclose(logits.cpu().numpy(), H, rtol=1e-4, atol=1e-4)

    # ---- dispatch on the GPU's own top-k table: bit-exact
    d = api.dispatch(idx, g["x"], w.E, C, d_ff=w.F, act=w.act, want_row_token=True)
    ref = O.dispatch(idx.cpu().numpy(), w.E, C)
    np.testing.assert_array_equal(d["pos"].cpu().numpy(), ref["pos"])
    np.testing.assert_array_equal(d["counts"].cpu().numpy(), ref["counts"])
    np.testing.assert_array_equal(d["offsets"].cpu().numpy(), ref["offsets"])
    assert int(d["dropped"].item()) == ref["dropped"]
    R = int(ref["offsets"][-1])
    rt = d["row_token"].cpu().numpy()[:R]
    # every kept (t, r) lands on row offsets[e] + pos, carrying token t exactly
    for t in range(w.T):
        for r in range(w.k):
            if ref["pos"][t, r] >= 0:
                row = ref["offsets"][idx[t, r].item()] + ref["pos"][t, r]
                assert rt[row] == t
    assert torch.equal(d["x_perm"][:R].cpu(), inp["x"][torch.from_numpy(rt.astype(np.int64))])

    # ---- expert FFN on the grouped rows
    y = api.expert_ffn(d["x_perm"], d["offsets"], g["W1"], g["W2"], w.T, w.k, C, w.act, W3=g["W3"],
                       b1=g["b1"], b2=g["b2"])
    yc = y[:R].cpu().numpy()
    xp = W.as_f64_numpy(d["x_perm"][:R].cpu())
    want = np.zeros_like(yc, dtype=np.float64)
    offs = ref["offsets"]
    for e in range(w.E):
        a, b = offs[e], offs[e + 1]
        if b > a:
            want[a:b] = O.expert(xp[a:b], e, w.act, F64Experts(inp["W1"]),
                                 None if inp["W3"] is None else F64Experts(inp["W3"]), F64Experts(inp["W2"]),
                                 None if inp["b1"] is None else F64Experts(inp["b1"]),
                                 None if inp["b2"] is None else F64Experts(inp["b2"]))
    tol = 1e-5 if w.dtype == torch.float32 else 1e-2
    assert rel_l2(yc, want) <= tol
    # every grouped row (each expert's segment-end rows and partial M tiles included)
    check_rows("y_perm", yc, want, tol)

    # ---- combine the GPU's expert rows: fp32 weighted sum in rank order
    out, moe = api.combine(y, idx, gates, d["pos"], d["offsets"], g["x"], w.E, C, w.dtype, d_ff=w.F, want_moe=True)
    yy = y.cpu().double().numpy()
    gw = gates.cpu().double().numpy()
    pos = ref["pos"]
    ref_moe = np.zeros((w.T, w.d))
    for t in range(w.T):
        for r in range(w.k):
            if pos[t, r] >= 0:
                ref_moe[t] += gw[t, r] * yy[offs[idx[t, r].item()] + pos[t, r]]
    np.testing.assert_allclose(moe.cpu().numpy(), ref_moe, rtol=1e-5, atol=1e-6)
    ref_out = W.as_f64_numpy(inp["x"]) + ref_moe
    # bf16 output rounding moves each element by at most 2^-8 of itself, so every row stays within 2^-8 (+ fp32 sums)
    out_tol = 1e-6 if w.dtype == torch.float32 else 4e-3
    assert rel_l2(out.float().cpu().numpy(), ref_out) <= out_tol
    check_rows("out", out.float().cpu().numpy(), ref_out, out_tol)
    # combine with no residual gives the expert sum alone
    out0, _ = api.combine(y, idx, gates, d["pos"], d["offsets"], None, w.E, C, w.dtype, d_ff=w.F)
    assert rel_l2(out0.float().cpu().numpy(), ref_moe) <= out_tol
    check_rows("out without residual", out0.float().cpu().numpy(), ref_moe, out_tol)


def test_route_near_tie_statistic():
    """Tokens whose k-th and (k+1)-th logits are within 1e-4 are counted."""
    T, d, E = 64, 64, 4
    x = torch.zeros(T, d, dtype=torch.bfloat16)
    x[:, 0] = 1.0
    Wg = torch.zeros(d, E)
    Wg[0] = torch.tensor([1.0, 0.99995, 0.5, 0.0])  # gap 5e-5 between experts 0 and 1
    stats = torch.zeros(2, dtype=torch.int64, device="cuda")
    idx, _, _ = api.route(x.cuda(), Wg.cuda(), 1, stats=stats)
    assert (idx.cpu()[:, 0] == 0).all()
    assert int(stats[1].item()) == T


def test_dispatch_bounded_wait_reports_timeout():
    """A dispatch tile that never publishes its totals makes the next tile's
    bounded wait run out: the error word says MOE_ERR_DEVICE_TIMEOUT, and the
    context stays usable for the next call."""
    lib = _lib.load()
    T, k, E, d = 3000, 2, 8, 64  # 6000 assignments = 2 dispatch tiles
    g = torch.Generator().manual_seed(3)
    idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).int().cuda()
    x = torch.randn(T, d, generator=g).to(torch.bfloat16).cuda()
    C = 2000
    shape = api.shape_of(T, d, E, k, 64, torch.bfloat16, "gelu")
    ws = api.new_workspace(shape, C)
    R = api.max_rows(shape, C)
    pos = torch.empty(T, k, dtype=torch.int32, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    dropped = torch.empty(1, dtype=torch.int64, device="cuda")
    x_perm = torch.empty(R, d, dtype=torch.bfloat16, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.moe_testing_dispatch_stalled(ctypes.byref(shape), C, P(idx), P(x), P(pos), P(counts), P(offsets),
                                          P(dropped), P(x_perm), 0, P(ws), ws.numel(),
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    assert api.get_device_error(ws) == 5  # MOE_ERR_DEVICE_TIMEOUT
    assert api.get_device_error(ws) == 0  # read clears it
    # the same workspace and context still dispatch correctly
    d2 = api.dispatch(idx, x, E, C, ws=ws)
    ref = O.dispatch(idx.cpu().numpy(), E, C)
    np.testing.assert_array_equal(d2["pos"].cpu().numpy(), ref["pos"])
    assert api.get_device_error(ws) == 0


@pytest.mark.parametrize("T,k,E,C", [(20000, 2, 16, 2600), (150000, 2, 8, 40000), (600, 3, 5, 300),
                                     (1000, 2, 128, 20), (2000, 2, 128, 40), (5000, 2, 8, 1000)],
                         ids=["40_small_tiles", "large_tiles", "single_cta_E5", "single_cta_E128", "tiles_E128",
                              "five_tiles"])
def test_dispatch_many_tiles(T, k, E, C):
    """Dispatch on one CTA (up to 2048 assignments) and across tiles, more
    than the 32-tile look-back window included (1024- and 4096-assignment
    tiles): slots, counts, offsets and drops bit-exact."""
    g = torch.Generator().manual_seed(T)
    logits = torch.randn(T, E, generator=g) + torch.linspace(1.0, -1.0, E)
    idx = logits.topk(k, dim=1).indices.int()
    x = torch.randn(T, 64, generator=g).to(torch.bfloat16)
    d = api.dispatch(idx.cuda(), x.cuda(), E, C)
    ref = O.dispatch(idx.numpy(), E, C)
    np.testing.assert_array_equal(d["pos"].cpu().numpy(), ref["pos"])
    np.testing.assert_array_equal(d["counts"].cpu().numpy(), ref["counts"])
    np.testing.assert_array_equal(d["offsets"].cpu().numpy(), ref["offsets"])
    assert int(d["dropped"].item()) == ref["dropped"]
    assert api.get_device_error(d["ws"]) == 0


@pytest.mark.parametrize("T", [300, 9000], ids=["single_cta", "tiled"])
def test_dispatch_out_of_range_expert_is_reported(T):
    """An expert id outside [0, E) takes no slot and sets MOE_ERR_BOUNDS; the
    other assignments are dispatched as if it were absent (both the one-CTA
    kernel and the tiled look-back kernel)."""
    k, E = 2, 6
    C = T * k // 3
    g = torch.Generator().manual_seed(9)
    idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).int()
    idx[17, 1] = E      # one past the last expert
    idx[250, 0] = -3    # negative
    x = torch.randn(T, 64, generator=g).to(torch.bfloat16)
    d = api.dispatch(idx.cuda(), x.cuda(), E, C)
    assert api.get_device_error(d["ws"]) == 6  # MOE_ERR_BOUNDS
    pos = d["pos"].cpu().numpy()
    assert pos[17, 1] == -1 and pos[250, 0] == -1
    clean = idx.numpy().copy()
    clean[17, 1] = -1
    clean[250, 0] = -1
    # the oracle on the table without the two bad assignments gives the same slots
    load = np.zeros(E, dtype=np.int64)
    for r in range(k):
        for t in range(T):
            e = clean[t, r]
            if e < 0:
                continue
            assert pos[t, r] == (load[e] if load[e] < C else -1)
            load[e] += 1
    np.testing.assert_array_equal(d["counts"].cpu().numpy(), np.minimum(load, C))

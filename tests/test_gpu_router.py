"""Router parity across launch plans: the thread-block cluster split over d
(1 to 16 CTAs per token tile), register tiles of 1 to 8 tokens per thread,
expert counts that are not multiples of four (scalar weight loads), weight
pointers that are not 16-byte aligned, the noise projection, fp32 and bf16
tokens, ragged token tiles and d not a multiple of the 32-wide slice.

Bar: top-k indices bit-exact against the fp64 oracle (the router certifies
its fp32 order or re-evaluates in fp64); gates within 1e-6 absolute; the fp32
logits within 1e-4 relative + absolute of the fp64 logits."""
import zlib

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_mixture_experts_51_b300 import api
from sparse_mixture_experts_51_b300 import workloads as W

pytestmark = pytest.mark.gpu

# (name, T, d, E, k, noisy, dtype)
PLANS = [
    ("small_T_wide_d", 40, 1024, 8, 2, False, torch.bfloat16),        # one tile, 16-CTA cluster
    ("decode_like", 128, 2048, 64, 6, False, torch.bfloat16),         # 8 tiles x up to 16 CTAs
    ("many_tokens_E8", 5000, 1024, 8, 2, False, torch.bfloat16),      # 2-token tiles, ragged last tile
    ("noisy_E64", 3000, 768, 64, 1, True, torch.bfloat16),            # 128 columns, 8-token tiles
    ("noisy_E128_k16", 300, 256, 128, 16, True, torch.bfloat16),      # 256 columns, widest tile
    ("odd_E5_noisy_fp32", 333, 96, 5, 2, True, torch.float32),        # scalar weight loads, 3 slices
    ("odd_E6_fp32_d48", 257, 48, 6, 3, False, torch.float32),         # d not a multiple of 32
    ("E3_top1_bf16", 1000, 64, 3, 1, False, torch.bfloat16),          # tiny column count
    ("E7_k7_all", 64, 128, 7, 7, False, torch.bfloat16),              # k = E
]


def _inputs(T, d, E, noisy, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, d, generator=g).to(dtype)
    Wg = torch.randn(d, E, generator=g) / d ** 0.5
    bg = torch.randn(E, generator=g) * 0.1
    Wn = torch.randn(d, E, generator=g) / d ** 0.5 if noisy else None
    eps = torch.randn(T, E, generator=g) if noisy else None
    return x, Wg, bg, Wn, eps


def _check(x, Wg, bg, Wn, eps, k, idx, gates, logits):
    f = W.as_f64_numpy
    H = O.logits(f(x), f(Wg), f(bg), f(Wn), f(eps))
    ref_idx = O.topk(H, k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    np.testing.assert_allclose(gates.cpu().numpy(), O.gates(H, ref_idx), rtol=0, atol=1e-6)
    np.testing.assert_allclose(logits.cpu().numpy(), H, rtol=1e-4, atol=1e-4)


@pytest.mark.parametrize("plan", PLANS, ids=lambda p: p[0])
def test_router_plans(plan):
    name, T, d, E, k, noisy, dtype = plan
    x, Wg, bg, Wn, eps = _inputs(T, d, E, noisy, dtype, seed=zlib.crc32(name.encode()) % 1000)
    cu = lambda t: None if t is None else t.cuda()
    idx, gates, logits = api.route(cu(x), cu(Wg), k, b_g=cu(bg), W_noise=cu(Wn), eps=cu(eps), want_logits=True)
    torch.cuda.synchronize()
    _check(x, Wg, bg, Wn, eps, k, idx, gates, logits)


def test_router_unaligned_weights():
    """Router weights that start 4 bytes past a 16-byte boundary are read with
    scalar loads; the result is the same."""
    T, d, E, k = 500, 256, 8, 2
    x, Wg, bg, Wn, eps = _inputs(T, d, E, True, torch.bfloat16, seed=77)
    big = torch.empty(d * E + 1, device="cuda")
    big[1:] = Wg.reshape(-1).cuda()
    Wg_u = big[1:].view(d, E)
    bign = torch.empty(d * E + 1, device="cuda")
    bign[1:] = Wn.reshape(-1).cuda()
    Wn_u = bign[1:].view(d, E)
    assert Wg_u.data_ptr() % 16 == 4
    idx, gates, logits = api.route(x.cuda(), Wg_u, k, b_g=bg.cuda(), W_noise=Wn_u, eps=eps.cuda(), want_logits=True)
    torch.cuda.synchronize()
    _check(x, Wg, bg, Wn, eps, k, idx, gates, logits)


def test_router_repeat_is_deterministic():
    T, d, E, k = 130, 2048, 64, 6
    x, Wg, bg, _, _ = _inputs(T, d, E, False, torch.bfloat16, seed=5)
    a = api.route(x.cuda(), Wg.cuda(), k, b_g=bg.cuda(), want_logits=True)
    b = api.route(x.cuda(), Wg.cuda(), k, b_g=bg.cuda(), want_logits=True)
    for u, v in zip(a, b):
        assert torch.equal(u, v)

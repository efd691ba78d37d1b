"""The margin of the tensor-core router filter, measured.

For long bf16 batches the router first computes approximate logits
g~ = x (hi + lo) on the tensor cores, where hi + lo is a two-part bf16 split
of each fp32 router column w (|w - hi - lo| <= 2^-16 |w|), and trusts each
g~ only to within delta = 2^-10 * 1.25 * ||x|| * ||w||: an expert whose upper
end stays below the k-th largest lower end is dropped without an exact
recomputation.  The products of bf16 operands are exact in fp32, but the
rounding of the tensor cores' fp32 accumulation is not specified, so the
margin is an assumption.  These tests measure the real error
|g~ - x.w| / (||x|| ||w||) (x.w in fp64 from the stored values) on inputs
built to make it large, and require it to stay below delta / 8."""
import ctypes
import math

import numpy as np
import pytest
import torch

from sparse_mixture_experts_51_b300 import _lib, api

pytestmark = pytest.mark.gpu

MARGIN = 2.0 ** -10  # the filter's delta, before its 1.25 inflation


def _filter(x, W_g, W_n=None):
    T, d = x.shape
    E = W_g.shape[1]
    nc = E * (2 if W_n is not None else 1)
    shape = api.shape_of(T, d, E, 2, 64, torch.bfloat16, "gelu")
    ws = api.new_workspace(shape, 0)
    out = torch.empty(T, nc, dtype=torch.float32, device="cuda")
    P = api._ptr
    st = _lib.load().moe_testing_router_filter(ctypes.byref(shape), P(x), P(W_g), P(W_n), P(out), P(ws), ws.numel(),
                                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    _lib.check(st, "moe_testing_router_filter")
    torch.cuda.synchronize()
    assert api.get_device_error(ws) == 0
    return out.cpu().double().numpy()


def _rel_error(x, W, approx):
    xd = x.cpu().double().numpy()
    Wd = W.cpu().double().numpy()
    exact = xd @ Wd
    scale = np.linalg.norm(xd, axis=1)[:, None] * np.linalg.norm(Wd, axis=0)[None, :]
    return np.abs(approx - exact) / scale


def _worst_split_columns(g, d, E):
    """fp32 values whose bf16 hi + lo split leaves the largest remainder:
    a mantissa with bits set just below lo's last bit (w = 2^e (1 + 2^-8 + ...
    + bits 17-23)), random signs and exponents."""
    mant = 1.0 + 2.0 ** -8 + sum(2.0 ** -i for i in range(17, 24))
    sign = torch.randint(0, 2, (d, E), generator=g).float() * 2 - 1
    expo = torch.randint(-6, 3, (d, E), generator=g).float()
    return (sign * mant * torch.pow(2.0, expo)).float()


@pytest.mark.parametrize("d", [768, 4096])
def test_filter_error_on_cancelling_columns_and_mixed_magnitudes(d):
    T, E = 2048, 64
    g = torch.Generator().manual_seed(d)
    # token rows whose elements span 2^-8 .. 2^8
    x = torch.randn(T, d, generator=g) * torch.pow(2.0, torch.randint(-8, 9, (T, d), generator=g).float())
    x = x.to(torch.bfloat16)
    W = torch.randn(d, E, generator=g) / math.sqrt(d)
    # columns 0-15: every product x[t,j] w[j] of the first half positive, of the
    # second half negative for token 0's signs, so the running sum climbs and cancels
    xs = torch.sign(x[0].float())
    half = d // 2
    for c in range(16):
        mag = torch.rand(d, generator=g) + 0.5
        W[:half, c] = xs[:half] * mag[:half]
        W[half:, c] = -xs[half:] * mag[half:]
    # columns 16-31: values with the worst two-part bf16 split
    W[:, 16:32] = _worst_split_columns(g, d, 16)
    W = W.contiguous().cuda()
    xg = x.cuda()
    err = _rel_error(x, W, _filter(xg, W))
    worst = float(err.max())
    print(f"d={d}: max |g~ - x.w| / (||x|| ||w||) = {worst:.3e} (delta/8 = {MARGIN / 8:.3e})")
    assert worst <= MARGIN / 8


def test_filter_error_with_noise_columns_at_the_switch_shape():
    """The Switch-style router's table: 64 gate and 64 noise columns, d = 768,
    tokens ~ N(0,1) (the columns of the noise weights are filtered too)."""
    T, d, E = 4096, 768, 64
    g = torch.Generator().manual_seed(5)
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    W_g = (torch.randn(d, E, generator=g) / math.sqrt(d)).contiguous()
    W_n = (torch.randn(d, E, generator=g) / math.sqrt(d)).contiguous()
    approx = _filter(x.cuda(), W_g.cuda(), W_n.cuda())
    err = np.concatenate([_rel_error(x, W_g, approx[:, :E]), _rel_error(x, W_n, approx[:, E:])], axis=1)
    worst = float(err.max())
    print(f"switch shape: max relative filter error {worst:.3e}")
    assert worst <= MARGIN / 8

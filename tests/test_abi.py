"""The C-ABI library loads, exports every symbol the header declares, and
rejects bad arguments on the host before anything reaches a GPU.  CPU only:
no call here launches a kernel (fake device pointers are never dereferenced
because validation fails first)."""
import ctypes
import os
import re

import pytest
import torch

from sparse_mixture_experts_51_b300 import _lib
from sparse_mixture_experts_51_b300._lib import MoeShape

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INC = os.path.join(ROOT, "include")

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3
FAKE = 0x7f0000000000  # 256-byte aligned, never dereferenced


def _declared():
    names = set()
    for f in os.listdir(INC):
        if f.endswith(".h"):
            src = open(os.path.join(INC, f)).read()
            names |= set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src))
    return names


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert {"moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_forward"} <= names
    for n in names:
        assert hasattr(lib, n), n
    # and the binding knows every declared signature
    assert names <= set(_lib.SIGNATURES) | {n for n in names if n.startswith("moe_testing_")}


def test_capacity(lib):
    assert lib.moe_capacity(64, 2, 4, 1.25) == 40
    assert lib.moe_capacity(4096, 2, 8, 1.25) == 1280
    assert lib.moe_capacity(16384, 2, 8, 4.0) == 16384
    assert lib.moe_capacity(32768, 1, 64, 1.0) == 512
    assert lib.moe_capacity(128, 6, 64, 2.0) == 24
    assert lib.moe_capacity(8, 1, 4, 1.0) == 2
    assert lib.moe_capacity(10, 1, 3, 1.0) == 4   # ceil(10/3)
    assert lib.moe_capacity(0, 1, 3, 1.0) == 0
    for bad in [(-1, 1, 4, 1.0), (8, 0, 4, 1.0), (8, 1, 0, 1.0), (8, 1, 4, 0.0), (8, 1, 4, float("nan")),
                (8, 1, 4, float("inf")), (1 << 40, 16, 1, 1.0)]:
        assert lib.moe_capacity(*bad) == -1, bad


def _shape(**kw):
    base = dict(T=64, d=64, E=4, k=2, d_ff=64, dtype=1, act=0)
    base.update(kw)
    return MoeShape(**base)


def _ws(lib, shape, C):
    n = ctypes.c_size_t(0)
    st = lib.moe_workspace_size(ctypes.byref(shape), C, ctypes.byref(n))
    return st, n.value


def test_workspace_size_and_shape_validation(lib):
    st, n = _ws(lib, _shape(), 40)
    assert st == OK and n > 0 and n % 256 == 0
    # grows with capacity-bounded rows
    assert _ws(lib, _shape(), 80)[1] >= n
    assert lib.moe_max_rows(ctypes.byref(_shape()), 40) == 128
    assert lib.moe_max_rows(ctypes.byref(_shape()), 10) == 40
    for kw, want in [(dict(T=-1), INVALID), (dict(d=0), INVALID), (dict(E=0), INVALID), (dict(k=0), INVALID),
                     (dict(k=5), INVALID), (dict(d_ff=0), INVALID), (dict(dtype=7), INVALID), (dict(act=9), INVALID),
                     (dict(E=129, k=2), UNSUPPORTED), (dict(E=32, k=17), UNSUPPORTED),
                     (dict(d=96), UNSUPPORTED), (dict(d_ff=100), UNSUPPORTED), (dict(dtype=0, d=30), UNSUPPORTED),
                     (dict(T=1 << 30, k=2), UNSUPPORTED)]:
        assert _ws(lib, _shape(**kw), 40)[0] == want, kw
    assert lib.moe_workspace_size(ctypes.byref(_shape()), -1, ctypes.byref(ctypes.c_size_t())) == INVALID
    assert lib.moe_workspace_size(None, 4, ctypes.byref(ctypes.c_size_t())) == INVALID


P = ctypes.c_void_p

# The calls below pass fake device pointers that validation must reject before
# any launch.  They only run where no GPU is visible, so a validation bug can
# never turn into a kernel reading a bogus address.
no_gpu = pytest.mark.skipif(torch.cuda.is_available(), reason="fake-pointer checks run on CPU-only hosts")


@no_gpu
def test_route_argument_errors(lib):
    s = _shape()
    f = P(FAKE)
    # missing W_g / idx / w
    assert lib.moe_route(ctypes.byref(s), f, None, None, None, None, f, f, None, None, None) == INVALID
    assert lib.moe_route(ctypes.byref(s), f, f, None, None, None, None, f, None, None, None) == INVALID
    # noise needs both W_noise and eps
    assert lib.moe_route(ctypes.byref(s), f, f, None, f, None, f, f, None, None, None) == INVALID
    assert lib.moe_route(ctypes.byref(s), f, f, None, None, f, f, f, None, None, None) == INVALID
    # misaligned tokens
    assert lib.moe_route(ctypes.byref(s), P(FAKE + 2), f, None, None, None, f, f, None, None, None) == UNSUPPORTED


@no_gpu
def test_dispatch_ffn_combine_argument_errors(lib):
    s = _shape()
    f = P(FAKE)
    st, n = _ws(lib, s, 40)
    # dispatch: null outputs, negative C, small / misaligned workspace
    assert lib.moe_dispatch(ctypes.byref(s), 40, f, f, f, None, f, f, f, None, f, n, None) == INVALID
    assert lib.moe_dispatch(ctypes.byref(s), -2, f, f, f, f, f, f, f, None, f, n, None) == INVALID
    assert lib.moe_dispatch(ctypes.byref(s), 40, f, f, f, f, f, f, f, None, f, n - 1, None) == WORKSPACE
    assert lib.moe_dispatch(ctypes.byref(s), 40, f, f, f, f, f, f, f, None, P(FAKE + 16), n, None) == WORKSPACE
    assert lib.moe_dispatch(ctypes.byref(s), 40, f, f, f, f, f, f, f, None, None, n, None) == WORKSPACE
    # expert ffn: GELU takes no W3; SwiGLU needs W3 and no b1
    sg = _shape(act=1)
    assert lib.moe_expert_ffn(ctypes.byref(s), 40, f, f, f, f, f, None, None, f, f, n, None) == INVALID
    assert lib.moe_expert_ffn(ctypes.byref(sg), 40, f, f, f, None, f, None, None, f, f, n, None) == INVALID
    assert lib.moe_expert_ffn(ctypes.byref(sg), 40, f, f, f, f, f, f, None, f, f, n, None) == INVALID
    assert lib.moe_expert_ffn(ctypes.byref(s), 40, f, f, P(FAKE + 8), None, f, None, None, f, f, n, None) == UNSUPPORTED
    # combine: missing pieces
    assert lib.moe_combine(ctypes.byref(s), 40, f, None, f, f, f, None, None, f, None, None) == INVALID
    assert lib.moe_combine(ctypes.byref(s), 40, None, f, f, f, f, None, None, f, None, None) == INVALID


@no_gpu
def test_forward_argument_errors(lib):
    s = _shape()
    f = P(FAKE)
    st, n = _ws(lib, s, 40)
    args = [f, f, None, None, None, f, None, f, None, None, None, f, None, None, None, None, None, None, None, None,
            None]
    # bad capacity factor with no override
    assert lib.moe_forward(ctypes.byref(s), 0.0, -1, *args, f, n, None) == INVALID
    # a workspace sized for C=10 (40 grouped rows) is too small for cf=1.25 (C=40, 128 rows)
    st, n10 = _ws(lib, s, 10)
    assert n10 < n
    assert lib.moe_forward(ctypes.byref(s), 1.25, -1, *args, f, n10, None) == WORKSPACE
    assert lib.moe_forward(ctypes.byref(s), 1.0, 40, *args, f, n10, None) == WORKSPACE
    # missing output
    bad = list(args)
    bad[11] = None
    assert lib.moe_forward(ctypes.byref(s), 1.25, -1, *bad, f, n, None) == INVALID


def test_status_strings(lib):
    for code, name in _lib.STATUS_NAMES.items():
        assert lib.moe_status_string(code).decode().startswith(name)
    assert b"unknown" in lib.moe_status_string(99)


@no_gpu
def test_routing_stats_argument_errors(lib):
    s = _shape()
    f = P(FAKE)
    st, n = _ws(lib, s, 0)
    # missing outputs or inputs
    assert lib.moe_routing_stats(ctypes.byref(s), f, f, f, f, None, f, f, f, n, None) == INVALID
    assert lib.moe_routing_stats(ctypes.byref(s), f, f, f, f, f, f, None, f, n, None) == INVALID
    assert lib.moe_routing_stats(ctypes.byref(s), None, f, f, f, f, f, f, f, n, None) == INVALID
    assert lib.moe_routing_stats(ctypes.byref(s), f, f, None, f, f, f, f, f, n, None) == INVALID
    # a bad shape
    assert lib.moe_routing_stats(ctypes.byref(_shape(k=5)), f, f, f, f, f, f, f, f, n, None) == INVALID
    # a workspace that is missing, misaligned or too small
    assert lib.moe_routing_stats(ctypes.byref(s), f, f, f, f, f, f, f, None, n, None) == WORKSPACE
    assert lib.moe_routing_stats(ctypes.byref(s), f, f, f, f, f, f, f, P(FAKE + 16), n, None) == WORKSPACE
    assert lib.moe_routing_stats(ctypes.byref(s), f, f, f, f, f, f, f, f, n - 256, None) == WORKSPACE


@no_gpu
def test_shared_expert_argument_errors(lib):
    from sparse_mixture_experts_51_b300._lib import MoeShared
    f = P(FAKE)
    s0 = _shape()                      # no shared experts
    s = _shape(d_ff_shared=128)        # GELU layer with a shared FFN of width 128
    sg = _shape(act=1, d_ff_shared=128)
    st, n = _ws(lib, s, 0)
    assert st == OK and n > _ws(lib, s0, 0)[1]  # the shared activations live in the workspace
    gelu_w = MoeShared(W1s=FAKE, W3s=None, W2s=FAKE, b1s=None, b2s=None)
    swiglu_no_w3 = MoeShared(W1s=FAKE, W3s=None, W2s=FAKE, b1s=None, b2s=None)
    gelu_with_w3 = MoeShared(W1s=FAKE, W3s=FAKE, W2s=FAKE, b1s=None, b2s=None)
    addr = ctypes.addressof
    # moe_shared_ffn: no shared width, missing weights, wrong W3 / b1 for the activation
    assert lib.moe_shared_ffn(ctypes.byref(s0), f, addr(gelu_w), f, f, n, None) == INVALID
    assert lib.moe_shared_ffn(ctypes.byref(s), f, None, f, f, n, None) == INVALID
    assert lib.moe_shared_ffn(ctypes.byref(sg), f, addr(swiglu_no_w3), f, f, n, None) == INVALID
    assert lib.moe_shared_ffn(ctypes.byref(s), f, addr(gelu_with_w3), f, f, n, None) == INVALID
    assert lib.moe_shared_ffn(ctypes.byref(s), f, addr(gelu_w), None, f, n, None) == INVALID
    # a workspace sized without the shared activations is too small
    assert lib.moe_shared_ffn(ctypes.byref(s), f, addr(gelu_w), f, f, _ws(lib, s0, 0)[1], None) == WORKSPACE
    # shape checks: negative or (bf16) non-multiple-of-64 shared width
    assert _ws(lib, _shape(d_ff_shared=-64), 40)[0] == INVALID
    assert _ws(lib, _shape(d_ff_shared=100), 40)[0] == UNSUPPORTED
    # moe_forward: shared weights required iff d_ff_shared > 0
    st, nf = _ws(lib, s, 40)
    args = [f, f, None, None, None, f, None, f, None, None, None, f, None, None, None, None, None, None, None, None,
            None]
    assert lib.moe_forward(ctypes.byref(s), 1.25, -1, *args, f, nf, None) == INVALID
    bad = list(args)
    bad[10] = addr(gelu_w)
    assert lib.moe_forward(ctypes.byref(s0), 1.25, -1, *bad, f, nf, None) == INVALID


@no_gpu
def test_expert_choice_argument_errors(lib):
    f = P(FAKE)
    tc = _shape()                      # token choice, T=64, E=4, k=2
    ec = _shape(routing=1)
    assert lib.moe_max_rows(ctypes.byref(ec), 40) == 4 * 40
    assert lib.moe_max_rows(ctypes.byref(ec), 100) == 4 * 64   # C' = min(C, T)
    assert _ws(lib, _shape(routing=7), 40)[0] == INVALID
    assert _ws(lib, _shape(routing=1, T=1 << 27, E=32, k=1), 40)[0] == UNSUPPORTED  # T*E >= 2^31
    st, n = _ws(lib, ec, 40)
    assert st == OK
    # expert choice keeps [T,E] tables the token-choice layer does not (a batch above 128 tokens,
    # where the token-choice layer has no fused decode FFN rows either)
    assert _ws(lib, _shape(T=300, routing=1), 40)[1] > _ws(lib, _shape(T=300), 40)[1]
    # the expert-choice route needs an expert-choice shape, its outputs and a workspace
    assert lib.moe_route_expert_choice(ctypes.byref(tc), 40, f, f, None, None, None, f, f, None, None, f, n,
                                       None) == INVALID
    assert lib.moe_route_expert_choice(ctypes.byref(ec), 40, f, f, None, None, None, None, f, None, None, f, n,
                                       None) == INVALID
    assert lib.moe_route_expert_choice(ctypes.byref(ec), 40, f, f, None, f, None, f, f, None, None, f, n,
                                       None) == INVALID  # W_noise without eps
    assert lib.moe_route_expert_choice(ctypes.byref(ec), 40, f, f, None, None, None, f, f, None, None, f,
                                       n - 256, None) == WORKSPACE
    # token-choice steps refuse an expert-choice shape
    assert lib.moe_dispatch(ctypes.byref(ec), 40, f, f, f, f, f, f, f, None, f, n, None) == INVALID
    assert lib.moe_combine(ctypes.byref(ec), 40, f, f, f, f, f, None, None, f, None, None) == INVALID
    # the forward takes no token-choice tables with expert choice
    args = [f, f, None, None, None, f, None, f, None, None, None, f, None, f, None, None, None, None, None, None,
            None]
    assert lib.moe_forward(ctypes.byref(ec), 1.25, -1, *args, f, n, None) == INVALID


@no_gpu
def test_overflow_and_gate_option_errors(lib):
    f = P(FAKE)
    assert _ws(lib, _shape(gates=2), 40)[0] == INVALID
    assert _ws(lib, _shape(overflow=2), 40)[0] == INVALID
    assert _ws(lib, _shape(routing=1, gates=1), 40)[0] == INVALID      # expert choice: gates are p by definition
    assert _ws(lib, _shape(routing=1, overflow=1), 40)[0] == INVALID   # expert choice: nothing overflows
    rr = _shape(overflow=1)
    st, n = _ws(lib, rr, 40)
    assert st == OK and n > _ws(lib, _shape(), 40)[1]  # room for the second dispatch pass
    # re-routing runs only inside moe_forward
    assert lib.moe_dispatch(ctypes.byref(rr), 40, f, f, f, f, f, f, f, None, f, n, None) == INVALID
    assert lib.moe_dispatch_noalloc(ctypes.byref(rr), 40, f, f, f, f, f, f, f, None, None, None) == INVALID


@no_gpu
def test_decode_sized_workspace_holds_the_fused_ffn_rows(lib):
    """A bf16 token-choice batch of at most 128 tokens with T*k >= 4E runs its
    expert FFN densely over every (expert, token): its workspace holds E*128
    hidden rows of d_ff bf16 values more than the grouped layout needs."""
    small = _shape(T=128, E=4, k=2, d_ff=128)      # 256 assignments >= 16: fused
    sparse = _shape(T=128, E=64, k=1, d_ff=128)    # 128 assignments < 256: grouped
    grouped = _shape(T=129, E=4, k=2, d_ff=128)    # above one 128-row tile: grouped
    f32 = _shape(T=128, E=4, k=2, d_ff=128, dtype=0)
    n_small = _ws(lib, small, 64)[1]
    assert n_small - _ws(lib, f32, 64)[1] >= 4 * 128 * 128 * 2 - 2 * (128 * 64 * 2 + 128 * 128 * 2)
    assert n_small > _ws(lib, grouped, 64)[1] - 16 * 1024
    assert _ws(lib, sparse, 64)[1] < 64 * 128 * 128 * 2

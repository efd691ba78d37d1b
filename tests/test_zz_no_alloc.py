"""moe_dispatch_noalloc: the dispatch entry point for callers that cannot
allocate device memory (a plug-in that is handed only its inputs and
outputs, or a serving loop with a fixed memory plan where cudaMalloc is not
allowed).  It keeps its scan state in a fixed array inside the library
instead of a caller workspace; its results must equal moe_dispatch's.

This file is collected last on purpose, and must pass both alone in a fresh
process (the first call sets up the array's device address) and after the
other GPU tests; test_noalloc_in_a_fresh_process runs the rest of the file
in a new Python process to check the first."""
import ctypes
import os
import subprocess
import sys

import pytest
import torch

from sparse_mixture_experts_51_b300 import _lib, api

pytestmark = pytest.mark.gpu

MAX_ASSIGNMENTS = 1 << 20


def _P(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _inputs(T, d, E, k, seed, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    # a skewed top-k table (distinct experts per token) so some experts overflow
    logits = torch.randn(T, E, generator=g) + torch.linspace(2.0, -2.0, E)
    idx = logits.topk(k, dim=1).indices.int().cuda()
    x = torch.randn(T, d, generator=g).to(dtype).cuda()
    return idx, x


def _noalloc(shape, C, idx, x):
    T, k, E, d = shape.T, shape.k, shape.E, shape.d
    R = api.max_rows(shape, C)
    dev = "cuda"
    out = dict(pos=torch.full((T, k), -7, dtype=torch.int32, device=dev),
               counts=torch.full((E,), -7, dtype=torch.int32, device=dev),
               offsets=torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
               dropped=torch.full((1,), -7, dtype=torch.int64, device=dev),
               x_perm=torch.zeros(max(R, 1), d, dtype=x.dtype, device=dev),
               row_token=torch.full((max(R, 1),), -1, dtype=torch.int32, device=dev),
               err=torch.full((1,), 123, dtype=torch.int32, device=dev))
    st = _lib.load().moe_dispatch_noalloc(
        ctypes.byref(shape), C, _P(idx), _P(x), _P(out["pos"]), _P(out["counts"]), _P(out["offsets"]),
        _P(out["dropped"]), _P(out["x_perm"]), _P(out["row_token"]), _P(out["err"]),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, _lib.STATUS_NAMES.get(st, st)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("T,d,E,k,cf", [(3000, 128, 16, 2, 0.8), (2600, 64, 8, 1, 1.0),
                                         (MAX_ASSIGNMENTS // 2, 64, 8, 2, 0.9)],
                         ids=["tiled_then_tiled", "tiled_then_one_cta", "256_large_tiles"])
def test_noalloc_dispatch_matches_workspace_dispatch_twice(T, d, E, k, cf):
    """Two calls in a row (different batches, so the second starts from the
    first call's leftover scratch) each equal the workspace entry point.  The
    cases cover the tiled look-back kernel (more than 2048 assignments) with
    1024-assignment tiles, the one-CTA kernel, and the largest size the fixed
    array holds: 2^20 assignments in 256 tiles of 4096."""
    for call, seed in enumerate((101, 202)):
        Tc = T if call == 0 else T // 2 + 1
        idx, x = _inputs(Tc, d, E, k, seed)
        C = api.capacity(Tc, k, E, cf)
        shape = api.shape_of(Tc, d, E, k, 64, x.dtype, "gelu")
        ref = api.dispatch(idx, x, E, C, want_row_token=True)
        got = _noalloc(shape, C, idx, x)
        R = int(ref["offsets"][-1].item())
        assert int(got["err"].item()) == 0
        for key in ("pos", "counts", "offsets", "dropped"):
            assert torch.equal(got[key], ref[key]), (call, key)
        assert torch.equal(got["x_perm"][:R], ref["x_perm"][:R]), call
        assert torch.equal(got["row_token"][:R], ref["row_token"][:R]), call
        assert int(ref["dropped"].item()) > 0  # the cases really overflow


def test_noalloc_rejects_sizes_beyond_its_array():
    """More than 2^20 assignments do not fit the fixed array: rejected before any work."""
    idx, x = _inputs(8, 64, 4, 2, 7)
    T = MAX_ASSIGNMENTS // 2 + 1  # T*k = 2^20 + 2 with k = 2
    shape = api.shape_of(T, 64, 4, 2, 64, torch.bfloat16, "gelu")
    st = _lib.load().moe_dispatch_noalloc(ctypes.byref(shape), 10, _P(idx), _P(x), _P(idx), _P(idx), _P(idx),
                                          _P(idx), _P(x), None, None, None)
    assert st == 2  # MOE_ERR_UNSUPPORTED


def test_noalloc_rejects_what_the_workspace_dispatch_rejects():
    """Shapes and pointers that moe_dispatch refuses are refused here too,
    before anything is enqueued: a bf16 width that is not a multiple of 64
    and a token matrix that is not 16-byte aligned."""
    idx, x = _inputs(64, 64, 4, 2, 8)
    lib = _lib.load()
    buf = torch.zeros(4096, dtype=torch.int32, device="cuda")
    bad_d = api.shape_of(64, 33, 4, 2, 64, torch.bfloat16, "gelu")
    st = lib.moe_dispatch_noalloc(ctypes.byref(bad_d), 40, _P(idx), _P(x), _P(buf), _P(buf), _P(buf), _P(buf),
                                  _P(buf), None, None, None)
    assert st == 2  # MOE_ERR_UNSUPPORTED
    shape = api.shape_of(63, 64, 4, 2, 64, torch.bfloat16, "gelu")
    x_odd = x.view(-1)[1:63 * 64 + 1]  # starts 2 bytes past an aligned address
    st = lib.moe_dispatch_noalloc(ctypes.byref(shape), 40, _P(idx), ctypes.c_void_p(x_odd.data_ptr()), _P(buf),
                                  _P(buf), _P(buf), _P(buf), _P(buf), None, None, None)
    assert st == 2
    ws = api.new_workspace(shape, 40)
    st = lib.moe_dispatch(ctypes.byref(shape), 40, _P(idx), ctypes.c_void_p(x_odd.data_ptr()), _P(buf), _P(buf),
                          _P(buf), _P(buf), _P(buf), None, _P(ws), ws.numel(), None)
    assert st == 2


def test_noalloc_in_a_fresh_process():
    """The other tests of this file, alone in a new process: the first call
    there finds the array's address itself."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-m", "gpu", "-p", "no:cacheprovider",
                        "-k", "not fresh_process", os.path.abspath(__file__)],
                       cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]

"""End-to-end parity of the CUDA path (through the C ABI) with the fp64 oracle.

Bar: top-k indices, slots, counts, offsets and drop count bit-exact; gates
within 1e-6 (fp32) / 1e-4 (bf16) absolute; layer output and the weighted
expert sum within relative L2 1e-5 (fp32 layers) / 1e-2 (bf16 layers)."""
import math

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from sparse_mixture_experts_51_b300 import api
from sparse_mixture_experts_51_b300 import workloads as W

from _parity import check_layer, edge_tokens, gpu_forward, oracle_forward, rel_l2, to_gpu

pytestmark = pytest.mark.gpu


def _run_full(w, C=None):
    inp = W.make_inputs(w)
    gpu = gpu_forward(w, to_gpu(inp), C=C)
    ref = oracle_forward(w, inp, C=C)
    check_layer(w, inp, gpu, ref)
    return inp, gpu, ref


def test_tiny_fp32_layer():
    """The tiny fp32 layer (T=64, d=32, E=4, top-2, GELU, C=40), whole batch."""
    _run_full(W.WORKLOADS["tiny_fp32"])


SMALL = [
    # several M tiles per expert with a ragged tail, SwiGLU, some drops
    W.Workload("swiglu_ragged", T=333, d=256, E=8, k=2, F=512, act=W.ACT_SWIGLU, capacity_factor=1.0,
               dtype=torch.bfloat16, seed=11),
    # GELU with the N tile wider than F on the last tile (F=320 = 256 + 64)
    W.Workload("gelu_ragged_n", T=517, d=192, E=6, k=2, F=320, act=W.ACT_GELU, capacity_factor=1.1,
               dtype=torch.bfloat16, seed=12),
    # Switch-style noisy top-1 with a Zipf-skewed bias and heavy drops
    W.Workload("noisy_top1", T=700, d=128, E=16, k=1, F=256, act=W.ACT_GELU, capacity_factor=1.0,
               dtype=torch.bfloat16, seed=13, noisy=True, zipf_bias=True),
    # fine-grained: many experts, top-6
    W.Workload("fine_grained", T=77, d=512, E=64, k=6, F=1408, act=W.ACT_SWIGLU, capacity_factor=2.0,
               dtype=torch.bfloat16, seed=14),
    # more than one dispatch tile (T*k > 4096) with drops
    W.Workload("multi_tile_dispatch", T=2500, d=128, E=8, k=2, F=128, act=W.ACT_SWIGLU, capacity_factor=0.9,
               dtype=torch.bfloat16, seed=15),
    # GELU with 256-row CTA tiles (more than four M tiles per expert), a ragged
    # last M tile and an N tile wider than F
    W.Workload("gelu_wide_m_tiles", T=3000, d=256, E=4, k=2, F=320, act=W.ACT_GELU, capacity_factor=1.0,
               dtype=torch.bfloat16, seed=17),
    # fp32 layer with nonzero-bias experts and noise
    W.Workload("fp32_noisy", T=150, d=48, E=5, k=2, F=40, act=W.ACT_GELU, capacity_factor=1.0,
               dtype=torch.float32, seed=16, noisy=True, zipf_bias=True, expert_bias=True),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_small_layers(w):
    _run_full(w)


def test_expert_biases_nonzero():
    """GELU experts with nonzero b1/b2 (bf16 path): the epilogue adds both biases."""
    w = W.Workload("gelu_bias", T=260, d=128, E=4, k=2, F=192, act=W.ACT_GELU, capacity_factor=1.5,
                   dtype=torch.bfloat16, seed=21)
    inp = W.make_inputs(w)
    g = torch.Generator().manual_seed(99)
    inp["b1"] = torch.randn(w.E, w.F, generator=g) * 0.5
    inp["b2"] = torch.randn(w.E, w.d, generator=g) * 0.5
    gpu = gpu_forward(w, to_gpu(inp))
    ref = oracle_forward(w, inp)
    check_layer(w, inp, gpu, ref)


def test_k_equals_E_no_drop():
    w = W.Workload("dense_mixture", T=100, d=64, E=4, k=4, F=128, act=W.ACT_SWIGLU, capacity_factor=1.0,
                   dtype=torch.bfloat16, seed=22)
    _, gpu, ref = _run_full(w, C=100)
    assert int(gpu["dropped"][0]) == 0


def test_zero_capacity_passes_tokens_through():
    w = W.Workload("all_dropped", T=64, d=64, E=4, k=2, F=64, act=W.ACT_GELU, capacity_factor=1.0,
                   dtype=torch.bfloat16, seed=23)
    inp, gpu, ref = _run_full(w, C=0)
    assert int(gpu["dropped"][0]) == 64 * 2
    assert torch.equal(gpu["out"], inp["x"])


def test_empty_batch():
    w = W.Workload("empty", T=0, d=64, E=4, k=2, F=64, act=W.ACT_GELU, capacity_factor=1.0,
                   dtype=torch.bfloat16, seed=24)
    inp = W.make_inputs(w)
    gpu = gpu_forward(w, to_gpu(inp), C=3)
    assert gpu["out"].shape == (0, 64)
    assert gpu["counts"].tolist() == [0] * 4 and gpu["offsets"].tolist() == [0] * 5
    assert int(gpu["dropped"][0]) == 0


def test_exact_ties_go_to_lower_expert():
    """Integer-valued tokens and duplicated router columns give exactly equal
    logits; the lower expert index must win, as in the oracle."""
    T, d, E, k = 96, 64, 8, 2
    g = torch.Generator().manual_seed(5)
    x = torch.randint(-2, 3, (T, d), generator=g).to(torch.bfloat16)
    Wg = torch.randint(-2, 3, (d, E), generator=g).float()
    Wg[:, 3] = Wg[:, 1]
    Wg[:, 6] = Wg[:, 1]
    Wg[:, 5] = Wg[:, 2]
    w = W.Workload("ties", T=T, d=d, E=E, k=k, F=64, act=W.ACT_GELU, capacity_factor=2.0,
                   dtype=torch.bfloat16, seed=25)
    inp = W.make_inputs(w)
    inp["x"], inp["W_g"] = x, Wg
    gpu = gpu_forward(w, to_gpu(inp))
    ref = oracle_forward(w, inp)
    H = ref["H"]
    assert (H[:, 1] == H[:, 3]).all()
    check_layer(w, inp, gpu, ref)
    # at least some tokens really had a tie inside their top k+1
    s = -np.sort(-H, axis=1)
    assert ((s[:, :k] - s[:, 1:k + 1]) == 0).any()
    # these ties are settled by the fp64 re-evaluation
    assert int(gpu["stats"][0]) > 0


def test_full_size_bf16_t4096():
    """The bf16 T=4096, d=1024, E=8 top-2 SwiGLU layer, whole batch (bench workload)."""
    _run_full(W.WORKLOADS["bf16_t4096"])


def test_full_size_decode_t128():
    """The decode-like T=128, d=2048, E=64 top-6 SwiGLU layer, whole batch."""
    _run_full(W.WORKLOADS["decode_t128"])


def _sampled(w, n_sample=48):
    """Routing, slots and drops for every token; outputs on a token sample
    that holds, besides random tokens and the first and last eight, every
    token with an assignment on an edge row of its expert's segment (first
    and last rows, the rows of partial M tiles): the rows the expert GEMMs
    store by their edge paths."""
    inp = W.make_inputs(w)
    gpu = gpu_forward(w, to_gpu(inp))
    rng = np.random.default_rng(w.seed)
    edges = edge_tokens(gpu["idx"].numpy(), gpu["pos"].numpy(), gpu["offsets"].numpy())
    toks = sorted(set(list(range(8)) + list(range(w.T - 8, w.T)) + rng.choice(w.T, n_sample, replace=False).tolist()
                      + edges))
    ref = oracle_forward(w, inp, tokens=toks)
    check_layer(w, inp, gpu, ref, tokens=toks)
    return inp, gpu, ref


def test_full_size_mixtral_sampled():
    """Mixtral-shaped T=16384, d=4096, F=14336 no-drop layer: routing, slots and
    drops for every token, outputs on a sample of tokens."""
    _, gpu, ref = _sampled(W.WORKLOADS["mixtral_t16384"], n_sample=24)
    assert ref["dropped"] == 0 and int(gpu["counts"].sum()) == 16384 * 2


def test_full_size_switch_top1_sampled():
    """Switch-style top-1 with forced overflow (T=32768, E=64, C=512, noisy, Zipf bias)."""
    inp, gpu, ref = _sampled(W.WORKLOADS["switch_top1"], n_sample=64)
    assert ref["dropped"] > 0
    assert (gpu["w"] == 1.0).all()


def test_determinism():
    w = SMALL[0]
    g = to_gpu(W.make_inputs(w))
    a = gpu_forward(w, g)
    b = gpu_forward(w, g)
    for key in ("out", "moe", "idx", "w", "pos", "counts", "offsets", "dropped"):
        assert torch.equal(a[key], b[key]), key


def test_cuda_graph_replay_matches_eager():
    """MoELayer.capture: a CUDA-graph replay of the forward gives the eager
    output bit for bit, also after new tokens are copied into the input."""
    w = SMALL[0]
    inp = W.make_inputs(w)
    g = to_gpu(inp)
    layer = api.MoELayer(g["W_g"], g["W1"], g["W2"], w.k, "swiglu", W3=g["W3"], capacity_factor=w.capacity_factor,
                         keep_routing=False)
    x = g["x"].clone()
    cap = layer.capture(x)
    eager = layer(x)
    torch.cuda.synchronize()
    assert torch.equal(cap.replay(), eager)
    x2 = torch.randn(x.shape, generator=torch.Generator().manual_seed(77)).to(x.dtype).cuda()
    x.copy_(x2)
    out2 = cap.replay().clone()
    torch.cuda.synchronize()
    assert torch.equal(out2, layer(x2))


def test_forward_timed_stage_events():
    """moe_forward_timed writes what moe_forward writes, and its six stage
    events (some NULL) record in order, eagerly and inside a CUDA graph."""
    import ctypes

    from sparse_mixture_experts_51_b300 import _lib

    w = W.WORKLOADS["bf16_t4096"].scaled(1024)
    inp = W.make_inputs(w)
    g = to_gpu(inp)
    C = api.capacity(w.T, w.k, w.E, w.capacity_factor)
    shape = api.shape_of(w.T, w.d, w.E, w.k, w.F, w.dtype, "swiglu")
    ws = api.new_workspace(shape, C, "cuda")
    lib = _lib.load()
    P = api._ptr

    def run(fn, out, *extra):
        s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        args = [ctypes.byref(shape), float(w.capacity_factor), -1, P(g["x"]), P(g["W_g"]), None, None, None,
                P(g["W1"]), P(g["W3"]), P(g["W2"]), None, None, None, P(out)] + [None] * 9 + [P(ws), ws.numel(), s]
        _lib.check(fn(*args, *extra), fn.__name__)

    ref = torch.empty(w.T, w.d, dtype=w.dtype, device="cuda")
    run(lib.moe_forward, ref)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for e in evs:
        e.record()
    torch.cuda.synchronize()
    arr = (ctypes.c_void_p * 6)(*[e.cuda_event if i != 4 else None for i, e in enumerate(evs)])
    out = torch.empty_like(ref)
    run(lib.moe_forward_timed, out, arr)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    spans = [evs[i].elapsed_time(evs[j]) for i, j in [(0, 1), (1, 2), (2, 3), (3, 5)]]
    assert all(sp >= 0 for sp in spans) and evs[0].elapsed_time(evs[5]) > 0
    # the same call captured into a graph: its events become external nodes that time every replay
    out2 = torch.zeros_like(ref)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run(lib.moe_forward_timed, out2, arr)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out2, ref)
    assert evs[0].elapsed_time(evs[5]) > 0
    assert api.get_device_error(ws) == 0


def test_kernel_launch_counter():
    """moe_kernel_launches counts the kernels a call enqueues: six for a bf16
    layer with the warp router (router, dispatch, gather, two expert GEMMs,
    combine); replaying a captured call enqueues nothing new."""
    from sparse_mixture_experts_51_b300 import _lib

    lib = _lib.load()
    w = W.WORKLOADS["bf16_t4096"].scaled(1024)
    g = to_gpu(W.make_inputs(w))
    layer = api.MoELayer(g["W_g"], g["W1"], g["W2"], w.k, "swiglu", W3=g["W3"], capacity_factor=w.capacity_factor)
    layer(g["x"])
    torch.cuda.synchronize()
    n0 = lib.moe_kernel_launches()
    layer(g["x"])
    assert lib.moe_kernel_launches() - n0 == 6
    cap = layer.capture(g["x"])
    n1 = lib.moe_kernel_launches()
    for _ in range(3):
        cap.replay()
    torch.cuda.synchronize()
    assert lib.moe_kernel_launches() == n1

"""Plain, slow fp64 CPU oracle for the forward pass of one sparse MoE layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code, table, constant
or helper with the CUDA library; both sides take their inputs from the
seeded generator in ``sparse_mixture_experts_51_b300.workloads``, which holds
none of the method's arithmetic.

Everything is evaluated in float64 from the values stored in the input
arrays (bf16 values widened exactly).  Each function names the passage of
the source pages it restates.  The pages are cited by title and section:

  [P1] "Mixture-of-Experts Sparse Model Scaling" (glossary page), sections
       "Mathematical Formulation", "Advanced Theory & Extensions", and the
       "Practical Labs" appendix (Lab 1 top-k router, Lab 2 load-balancing
       loss, Lab 3 capacity).
  [P2] "Mixture-of-experts Models" (book chapter), Level 2 "Router scores
       become a sparse dispatch decision", "Top-k selection has ties",
       "Capacity limits make dispatch observable" (Figure 44.4); Level 3
       "Load balancing has probability, assignment, and quality diagnostics".
  [P3] "Scaling Capacity via Sparse Mixture of Experts (MoE) Architectures",
       the SimpleRouter listing.
  [P4] "LLM part 09: Sparse Mixture-of-Experts (MoE)", section 1 (output
       equation), section 2 (noisy top-k gating), section 3 (capacity),
       section 4 (auxiliary load-balancing loss).
  [P5] "3D mixture-of-experts routing lab", the "Capacity" card.

Readings taken where the pages are silent or disagree:
  * gates are renormalised over the selected experts ([P1] Lab 1, [P2]
    Level 2, [P3] SimpleRouter, [P4] s2 all do so; [P1]'s displayed
    equation does not, and is the minority reading);
  * ties in the top-k order go to the lower expert index;
  * capacity C = ceil(cf * T * k / E) in float64 ([P5] capacity card);
  * dispatch priority is rank-major: every token's first choice, in token
    order, before any second choice; an assignment is kept iff fewer than C
    earlier assignments went to the same expert ([P1] Lab 3 generalised);
  * a dropped assignment contributes nothing; the gates of the survivors
    are NOT renormalised again; the residual carries the token
    ([P1] "Advanced Theory", [P4] s3);
  * GELU is the exact erf form; SwiGLU is silu(x W1^T) * (x W3^T); the
    noise branch has no bias; softplus(z) = max(z,0) + log1p(exp(-|z|));
    SwiGLU experts take no b1 (b2 is optional for both forms).
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np

try:
    from scipy.special import erf as _erf
except ImportError:  # pragma: no cover - scipy is present in the image
    _erf = np.vectorize(math.erf, otypes=[np.float64])

GELU = 0
SWIGLU = 1


# --------------------------------------------------------------------------
# routing
# --------------------------------------------------------------------------

def softplus(z: np.ndarray) -> np.ndarray:
    """softplus(z) = ln(1 + e^z), written in the overflow-free form."""
    z = np.asarray(z, dtype=np.float64)
    return np.maximum(z, 0.0) + np.log1p(np.exp(-np.abs(z)))


def logits(x, W_g, b_g=None, W_noise=None, eps=None) -> np.ndarray:
    """Router logits H[t,e] ([P4] s2 noisy top-k gating; [P1] "Mathematical
    Formulation": g_i(x) is a linear transform of x; [P3] SimpleRouter's
    nn.Linear carries a bias).

        H = x W_g + b_g + eps * softplus(x W_noise)

    x [T,d], W_g [d,E], b_g [E] or None, W_noise [d,E] or None, eps [T,E] or None.
    The noise term is present only when both W_noise and eps are given.
    """
    x = np.asarray(x, dtype=np.float64)
    H = x @ np.asarray(W_g, dtype=np.float64)
    if b_g is not None:
        H = H + np.asarray(b_g, dtype=np.float64)[None, :]
    if W_noise is not None and eps is not None:
        H = H + np.asarray(eps, dtype=np.float64) * softplus(x @ np.asarray(W_noise, dtype=np.float64))
    return H


def topk(H: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest logits per token, largest first ([P4] s2 TopK;
    [P1] Lab 1 ranks experts by descending probability; softmax is monotone
    so ranking logits ranks probabilities).  Equal logits go to the lower
    expert index: a stable sort of -H keeps index order among equals.
    Returns int64 [T,k].
    """
    H = np.asarray(H, dtype=np.float64)
    order = np.argsort(-H, axis=1, kind="stable")
    return order[:, :k].astype(np.int64)


def gates(H: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Gate weights w[t,r] = softmax over the k selected logits ([P4] s2:
    G = Softmax(TopK(H)); equal to the renormalised top-k probabilities of
    [P1] Lab 1 and [P2] Level 2).  Shifted by the largest selected logit.
    """
    sel = np.take_along_axis(np.asarray(H, dtype=np.float64), idx, axis=1)
    z = np.exp(sel - sel.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


def gates_raw(H: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Un-renormalised gates: w[t,r] = p_i(x) for i = idx[t,r], the full
    softmax over all experts ([P1] "Mathematical Formulation": the layer
    output weights each selected expert by its routing probability)."""
    P = softmax_rows(H)
    return np.take_along_axis(P, np.asarray(idx, dtype=np.int64), axis=1)


def capacity(T: int, k: int, E: int, capacity_factor: float) -> int:
    """Expert capacity C = ceil(factor * tokens * k / experts) ([P5] Capacity
    card; [P4] s3 gives the k=1 form)."""
    return int(math.ceil(float(capacity_factor) * float(T) * float(k) / float(E)))


def dispatch(idx: np.ndarray, E: int, C: int) -> dict:
    """Capacity-limited first-come dispatch ([P1] Lab 3; [P2] "Capacity limits
    make dispatch observable").

    Assignments are visited in priority order: rank 0 of every token in token
    order, then rank 1, and so on.  An assignment takes the next slot of its
    expert while the expert has fewer than C; otherwise it is dropped.

    Returns dict with
      pos     int64 [T,k]  slot within the expert's segment, -1 if dropped
      load    int64 [E]    assignments requested per expert (before the cap)
      counts  int64 [E]    kept assignments per expert = min(load, C)
      offsets int64 [E+1]  exclusive prefix sum of counts (segment starts)
      dropped int          number of dropped assignments
    """
    idx = np.asarray(idx, dtype=np.int64)
    T, k = idx.shape
    load = np.zeros(E, dtype=np.int64)
    pos = np.full((T, k), -1, dtype=np.int64)
    dropped = 0
    for r in range(k):
        for t in range(T):
            e = int(idx[t, r])
            slot = int(load[e])
            load[e] += 1
            if slot < C:
                pos[t, r] = slot
            else:
                dropped += 1
    counts = np.minimum(load, C)
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    return dict(pos=pos, load=load, counts=counts, offsets=offsets, dropped=int(dropped))


def softmax_rows(H: np.ndarray) -> np.ndarray:
    """Router probabilities p[t,e] = softmax over all E experts of H[t]
    ([P2] Level 2: a softmax turns the router scores into weights)."""
    H = np.asarray(H, dtype=np.float64)
    z = np.exp(H - H.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


def expert_choice(H: np.ndarray, C: int) -> dict:
    """Expert-choice routing ([P1] "Advanced Theory & Extensions": each expert
    selects from the batch the top tokens it wants, up to its capacity, so
    every expert is filled; a token may be taken by no expert or by several).

    Readings: expert e ranks the tokens by its router score H[t,e] (the
    logit: [P2] Level 2 calls the router's per-expert outputs scores) and
    takes the min(C, T) highest, equal scores going to the lower token index;
    the gate of a chosen (t, e) is the router probability p[t,e] (softmax
    over all E experts), not renormalised over the experts that chose t.

    Returns sel int64 [E, C'] (chosen tokens of each expert, ascending),
    gates [E, C'] (p of those pairs), chosen bool [T,E], counts [E] (= C'),
    dropped (tokens no expert chose).
    """
    H = np.asarray(H, dtype=np.float64)
    T, E = H.shape
    Cp = min(int(C), T)
    P = softmax_rows(H)
    sel = np.zeros((E, Cp), dtype=np.int64)
    chosen = np.zeros((T, E), dtype=bool)
    for e in range(E):
        # a stable sort of -H keeps lower token indices first among equal scores
        top = np.sort(np.argsort(-H[:, e], kind="stable")[:Cp])
        sel[e] = top
        chosen[top, e] = True
    gates = np.array([[P[t, e] for t in sel[e]] for e in range(E)], dtype=np.float64).reshape(E, Cp)
    counts = np.full(E, Cp, dtype=np.int64)
    dropped = int(T - np.count_nonzero(chosen.any(axis=1)))
    return dict(sel=sel, gates=gates, chosen=chosen, counts=counts, dropped=dropped, P=P)


def reroute(idx: np.ndarray, disp: dict, backup: np.ndarray, C: int) -> dict:
    """Overflow re-routing to a backup expert ([P2] "Capacity limits make
    dispatch observable" and "Overflow handling defines an output contract":
    a full expert's assignment may be sent to a backup, lower-ranked expert;
    [P3]: routed to a secondary expert).

    Readings: a token's backup is its (k+1)-th ranked expert (``backup[t]``,
    -1 when k = E); only the token's first dropped assignment (lowest rank)
    asks for it, since an expert takes a token once; the requests are served
    after the capacity dispatch, first-come in the same priority order (rank
    r, then token t), while the backup has fewer than C assignments; a
    rerouted assignment keeps its gate; the rest stay dropped.

    Returns idx (the expert each assignment is finally sent to), pos, counts,
    offsets, dropped (after re-routing) and rerouted (how many were moved).
    """
    idx = np.array(idx, dtype=np.int64, copy=True)
    pos = np.array(disp["pos"], dtype=np.int64, copy=True)
    T, k = idx.shape
    E = len(disp["counts"])
    load = np.array(disp["counts"], dtype=np.int64, copy=True)
    first = {}
    for t in range(T):
        for r in range(k):
            if pos[t, r] < 0:
                first[t] = r
                break
    rerouted = 0
    for r in range(k):          # priority order: rank, then token
        for t in range(T):
            if first.get(t) != r:
                continue
            e = int(backup[t])
            if e >= 0 and load[e] < C:
                idx[t, r] = e
                pos[t, r] = load[e]
                load[e] += 1
                rerouted += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + load[e]
    dropped = int(np.count_nonzero(pos < 0))
    return dict(idx=idx, pos=pos, counts=load, offsets=offsets, dropped=dropped, rerouted=rerouted)


# --------------------------------------------------------------------------
# experts
# --------------------------------------------------------------------------

def gelu(a: np.ndarray) -> np.ndarray:
    """Exact GELU: a * Phi(a) = a * (1 + erf(a / sqrt 2)) / 2 (erf from scipy)."""
    a = np.asarray(a, dtype=np.float64)
    return a * 0.5 * (1.0 + _erf(a / math.sqrt(2.0)))


def silu(a: np.ndarray) -> np.ndarray:
    """SiLU: a * sigmoid(a)."""
    a = np.asarray(a, dtype=np.float64)
    return a / (1.0 + np.exp(-a))


def expert(xr: np.ndarray, e: int, act: int, W1, W3, W2, b1=None, b2=None) -> np.ndarray:
    """Output of expert e on rows xr [n,d] ([P1] "Core Concepts": each expert
    is a feed-forward network with the architecture of the dense FFN it
    replaces; the GELU and SwiGLU forms are the two the layer supports).

      GELU   : y = gelu(xr W1[e]^T + b1[e]) W2[e]^T + b2[e]
      SwiGLU : y = (silu(xr W1[e]^T) * (xr W3[e]^T)) W2[e]^T (+ b2[e])

    Weights are in nn.Linear layout: W1, W3 [E,F,d], W2 [E,d,F].
    """
    xr = np.asarray(xr, dtype=np.float64)
    w1 = np.asarray(W1[e], dtype=np.float64)
    a = xr @ w1.T
    if act == GELU:
        if b1 is not None:
            a = a + np.asarray(b1[e], dtype=np.float64)[None, :]
        h = gelu(a)
    elif act == SWIGLU:
        w3 = np.asarray(W3[e], dtype=np.float64)
        h = silu(a) * (xr @ w3.T)
    else:
        raise ValueError(f"unknown activation {act}")
    y = h @ np.asarray(W2[e], dtype=np.float64).T
    if b2 is not None:
        y = y + np.asarray(b2[e], dtype=np.float64)[None, :]
    return y


def shared_experts(x, act: int, W1s, W2s, W3s=None, b1s=None, b2s=None, tokens=None) -> np.ndarray:
    """Sum of the shared experts' outputs for each token ([P1] "Advanced
    Theory & Extensions": fine-grained designs add dedicated shared experts
    that every token passes through unconditionally; [P1] "Real-World
    Applications" names DeepSeek-MoE for this design).

    Readings: a shared expert has the routed experts' form (``expert``) and
    enters with weight 1 (the pages give it no gate); S shared experts are
    summed in order s = 0..S-1.
    W1s, W3s [S,F_s,d], W2s [S,d,F_s], b1s [S,F_s], b2s [S,d] (nn.Linear layout).
    Returns [n,d] for the rows in ``tokens`` (all tokens when None).
    """
    x = np.asarray(x, dtype=np.float64)
    toks = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens, dtype=np.int64)
    xs = x[toks]
    y = np.zeros_like(xs)
    for s in range(len(W1s)):
        y = y + expert(xs, s, act, W1s, W3s, W2s, b1s, b2s)
    return y


# --------------------------------------------------------------------------
# whole layer
# --------------------------------------------------------------------------

def combine(x, idx, w, pos, expert_out, residual=True, tokens=None, shared_out=None) -> dict:
    """Weighted combination y = sum_i G(x)_i E_i(x) over the kept assignments
    ([P4] s1; [P1] "Mathematical Formulation"; [P1] Lab 1 accumulates
    weight * expert output per token), plus the residual that carries a
    dropped token through unchanged ([P1] "Advanced Theory"; [P4] s3).

    expert_out[(t, r)] holds E_{idx[t,r]}(x_t) for every kept (t, r) of the
    tokens evaluated.  Ranks are summed in order 0..k-1; ``shared_out`` [n,d]
    (the shared experts' sum for the same rows, or None) is added after them.
    Returns moe [n,d] (everything the experts add) and out = x + moe for the
    rows in ``tokens`` (all tokens when None).
    """
    x = np.asarray(x, dtype=np.float64)
    T, k = idx.shape
    toks = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    moe = np.zeros((len(toks), x.shape[1]), dtype=np.float64)
    for i, t in enumerate(toks):
        for r in range(k):
            if pos[t, r] >= 0:
                moe[i] += w[t, r] * expert_out[(int(t), r)]
    if shared_out is not None:
        moe = moe + np.asarray(shared_out, dtype=np.float64)
    out = x[toks] + moe if residual else moe.copy()
    return dict(moe=moe, out=out)


def forward(x, W_g, k: int, act: int, W1, W2, W3=None, b1=None, b2=None,
            b_g=None, W_noise=None, eps=None, capacity_factor: Optional[float] = None,
            C: Optional[int] = None, tokens=None, idx_override=None, shared: Optional[dict] = None,
            gate_mode: str = "renorm", overflow: str = "drop") -> dict:
    """Forward pass of one sparse MoE layer, step by step.

    1 logits ([P4] s2) -> 2 top-k ([P4] s2) -> 3 gates ([P4] s2) ->
    4 capacity ([P5]) -> 5 dispatch ([P1] Lab 3) -> 6 experts on the kept
    assignments -> 7 combine + residual ([P4] s1, s3).
    ``shared``: optional shared experts (keys W1s, W2s and optionally W3s,
    b1s, b2s, as in ``shared_experts``), applied to every token and added in
    the combine.  ``gate_mode``: "renorm" (softmax over the k selected
    logits) or "raw" (``gates_raw``).  ``overflow``: "drop" or "reroute"
    (``reroute``, after the dispatch).

    ``tokens``: evaluate experts and combine only for these token ids
    (routing and dispatch always cover the whole batch, since capacity
    couples all tokens).  ``idx_override``: dispatch/combine a given top-k
    index table instead of the oracle's own (used to check the later stages
    on another router's decisions); gates still come from the oracle's H.
    """
    x = np.asarray(x, dtype=np.float64)
    T, d = x.shape
    E = np.asarray(W_g).shape[1]
    H = logits(x, W_g, b_g, W_noise, eps)
    idx = topk(H, k) if idx_override is None else np.asarray(idx_override, dtype=np.int64)
    w = gates(H, idx) if gate_mode == "renorm" else gates_raw(H, idx)
    if C is None:
        C = capacity(T, k, E, capacity_factor)
    disp = dispatch(idx, E, C)
    if overflow == "reroute":
        backup = topk(H, k + 1)[:, k] if k < E else np.full(T, -1, dtype=np.int64)
        rr = reroute(idx, disp, backup, C)
        idx = rr["idx"]
        disp = dict(disp, pos=rr["pos"], counts=rr["counts"], offsets=rr["offsets"], dropped=rr["dropped"],
                    rerouted=rr["rerouted"], backup=backup)
    pos = disp["pos"]
    toks = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    per_expert = [[] for _ in range(E)]
    for t in toks:
        for r in range(k):
            if pos[t, r] >= 0:
                per_expert[int(idx[t, r])].append((int(t), r))
    expert_out = {}
    for e in range(E):
        pairs = per_expert[e]
        if not pairs:
            continue
        rows = np.stack([x[t] for t, _ in pairs])
        y = expert(rows, e, act, W1, W3, W2, b1, b2)
        for i, p in enumerate(pairs):
            expert_out[p] = y[i]
    sh = None
    if shared is not None:
        sh = shared_experts(x, act, shared["W1s"], shared["W2s"], shared.get("W3s"), shared.get("b1s"),
                            shared.get("b2s"), tokens=toks)
    comb = combine(x, idx, w, pos, expert_out, residual=True, tokens=toks, shared_out=sh)
    return dict(H=H, idx=idx, w=w, C=C, tokens=toks, shared_out=sh, **disp, **comb)


def forward_expert_choice(x, W_g, act: int, W1, W2, W3=None, b1=None, b2=None, b_g=None, W_noise=None, eps=None,
                          C: Optional[int] = None, capacity_factor: Optional[float] = None, k: int = 1,
                          tokens=None, shared: Optional[dict] = None) -> dict:
    """Forward pass of one MoE layer with expert-choice routing ([P1]
    "Advanced Theory & Extensions").

    1 logits ([P4] s2) -> 2 each expert's top-C tokens (``expert_choice``)
    -> 3 every expert on its chosen tokens -> 4 out[t] = x[t] + sum over the
    experts e that chose t, in order e = 0..E-1, of p[t,e] * E_e(x_t)
    (+ the shared experts), the residual carrying a token no expert chose.
    C defaults to the token-choice capacity ceil(cf * T * k / E) ([P5]), k
    being the average number of experts per token.
    """
    x = np.asarray(x, dtype=np.float64)
    T, d = x.shape
    E = np.asarray(W_g).shape[1]
    H = logits(x, W_g, b_g, W_noise, eps)
    if C is None:
        C = capacity(T, k, E, capacity_factor)
    ec = expert_choice(H, C)
    toks = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    want = set(int(t) for t in toks)
    contrib = {}
    for e in range(E):
        rows = [int(t) for t in ec["sel"][e] if int(t) in want]
        if not rows:
            continue
        y = expert(x[rows], e, act, W1, W3, W2, b1, b2)
        for i, t in enumerate(rows):
            contrib[(t, e)] = ec["P"][t, e] * y[i]
    moe = np.zeros((len(toks), d), dtype=np.float64)
    for i, t in enumerate(toks):
        for e in range(E):
            if ec["chosen"][t, e]:
                moe[i] += contrib[(int(t), e)]
    sh = None
    if shared is not None:
        sh = shared_experts(x, act, shared["W1s"], shared["W2s"], shared.get("W3s"), shared.get("b1s"),
                            shared.get("b2s"), tokens=toks)
        moe = moe + sh
    return dict(H=H, C=C, tokens=toks, moe=moe, out=x[toks] + moe, shared_out=sh, **ec)


def near_ties(H: np.ndarray, k: int, thresh: float = 1e-4) -> dict:
    """Near-tie report: tokens whose k-th and (k+1)-th largest logits differ
    by less than ``thresh``, and tokens with any adjacent gap under ``thresh``
    among their k+1 largest logits (a swap inside the top k changes the rank
    order, hence the dispatch priority)."""
    H = np.asarray(H, dtype=np.float64)
    E = H.shape[1]
    s = -np.sort(-H, axis=1)
    boundary = np.zeros(H.shape[0], dtype=bool)
    if k < E:
        boundary = (s[:, k - 1] - s[:, k]) < thresh
    m = min(k + 1, E)
    inner = np.zeros(H.shape[0], dtype=bool)
    for j in range(m - 1):
        inner |= (s[:, j] - s[:, j + 1]) < thresh
    return dict(boundary=np.nonzero(boundary)[0], any_adjacent=np.nonzero(inner)[0])


# --------------------------------------------------------------------------
# routing diagnostics and the auxiliary load-balancing loss
# --------------------------------------------------------------------------

def routing_stats(H: np.ndarray, idx: np.ndarray, counts: np.ndarray, dropped: int) -> dict:
    """Routing diagnostics of one batch and the auxiliary load-balancing loss.

    [P1] "Mathematical Formulation": L_aux = N * sum_i f_i * P_i, f_i the
    fraction of the batch dispatched to expert i (a hard count), P_i the mean
    routing probability of expert i over the batch; uniform routing gives
    exactly 1.  [P1] Lab 2 takes P from the full softmax of the router logits.
    [P4] s4 states the same loss with the coefficient alpha left to the
    trainer.  [P2] Level 3 (load-balancing diagnostics) asks for the
    probability mass and the realised loads together, with overflow,
    utilisation and a named imbalance measure.

    Readings (top-k): f_i counts every selected assignment (t, r) with
    idx[t,r] = i before the capacity cut, divided by T*k, so f sums to 1; P
    is the mean over tokens of softmax(H[t]) over all E experts (the noisy
    logits when noise is used).

    H [T,E] logits, idx [T,k] selected experts, counts [E] kept assignments
    (after capacity), dropped = assignments over capacity.
    Returns f [E], P [E], aux_loss, entropy (mean over tokens of
    -sum_e p ln p, nats), load_cv (population std / mean of the
    pre-capacity loads), kept_cv (same for counts), utilisation (fraction of
    experts with a kept assignment), overflow (dropped / (T*k)).
    """
    H = np.asarray(H, dtype=np.float64)
    T, E = H.shape
    idx = np.asarray(idx, dtype=np.int64)
    k = idx.shape[1]
    counts = np.asarray(counts, dtype=np.float64)
    if T == 0:
        zero = np.zeros(E)
        return dict(f=zero, P=zero, aux_loss=0.0, entropy=0.0, load_cv=0.0, kept_cv=0.0, utilisation=0.0,
                    overflow=0.0, loads=zero)
    p = np.exp(H - H.max(axis=1, keepdims=True))
    p = p / p.sum(axis=1, keepdims=True)
    P = p.mean(axis=0)
    loads = np.bincount(idx.reshape(-1), minlength=E).astype(np.float64)
    f = loads / float(T * k)
    aux = float(E) * float(np.sum(f * P))
    with np.errstate(divide="ignore", invalid="ignore"):
        plogp = np.where(p > 0.0, p * np.log(p), 0.0)
    entropy = float(-plogp.sum(axis=1).mean())

    def cv(v):
        m = v.mean()
        return float(np.sqrt(((v - m) ** 2).mean()) / m) if m > 0 else 0.0

    return dict(f=f, P=P, aux_loss=aux, entropy=entropy, load_cv=cv(loads), kept_cv=cv(counts),
                utilisation=float((counts > 0).sum()) / E, overflow=float(dropped) / float(T * k), loads=loads)

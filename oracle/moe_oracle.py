"""Plain, slow CPU oracle for the single-GPU MoE feed-forward layer forward pass.

TEST INFRASTRUCTURE ONLY.  This module exists to check the CUDA library.  Only the
test suite, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl
reference`` legs of ``bench.py`` may import it.  The product path never calls it,
and it shares no code with the CUDA path.

Every function works in float64 on NumPy arrays.  Inputs given in bf16 are passed
in already widened (bf16 -> float is exact), so the oracle sees the same values as
the kernels.  The one place where a floating-point value decides an integer is the
expert selection: it is taken on float32 router logits, the precision the kernels
use, with ties broken towards the lower expert id.

Sources (page titles as printed; sections as headed on each page):

* P1 = "MoE大模型的智能调度：从1.8万亿参数到每token仅激活2%的工程真相",
  section 2.2 "MoE 架构的三层核心组件：路由层、专家层、融合层"
  (routing steps 1-4, the expert layer, the gated sum of the fusion layer).
* P3 = the page opening "MoE通过稀疏激活降低每个token的计算量但增加了服务系统的复杂度",
  sections "MoE层的结构与token路由" (weighted sum over the selected set S(x),
  shared experts), "一个批次如何变成各专家专属的矩阵" (assignments, grouping by
  expert, the four-token worked example) and "单机MoE执行流水线" (router scores,
  top-k, permutation with an inverse map, grouped GEMM, activation and output
  projection, un-permute and weighted accumulation).

Readings taken where the pages are silent or ambiguous (each is listed in the
design notes of the repository):

* Router = one linear map with an optional per-expert bias, L = x W_r^T + b.
* Softmax over the K selected logits (equal, in exact arithmetic, to a softmax over
  all E experts renormalised over the K).
* Gate drop: a slot k >= 1 whose renormalised gate is strictly below the threshold
  is dropped (id -1, gate 0) and the survivors are renormalised once; slot 0 is
  never dropped.  Dropped assignments are not dispatched.
* Expert FFN = SwiGLU: h = silu(x W_g^T) * (x W_u^T), o = h W_d^T, with the gate and
  up weights stacked as W_gu = [W_g; W_u] of shape [2I, H] and W_d of shape [H, I].
* Rows of an expert's group are ordered by ascending token id.
* A shared expert (if any) is added with weight 1 after the routed sum.

Parity pins: every function here is pinned by ``tests/test_oracle_*.py`` against
the worked example of P3, closed forms, hand-computable special cases, invariants
and a scalar brute force on tiny inputs.  The full-size configs are pinned only
through those functions ("parity unpinned" beyond them).
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "router_logits",
    "topk_softmax",
    "gate_drop",
    "route",
    "capacity",
    "route_capacity",
    "permute",
    "quantize_e4m3",
    "quantize_rows_fp8",
    "expert_gate_up_fp8",
    "expert_down_fp8",
    "silu",
    "swiglu_ffn",
    "expert_gate_up",
    "expert_down",
    "grouped_ffn",
    "combine",
    "moe_layer",
    "moe_layer_tokens",
]


def router_logits(x, w_router, bias=None):
    """Router scores: one logit per expert per token.

    P1 §2.2, routing step 1 (the router maps the hidden state h to one logit per
    expert); P3 "MoE层的结构与token路由" (the router scores every expert for the
    token).  Computed in float64: L[t, e] = sum_h x[t, h] * W_r[e, h] (+ b[e]).
    x: [T, H], w_router: [E, H], bias: [E] or None.  Returns [T, E] float64.
    """
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w_router, dtype=np.float64)
    logits = x @ w.T
    if bias is not None:
        logits = logits + np.asarray(bias, dtype=np.float64)[None, :]
    return logits


def topk_softmax(logits32, K):
    """Top-k selection and softmax over the selected logits.

    P1 §2.2, routing step 2 (take the top-k logits and normalise them with a
    softmax into w_1..w_k); P3 "单机MoE执行流水线" (top-k keeps the chosen expert
    indices and their weights).

    logits32: [T, E] values that are float32 numbers (the selection is made on
    float32, the kernels' precision).  Order per token: logit descending, ties to
    the lower expert id.  Gates in float64:
        w_k = exp(l_k - l_0) / sum_{j<K} exp(l_j - l_0).
    Returns ids [T, K] int32 and w [T, K] float64, slot 0 = largest logit.
    """
    L = np.asarray(logits32, dtype=np.float32).astype(np.float64)
    T, E = L.shape
    if not 1 <= K <= E:
        raise ValueError("need 1 <= K <= E")
    ids = np.empty((T, K), dtype=np.int32)
    w = np.empty((T, K), dtype=np.float64)
    experts = np.arange(E)
    for t in range(T):
        # lexsort sorts by the last key first: primary -logit, secondary expert id
        order = np.lexsort((experts, -L[t]))
        top = order[:K]
        ids[t] = top
        z = np.exp(L[t, top] - L[t, top[0]])
        w[t] = z / z.sum()
    return ids, w


def gate_drop(ids, w, theta):
    """Below-threshold gate drop with one renormalisation.

    P1 §2.2, routing step 3: a selected expert whose weight is below the (tunable)
    threshold is set to zero and the remaining weights are renormalised; the page
    gives 0.05 as DeepSeek's value.  Reading: strict comparison w < theta, applied
    to the renormalised top-k gates, slot 0 never dropped, one pass.  A dropped slot
    gets id -1 and gate 0.  theta == 0 disables the drop.
    """
    ids = np.array(ids, dtype=np.int32, copy=True)
    w = np.array(w, dtype=np.float64, copy=True)
    if theta <= 0.0:
        return ids, w
    T, K = ids.shape
    for t in range(T):
        for k in range(1, K):
            if w[t, k] < theta:
                ids[t, k] = -1
                w[t, k] = 0.0
        w[t] = w[t] / w[t].sum()
    return ids, w


def route(logits32, K, theta=0.0):
    """Routing = top-k softmax followed by the gate drop (P1 §2.2, steps 2 and 3)."""
    ids, w = topk_softmax(logits32, K)
    return gate_drop(ids, w, theta)


def capacity(T, K, E, factor_tenths=12):
    """Per-expert capacity of a batch: ceil(T * K / E * 1.2).

    P1 §3.2, trap 2: capacity = (batch_size * seq_len * k) / num_experts * 1.2, the
    batch's assignments spread evenly with a 1.2 safety factor.  Reading: T = batch_size
    * seq_len tokens, rounded up to a whole number of rows, computed exactly in integers.
    """
    return (factor_tenths * T * K + 10 * E - 1) // (10 * E)


def route_capacity(logits32, K, theta=0.0, cap=None):
    """Routing with a per-expert capacity (P1 §3.2, trap 2).

    The page inserts a capacity check into routing: once an expert has been chosen
    `cap` times, its logit is set to -inf and the token chooses again.  Reading: tokens
    are routed one after another in token order.  For token t, an expert is available
    when fewer than `cap` of the assignments kept so far (tokens before t, after their
    gate drop) went to it.  The token then takes the top-k of the available experts only
    (logit descending, ties to the lower id), with a softmax over those and the gate drop
    of `gate_drop`.  Its kept assignments then count against the experts' capacity.  If
    fewer than K experts are available, the missing slots hold id -1 and gate 0.

    Returns ids [T, K] int32 and w [T, K] float64, as `route`.
    """
    L = np.asarray(logits32, dtype=np.float32).astype(np.float64)
    T, E = L.shape
    if not 1 <= K <= E:
        raise ValueError("need 1 <= K <= E")
    if cap is None:
        cap = capacity(T, K, E)
    count = np.zeros(E, dtype=np.int64)
    ids = np.full((T, K), -1, dtype=np.int32)
    w = np.zeros((T, K), dtype=np.float64)
    experts = np.arange(E)
    for t in range(T):
        avail = experts[count < cap]
        if len(avail) == 0:
            continue
        order = avail[np.lexsort((avail, -L[t, avail]))]
        top = order[:K]
        z = np.exp(L[t, top] - L[t, top[0]])
        row_ids = np.full(K, -1, dtype=np.int32)
        row_w = np.zeros(K)
        row_ids[:len(top)] = top
        row_w[:len(top)] = z / z.sum()
        row_ids, row_w = gate_drop(row_ids[None, :], row_w[None, :], theta)
        ids[t], w[t] = row_ids[0], row_w[0]
        for e in ids[t]:
            if e >= 0:
                count[e] += 1
    return ids, w


def permute(ids, E):
    """Dispatch: group the assignments by expert into contiguous row blocks.

    P3 "一个批次如何变成各专家专属的矩阵": every (token, expert, weight) triple is an
    assignment; assignments are grouped by expert, each group becomes a matrix
    with as many rows as it has assignments, and the source token id is kept next
    to every row.  P3 "单机MoE执行流水线": the permutation writes token rows in
    expert order and records an inverse map for the combine.

    ids: [T, K] int32, -1 = dropped.  Rows are ordered by (expert, token).
    Returns counts [E], offsets [E+1] (exclusive scan of counts), perm [M] (the
    source token of each row) and inv [T, K] (the row of each assignment, -1 if
    dropped), where M = number of kept assignments.
    """
    ids = np.asarray(ids, dtype=np.int64)
    T, K = ids.shape
    triples = [(int(ids[t, k]), t, k) for t in range(T) for k in range(K) if ids[t, k] >= 0]
    triples.sort()  # by expert, then token (a token never picks one expert twice)
    counts = np.zeros(E, dtype=np.int32)
    for e, _, _ in triples:
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    perm = np.array([t for _, t, _ in triples], dtype=np.int32)
    inv = np.full((T, K), -1, dtype=np.int32)
    for r, (_, t, k) in enumerate(triples):
        inv[t, k] = r
    return counts, offsets, perm, inv


def silu(z):
    """silu(z) = z / (1 + exp(-z)), in float64."""
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def swiglu_ffn(x_rows, w_gate_up, w_down):
    """One expert's feed-forward network on a block of rows.

    P1 §2.2 (expert layer: every expert is a two-layer FFN of the same shape with
    its own weights); P3 "单机MoE执行流水线" (each expert applies its activation and
    output projection).  The activation is SwiGLU (a reading; the pages name none):
        g = x W_g^T, u = x W_u^T, h = silu(g) * u, o = h W_d^T
    x_rows: [R, H]; w_gate_up: [2I, H] with rows 0..I-1 = W_g and I..2I-1 = W_u;
    w_down: [H, I].  Returns o: [R, H] float64 (h is not rounded).
    """
    return expert_down(expert_gate_up(x_rows, w_gate_up), w_down)


def expert_gate_up(x_rows, w_gate_up):
    """First half of the expert FFN: h = silu(x W_g^T) * (x W_u^T), float64.

    x_rows: [R, H]; w_gate_up: [2I, H] (rows 0..I-1 = W_g, I..2I-1 = W_u).  Returns [R, I].
    """
    x = np.asarray(x_rows, dtype=np.float64)
    wgu = np.asarray(w_gate_up, dtype=np.float64)
    I = wgu.shape[0] // 2
    return silu(x @ wgu[:I].T) * (x @ wgu[I:].T)


E4M3_MAX = 448.0


def quantize_e4m3(v32):
    """Round float32 values to the nearest FP8 E4M3 value (1 sign, 4 exponent bits with
    bias 7, 3 mantissa bits, no infinities; largest finite 448, smallest subnormal 2^-9),
    ties to even, saturating: anything beyond 448 in magnitude becomes +-448.

    Low-precision experts: P1 §4.1 quantises the resident experts' weights to 8 bits
    (INT8) to save memory.  Reading: the 8-bit format that the target's tensor cores run at
    full rate, FP8 E4M3, with one scale per row.  Returns float64 values that are exactly
    representable in E4M3.
    """
    v = np.asarray(v32, dtype=np.float32).astype(np.float64)
    a = np.abs(v)
    out = np.zeros_like(a)
    nz = a > 0
    e = np.floor(np.log2(np.where(nz, a, 1.0)))
    e = np.maximum(e, -6.0)               # below 2^-6 the spacing stays 2^-9 (subnormals)
    quantum = np.exp2(e - 3.0)            # 3 mantissa bits
    q = np.round(a / quantum) * quantum   # np.round: halves to even, exact for these powers of 2
    q = np.minimum(q, E4M3_MAX)
    out[nz] = q[nz]
    return np.copysign(out, v)


def quantize_rows_fp8(a):
    """Per-row E4M3 quantisation of a [rows, cols] matrix: scale = amax(|row|) / 448 in
    float32 (1 for an all-zero row) and codes = E4M3(row * (1 / scale)): the reciprocal of
    the scale and the product, each rounded to float32, which is the precision the kernels
    take this decision in (the page fixes none).  Returns (codes as float64 values, scales
    as float32), with row ~= codes * scale."""
    a32 = np.asarray(a, dtype=np.float32)
    amax = np.abs(a32).max(axis=1)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    inv = (np.float32(1.0) / scale).astype(np.float32)
    codes = quantize_e4m3((a32 * inv[:, None]).astype(np.float32))
    return codes, scale


def expert_gate_up_fp8(x_codes, x_scale, w_codes, w_scale):
    """The gate/up half of the expert FFN on E4M3 operands: every dot product of codes is
    exact in float64, then scaled by the token row's and the weight row's scales;
    h = silu(g) * u as in `expert_gate_up`.  w rows 0..I-1 are the gate, I..2I-1 the up."""
    acc = (np.asarray(x_codes, dtype=np.float64) @ np.asarray(w_codes, dtype=np.float64).T)
    acc = acc * np.asarray(x_scale, dtype=np.float64)[:, None] * \
        np.asarray(w_scale, dtype=np.float64)[None, :]
    I = acc.shape[1] // 2
    return silu(acc[:, :I]) * acc[:, I:]


def expert_down_fp8(h_codes, h_scale, w_codes, w_scale):
    """The output projection on E4M3 operands: o[r, n] = h_scale[r] * w_scale[n] *
    sum_k hq[r, k] wq[n, k], the code dot products exact in float64 (W_d rows = output
    channels, one scale each)."""
    acc = np.asarray(h_codes, dtype=np.float64) @ np.asarray(w_codes, dtype=np.float64).T
    return acc * np.asarray(h_scale, dtype=np.float64)[:, None] * \
        np.asarray(w_scale, dtype=np.float64)[None, :]


def expert_down(h_rows, w_down):
    """Second half of the expert FFN, the output projection: o = h W_d^T, float64.

    h_rows: [R, I]; w_down: [H, I].  Returns [R, H].
    """
    return np.asarray(h_rows, dtype=np.float64) @ np.asarray(w_down, dtype=np.float64).T


def grouped_ffn(x_perm, offsets, w_gate_up, w_down):
    """Every expert runs its FFN on its own contiguous row group.

    P3 "一个批次如何变成各专家专属的矩阵" / "单机MoE执行流水线": the grouped GEMM runs
    the experts' matrices (rows may differ per expert) and grouping only changes
    the number of launches, not the matrices.  Here: a plain loop over experts.
    x_perm: [M, H]; offsets: [E+1]; w_gate_up: [E, 2I, H]; w_down: [E, H, I].
    Returns out_perm: [M, H] float64.
    """
    x_perm = np.asarray(x_perm, dtype=np.float64)
    M, H = x_perm.shape
    out = np.zeros((M, H), dtype=np.float64)
    E = len(offsets) - 1
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 > r0:
            out[r0:r1] = swiglu_ffn(x_perm[r0:r1], w_gate_up[e], w_down[e])
    return out


def combine(out_perm, inv, w, shared_out=None):
    """Un-permute and gated weighted sum back to token order.

    P1 §2.2 step 4 and the fusion layer (output = sum of gate_i * Expert_i(h));
    P3 "MoE层的结构与token路由" (y = sum over the selected set S(x) of
    w_e(x) E_e(x), and only the selected experts enter the sum);
    P3 "单机MoE执行流水线" (restore token order with the inverse map, apply the
    route weights and add up contributions with the same token id).
        y[t] = sum_{k: inv[t,k] >= 0} w[t,k] * out_perm[inv[t,k]]  (+ shared_out[t])
    Returns y: [T, H] float64.
    """
    out_perm = np.asarray(out_perm, dtype=np.float64)
    inv = np.asarray(inv)
    w = np.asarray(w, dtype=np.float64)
    T, K = inv.shape
    H = out_perm.shape[1]
    y = np.zeros((T, H), dtype=np.float64)
    for t in range(T):
        for k in range(K):
            r = int(inv[t, k])
            if r >= 0:
                y[t] += w[t, k] * out_perm[r]
    if shared_out is not None:
        y = y + np.asarray(shared_out, dtype=np.float64)
    return y


def _logits32(x, w_router, bias):
    """Router logits rounded to float32, the precision the selection is taken in."""
    return router_logits(x, w_router, bias).astype(np.float32)


def moe_layer(x, w_router, w_gate_up, w_down, K, theta=0.0, router_bias=None,
              w_shared_gate_up=None, w_shared_down=None, logits=None):
    """The whole layer, stage by stage, in the order P3 "单机MoE执行流水线" gives.

    router scores -> top-k (+ gate drop) -> permutation with inverse map ->
    per-expert SwiGLU FFN on the grouped rows -> un-permute and weighted sum,
    plus the shared expert (P3 "MoE层的结构与token路由": a shared expert is not
    scored by the router and runs for every token).
    If ``logits`` is given (float32 [T, E]), it replaces the router scores.
    Returns a dict with every intermediate and ``y`` [T, H] float64.
    """
    x = np.asarray(x, dtype=np.float64)
    E = w_gate_up.shape[0]
    L32 = _logits32(x, w_router, router_bias) if logits is None else np.asarray(logits, np.float32)
    ids, w = route(L32, K, theta)
    counts, offsets, perm, inv = permute(ids, E)
    x_perm = x[perm] if len(perm) else np.zeros((0, x.shape[1]))
    out_perm = grouped_ffn(x_perm, offsets, w_gate_up, w_down)
    shared = None
    if w_shared_gate_up is not None:
        shared = swiglu_ffn(x, w_shared_gate_up, w_shared_down)
    y = combine(out_perm, inv, w, shared)
    return dict(logits=L32, ids=ids, w=w, counts=counts, offsets=offsets, perm=perm,
                inv=inv, x_perm=x_perm, out_perm=out_perm, shared=shared, y=y)


def moe_layer_tokens(x_tokens, w_router, w_gate_up, w_down, K, theta=0.0, router_bias=None,
                     w_shared_gate_up=None, w_shared_down=None, logits=None):
    """The layer output for a subset of tokens, token by token.

    Each token's output depends only on its own row (P3 "MoE层的结构与token路由":
    the FFN transforms each token position independently), so a sample of tokens
    can be checked at any batch size.  x_tokens: [S, H]; optional float32 logits
    [S, E] replace the router scores.  Returns ids, w, y [S, H].
    """
    x = np.asarray(x_tokens, dtype=np.float64)
    L32 = _logits32(x, w_router, router_bias) if logits is None else np.asarray(logits, np.float32)
    ids, w = route(L32, K, theta)
    S, H = x.shape
    y = np.zeros((S, H), dtype=np.float64)
    # Each selected expert is evaluated once on the sampled rows that chose it;
    # row s of the result is exactly that expert applied to token s alone.
    for e in np.unique(ids[ids >= 0]):
        rows, slots = np.nonzero(ids == e)
        o = swiglu_ffn(x[rows], w_gate_up[e], w_down[e])
        y[rows] += w[rows, slots][:, None] * o
    if w_shared_gate_up is not None:
        y += swiglu_ffn(x, w_shared_gate_up, w_shared_down)
    return dict(logits=L32, ids=ids, w=w, y=y)

"""Shared test helpers: buffers for the C ABI, oracle inputs, routing ambiguity.

Where floating point decides an integer (which experts are selected, whether a gate is
dropped), the GPU and the oracle can legitimately disagree when the deciding values lie
within rounding error of each other.  Such tokens are "ambiguous": their ids are only
checked for validity and they are left out of output comparisons; every other token
must match exactly.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

# Tolerances of the layer output against the float64 oracle (bf16 inputs, fp32
# accumulation): max-abs and relative L2 of the fp32 combine accumulator y_f32.
Y_MAX_ABS = 2e-2
Y_REL_L2 = 1e-2
# float32 layers: tolerance derived from fp32 accumulation of a few thousand terms.
Y32_MAX_ABS = 1e-3
Y32_REL_L2 = 1e-3
# Logit agreement (fp32 accumulation vs float64) and the decision margins built on it.
LOGIT_ATOL = 5e-5
GATE_ATOL = 2e-6


def f64(t):
    return synth.to_numpy_f64(t)


def cuda_empty(shape, dtype):
    return torch.empty(shape, dtype=dtype, device="cuda")


def ambiguous_tokens(L, K, theta, w_ref, margin=LOGIT_ATOL):
    """Tokens whose routing can flip within `margin` of logit error (or whose gates lie
    within GATE_ATOL of the drop threshold).  margin=None: the logits are shared exactly,
    only the threshold decision can differ."""
    L = np.asarray(L, dtype=np.float64)
    T, E = L.shape
    amb = np.zeros(T, dtype=bool)
    if T == 0:
        return amb
    s = -np.sort(-L, axis=1)
    if margin is not None:
        m = min(K + 1, E)
        gaps = s[:, :m - 1] - s[:, 1:m]
        tol = margin * np.maximum(1.0, np.abs(s[:, :m - 1]))
        amb |= (gaps <= tol).any(axis=1)
    if theta > 0 and w_ref is not None:
        amb |= (np.abs(np.asarray(w_ref)[:, 1:] - theta) <= GATE_ATOL).any(axis=1)
        # a near-threshold gate before renormalisation also counts
        z = np.exp(s[:, :K] - s[:, :1])
        w0 = z / z.sum(axis=1, keepdims=True)
        amb |= (np.abs(w0[:, 1:] - theta) <= 10 * GATE_ATOL).any(axis=1)
    return amb


def check_valid_selection(L, ids, K, margin=LOGIT_ATOL):
    """The kept ids of one token are a valid descending top selection of logits L within
    `margin`: distinct, in descending order, and none below an expert left out.  (Dropped
    slots carry -1; their experts have smaller logits than every kept one.)"""
    sel = [int(e) for e in ids if e >= 0]
    assert int(ids[0]) >= 0 and len(set(sel)) == len(sel)
    tol = margin * max(1.0, float(np.max(np.abs(L))))
    vals = [float(L[e]) for e in sel]
    for a, b in zip(vals, vals[1:]):
        assert a >= b - tol
    rest = [float(L[e]) for e in range(len(L)) if e not in set(sel)]
    if rest:
        assert min(vals) >= max(rest) - tol


def compare_routing(L_ref32, ids_gpu, w_gpu, ids_ref, w_ref, K, theta, margin=LOGIT_ATOL):
    """ids bit-exact and gates close on unambiguous tokens; valid elsewhere.
    Returns the boolean mask of ambiguous tokens."""
    amb = ambiguous_tokens(L_ref32, K, theta, w_ref, margin)
    ok = ~amb
    np.testing.assert_array_equal(ids_gpu[ok], ids_ref[ok])
    np.testing.assert_allclose(w_gpu[ok], w_ref[ok], rtol=0, atol=1e-5)
    for t in np.nonzero(amb)[0]:
        check_valid_selection(L_ref32[t], ids_gpu[t], K)
        assert abs(float(w_gpu[t].sum()) - 1.0) < 1e-5
    return amb


def assert_close_y(got, want, max_abs=Y_MAX_ABS, rel_l2=Y_REL_L2, what="y"):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape
    if got.size == 0:
        return 0.0, 0.0
    err = float(np.abs(got - want).max())
    nrm = float(np.linalg.norm(want))
    rel = float(np.linalg.norm(got - want) / nrm) if nrm > 0 else err
    assert err <= max_abs and rel <= rel_l2, f"{what}: max-abs {err:.3g} (<= {max_abs}), rel-L2 {rel:.3g} (<= {rel_l2})"
    return err, rel


def bf16_half_ulp(v):
    """Half the spacing of bfloat16 numbers at |v| (8 significant bits): the most a correct
    round-to-nearest store can move a value."""
    a = np.maximum(np.abs(np.asarray(v, dtype=np.float64)), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 8)


def assert_close_y_rounded(got_bf16, want, max_abs=Y_MAX_ABS, rel_l2=Y_REL_L2, what="y (bf16)"):
    """The rounded bf16 output against the float64 oracle: every element within max_abs plus
    half a bf16 ulp of the oracle's value (the store's own rounding, which exceeds max_abs
    where |y| >= 8), and relative L2 within rel_l2."""
    got = np.asarray(got_bf16, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape
    if got.size == 0:
        return
    excess = np.abs(got - want) - (max_abs + bf16_half_ulp(want))
    nrm = float(np.linalg.norm(want))
    rel = float(np.linalg.norm(got - want) / nrm) if nrm > 0 else 0.0
    assert excess.max() <= 0 and rel <= rel_l2, \
        f"{what}: worst excess over max-abs + half ulp {excess.max():.3g}, rel-L2 {rel:.3g} (<= {rel_l2})"


class LayerRun:
    """Buffers and one moe_layer_forward call of a workload on the GPU."""

    def __init__(self, moe, shape, inputs, T=None, flags=0):
        self.moe = moe
        self.shape = shape
        self.inp = inputs
        self.T = inputs["x"].shape[0] if T is None else T
        s = shape
        dt = moe.BF16 if s.dtype == "bf16" else moe.F32
        self.cfg = moe.MoEConfig.make(self.T, s.H, s.E, s.K, s.I, s.I_shared, s.theta, dt, flags)
        self.ws = torch.empty(moe.workspace_size(self.cfg), dtype=torch.uint8, device="cuda")
        self.y = torch.empty(self.T, s.H, dtype=s.torch_dtype, device="cuda")
        self.y32 = torch.empty(self.T, s.H, dtype=torch.float32, device="cuda")

    def run(self, stream=None):
        i = self.inp
        self.moe.layer_forward(self.cfg, i["x"], i["w_router"], i["router_bias"], i["w_gate_up"],
                               i["w_down"], i.get("w_shared_gate_up"), i.get("w_shared_down"),
                               self.y, self.y32, self.ws, stream=stream)

    def view(self, name, shape, dtype):
        """A torch view of one intermediate the layer left in the workspace."""
        addr = self.moe.workspace_views(self.cfg, self.ws)[name]
        off = addr - self.ws.data_ptr()
        n = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
        return self.ws[off:off + n].view(dtype).view(*shape)

    def routing(self):
        T, K, E = self.T, self.shape.K, self.shape.E
        return dict(
            logits=self.view("logits", (T, E), torch.float32).cpu().numpy(),
            ids=self.view("topk_ids", (T, K), torch.int32).cpu().numpy(),
            w=self.view("topk_w", (T, K), torch.float32).cpu().numpy(),
            counts=self.view("counts", (E,), torch.int32).cpu().numpy(),
            offsets=self.view("offsets", (E + 1,), torch.int32).cpu().numpy(),
            perm=self.view("perm", (T * K,), torch.int32).cpu().numpy(),
            inv=self.view("inv", (T, K), torch.int32).cpu().numpy(),
        )


class ExpertSlices:
    """Lazy float64 host copies of one expert's weights, indexed like the full array."""

    def __init__(self, w):
        self.w = w
        self.shape = tuple(w.shape)

    def __getitem__(self, e):
        return f64(self.w[int(e)])


def capacity_gate_margin(L, K, theta, ids):
    """Smallest |pre-drop gate - theta| over slots >= 1 in the token-by-token capacity
    routing whose result is `ids`: the replay recovers each token's available top-k."""
    if theta <= 0:
        return np.inf
    L = L.astype(np.float64)
    T, E = L.shape
    cap = oracle.capacity(T, K, E)
    count = np.zeros(E, dtype=np.int64)
    m = np.inf
    for t in range(T):
        avail = np.nonzero(count < cap)[0]
        top = avail[np.lexsort((avail, -L[t, avail]))][:K]
        if len(top) > 1:
            z = np.exp(L[t, top] - L[t, top[0]])
            m = min(m, float(np.abs(z[1:] / z.sum() - theta).min()))
        for e in ids[t]:
            if e >= 0:
                count[e] += 1
    return m

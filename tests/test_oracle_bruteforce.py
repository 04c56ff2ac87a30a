"""The oracle against a scalar brute force on tiny inputs, and its invariants.

The brute force evaluates EVERY expert on EVERY token with scalar Python loops and
forms y = sum_e g_e * E_e(x), where g is the full softmax over all E experts
renormalised over the top-K by probability, scattered to E slots with zeros
elsewhere ("the sum covers only the selected experts", page opening
"MoE通过稀疏激活…", section "MoE层的结构与token路由").  It shares no code path with
the oracle's grouped pipeline (no permutation, no inverse map, no top-k softmax).

Invariants (same page, sections "一个批次如何变成各专家专属的矩阵" and
"单机MoE执行流水线"): there are T*K assignments minus drops; every token comes back
to its own position through the inverse map; kept gates sum to 1; permuting and
then un-permuting with unit weights is the identity.
"""

import math

import numpy as np
import pytest

import oracle


def _brute_force(x, w_router, bias, w_gate_up, w_down, K, theta, ws_gu=None, ws_d=None):
    T, H = x.shape
    E = w_router.shape[0]
    I = w_gate_up.shape[1] // 2

    def ffn(xt, wgu, wd, Ie):
        h = []
        for i in range(Ie):
            g = sum(float(xt[j]) * float(wgu[i, j]) for j in range(H))
            u = sum(float(xt[j]) * float(wgu[Ie + i, j]) for j in range(H))
            h.append(g / (1.0 + math.exp(-g)) * u)
        return [sum(h[i] * float(wd[j, i]) for i in range(Ie)) for j in range(H)]

    y = np.zeros((T, H))
    for t in range(T):
        logits = []
        for e in range(E):
            s = sum(float(x[t, j]) * float(w_router[e, j]) for j in range(H))
            if bias is not None:
                s += float(bias[e])
            logits.append(float(np.float32(s)))     # selection is taken on float32 logits
        m = max(logits)
        p = [math.exp(l - m) for l in logits]
        z = sum(p)
        p = [v / z for v in p]
        chosen = sorted(range(E), key=lambda e: (-logits[e], e))[:K]
        g = [p[e] for e in chosen]
        s = sum(g)
        g = [v / s for v in g]
        if theta > 0:
            g = [g[0]] + [v if v >= theta else 0.0 for v in g[1:]]
            s = sum(g)
            g = [v / s for v in g]
        for e, ge in zip(chosen, g):
            if ge == 0.0:
                continue
            o = ffn(x[t], w_gate_up[e], w_down[e], I)
            y[t] += ge * np.array(o)
        if ws_gu is not None:
            y[t] += np.array(ffn(x[t], ws_gu, ws_d, ws_gu.shape[0] // 2))
    return y


CASES = [
    # T, H, E, K, I, theta, bias, shared I
    (5, 8, 4, 2, 3, 0.0, False, 0),
    (9, 16, 8, 2, 16, 0.0, True, 0),
    (16, 32, 8, 3, 8, 0.0, False, 0),
    (11, 12, 6, 4, 5, 0.2, True, 0),
    (7, 10, 5, 5, 4, 0.15, False, 6),
    (13, 24, 8, 1, 8, 0.0, True, 4),
    (6, 8, 3, 3, 2, 0.3, True, 3),
]


@pytest.mark.parametrize("T,H,E,K,I,theta,use_bias,Is", CASES)
@pytest.mark.parametrize("seed", [0, 1])
def test_oracle_equals_dense_brute_force(T, H, E, K, I, theta, use_bias, Is, seed):
    rng = np.random.default_rng(100 + seed)
    x = rng.standard_normal((T, H))
    wr = rng.standard_normal((E, H)) / math.sqrt(H)
    wgu = rng.standard_normal((E, 2 * I, H)) * 0.5
    wd = rng.standard_normal((E, H, I)) * 0.5
    bias = rng.standard_normal(E).astype(np.float32) if use_bias else None
    ws_gu = rng.standard_normal((2 * Is, H)) * 0.5 if Is else None
    ws_d = rng.standard_normal((H, Is)) * 0.5 if Is else None
    out = oracle.moe_layer(x, wr, wgu, wd, K, theta, bias, ws_gu, ws_d)
    want = _brute_force(x, wr, bias, wgu, wd, K, theta, ws_gu, ws_d)
    np.testing.assert_allclose(out["y"], want, rtol=1e-9, atol=1e-9)
    tok = oracle.moe_layer_tokens(x[::2], wr, wgu, wd, K, theta, bias, ws_gu, ws_d)
    np.testing.assert_allclose(tok["y"], want[::2], rtol=1e-9, atol=1e-9)


def _check_invariants(x, ids, w, E, theta):
    T, K = ids.shape
    counts, offsets, perm, inv = oracle.permute(ids, E)
    kept = ids >= 0
    M = int(kept.sum())
    assert int(counts.sum()) == M == len(perm)
    assert offsets[0] == 0 and (np.diff(offsets) == counts).all()
    assert (kept[:, 0]).all()                     # slot 0 is never dropped
    for t in range(T):                            # dropped slots form a suffix
        k_kept = kept[t].sum()
        assert kept[t, :k_kept].all()
        assert abs(w[t].sum() - 1.0) < 1e-12
        if theta > 0:
            assert (w[t, 1:k_kept] >= theta).all()
    seen = np.zeros(M, dtype=int)
    for t in range(T):
        for k in range(K):
            r = inv[t, k]
            if ids[t, k] < 0:
                assert r == -1
                continue
            assert offsets[ids[t, k]] <= r < offsets[ids[t, k] + 1]
            assert perm[r] == t
            seen[r] += 1
    assert (seen == 1).all()
    for e in range(E):                            # rows of a group in ascending token order
        grp = perm[offsets[e]:offsets[e + 1]]
        assert (np.diff(grp) > 0).all()
    x_perm = x[perm]
    for t in range(T):
        for k in range(K):
            if inv[t, k] >= 0:
                assert (x_perm[inv[t, k]] == x[t]).all()
    # permute then un-permute with unit weights: each token comes back K' times
    unit = np.where(kept, 1.0, 0.0)
    back = oracle.combine(x_perm, inv, unit)
    np.testing.assert_array_equal(back, x * kept.sum(1)[:, None])


@pytest.mark.parametrize("seed", range(6))
def test_routing_and_dispatch_invariants(seed):
    rng = np.random.default_rng(seed)
    T = int(rng.integers(0, 40))
    E = int(rng.integers(1, 20))
    K = int(rng.integers(1, E + 1))
    theta = float(rng.choice([0.0, 0.05, 0.2]))
    x = rng.integers(-50, 50, (T, 3)).astype(np.float64)   # exact sums
    L = (rng.standard_normal((T, E)) * rng.choice([0.1, 1.0, 5.0])).astype(np.float32)
    if seed % 2:
        L = np.round(L)                           # many exact ties
    ids, w = oracle.route(L, K, theta)
    _check_invariants(x, ids, w, E, theta)


try:
    import hypothesis as hyp
except ImportError:          # only the property search needs it; the cases above do not
    hyp = None


def _invariants_case(T, E, K, theta, seed, scale, halves):
    rng = np.random.default_rng(seed)
    L = (rng.standard_normal((T, E)) * scale).astype(np.float32)
    if halves:
        L = np.round(L * 2) / 2
    ids, w = oracle.route(L, K, theta)
    _check_invariants(rng.integers(-50, 50, (T, 2)).astype(np.float64), ids, w, E, theta)


if hyp is not None:
    st = hyp.strategies

    @hyp.settings(max_examples=60, deadline=None)
    @hyp.given(T=st.integers(0, 24), E=st.integers(1, 12), data=st.data())
    def test_invariants_property(T, E, data):
        _invariants_case(T, E, data.draw(st.integers(1, E)),
                         data.draw(st.sampled_from([0.0, 0.01, 0.1, 0.3])),
                         data.draw(st.integers(0, 2**31 - 1)),
                         data.draw(st.sampled_from([0.01, 1.0, 10.0])),
                         data.draw(st.booleans()))
else:
    def test_invariants_property():
        """The same search space as the hypothesis property, drawn from a seeded generator
        where hypothesis is not installed, so the invariants still run everywhere."""
        rng = np.random.default_rng(2024)
        for _ in range(60):
            E = int(rng.integers(1, 13))
            _invariants_case(int(rng.integers(0, 25)), E, int(rng.integers(1, E + 1)),
                             float(rng.choice([0.0, 0.01, 0.1, 0.3])),
                             int(rng.integers(0, 2**31 - 1)),
                             float(rng.choice([0.01, 1.0, 10.0])), bool(rng.integers(0, 2)))

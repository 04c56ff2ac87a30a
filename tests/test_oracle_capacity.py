"""Pins of the oracle's capacity-limited routing (P1 §3.2, trap 2: capacity =
(batch_size * seq_len * k) / num_experts * 1.2; an expert chosen that many times gets
logit -inf and the token chooses again).

Pinned by: the capacity formula at exact and rounded values; hand-worked batches
(K = 1, K = 2 with a closed-form gate, the gate drop freeing capacity, a token left with
no available expert); the special case that reduces to plain routing (no expert reaches
its capacity); invariants; and an independent algorithm, the fixed point of a
whole-batch iteration, which must select exactly what the token-by-token rule selects.
"""

import math

import numpy as np
import pytest

from oracle import moe_oracle as oracle

import synth


def test_capacity_formula():
    # ceil(1.2 * T * K / E) computed exactly: 1.2 * 100 / 12 is 10, not 10.000...2
    assert oracle.capacity(100, 1, 12) == 10
    assert oracle.capacity(5, 1, 4) == 2          # 1.5 -> 2
    assert oracle.capacity(10, 2, 8) == 3         # 3.0 exactly
    assert oracle.capacity(8192, 8, 128) == 615   # 614.4 -> 615
    assert oracle.capacity(16384, 8, 256) == 615
    assert oracle.capacity(1, 8, 128) == 1
    for T, K, E in [(7, 3, 5), (333, 2, 24), (4096, 2, 8), (64, 8, 128)]:
        exact = 12 * T * K / (10 * E)
        assert oracle.capacity(T, K, E) == math.ceil(exact - 1e-12)


def test_hand_batch_top1():
    # every token prefers e0 > e1 > e2 > e3; cap = ceil(1.2 * 5 / 4) = 2
    L = np.array([[4, 3, 2, 1]] * 5, dtype=np.float32)
    ids, w = oracle.route_capacity(L, 1)
    np.testing.assert_array_equal(ids[:, 0], [0, 0, 1, 1, 2])
    np.testing.assert_array_equal(w, np.ones((5, 1)))


def test_hand_batch_top2_closed_form_gate():
    # cap = ceil(1.2 * 4 * 2 / 4) = 3: tokens 0-2 fill e0 and e1, token 3 gets e2, e3
    L = np.array([[4, 3, 2, 1]] * 4, dtype=np.float32)
    ids, w = oracle.route_capacity(L, 2)
    np.testing.assert_array_equal(ids, [[0, 1], [0, 1], [0, 1], [2, 3]])
    s = 1.0 / (1.0 + math.exp(-1.0))  # K = 2: w_0 = sigmoid(l_0 - l_1)
    np.testing.assert_allclose(w, [[s, 1 - s]] * 4, rtol=1e-12)


def test_dropped_gates_do_not_use_capacity():
    L = np.array([[5, 0, -5, -9]] * 3, dtype=np.float32)
    # with the drop (second gates ~0.0067 and ~0.018 are below 0.05) each token keeps one
    # expert, and only that one counts against cap = 1
    ids, w = oracle.route_capacity(L, 2, theta=0.05, cap=1)
    np.testing.assert_array_equal(ids, [[0, -1], [1, -1], [2, -1]])
    np.testing.assert_array_equal(w, [[1, 0]] * 3)
    # without it token 0 fills e0, e1 and token 1 fills e2, e3: token 2 has nothing left
    ids, w = oracle.route_capacity(L, 2, theta=0.0, cap=1)
    np.testing.assert_array_equal(ids, [[0, 1], [2, 3], [-1, -1]])
    np.testing.assert_array_equal(w[2], [0, 0])
    np.testing.assert_allclose(w[:2].sum(axis=1), 1.0)


@pytest.mark.parametrize("theta", [0.0, 0.05])
def test_reduces_to_plain_routing_without_overflow(theta):
    L = synth.random_logits(300, 16, seed=3, scale=1.5).numpy()
    ids0, w0 = oracle.route(L, 4, theta)
    ids, w = oracle.route_capacity(L, 4, theta, cap=300)  # no expert can fill up
    np.testing.assert_array_equal(ids, ids0)
    np.testing.assert_allclose(w, w0, rtol=0, atol=0)


def _fixed_point(L, K, theta, cap):
    """The whole-batch iteration: f[e] = index of the token holding e's cap-th kept
    assignment in the current routing (or T); every token re-selects its top-k among
    experts with f[e] >= t; repeat until nothing changes.  Written independently of the
    token-by-token loop; its fixed point is the sequential routing."""
    L = np.asarray(L, dtype=np.float32).astype(np.float64)
    T, E = L.shape
    f = np.full(E, T)
    for _ in range(T + 2):
        ids = np.full((T, K), -1, dtype=np.int32)
        w = np.zeros((T, K))
        for t in range(T):
            ok = f >= t
            cand = [e for e in sorted(range(E), key=lambda e: (-L[t, e], e)) if ok[e]][:K]
            if not cand:
                continue
            z = np.exp(L[t, cand] - L[t, cand[0]])
            row_i = np.array(cand + [-1] * (K - len(cand)), dtype=np.int32)
            row_w = np.concatenate([z / z.sum(), np.zeros(K - len(cand))])
            if theta > 0:
                for k in range(1, K):
                    if row_w[k] < theta:
                        row_i[k], row_w[k] = -1, 0.0
                row_w = row_w / row_w.sum()
            ids[t], w[t] = row_i, row_w
        nf = np.full(E, T)
        for e in range(E):
            holders = [t for t in range(T) if (ids[t] == e).any()]
            if len(holders) >= cap:
                nf[e] = holders[cap - 1]
        if (nf == f).all():
            return ids, w
        f = nf
    raise AssertionError("no fixed point")


@pytest.mark.parametrize("T,E,K,theta,skew", [
    (60, 8, 2, 0.0, 3.0), (80, 16, 4, 0.05, 2.0), (40, 6, 3, 0.1, 4.0), (50, 12, 1, 0.0, 5.0),
])
def test_sequential_rule_equals_whole_batch_fixed_point(T, E, K, theta, skew):
    rng = np.random.default_rng(T * E + K)
    L = (rng.standard_normal((T, E)) + skew * np.linspace(1, 0, E)).astype(np.float32)
    cap = oracle.capacity(T, K, E)
    ids, w = oracle.route_capacity(L, K, theta)
    ids_fp, w_fp = _fixed_point(L, K, theta, cap)
    np.testing.assert_array_equal(ids, ids_fp)
    np.testing.assert_allclose(w, w_fp, rtol=1e-12, atol=0)
    # the skew makes the capacity bind: some token must have been re-routed
    assert not np.array_equal(ids, oracle.route(L, K, theta)[0])


@pytest.mark.parametrize("T,E,K,theta,skew", [(500, 32, 4, 0.0, 3.0), (400, 8, 2, 0.05, 6.0)])
def test_invariants(T, E, K, theta, skew):
    rng = np.random.default_rng(T + E)
    L = (rng.standard_normal((T, E)) + skew * np.linspace(1, 0, E)).astype(np.float32)
    cap = oracle.capacity(T, K, E)
    ids, w = oracle.route_capacity(L, K, theta)
    counts = np.bincount(ids[ids >= 0], minlength=E)
    assert counts.max() <= cap and counts.sum() <= T * K
    for t in range(T):
        kept = ids[t][ids[t] >= 0]
        assert len(set(kept.tolist())) == len(kept)
        assert (ids[t][len(kept):] == -1).all()  # dropped / missing slots form a suffix
        if len(kept):
            np.testing.assert_allclose(w[t].sum(), 1.0, rtol=1e-12)
            # gates descend with the logits (slot 0 = best available expert)
            assert (np.diff(L[t, kept]) <= 0).all()

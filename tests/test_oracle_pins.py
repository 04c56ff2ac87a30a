"""Pins of the CPU oracle against facts fixed outside the oracle itself.

* the four-token, four-expert, top-two worked example printed on the page opening
  "MoE通过稀疏激活降低每个token的计算量…", section "一个批次如何变成各专家专属的矩阵"
  (tests/golden/worked_example.json);
* closed forms: the K=2 softmax is the logistic function of the logit gap; K=1 gives
  a gate of exactly 1; silu(ln 3) = (3/4) ln 3;
* hand-computable SwiGLU experts with distinct gate, up and down roles;
* the gate-drop rule of "MoE大模型的智能调度…" §2.2 step 3 on hand-made gates.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _load_example(golden_dir):
    with open(os.path.join(golden_dir, "worked_example.json")) as f:
        return json.load(f)


def _example_logits(ex):
    """Float32 logits whose top-2 softmax reproduces the printed route weights.

    Chosen experts get ln(weight); the others get -30, which no top-2 choice can
    reach, so the selection is the printed one and the softmax over the two kept
    logits equals the printed weights up to float32 rounding of ln(weight).
    """
    T, E = ex["T"], ex["E"]
    L = np.full((T, E), -30.0, dtype=np.float32)
    for t in range(T):
        for name, wt in ex["choices"][f"T{t + 1}"]:
            L[t, int(name[1:]) - 1] = np.float32(math.log(wt))
    return L


def test_worked_example_routing(golden_dir):
    ex = _load_example(golden_dir)
    ids, w = oracle.route(_example_logits(ex), ex["K"], 0.0)
    for t in range(ex["T"]):
        printed = sorted(((int(n[1:]) - 1, wt) for n, wt in ex["choices"][f"T{t + 1}"]),
                         key=lambda p: -p[1])
        assert [int(i) for i in ids[t]] == [e for e, _ in printed]
        np.testing.assert_allclose(w[t], [wt for _, wt in printed], rtol=0, atol=1e-6)
        assert abs(w[t].sum() - 1.0) < 1e-12


def test_worked_example_dispatch(golden_dir):
    ex = _load_example(golden_dir)
    ids, _ = oracle.route(_example_logits(ex), ex["K"], 0.0)
    counts, offsets, perm, inv = oracle.permute(ids, ex["E"])
    assert counts.tolist() == ex["group_rows"]
    assert int(counts.sum()) == ex["assignments"]
    assert offsets.tolist() == ex["derived"]["offsets"]
    for e in range(ex["E"]):
        toks = [f"T{int(t) + 1}" for t in perm[offsets[e]:offsets[e + 1]]]
        assert toks == ex["groups"][f"E{e + 1}"]
    assert [f"T{int(t) + 1}" for t in perm] == ex["derived"]["perm_tokens"]
    # the inverse map sends every assignment back to the row holding its token
    for t in range(ex["T"]):
        for k in range(ex["K"]):
            assert perm[inv[t, k]] == t


def test_worked_example_combine(golden_dir):
    ex = _load_example(golden_dir)
    ids, w = oracle.route(_example_logits(ex), ex["K"], 0.0)
    _, _, _, inv = oracle.permute(ids, ex["E"])
    rng = np.random.default_rng(7)
    out_perm = rng.standard_normal((ex["assignments"], 5))
    y = oracle.combine(out_perm, inv, w)
    for t in range(ex["T"]):
        want = sum(wt * out_perm[row] for wt, row in ex["derived"]["combine"][f"T{t + 1}"])
        np.testing.assert_allclose(y[t], want, rtol=0, atol=5e-6)


def test_two_way_softmax_is_logistic():
    rng = np.random.default_rng(1)
    L = rng.standard_normal((64, 6)).astype(np.float32) * 3
    ids, w = oracle.topk_softmax(L, 2)
    for t in range(64):
        gap = float(L[t, ids[t, 0]]) - float(L[t, ids[t, 1]])
        assert gap >= 0
        assert abs(w[t, 0] - 1.0 / (1.0 + math.exp(-gap))) < 1e-12
        assert abs(w[t, 1] - 1.0 / (1.0 + math.exp(gap))) < 1e-12


def test_top1_gate_is_one_and_argmax():
    rng = np.random.default_rng(2)
    L = rng.standard_normal((50, 9)).astype(np.float32)
    ids, w = oracle.topk_softmax(L, 1)
    assert (ids[:, 0] == np.argmax(L, axis=1)).all()
    assert (w == 1.0).all()


def test_topk_ties_go_to_lower_expert():
    L = np.array([[1, 1, 1, 1],
                  [0, 2, 2, 1],
                  [5, 3, 5, 3],
                  [-1, -1, -2, -1]], dtype=np.float32)
    ids, w = oracle.topk_softmax(L, 2)
    assert ids.tolist() == [[0, 1], [1, 2], [0, 2], [0, 1]]
    np.testing.assert_allclose(w[0], [0.5, 0.5])
    ids3, _ = oracle.topk_softmax(L, 3)
    assert ids3.tolist() == [[0, 1, 2], [1, 2, 3], [0, 2, 1], [0, 1, 3]]


def test_topk_k_equals_e_is_full_softmax_sorted():
    rng = np.random.default_rng(3)
    L = rng.standard_normal((10, 5)).astype(np.float32)
    ids, w = oracle.topk_softmax(L, 5)
    for t in range(10):
        assert sorted(ids[t].tolist()) == [0, 1, 2, 3, 4]
        z = np.exp(L[t].astype(np.float64))
        np.testing.assert_allclose(w[t], (z / z.sum())[ids[t]], rtol=1e-12)
        assert all(L[t, ids[t, k]] >= L[t, ids[t, k + 1]] for k in range(4))


@pytest.mark.parametrize("gates,theta,want_w,want_kept", [
    ([0.95, 0.05], 0.05, [0.95, 0.05], [True, True]),          # equal to the threshold: kept
    ([0.9501, 0.0499], 0.05, [1.0, 0.0], [True, False]),        # just below: dropped
    ([0.7, 0.2, 0.06, 0.04], 0.05, [0.7 / 0.96, 0.2 / 0.96, 0.06 / 0.96, 0.0],
     [True, True, True, False]),
    ([0.97, 0.01, 0.01, 0.01], 0.05, [1.0, 0.0, 0.0, 0.0], [True, False, False, False]),
    ([0.3, 0.25, 0.25, 0.2], 0.5, [1.0, 0.0, 0.0, 0.0], [True, False, False, False]),  # slot 0 kept
    ([0.6, 0.3, 0.1], 0.0, [0.6, 0.3, 0.1], [True, True, True]),  # threshold off
])
def test_gate_drop_hand_cases(gates, theta, want_w, want_kept):
    K = len(gates)
    ids = np.arange(K, dtype=np.int32)[None, :] + 3
    ids2, w2 = oracle.gate_drop(ids, np.array([gates]), theta)
    np.testing.assert_allclose(w2[0], want_w, rtol=0, atol=1e-15)
    assert [(i >= 0) for i in ids2[0]] == want_kept
    assert all(ids2[0, k] == ids[0, k] for k in range(K) if want_kept[k])


def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(math.log(3.0)) - 0.75 * math.log(3.0)) < 1e-15
    assert abs(oracle.silu(-math.log(3.0)) + 0.25 * math.log(3.0)) < 1e-15
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12
    assert abs(oracle.silu(-40.0)) < 1e-12


def test_swiglu_roles_by_hand():
    """H=3, I=2 expert whose every weight has a distinct, hand-checkable role."""
    a, b, c = math.log(3.0), 2.0, -1.5
    x = np.array([[a, b, c]])
    w_gate_up = np.array([
        [1.0, 0.0, 0.0],   # g0 = a
        [0.0, 0.0, 0.0],   # g1 = 0  -> h1 = 0 whatever u1 is
        [0.0, 1.0, 0.0],   # u0 = b
        [0.0, 0.0, 1.0],   # u1 = c
    ])
    w_down = np.array([
        [1.0, 7.0],
        [-2.0, 5.0],
        [0.0, 3.0],
    ])  # [H, I]: o_j = sum_i h_i * w_down[j, i]
    h0 = 0.75 * a * b
    o = oracle.swiglu_ffn(x, w_gate_up, w_down)
    np.testing.assert_allclose(o[0], [h0, -2.0 * h0, 0.0], rtol=0, atol=1e-15)


def test_single_expert_top1_is_dense_mlp_and_zero_gate_gives_zero():
    rng = np.random.default_rng(4)
    T, H, I = 7, 6, 5
    x = rng.standard_normal((T, H))
    wgu = rng.standard_normal((1, 2 * I, H))
    wd = rng.standard_normal((1, H, I))
    wr = rng.standard_normal((1, H))
    out = oracle.moe_layer(x, wr, wgu, wd, K=1)
    assert (out["ids"] == 0).all() and (out["w"] == 1.0).all()
    # dense MLP written as scalar loops from the definitions
    for t in range(T):
        h = []
        for i in range(I):
            g = sum(x[t, j] * wgu[0, i, j] for j in range(H))
            u = sum(x[t, j] * wgu[0, I + i, j] for j in range(H))
            h.append(g / (1.0 + math.exp(-g)) * u)
        want = [sum(h[i] * wd[0, j, i] for i in range(I)) for j in range(H)]
        np.testing.assert_allclose(out["y"][t], want, rtol=1e-12, atol=1e-12)
    wgu0 = wgu.copy()
    wgu0[:, :I, :] = 0.0
    assert np.abs(oracle.moe_layer(x, wr, wgu0, wd, K=1)["y"]).max() == 0.0


def test_empty_and_single_token():
    rng = np.random.default_rng(5)
    H, E, I = 8, 4, 3
    wgu = rng.standard_normal((E, 2 * I, H))
    wd = rng.standard_normal((E, H, I))
    wr = rng.standard_normal((E, H))
    out0 = oracle.moe_layer(np.zeros((0, H)), wr, wgu, wd, K=2)
    assert out0["y"].shape == (0, H)
    assert out0["counts"].tolist() == [0] * E and out0["offsets"].tolist() == [0] * (E + 1)
    x1 = rng.standard_normal((1, H))
    out1 = oracle.moe_layer(x1, wr, wgu, wd, K=2)
    assert int(out1["counts"].sum()) == 2
    e0, e1 = out1["ids"][0]
    want = (out1["w"][0, 0] * oracle.swiglu_ffn(x1, wgu[e0], wd[e0])
            + out1["w"][0, 1] * oracle.swiglu_ffn(x1, wgu[e1], wd[e1]))
    np.testing.assert_allclose(out1["y"], want, rtol=1e-13)


def test_all_tokens_to_one_expert_and_forced_empty_experts():
    rng = np.random.default_rng(6)
    T, H, E, I = 12, 8, 6, 4
    x = rng.standard_normal((T, H))
    wgu = rng.standard_normal((E, 2 * I, H))
    wd = rng.standard_normal((E, H, I))
    wr = rng.standard_normal((E, H)) * 0.01
    bias = np.array([0, -1e4, 50.0, -1e4, 0, -1e4], dtype=np.float32)
    out = oracle.moe_layer(x, wr, wgu, wd, K=1, router_bias=bias)
    assert out["counts"].tolist() == [0, 0, T, 0, 0, 0]
    out2 = oracle.moe_layer(x, wr, wgu, wd, K=2, router_bias=bias)
    assert out2["counts"][1] == out2["counts"][3] == out2["counts"][5] == 0
    assert out2["counts"][2] == T

"""Planted mistakes in the oracle (on the CPU) must be caught by its pins.

Each case replaces one oracle function with a plausible wrong variant (a dropped
term, a wrong sign, swapped operands, a reversed tie-break, an off-by-one) and
checks that at least one pin test then fails.
"""

import numpy as np
import pytest

import oracle
import oracle.moe_oracle as om
from tests import test_oracle_bruteforce as bf
from tests import test_oracle_fp8 as fp8_pins
from tests import test_oracle_pins as pins


def _patch(monkeypatch, name, fn):
    monkeypatch.setattr(om, name, fn)
    monkeypatch.setattr(oracle, name, fn)


def _silu_wrong_sign(z):
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(z))


def _swiglu_swapped(x_rows, w_gate_up, w_down):
    x = np.asarray(x_rows, dtype=np.float64)
    wgu = np.asarray(w_gate_up, dtype=np.float64)
    I = wgu.shape[0] // 2
    g = x @ wgu[I:].T
    u = x @ wgu[:I].T
    return (om.silu(g) * u) @ np.asarray(w_down, dtype=np.float64).T


def _swiglu_down_transposed(x_rows, w_gate_up, w_down):
    x = np.asarray(x_rows, dtype=np.float64)
    wgu = np.asarray(w_gate_up, dtype=np.float64)
    I = wgu.shape[0] // 2
    h = om.silu(x @ wgu[:I].T) * (x @ wgu[I:].T)
    wd = np.asarray(w_down, dtype=np.float64)
    return (h @ wd.reshape(wd.shape[1], wd.shape[0]))


def _combine_drops_last_slot(out_perm, inv, w, shared_out=None):
    inv = np.array(inv, copy=True)
    inv[:, -1] = -1
    return _orig_combine(out_perm, inv, w, shared_out)


def _topk_high_id_wins(logits32, K):
    L = np.asarray(logits32, dtype=np.float32).astype(np.float64)
    T, E = L.shape
    ids = np.empty((T, K), dtype=np.int32)
    w = np.empty((T, K))
    for t in range(T):
        order = np.lexsort((-np.arange(E), -L[t]))[:K]
        ids[t] = order
        z = np.exp(L[t, order] - L[t, order[0]])
        w[t] = z / z.sum()
    return ids, w


def _gate_drop_le(ids, w, theta):
    ids = np.array(ids, dtype=np.int32, copy=True)
    w = np.array(w, dtype=np.float64, copy=True)
    if theta <= 0:
        return ids, w
    for t in range(ids.shape[0]):
        for k in range(1, ids.shape[1]):
            if w[t, k] <= theta:
                ids[t, k], w[t, k] = -1, 0.0
        w[t] /= w[t].sum()
    return ids, w


def _gate_drop_no_renorm(ids, w, theta):
    ids = np.array(ids, dtype=np.int32, copy=True)
    w = np.array(w, dtype=np.float64, copy=True)
    if theta <= 0:
        return ids, w
    for t in range(ids.shape[0]):
        for k in range(1, ids.shape[1]):
            if w[t, k] < theta:
                ids[t, k], w[t, k] = -1, 0.0
    return ids, w


def _permute_offsets_inclusive(ids, E):
    counts, offsets, perm, inv = _orig_permute(ids, E)
    return counts, np.concatenate([offsets[1:], offsets[-1:]]), perm, inv


def _permute_tokens_descending(ids, E):
    ids = np.asarray(ids, dtype=np.int64)
    T, K = ids.shape
    tr = sorted(((int(ids[t, k]), -t, k) for t in range(T) for k in range(K) if ids[t, k] >= 0))
    counts = np.bincount([e for e, _, _ in tr], minlength=E).astype(np.int32)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    perm = np.array([-t for _, t, _ in tr], dtype=np.int32)
    inv = np.full((T, K), -1, dtype=np.int32)
    for r, (_, t, k) in enumerate(tr):
        inv[-t, k] = r
    return counts, offsets, perm, inv


_orig_combine = om.combine
_orig_permute = om.permute


def _all_pins(golden_dir):
    pins.test_worked_example_routing(golden_dir)
    pins.test_worked_example_dispatch(golden_dir)
    pins.test_worked_example_combine(golden_dir)
    pins.test_two_way_softmax_is_logistic()
    pins.test_topk_ties_go_to_lower_expert()
    for args in [([0.95, 0.05], 0.05, [0.95, 0.05], [True, True]),
                 ([0.7, 0.2, 0.06, 0.04], 0.05, [0.7 / 0.96, 0.2 / 0.96, 0.06 / 0.96, 0.0],
                  [True, True, True, False])]:
        pins.test_gate_drop_hand_cases(*args)
    pins.test_silu_closed_forms()
    pins.test_swiglu_roles_by_hand()
    pins.test_single_expert_top1_is_dense_mlp_and_zero_gate_gives_zero()
    bf.test_oracle_equals_dense_brute_force(9, 16, 8, 2, 16, 0.0, True, 0, 0)
    bf.test_oracle_equals_dense_brute_force(11, 12, 6, 4, 5, 0.2, True, 0, 0)


@pytest.mark.parametrize("name,bad", [
    ("silu", _silu_wrong_sign),
    ("swiglu_ffn", _swiglu_swapped),
    ("swiglu_ffn", _swiglu_down_transposed),
    ("combine", _combine_drops_last_slot),
    ("topk_softmax", _topk_high_id_wins),
    ("gate_drop", _gate_drop_le),
    ("gate_drop", _gate_drop_no_renorm),
    ("permute", _permute_offsets_inclusive),
    ("permute", _permute_tokens_descending),
])
def test_planted_mistake_is_caught(monkeypatch, golden_dir, name, bad):
    _all_pins(golden_dir)            # the real oracle passes every pin
    _patch(monkeypatch, name, bad)
    with pytest.raises(AssertionError):
        _all_pins(golden_dir)


# FP8 experts (P1 §4.1, 8-bit expert weights): plausible slips in applying the per-row and
# per-channel scales.  The unit-scale pins cannot see them; the hand-worked cases with
# distinct power-of-two scales and the dequantised-operand comparison must.

def _gate_up_fp8_divides_scales(x_codes, x_scale, w_codes, w_scale):
    acc = np.asarray(x_codes, np.float64) @ np.asarray(w_codes, np.float64).T
    acc = acc / np.asarray(x_scale, np.float64)[:, None] / np.asarray(w_scale, np.float64)[None, :]
    I = acc.shape[1] // 2
    return om.silu(acc[:, :I]) * acc[:, I:]


def _gate_up_fp8_gate_scales_on_up(x_codes, x_scale, w_codes, w_scale):
    ws = np.asarray(w_scale, np.float64)
    I = ws.shape[0] // 2
    ws = np.concatenate([ws[:I], ws[:I]])
    acc = (np.asarray(x_codes, np.float64) @ np.asarray(w_codes, np.float64).T) * \
        np.asarray(x_scale, np.float64)[:, None] * ws[None, :]
    return om.silu(acc[:, :I]) * acc[:, I:]


def _down_fp8_divides_scales(h_codes, h_scale, w_codes, w_scale):
    acc = np.asarray(h_codes, np.float64) @ np.asarray(w_codes, np.float64).T
    return acc / np.asarray(h_scale, np.float64)[:, None] / np.asarray(w_scale, np.float64)[None, :]


def _down_fp8_row_scale_per_channel(h_codes, h_scale, w_codes, w_scale):
    acc = np.asarray(h_codes, np.float64) @ np.asarray(w_codes, np.float64).T
    hs = np.resize(np.asarray(h_scale, np.float64), acc.shape[1])
    return acc * hs[None, :] * np.asarray(w_scale, np.float64)[None, :]


def _fp8_pins():
    fp8_pins.test_fp8_gate_up_reduces_to_plain_on_exact_operands()
    fp8_pins.test_fp8_down_reduces_to_plain_on_exact_operands()
    fp8_pins.test_fp8_gate_up_hand_worked()
    fp8_pins.test_fp8_down_hand_worked()
    fp8_pins.test_fp8_products_equal_plain_products_of_dequantised_operands()


@pytest.mark.parametrize("name,bad", [
    ("expert_gate_up_fp8", _gate_up_fp8_divides_scales),
    ("expert_gate_up_fp8", _gate_up_fp8_gate_scales_on_up),
    ("expert_down_fp8", _down_fp8_divides_scales),
    ("expert_down_fp8", _down_fp8_row_scale_per_channel),
])
def test_planted_fp8_scale_mistake_is_caught(monkeypatch, name, bad):
    _fp8_pins()                      # the real oracle passes every FP8 pin
    monkeypatch.setattr(om, name, bad)
    with pytest.raises(AssertionError):
        _fp8_pins()

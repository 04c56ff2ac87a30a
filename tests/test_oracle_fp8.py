"""Pins of the oracle's FP8 (E4M3) expert path: the quantiser against the format's
definition (hand values: representable numbers, ties to even, subnormals, saturation) and
against PyTorch's independent float8_e4m3fn conversion; the per-row scaling; and the FP8
gate/up, which must reduce to the plain gate/up when the operands are already E4M3 values
with unit scales.

Low-precision experts: P1 §4.1 quantises the resident experts' weights to 8 bits.
"""

import numpy as np
import pytest
import torch

from oracle import moe_oracle as oracle


def test_e4m3_hand_values():
    v = np.array([0.0, 1.0, -1.0, 448.0, 1.125, 1.0625, 1.1875, 2.0 ** -9, 2.0 ** -10,
                  3 * 2.0 ** -10, 300.0, 464.0, 1e6, -1e6, 2.0 ** -6, 0.013], dtype=np.float32)
    want = [0.0, 1.0, -1.0, 448.0, 1.125,
            1.0,      # 1.0625 is halfway between 1 and 1.125: ties to even (1.000)
            1.25,     # 1.1875 halfway between 1.125 and 1.25: to even (1.010)
            2.0 ** -9,  # smallest subnormal
            0.0,      # half of it: ties to even (zero)
            2.0 ** -8,  # 1.5 quanta: to even (2 quanta)
            288.0,    # spacing 32 above 256
            448.0,    # beyond the largest finite value: saturates
            448.0, -448.0,
            2.0 ** -6,  # smallest normal
            0.013671875]  # 7 subnormal quanta of 2^-9
    np.testing.assert_array_equal(oracle.quantize_e4m3(v), want)


def test_e4m3_matches_an_independent_conversion():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(20000) * 60, rng.standard_normal(20000) * 0.01,
                        rng.uniform(-448, 448, 20000)]).astype(np.float32)
    v = np.clip(v, -448, 448)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(oracle.quantize_e4m3(v), ref)
    # every E4M3 value is a fixed point
    allv = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    allv = allv[np.isfinite(allv)]
    np.testing.assert_array_equal(oracle.quantize_e4m3(allv.astype(np.float32)), allv)


def test_row_scaling():
    rng = np.random.default_rng(2)
    a = (rng.standard_normal((64, 300)) * rng.uniform(0.01, 10, (64, 1))).astype(np.float32)
    a[5] = 0.0
    codes, scale = oracle.quantize_rows_fp8(a)
    assert scale.dtype == np.float32 and scale[5] == 1.0 and (codes[5] == 0).all()
    np.testing.assert_array_equal(np.abs(codes).max(axis=1)[np.arange(64) != 5], 448.0)
    # E4M3 keeps 3 mantissa bits: relative error <= 2^-4 for normal codes; subnormal codes
    # (|code| < 2^-6) are within half a quantum, 2^-10, of the row's scaled value
    deq = codes * scale[:, None]
    err = np.abs(deq - a)
    bound = np.maximum(np.abs(a) * 2.0 ** -4, 2.0 ** -10 * scale[:, None]) * (1 + 1e-6)
    assert (err <= bound).all()


def test_fp8_gate_up_reduces_to_plain_on_exact_operands():
    rng = np.random.default_rng(3)
    x = oracle.quantize_e4m3((rng.standard_normal((40, 64)) * 0.5).astype(np.float32))
    w = oracle.quantize_e4m3((rng.standard_normal((2 * 24, 64)) * 0.5).astype(np.float32))
    h8 = oracle.expert_gate_up_fp8(x, np.ones(40, np.float32), w, np.ones(48, np.float32))
    np.testing.assert_allclose(h8, oracle.expert_gate_up(x, w), rtol=1e-15, atol=0)
    # scales multiply the gate and up pre-activations row- and column-wise
    sx = rng.uniform(0.5, 2, 40).astype(np.float32)
    sw = rng.uniform(0.5, 2, 48).astype(np.float32)
    g = (x @ w[:24].T) * sx[:, None] * sw[None, :24]
    u = (x @ w[24:].T) * sx[:, None] * sw[None, 24:]
    np.testing.assert_allclose(oracle.expert_gate_up_fp8(x, sx, w, sw), oracle.silu(g) * u,
                               rtol=1e-12)


def test_fp8_down_reduces_to_plain_on_exact_operands():
    rng = np.random.default_rng(4)
    h = oracle.quantize_e4m3((rng.standard_normal((30, 96)) * 2).astype(np.float32))
    w = oracle.quantize_e4m3((rng.standard_normal((40, 96)) * 2).astype(np.float32))
    np.testing.assert_allclose(
        oracle.expert_down_fp8(h, np.ones(30, np.float32), w, np.ones(40, np.float32)),
        oracle.expert_down(h, w), rtol=1e-15, atol=0)
    sh = rng.uniform(0.5, 2, 30).astype(np.float32)
    sw = rng.uniform(0.5, 2, 40).astype(np.float32)
    np.testing.assert_allclose(oracle.expert_down_fp8(h, sh, w, sw),
                               (h @ w.T) * sh[:, None] * sw[None, :], rtol=1e-12)

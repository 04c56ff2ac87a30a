"""Pins of the oracle's FP8 (E4M3) expert path: the quantiser against the format's
definition (hand values: representable numbers, ties to even, subnormals, saturation) and
against PyTorch's independent float8_e4m3fn conversion; the per-row scaling; and the FP8
gate/up, which must reduce to the plain gate/up when the operands are already E4M3 values
with unit scales; hand-worked FP8 gate/up and down cases with a distinct power-of-two
scale on every row and every output channel (each expected value written out below); and
the FP8 products against the plain float64 products of the dequantised operands.

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


# Hand-worked FP8 gate/up, I = 2, H = 4.  Every code is an E4M3 value and every scale a
# power of two, so each scaled dot product below is exact.
#   x codes  row 0: [1, 2, 0, -1]   scale 2
#            row 1: [0.5, 0, 3, 1]  scale 1/4
#   w codes  gate 0: [1, 0, 0, 0]  scale 1      gate 1: [0, 1, 1, 0]  scale 4
#            up 0:   [0, 0, 0, 1]  scale 1/2    up 1:   [2, 0, 0, 0]  scale 8
# Code dot products (row 0 / row 1): gate0 1 / 0.5, gate1 2 / 3, up0 -1 / 1, up1 2 / 1.
# Times the row scale and the channel scale:
#   g = [[2*1*1, 2*4*2], [0.25*1*0.5, 0.25*4*3]]     = [[2, 16], [0.125, 3]]
#   u = [[2*0.5*-1, 2*8*2], [0.25*0.5*1, 0.25*8*1]]  = [[-1, 32], [0.125, 2]]
# h = silu(g) * u with silu(z) = z / (1 + e^-z), where e^-2 = 0.1353352832366127,
# e^-16 = 1.1253517471925912e-07, e^-0.125 = 0.8824969025845955, e^-3 = 0.049787068367863944:
#   silu(2) = 1.7615941559557646, silu(16) = 15.999998199437407,
#   silu(0.125) = 0.0664011716717195, silu(3) = 2.8577223804673.
_GU_X = np.array([[1, 2, 0, -1], [0.5, 0, 3, 1]], np.float64)
_GU_SX = np.array([2, 0.25], np.float32)
_GU_W = np.array([[1, 0, 0, 0], [0, 1, 1, 0], [0, 0, 0, 1], [2, 0, 0, 0]], np.float64)
_GU_SW = np.array([1, 4, 0.5, 8], np.float32)
_GU_H = np.array([[1.7615941559557646 * -1, 15.999998199437407 * 32],
                  [0.0664011716717195 * 0.125, 2.8577223804673 * 2]])


def test_fp8_gate_up_hand_worked():
    np.testing.assert_allclose(oracle.expert_gate_up_fp8(_GU_X, _GU_SX, _GU_W, _GU_SW), _GU_H,
                               rtol=1e-12, atol=0)


# Hand-worked FP8 down projection, I = 4, H = 3.
#   h codes row 0: [1, -2, 0, 0.5]  scale 1/2     row 1: [0, 1, 1, 1]  scale 4
#   w codes out 0: [1, 1, 0, 0]  scale 2;  out 1: [0, 0, 4, 2]  scale 1/8;  out 2: [2, 0, 0, 1]  scale 1
# Code dot products: row 0 -> [-1, 1, 2.5], row 1 -> [1, 6, 1].
#   o[0] = 0.5 * [2*-1, 0.125*1, 1*2.5] = [-1, 0.0625, 1.25]
#   o[1] = 4 * [2*1, 0.125*6, 1*1]      = [8, 3, 4]
def test_fp8_down_hand_worked():
    h = np.array([[1, -2, 0, 0.5], [0, 1, 1, 1]], np.float64)
    w = np.array([[1, 1, 0, 0], [0, 0, 4, 2], [2, 0, 0, 1]], np.float64)
    o = oracle.expert_down_fp8(h, np.array([0.5, 4], np.float32), w,
                               np.array([2, 0.125, 1], np.float32))
    np.testing.assert_array_equal(o, [[-1, 0.0625, 1.25], [8, 3, 4]])


def test_fp8_products_equal_plain_products_of_dequantised_operands():
    """Quantise real rows, then compare the FP8 products with the plain float64 gate/up and
    down of the dequantised operands (codes * scale, applied to each operand before the
    product): the scales may be moved out of the dot products only if they multiply."""
    rng = np.random.default_rng(5)
    xq, sx = oracle.quantize_rows_fp8(rng.standard_normal((24, 64)).astype(np.float32) *
                                      rng.uniform(0.1, 8, (24, 1)).astype(np.float32))
    wq, sw = oracle.quantize_rows_fp8(rng.standard_normal((40, 64)).astype(np.float32) *
                                      rng.uniform(0.01, 0.5, (40, 1)).astype(np.float32))
    x_deq = xq * sx.astype(np.float64)[:, None]
    w_deq = wq * sw.astype(np.float64)[:, None]
    np.testing.assert_allclose(oracle.expert_gate_up_fp8(xq, sx, wq, sw),
                               oracle.expert_gate_up(x_deq, w_deq), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(oracle.expert_down_fp8(xq, sx, wq, sw),
                               oracle.expert_down(x_deq, w_deq), rtol=1e-12, atol=1e-15)

"""Pins for the oracle's input gradient of the layer, dL/dx = U^^H g + W^^T conj(g).

Sources: "Fairy2i-W2" model card, "Widely-linear transformation" (y = Ux + W
conj(x)) and the quantization-aware training paragraph of "Fairy2i:
Ultra-Low-Bit LLM Quantization Using Complex Weights {±1, ±i}" (training
through the quantized layer with the straight-through estimator, which needs
the gradient with respect to the layer input).

The gradient is pinned to the forward evaluation (itself pinned in
test_oracle_linear.py) by the adjoint identity, and to the real form of the
layer (the inverse of Theorem 1: R11 = Re U + Re W, R12 = Im W - Im U,
R21 = Im U + Im W, R22 = Re U - Re W) by a plain transpose.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_complex_valued_fairy2i_b300 import inputs

CASES = [(8, 12, 1, 1), (16, 40, 2, 3), (33, 17, 3, 2), (5, 70, 4, 1)]


def _bf16(x: np.ndarray) -> np.ndarray:
    return inputs.bf16_bits(torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16))


def _layer(n, m, T, seed):
    R = np.random.default_rng(seed).normal(0, 0.02, (2 * n, 2 * m)).astype(np.float32)
    U, W = oracle.convert_f32(R)
    return oracle.quantize(U, T), oracle.quantize(W, T)


def _g(M, n, seed):
    return np.random.default_rng(seed).normal(size=(M, 2 * n)).astype(np.float32)


@pytest.mark.parametrize("n,m,T,M", CASES)
def test_adjoint_identity_with_the_forward(n, m, T, M):
    """<y(x), g> = <x, dL/dx(g)> over the real vectors [Re | Im]."""
    qU, qW = _layer(n, m, T, 10 * n + m)
    x = _bf16(np.random.default_rng(2).normal(size=(M, 2 * m)))
    g = _g(M, n, 3)
    y = oracle.linear_mulfree(qU, qW, x)
    gx = oracle.linear_grad_x_mulfree(qU, qW, g)
    xf = oracle.bf16_bits_to_f64(x)
    lhs = np.sum(y * g.astype(np.float64), axis=1)
    rhs = np.sum(xf * gx, axis=1)
    scale = np.linalg.norm(y, axis=1) * np.linalg.norm(g, axis=1)
    assert np.all(np.abs(lhs - rhs) <= 1e-12 * scale)


@pytest.mark.parametrize("n,m,T,M", CASES)
def test_mulfree_equals_dense(n, m, T, M):
    qU, qW = _layer(n, m, T, n + 7 * m)
    g = _g(M, n, 4)
    a = oracle.linear_grad_x_mulfree(qU, qW, g)
    b = oracle.linear_grad_x_dense(oracle.dequantize(qU.codes, qU.scales),
                                   oracle.dequantize(qW.codes, qW.scales), g)
    assert np.linalg.norm(a - b) <= 1e-12 * np.linalg.norm(b)


@pytest.mark.parametrize("n,m,T", [(6, 9, 1), (12, 20, 2)])
def test_equals_transpose_of_real_form(n, m, T):
    qU, qW = _layer(n, m, T, 5 * n + m)
    Uh = oracle.dequantize(qU.codes, qU.scales)
    Wh = oracle.dequantize(qW.codes, qW.scales)
    R = np.block([[Uh.real + Wh.real, Wh.imag - Uh.imag],
                  [Uh.imag + Wh.imag, Uh.real - Wh.real]])
    g = _g(2, n, 5)
    gx = oracle.linear_grad_x_mulfree(qU, qW, g)
    want = g.astype(np.float64) @ R  # rows of (R^T g)
    assert np.linalg.norm(gx - want) <= 1e-12 * np.linalg.norm(want)


def test_u_only_single_stage_is_conjugate_transpose_product():
    n, m = 7, 11
    qU, qW = _layer(n, m, 1, 77)
    qW.scales[...] = 0.0  # W contributes nothing
    Uh = oracle.dequantize(qU.codes, qU.scales)
    g = _g(1, n, 6)
    gc = g[0, :n].astype(np.float64) + 1j * g[0, n:]
    want = np.conj(Uh).T @ gc
    gx = oracle.linear_grad_x_mulfree(qU, qW, g)[0]
    assert np.allclose(gx[:m], want.real, rtol=0, atol=1e-12)
    assert np.allclose(gx[m:], want.imag, rtol=0, atol=1e-12)


def test_single_code_each_kind():
    """One nonzero code per matrix, checked against the hand-derived value of
    conj(c) g (U) and c conj(g) (W) for c in {+1, -1, +i, -i}."""
    n, m, T = 1, 1, 1
    g = np.array([[0.75, -1.25]], np.float32)  # g = 0.75 - 1.25 i
    gc = 0.75 - 1.25j
    for code, c in enumerate((1, -1, 1j, -1j)):
        for X in range(2):
            codes = np.zeros((T, n, m), np.uint8)
            codes[0, 0, 0] = code
            scales = np.zeros((T, 2, n), np.float32)
            scales[0, 0 if code < 2 else 1, 0] = 0.5
            zero = oracle.Quantized(np.zeros((T, n, m), np.uint8), np.zeros((T, 2, n), np.float32), None, None)
            q = oracle.Quantized(codes, scales, None, None)
            qU, qW = (q, zero) if X == 0 else (zero, q)
            gx = oracle.linear_grad_x_mulfree(qU, qW, g)[0]
            want = np.conj(0.5 * c) * gc if X == 0 else 0.5 * c * np.conj(gc)
            assert gx[0] == pytest.approx(want.real, abs=0) and gx[1] == pytest.approx(want.imag, abs=0)

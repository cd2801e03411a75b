"""Pins for the oracle's layer evaluation y = U^ x + W^ conj(x).

Sources: "Fairy2i-W2" model card, "Widely-linear transformation" (y = Ux + W
conj(x)); "Fairy2i: Ultra-Low-Bit LLM Quantization Using Complex Weights
{±1, ±i}", "Industry implications: multiplication-free inference" (adds,
subtracts, re/im swaps); "The 2-bit complex model rivals full precision ..."
(36kr), the multiplication-free paragraph.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_complex_valued_fairy2i_b300 import inputs


def _bf16(x: np.ndarray) -> np.ndarray:
    return inputs.bf16_bits(torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16))


def _layer(n, m, T, seed):
    R = np.random.default_rng(seed).normal(0, 0.02, (2 * n, 2 * m)).astype(np.float32)
    U, W = oracle.convert_f32(R)
    return R, U, W, oracle.quantize(U, T), oracle.quantize(W, T)


def _xc(xbits):
    xf = oracle.bf16_bits_to_f64(xbits)
    m = xf.shape[1] // 2
    return xf[:, :m] + 1j * xf[:, m:]


@pytest.mark.parametrize("n,m,T,M", [(8, 12, 1, 1), (16, 40, 2, 3), (33, 17, 3, 2)])
def test_mulfree_equals_dense_dequantized(n, m, T, M):
    _, _, _, qU, qW = _layer(n, m, T, n + m)
    x = _bf16(np.random.default_rng(1).normal(size=(M, 2 * m)))
    y1 = oracle.linear_mulfree(qU, qW, x)
    y2 = oracle.linear_dense(oracle.dequantize(qU.codes, qU.scales),
                             oracle.dequantize(qW.codes, qW.scales), x)
    assert np.linalg.norm(y1 - y2) <= 1e-12 * np.linalg.norm(y2)


def test_dense_matches_numpy_complex_matmul():
    n, m, T, M = 12, 20, 2, 4
    _, _, _, qU, qW = _layer(n, m, T, 99)
    x = _bf16(np.random.default_rng(2).normal(size=(M, 2 * m)))
    Uh = oracle.dequantize(qU.codes, qU.scales)
    Wh = oracle.dequantize(qW.codes, qW.scales)
    xc = _xc(x)
    want = xc @ Uh.T + np.conj(xc) @ Wh.T
    got = oracle.linear_mulfree(qU, qW, x)
    np.testing.assert_allclose(got[:, :n], want.real, rtol=0, atol=1e-12)
    np.testing.assert_allclose(got[:, n:], want.imag, rtol=0, atol=1e-12)


def test_real_form_of_the_quantized_layer():
    """Rebuild the real 2n x 2m matrix from U^, W^ by the inverse block map
    and apply it to the real activation row [Re x | Im x]."""
    n, m, T = 10, 14, 2
    _, _, _, qU, qW = _layer(n, m, T, 5)
    Uh = oracle.dequantize(qU.codes, qU.scales)
    Wh = oracle.dequantize(qW.codes, qW.scales)
    Rh = np.block([[Uh.real + Wh.real, Wh.imag - Uh.imag],
                   [Uh.imag + Wh.imag, Uh.real - Wh.real]])
    x = _bf16(np.random.default_rng(3).normal(size=(2, 2 * m)))
    want = oracle.bf16_bits_to_f64(x) @ Rh.T
    got = oracle.linear_mulfree(qU, qW, x)
    assert np.linalg.norm(got - want) <= 1e-12 * np.linalg.norm(want)


def test_quantized_layer_approximates_real_layer():
    """At T = 3 the quantized layer tracks R x~ (rel-L2 well below 1)."""
    n, m, T = 64, 64, 3
    R, _, _, qU, qW = _layer(n, m, T, 17)
    x = _bf16(np.random.default_rng(4).normal(size=(4, 2 * m)))
    want = oracle.bf16_bits_to_f64(x) @ R.astype(np.float64).T
    got = oracle.linear_mulfree(qU, qW, x)
    assert np.linalg.norm(got - want) / np.linalg.norm(want) < 0.4


def test_u_only_layer_is_a_complex_matvec():
    """W = 0: every W code is +1 with scale 0, y = U^ x exactly."""
    n, m = 7, 9
    _, U, _, qU, _ = _layer(n, m, 1, 8)
    qW = oracle.quantize(np.zeros((n, m), np.complex64), 1)
    x = _bf16(np.random.default_rng(5).normal(size=(1, 2 * m)))
    y = oracle.linear_mulfree(qU, qW, x)
    want = oracle.dequantize(qU.codes, qU.scales) @ _xc(x)[0]
    np.testing.assert_allclose(y[0, :n], want.real, atol=1e-13)
    np.testing.assert_allclose(y[0, n:], want.imag, atol=1e-13)


def test_lossless_codebook_layer_equals_exact_widely_linear_map():
    """U, W on the codebook => one stage is exact and the layer equals
    U x + W conj(x) computed by numpy.  A wrong conjugation or a swapped
    re/im sign anywhere in the epilogue fails this."""
    rng = np.random.default_rng(11)
    n, m = 5, 16

    def on_codebook():
        c = rng.uniform(0.1, 1, n).astype(np.float32)
        d = rng.uniform(0.1, 1, n).astype(np.float32)
        codes = rng.integers(0, 4, (n, m))
        return np.choose(codes, [c[:, None] + 0j, -c[:, None] + 0j,
                                 1j * d[:, None], -1j * d[:, None]]).astype(np.complex64)

    U, W = on_codebook(), on_codebook()
    qU, qW = oracle.quantize(U, 1), oracle.quantize(W, 1)
    x = _bf16(rng.normal(size=(3, 2 * m)))
    xc = _xc(x)
    want = xc @ U.astype(np.complex128).T + np.conj(xc) @ W.astype(np.complex128).T
    got = oracle.linear_mulfree(qU, qW, x)
    np.testing.assert_allclose(got[:, :n], want.real, atol=1e-12)
    np.testing.assert_allclose(got[:, n:], want.imag, atol=1e-12)


def test_bf16_widening_matches_torch():
    v = torch.randn(1000).to(torch.bfloat16)
    bits = inputs.bf16_bits(v)
    assert np.array_equal(oracle.bf16_bits_to_f64(bits), v.to(torch.float64).numpy())


def test_zero_tokens():
    _, _, _, qU, qW = _layer(4, 4, 1, 1)
    y = oracle.linear_mulfree(qU, qW, np.zeros((0, 8), np.uint16))
    assert y.shape == (0, 8)

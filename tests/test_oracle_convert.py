"""Pins for the oracle's widely-linear conversion (Theorem 1).

Source: "Fairy2i: Ultra-Low-Bit LLM Quantization Using Complex Weights {±1, ±i}",
Step 1 (Theorem 1 and its block formulas); "Fairy2i-W2" model card,
"Widely-linear transformation" (y = Ux + W conj(x), lossless and unique).
Each test checks the oracle against a fact fixed by the pages or by linear
algebra, never against a retyped copy of the block formulas.
"""
import numpy as np
import pytest

import oracle


def _R(n, m, seed, std=0.02):
    return np.random.default_rng(seed).normal(0.0, std, (2 * n, 2 * m)).astype(np.float32)


def _realform(y):
    return np.concatenate([y.real, y.imag], axis=-1)


@pytest.mark.parametrize("n,m", [(1, 1), (3, 5), (16, 8), (33, 47)])
def test_theorem1_equivalence(n, m):
    """R [Re x; Im x] == realform(U x + W conj(x)) to 1e-12 (fp64)."""
    R = _R(n, m, 1 + n * m)
    U, W = oracle.convert_f64(R)
    rng = np.random.default_rng(7)
    for _ in range(4):
        x = rng.normal(size=m) + 1j * rng.normal(size=m)
        ref = R.astype(np.float64) @ np.concatenate([x.real, x.imag])
        got = _realform(U @ x + W @ np.conj(x))
        assert np.linalg.norm(got - ref) <= 1e-12 * np.linalg.norm(ref)


def test_theorem1_is_not_the_interleaved_stacking():
    """The halves stacking is the one under which the formulas hold: with an
    interleaved real vector the same U, W do not reproduce R."""
    n, m = 4, 6
    R = _R(n, m, 3)
    U, W = oracle.convert_f64(R)
    x = np.random.default_rng(1).normal(size=m) + 1j * np.random.default_rng(2).normal(size=m)
    inter = np.empty(2 * m)
    inter[0::2], inter[1::2] = x.real, x.imag
    ref_inter = R.astype(np.float64) @ inter
    got = _realform(U @ x + W @ np.conj(x))
    assert np.linalg.norm(got - ref_inter) > 1e-3 * np.linalg.norm(ref_inter)


def test_inverse_map_reproduces_R_exactly():
    """Lossless: R11 = ReU+ReW, R12 = ImW-ImU, R21 = ImU+ImW, R22 = ReU-ReW."""
    n, m = 9, 13
    R = _R(n, m, 11)
    U, W = oracle.convert_f64(R)
    back = np.block([[U.real + W.real, W.imag - U.imag],
                     [U.imag + W.imag, U.real - W.real]])
    assert np.array_equal(back, R.astype(np.float64))


def test_textbook_complex_matrix_gives_W_zero():
    """R = [[A, -B], [B, A]] is the real form of A + iB: W = 0, U = A + iB."""
    rng = np.random.default_rng(5)
    A = rng.normal(size=(6, 7)).astype(np.float32)
    B = rng.normal(size=(6, 7)).astype(np.float32)
    R = np.block([[A, -B], [B, A]])
    U, W = oracle.convert_f64(R)
    assert np.array_equal(W, np.zeros_like(W))
    assert np.array_equal(U, A.astype(np.float64) + 1j * B.astype(np.float64))


def test_conjugate_linear_matrix_gives_U_zero():
    """R = [[A, B], [B, -A]] is x -> (A + iB) conj(x): U = 0, W = A + iB."""
    rng = np.random.default_rng(6)
    A = rng.normal(size=(5, 4)).astype(np.float32)
    B = rng.normal(size=(5, 4)).astype(np.float32)
    R = np.block([[A, B], [B, -A]])
    U, W = oracle.convert_f64(R)
    assert np.array_equal(U, np.zeros_like(U))
    assert np.array_equal(W, A.astype(np.float64) + 1j * B.astype(np.float64))


def test_identity():
    R = np.eye(10, dtype=np.float32)
    U, W = oracle.convert_f64(R)
    assert np.array_equal(U, np.eye(5))
    assert np.array_equal(W, np.zeros((5, 5)))


def test_float32_mode_is_the_rounded_exact_result():
    """Sum-then-halve in float32 equals the exact result rounded once."""
    n, m = 32, 40
    R = _R(n, m, 21)
    U64, W64 = oracle.convert_f64(R)
    U32, W32 = oracle.convert_f32(R)
    for a, b in ((U32, U64), (W32, W64)):
        assert np.array_equal(a.real, b.real.astype(np.float32))
        assert np.array_equal(a.imag, b.imag.astype(np.float32))


def test_conversion_is_linear_and_injective():
    """Uniqueness: the map is linear, and a nonzero R never maps to (0, 0)."""
    n, m = 3, 4
    rng = np.random.default_rng(8)
    for _ in range(20):
        R = np.zeros((2 * n, 2 * m), np.float32)
        R[rng.integers(2 * n), rng.integers(2 * m)] = 1.0
        U, W = oracle.convert_f64(R)
        assert np.count_nonzero(U) + np.count_nonzero(W) == 2

"""Pins for the oracle's phase-aware recursive residual quantizer.

Sources: "Fairy2i: Ultra-Low-Bit LLM Quantization Using Complex Weights {±1, ±i}",
Step 2 (b(w) = argmax Re(w conj(s)), axis-wise scales, dequantization) and
Step 3 (R^(t+1) = R^(t) - W~^(t)); "Fairy2i-W2" model card, "Phase-aware complex
quantization" and "Recursive residual quantization".
"""
import math
import os

import numpy as np
import pytest

import oracle

CODEBOOK = (1 + 0j, -1 + 0j, 1j, -1j)


def _brute_force_code(w: complex) -> int:
    """Independent restatement with Python complex numbers: first maximum."""
    vals = [(w * s.conjugate()).real for s in CODEBOOK]
    best = 0
    for c in range(1, 4):
        if vals[c] > vals[best]:
            best = c
    return best


def test_projection_brute_force_all_small_values():
    """Every complex value with parts in {0, -0, +-1, +-2}: all tie cases occur."""
    parts = [0.0, -0.0, 1.0, -1.0, 2.0, -2.0]
    vals = [complex(a, b) for a in parts for b in parts]
    Z = np.array(vals, dtype=np.complex64).reshape(6, 6)
    # keep signed zeros: build the float pairs directly
    Zp = np.array([[a, b] for a in parts for b in parts], np.float32).reshape(6, 6, 2)
    Zc = Zp.view(np.complex64)[..., 0]
    q = oracle.quantize(Zc, 1)
    for idx, w in enumerate(vals):
        assert q.codes[0].reshape(-1)[idx] == _brute_force_code(w), w
    assert Z.shape == (6, 6)


def test_projection_brute_force_random_tiny_matrices():
    rng = np.random.default_rng(0)
    for shape in [(1, 1), (2, 3), (4, 4), (3, 1)]:
        vals = rng.integers(-2, 3, size=shape + (2,)).astype(np.float32)
        Zc = np.ascontiguousarray(vals).view(np.complex64)[..., 0]
        q = oracle.quantize(Zc, 1)
        for idx in np.ndindex(shape):
            assert q.codes[0][idx] == _brute_force_code(complex(Zc[idx]))


def test_projection_golden_ties(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "projection_ties.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                re_s, im_s, code_s = line.split()
                rows.append((float(re_s), float(im_s), int(code_s)))
    Zp = np.array([[r, i] for r, i, _ in rows], np.float32).reshape(1, len(rows), 2)
    q = oracle.quantize(Zp.view(np.complex64)[..., 0], 1)
    assert list(q.codes[0, 0]) == [c for _, _, c in rows]


def _read_worked(golden_dir):
    d = {}
    with open(os.path.join(golden_dir, "worked_example_1x4.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                k, *v = line.split()
                d[k] = [float(t) for t in v]
    return d


def test_worked_example(golden_dir):
    d = _read_worked(golden_dir)
    U = (np.array(d["u_re"], np.float32) + 1j * np.array(d["u_im"], np.float32)).astype(np.complex64)
    q = oracle.quantize(U[None, :], 2, keep_residuals=True)
    assert list(q.codes[0, 0]) == [int(c) for c in d["codes0"]]
    assert list(q.codes[1, 0]) == [int(c) for c in d["codes1"]]
    np.testing.assert_allclose(q.scales[0, :, 0], d["scales0"], rtol=1e-6)
    np.testing.assert_allclose(q.scales[1, :, 0], d["scales1"], rtol=1e-6)
    np.testing.assert_allclose(q.resid[2, 0].real, d["r2_re"], atol=1e-6)
    np.testing.assert_allclose(q.resid[2, 0].imag, d["r2_im"], atol=1e-6)
    # layer with W = 0 and x = e_0 returns the dequantized U[0]
    qW = oracle.quantize(np.zeros((1, 4), np.complex64), 2)
    x = np.zeros((1, 8), np.uint16)
    x[0, 0] = 0x3F80  # bfloat16 1.0
    y = oracle.linear_mulfree(q, qW, x)
    np.testing.assert_allclose(y[0], d["y_e0"], rtol=1e-6)


def _stats_matrix(n=256, m=256, seed=20251203 + 1000):
    """Config-1-like U: convert of R ~ N(0, 0.02^2)."""
    R = np.random.default_rng(seed).normal(0, 0.02, (2 * n, 2 * m)).astype(np.float32)
    U, W = oracle.convert_f32(R)
    return U, W


def test_scale_integer_rule_matches_plain_mean():
    """|s - mean| <= 2^(e-48) (truncation) + half an ulp of float32."""
    U, _ = _stats_matrix(64, 300)
    q = oracle.quantize(U, 3, keep_residuals=True)
    for t in range(3):
        for ax in range(2):
            s = q.scales[t, ax].astype(np.float64)
            mu = q.mean64[t, ax]
            r = q.resid[t]
            comp = r.real if ax == 0 else r.imag
            on = (q.codes[t] <= 1) if ax == 0 else (q.codes[t] >= 2)
            vmax = np.where(on, np.abs(comp), 0).max(axis=1).astype(np.float64)
            e = np.floor(np.log2(np.where(vmax > 0, vmax, 1.0)))
            bound = 2.0 ** (e - 48) + np.abs(mu) * 2.0 ** -24
            assert np.all(np.abs(s - mu) <= bound)


def test_scale_rule_adversarial_spread():
    """One large value and many tiny ones on the same axis."""
    m = 2000
    re = np.full(m, 1e-7, np.float32)
    re[0] = 3.0
    Z = (re + 1j * np.zeros(m, np.float32)).astype(np.complex64)[None, :]
    q = oracle.quantize(Z, 1, keep_residuals=True)
    exact = (3.0 + (m - 1) * float(np.float32(1e-7))) / m
    assert abs(q.scales[0, 0, 0] - exact) <= 2.0 ** (1 - 48) + exact * 2.0 ** -24
    assert q.scales[0, 1, 0] == 0.0  # empty imaginary axis


def test_scale_is_least_squares_optimal_given_codes():
    """s minimises sum (|v| - s)^2 over the axis: f(s) < f(s(1 +- 1e-3))."""
    U, _ = _stats_matrix(32, 128)
    q = oracle.quantize(U, 2, keep_residuals=True)
    for t in range(2):
        for ax in range(2):
            comp = q.resid[t].real if ax == 0 else q.resid[t].imag
            on = (q.codes[t] <= 1) if ax == 0 else (q.codes[t] >= 2)
            for j in range(U.shape[0]):
                v = np.abs(comp[j][on[j]]).astype(np.float64)
                s = float(q.scales[t, ax, j])
                f = lambda z: float(((v - z) ** 2).sum())  # noqa: E731
                assert f(s) < f(s * (1 + 1e-3)) and f(s) < f(s * (1 - 1e-3))


def test_closed_form_statistics_gaussian_weights():
    """R iid N(0, sigma^2) => U circular Gaussian, Re/Im iid N(0, sigma^2/2):
       P(real-coded) = 1/2; E[stage-0 scale] = (sigma/sqrt 2) * 2/sqrt(pi);
       ||r^(1)||^2 / ||U||^2 -> 1 - 2/pi."""
    U, W = _stats_matrix()
    for Z in (U, W):
        q = oracle.quantize(Z, 1, keep_residuals=True)
        frac_real = float(np.mean(q.codes[0] <= 1))
        assert abs(frac_real - 0.5) < 0.01
        expected = 0.02 / math.sqrt(2) * 2 / math.sqrt(math.pi)  # 0.015958
        for ax in range(2):
            assert abs(float(q.scales[0, ax].mean()) / expected - 1) < 0.01
        ratio = float(np.sum(np.abs(q.resid[1].astype(np.complex128)) ** 2)
                      / np.sum(np.abs(Z.astype(np.complex128)) ** 2))
        assert abs(ratio - (1 - 2 / math.pi)) < 0.01


def test_residual_recursion_and_telescoping():
    """r^(t+1) = r^(t) - W~^(t) in float32; sum_t W~^(t) + r^(T) = Z; the
    residual norm never grows (s = 0 is feasible and s is optimal)."""
    U, _ = _stats_matrix(48, 96)
    T = 4
    q = oracle.quantize(U, T, keep_residuals=True)
    total = np.zeros(U.shape, np.complex128)
    prev = np.inf
    for t in range(T):
        stage = oracle.dequantize(q.codes[t:t + 1], q.scales[t:t + 1])
        total += stage
        r, r1 = q.resid[t], q.resid[t + 1]
        want_re = (r.real - stage.real.astype(np.float32)).astype(np.float32)
        want_im = (r.imag - stage.imag.astype(np.float32)).astype(np.float32)
        assert np.array_equal(r1.real, want_re) and np.array_equal(r1.imag, want_im)
        norm = float(np.linalg.norm(r1.astype(np.complex128)))
        assert norm <= prev
        prev = norm
    recon = total + q.resid[T].astype(np.complex128)
    assert np.max(np.abs(recon - U.astype(np.complex128))) < 1e-7


def test_stages_reduce_error():
    U, _ = _stats_matrix(64, 128)
    errs = []
    for T in (1, 2, 3):
        q = oracle.quantize(U, T)
        errs.append(np.linalg.norm(oracle.dequantize(q.codes, q.scales) - U))
    assert errs[0] > errs[1] > errs[2]


def test_lossless_on_codebook_values():
    """Rows whose entries are exactly +-c_j or +-i d_j are reproduced by one
    stage: the scales are c_j, d_j and the residual is exactly zero."""
    rng = np.random.default_rng(3)
    n, m = 6, 20
    c = rng.uniform(0.1, 1.0, n).astype(np.float32)
    d = rng.uniform(0.1, 1.0, n).astype(np.float32)
    codes = rng.integers(0, 4, (n, m))
    codes[:, 0], codes[:, 1] = 0, 2  # both axes non-empty
    vals = np.choose(codes, [c[:, None] + 0j, -c[:, None] + 0j, 1j * d[:, None], -1j * d[:, None]])
    Z = vals.astype(np.complex64)
    q = oracle.quantize(Z, 2, keep_residuals=True)
    assert np.array_equal(q.codes[0], codes)
    assert np.array_equal(q.scales[0, 0], c) and np.array_equal(q.scales[0, 1], d)
    assert not np.any(q.resid[1])
    # second stage of an all-zero residual: every code +1, every scale 0
    assert np.all(q.codes[1] == 0) and not np.any(q.scales[1])


def test_nonfinite_rejected():
    Z = np.zeros((2, 3), np.complex64)
    Z[1, 2] = np.nan
    with pytest.raises(oracle.NonFiniteInput):
        oracle.quantize(Z, 1)
    Z[1, 2] = np.inf
    with pytest.raises(oracle.NonFiniteInput):
        oracle.quantize(Z, 1)


def test_scale_rounding_golden(golden_dir):
    """Hand-derived scales at float32 rounding boundaries (normal and
    subnormal); pins the 48-bit integer mean and the round-to-nearest-even."""
    with open(os.path.join(golden_dir, "scale_rounding.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            name, *vals = line.split()
            re = np.array([float(v) for v in vals[:-1]], np.float32)
            want = np.float32(float(vals[-1]))
            Z = (re + 1j * np.zeros_like(re)).astype(np.complex64)[None, :]
            q = oracle.quantize(Z, 1)
            assert q.scales[0, 0, 0] == want, name

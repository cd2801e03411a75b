"""GPU parity of the fp16 form of the dequantized GEMM (FAIRY2I_ALGO_TCGEN05_DQ16) on
layout 3, through the C ABI, against the oracle's exact sum.

The form rounds each entry of the summed real matrix (its row scaled by a power of two)
once to fp16, relative error at most 2^-11 = 4.9e-4 per entry, and carries every
activation exactly (a bfloat16 value scaled by a power of two into the fp16 range); the
products are exact and summed in fp32.  The output error relative to the exact sum is a
weighted mean of the entries' relative errors, so it stays below 2^-11 plus the fp32
summation error: bar 6e-4 (measured values are near 2.8e-4, the mean of a uniform
rounding error), inside the layer's 1e-3.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import bit_complex_valued_fairy2i_b300 as f2i
from bit_complex_valued_fairy2i_b300 import inputs

pytestmark = pytest.mark.gpu

DQ16_REL_L2 = 6e-4
L3 = f2i.LAYOUT_LUT
SHAPES = [(8, 64), (37, 136), (33, 200), (256, 256), (300, 704), (64, 1024), (40, 320), (130, 2056)]


def rel_l2(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


def _R(n, m, seed):
    return inputs.weight_R(97, seed, 2 * n, 2 * m)


def _x(M, m, seed, outliers=False):
    return inputs.activations(97, seed, M, 2 * m, outliers=outliers)


def _layer(R, T):
    """(GPU layout-3 layer, oracle U and W layers) of a real weight R."""
    U, W = f2i.convert(R.cuda())
    q = f2i.quantize(U, W, T, layout=L3)
    Uo, Wo = oracle.convert_f32(R.numpy())
    return q, oracle.quantize(Uo, T), oracle.quantize(Wo, T)


@pytest.mark.parametrize("n,m", SHAPES)
@pytest.mark.parametrize("M", [1, 7, 40, 130, 256, 300, 513])  # N = 16, 16, 48, 144, 256, 256 (x2), 256 (x2)
def test_dq16_parity(n, m, M):
    q, qU, qW = _layer(_R(n, m, 11 * n + m), 2)
    x = _x(M, m, n + 3 * m)
    y = f2i.linear(q, x.cuda(), algo="tcgen05_dq16").cpu().numpy()
    err = rel_l2(y, oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x)))
    assert err <= DQ16_REL_L2, err


@pytest.mark.parametrize("T", [1, 3, 4])
@pytest.mark.parametrize("M", [40, 300])  # one token tile of 48; two of 256 per decoded pair at T = 1
def test_dq16_parity_stages(T, M):
    q, qU, qW = _layer(_R(72, 520, 60 + T), T)
    x = _x(M, 520, 19 + T, outliers=True)
    y = f2i.linear(q, x.cuda(), algo="tcgen05_dq16").cpu().numpy()
    assert rel_l2(y, oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))) <= DQ16_REL_L2


def test_dq16_token_magnitudes():
    """Tokens scaled by 2^-60, 2^-20, 1, 2^20 and 2^100 (bfloat16 holds them, fp16 does
    not without the per-token power of two), a token of zeros, and a token whose
    values span 2^-30 .. 1: every token within the bar (zeros exactly zero)."""
    n, m = 96, 264
    q, qU, qW = _layer(_R(n, m, 5), 2)
    x = _x(7, m, 6).double()
    for t, e in enumerate([-60, -20, 0, 20, 100]):
        x[t] *= 2.0 ** e
    x[5] = 0.0
    x[6] *= torch.tensor([2.0 ** -(k % 31) for k in range(2 * m)], dtype=torch.float64)
    x = x.to(torch.bfloat16)
    y = f2i.linear(q, x.cuda(), algo="tcgen05_dq16").cpu().numpy()
    want = oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))
    for t in (0, 1, 2, 3, 4, 6):
        assert rel_l2(y[t], want[t]) <= DQ16_REL_L2, t
    assert np.all(y[5] == 0.0)


def test_dq16_row_scale_magnitudes():
    """Real rows scaled by powers of two from 2^-40 to 2^40 (weight scales of 2^-45 ..
    2^35), so every row takes its own power of two: rows within the bar one by one."""
    n, m = 64, 200
    R = _R(n, m, 8).double()
    exps = torch.tensor([float(-40 + 10 * (j % 9)) for j in range(2 * n)], dtype=torch.float64)
    Rs = (R * torch.pow(2.0, exps)[:, None]).float()
    q, qU, qW = _layer(Rs, 2)
    x = _x(20, m, 9)
    y = f2i.linear(q, x.cuda(), algo="tcgen05_dq16").cpu().numpy()
    want = oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))
    for j in range(n):  # output j holds Re y_j and Im y_j, from real rows j and n + j
        cols = [j, n + j]
        assert rel_l2(y[:, cols], want[:, cols]) <= DQ16_REL_L2, j


def test_dq16_nonfinite_token():
    """A token holding Inf or NaN gives non-finite outputs; the other tokens are unaffected."""
    n, m = 40, 256
    q, qU, qW = _layer(_R(n, m, 12), 2)
    x = _x(5, m, 13)
    want = oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))
    x[1, 7] = float("inf")
    x[3, m + 2] = float("nan")
    y = f2i.linear(q, x.cuda(), algo="tcgen05_dq16").cpu().numpy()
    assert not np.isfinite(y[1]).any() and not np.isfinite(y[3]).any()
    for t in (0, 2, 4):
        assert rel_l2(y[t], want[t]) <= DQ16_REL_L2


@pytest.mark.parametrize("M", [33, 300])
def test_dq16_group_over_several_launches(M):
    """11 layers: two launches of at most 8, both converting their activations into the
    same workspace in stream order."""
    shapes = [(40 + 8 * i, 256 + 64 * (i % 5)) for i in range(11)]
    qs, xs, wants = [], [], []
    for i, (n, m) in enumerate(shapes):
        q, qU, qW = _layer(_R(n, m, 900 + i), 2)
        qs.append(q)
        x = _x(M, m, 950 + i)
        xs.append(x.cuda())
        wants.append(oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x)))
    ys = f2i.linear_group(qs, xs, algo="tcgen05_dq16")
    for y, want in zip(ys, wants):
        assert rel_l2(y.cpu().numpy(), want) <= DQ16_REL_L2


def test_dq16_is_auto_with_workspace():
    """With a workspace AUTO takes the fp16 form from 10 tokens: the same bits as the
    explicit call; without one (the plain entry point) the bfloat16 form."""
    n, m = 100, 600
    q, qU, qW = _layer(_R(n, m, 14), 2)
    lib = f2i.load_library()
    x = _x(11, m, 15).cuda()
    a = f2i.linear(q, x)
    b = f2i.linear(q, x, algo="tcgen05_dq16")
    assert torch.equal(a, b)
    y = torch.empty_like(a)
    d = q.desc()
    assert lib.fairy2i_linear(ctypes.byref(d), x.data_ptr(), 11, y.data_ptr(), None) == 0
    assert torch.equal(y, f2i.linear(q, x, algo="tcgen05_dq"))


def _sample_rows(n, count, seed):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(n, size=min(count, n), replace=False).tolist())
    rows.update({0, n - 1, min(31, n - 1), min(64, n - 1)})
    return np.array(sorted(rows))


@pytest.mark.parametrize("M", [16, 2048])
def test_dq16_full_size_block_sampled(M):
    """The seven LLaMA-2-7B projections in one grouped call through AUTO (the fp16 form):
    16 tokens (batched decode) and 2048 with 1 % outliers x10 (the prefill workload), on
    sampled rows and tokens."""
    qs, xs, samples = [], [], []
    for pi, (name, out_f, in_f) in enumerate(inputs.LLAMA2_7B_BLOCK):
        n = out_f // 2
        R = inputs.weight_R(5, pi, out_f, in_f)
        qs.append(f2i.convert_quantize(R.cuda(), 2, layout=L3))
        x = inputs.activations(5, pi, M, in_f, outliers=M > 16)
        xs.append(x.cuda())
        rows = _sample_rows(n, 6, pi)
        Rs = torch.cat([R[rows], R[n + rows]]).numpy()
        Uo, Wo = oracle.convert_f32(Rs)
        toks = np.unique(np.array([0, 1, M // 2, M - 1]))
        want = oracle.linear_mulfree(oracle.quantize(Uo, 2), oracle.quantize(Wo, 2), inputs.bf16_bits(x[toks]))
        samples.append((rows, toks, want))
    ys = f2i.linear_group(qs, xs)
    for q, y, (rows, toks, want) in zip(qs, ys, samples):
        y = y.cpu().numpy()[toks]
        got = np.concatenate([y[:, rows], y[:, q.n + rows]], axis=1)
        assert rel_l2(got, want) <= DQ16_REL_L2


@pytest.mark.parametrize("algo,M", [("lut", 1), ("lut", 3), ("lut", 5), ("tcgen05_dq", 40), ("tcgen05_dq16", 40),
                                    ("tcgen05_dq16", 300), ("auto", 16)])
def test_bf16_outputs_are_the_rounded_fp32_outputs(algo, M):
    """fairy2i_linear_group_ws_out with bfloat16 outputs: every element equals the float32
    call's element rounded to nearest even, for one-window layers (written by the table
    lookup's decode launch) and several-window ones (written by its summing launch), and for
    both forms of the dequantized GEMM."""
    shapes = [(40, 256), (37, 600), (64, 1024)]
    qs, xs = [], []
    for i, (n, m) in enumerate(shapes):
        qs.append(_layer(_R(n, m, 70 + i), 2)[0])
        xs.append(_x(M, m, 80 + i).cuda())
    y32 = f2i.linear_group(qs, xs, algo=algo)
    y16 = f2i.linear_group(qs, xs, algo=algo, out_dtype=torch.bfloat16)
    for a, b in zip(y32, y16):
        assert b.dtype == torch.bfloat16 and torch.equal(a.to(torch.bfloat16), b)


@pytest.mark.parametrize("layout,algo,M", [(L3, "lut", 1), (L3, "tcgen05_dq16", 40), (L3, "auto", 3), (2, "mma", 2),
                                           (2, "tcgen05", 33)])
def test_group_call_prepared_once(layout, algo, M):
    """GroupCall: arguments built once, then called again after the inputs changed in place;
    every call equals a fresh linear_group call on the same inputs, bit for bit."""
    shapes = [(40, 256), (37, 600)]
    qs, xs = [], []
    for i, (n, m) in enumerate(shapes):
        U, W = f2i.convert(_R(n, m, 40 + i).cuda())
        qs.append(f2i.quantize(U, W, 2, layout=layout))
        xs.append(_x(M, m, 50 + i).cuda())
    call = f2i.GroupCall(qs, xs, algo=algo)
    for step in range(3):
        got = [y.clone() for y in call()]
        want = f2i.linear_group(qs, xs, algo=algo)
        for a, b in zip(got, want):
            assert torch.equal(a, b), step
        for x in xs:
            x.mul_(-2)  # exact in bfloat16

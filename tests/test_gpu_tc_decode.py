"""GPU parity of the 2:4-sparse tensor-core decode (tcgen05.mma.sp) against the
oracle, through the C ABI.

The path represents each bfloat16 activation as two e4m3 terms under a
per-token power of two; the sum is exact for every entry within 2^-13 of the
token's largest magnitude, so outputs agree with the fp64 oracle to fp32
accumulation error.  Bar: relative L2 1e-3 as for every decode path, and 1e-5
for ordinary activations.
"""
import numpy as np
import pytest
import torch

import oracle
import bit_complex_valued_fairy2i_b300 as f2i
from bit_complex_valued_fairy2i_b300 import inputs

pytestmark = pytest.mark.gpu

ALGO = "tcgen05_sp"
REL_L2 = 1e-3
TIGHT = 1e-5


def rel_l2(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


def _layer(n, m, T, seed):
    R = inputs.weight_R(98, seed, 2 * n, 2 * m)
    U, W = f2i.convert(R.cuda())
    q = f2i.quantize(U, W, T)
    Uo, Wo = oracle.convert_f32(R.numpy())
    return q, oracle.quantize(Uo, T), oracle.quantize(Wo, T)


def _x(M, m, seed, outliers=False):
    return inputs.activations(98, seed, M, 2 * m, outliers=outliers)


# (n, m): partial row tiles for every R; odd column-block counts (the 4-D tail
# map); m not a multiple of 8 (per-element activation loads); one column.
SHAPES = [(70, 300), (64, 256), (33, 64), (130, 1000), (5, 77), (17, 1), (96, 4160)]


@pytest.mark.parametrize("n,m", SHAPES)
@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_tc_decode_shapes_and_stages(n, m, T):
    q, qU, qW = _layer(n, m, T, 10 * n + m + T)
    x = _x(2, m, n + m)
    y = f2i.linear(q, x.cuda(), algo=ALGO).cpu().numpy()
    err = rel_l2(y, oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x)))
    assert err <= TIGHT, err


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 6, 7, 8])
def test_tc_decode_token_counts(M):
    n, m, T = 96, 640, 2
    q, qU, qW = _layer(n, m, T, 300 + M)
    x = _x(M, m, 400 + M, outliers=True)
    y = f2i.linear(q, x.cuda(), algo=ALGO).cpu().numpy()
    want = oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))
    for t in range(M):
        assert rel_l2(y[t], want[t]) <= TIGHT, t


def test_tc_decode_dynamic_range_inside_a_token():
    """One huge entry next to tiny ones: entries far below the token's largest
    magnitude lose bits, and the output error stays inside the bar."""
    n, m = 64, 512
    q, qU, qW = _layer(n, m, 2, 5)
    x = _x(3, m, 6).float()
    x[0, 7] = 3.0e4
    x[1] *= 1e-3
    x[1, 100] = 1.0e3
    x[2, :m] *= 1e6
    x = x.to(torch.bfloat16)
    y = f2i.linear(q, x.cuda(), algo=ALGO).cpu().numpy()
    want = oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))
    for t in range(3):
        assert rel_l2(y[t], want[t]) <= REL_L2, t


def test_tc_decode_nonfinite_token_gives_nan():
    """A token holding Inf or NaN gets NaN outputs; the other tokens are
    unaffected."""
    n, m = 40, 256
    q, qU, qW = _layer(n, m, 2, 8)
    x = _x(3, m, 9).float()
    x[0, 3] = float("inf")
    x[2, m + 5] = float("nan")
    x = x.to(torch.bfloat16)
    y = f2i.linear(q, x.cuda(), algo=ALGO).cpu().numpy()
    assert np.all(np.isnan(y[0])) and np.all(np.isnan(y[2]))
    want = oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x[1:2]))
    assert rel_l2(y[1:2], want) <= TIGHT


def test_tc_decode_zero_input():
    q, _, _ = _layer(40, 256, 2, 11)
    y = f2i.linear(q, torch.zeros((3, 512), dtype=torch.bfloat16, device="cuda"), algo=ALGO)
    assert not torch.any(y)


def test_tc_decode_group_over_several_launches():
    """Eleven layers of mixed shapes: more than one launch's worth of layers,
    each CTA taking tiles of several layers; equal to the layers one by one."""
    shapes = [(70, 300), (64, 256), (130, 1000), (5, 77), (96, 640), (48, 130), (256, 512), (33, 64),
              (90, 700), (16, 2048), (200, 192)]
    qs, xs, wants = [], [], []
    for i, (n, m) in enumerate(shapes):
        q, qU, qW = _layer(n, m, 2, 600 + i)
        x = _x(2, m, 700 + i)
        qs.append(q)
        xs.append(x.cuda())
        wants.append(oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x)))
    ys = f2i.linear_group(qs, xs, algo=ALGO)
    for q, x, y, want in zip(qs, xs, ys, wants):
        assert rel_l2(y.cpu().numpy(), want) <= TIGHT
        assert torch.equal(y, f2i.linear(q, x, algo=ALGO))


def test_tc_decode_deterministic():
    q, _, _ = _layer(300, 700, 2, 12)
    x = _x(5, 700, 13).cuda()
    assert torch.equal(f2i.linear(q, x, algo=ALGO), f2i.linear(q, x, algo=ALGO))


def test_tc_decode_unsupported_requests():
    q, _, _ = _layer(16, 64, 2, 14)
    with pytest.raises(RuntimeError):
        f2i.linear(q, _x(9, 64, 1).cuda(), algo=ALGO)  # more than 8 tokens
    q8, _, _ = _layer(16, 64, 5, 15)
    with pytest.raises(RuntimeError):
        f2i.linear(q8, _x(1, 64, 1).cuda(), algo=ALGO)  # more than 4 stages

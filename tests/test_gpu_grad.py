"""GPU parity of the input gradient dL/dx = U^^H g + W^^T conj(g) against the
oracle, through the C ABI.  fp32 accumulation of fp32 gradients: bar rel-L2
1e-5 (the layer bar is 1e-3)."""
import numpy as np
import pytest
import torch

import oracle
import bit_complex_valued_fairy2i_b300 as f2i
from bit_complex_valued_fairy2i_b300 import inputs

pytestmark = pytest.mark.gpu

TIGHT = 1e-5


def rel_l2(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


def _layer(n, m, T, seed, R=None):
    if R is None:
        R = inputs.weight_R(97, seed, 2 * n, 2 * m)
    U, W = f2i.convert(R.cuda())
    q = f2i.quantize(U, W, T)
    Uo, Wo = oracle.convert_f32(R.numpy())
    return q, oracle.quantize(Uo, T), oracle.quantize(Wo, T)


def _g(M, n, seed):
    return torch.from_numpy(np.random.default_rng(seed).normal(size=(M, 2 * n)).astype(np.float32))


@pytest.mark.parametrize("n,m", [(1, 1), (8, 64), (37, 130), (70, 300), (256, 256), (13, 2049), (130, 1000)])
@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_grad_x_parity(n, m, T):
    q, qU, qW = _layer(n, m, T, 10 * n + m + T)
    g = _g(2, n, n + m)
    gx = f2i.linear_grad_x(q, g.cuda()).cpu().numpy()
    err = rel_l2(gx, oracle.linear_grad_x_mulfree(qU, qW, g.numpy()))
    assert err <= TIGHT, err


@pytest.mark.parametrize("M", [1, 2, 3, 5])
def test_grad_x_token_counts(M):
    n, m = 96, 640
    q, qU, qW = _layer(n, m, 2, 300 + M)
    g = _g(M, n, 400 + M)
    gx = f2i.linear_grad_x(q, g.cuda()).cpu().numpy()
    want = oracle.linear_grad_x_mulfree(qU, qW, g.numpy())
    for t in range(M):
        assert rel_l2(gx[t], want[t]) <= TIGHT, t


def test_grad_x_adjoint_of_the_gpu_forward():
    """<y(x), g> = <x, dL/dx(g)> with both sides computed on the GPU."""
    n, m = 300, 700
    q, _, _ = _layer(n, m, 2, 12)
    x = inputs.activations(97, 5, 3, 2 * m)
    g = _g(3, n, 6)
    y = f2i.linear(q, x.cuda(), algo="addsub").cpu().double()
    gx = f2i.linear_grad_x(q, g.cuda()).cpu().double()
    lhs = (y * g.double()).sum(dim=1)
    rhs = (x.double() * gx).sum(dim=1)
    assert torch.all((lhs - rhs).abs() <= 1e-5 * y.norm(dim=1) * g.double().norm(dim=1))


@pytest.mark.parametrize("name,out_f,in_f", inputs.LLAMA2_7B_BLOCK[3:])  # o, gate, up, down
def test_grad_x_full_size_sampled_columns(name, out_f, in_f):
    """LLaMA-2-7B-shaped projection at full size; the oracle on a sample of
    input columns (column k of the gradient depends on column k of the codes)."""
    pi = [p[0] for p in inputs.LLAMA2_7B_BLOCK].index(name)
    n, m, T = out_f // 2, in_f // 2, 2
    R = inputs.weight_R(2, pi, out_f, in_f)
    U, W = f2i.convert(R.cuda())
    q = f2i.quantize(U, W, T)
    rng = np.random.default_rng(pi)
    cols = np.unique(np.concatenate([[0, 1, 63, 64, m - 1], rng.choice(m, size=19, replace=False)]))
    Uo, Wo = oracle.convert_f32(R.numpy())  # the oracle's own codes and scales of every row
    oU, oW = oracle.quantize(Uo, T), oracle.quantize(Wo, T)
    qU = oracle.Quantized(np.ascontiguousarray(oU.codes[:, :, cols]), oU.scales, None, None)
    qW = oracle.Quantized(np.ascontiguousarray(oW.codes[:, :, cols]), oW.scales, None, None)
    g = _g(1, n, 50 + pi)
    want = oracle.linear_grad_x_mulfree(qU, qW, g.numpy())
    gx = f2i.linear_grad_x(q, g.cuda()).cpu().numpy()
    got = np.concatenate([gx[:, cols], gx[:, m + cols]], axis=1)
    assert rel_l2(got, want) <= TIGHT


def test_grad_x_deterministic_and_zero_tokens():
    q, _, _ = _layer(300, 700, 2, 13)
    g = _g(3, 300, 7).cuda()
    assert torch.equal(f2i.linear_grad_x(q, g), f2i.linear_grad_x(q, g))
    assert f2i.linear_grad_x(q, torch.zeros((0, 600), device="cuda")).shape == (0, 1400)


@pytest.mark.parametrize("M", [1, 3])
def test_grad_x_group_equals_single_launches(M):
    """One launch over layers of mixed shapes (partial row tiles, an odd column
    block count, a ragged last block) gives each layer's single-launch result
    bit for bit, and the oracle's."""
    shapes = [(37, 130), (256, 256), (13, 2049), (70, 300), (8, 64)]
    qs, gs, wants = [], [], []
    for i, (n, m) in enumerate(shapes):
        q, qU, qW = _layer(n, m, 2, 900 + i)
        g = _g(M, n, 950 + i)
        qs.append(q)
        gs.append(g.cuda())
        wants.append(oracle.linear_grad_x_mulfree(qU, qW, g.numpy()))
    gxs = f2i.linear_grad_x_group(qs, gs)
    for q, g, gx, want in zip(qs, gs, gxs, wants):
        assert torch.equal(gx, f2i.linear_grad_x(q, g))
        assert rel_l2(gx.cpu().numpy(), want) <= TIGHT

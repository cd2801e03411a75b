"""GPU parity of the tcgen05 prefill path (large token counts) against the oracle.

The prefill evaluates the same sum as the decode path as a dense ternary
contraction on the tensor cores; every product is exact, so the bar is the
same as for decode: outputs within relative L2 error 1e-3 of the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import bit_complex_valued_fairy2i_b300 as f2i
from bit_complex_valued_fairy2i_b300 import inputs

pytestmark = pytest.mark.gpu

REL_L2 = 1e-3


def rel_l2(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


def _R(n, m, seed):
    return inputs.weight_R(98, seed, 2 * n, 2 * m)


def _x(M, m, seed, outliers=True):
    return inputs.activations(98, seed, M, 2 * m, outliers=outliers)


def _layer(R, T):
    U, W = f2i.convert(R.cuda())
    q = f2i.quantize(U, W, T)
    Uo, Wo = oracle.convert_f32(R.numpy())
    return q, oracle.quantize(Uo, T), oracle.quantize(Wo, T)


# (n, m): several row tiles, ragged row tiles, m with a partial 64-column block
SHAPES = [(8, 64), (37, 136), (256, 256), (300, 704), (16, 1024), (130, 2048)]


@pytest.mark.parametrize("n,m", SHAPES)
@pytest.mark.parametrize("M", [1, 5, 128, 129, 300])
def test_prefill_parity(n, m, M):
    R = _R(n, m, 7 * n + m)
    q, qU, qW = _layer(R, 2)
    x = _x(M, m, n + 3 * m + M)
    y = f2i.linear(q, x.cuda(), algo="tcgen05").cpu().numpy()
    want = oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))
    assert rel_l2(y, want) <= REL_L2


@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_prefill_parity_stages(T):
    n, m, M = 72, 520, 200
    R = _R(n, m, 60 + T)
    q, qU, qW = _layer(R, T)
    x = _x(M, m, 13)
    y = f2i.linear(q, x.cuda(), algo="tcgen05").cpu().numpy()
    want = oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))
    assert rel_l2(y, want) <= REL_L2
    # per token too: no token may be wrong while the total passes
    for t in range(0, M, 37):
        assert rel_l2(y[t], want[t]) <= REL_L2


def test_prefill_matches_decode_path():
    n, m, M = 100, 512, 70
    R = _R(n, m, 3)
    q, _, _ = _layer(R, 2)
    x = _x(M, m, 4).cuda()
    y_tc = f2i.linear(q, x, algo="tcgen05")
    y_mma = f2i.linear(q, x, algo="mma")
    assert rel_l2(y_tc.cpu().numpy(), y_mma.cpu().numpy()) <= 1e-5


def test_prefill_auto_dispatch_and_unsupported():
    R = _R(16, 100, 5)  # m = 100 is not a multiple of 8: no TMA row stride
    q, qU, qW = _layer(R, 2)
    x = _x(200, 100, 6)
    with pytest.raises(f2i.Fairy2iError) as e:
        f2i.linear(q, x.cuda(), algo="tcgen05")
    assert e.value.status == 4
    y = f2i.linear(q, x.cuda()).cpu().numpy()  # auto falls back to the decode kernel
    assert rel_l2(y, oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))) <= REL_L2


def test_prefill_zero_tokens_and_zero_input():
    R = _R(24, 128, 7)
    q, _, _ = _layer(R, 2)
    y = f2i.linear(q, torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda"), algo="tcgen05")
    assert y.shape == (0, 48)
    y = f2i.linear(q, torch.zeros((300, 256), dtype=torch.bfloat16, device="cuda"), algo="tcgen05")
    assert not torch.any(y)


def test_prefill_extreme_activation_range():
    n, m = 40, 256
    R = _R(n, m, 8)
    q, qU, qW = _layer(R, 2)
    x = torch.cat([_x(64, m, 1) * 1e-20, _x(64, m, 2) * 1e20, _x(64, m, 3)]).to(torch.bfloat16)
    y = f2i.linear(q, x.cuda(), algo="tcgen05").cpu().numpy()
    want = oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))
    for t in (0, 63, 64, 127, 128, 191):
        assert rel_l2(y[t], want[t]) <= REL_L2


def test_prefill_deterministic_and_group_equals_single():
    shapes = [(40, 256), (130, 2048), (64, 64)]
    qs, xs = [], []
    for i, (n, m) in enumerate(shapes):
        q, _, _ = _layer(_R(n, m, 300 + i), 2)
        qs.append(q)
        xs.append(_x(150, m, 400 + i).cuda())
    ys = f2i.linear_group(qs, xs, algo="tcgen05")
    for q, x, y in zip(qs, xs, ys):
        y1 = f2i.linear(q, x, algo="tcgen05")
        assert torch.equal(y, y1)
        assert torch.equal(y1, f2i.linear(q, x, algo="tcgen05"))


def _sample_rows(n, count=16, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(n, size=min(count, n), replace=False).tolist())
    rows.update({0, n - 1, min(15, n - 1), min(16, n - 1)})
    return np.array(sorted(rows))


def test_full_size_block_prefill_sampled():
    """The seven LLaMA-2-7B projections of a block at M = 2048 tokens with 1 %
    outliers x10 (the prefill workload), one grouped launch, checked on
    sampled output rows and sampled tokens against the oracle."""
    M = 2048
    qs, xs, samples = [], [], []
    for pi, (name, out_f, in_f) in enumerate(inputs.LLAMA2_7B_BLOCK):
        n = out_f // 2
        R = inputs.weight_R(4, pi, out_f, in_f)
        U, W = f2i.convert(R.cuda())
        qs.append(f2i.quantize(U, W, 2))
        del U, W
        x = inputs.activations(4, pi, M, in_f, outliers=True)
        xs.append(x.cuda())
        rows = _sample_rows(n, seed=pi)
        toks = np.array(sorted(set(np.random.default_rng(pi).choice(M, 48, replace=False).tolist()) | {0, M - 1}))
        Rs = torch.cat([R[rows], R[n + rows]]).numpy()
        Uo, Wo = oracle.convert_f32(Rs)
        qU, qW = oracle.quantize(Uo, 2), oracle.quantize(Wo, 2)
        want = oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x[torch.from_numpy(toks)]))
        samples.append((rows, toks, want))
    ys = f2i.linear_group(qs, xs, algo="tcgen05")
    for q, y, (rows, toks, want) in zip(qs, ys, samples):
        y = y[torch.from_numpy(toks).cuda()].cpu().numpy()
        got = np.concatenate([y[:, rows], y[:, q.n + rows]], axis=1)
        assert rel_l2(got, want) <= REL_L2

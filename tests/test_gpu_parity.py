"""GPU parity: the CUDA path through the C ABI against the oracle.

Bars: converted weights, codes and scales bit-exact; layer outputs within
relative L2 error 1e-3 (fp32 accumulation of bfloat16 activations).
"""
import numpy as np
import pytest
import torch

import oracle
import bit_complex_valued_fairy2i_b300 as f2i
from bit_complex_valued_fairy2i_b300 import inputs

pytestmark = pytest.mark.gpu

REL_L2 = 1e-3
DECODE_ALGOS = ("addsub", "mma", "tcgen05_sp")


def rel_l2(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


def _R(n, m, seed):
    return inputs.weight_R(99, seed, 2 * n, 2 * m)


def _x(M, m, seed, outliers=False):
    return inputs.activations(99, seed, M, 2 * m, outliers=outliers)


def _gpu_layer(R, T):
    U, W = f2i.convert(R.cuda())
    q = f2i.quantize(U, W, T)
    return U, W, q


def _oracle_layer(R, T):
    U, W = oracle.convert_f32(R.numpy())
    return U, W, oracle.quantize(U, T), oracle.quantize(W, T)


SHAPES = [(1, 1), (8, 64), (37, 130), (256, 256), (300, 700), (64, 1024), (13, 2049)]


@pytest.mark.parametrize("n,m", SHAPES + [(5, 6), (16, 10)])
def test_convert_bit_exact(n, m):
    R = _R(n, m, n * 1000 + m)
    U, W = f2i.convert(R.cuda())
    Uo, Wo = oracle.convert_f32(R.numpy())
    assert np.array_equal(U.cpu().numpy().view(np.uint64), Uo.view(np.uint64))
    assert np.array_equal(W.cpu().numpy().view(np.uint64), Wo.view(np.uint64))


@pytest.mark.parametrize("n,m", SHAPES)
@pytest.mark.parametrize("T", [1, 2, 3])
def test_quantize_bit_exact(n, m, T):
    R = _R(n, m, 7 + n + m)
    _, _, q = _gpu_layer(R, T)
    _, _, qU, qW = _oracle_layer(R, T)
    codes = f2i.unpack_codes(q).cpu().numpy()
    assert np.array_equal(codes[0], qU.codes)
    assert np.array_equal(codes[1], qW.codes)
    sc = q.scales.cpu().numpy()
    assert np.array_equal(sc[0].view(np.uint32), qU.scales.view(np.uint32))
    assert np.array_equal(sc[1].view(np.uint32), qW.scales.view(np.uint32))


def test_quantize_golden_rounding_cases(golden_dir):
    """The hand-derived float32 rounding-boundary scales, on the GPU."""
    import os
    with open(os.path.join(golden_dir, "scale_rounding.txt")) as fh:
        for line in fh:
            line = line.split("#")[0].strip()
            if not line:
                continue
            _, *vals = line.split()
            re = torch.tensor([float(v) for v in vals[:-1]], dtype=torch.float32)
            want = np.float32(float(vals[-1]))
            U = torch.complex(re, torch.zeros_like(re))[None, :].cuda()
            q = f2i.quantize(U, torch.zeros_like(U), 1)
            assert q.scales[0, 0, 0, 0].item() == want


@pytest.mark.parametrize("T", [1, 2, 3, 4, 8])
def test_quantize_bit_exact_more_stages(T):
    R = _R(40, 300, 31 + T)
    _, _, q = _gpu_layer(R, T)
    _, _, qU, qW = _oracle_layer(R, T)
    codes = f2i.unpack_codes(q).cpu().numpy()
    assert np.array_equal(codes[0], qU.codes) and np.array_equal(codes[1], qW.codes)
    sc = q.scales.cpu().numpy()
    assert np.array_equal(sc[0], qU.scales) and np.array_equal(sc[1], qW.scales)


def test_quantize_ties_and_zeros():
    vals = [(1, 1), (-1, 1), (1, -1), (-1, -1), (0, 0), (-0.0, 0), (0, -0.0), (-0.0, -0.0), (2, -2), (0, 3)]
    re = torch.tensor([v[0] for v in vals], dtype=torch.float32)
    im = torch.tensor([v[1] for v in vals], dtype=torch.float32)
    U = torch.complex(re, im)[None, :].cuda()
    q = f2i.quantize(U, U.clone(), 2)
    Uo = (re.numpy() + 1j * im.numpy()).astype(np.complex64)[None, :]
    qo = oracle.quantize(Uo, 2)
    assert np.array_equal(f2i.unpack_codes(q).cpu().numpy()[0], qo.codes)


def test_quantize_nonfinite_reported():
    U = torch.zeros((4, 8), dtype=torch.complex64, device="cuda")
    U[2, 3] = complex(float("nan"), 0.0)
    with pytest.raises(f2i.Fairy2iError) as e:
        f2i.quantize(U, torch.zeros_like(U), 1)
    assert e.value.status == 3
    # the error word is cleared: a clean call succeeds afterwards
    f2i.quantize(torch.ones_like(U), torch.zeros_like(U), 1)


@pytest.mark.parametrize("algo", DECODE_ALGOS)
@pytest.mark.parametrize("n,m", SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 8])
def test_linear_parity(algo, n, m, M):
    T = 2
    R = _R(n, m, 3 * n + m)
    _, _, q = _gpu_layer(R, T)
    _, _, qU, qW = _oracle_layer(R, T)
    x = _x(M, m, n + 5 * m)
    y = f2i.linear(q, x.cuda(), algo=algo).cpu().numpy()
    want = oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))
    err = rel_l2(y, want)
    assert err <= REL_L2, err
    if algo == "addsub":
        assert err <= 1e-5, err  # fp32 accumulation of exact bfloat16 values


@pytest.mark.parametrize("algo", DECODE_ALGOS)
@pytest.mark.parametrize("T", [1, 3, 4])
def test_linear_parity_stages(algo, T):
    n, m, M = 72, 520, 3
    R = _R(n, m, 50 + T)
    _, _, q = _gpu_layer(R, T)
    _, _, qU, qW = _oracle_layer(R, T)
    x = _x(M, m, 9)
    y = f2i.linear(q, x.cuda(), algo=algo).cpu().numpy()
    assert rel_l2(y, oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))) <= REL_L2


def test_linear_addsub_many_stages():
    n, m, M, T = 24, 200, 2, 8
    R = _R(n, m, 77)
    _, _, q = _gpu_layer(R, T)
    _, _, qU, qW = _oracle_layer(R, T)
    x = _x(M, m, 10)
    y = f2i.linear(q, x.cuda(), algo="addsub").cpu().numpy()
    assert rel_l2(y, oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))) <= 1e-5


@pytest.mark.parametrize("algo", ("addsub", "mma"))  # the sparse tensor-core decode takes M <= 8
def test_linear_more_tokens_than_one_launch(algo):
    n, m, M = 40, 256, 19
    R = _R(n, m, 5)
    _, _, q = _gpu_layer(R, 2)
    _, _, qU, qW = _oracle_layer(R, 2)
    x = _x(M, m, 11, outliers=True)
    y = f2i.linear(q, x.cuda(), algo=algo).cpu().numpy()
    assert rel_l2(y, oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))) <= REL_L2


@pytest.mark.parametrize("algo", DECODE_ALGOS)
def test_linear_extreme_activation_range(algo):
    """Tokens whose largest magnitude is tiny or huge (the fp8 path rescales
    each token's real and imaginary halves by a power of two)."""
    n, m = 16, 128
    R = _R(n, m, 6)
    _, _, q = _gpu_layer(R, 2)
    _, _, qU, qW = _oracle_layer(R, 2)
    x = torch.cat([_x(1, m, 1) * 1e-20, _x(1, m, 2) * 1e20, _x(1, m, 3)]).to(torch.bfloat16)
    y = f2i.linear(q, x.cuda(), algo=algo).cpu().numpy()
    want = oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))
    for t in range(3):
        assert rel_l2(y[t], want[t]) <= REL_L2


def test_linear_zero_tokens_and_zero_input():
    R = _R(8, 64, 2)
    _, _, q = _gpu_layer(R, 2)
    y = f2i.linear(q, torch.zeros((0, 128), dtype=torch.bfloat16, device="cuda"))
    assert y.shape == (0, 16)
    for algo in DECODE_ALGOS:
        y = f2i.linear(q, torch.zeros((2, 128), dtype=torch.bfloat16, device="cuda"), algo=algo)
        assert not torch.any(y)


@pytest.mark.parametrize("algo", DECODE_ALGOS)
def test_linear_deterministic(algo):
    R = _R(300, 700, 4)
    _, _, q = _gpu_layer(R, 2)
    x = _x(3, 700, 4).cuda()
    y1 = f2i.linear(q, x, algo=algo)
    y2 = f2i.linear(q, x, algo=algo)
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("algo", DECODE_ALGOS)
def test_group_equals_single_launches(algo):
    shapes = [(40, 256), (13, 2049), (64, 64)]
    qs, xs = [], []
    for i, (n, m) in enumerate(shapes):
        _, _, q = _gpu_layer(_R(n, m, 100 + i), 2)
        qs.append(q)
        xs.append(_x(2, m, 200 + i).cuda())
    ys = f2i.linear_group(qs, xs, algo=algo)
    for q, x, y in zip(qs, xs, ys):
        assert torch.equal(y, f2i.linear(q, x, algo=algo))


def _sample_rows(n, count=24, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(n, size=min(count, n), replace=False).tolist())
    rows.update({0, n - 1, min(7, n - 1), min(8, n - 1)})
    return np.array(sorted(rows))


def _oracle_rows(R, rows, T):
    """Oracle on a subset of output rows: rows j of U and W depend only on
    rows j and n + j of R."""
    n = R.shape[0] // 2
    Rs = torch.cat([R[rows], R[n + rows]]).numpy()
    return _oracle_layer(torch.from_numpy(Rs), T)


@pytest.mark.parametrize("T", [1, 2, 3])
@pytest.mark.parametrize("name,out_f,in_f", inputs.LLAMA2_7B_BLOCK[3:])  # o, gate, up, down
def test_full_size_projection_sampled(name, out_f, in_f, T):
    """LLaMA-2-7B-shaped projection at full size, T = 1, 2, 3 (the stack's stage
    counts): codes and scales bit-exact and outputs within the bar on sampled rows."""
    pi = [p[0] for p in inputs.LLAMA2_7B_BLOCK].index(name)
    n, m = out_f // 2, in_f // 2
    R = inputs.weight_R(2, pi, out_f, in_f)
    _, _, q = _gpu_layer(R, T)
    rows = _sample_rows(n, seed=pi)
    _, _, qU, qW = _oracle_rows(R, rows, T)
    codes = f2i.unpack_codes(q)[:, :, torch.from_numpy(rows).cuda()].cpu().numpy()
    assert np.array_equal(codes[0], qU.codes) and np.array_equal(codes[1], qW.codes)
    sc = q.scales[:, :, :, torch.from_numpy(rows).cuda()].cpu().numpy()
    assert np.array_equal(sc[0], qU.scales) and np.array_equal(sc[1], qW.scales)
    x = inputs.activations(2, pi, 1, in_f)
    want = oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))
    for algo in DECODE_ALGOS:
        y = f2i.linear(q, x.cuda(), algo=algo).cpu().numpy()
        got = np.concatenate([y[:, rows], y[:, n + rows]], axis=1)
        assert rel_l2(got, want) <= REL_L2, algo


@pytest.mark.parametrize("T", [1, 2, 3])
def test_full_size_block_group_decode_sampled(T):
    """The seven projections of a block in one grouped launch, M = 1, T = 1, 2, 3."""
    qs, xs, samples = [], [], []
    for pi, (name, out_f, in_f) in enumerate(inputs.LLAMA2_7B_BLOCK):
        n = out_f // 2
        R = inputs.weight_R(2, pi, out_f, in_f)
        q = f2i.convert_quantize(R.cuda(), T)
        qs.append(q)
        x = inputs.activations(2, pi, 1, in_f)
        xs.append(x.cuda())
        rows = _sample_rows(n, count=8, seed=pi)
        _, _, qU, qW = _oracle_rows(R, rows, T)
        samples.append((rows, oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))))
    ys = f2i.linear_group(qs, xs)
    for q, y, (rows, want) in zip(qs, ys, samples):
        y = y.cpu().numpy()
        got = np.concatenate([y[:, rows], y[:, q.n + rows]], axis=1)
        assert rel_l2(got, want) <= REL_L2


@pytest.mark.parametrize("M", [16, 32, 64])
@pytest.mark.parametrize("name,out_f,in_f", [inputs.LLAMA2_7B_BLOCK[4], inputs.LLAMA2_7B_BLOCK[6]])  # gate, down
def test_full_size_auto_batched_decode_sampled(name, out_f, in_f, M):
    """Batched decode at M = 16, 32, 64 through AUTO on full-size gate and down
    projections: the tcgen05 path with one partial 128-token tile at real m."""
    pi = [p[0] for p in inputs.LLAMA2_7B_BLOCK].index(name)
    n = out_f // 2
    R = inputs.weight_R(3, pi, out_f, in_f)
    q = f2i.convert_quantize(R.cuda(), 2)
    rows = _sample_rows(n, count=12, seed=M + pi)
    _, _, qU, qW = _oracle_rows(R, rows, 2)
    x = inputs.activations(3, pi, M, in_f)
    want = oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))
    y = f2i.linear(q, x.cuda()).cpu().numpy()
    got = np.concatenate([y[:, rows], y[:, n + rows]], axis=1)
    assert rel_l2(got, want) <= REL_L2


@pytest.mark.parametrize("T,M", [(3, 6), (4, 8), (1, 5), (2, 7)])
def test_linear_parity_wide_variants(T, M):
    """The decode instances with several token pairs per launch and 2T = 6 or 8
    code planes (the largest register footprints)."""
    n, m = 48, 384
    R = _R(n, m, 80 + 10 * T + M)
    _, _, q = _gpu_layer(R, T)
    _, _, qU, qW = _oracle_layer(R, T)
    x = _x(M, m, 90 + M)
    want = oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))
    for algo in DECODE_ALGOS:
        y = f2i.linear(q, x.cuda(), algo=algo).cpu().numpy()
        assert rel_l2(y, want) <= REL_L2, algo


def test_group_split_by_activation_width():
    """At 4 tokens a 7200-column layer's staged activations fit neither one
    16-warp CTA nor two 8-warp CTAs per SM, so the group is launched per
    activation width; results must not depend on it."""
    shapes = [(40, 256), (13, 7200), (64, 64), (24, 7200)]
    qs, xs, wants = [], [], []
    for i, (n, m) in enumerate(shapes):
        R = _R(n, m, 500 + i)
        _, _, q = _gpu_layer(R, 2)
        _, _, qU, qW = _oracle_layer(R, 2)
        x = _x(4, m, 600 + i)
        qs.append(q)
        xs.append(x.cuda())
        wants.append(oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x)))
    ys = f2i.linear_group(qs, xs, algo="mma")
    for q, x, y, want in zip(qs, xs, ys, wants):
        assert rel_l2(y.cpu().numpy(), want) <= REL_L2
        assert torch.equal(y, f2i.linear(q, x, algo="mma"))


@pytest.mark.parametrize("T,M", [(4, 2), (2, 2), (3, 2)])
def test_decode_both_launch_shapes(T, M):
    """The same call takes one 16-warp CTA per SM when the buffers fit and two
    (or one) 8-warp CTAs when a wide layer's staged activations do not: both
    against the oracle, in one group and alone."""
    wide_m = {4: 9000, 2: 15000, 3: 14000}[T]  # within the quantizer's m <= 16384
    shapes = [(40, 512), (24, wide_m)]
    qs, xs, wants = [], [], []
    for i, (n, m) in enumerate(shapes):
        R = _R(n, m, 700 + 10 * T + i)
        _, _, q = _gpu_layer(R, T)
        _, _, qU, qW = _oracle_layer(R, T)
        x = _x(M, m, 800 + i)
        qs.append(q)
        xs.append(x.cuda())
        wants.append(oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x)))
    ys = f2i.linear_group(qs, xs, algo="mma")
    for q, x, y, want in zip(qs, xs, ys, wants):
        assert rel_l2(y.cpu().numpy(), want) <= REL_L2
        assert rel_l2(f2i.linear(q, x, algo="mma").cpu().numpy(), want) <= REL_L2


def test_bounded_wait_gives_up_and_reports_timeout():
    """The bounded mbarrier wait used by the prefill kernel, run on a barrier that
    nothing arrives at: it must give up after its limit, report TIMEOUT through the
    error word, clear it, and leave the context usable."""
    f2i.selftest_bounded_wait(10000)  # 10 ms
    with pytest.raises(f2i.Fairy2iError) as e:
        f2i.sync_status()
    assert e.value.status == 6
    f2i.sync_status()  # cleared
    R = _R(8, 64, 1)
    _, _, q = _gpu_layer(R, 2)
    _, _, qU, qW = _oracle_layer(R, 2)
    x = _x(200, 64, 2)
    y = f2i.linear(q, x.cuda(), algo="tcgen05").cpu().numpy()
    assert rel_l2(y, oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))) <= REL_L2


@pytest.mark.parametrize("n,m", [(37, 130), (256, 256), (13, 2049), (300, 700)])
@pytest.mark.parametrize("T", [1, 2, 3])
def test_convert_quantize_fused_equals_two_pass(n, m, T):
    """One pass from R gives the codes and scales of convert + quantize, bit for bit,
    and the oracle's."""
    R = _R(n, m, 40 + n + m)
    q2 = f2i.convert_quantize(R.cuda(), T)
    _, _, q1 = _gpu_layer(R, T)
    assert torch.equal(f2i.unpack_codes(q2), f2i.unpack_codes(q1))
    assert torch.equal(q2.scales, q1.scales)
    _, _, qU, qW = _oracle_layer(R, T)
    codes = f2i.unpack_codes(q2).cpu().numpy()
    assert np.array_equal(codes[0], qU.codes) and np.array_equal(codes[1], qW.codes)


def test_convert_quantize_nonfinite_reported():
    R = torch.zeros((8, 16), dtype=torch.float32)
    R[5, 3] = float("inf")
    with pytest.raises(f2i.Fairy2iError) as e:
        f2i.convert_quantize(R.cuda(), 1)
    assert e.value.status == 3

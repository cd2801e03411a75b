"""GPU parity of layout 3 and the table-lookup decode, through the C ABI, against the oracle.

Bars: codes and scales bit-exact (the packed bytes also equal a packing of the
oracle's codes by the byte rule documented in include/fairy2i.h); outputs
within relative L2 error 1e-3 of the oracle's exact sum.
"""
import numpy as np
import pytest
import torch

import oracle
import bit_complex_valued_fairy2i_b300 as f2i
from bit_complex_valued_fairy2i_b300 import inputs

pytestmark = pytest.mark.gpu

REL_L2 = 1e-3
L3 = f2i.LAYOUT_LUT


def rel_l2(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


def _R(n, m, seed):
    return inputs.weight_R(98, seed, 2 * n, 2 * m)


def _x(M, m, seed, outliers=False):
    return inputs.activations(98, seed, M, 2 * m, outliers=outliers)


def _gpu_layer(R, T, layout=L3):
    U, W = f2i.convert(R.cuda())
    return f2i.quantize(U, W, T, layout=layout)


def _oracle_layer(R, T):
    U, W = oracle.convert_f32(R.numpy())
    return oracle.quantize(U, T), oracle.quantize(W, T)


def _slots(m, w):
    rest = m - 256 * w
    if rest >= 256:
        return 4
    nc = -(-rest // 64)
    return 4 if nc == 3 else nc


def pack_layout3(planes, n, m):
    """Layout-3 bytes of canonical codes [2T][n][m], by the documented rule:
    per (row, group of 8 columns) a sign byte and a q byte (sign XOR imaginary
    flag); byte i of row r in slot jj of a window with nb slots holds group
    (r & (8 nb - 1)) ^ (8 jj + i); order [window][tile][plane][slot][row][16]."""
    P = planes.shape[0]
    tiles, windows = -(-n // 32), -(-m // 256)
    row_slots = sum(_slots(m, w) for w in range(windows))
    out = np.zeros(tiles * P * 512 * row_slots, np.uint8)
    mp = windows * 256
    sign = np.zeros((P, n, mp), np.uint8)
    imag = np.zeros((P, n, mp), np.uint8)
    sign[:, :, :m] = planes & 1
    imag[:, :, :m] = (planes >> 1) & 1
    weights = (1 << np.arange(8)).astype(np.uint32)
    sb = (sign.reshape(P, n, -1, 8) * weights).sum(-1).astype(np.uint8)  # [P][n][groups]
    qb = ((sign ^ imag).reshape(P, n, -1, 8) * weights).sum(-1).astype(np.uint8)
    j = np.arange(n)[:, None]
    for w in range(windows):
        nb = _slots(m, w)
        g = np.arange(8 * nb)[None, :]
        tau, r = j // 32, j % 32
        a = (r >> 3) & 3
        jj = (g >> 3) ^ (a & (nb - 1))
        i = (g & 7) ^ (r & 7)
        for p in range(P):
            off = w * tiles * P * 2048 + (tau * P + p) * nb * 512 + jj * 512 + r * 16 + i
            out[off] = sb[p][:, 32 * w + g[0]]
            out[off + 8] = qb[p][:, 32 * w + g[0]]
    return out


SHAPES = [(1, 1), (8, 64), (37, 130), (33, 200), (256, 256), (300, 700), (64, 1024), (13, 2049), (40, 320)]


@pytest.mark.parametrize("n,m", SHAPES)
@pytest.mark.parametrize("T", [1, 2, 3])
def test_quantize_layout3_bit_exact(n, m, T):
    R = _R(n, m, 7 + n + m)
    q = _gpu_layer(R, T)
    qU, qW = _oracle_layer(R, T)
    codes = f2i.unpack_codes(q).cpu().numpy()
    assert np.array_equal(codes[0], qU.codes) and np.array_equal(codes[1], qW.codes)
    sc = q.scales.cpu().numpy()
    assert np.array_equal(sc[0].view(np.uint32), qU.scales.view(np.uint32))
    assert np.array_equal(sc[1].view(np.uint32), qW.scales.view(np.uint32))
    want = pack_layout3(np.concatenate([qU.codes, qW.codes]), n, m)
    assert np.array_equal(q.codes.cpu().numpy(), want)


@pytest.mark.parametrize("T", [4, 8])
def test_quantize_layout3_more_stages(T):
    n, m = 40, 300
    R = _R(n, m, 31 + T)
    q = _gpu_layer(R, T)
    qU, qW = _oracle_layer(R, T)
    assert np.array_equal(q.codes.cpu().numpy(), pack_layout3(np.concatenate([qU.codes, qW.codes]), n, m))
    sc = q.scales.cpu().numpy()
    assert np.array_equal(sc[0], qU.scales) and np.array_equal(sc[1], qW.scales)


@pytest.mark.parametrize("n,m", [(37, 130), (256, 256), (13, 2049), (300, 700)])
@pytest.mark.parametrize("T", [1, 2])
def test_convert_quantize_layout3(n, m, T):
    """The one-pass path writes the same layout-3 bytes and scales as convert + quantize,
    and the same canonical codes as layout 2."""
    R = _R(n, m, 40 + n + m)
    q3 = f2i.convert_quantize(R.cuda(), T, layout=L3)
    q3b = _gpu_layer(R, T)
    assert torch.equal(q3.codes, q3b.codes) and torch.equal(q3.scales, q3b.scales)
    q2 = _gpu_layer(R, T, layout=2)
    assert torch.equal(f2i.unpack_codes(q3), f2i.unpack_codes(q2))
    assert torch.equal(q3.scales, q2.scales)


def test_quantize_layout3_overwrites_old_bytes():
    """Layout 3 writes every byte (no clearing pass): a buffer full of ones is
    fully overwritten, padding rows of the last tile included."""
    n, m, T = 37, 200, 2
    R = _R(n, m, 3)
    q = f2i.Packed.empty(n, m, T, "cuda", L3)
    q.codes.fill_(0xFF)
    U, W = f2i.convert(R.cuda())
    f2i.quantize(U, W, T, out=q)
    qU, qW = _oracle_layer(R, T)
    assert np.array_equal(q.codes.cpu().numpy(), pack_layout3(np.concatenate([qU.codes, qW.codes]), n, m))


@pytest.mark.parametrize("n,m", SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 9])
def test_lut_linear_parity(n, m, M):
    T = 2
    R = _R(n, m, 3 * n + m)
    q = _gpu_layer(R, T)
    qU, qW = _oracle_layer(R, T)
    x = _x(M, m, n + 5 * m)
    y = f2i.linear(q, x.cuda()).cpu().numpy()
    want = oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))
    assert rel_l2(y, want) <= REL_L2


@pytest.mark.parametrize("T,M", [(1, 1), (1, 4), (1, 7), (3, 1), (3, 2), (3, 5), (4, 1), (4, 3)])
def test_lut_linear_parity_stages(T, M):
    n, m = 72, 520
    R = _R(n, m, 50 + T)
    q = _gpu_layer(R, T)
    qU, qW = _oracle_layer(R, T)
    x = _x(M, m, 9 + M)
    y = f2i.linear(q, x.cuda(), algo="lut").cpu().numpy()
    assert rel_l2(y, oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))) <= REL_L2


def test_lut_outliers_and_extreme_ranges():
    """Each window's table is scaled by its own power of two: tokens whose
    largest magnitude is tiny or huge, and 1 % outliers x10, keep the bar."""
    n, m = 40, 700
    R = _R(n, m, 6)
    q = _gpu_layer(R, 2)
    qU, qW = _oracle_layer(R, 2)
    x = torch.cat([_x(1, m, 1) * 1e-20, _x(1, m, 2) * 1e20, _x(1, m, 3, outliers=True),
                   _x(1, m, 4) * 1e-38]).to(torch.bfloat16)
    y = f2i.linear(q, x.cuda()).cpu().numpy()
    want = oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))
    for t in range(x.shape[0]):
        assert rel_l2(y[t], want[t]) <= REL_L2, t


def test_lut_one_window_with_a_huge_entry():
    """A single outlier 1e30 beside ordinary entries of the same window: the other
    tokens and rows stay within the bar of the exact sum."""
    n, m = 16, 512
    R = _R(n, m, 8)
    q = _gpu_layer(R, 2)
    qU, qW = _oracle_layer(R, 2)
    x = _x(2, m, 5)
    x[0, 3] = 1e30
    x = x.to(torch.bfloat16)
    y = f2i.linear(q, x.cuda()).cpu().numpy()
    want = oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))
    assert rel_l2(y, want) <= REL_L2


def test_lut_zero_tokens_zero_input_and_nonfinite():
    R = _R(40, 600, 2)
    q = _gpu_layer(R, 2)
    assert f2i.linear(q, torch.zeros((0, 1200), dtype=torch.bfloat16, device="cuda")).shape == (0, 80)
    assert not torch.any(f2i.linear(q, torch.zeros((3, 1200), dtype=torch.bfloat16, device="cuda")))
    x = _x(2, 600, 7).cuda()
    x[1, 10] = float("inf")
    y = f2i.linear(q, x)
    assert torch.all(torch.isfinite(y[0]))
    assert not torch.any(torch.isfinite(y[1]))


def test_lut_deterministic_and_workspace_reuse():
    """Repeated calls with one workspace: bit-identical outputs (fixed summation
    order), whatever the workspace held before (it needs no initialisation)."""
    R = _R(300, 1500, 4)
    q = _gpu_layer(R, 2)
    x = _x(3, 1500, 4).cuda()
    ws = f2i.workspace([q], 3, "cuda")
    y0 = f2i.linear(q, x, ws=ws)
    for fill in (0x00, 0xFF, 0x7F):
        ws.fill_(fill)
        assert torch.equal(f2i.linear(q, x, ws=ws), y0)


def test_lut_group_equals_single_launches():
    shapes = [(40, 256), (13, 2049), (64, 64), (300, 700), (33, 5504)]
    qs, xs, wants = [], [], []
    for i, (n, m) in enumerate(shapes):
        R = _R(n, m, 100 + i)
        qs.append(_gpu_layer(R, 2))
        x = _x(2, m, 200 + i)
        xs.append(x.cuda())
        qU, qW = _oracle_layer(R, 2)
        wants.append(oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x)))
    ys = f2i.linear_group(qs, xs)
    for q, x, y, want in zip(qs, xs, ys, wants):
        assert torch.equal(y, f2i.linear(q, x))
        assert rel_l2(y.cpu().numpy(), want) <= REL_L2


def test_lut_many_layers_several_launches():
    """More than 32 layers in a group (several launches sharing the workspace)."""
    qs, xs = [], []
    for i in range(37):
        n, m = 16 + 8 * (i % 5), 256 + 64 * (i % 7)
        qs.append(_gpu_layer(_R(n, m, 300 + i), 2))
        xs.append(_x(1, m, 400 + i).cuda())
    ys = f2i.linear_group(qs, xs)
    for q, x, y in zip(qs, xs, ys):
        assert torch.equal(y, f2i.linear(q, x))


def test_lut_cuda_graph_replay():
    R = _R(200, 1000, 12)
    q = _gpu_layer(R, 2)
    qU, qW = _oracle_layer(R, 2)
    x = _x(1, 1000, 13)
    xd = x.cuda()
    y = torch.empty((1, 400), device="cuda")
    f2i.linear(q, xd, out=y)  # first call outside capture (workspace, attributes)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        f2i.linear(q, xd, out=y)
    y.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert rel_l2(y.cpu().numpy(), oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))) <= REL_L2


def test_lut_errors():
    R = _R(40, 600, 2)
    q = _gpu_layer(R, 2)
    x = _x(1, 600, 1).cuda()
    lib = f2i.load_library()
    import ctypes
    d = q.desc()
    y = torch.empty((1, 80), device="cuda")
    # plain entry point: the table lookup needs the workspace entry point
    assert lib.fairy2i_linear_ex(ctypes.byref(d), x.data_ptr(), 1, y.data_ptr(), 5, None) == 4
    need = lib.fairy2i_linear_workspace_bytes(ctypes.byref(d), 1, 1)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    assert lib.fairy2i_linear_ws(ctypes.byref(d), x.data_ptr(), 1, y.data_ptr(), 0, ws.data_ptr(), 16,
                                 None) == 1  # the table lookup needs 1536 bytes here
    assert lib.fairy2i_linear_ws(ctypes.byref(d), x.data_ptr(), 1, y.data_ptr(), 2, ws.data_ptr(), need,
                                 None) == 4  # mma does not read layout 3
    with pytest.raises(f2i.Fairy2iError):
        f2i.linear_grad_x(q, torch.zeros((1, 80), device="cuda"))
    q2 = _gpu_layer(R, 2, layout=2)
    with pytest.raises(f2i.Fairy2iError):
        f2i.linear_group([q, q2], [x, x])
    f2i.sync_status()


def _sample_rows(n, count=24, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(n, size=min(count, n), replace=False).tolist())
    rows.update({0, n - 1, min(31, n - 1), min(32, n - 1)})
    return np.array(sorted(rows))


def _oracle_rows(R, rows, T):
    n = R.shape[0] // 2
    Rs = torch.cat([R[rows], R[n + rows]]).numpy()
    return _oracle_layer(torch.from_numpy(Rs), T)


@pytest.mark.parametrize("T", [1, 2, 3])
@pytest.mark.parametrize("name,out_f,in_f", [inputs.LLAMA2_7B_BLOCK[0], inputs.LLAMA2_7B_BLOCK[4],
                                             inputs.LLAMA2_7B_BLOCK[6]])  # q, gate, down
def test_full_size_projection_layout3_sampled(name, out_f, in_f, T):
    """LLaMA-2-7B-shaped projections at full size, T = 1, 2, 3: layout-3 codes and
    scales bit-exact on sampled rows and table-lookup outputs within the bar (M = 1, 2)."""
    pi = [p[0] for p in inputs.LLAMA2_7B_BLOCK].index(name)
    n, m = out_f // 2, in_f // 2
    R = inputs.weight_R(5, pi, out_f, in_f)
    q = f2i.convert_quantize(R.cuda(), T, layout=L3)
    rows = _sample_rows(n, seed=pi)
    qU, qW = _oracle_rows(R, rows, T)
    ri = torch.from_numpy(rows).cuda()
    codes = f2i.unpack_codes(q)[:, :, ri].cpu().numpy()
    assert np.array_equal(codes[0], qU.codes) and np.array_equal(codes[1], qW.codes)
    sc = q.scales[:, :, :, ri].cpu().numpy()
    assert np.array_equal(sc[0], qU.scales) and np.array_equal(sc[1], qW.scales)
    x = inputs.activations(5, pi, 2, in_f)
    want = oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))
    y = f2i.linear(q, x.cuda()).cpu().numpy()
    got = np.concatenate([y[:, rows], y[:, n + rows]], axis=1)
    assert rel_l2(got, want) <= REL_L2


@pytest.mark.parametrize("M", [1, 4, 9, 11])  # 9: AUTO's last table-lookup count; 11: 3 + 2 + 2 + 2 + 2
def test_full_size_block_group_layout3_sampled(M):
    """The seven projections of a block in one grouped table-lookup launch (the
    benchmark's launch), against the oracle on sampled rows."""
    qs, xs, samples = [], [], []
    for pi, (name, out_f, in_f) in enumerate(inputs.LLAMA2_7B_BLOCK):
        n = out_f // 2
        R = inputs.weight_R(2, pi, out_f, in_f)
        qs.append(f2i.convert_quantize(R.cuda(), 2, layout=L3))
        x = inputs.activations(2, pi, M, in_f)
        xs.append(x.cuda())
        rows = _sample_rows(n, count=8, seed=pi)
        qU, qW = _oracle_rows(R, rows, 2)
        samples.append((rows, oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))))
    ys = f2i.linear_group(qs, xs, algo="lut")
    for q, y, (rows, want) in zip(qs, ys, samples):
        y = y.cpu().numpy()
        got = np.concatenate([y[:, rows], y[:, q.n + rows]], axis=1)
        assert rel_l2(got, want) <= REL_L2


# ---------------------------------------------------------------------------
# the dequantized GEMM over layout 3 (FAIRY2I_ALGO_TCGEN05_DQ)
# ---------------------------------------------------------------------------
# R^ is carried as two bfloat16 terms (<= 2^-18 relative per entry) and summed in fp32 by
# the tensor cores over 2 (2m) / 16 steps (up to 1376 for m = 5504; each may lose up to
# 2^-23 of the running sum if the adder truncates): bar 1e-4, ten times inside the
# layer's 1e-3 (measured 1.06e-5 on the full-size block with outliers)
DQ_REL_L2 = 1e-4
DQ_SHAPES = [(8, 64), (37, 136), (33, 200), (256, 256), (300, 704), (64, 1024), (40, 320), (130, 2056)]


@pytest.mark.parametrize("n,m", DQ_SHAPES)
@pytest.mark.parametrize("M", [1, 7, 40, 130, 256, 300, 513])  # N = 16, 16, 48, 144, 256, 256 (x2), 256 (x2)
def test_dq_parity(n, m, M):
    R = _R(n, m, 11 * n + m)
    q = _gpu_layer(R, 2)
    qU, qW = _oracle_layer(R, 2)
    x = _x(M, m, n + 3 * m)
    y = f2i.linear(q, x.cuda(), algo="tcgen05_dq").cpu().numpy()
    err = rel_l2(y, oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x)))
    assert err <= DQ_REL_L2, err


@pytest.mark.parametrize("T", [1, 3, 4])
@pytest.mark.parametrize("M", [40, 300])  # one token tile of 48; two of 256 per decoded pair
def test_dq_parity_stages(T, M):
    n, m = 72, 520
    R = _R(n, m, 60 + T)
    q = _gpu_layer(R, T)
    qU, qW = _oracle_layer(R, T)
    x = _x(M, m, 19 + T, outliers=True)
    y = f2i.linear(q, x.cuda(), algo="tcgen05_dq").cpu().numpy()
    assert rel_l2(y, oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))) <= DQ_REL_L2


def test_dq_plain_entry_and_auto():
    """Layout 3 through the plain entry points (no workspace) takes the dequantized
    GEMM at any token count; with a workspace AUTO switches to the fp16 form from 10 tokens."""
    import ctypes
    n, m = 100, 600
    R = _R(n, m, 5)
    q = _gpu_layer(R, 2)
    qU, qW = _oracle_layer(R, 2)
    lib = f2i.load_library()
    for M in (1, 9, 10):
        x = _x(M, m, 30 + M)
        xd = x.cuda()
        y = torch.empty((M, 2 * n), device="cuda")
        d = q.desc()
        assert lib.fairy2i_linear(ctypes.byref(d), xd.data_ptr(), M, y.data_ptr(), None) == 0
        want = oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x))
        assert rel_l2(y.cpu().numpy(), want) <= DQ_REL_L2
        assert rel_l2(f2i.linear(q, xd).cpu().numpy(), want) <= REL_L2  # AUTO with the binding's workspace
    # m not a multiple of 8: the dequantized GEMM is refused, so the plain entry has
    # nothing to run; with a workspace the table lookup serves at any token count
    R7 = _R(16, 100, 6)
    q7 = _gpu_layer(R7, 2)
    x7 = _x(40, 100, 7)
    d7 = q7.desc()
    y7 = torch.empty((40, 32), device="cuda")
    xd7 = x7.cuda()
    assert lib.fairy2i_linear(ctypes.byref(d7), xd7.data_ptr(), 40, y7.data_ptr(), None) == 4
    assert lib.fairy2i_linear_ex(ctypes.byref(d7), xd7.data_ptr(), 40, y7.data_ptr(), 6, None) == 4
    qU7, qW7 = _oracle_layer(R7, 2)
    want7 = oracle.linear_mulfree(qU7, qW7, inputs.bf16_bits(x7))
    assert rel_l2(f2i.linear(q7, xd7).cpu().numpy(), want7) <= REL_L2


@pytest.mark.parametrize("M", [33, 300])  # the longest-first deal with one and with two token tiles
def test_dq_group_over_several_launches(M):
    shapes = [(40 + 8 * i, 256 + 64 * (i % 5)) for i in range(11)]  # 11 layers: two launches of <= 8
    qs, xs, wants = [], [], []
    for i, (n, m) in enumerate(shapes):
        R = _R(n, m, 900 + i)
        qs.append(_gpu_layer(R, 2))
        x = _x(M, m, 950 + i)
        xs.append(x.cuda())
        qU, qW = _oracle_layer(R, 2)
        wants.append(oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x)))
    ys = f2i.linear_group(qs, xs, algo="tcgen05_dq")
    for y, want in zip(ys, wants):
        assert rel_l2(y.cpu().numpy(), want) <= DQ_REL_L2


def test_dq_full_size_block_prefill_sampled():
    """The seven LLaMA-2-7B projections at 2048 tokens with 1 % outliers x10 (the
    prefill workload), one grouped call, against the oracle on sampled rows."""
    M = 2048
    qs, xs, samples = [], [], []
    for pi, (name, out_f, in_f) in enumerate(inputs.LLAMA2_7B_BLOCK):
        n = out_f // 2
        R = inputs.weight_R(4, pi, out_f, in_f)
        qs.append(f2i.convert_quantize(R.cuda(), 2, layout=L3))
        x = inputs.activations(4, pi, M, in_f, outliers=True)
        xs.append(x.cuda())
        rows = _sample_rows(n, count=6, seed=pi)
        qU, qW = _oracle_rows(R, rows, 2)
        toks = np.array([0, 1, 255, 256, 1000, M - 1])
        samples.append((rows, toks, oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x[toks]))))
    ys = f2i.linear_group(qs, xs, algo="tcgen05_dq")
    for q, y, (rows, toks, want) in zip(qs, ys, samples):
        y = y.cpu().numpy()[toks]
        got = np.concatenate([y[:, rows], y[:, q.n + rows]], axis=1)
        assert rel_l2(got, want) <= DQ_REL_L2


@pytest.mark.parametrize("M", [16, 64, 256])  # value tables up to 64 tokens, the per-plane decode above
def test_dq_full_size_block_batched_sampled(M):
    """The seven LLaMA-2-7B projections at batched-decode token counts through the bfloat16
    form (one grouped call; AUTO takes the fp16 form, tested beside it), against the oracle
    on sampled rows and tokens."""
    qs, xs, samples = [], [], []
    for pi, (name, out_f, in_f) in enumerate(inputs.LLAMA2_7B_BLOCK):
        n = out_f // 2
        R = inputs.weight_R(3, pi, out_f, in_f)
        qs.append(f2i.convert_quantize(R.cuda(), 2, layout=L3))
        x = inputs.activations(3, pi, M, in_f)
        xs.append(x.cuda())
        rows = _sample_rows(n, count=6, seed=pi + M)
        qU, qW = _oracle_rows(R, rows, 2)
        toks = np.unique(np.array([0, 1, M // 2, M - 1]))
        samples.append((rows, toks, oracle.linear_mulfree(qU, qW, inputs.bf16_bits(x[toks]))))
    ys = f2i.linear_group(qs, xs, algo="tcgen05_dq")
    for q, y, (rows, toks, want) in zip(qs, ys, samples):
        y = y.cpu().numpy()[toks]
        got = np.concatenate([y[:, rows], y[:, q.n + rows]], axis=1)
        assert rel_l2(got, want) <= DQ_REL_L2


@pytest.mark.parametrize("layout", [2, L3])
@pytest.mark.parametrize("T", [1, 2, 3])
def test_quantize_extreme_row_magnitudes_bit_exact(layout, T):
    """Rows scaled by powers of two from 2^-130 (subnormal weights) to 2^100, rows at the
    2^-79 boundary between the quantizer's fp32 and integer-shift sum paths, and rows with one
    large entry among tiny ones (per-weight truncation of the exact axis sums): codes and
    scales bit-exact against the oracle in both layouts."""
    n, m = 48, 200
    R = _R(n, m, 77 + T)
    exps = [-130, -110, -100, -81, -80, -79, -78, -77, -60, -20, 0, 20, 60, 100]
    rows = torch.arange(2 * n) % n
    scale = torch.tensor([2.0 ** exps[int(j) % len(exps)] for j in rows], dtype=torch.float64)
    Rs = (R.double() * scale[:, None]).float()
    # rows 40..47 of both halves: one entry of ordinary size among entries 2^-30 smaller
    Rs[40:48] *= 2.0 ** -30
    Rs[n + 40:n + 48] *= 2.0 ** -30
    Rs[40:48, 3] = 1.5
    Rs[n + 40:n + 48, m + 7] = -0.75
    U, W = f2i.convert(Rs.cuda())
    q = f2i.quantize(U, W, T, layout=layout)
    qU, qW = _oracle_layer(Rs, T)
    codes = f2i.unpack_codes(q).cpu().numpy()
    assert np.array_equal(codes[0], qU.codes) and np.array_equal(codes[1], qW.codes)
    sc = q.scales.cpu().numpy()
    assert np.array_equal(sc[0].view(np.uint32), qU.scales.view(np.uint32))
    assert np.array_equal(sc[1].view(np.uint32), qW.scales.view(np.uint32))
    f2i.sync_status()

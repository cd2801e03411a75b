"""Guard bands around every output and workspace: out-of-bounds writes, checked on the GPU.

The device sanitizer is not available on the test machines, so writes past an output's end
(or before its start) are caught another way: each output -- converted weights, packed codes
and scales, layer outputs in float32 and bfloat16, input gradients, the canonical code view and
the caller workspace sized exactly as the size query says -- is placed inside a larger device
buffer whose 4 KB bands on both sides hold a fixed byte pattern, and the bands are compared
byte for byte after the call.  Shapes have ragged tails (n, m and M off every tile size) so
that the last tiles, windows and token tiles are partial.
"""
import ctypes

import pytest
import torch

import bit_complex_valued_fairy2i_b300 as f2i
from bit_complex_valued_fairy2i_b300 import inputs

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side (a multiple of 256: the payload keeps its alignment)
PATTERN = 0xA5
L3 = f2i.LAYOUT_LUT


class Guarded:
    """A payload of `nbytes` inside a buffer with a guard band on each side."""

    def __init__(self, nbytes: int):
        self.nbytes = nbytes
        self.buf = torch.full((GUARD + nbytes + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")

    def view(self, dtype, shape):
        t = self.buf[GUARD:GUARD + self.nbytes]
        return t.view(dtype).view(shape) if len(shape) else t.view(dtype)

    def ptr(self) -> int:
        return self.buf.data_ptr() + GUARD

    def assert_intact(self, what: str):
        torch.cuda.synchronize()
        lo, hi = self.buf[:GUARD], self.buf[GUARD + self.nbytes:]
        assert bool((lo == PATTERN).all()), f"{what}: write before the buffer"
        assert bool((hi == PATTERN).all()), f"{what}: write past the buffer"


def _elem(dtype):
    return torch.tensor([], dtype=dtype).element_size()


def guarded_tensor(shape, dtype):
    n = 1
    for s in shape:
        n *= s
    g = Guarded(max(n * _elem(dtype), 16))
    return g, (g.view(dtype, shape) if n else None)


def guarded_packed(n, m, T, layout):
    gc = Guarded(f2i.codes_bytes(n, m, T, layout))
    gs = Guarded(f2i.scales_count(n, T) * 4)
    q = f2i.Packed(n, m, T, gc.view(torch.uint8, (gc.nbytes,)), gs.view(torch.float32, (2, T, 2, n)), layout)
    return q, gc, gs


SHAPES = [(37, 130), (33, 2049), (300, 704)]


@pytest.mark.parametrize("n,m", SHAPES)
def test_convert_writes_inside_U_and_W(n, m):
    lib = f2i.load_library()
    R = inputs.weight_R(95, 0, 2 * n, 2 * m).cuda()
    gu, U = guarded_tensor((n, m), torch.complex64)
    gw, W = guarded_tensor((n, m), torch.complex64)
    assert lib.fairy2i_convert(R.data_ptr(), 2 * n, 2 * m, U.data_ptr(), W.data_ptr(), None) == 0
    gu.assert_intact("convert U")
    gw.assert_intact("convert W")
    U2, W2 = f2i.convert(R)
    assert torch.equal(U, U2) and torch.equal(W, W2)


@pytest.mark.parametrize("layout", [2, L3])
@pytest.mark.parametrize("T", [1, 2, 3])
@pytest.mark.parametrize("n,m", SHAPES)
def test_quantize_writes_inside_codes_and_scales(n, m, T, layout):
    R = inputs.weight_R(95, 1, 2 * n, 2 * m).cuda()
    U, W = f2i.convert(R)
    for fused in (False, True):
        q, gc, gs = guarded_packed(n, m, T, layout)
        if fused:
            f2i.convert_quantize(R, T, out=q)
        else:
            f2i.quantize(U, W, T, out=q)
        gc.assert_intact(f"codes (fused={fused})")
        gs.assert_intact(f"scales (fused={fused})")
    # the canonical view of the codes
    lib = f2i.load_library()
    go, out = guarded_tensor((2, T, n, m), torch.uint8)
    d = q.desc()
    assert lib.fairy2i_unpack_codes(ctypes.byref(d), out.data_ptr(), None) == 0
    go.assert_intact("unpack_codes")


def _layer(n, m, T, layout, seed):
    R = inputs.weight_R(95, seed, 2 * n, 2 * m).cuda()
    return f2i.convert_quantize(R, T, layout=layout)


@pytest.mark.parametrize("algo,M", [("addsub", 3), ("mma", 1), ("mma", 9), ("tcgen05", 33), ("tcgen05_sp", 5)])
@pytest.mark.parametrize("n,m", [(37, 136), (300, 704)])
def test_layout2_linear_writes_inside_y(algo, M, n, m):
    q = _layer(n, m, 2, 2, 3)
    x = inputs.activations(95, 4, M, 2 * m).cuda()
    gy, y = guarded_tensor((M, 2 * n), torch.float32)
    f2i.linear(q, x, algo=algo, out=y)
    f2i.sync_status()
    gy.assert_intact(f"{algo} y")
    assert torch.isfinite(y).all()


@pytest.mark.parametrize("algo,M", [("lut", 1), ("lut", 3), ("lut", 4), ("tcgen05_dq", 33), ("tcgen05_dq", 300),
                                    ("tcgen05_dq16", 17), ("tcgen05_dq16", 300), ("auto", 12)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_layout3_linear_writes_inside_y_and_the_workspace(algo, M, out_dtype):
    """A group of three layers (one and several windows, ragged n and m), the workspace
    exactly as large as the size query says."""
    lib = f2i.load_library()
    shapes = [(40, 256), (37, 600), (131, 1032)]
    qs = [_layer(n, m, 2, L3, 10 + i) for i, (n, m) in enumerate(shapes)]
    xs = [inputs.activations(95, 20 + i, M, 2 * m).cuda() for i, (n, m) in enumerate(shapes)]
    descs = (f2i.PackedDesc * len(qs))(*[q.desc() for q in qs])
    need = int(lib.fairy2i_linear_workspace_bytes(descs, len(qs), M))
    gws = Guarded(max(need, 16))
    ws = gws.view(torch.uint8, (gws.nbytes,))
    guards = [guarded_tensor((M, 2 * n), out_dtype) for n, _ in shapes]
    ys = [g[1] for g in guards]
    f2i.linear_group(qs, xs, ys, algo=algo, ws=ws, out_dtype=out_dtype)
    f2i.sync_status()
    for i, (g, _) in enumerate(guards):
        g.assert_intact(f"{algo} y[{i}]")
    gws.assert_intact(f"{algo} workspace of {need} bytes")
    for y in ys:
        assert torch.isfinite(y.float()).all()


@pytest.mark.parametrize("M", [1, 2, 5])
def test_grad_x_writes_inside_gx(M):
    qs = [_layer(n, m, 2, 2, 30 + i) for i, (n, m) in enumerate([(37, 130), (64, 200)])]
    gen = torch.Generator().manual_seed(7)
    gys = [torch.randn((M, 2 * q.n), generator=gen).cuda() for q in qs]
    guards = [guarded_tensor((M, 2 * q.m), torch.float32) for q in qs]
    f2i.linear_grad_x_group(qs, gys, [g[1] for g in guards])
    f2i.sync_status()
    for i, (g, _) in enumerate(guards):
        g.assert_intact(f"grad_x gx[{i}]")

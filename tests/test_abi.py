"""C ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest
import torch

import bit_complex_valued_fairy2i_b300 as f2i
from bit_complex_valued_fairy2i_b300 import build as f2i_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fairy2i.h")


@pytest.fixture(scope="module")
def lib():
    f2i_build.build()
    return f2i.load_library()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fairy2i_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("fairy2i_convert", "fairy2i_quantize", "fairy2i_linear", "fairy2i_unpack_codes",
                     "fairy2i_last_error", "fairy2i_codes_bytes"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert sorted(f2i.EXPORTED) == _declared()


def test_sizes(lib):
    # 2 bits per code: 2 matrices x T planes x n x m codes / 4 codes per byte
    assert f2i.codes_bytes(2048, 2048, 2) == 2 * 2 * 2048 * 2048 // 4
    assert f2i.codes_bytes(5504, 2048, 2) == 2 * 2 * 5504 * 2048 // 4
    assert f2i.codes_bytes(2048, 5504, 2) == 2 * 2 * 2048 * 5504 // 4
    # padding to 16 rows x 64 columns
    assert f2i.codes_bytes(1, 1, 1) == 2 * 256
    assert f2i.codes_bytes(9, 65, 1) == 2 * 2 * 256
    assert f2i.codes_bytes(17, 65, 1) == 2 * 2 * 2 * 256
    assert f2i.scales_count(100, 3) == 4 * 3 * 100
    assert f2i.codes_bytes(0, 4, 1) == 0 and f2i.codes_bytes(4, 4, 9) == 0
    assert lib.fairy2i_layout_version() == f2i.LAYOUT_VERSION


def test_block_packed_bytes_match_the_stated_figure(lib):
    """One LLaMA-2-7B block at T=2: codes + fp32 scales = 51,273,728 bytes."""
    shapes = [(2048, 2048)] * 4 + [(5504, 2048)] * 2 + [(2048, 5504)]
    total = sum(f2i.codes_bytes(n, m, 2) + 4 * f2i.scales_count(n, 2) for n, m in shapes)
    assert total == 51_273_728


def _err(lib):
    return lib.fairy2i_last_error().decode()


def test_convert_rejects_bad_arguments(lib):
    p = ctypes.c_void_p(256)
    assert lib.fairy2i_convert(None, 4, 4, p, p, None) == 1
    assert lib.fairy2i_convert(p, 3, 4, p, p, None) == 2
    assert "even" in _err(lib)
    assert lib.fairy2i_convert(p, 4, 0, p, p, None) == 2
    assert lib.fairy2i_convert(ctypes.c_void_p(258), 4, 4, p, p, None) == 1
    assert "aligned" in _err(lib)


def _desc(n=4, m=4, T=1, codes=256, scales=256, version=f2i.LAYOUT_VERSION):
    return f2i.PackedDesc(version, T, n, m, codes, scales)


def test_quantize_rejects_bad_arguments(lib):
    p = ctypes.c_void_p(256)
    d = _desc()
    assert lib.fairy2i_quantize(None, p, 4, 4, 1, ctypes.byref(d), None) == 1
    bad = _desc(version=99)
    assert lib.fairy2i_quantize(p, p, 4, 4, 1, ctypes.byref(bad), None) == 1
    assert lib.fairy2i_quantize(p, p, 4, 4, 2, ctypes.byref(d), None) == 2  # T mismatch
    t9 = _desc(T=9)
    assert lib.fairy2i_quantize(p, p, 4, 4, 9, ctypes.byref(t9), None) == 4
    big = _desc(m=16385)
    assert lib.fairy2i_quantize(p, p, 4, 16385, 1, ctypes.byref(big), None) == 4
    unal = _desc(codes=264)
    assert lib.fairy2i_quantize(p, p, 4, 4, 1, ctypes.byref(unal), None) == 1
    assert lib.fairy2i_quantize(p, p, 4, 4, 1, None, None) == 1


def test_linear_rejects_bad_arguments(lib):
    p = ctypes.c_void_p(256)
    d = _desc()
    assert lib.fairy2i_linear(None, p, 1, p, None) == 1
    assert lib.fairy2i_linear(ctypes.byref(d), None, 1, p, None) == 1
    assert lib.fairy2i_linear(ctypes.byref(d), None, 0, None, None) == 0  # M = 0: pointers unused
    assert lib.fairy2i_linear(ctypes.byref(d), p, -1, p, None) == 2
    assert lib.fairy2i_linear(ctypes.byref(d), ctypes.c_void_p(258), 1, p, None) == 1
    assert lib.fairy2i_linear_ex(ctypes.byref(d), p, 1, p, 8, None) == 1  # no such algo
    assert lib.fairy2i_linear_ex(ctypes.byref(d), p, 1, p, 7, None) == 4  # the fp16 dequantized GEMM: layout 3
    assert lib.fairy2i_linear_ex(ctypes.byref(d), p, 1, p, -1, None) == 1
    assert lib.fairy2i_linear_ex(ctypes.byref(d), p, 1, p, 5, None) == 4  # the table lookup reads layout 3 only
    assert lib.fairy2i_linear_ex(ctypes.byref(d), p, 1, p, 6, None) == 4  # so does the dequantized GEMM
    # the sparse tensor-core decode takes at most 8 tokens and 4 stages (checked before any launch)
    assert lib.fairy2i_linear_ex(ctypes.byref(d), p, 9, p, 4, None) == 4
    t5 = _desc(T=5)
    assert lib.fairy2i_linear_ex(ctypes.byref(t5), p, 1, p, 4, None) == 4
    zero = _desc(n=0)
    assert lib.fairy2i_linear(ctypes.byref(zero), p, 1, p, None) == 2
    # M = 0 with valid arguments is a no-op that launches nothing
    assert lib.fairy2i_linear(ctypes.byref(d), p, 0, p, None) == 0
    descs = (f2i.PackedDesc * 1)(d)
    arr = (ctypes.c_void_p * 1)(256)
    assert lib.fairy2i_linear_group(descs, arr, arr, 0, 1, 0, None) == 1
    assert lib.fairy2i_linear_group(descs, arr, arr, 300, 1, 0, None) == 1


def test_linear_grad_x_rejects_bad_arguments(lib):
    p = ctypes.c_void_p(256)
    d = _desc()
    assert lib.fairy2i_linear_grad_x(None, p, 1, p, None) == 1
    assert lib.fairy2i_linear_grad_x(ctypes.byref(d), None, 1, p, None) == 1
    assert lib.fairy2i_linear_grad_x(ctypes.byref(d), p, -1, p, None) == 2
    assert lib.fairy2i_linear_grad_x(ctypes.byref(d), ctypes.c_void_p(260), 1, p, None) == 1
    assert lib.fairy2i_linear_grad_x(ctypes.byref(d), p, 0, p, None) == 0  # no tokens: nothing launched
    assert lib.fairy2i_linear_grad_x(ctypes.byref(d), p, 20000, p, None) == 4


def test_linear_grad_x_group_rejects_bad_arguments(lib):
    d = _desc()
    descs = (f2i.PackedDesc * 2)(d, _desc(T=3))
    arr = (ctypes.c_void_p * 2)(256, 512)
    assert lib.fairy2i_linear_grad_x_group(descs, arr, arr, 0, 1, None) == 1  # count 0
    assert lib.fairy2i_linear_grad_x_group(descs, arr, arr, 300, 1, None) == 1  # count above 256
    assert lib.fairy2i_linear_grad_x_group(descs, None, arr, 1, 1, None) == 1  # NULL array
    assert lib.fairy2i_linear_grad_x_group(descs, arr, arr, 2, 1, None) == 2  # mixed T
    assert lib.fairy2i_linear_grad_x_group(descs, arr, arr, 1, -1, None) == 2  # negative M
    assert lib.fairy2i_linear_grad_x_group(descs, arr, arr, 1, 0, None) == 0  # no tokens: nothing launched
    nulls = (ctypes.c_void_p * 1)(None)
    assert lib.fairy2i_linear_grad_x_group(descs, nulls, arr, 1, 1, None) == 1  # NULL gradient


def test_convert_quantize_rejects_bad_arguments(lib):
    p = ctypes.c_void_p(256)
    d = _desc(n=2, m=2, T=1)
    assert lib.fairy2i_convert_quantize(None, 4, 4, 1, ctypes.byref(d), None) == 1
    assert lib.fairy2i_convert_quantize(p, 3, 4, 1, ctypes.byref(d), None) == 2
    assert lib.fairy2i_convert_quantize(p, 4, 4, 2, ctypes.byref(d), None) == 2  # T differs
    assert lib.fairy2i_convert_quantize(p, 6, 4, 1, ctypes.byref(d), None) == 2  # n differs


def test_selftest_rejects_bad_limit(lib):
    assert lib.fairy2i_selftest_bounded_wait(0, None) == 1
    assert lib.fairy2i_selftest_bounded_wait(2000000, None) == 1


def test_unpack_rejects_bad_arguments(lib):
    d = _desc()
    assert lib.fairy2i_unpack_codes(ctypes.byref(d), None, None) == 1
    assert lib.fairy2i_unpack_codes(None, ctypes.c_void_p(256), None) == 1


def test_python_wrappers_reject_host_tensors(lib):
    """The Python layer marshals arguments only: host tensors are refused before
    anything reaches the library (there is no CPU fallback)."""
    q = f2i.Packed(4, 8, 2, torch.zeros(f2i.codes_bytes(4, 8, 2), dtype=torch.uint8),
                   torch.zeros((2, 2, 2, 4)))
    with pytest.raises(ValueError):
        f2i.linear(q, torch.zeros((1, 16), dtype=torch.bfloat16))  # host tensor
    with pytest.raises(ValueError):
        f2i.linear_grad_x(q, torch.zeros((1, 8)))  # host tensor
    with pytest.raises(ValueError):
        f2i.GroupCall([q], [torch.zeros((1, 16), dtype=torch.bfloat16)])  # host tensor
    # the algorithm names map onto the header's fairy2i_algo values
    assert f2i.ALGO == {"auto": 0, "addsub": 1, "mma": 2, "tcgen05": 3, "tcgen05_sp": 4, "lut": 5,
                        "tcgen05_dq": 6, "tcgen05_dq16": 7}


def test_layout3_sizes(lib):
    L3 = f2i.LAYOUT_LUT
    # 2 bits per code for every LLaMA-2-7B projection (n a multiple of 32, m of 64)
    for n, m in [(2048, 2048), (5504, 2048), (2048, 5504)]:
        assert f2i.codes_bytes(n, m, 2, L3) == 2 * 2 * n * m // 4
    # padding: rows to 32; a last partial window keeps 1, 2 or 4 blocks of 64 columns (3 -> 4)
    assert f2i.codes_bytes(1, 1, 1, L3) == 2 * 512
    assert f2i.codes_bytes(1, 129, 1, L3) == 2 * 512 * 4
    assert f2i.codes_bytes(1, 100, 1, L3) == 2 * 512 * 2
    assert f2i.codes_bytes(33, 256, 1, L3) == 2 * 2 * 512 * 4
    assert f2i.codes_bytes(1, 257, 3, L3) == 6 * 512 * 5
    assert f2i.codes_bytes(4, 4, 1, 7) == 0


def test_layout3_workspace_bytes(lib):
    """The larger of the table lookup's need (one float2 partial output per (row of a
    32-row tile, window of 256 columns, token of a launch) for the layers with several
    windows) and, for m a multiple of 8, the fp16 dequantized GEMM's (per layer of a
    launch, the fp16 copy of x and a float per token, each rounded up to 256 bytes)."""
    def ws(descs, M):
        arr = (f2i.PackedDesc * len(descs))(*descs)
        return lib.fairy2i_linear_workspace_bytes(arr, len(descs), M)
    L3 = f2i.LAYOUT_LUT
    q = _desc(n=2048, m=2048, T=2, version=L3)
    assert ws([q], 1) == 64 * 8 * 32 * 8
    # at T = 2, launches of 2 tokens (the first of 3 when M is odd) share it
    assert ws([q], 2) == ws([q], 4) == ws([q], 10) == 64 * 8 * 2 * 32 * 8
    assert ws([q], 3) == ws([q], 9) == 64 * 8 * 3 * 32 * 8
    assert ws([_desc(n=2048, m=2048, T=3, version=L3)], 9) == 64 * 8 * 2 * 32 * 8
    # one window: the table lookup writes y directly; the fp16 copy of one token remains
    assert ws([_desc(n=100, m=256, T=2, version=L3)], 1) == 1024 + 256
    assert ws([_desc(n=100, m=250, T=2, version=L3)], 1) == 0  # and none for m not a multiple of 8
    r256 = lambda v: (v + 255) // 256 * 256
    assert ws([q], 2048) == r256(2048 * 4 * 2048) + r256(2048 * 4)
    # nine layers: launches of 8 and 1 reuse the workspace, so the larger launch sets it
    nine = [_desc(n=64, m=8 * (i + 1), T=2, version=L3) for i in range(9)]
    assert ws(nine, 100) == sum(r256(100 * 4 * 8 * (i + 1)) + r256(400) for i in range(8))
    assert ws([_desc(n=2048, m=2048, T=2)], 1) == 0  # layout 2
    assert ws([q], 0) == 0


def test_dq16_host_errors(lib):
    """The fp16 dequantized GEMM's argument checks (all before any launch)."""
    p = ctypes.c_void_p(256)
    L3 = f2i.LAYOUT_LUT
    d = _desc(n=4, m=600, T=2, version=L3)
    assert lib.fairy2i_linear_ex(ctypes.byref(d), p, 16, p, 7, None) == 4  # needs a workspace
    assert "workspace" in _err(lib)
    assert lib.fairy2i_linear_ws(ctypes.byref(d), p, 16, p, 7, None, 0, None) == 1  # workspace missing
    assert lib.fairy2i_linear_ws(ctypes.byref(d), p, 16, p, 7, p, 16, None) == 1  # too small
    assert lib.fairy2i_linear_ws(ctypes.byref(d), p, 16, p, 7, ctypes.c_void_p(272), 1 << 20, None) == 1
    d7 = _desc(n=4, m=100, T=2, version=L3)
    assert lib.fairy2i_linear_ws(ctypes.byref(d7), p, 16, p, 7, p, 1 << 20, None) == 4  # m not a multiple of 8
    d2 = _desc(n=4, m=600, T=2)
    assert lib.fairy2i_linear_ws(ctypes.byref(d2), p, 16, p, 7, p, 1 << 20, None) == 4  # layout 2
    assert lib.fairy2i_linear_ex(ctypes.byref(d), p, 16, p, 8, None) == 1  # no such algo


def test_bf16_output_host_errors(lib):
    """fairy2i_linear_group_ws_out: an unknown output type, and bfloat16 outputs for
    layout-2 layers, are refused before any launch."""
    p = ctypes.c_void_p(256)
    xp = (ctypes.c_void_p * 1)(p)
    yp = (ctypes.c_void_p * 1)(p)
    d3 = (f2i.PackedDesc * 1)(_desc(n=4, m=600, T=2, version=f2i.LAYOUT_LUT))
    assert lib.fairy2i_linear_group_ws_out(d3, xp, yp, 1, 16, 0, 2, p, 1 << 20, None) == 1
    d2 = (f2i.PackedDesc * 1)(_desc(n=4, m=600, T=2))
    assert lib.fairy2i_linear_group_ws_out(d2, xp, yp, 1, 16, 0, 1, p, 1 << 20, None) == 4
    assert "layout-3" in _err(lib)


def test_layout3_host_errors(lib):
    p = ctypes.c_void_p(256)
    L3 = f2i.LAYOUT_LUT
    d = _desc(n=4, m=600, T=2, version=L3)
    # without a workspace the table lookup is refused; m = 600 is a multiple of 8, so AUTO takes
    # the dequantized GEMM (which would launch, so it is not called here without a GPU)
    assert lib.fairy2i_linear_ex(ctypes.byref(d), p, 1, p, 5, None) == 4
    assert "workspace" in _err(lib)
    assert lib.fairy2i_linear_ws(ctypes.byref(d), p, 1, p, 0, None, 0, None) == 1  # workspace missing
    assert lib.fairy2i_linear_ws(ctypes.byref(d), p, 1, p, 0, p, 16, None) == 1  # workspace too small
    assert lib.fairy2i_linear_ws(ctypes.byref(d), p, 1, p, 0, ctypes.c_void_p(272), 1 << 20, None) == 1  # misaligned
    assert lib.fairy2i_linear_ws(ctypes.byref(d), p, 1, p, 2, p, 1 << 20, None) == 4  # mma does not read layout 3
    t5 = _desc(n=4, m=600, T=5, version=L3)
    assert lib.fairy2i_linear_ws(ctypes.byref(t5), p, 1, p, 0, p, 1 << 20, None) == 4
    assert lib.fairy2i_linear_ws(ctypes.byref(d), p, 0, p, 0, None, 0, None) == 0  # no tokens
    # the dequantized GEMM reads x by TMA in two halves: m must be a multiple of 8; the plain
    # entry (no workspace) then has nothing to run, explicitly or through AUTO (no launch)
    d100 = _desc(n=4, m=100, T=2, version=L3)
    assert lib.fairy2i_linear_ex(ctypes.byref(d100), p, 20, p, 6, None) == 4
    assert "multiple of 8" in _err(lib)
    assert lib.fairy2i_linear(ctypes.byref(d100), p, 20, p, None) == 4
    assert lib.fairy2i_linear_ws(ctypes.byref(d100), p, 20, p, 6, p, 1 << 20, None) == 4
    # layout-2 descriptors are refused by the layout-3 kernels before any launch
    d2 = _desc(n=4, m=600, T=2)
    assert lib.fairy2i_linear_ex(ctypes.byref(d2), p, 20, p, 6, None) == 4
    descs = (f2i.PackedDesc * 2)(d, _desc(n=4, m=600, T=2))
    arr = (ctypes.c_void_p * 2)(256, 512)
    assert lib.fairy2i_linear_group_ws(descs, arr, arr, 2, 1, 0, p, 1 << 20, None) == 2  # mixed layouts
    assert lib.fairy2i_linear_grad_x(ctypes.byref(d), p, 1, p, None) == 4  # the gradient reads layout 2


def test_mma_decode_rejects_code_planes_beyond_32bit_offsets(lib):
    """The mma decode addresses a layer's planes with 32-bit offsets: a layer whose
    2T planes exceed 4 GB is refused on the host (AUTO takes the add/subtract path)."""
    p = ctypes.c_void_p(256)
    big = _desc(n=300000, m=16384, T=2)
    assert lib.fairy2i_linear_ex(ctypes.byref(big), p, 1, p, 2, None) == 4
    assert "32-bit" in _err(lib)


def test_packed_descriptor_follows_its_tensors(lib):
    """The binding builds a layer's C descriptor once; assigning a field, or code and scale
    storage that moved, gives a fresh one with the current pointers and shape."""
    codes = torch.zeros(64, dtype=torch.uint8)
    scales = torch.zeros(2 * 2 * 2 * 8)
    q = f2i.Packed(8, 16, 2, codes, scales, layout=3)
    d1 = q.desc()
    assert q.desc() is d1
    assert (d1.n, d1.m, d1.T, d1.version) == (8, 16, 2, 3)
    assert d1.codes == codes.data_ptr() and d1.scales == scales.data_ptr()
    q.codes = torch.zeros(128, dtype=torch.uint8)  # a new tensor in the field
    d2 = q.desc()
    assert d2 is not d1 and d2.codes == q.codes.data_ptr()
    q.n = 4  # any field assignment
    assert q.desc().n == 4
    q.scales.set_(torch.zeros(64).untyped_storage())  # same tensor object, storage moved
    assert q.desc().scales == q.scales.data_ptr()

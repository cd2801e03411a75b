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
    assert lib.fairy2i_linear_ex(ctypes.byref(d), p, 1, p, 7, None) == 1
    assert lib.fairy2i_linear_ex(ctypes.byref(d), p, 1, p, 5, None) == 1
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
    # the algorithm names map onto the header's fairy2i_algo values
    assert f2i.ALGO == {"auto": 0, "addsub": 1, "mma": 2, "tcgen05": 3, "tcgen05_sp": 4}

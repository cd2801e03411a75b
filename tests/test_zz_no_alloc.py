"""The no-allocation entry point (fairy2i_linear_group_static), checked on the GPU.

Some callers may not allocate device memory at all (a plugin whose host
process owns every byte of the GPU through its own allocator, a real-time loop
that forbids allocation after start-up).  For them the table-lookup decode can
use a fixed scratch array inside the library instead of a caller workspace.
This file is named to be collected last, so that a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import bit_complex_valued_fairy2i_b300 as f2i
from bit_complex_valued_fairy2i_b300 import build as f2i_build
from bit_complex_valued_fairy2i_b300 import inputs

pytestmark = pytest.mark.gpu

REL_L2 = 1e-3  # the outputs' bar used by every parity test


def _rel_l2(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


@pytest.fixture(scope="module")
def lib():
    f2i_build.build()
    return f2i.load_library()


def _layers():
    """Layout-3 layers with several windows (so partial outputs go through the scratch)."""
    qs = []
    for i, (n, m) in enumerate([(300, 700), (5504 // 8, 2048), (40, 5504)]):
        R = inputs.weight_R(96, i, 2 * n, 2 * m).cuda()
        qs.append(f2i.convert_quantize(R, 2, layout=f2i.LAYOUT_LUT))
    return qs


def _call_static(lib, qs, xs):
    ys = [torch.full((x.shape[0], 2 * q.n), float("nan"), device="cuda") for q, x in zip(qs, xs)]
    descs = (f2i.PackedDesc * len(qs))(*[q.desc() for q in qs])
    xp = (ctypes.c_void_p * len(qs))(*[x.data_ptr() for x in xs])
    yp = (ctypes.c_void_p * len(qs))(*[y.data_ptr() for y in ys])
    stream = torch.cuda.current_stream().cuda_stream
    st = lib.fairy2i_linear_group_static(descs, xp, yp, len(qs), xs[0].shape[0], stream)
    assert st == 0, lib.fairy2i_last_error().decode()
    torch.cuda.synchronize()
    return ys


def test_static_scratch_matches_workspace_entry_point_twice(lib):
    """Two calls in a row through the C ABI, each against fairy2i_linear_group_ws
    with a caller workspace: the second call sees the first call's leftovers in
    the shared scratch and must not depend on them."""
    qs = _layers()
    for call, M in enumerate((3, 1)):
        xs = [inputs.activations(96, 10 * call + i, M, 2 * q.m).cuda() for i, q in enumerate(qs)]
        got = _call_static(lib, qs, xs)
        want = f2i.linear_group(qs, xs)  # the workspace entry point
        torch.cuda.synchronize()
        for g, w in zip(got, want):
            assert _rel_l2(g.cpu().numpy(), w.cpu().numpy()) <= REL_L2


def test_static_scratch_refuses_what_does_not_fit(lib):
    """Layers whose partial outputs exceed the fixed scratch are refused with a
    message, and nothing is launched."""
    q = f2i.Packed.empty(16384, 16384, 2, "cuda", f2i.LAYOUT_LUT)
    x = torch.zeros((4, 2 * q.m), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((4, 2 * q.n), device="cuda")
    descs = (f2i.PackedDesc * 1)(q.desc())
    xp = (ctypes.c_void_p * 1)(x.data_ptr())
    yp = (ctypes.c_void_p * 1)(y.data_ptr())
    st = lib.fairy2i_linear_group_static(descs, xp, yp, 1, 4, None)
    assert st == 4 and "scratch" in lib.fairy2i_last_error().decode()
    assert not torch.any(y)

"""Fairy2i widely-linear 2-bit complex linear layer on B300 (sm_103a).

Thin Python binding over the C ABI in ``include/fairy2i.h`` (libfairy2i.so,
built in-tree by ``build.py``).  This module only marshals arguments: device
memory comes from PyTorch tensors, every step of the layer runs in the
library's CUDA kernels.  There is no CPU fallback; if the library or a GPU is
missing, calls raise.

    U, W = convert(R)                 # R: cuda float32 [2n, 2m]
    q = quantize(U, W, T=2)           # packed 2-bit codes + per-row scales
    y = linear(q, x)                  # x: cuda bfloat16 [M, 2m] -> y float32 [M, 2n]

    q3 = quantize(U, W, T=2, layout=3)   # the table-lookup decode layout
    y = linear(q3, x)                    # table-lookup decode; workspace kept per (device, stream)
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfairy2i.so")

OK = 0
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "SHAPE", 3: "NONFINITE", 4: "UNSUPPORTED", 5: "CUDA",
                6: "TIMEOUT"}
ALGO = {"auto": 0, "addsub": 1, "mma": 2, "tcgen05": 3, "tcgen05_sp": 4, "lut": 5, "tcgen05_dq": 6, "tcgen05_dq16": 7}
LAYOUT_VERSION = 2
LAYOUT_LUT = 3

# every extern "C" symbol declared in include/fairy2i.h
EXPORTED = (
    "fairy2i_codes_bytes", "fairy2i_scales_count", "fairy2i_convert", "fairy2i_quantize",
    "fairy2i_linear", "fairy2i_linear_ex", "fairy2i_linear_group", "fairy2i_unpack_codes",
    "fairy2i_sync_status", "fairy2i_last_error", "fairy2i_layout_version", "fairy2i_selftest_bounded_wait",
    "fairy2i_convert_quantize", "fairy2i_linear_grad_x", "fairy2i_linear_grad_x_group",
    "fairy2i_codes_bytes_layout", "fairy2i_linear_ws", "fairy2i_linear_group_ws", "fairy2i_linear_workspace_bytes",
    "fairy2i_linear_group_static", "fairy2i_linear_group_ws_out",
)
OUT = {torch.float32: 0, torch.bfloat16: 1}  # fairy2i_out


class Fairy2iError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class PackedDesc(ctypes.Structure):
    _fields_ = [("version", ctypes.c_int32), ("T", ctypes.c_int32), ("n", ctypes.c_int64),
                ("m", ctypes.c_int64), ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libfairy2i.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libfairy2i.so not found at {path}; run bit_complex_valued_fairy2i_b300/build.py")
    lib = ctypes.CDLL(path)
    P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    PD = ctypes.POINTER(PackedDesc)
    sig = {
        "fairy2i_codes_bytes": (SZ, [I64, I64, I32]),
        "fairy2i_scales_count": (SZ, [I64, I32]),
        "fairy2i_convert": (ctypes.c_int, [P, I64, I64, P, P, P]),
        "fairy2i_quantize": (ctypes.c_int, [P, P, I64, I64, I32, PD, P]),
        "fairy2i_linear": (ctypes.c_int, [PD, P, I64, P, P]),
        "fairy2i_linear_ex": (ctypes.c_int, [PD, P, I64, P, ctypes.c_int, P]),
        "fairy2i_linear_group": (ctypes.c_int, [PD, ctypes.POINTER(P), ctypes.POINTER(P), I32, I64,
                                                ctypes.c_int, P]),
        "fairy2i_unpack_codes": (ctypes.c_int, [PD, P, P]),
        "fairy2i_sync_status": (ctypes.c_int, [P]),
        "fairy2i_last_error": (ctypes.c_char_p, []),
        "fairy2i_layout_version": (I32, []),
        "fairy2i_selftest_bounded_wait": (ctypes.c_int, [I32, P]),
        "fairy2i_convert_quantize": (ctypes.c_int, [P, I64, I64, I32, PD, P]),
        "fairy2i_linear_grad_x": (ctypes.c_int, [PD, P, I64, P, P]),
        "fairy2i_linear_grad_x_group": (ctypes.c_int, [PD, ctypes.POINTER(P), ctypes.POINTER(P), I32, I64, P]),
        "fairy2i_codes_bytes_layout": (SZ, [I64, I64, I32, I32]),
        "fairy2i_linear_ws": (ctypes.c_int, [PD, P, I64, P, ctypes.c_int, P, SZ, P]),
        "fairy2i_linear_group_ws": (ctypes.c_int, [PD, ctypes.POINTER(P), ctypes.POINTER(P), I32, I64, ctypes.c_int,
                                                   P, SZ, P]),
        "fairy2i_linear_workspace_bytes": (SZ, [PD, I32, I64]),
        "fairy2i_linear_group_static": (ctypes.c_int, [PD, ctypes.POINTER(P), ctypes.POINTER(P), I32, I64, P]),
        "fairy2i_linear_group_ws_out": (ctypes.c_int, [PD, ctypes.POINTER(P), ctypes.POINTER(P), I32, I64,
                                                       ctypes.c_int, ctypes.c_int, P, SZ, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    if lib.fairy2i_layout_version() != LAYOUT_VERSION:
        raise ImportError("libfairy2i.so layout version mismatch")
    _lib = lib
    return lib


def _check(status: int):
    if status != OK:
        raise Fairy2iError(status, load_library().fairy2i_last_error().decode())


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device_index: int | None = None) -> int:
    """The CUDA stream handle: ``stream`` itself, else the current stream of ``device_index``
    (or of the current device)."""
    if stream is None:
        if _raw_stream is not None:
            return int(_raw_stream(torch.cuda.current_device() if device_index is None else device_index))
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def codes_bytes(n: int, m: int, T: int, layout: int = LAYOUT_VERSION) -> int:
    return int(load_library().fairy2i_codes_bytes_layout(n, m, T, layout))


def scales_count(n: int, T: int) -> int:
    return int(load_library().fairy2i_scales_count(n, T))


@dataclass
class Packed:
    """Packed quantized layer: device codes (uint8) and scales [2][T][2][n].
    ``layout`` is the code layout version: 2 (every kernel) or 3 (the table-lookup decode)."""
    n: int
    m: int
    T: int
    codes: torch.Tensor
    scales: torch.Tensor
    layout: int = LAYOUT_VERSION

    def desc(self) -> PackedDesc:
        """The C descriptor, built once and rebuilt after any field is assigned or when the
        code or scale storage has moved."""
        d = self.__dict__.get("_desc")
        if d is None or d.codes != self.codes.data_ptr() or d.scales != self.scales.data_ptr():
            d = PackedDesc(self.layout, self.T, self.n, self.m, self.codes.data_ptr(), self.scales.data_ptr())
            self.__dict__["_desc"] = d
        return d

    def __setattr__(self, name, value):
        self.__dict__.pop("_desc", None)
        object.__setattr__(self, name, value)

    @property
    def nbytes(self) -> int:
        """Packed bytes streamed per evaluation: codes + scales."""
        return self.codes.numel() + 4 * self.scales.numel()

    @staticmethod
    def empty(n: int, m: int, T: int, device="cuda", layout: int = LAYOUT_VERSION) -> "Packed":
        nb = codes_bytes(n, m, T, layout)
        ns = scales_count(n, T)
        if nb == 0 or ns == 0:
            raise Fairy2iError(4, f"unsupported shape n={n} m={m} T={T} layout={layout}")
        codes = torch.empty(nb, dtype=torch.uint8, device=device)
        scales = torch.empty(ns, dtype=torch.float32, device=device).view(2, T, 2, n)
        return Packed(n, m, T, codes, scales, layout)


def convert(R: torch.Tensor, stream=None):
    """Real [2n, 2m] float32 weight -> complex64 (U, W), each [n, m]."""
    _dev(R, "R")
    if R.dtype != torch.float32 or R.dim() != 2:
        raise ValueError("R must be a 2-D float32 tensor")
    n, m = R.shape[0] // 2, R.shape[1] // 2
    U = torch.empty((n, m), dtype=torch.complex64, device=R.device)
    W = torch.empty((n, m), dtype=torch.complex64, device=R.device)
    _check(load_library().fairy2i_convert(R.data_ptr(), R.shape[0], R.shape[1], U.data_ptr(), W.data_ptr(),
                                          _stream(stream)))
    return U, W


def quantize(U: torch.Tensor, W: torch.Tensor, T: int = 2, out: Packed | None = None, stream=None,
             check: bool = True, layout: int = LAYOUT_VERSION) -> Packed:
    """Phase-aware recursive residual quantization of U and W (complex64 [n, m]) into
    code layout ``layout`` (ignored when ``out`` is given: its own layout is written).
    With ``check`` the stream is synchronized and a non-finite weight raises."""
    _dev(U, "U")
    _dev(W, "W")
    if U.dtype != torch.complex64 or W.dtype != torch.complex64 or U.shape != W.shape or U.dim() != 2:
        raise ValueError("U and W must be complex64 tensors of the same 2-D shape")
    n, m = U.shape
    q = out if out is not None else Packed.empty(n, m, T, U.device, layout)
    d = q.desc()
    _check(load_library().fairy2i_quantize(U.data_ptr(), W.data_ptr(), n, m, T, ctypes.byref(d), _stream(stream)))
    if check:
        sync_status(stream)
    return q


def convert_quantize(R: torch.Tensor, T: int = 2, out: Packed | None = None, stream=None,
                     check: bool = True, layout: int = LAYOUT_VERSION) -> Packed:
    """Real [2n, 2m] float32 weight -> packed layer, in one pass (the same codes and
    scales as quantize(*convert(R), T))."""
    _dev(R, "R")
    if R.dtype != torch.float32 or R.dim() != 2:
        raise ValueError("R must be a 2-D float32 tensor")
    n, m = R.shape[0] // 2, R.shape[1] // 2
    q = out if out is not None else Packed.empty(n, m, T, R.device, layout)
    d = q.desc()
    _check(load_library().fairy2i_convert_quantize(R.data_ptr(), R.shape[0], R.shape[1], T, ctypes.byref(d),
                                                   _stream(stream)))
    if check:
        sync_status(stream)
    return q


_workspaces: dict = {}
_ws_bytes: dict = {}  # (layer shapes, M) -> workspace bytes


def workspace(qs, M: int, device, stream=None, descs=None) -> torch.Tensor | None:
    """The device scratch of the table-lookup decode for these layers and token count,
    kept per (device, stream) and grown when a call needs more (None if none is needed).
    Calls on one stream run in order, so they can share it."""
    count = len(qs)
    shapes = (tuple((q.layout, q.T, q.n, q.m) for q in qs), M)
    need = _ws_bytes.get(shapes)
    if need is None:
        if descs is None:
            descs = (PackedDesc * count)(*[q.desc() for q in qs])
        need = int(load_library().fairy2i_linear_workspace_bytes(descs, count, M))
        _ws_bytes[shapes] = need
    if need == 0:
        return None
    dev = torch.device(device)
    index = dev.index if dev.index is not None else torch.cuda.current_device()
    key = (index, _stream(stream, index))
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
        _workspaces[key] = ws
    return ws


def linear(q: Packed, x: torch.Tensor, algo: str = "auto", out: torch.Tensor | None = None,
           stream=None, ws: torch.Tensor | None = None) -> torch.Tensor:
    """y = U^ x + W^ conj(x) for x bfloat16 [M, 2m] ([Re x | Im x] rows) -> y float32 [M, 2n].
    A layout-3 layer goes through the table-lookup decode with workspace ``ws`` (by default
    the one kept for this device and stream)."""
    _dev(x, "x")
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] != 2 * q.m:
        raise ValueError(f"x must be bfloat16 [M, {2 * q.m}]")
    y = out if out is not None else torch.empty((x.shape[0], 2 * q.n), dtype=torch.float32, device=x.device)
    d = q.desc()
    s = _stream(stream, x.get_device())
    if q.layout == LAYOUT_LUT:
        if ws is None:
            ws = workspace([q], x.shape[0], x.device, s)
        wp, wn = (ws.data_ptr(), ws.numel()) if ws is not None else (None, 0)
        _check(load_library().fairy2i_linear_ws(ctypes.byref(d), x.data_ptr(), x.shape[0], y.data_ptr(), ALGO[algo],
                                                wp, wn, s))
        return y
    _check(load_library().fairy2i_linear_ex(ctypes.byref(d), x.data_ptr(), x.shape[0], y.data_ptr(), ALGO[algo], s))
    return y


def linear_grad_x(q: Packed, gy: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """dL/dx = U^^H g + W^^T conj(g) for gy float32 [M, 2n] ([dRe y | dIm y]) -> gx float32 [M, 2m]."""
    _dev(gy, "gy")
    if gy.dtype != torch.float32 or gy.dim() != 2 or gy.shape[1] != 2 * q.n:
        raise ValueError(f"gy must be float32 [M, {2 * q.n}]")
    gx = out if out is not None else torch.empty((gy.shape[0], 2 * q.m), dtype=torch.float32, device=gy.device)
    d = q.desc()
    _check(load_library().fairy2i_linear_grad_x(ctypes.byref(d), gy.data_ptr(), gy.shape[0], gx.data_ptr(),
                                                _stream(stream)))
    return gx


def linear_grad_x_group(qs, gys, outs=None, stream=None):
    """Input gradients of several layers (same T and token count) in one launch."""
    count = len(qs)
    M = gys[0].shape[0]
    if outs is None:
        outs = [torch.empty((M, 2 * q.m), dtype=torch.float32, device=g.device) for q, g in zip(qs, gys)]
    for q, g, gx in zip(qs, gys, outs):
        _dev(g, "gy")
        _dev(gx, "gx")
        if g.dtype != torch.float32 or g.shape != (M, 2 * q.n) or gx.shape != (M, 2 * q.m):
            raise ValueError("group members need matching gy [M, 2n] and gx [M, 2m] float32")
    descs = (PackedDesc * count)(*[q.desc() for q in qs])
    gp = (ctypes.c_void_p * count)(*[g.data_ptr() for g in gys])
    xp = (ctypes.c_void_p * count)(*[gx.data_ptr() for gx in outs])
    _check(load_library().fairy2i_linear_grad_x_group(descs, gp, xp, count, M, _stream(stream)))
    return outs


class GroupCall:
    """A grouped linear call prepared once: layers, inputs, outputs, algorithm, stream and
    workspace fixed, the C arguments (descriptor array, pointer arrays) built here.  Calling it
    issues the launches again with no per-call marshalling -- for loops that reuse the same
    buffers (a serving step, a benchmark): the tensors' contents may change between calls, the
    tensors themselves may not.  The stream is fixed too (the current one when prepared, unless
    given): prepare a call inside a CUDA-graph capture to have it captured.  ``ys`` (allocated
    if not given) are the outputs."""

    def __init__(self, qs, xs, ys=None, algo: str = "auto", stream=None, ws: torch.Tensor | None = None,
                 out_dtype=torch.float32):
        count = len(qs)
        M = xs[0].shape[0]
        if out_dtype not in OUT:
            raise ValueError("out_dtype must be torch.float32 or torch.bfloat16")
        if ys is None:
            ys = [torch.empty((M, 2 * q.n), dtype=out_dtype, device=x.device) for q, x in zip(qs, xs)]
        for q, x, y in zip(qs, xs, ys):
            _dev(x, "x")
            _dev(y, "y")
            if x.dtype != torch.bfloat16 or x.shape != (M, 2 * q.m) or y.shape != (M, 2 * q.n) or y.dtype != out_dtype:
                raise ValueError("group members need matching x [M, 2m] bfloat16 and y [M, 2n] of out_dtype")
        lib = load_library()
        descs = (PackedDesc * count)(*[q.desc() for q in qs])
        xp = (ctypes.c_void_p * count)(*[x.data_ptr() for x in xs])
        yp = (ctypes.c_void_p * count)(*[y.data_ptr() for y in ys])
        s = _stream(stream, xs[0].get_device())
        if qs[0].layout == LAYOUT_LUT:
            if ws is None:
                ws = workspace(qs, M, xs[0].device, s, descs)
            wp, wn = (ws.data_ptr(), ws.numel()) if ws is not None else (None, 0)
            if out_dtype == torch.float32:
                self._fn, self._args = lib.fairy2i_linear_group_ws, (descs, xp, yp, count, M, ALGO[algo], wp, wn, s)
            else:
                self._fn = lib.fairy2i_linear_group_ws_out
                self._args = (descs, xp, yp, count, M, ALGO[algo], OUT[out_dtype], wp, wn, s)
        else:
            if out_dtype != torch.float32:
                raise ValueError("bfloat16 outputs are written for layout-3 layers only")
            self._fn, self._args = lib.fairy2i_linear_group, (descs, xp, yp, count, M, ALGO[algo], s)
        # the tensors whose addresses the arguments hold stay alive with the call
        self._keep = (list(qs), list(xs), ws)
        self.ys = ys

    def __call__(self):
        _check(self._fn(*self._args))
        return self.ys


def linear_group(qs, xs, ys=None, algo: str = "auto", stream=None, ws: torch.Tensor | None = None,
                 out_dtype=torch.float32):
    """Evaluate several layers (same T, layout and token count) in one launch; layout-3 layers
    use workspace ``ws`` (by default the one kept for this device and stream) and may write
    bfloat16 outputs (``out_dtype``: the float32 result rounded once).  For a loop over the same
    buffers, ``GroupCall`` prepares the arguments once."""
    return GroupCall(qs, xs, ys, algo, stream, ws, out_dtype)()


def linear_group_static(qs, xs, ys=None, stream=None):
    """The table-lookup decode of layout-3 layers with the library's own fixed scratch (no
    workspace, nothing allocated on the device by the library): for callers that may not
    allocate device memory.  Calls that overlap on the GPU share that scratch and race."""
    count = len(qs)
    M = xs[0].shape[0]
    if ys is None:
        ys = [torch.empty((M, 2 * q.n), dtype=torch.float32, device=x.device) for q, x in zip(qs, xs)]
    for q, x, y in zip(qs, xs, ys):
        _dev(x, "x")
        _dev(y, "y")
        if x.dtype != torch.bfloat16 or x.shape != (M, 2 * q.m) or y.shape != (M, 2 * q.n):
            raise ValueError("group members need matching x [M, 2m] bfloat16 and y [M, 2n] float32")
    descs = (PackedDesc * count)(*[q.desc() for q in qs])
    xp = (ctypes.c_void_p * count)(*[x.data_ptr() for x in xs])
    yp = (ctypes.c_void_p * count)(*[y.data_ptr() for y in ys])
    _check(load_library().fairy2i_linear_group_static(descs, xp, yp, count, M, _stream(stream)))
    return ys


def unpack_codes(q: Packed, stream=None) -> torch.Tensor:  # either layout
    """Canonical codes uint8 [2, T, n, m] (0=+1, 1=-1, 2=+i, 3=-i) on the device."""
    out = torch.empty((2, q.T, q.n, q.m), dtype=torch.uint8, device=q.codes.device)
    d = q.desc()
    _check(load_library().fairy2i_unpack_codes(ctypes.byref(d), out.data_ptr(), _stream(stream)))
    return out


def selftest_bounded_wait(limit_us: int = 10000, stream=None):
    """Run the bounded-wait self-test; a following sync_status() raises TIMEOUT."""
    _check(load_library().fairy2i_selftest_bounded_wait(limit_us, _stream(stream)))


def sync_status(stream=None):
    """Synchronize the stream and raise if a kernel reported an error."""
    _check(load_library().fairy2i_sync_status(_stream(stream)))

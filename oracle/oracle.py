"""Reference oracle for the Fairy2i widely-linear layer -- TEST INFRASTRUCTURE.

Thin ctypes marshalling over ``fairy2i_oracle.c`` (plain C, double precision).
Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The product library never does, and it
shares no code with the CUDA path.

Array conventions (numpy, C order):
  R       float32 [2n, 2m]
  U, W    complex64 (float32 pairs) or complex128 [n, m]
  codes   uint8 [T, n, m]   canonical values 0=+1, 1=-1, 2=+i, 3=-i
  scales  float32 [T, 2, n] axis 0 = real, axis 1 = imaginary
  x       uint16 bfloat16 bit patterns [M, 2m] = [Re x | Im x]
  y       float64 [M, 2n]   = [Re y | Im y]
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fairy2i_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")

OK, BAD_ARG, NONFINITE = 0, 1, 2


class OracleError(RuntimeError):
    pass


class NonFiniteInput(OracleError):
    pass


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no contraction of a*b+c into fused ops)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
             "-shared", "-o", tmp, _SRC, "-lm"],
            check=True)
        os.replace(tmp, _LIB)
    return _LIB


_lib_handle = None


def _lib():
    global _lib_handle
    if _lib_handle is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I32 = ctypes.c_int32
        lib.oracle_convert_f64.argtypes = [P, I64, I64, P, P]
        lib.oracle_convert_f32.argtypes = [P, I64, I64, P, P]
        lib.oracle_quantize.argtypes = [P, I64, I64, I32, P, P, P, P, P, P]
        lib.oracle_dequantize.argtypes = [P, P, I64, I64, I32, P]
        lib.oracle_linear_mulfree.argtypes = [P, P, P, P, I64, I64, I32, P, I64, P]
        lib.oracle_linear_dense.argtypes = [P, P, I64, I64, P, I64, P]
        lib.oracle_linear_grad_x.argtypes = [P, P, P, P, I64, I64, I32, P, I64, P]
        for f in (lib.oracle_convert_f64, lib.oracle_convert_f32, lib.oracle_quantize,
                  lib.oracle_dequantize, lib.oracle_linear_mulfree, lib.oracle_linear_dense,
                  lib.oracle_linear_grad_x):
            f.restype = ctypes.c_int
        _lib_handle = lib
    return _lib_handle


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int):
    if rc == NONFINITE:
        raise NonFiniteInput("non-finite weight")
    if rc != OK:
        raise OracleError(f"oracle returned {rc}")


def _as_pairs(Z: np.ndarray, dtype) -> np.ndarray:
    """complex [n, m] -> contiguous real pairs [n, m, 2] of dtype."""
    Z = np.ascontiguousarray(Z)
    pairs = np.empty(Z.shape + (2,), dtype=dtype)
    pairs[..., 0] = Z.real
    pairs[..., 1] = Z.imag
    return pairs


def convert_f64(R: np.ndarray):
    """Theorem 1 block formulas in double.  Returns (U, W) complex128 [n, m]."""
    R = np.ascontiguousarray(R, dtype=np.float32)
    n, m = R.shape[0] // 2, R.shape[1] // 2
    U = np.empty((n, m, 2), np.float64)
    W = np.empty((n, m, 2), np.float64)
    _check(_lib().oracle_convert_f64(_ptr(R), n, m, _ptr(U), _ptr(W)))
    return U[..., 0] + 1j * U[..., 1], W[..., 0] + 1j * W[..., 1]


def convert_f32(R: np.ndarray):
    """Block formulas with float32 rounding per operation.  (U, W) complex64."""
    R = np.ascontiguousarray(R, dtype=np.float32)
    n, m = R.shape[0] // 2, R.shape[1] // 2
    U = np.empty((n, m, 2), np.float32)
    W = np.empty((n, m, 2), np.float32)
    _check(_lib().oracle_convert_f32(_ptr(R), n, m, _ptr(U), _ptr(W)))
    return U.view(np.complex64)[..., 0], W.view(np.complex64)[..., 0]


@dataclass
class Quantized:
    codes: np.ndarray      # uint8 [T, n, m]
    scales: np.ndarray     # float32 [T, 2, n]
    resid: np.ndarray | None   # complex64 [T+1, n, m]; resid[0] is the input
    mean64: np.ndarray | None  # float64 [T, 2, n] plain double means


def quantize(Z: np.ndarray, T: int, keep_residuals: bool = False) -> Quantized:
    """Phase-aware recursive residual quantization of one complex matrix."""
    Zp = _as_pairs(np.asarray(Z, dtype=np.complex64), np.float32)
    n, m = Zp.shape[0], Zp.shape[1]
    codes = np.empty((T, n, m), np.uint8)
    scales = np.empty((T, 2, n), np.float32)
    resid = np.empty((T + 1, n, m, 2), np.float32) if keep_residuals else None
    mean64 = np.empty((T, 2, n), np.float64) if keep_residuals else None
    work = np.empty((n, m, 2), np.float32)
    axis_buf = np.empty((m,), np.float32)
    _check(_lib().oracle_quantize(_ptr(Zp), n, m, T, _ptr(codes), _ptr(scales), _ptr(resid),
                                  _ptr(mean64), _ptr(work), _ptr(axis_buf)))
    rc = resid.view(np.complex64)[..., 0] if resid is not None else None
    return Quantized(codes, scales, rc, mean64)


def dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Sum of dequantized stages, complex128 [n, m]."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    T, n, m = codes.shape
    Z = np.empty((n, m, 2), np.float64)
    _check(_lib().oracle_dequantize(_ptr(codes), _ptr(scales), n, m, T, _ptr(Z)))
    return Z[..., 0] + 1j * Z[..., 1]


def _x_bits(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        raise TypeError("x must be bfloat16 bit patterns (uint16)")
    if x.ndim == 1:
        x = x[None, :]
    return x


def linear_mulfree(qU: Quantized, qW: Quantized, x: np.ndarray) -> np.ndarray:
    """y = U^ x + W^ conj(x) by adds/subtracts and one scale per stage/axis."""
    x = _x_bits(x)
    T, n, m = qU.codes.shape
    assert qW.codes.shape == (T, n, m) and x.shape[1] == 2 * m
    M = x.shape[0]
    y = np.empty((M, 2 * n), np.float64)
    cu = np.ascontiguousarray(qU.codes)
    cw = np.ascontiguousarray(qW.codes)
    su = np.ascontiguousarray(qU.scales, dtype=np.float32)
    sw = np.ascontiguousarray(qW.scales, dtype=np.float32)
    _check(_lib().oracle_linear_mulfree(_ptr(cu), _ptr(su), _ptr(cw), _ptr(sw),
                                        n, m, T, _ptr(x), M, _ptr(y)))
    return y


def linear_dense(Uhat: np.ndarray, What: np.ndarray, x: np.ndarray) -> np.ndarray:
    """y = U^ x + W^ conj(x) with complex products (U^, W^ complex [n, m])."""
    x = _x_bits(x)
    n, m = Uhat.shape
    Up = _as_pairs(np.asarray(Uhat, np.complex128), np.float64)
    Wp = _as_pairs(np.asarray(What, np.complex128), np.float64)
    M = x.shape[0]
    y = np.empty((M, 2 * n), np.float64)
    _check(_lib().oracle_linear_dense(_ptr(Up), _ptr(Wp), n, m, _ptr(x), M, _ptr(y)))
    return y


def linear_grad_x_mulfree(qU: Quantized, qW: Quantized, g: np.ndarray) -> np.ndarray:
    """dL/dx = U^^H g + W^^T conj(g) for g = [dRe y | dIm y] float32 [M, 2n], by one scale multiply
    per row, stage and axis and adds/subtracts over the codes; returns [dRe x | dIm x] [M, 2m]."""
    g = np.ascontiguousarray(g, dtype=np.float32)
    if g.ndim == 1:
        g = g[None, :]
    T, n, m = qU.codes.shape
    assert qW.codes.shape == (T, n, m) and g.shape[1] == 2 * n
    M = g.shape[0]
    gx = np.empty((M, 2 * m), np.float64)
    cu = np.ascontiguousarray(qU.codes)
    cw = np.ascontiguousarray(qW.codes)
    su = np.ascontiguousarray(qU.scales, dtype=np.float32)
    sw = np.ascontiguousarray(qW.scales, dtype=np.float32)
    _check(_lib().oracle_linear_grad_x(_ptr(cu), _ptr(su), _ptr(cw), _ptr(sw), n, m, T, _ptr(g), M, _ptr(gx)))
    return gx


def linear_grad_x_dense(Uhat: np.ndarray, What: np.ndarray, g: np.ndarray) -> np.ndarray:
    """The same gradient with complex matrix products of the dequantized U^, W^ (complex [n, m])."""
    g = np.asarray(g, np.float64)
    if g.ndim == 1:
        g = g[None, :]
    n, m = Uhat.shape
    gc = g[:, :n] + 1j * g[:, n:]
    gxc = gc @ np.conj(Uhat) + np.conj(gc) @ What  # row form of U^^H g + W^^T conj(g)
    return np.concatenate([gxc.real, gxc.imag], axis=1)


def bf16_bits_to_f64(x: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns (uint16) to float64."""
    x = np.asarray(x, dtype=np.uint16)
    return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)

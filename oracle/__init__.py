"""NVFP4 oracle: a plain, single-threaded CPU reference (C++, fp32 quantizer
steps and an fp64 matmul).

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import it.  It shares no code with the CUDA
library and never imports it.

Functions and what pins them (tests/test_oracle.py):

* ``e2m1_value`` / ``e4m3_value`` -- element decode from the type definitions
  (OCP MX v1.0 E2M1; OCP FP8 E4M3 "fn").  Pinned by the exhaustive 16-entry
  table and by all 256 bytes against torch.float8_e4m3fn.
* ``e4m3_encode`` / ``e2m1_encode`` -- round to nearest, ties to even,
  saturating.  Pinned by torch's fp8 cast and by brute-force argmin.
* ``quantize`` / ``quantize_rows`` / ``tensor_scale`` -- the NVFP4 recipe
  (tensor scale g/(6*448); block scale E4M3(block amax/6/s); codes
  E2M1(x/d)).  Pinned by hand-worked blocks (tests/golden/) and by the
  round-trip error bound.
* ``dequant`` and ``matmul_abt`` -- the plain definitions; pinned by exact
  rational brute force on tiny shapes and closed forms.
* ``reference_gemm`` -- Y = Xhat W^T with Xhat = X for M <= 16 and
  dequant(quantize(X)) for M > 16.
* ``e8m0_value`` / ``mx_quantize`` / ``mx_dequant`` -- MXFP4 (OCP MX v1.0:
  32-element blocks, E8M0 scale 2^(floor(log2 amax) - 2), E2M1 elements).
  Pinned by hand-worked blocks (tests/golden/mx_*.txt), by all 255 finite
  E8M0 bytes against torch.float8_e8m0fnu where torch has it and against
  powers of two, and by the definition's invariants (the scale is the
  largest power of two that keeps the block max below 8 times it; no code
  but the clipped ones errs by more than half an E2M1 step).
* ``silu`` / ``reference_swiglu`` -- the gate/up MLP activation
  h = silu(g) * u (silu(v) = v / (1 + e^-v)) on reference_gemm's g and u, in
  fp64, with the band derived in reference_swiglu.  silu pinned by
  scipy.special.expit; the band by its own properties (it admits the
  correctly rounded result under the worst g/u errors it allows and rejects
  a dropped block of g).
* ``fp8_tensor_scale`` / ``fp8_quantize_rows`` / ``fp8_quantize`` /
  ``fp8_dequant`` -- FP8 E4M3 weights with one fp32 scale g/448.  Pinned by
  hand-worked values (tests/golden/fp8_*.txt) and by torch's fp8 cast of
  x / s8 (the same correctly rounded division).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libnvfp4_oracle.so")
_lib = None

DECODE_M_MAX = 16


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (single-threaded, no FP contraction)."""
    src = os.path.join(_HERE, "nvfp4_oracle.cpp")
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared",
                               "-ffp-contract=off", "-fno-fast-math", src, "-o", tmp])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P, I64, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float
    lib.orc_e2m1_value.restype = ctypes.c_double
    lib.orc_e2m1_value.argtypes = [ctypes.c_uint8]
    lib.orc_e4m3_value.restype = ctypes.c_double
    lib.orc_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.orc_e4m3_encode.restype = ctypes.c_uint8
    lib.orc_e4m3_encode.argtypes = [F]
    lib.orc_e2m1_encode.restype = ctypes.c_uint8
    lib.orc_e2m1_encode.argtypes = [F]
    lib.orc_tensor_scale.restype = ctypes.c_int
    lib.orc_tensor_scale.argtypes = [P, I64, I64, I64, P, P]
    lib.orc_quantize_rows.restype = None
    lib.orc_quantize_rows.argtypes = [P, I64, I64, I64, F, P, P]
    lib.orc_quantize.restype = ctypes.c_int
    lib.orc_quantize.argtypes = [P, I64, I64, I64, P, P, P]
    lib.orc_dequant.restype = None
    lib.orc_dequant.argtypes = [P, P, F, I64, I64, P]
    lib.orc_bf16_to_f64.restype = None
    lib.orc_bf16_to_f64.argtypes = [P, I64, P]
    lib.orc_matmul_abt.restype = None
    lib.orc_matmul_abt.argtypes = [P, I64, P, I64, I64, P, P]
    lib.orc_e8m0_value.restype = ctypes.c_double
    lib.orc_e8m0_value.argtypes = [ctypes.c_uint8]
    lib.orc_mx_quantize.restype = ctypes.c_int
    lib.orc_mx_quantize.argtypes = [P, I64, I64, I64, P, P]
    lib.orc_mx_dequant.restype = None
    lib.orc_mx_dequant.argtypes = [P, P, I64, I64, P]
    lib.orc_fp8_tensor_scale.restype = ctypes.c_int
    lib.orc_fp8_tensor_scale.argtypes = [P, I64, I64, I64, P]
    lib.orc_fp8_quantize_rows.restype = None
    lib.orc_fp8_quantize_rows.argtypes = [P, I64, I64, I64, F, P]
    lib.orc_fp8_dequant.restype = None
    lib.orc_fp8_dequant.argtypes = [P, F, I64, P]
    _lib = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags.c_contiguous
    return a.ctypes.data


def e2m1_value(code: int) -> float:
    return _load().orc_e2m1_value(code)


def e4m3_value(byte: int) -> float:
    return _load().orc_e4m3_value(byte)


def e4m3_encode(u: float) -> int:
    return _load().orc_e4m3_encode(u)


def e2m1_encode(q: float) -> int:
    return _load().orc_e2m1_encode(q)


def tensor_scale(x_bf16: np.ndarray) -> tuple[float, float, bool]:
    """(global amax, tensor scale g/2688, nonfinite flag) of a [rows, K] uint16 array."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, K = x.shape
    g = np.zeros(1, np.float32)
    s = np.zeros(1, np.float32)
    bad = _load().orc_tensor_scale(_ptr(x), rows, K, K, _ptr(g), _ptr(s))
    return float(g[0]), float(s[0]), bool(bad)


def quantize_rows(x_bf16: np.ndarray, s: float) -> tuple[np.ndarray, np.ndarray]:
    """Quantize rows with a given tensor scale -> (codes [rows,K/2], scales [rows,K/16])."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, K = x.shape
    codes = np.empty((rows, K // 2), np.uint8)
    scales = np.empty((rows, K // 16), np.uint8)
    _load().orc_quantize_rows(_ptr(x), rows, K, K, np.float32(s), _ptr(codes), _ptr(scales))
    return codes, scales


def quantize(x_bf16: np.ndarray) -> tuple[np.ndarray, np.ndarray, float, bool]:
    """Whole tensor -> (codes, scales, tensor scale, nonfinite flag)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, K = x.shape
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    codes = np.empty((rows, K // 2), np.uint8)
    scales = np.empty((rows, K // 16), np.uint8)
    s = np.zeros(1, np.float32)
    bad = _load().orc_quantize(_ptr(x), rows, K, K, _ptr(codes), _ptr(scales), _ptr(s))
    return codes, scales, float(s[0]), bool(bad)


def dequant(codes: np.ndarray, scales: np.ndarray, s: float) -> np.ndarray:
    """fp64 [rows, K] values e2m1 * e4m3 * s."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    rows, K = codes.shape[0], codes.shape[1] * 2
    out = np.empty((rows, K), np.float64)
    _load().orc_dequant(_ptr(codes), _ptr(scales), np.float32(s), rows, K, _ptr(out))
    return out


def bf16_to_f64(x_bf16: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    out = np.empty(x.shape, np.float64)
    _load().orc_bf16_to_f64(_ptr(x), x.size, _ptr(out))
    return out


def matmul_abt(a: np.ndarray, b: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """(A B^T, |A| |B|^T) accumulated in fp64; a [M,K], b [N,K]."""
    a = np.ascontiguousarray(a, dtype=np.float64)
    b = np.ascontiguousarray(b, dtype=np.float64)
    M, K = a.shape
    N = b.shape[0]
    y = np.empty((M, N), np.float64)
    bound = np.empty((M, N), np.float64)
    _load().orc_matmul_abt(_ptr(a), M, _ptr(b), N, K, _ptr(y), _ptr(bound))
    return y, bound


def activation_hat(x_bf16: np.ndarray, M_total: int, s_x: float | None = None) -> np.ndarray:
    """The X operand the method multiplies: bf16 X itself for decode-sized M
    (<= 16), dequant(quantize(X)) for larger M.  For a row sample of a large
    X, pass the tensor scale of the whole X as s_x."""
    if M_total <= DECODE_M_MAX:
        return bf16_to_f64(x_bf16)
    if s_x is None:
        _, s_x, _ = tensor_scale(x_bf16)
    c, sc = quantize_rows(x_bf16, s_x)
    return dequant(c, sc, s_x)


def reference_gemm(x_bf16: np.ndarray, M_total: int, w_codes: np.ndarray,
                   w_scales: np.ndarray, s_w: float, s_x: float | None = None):
    """(y_ref, bound) for rows of X against rows of W, in fp64."""
    xh = activation_hat(x_bf16, M_total, s_x)
    wh = dequant(w_codes, w_scales, s_w)
    return matmul_abt(xh, wh)


BF16_UNIT_ROUNDOFF = 2.0 ** -8


def tolerance(bound: np.ndarray, y_ref: np.ndarray | None = None) -> np.ndarray:
    """Per-element acceptance band for a bf16 result:
    |y - y_ref| <= 2e-3 * sum|x w| + 1e-5 + 2^-8 * |y_ref|.

    The first two terms are the stated bound on the arithmetic.  The last is
    the rounding of the result to bf16 (8 significant bits, unit roundoff
    2^-8): the exactly rounded bf16 value of y_ref can itself differ from
    y_ref by up to 2^-8 |y_ref|, which exceeds 2e-3 * sum|x w| whenever
    |y_ref| > 0.512 * sum|x w| (short or one-signed sums)."""
    tol = 2e-3 * bound + 1e-5
    if y_ref is not None:
        tol = tol + BF16_UNIT_ROUNDOFF * np.abs(y_ref)
    return tol


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |v| (normal range)."""
    _, e = np.frexp(np.abs(np.asarray(v, dtype=np.float64)))
    return np.ldexp(1.0, e - 8)


def tight_tolerance(bound: np.ndarray, y_ref: np.ndarray) -> np.ndarray:
    """A stricter band for kernels whose products are exact and whose sums are
    fp32: one bf16 ulp of y_ref plus 2^-14 * sum|x w| (room for ~1000 fp32
    roundings).  A dropped or doubled block moves y by far more than this."""
    return bf16_ulp(y_ref) + 2.0 ** -14 * bound + 1e-30


# ---- MXFP4 -------------------------------------------------------------------

def e8m0_value(byte: int) -> float:
    return _load().orc_e8m0_value(byte)


def mx_quantize(x_bf16: np.ndarray) -> tuple[np.ndarray, np.ndarray, bool]:
    """[rows, K] uint16 -> (codes [rows, K/2], E8M0 scales [rows, K/32], nonfinite flag)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, K = x.shape
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    codes = np.empty((rows, K // 2), np.uint8)
    scales = np.empty((rows, K // 32), np.uint8)
    bad = _load().orc_mx_quantize(_ptr(x), rows, K, K, _ptr(codes), _ptr(scales))
    return codes, scales, bool(bad)


def mx_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """fp64 [rows, K] values e2m1 * 2^(scale - 127)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    rows, K = codes.shape[0], codes.shape[1] * 2
    out = np.empty((rows, K), np.float64)
    _load().orc_mx_dequant(_ptr(codes), _ptr(scales), rows, K, _ptr(out))
    return out


def mx_reference_gemm(x_bf16: np.ndarray, M_total: int, w_codes: np.ndarray,
                      w_scales: np.ndarray, s_x: float | None = None):
    """(y_ref, bound) for rows of X against rows of an MXFP4 weight, in fp64
    (X as in reference_gemm: bf16 for M <= 16, its NVFP4 quantization for
    larger M)."""
    return matmul_abt(activation_hat(x_bf16, M_total, s_x), mx_dequant(w_codes, w_scales))


# ---- FP8 E4M3 weights ----------------------------------------------------------

def fp8_tensor_scale(x_bf16: np.ndarray) -> tuple[float, bool]:
    """(s8 = global amax / 448, nonfinite flag)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, K = x.shape
    s = np.zeros(1, np.float32)
    bad = _load().orc_fp8_tensor_scale(_ptr(x), rows, K, K, _ptr(s))
    return float(s[0]), bool(bad)


def fp8_quantize_rows(x_bf16: np.ndarray, s8: float) -> np.ndarray:
    """E4M3 codes [rows, K] of x / s8."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    rows, K = x.shape
    codes = np.empty((rows, K), np.uint8)
    _load().orc_fp8_quantize_rows(_ptr(x), rows, K, K, np.float32(s8), _ptr(codes))
    return codes


def fp8_quantize(x_bf16: np.ndarray) -> tuple[np.ndarray, float, bool]:
    """Whole tensor -> (codes [rows, K], s8, nonfinite flag)."""
    s8, bad = fp8_tensor_scale(x_bf16)
    return fp8_quantize_rows(x_bf16, s8), s8, bad


def fp8_dequant(codes: np.ndarray, s8: float) -> np.ndarray:
    """fp64 values e4m3(code) * s8, same shape as codes."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().orc_fp8_dequant(_ptr(c), np.float32(s8), c.size, _ptr(out))
    return out


def fp8_reference_gemm(x_bf16: np.ndarray, w_codes: np.ndarray, s8: float):
    """(y_ref, bound) for a decode-sized X against an FP8 weight, in fp64."""
    return matmul_abt(bf16_to_f64(x_bf16), fp8_dequant(w_codes, s8))


# ---- gate/up MLP activation (SwiGLU) ------------------------------------------------

SILU_SLOPE_MAX = 1.1  # max |d silu / dv| = 1.0998 (at v = 2.3994)


def silu(v: np.ndarray) -> np.ndarray:
    """silu(v) = v / (1 + e^-v), fp64 (exp overflow for v < -709 gives -0)."""
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def reference_swiglu(x_bf16: np.ndarray, M_total: int, gate, up, s_x: float | None = None):
    """(h_ref, tol) for h = silu(g) * u with g = X Wg^T and u = X Wu^T as
    reference_gemm forms them (gate and up: (codes, scales, tensor scale)).

    The band: g and u reach the epilogue in fp32 from exact products summed
    in fp32, so |dg| <= t_g = 2^-14 sum|x w_g| + 2^-22 |g| (the tight band of
    the GEMM without its bf16 term, plus the rounding of the scale factor);
    likewise t_u.  Then |silu(g') u' - silu(g) u| <= 1.1 t_g (|u| + t_u) +
    |silu(g)| t_u, the fp32 evaluation of silu and the product adds at most
    2^-20 of |silu(g')| |u'|, and the result is rounded to bf16 (2^-8 of
    itself)."""
    g, bg = reference_gemm(x_bf16, M_total, *gate, s_x=s_x)
    u, bu = reference_gemm(x_bf16, M_total, *up, s_x=s_x)
    tg = 2.0 ** -14 * bg + 2.0 ** -22 * np.abs(g)
    tu = 2.0 ** -14 * bu + 2.0 ** -22 * np.abs(u)
    sg = np.abs(silu(g))
    a = SILU_SLOPE_MAX * tg * (np.abs(u) + tu) + sg * tu
    a = a + 2.0 ** -20 * (sg + SILU_SLOPE_MAX * tg) * (np.abs(u) + tu)
    h = silu(g) * u
    tol = a + BF16_UNIT_ROUNDOFF * (np.abs(h) + a) + 1e-30
    return h, tol

"""Python binding of libimp_nvfp4 (include/imp_nvfp4.h).

Argument marshalling only: every step of the quantizer and the linear layer
runs in the library's CUDA kernels.  The C entry points are exposed under
their own names (``imp_nvfp4_quantize``, ``imp_nvfp4_gemm``, ...) and take raw
integers (device addresses, sizes, a cudaStream_t handle).  ``quantize`` and
``gemm`` wrap them for torch CUDA tensors: they allocate outputs and the
workspace with torch and pass the current stream.

The shared library is loaded on first use (or by ``load()``); if it has not
been built (``python -m nvfp4_weight_quantized_02_gb300.build``) that raises
ImportError: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
from dataclasses import dataclass

from .build import INCLUDE, LIB

__all__ = [
    "IMP_OK", "IMP_DEV_OK", "IMP_DEV_NONFINITE_INPUT", "IMP_DEV_TIMEOUT", "ImpNvfp4Tensor",
    "imp_nvfp4_quantize", "imp_nvfp4_gemm", "imp_nvfp4_quantize_workspace_size",
    "imp_nvfp4_gemm_workspace_size", "imp_nvfp4_gemm_plan", "imp_status_string", "NVFP4Tensor",
    "quantize", "gemm",
    "library_path", "header_functions", "ImpError", "load", "imp_nvfp4_mma_scales_size",
    "imp_nvfp4_prepare_mma", "imp_nvfp4_quantize_mma", "imp_nvfp4_gemm_fp4", "prepare_mma",
    "imp_nvfp4_gemm_fp4_workspace_size",
    "imp_nvfp4_quantize_noalloc", "imp_nvfp4_mma_codes_size", "imp_nvfp4_gemm_mma",
    "quantize_mma", "gemm_fp4", "gemm_mma", "imp_selftest_bounded_wait",
    "ImpNvfp4Group", "IMP_NVFP4_MAX_GROUPS", "imp_nvfp4_gemm_grouped",
    "imp_nvfp4_gemm_grouped_workspace_size", "imp_nvfp4_gemm_grouped_plan", "gemm_grouped",
    "IMP_DEV_RANGE", "ImpMxfp4Tensor", "ImpFp8Tensor", "imp_mxfp4_quantize",
    "imp_mxfp4_to_nvfp4", "imp_mxfp4_to_nvfp4_workspace_size", "imp_fp8_quantize",
    "imp_fp8_quantize_workspace_size", "imp_fp8_gemm", "imp_fp8_gemm_workspace_size",
    "imp_fp8_gemm_plan", "MXFP4Tensor", "FP8Tensor", "mxfp4_quantize", "mxfp4_to_nvfp4",
    "fp8_quantize", "gemm_fp8", "imp_nvfp4_gemm_swiglu", "imp_nvfp4_gemm_swiglu_workspace_size",
    "imp_nvfp4_quantize_mma_amax", "gemm_swiglu", "quantize_mma_amax",
]

IMP_OK = 0
IMP_ERR_INVALID_ARG = 1
IMP_ERR_UNSUPPORTED_SHAPE = 2
IMP_ERR_MISALIGNED = 3
IMP_ERR_WORKSPACE_TOO_SMALL = 4
IMP_ERR_CUDA = 5
IMP_DEV_OK = 0
IMP_DEV_NONFINITE_INPUT = 1
IMP_DEV_TIMEOUT = 2
IMP_DEV_RANGE = 4
DECODE_M_MAX = 16
IMP_NVFP4_MAX_GROUPS = 4

class ImpNvfp4Tensor(ctypes.Structure):
    """ctypes mirror of imp_nvfp4_tensor."""
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("tensor_scale", ctypes.c_void_p), ("rows", ctypes.c_int64), ("K", ctypes.c_int64)]


class ImpNvfp4Group(ctypes.Structure):
    """ctypes mirror of imp_nvfp4_group."""
    _fields_ = [("w", ImpNvfp4Tensor), ("y_bf16", ctypes.c_void_p), ("ldy", ctypes.c_int64)]


class ImpNvfp4ChainLink(ctypes.Structure):
    """ctypes mirror of imp_nvfp4_chain_link."""
    _fields_ = [("groups", ctypes.POINTER(ImpNvfp4Group)), ("n_groups", ctypes.c_int32),
                ("x_bf16", ctypes.c_void_p), ("ldx", ctypes.c_int64), ("x_swiglu", ctypes.c_int32)]


class ImpMxfp4Tensor(ctypes.Structure):
    """ctypes mirror of imp_mxfp4_tensor."""
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("rows", ctypes.c_int64),
                ("K", ctypes.c_int64)]


class ImpFp8Tensor(ctypes.Structure):
    """ctypes mirror of imp_fp8_tensor."""
    _fields_ = [("codes", ctypes.c_void_p), ("tensor_scale", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("K", ctypes.c_int64)]


_lib = None


def _L():
    """The loaded library.  Raises ImportError if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB):
        raise ImportError(f"libimp_nvfp4.so is not built ({LIB}); run "
                          "python -m nvfp4_weight_quantized_02_gb300.build")
    lib = ctypes.CDLL(LIB)
    P, I64, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    lib.imp_nvfp4_quantize_workspace_size.restype = SZ
    lib.imp_nvfp4_quantize_workspace_size.argtypes = [I64, I64]
    lib.imp_nvfp4_quantize.restype = ctypes.c_int
    lib.imp_nvfp4_quantize.argtypes = [P, I64, I64, I64, ctypes.POINTER(ImpNvfp4Tensor), P, P, SZ, P]
    lib.imp_nvfp4_gemm_workspace_size.restype = SZ
    lib.imp_nvfp4_gemm_workspace_size.argtypes = [I64, I64, I64]
    lib.imp_nvfp4_gemm_plan.restype = ctypes.c_int32
    lib.imp_nvfp4_gemm_plan.argtypes = [I64, I64, I64, ctypes.POINTER(ctypes.c_char_p)]
    lib.imp_nvfp4_gemm.restype = ctypes.c_int
    lib.imp_nvfp4_gemm.argtypes = [P, I64, I64, I64, ctypes.POINTER(ImpNvfp4Tensor), P, I64, P, P,
                                   SZ, P]
    lib.imp_status_string.restype = ctypes.c_char_p
    lib.imp_selftest_bounded_wait.restype = ctypes.c_int
    lib.imp_selftest_bounded_wait.argtypes = [P, P]
    lib.imp_status_string.argtypes = [ctypes.c_int]
    T = ctypes.POINTER(ImpNvfp4Tensor)
    lib.imp_nvfp4_mma_scales_size.restype = SZ
    lib.imp_nvfp4_mma_scales_size.argtypes = [I64, I64]
    lib.imp_nvfp4_mma_codes_size.restype = SZ
    lib.imp_nvfp4_mma_codes_size.argtypes = [I64, I64]
    lib.imp_nvfp4_prepare_mma.restype = ctypes.c_int
    lib.imp_nvfp4_prepare_mma.argtypes = [T, P, SZ, P, SZ, P]
    lib.imp_nvfp4_gemm_mma.restype = ctypes.c_int
    lib.imp_nvfp4_gemm_mma.argtypes = [P, I64, I64, I64, T, P, I64, P, P, SZ, P]
    lib.imp_nvfp4_gemm_mma_swiglu.restype = ctypes.c_int
    lib.imp_nvfp4_gemm_mma_swiglu.argtypes = [P, P, I64, I64, I64, T, P, I64, P, P, SZ, P]
    lib.imp_nvfp4_gemm_mma_swiglu_plan.restype = ctypes.c_int32
    lib.imp_nvfp4_gemm_mma_swiglu_plan.argtypes = [I64, I64, I64, ctypes.POINTER(ctypes.c_char_p)]
    lib.imp_nvfp4_quantize_mma.restype = ctypes.c_int
    lib.imp_nvfp4_quantize_mma.argtypes = [P, I64, I64, I64, T, P, P, SZ, P]
    lib.imp_nvfp4_quantize_noalloc.restype = ctypes.c_int
    lib.imp_nvfp4_quantize_noalloc.argtypes = [P, I64, I64, I64, T, P, P]
    lib.imp_nvfp4_gemm_fp4.restype = ctypes.c_int
    lib.imp_nvfp4_gemm_fp4.argtypes = [T, T, P, I64, P, P, SZ, P]
    lib.imp_nvfp4_gemm_fp4_workspace_size.restype = SZ
    lib.imp_nvfp4_gemm_fp4_workspace_size.argtypes = [I64, I64, I64]
    PI64 = ctypes.POINTER(I64)
    lib.imp_nvfp4_gemm_grouped_workspace_size.restype = SZ
    lib.imp_nvfp4_gemm_grouped_workspace_size.argtypes = [I64, I64, PI64, ctypes.c_int32]
    lib.imp_nvfp4_gemm_grouped_plan.restype = ctypes.c_int32
    lib.imp_nvfp4_gemm_grouped_plan.argtypes = [I64, I64, PI64, ctypes.c_int32,
                                                ctypes.POINTER(ctypes.c_char_p)]
    lib.imp_nvfp4_gemm_grouped.restype = ctypes.c_int
    lib.imp_nvfp4_gemm_grouped.argtypes = [P, I64, I64, I64, ctypes.POINTER(ImpNvfp4Group),
                                           ctypes.c_int32, P, P, SZ, P]
    CL = ctypes.POINTER(ImpNvfp4ChainLink)
    lib.imp_nvfp4_gemm_chain_workspace_size.restype = SZ
    lib.imp_nvfp4_gemm_chain_workspace_size.argtypes = [I64, CL, ctypes.c_int32]
    lib.imp_nvfp4_gemm_chain_plan.restype = ctypes.c_int32
    lib.imp_nvfp4_gemm_chain_plan.argtypes = [I64, CL, ctypes.c_int32]
    lib.imp_nvfp4_gemm_chain.restype = ctypes.c_int
    lib.imp_nvfp4_gemm_chain.argtypes = [I64, CL, ctypes.c_int32, P, P, SZ, P]
    MX, F8 = ctypes.POINTER(ImpMxfp4Tensor), ctypes.POINTER(ImpFp8Tensor)
    lib.imp_mxfp4_quantize.restype = ctypes.c_int
    lib.imp_mxfp4_quantize.argtypes = [P, I64, I64, I64, MX, P, P]
    lib.imp_mxfp4_to_nvfp4_workspace_size.restype = SZ
    lib.imp_mxfp4_to_nvfp4_workspace_size.argtypes = []
    lib.imp_mxfp4_to_nvfp4.restype = ctypes.c_int
    lib.imp_mxfp4_to_nvfp4.argtypes = [MX, ctypes.POINTER(ImpNvfp4Tensor), P, P, SZ, P]
    lib.imp_fp8_quantize_workspace_size.restype = SZ
    lib.imp_fp8_quantize_workspace_size.argtypes = [I64, I64]
    lib.imp_fp8_quantize.restype = ctypes.c_int
    lib.imp_fp8_quantize.argtypes = [P, I64, I64, I64, F8, P, P, SZ, P]
    lib.imp_fp8_gemm_workspace_size.restype = SZ
    lib.imp_fp8_gemm_workspace_size.argtypes = [I64, I64, I64]
    lib.imp_fp8_gemm_plan.restype = ctypes.c_int32
    lib.imp_fp8_gemm_plan.argtypes = [I64, I64, I64, ctypes.POINTER(ctypes.c_char_p)]
    lib.imp_fp8_gemm.restype = ctypes.c_int
    lib.imp_fp8_gemm.argtypes = [P, I64, I64, I64, F8, P, I64, P, P, SZ, P]
    lib.imp_nvfp4_gemm_swiglu_workspace_size.restype = SZ
    lib.imp_nvfp4_gemm_swiglu_workspace_size.argtypes = [I64, I64, I64]
    lib.imp_nvfp4_gemm_swiglu.restype = ctypes.c_int
    lib.imp_nvfp4_gemm_swiglu.argtypes = [P, I64, I64, I64, T, T, P, I64, P, P, P, SZ, P]
    lib.imp_nvfp4_quantize_mma_amax.restype = ctypes.c_int
    lib.imp_nvfp4_quantize_mma_amax.argtypes = [P, I64, I64, I64, P, T, P, P]
    _lib = lib
    return lib


def load() -> ctypes.CDLL:
    """Load the library now (ImportError if it is missing)."""
    return _L()


def library_path() -> str:
    return LIB


def header_functions() -> list[str]:
    """Names of the functions declared in include/imp_nvfp4.h."""
    text = open(os.path.join(INCLUDE, "imp_nvfp4.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(imp_\w+)\s*\(", text)))


def imp_status_string(status: int) -> str:
    return _L().imp_status_string(status).decode()


def imp_nvfp4_quantize_workspace_size(rows: int, K: int) -> int:
    return _L().imp_nvfp4_quantize_workspace_size(rows, K)


def imp_nvfp4_gemm_workspace_size(M: int, N: int, K: int) -> int:
    return _L().imp_nvfp4_gemm_workspace_size(M, N, K)


def imp_selftest_bounded_wait(dev_status: int, stream: int | None) -> int:
    return _L().imp_selftest_bounded_wait(dev_status, stream)


def imp_nvfp4_gemm_plan(M: int, N: int, K: int) -> tuple[int, str | None]:
    """(kernel launches of one imp_nvfp4_gemm call, name of the kernel that
    streams W) on the current device; (0, None) for rejected shapes."""
    name = ctypes.c_char_p()
    n = _L().imp_nvfp4_gemm_plan(M, N, K, ctypes.byref(name))
    return n, (name.value.decode() if name.value else None)


def imp_nvfp4_quantize(x_bf16: int, rows: int, K: int, ldx: int, out: ImpNvfp4Tensor,
                       dev_status: int | None, workspace: int | None, ws_bytes: int,
                       stream: int | None) -> int:
    return _L().imp_nvfp4_quantize(x_bf16, rows, K, ldx, ctypes.byref(out), dev_status, workspace,
                                   ws_bytes, stream)


def imp_nvfp4_gemm(x_bf16: int, M: int, K: int, ldx: int, w: ImpNvfp4Tensor, y_bf16: int,
                   ldy: int, dev_status: int | None, workspace: int | None, ws_bytes: int,
                   stream: int | None) -> int:
    return _L().imp_nvfp4_gemm(x_bf16, M, K, ldx, ctypes.byref(w), y_bf16, ldy, dev_status,
                               workspace, ws_bytes, stream)


def imp_nvfp4_mma_scales_size(rows: int, K: int) -> int:
    return _L().imp_nvfp4_mma_scales_size(rows, K)


def imp_nvfp4_mma_codes_size(rows: int, K: int) -> int:
    return _L().imp_nvfp4_mma_codes_size(rows, K)


def imp_nvfp4_prepare_mma(t: ImpNvfp4Tensor, mma_codes: int | None, codes_bytes: int,
                          mma_scales: int | None, scales_bytes: int, stream: int | None) -> int:
    return _L().imp_nvfp4_prepare_mma(ctypes.byref(t), mma_codes, codes_bytes, mma_scales,
                                      scales_bytes, stream)


def imp_nvfp4_gemm_mma(x_bf16: int, M: int, K: int, ldx: int, w: ImpNvfp4Tensor, y_bf16: int,
                       ldy: int, dev_status: int | None, workspace: int | None, ws_bytes: int,
                       stream: int | None) -> int:
    return _L().imp_nvfp4_gemm_mma(x_bf16, M, K, ldx, ctypes.byref(w), y_bf16, ldy, dev_status,
                                   workspace, ws_bytes, stream)


def imp_nvfp4_gemm_mma_swiglu(gate_bf16: int, up_bf16: int, M: int, K: int, ld: int,
                              w: ImpNvfp4Tensor, y_bf16: int, ldy: int, dev_status: int | None,
                              workspace: int | None, ws_bytes: int, stream: int | None) -> int:
    return _L().imp_nvfp4_gemm_mma_swiglu(gate_bf16, up_bf16, M, K, ld, ctypes.byref(w), y_bf16,
                                          ldy, dev_status, workspace, ws_bytes, stream)


def imp_nvfp4_gemm_mma_swiglu_plan(M: int, N: int, K: int) -> tuple[int, str | None]:
    name = ctypes.c_char_p()
    n = _L().imp_nvfp4_gemm_mma_swiglu_plan(M, N, K, ctypes.byref(name))
    return n, (name.value.decode() if name.value else None)


def imp_nvfp4_quantize_mma(x_bf16: int, rows: int, K: int, ldx: int, out: ImpNvfp4Tensor,
                           dev_status: int | None, workspace: int | None, ws_bytes: int,
                           stream: int | None) -> int:
    return _L().imp_nvfp4_quantize_mma(x_bf16, rows, K, ldx, ctypes.byref(out), dev_status,
                                       workspace, ws_bytes, stream)


def imp_nvfp4_quantize_noalloc(x_bf16: int, rows: int, K: int, ldx: int, out: ImpNvfp4Tensor,
                               dev_status: int | None, stream: int | None) -> int:
    """The quantizer without caller workspace (its scratch is a fixed array
    inside the library); for callers that cannot allocate at call time."""
    return _L().imp_nvfp4_quantize_noalloc(x_bf16, rows, K, ldx, ctypes.byref(out), dev_status,
                                           stream)


def imp_nvfp4_gemm_fp4_workspace_size(M: int, N: int, K: int) -> int:
    return _L().imp_nvfp4_gemm_fp4_workspace_size(M, N, K)


def imp_nvfp4_gemm_fp4(xq: ImpNvfp4Tensor, wq: ImpNvfp4Tensor, y_bf16: int, ldy: int,
                       dev_status: int | None, workspace: int | None, ws_bytes: int,
                       stream: int | None) -> int:
    return _L().imp_nvfp4_gemm_fp4(ctypes.byref(xq), ctypes.byref(wq), y_bf16, ldy, dev_status,
                                   workspace, ws_bytes, stream)


def _i64s(N) -> "ctypes.Array":
    return (ctypes.c_int64 * len(N))(*N)


def imp_nvfp4_gemm_grouped_workspace_size(M: int, K: int, N: list[int]) -> int:
    return _L().imp_nvfp4_gemm_grouped_workspace_size(M, K, _i64s(N), len(N))


def imp_nvfp4_gemm_grouped_plan(M: int, K: int, N: list[int]) -> tuple[int, str | None]:
    """(kernel launches of one imp_nvfp4_gemm_grouped call, name of the first
    weight-streaming kernel); (0, None) if rejected."""
    name = ctypes.c_char_p()
    n = _L().imp_nvfp4_gemm_grouped_plan(M, K, _i64s(N), len(N), ctypes.byref(name))
    return n, (name.value.decode() if name.value else None)


def imp_nvfp4_gemm_grouped(x_bf16: int, M: int, K: int, ldx: int, groups: list[ImpNvfp4Group],
                           dev_status: int | None, workspace: int | None, ws_bytes: int,
                           stream: int | None) -> int:
    arr = (ImpNvfp4Group * len(groups))(*groups)
    return _L().imp_nvfp4_gemm_grouped(x_bf16, M, K, ldx, arr, len(groups), dev_status,
                                       workspace, ws_bytes, stream)


class ChainLinks:
    """A host array of imp_nvfp4_chain_link built from (groups, x_bf16, ldx
    [, x_swiglu]) tuples (x_bf16 None: the previous link's first output, or
    with x_swiglu the activation of its first two); keeps the groups' arrays
    alive for as long as it lives."""

    def __init__(self, links: list):
        links = [tuple(l) + (0,) * (4 - len(l)) for l in links]
        self._groups = [(ImpNvfp4Group * len(l[0]))(*l[0]) for l in links]
        self.array = (ImpNvfp4ChainLink * len(links))(*[
            ImpNvfp4ChainLink(ctypes.cast(ga, ctypes.POINTER(ImpNvfp4Group)), len(g), x, ldx, sw)
            for ga, (g, x, ldx, sw) in zip(self._groups, links)])
        self.n = len(links)


def imp_nvfp4_gemm_chain_workspace_size(M: int, links: ChainLinks) -> int:
    return _L().imp_nvfp4_gemm_chain_workspace_size(M, links.array, links.n)


def imp_nvfp4_gemm_chain_plan(M: int, links: ChainLinks) -> int:
    """1: one persistent launch; 0: one grouped call per link (or rejected)."""
    return _L().imp_nvfp4_gemm_chain_plan(M, links.array, links.n)


def imp_nvfp4_gemm_chain(M: int, links: ChainLinks, dev_status: int | None, workspace: int | None,
                         ws_bytes: int, stream: int | None) -> int:
    return _L().imp_nvfp4_gemm_chain(M, links.array, links.n, dev_status, workspace, ws_bytes,
                                      stream)


def imp_mxfp4_quantize(x_bf16: int, rows: int, K: int, ldx: int, out: ImpMxfp4Tensor,
                       dev_status: int | None, stream: int | None) -> int:
    return _L().imp_mxfp4_quantize(x_bf16, rows, K, ldx, ctypes.byref(out), dev_status, stream)


def imp_mxfp4_to_nvfp4_workspace_size() -> int:
    return _L().imp_mxfp4_to_nvfp4_workspace_size()


def imp_mxfp4_to_nvfp4(t: ImpMxfp4Tensor, out: ImpNvfp4Tensor, dev_status: int | None,
                       workspace: int | None, ws_bytes: int, stream: int | None) -> int:
    return _L().imp_mxfp4_to_nvfp4(ctypes.byref(t), ctypes.byref(out), dev_status, workspace,
                                   ws_bytes, stream)


def imp_fp8_quantize_workspace_size(rows: int, K: int) -> int:
    return _L().imp_fp8_quantize_workspace_size(rows, K)


def imp_fp8_quantize(x_bf16: int, rows: int, K: int, ldx: int, out: ImpFp8Tensor,
                     dev_status: int | None, workspace: int | None, ws_bytes: int,
                     stream: int | None) -> int:
    return _L().imp_fp8_quantize(x_bf16, rows, K, ldx, ctypes.byref(out), dev_status, workspace,
                                 ws_bytes, stream)


def imp_fp8_gemm_workspace_size(M: int, N: int, K: int) -> int:
    return _L().imp_fp8_gemm_workspace_size(M, N, K)


def imp_fp8_gemm_plan(M: int, N: int, K: int) -> tuple[int, str | None]:
    name = ctypes.c_char_p()
    n = _L().imp_fp8_gemm_plan(M, N, K, ctypes.byref(name))
    return n, (name.value.decode() if name.value else None)


def imp_fp8_gemm(x_bf16: int, M: int, K: int, ldx: int, w: ImpFp8Tensor, y_bf16: int, ldy: int,
                 dev_status: int | None, workspace: int | None, ws_bytes: int,
                 stream: int | None) -> int:
    return _L().imp_fp8_gemm(x_bf16, M, K, ldx, ctypes.byref(w), y_bf16, ldy, dev_status,
                             workspace, ws_bytes, stream)


def imp_nvfp4_gemm_swiglu_workspace_size(M: int, N: int, K: int) -> int:
    return _L().imp_nvfp4_gemm_swiglu_workspace_size(M, N, K)


def imp_nvfp4_gemm_swiglu(x_bf16: int, M: int, K: int, ldx: int, w_gate: ImpNvfp4Tensor,
                          w_up: ImpNvfp4Tensor, h_bf16: int, ldh: int, h_amax: int,
                          dev_status: int | None, workspace: int | None, ws_bytes: int,
                          stream: int | None) -> int:
    return _L().imp_nvfp4_gemm_swiglu(x_bf16, M, K, ldx, ctypes.byref(w_gate), ctypes.byref(w_up),
                                      h_bf16, ldh, h_amax, dev_status, workspace, ws_bytes, stream)


def imp_nvfp4_quantize_mma_amax(x_bf16: int, rows: int, K: int, ldx: int, amax: int,
                                out: ImpNvfp4Tensor, dev_status: int | None,
                                stream: int | None) -> int:
    return _L().imp_nvfp4_quantize_mma_amax(x_bf16, rows, K, ldx, amax, ctypes.byref(out),
                                            dev_status, stream)


class ImpError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {imp_status_string(status)}")
        self.status = status


# ---- torch convenience layer (allocation + marshalling) ----------------------

@dataclass
class NVFP4Tensor:
    """Device NVFP4 tensor: codes uint8[rows][K/2], scales uint8[rows][K/16],
    tensor_scale float32[1] -- or, with layout "mma" (prepare_mma), codes and
    scales as flat arrays in the tensor-core layout, shape=(rows, K)."""
    codes: "object"
    scales: "object"
    tensor_scale: "object"
    shape: "tuple | None" = None
    layout: str = "rows"

    @property
    def rows(self) -> int:
        return self.shape[0] if self.shape else self.codes.shape[0]

    @property
    def K(self) -> int:
        return self.shape[1] if self.shape else self.codes.shape[1] * 2

    def c_struct(self) -> ImpNvfp4Tensor:
        return ImpNvfp4Tensor(self.codes.data_ptr(), self.scales.data_ptr(),
                              self.tensor_scale.data_ptr(), self.rows, self.K)

    @staticmethod
    def empty(rows: int, K: int, device="cuda"):
        import torch
        return NVFP4Tensor(torch.empty((rows, K // 2), dtype=torch.uint8, device=device),
                           torch.empty((rows, K // 16), dtype=torch.uint8, device=device),
                           torch.empty(1, dtype=torch.float32, device=device))


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def quantize(x, out: NVFP4Tensor | None = None, dev_status=None, stream=None) -> NVFP4Tensor:
    """Quantize a 2-D bf16 CUDA tensor (row stride may exceed K) to NVFP4."""
    import torch
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, K = x.shape
    if out is None:
        out = NVFP4Tensor.empty(rows, K, device=x.device)
    ws_bytes = imp_nvfp4_quantize_workspace_size(rows, K)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=x.device)
    st = imp_nvfp4_quantize(x.data_ptr(), rows, K, x.stride(0), out.c_struct(),
                            None if dev_status is None else dev_status.data_ptr(), ws.data_ptr(),
                            ws_bytes, _stream_handle(stream))
    if st != IMP_OK:
        raise ImpError(st, "imp_nvfp4_quantize")
    return out


def gemm(x, w: NVFP4Tensor, y=None, dev_status=None, stream=None, workspace=None):
    """Y = X W^T for a 2-D bf16 CUDA tensor X and an NVFP4 weight."""
    import torch
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    N = w.rows
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    ws_bytes = imp_nvfp4_gemm_workspace_size(M, N, K)
    if workspace is None and ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=x.device)
    st = imp_nvfp4_gemm(x.data_ptr(), M, K, x.stride(0), w.c_struct(), y.data_ptr(), y.stride(0),
                        None if dev_status is None else dev_status.data_ptr(),
                        None if workspace is None else workspace.data_ptr(), ws_bytes,
                        _stream_handle(stream))
    if st != IMP_OK:
        raise ImpError(st, "imp_nvfp4_gemm")
    return y


def prepare_mma(w: NVFP4Tensor, stream=None) -> NVFP4Tensor:
    """The same weight in the tensor-core (MMA) layout: code tiles and scale
    atoms (flat uint8 arrays); the tensor scale is shared with `w`."""
    import torch
    assert w.layout == "rows"
    cb = imp_nvfp4_mma_codes_size(w.rows, w.K)
    sb = imp_nvfp4_mma_scales_size(w.rows, w.K)
    codes = torch.empty(cb, dtype=torch.uint8, device=w.codes.device)
    sc = torch.empty(sb, dtype=torch.uint8, device=w.codes.device)
    st = imp_nvfp4_prepare_mma(w.c_struct(), codes.data_ptr(), cb, sc.data_ptr(), sb,
                               _stream_handle(stream))
    if st != IMP_OK:
        raise ImpError(st, "imp_nvfp4_prepare_mma")
    return NVFP4Tensor(codes, sc, w.tensor_scale, shape=(w.rows, w.K), layout="mma")


def _struct(t: NVFP4Tensor) -> ImpNvfp4Tensor:
    return ImpNvfp4Tensor(t.codes.data_ptr(), t.scales.data_ptr(), t.tensor_scale.data_ptr(),
                          t.rows, t.K)


def quantize_mma(x, dev_status=None, stream=None) -> NVFP4Tensor:
    """Quantize a bf16 CUDA matrix with its scales in the tensor-core atom layout."""
    import torch
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, K = x.shape
    out = NVFP4Tensor(torch.empty((rows, K // 2), dtype=torch.uint8, device=x.device),
                      torch.empty(imp_nvfp4_mma_scales_size(rows, K), dtype=torch.uint8,
                                  device=x.device),
                      torch.empty(1, dtype=torch.float32, device=x.device))
    ws_bytes = imp_nvfp4_quantize_workspace_size(rows, K)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=x.device)
    st = imp_nvfp4_quantize_mma(x.data_ptr(), rows, K, x.stride(0), _struct(out),
                                None if dev_status is None else dev_status.data_ptr(),
                                ws.data_ptr(), ws_bytes, _stream_handle(stream))
    if st != IMP_OK:
        raise ImpError(st, "imp_nvfp4_quantize_mma")
    return out


def gemm_fp4(xq: NVFP4Tensor, wq: NVFP4Tensor, y=None, dev_status=None, stream=None,
             workspace=None, stream_k=False):
    """Y = Xq Wq^T on the block-scaled FP4 tensor cores (atom-layout scales).
    Whole 128 x 256 tiles per CTA; stream_k=True splits the (tile, K step)
    work evenly over the SMs instead (allocates the workspace if none is
    passed)."""
    import torch
    assert wq.layout == "mma"
    M, N = xq.rows, wq.rows
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=xq.codes.device)
    ws_bytes = imp_nvfp4_gemm_fp4_workspace_size(M, N, xq.K) if stream_k else 0
    if stream_k and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=xq.codes.device)
    st = imp_nvfp4_gemm_fp4(_struct(xq), _struct(wq), y.data_ptr(), y.stride(0),
                            None if dev_status is None else dev_status.data_ptr(),
                            workspace.data_ptr() if stream_k else None, ws_bytes,
                            _stream_handle(stream))
    if st != IMP_OK:
        raise ImpError(st, "imp_nvfp4_gemm_fp4")
    return y


def gemm_mma(x, w: NVFP4Tensor, y=None, dev_status=None, stream=None, workspace=None):
    """Y = X W^T for a bf16 CUDA matrix X and a weight in MMA layout
    (prepare_mma): the serving path."""
    import torch
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    assert w.layout == "mma"
    M, K = x.shape
    N = w.rows
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    ws_bytes = imp_nvfp4_gemm_workspace_size(M, N, K)
    if workspace is None and ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=x.device)
    st = imp_nvfp4_gemm_mma(x.data_ptr(), M, K, x.stride(0), w.c_struct(), y.data_ptr(),
                            y.stride(0), None if dev_status is None else dev_status.data_ptr(),
                            None if workspace is None else workspace.data_ptr(), ws_bytes,
                            _stream_handle(stream))
    if st != IMP_OK:
        raise ImpError(st, "imp_nvfp4_gemm_mma")
    return y


def gemm_mma_swiglu(gate, up, w: NVFP4Tensor, y=None, dev_status=None, stream=None,
                    workspace=None):
    """Y = bf16(silu(gate) * up) W^T at decode sizes (M <= 16), the
    activation formed inside the call (imp_nvfp4_gemm_mma_swiglu)."""
    import torch
    for t in (gate, up):
        assert t.dtype == torch.bfloat16 and t.dim() == 2 and t.stride(1) == 1
    assert gate.shape == up.shape and gate.stride(0) == up.stride(0) and w.layout == "mma"
    M, K = gate.shape
    N = w.rows
    if y is None:  # row stride rounded up to a multiple of 8 elements
        y = torch.empty((M, (N + 7) // 8 * 8), dtype=torch.bfloat16, device=gate.device)[:, :N]
    ws_bytes = imp_nvfp4_gemm_workspace_size(M, N, K)
    if workspace is None and ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=gate.device)
    st = imp_nvfp4_gemm_mma_swiglu(gate.data_ptr(), up.data_ptr(), M, K, gate.stride(0),
                                   w.c_struct(), y.data_ptr(), y.stride(0),
                                   None if dev_status is None else dev_status.data_ptr(),
                                   None if workspace is None else workspace.data_ptr(), ws_bytes,
                                   _stream_handle(stream))
    if st != IMP_OK:
        raise ImpError(st, "imp_nvfp4_gemm_mma_swiglu")
    return y


def gemm_grouped(x, ws: list, ys=None, dev_status=None, stream=None, workspace=None):
    """[X W_g^T for W_g in ws] in one call for weights in MMA layout
    (prepare_mma) sharing K: one X split and one weight stream for all of
    them at M <= 2."""
    import torch
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    assert all(w.layout == "mma" for w in ws)
    M, K = x.shape
    N = [w.rows for w in ws]
    if ys is None:  # row strides rounded up to a multiple of 8 elements
        ys = [torch.empty((M, (n + 7) // 8 * 8), dtype=torch.bfloat16, device=x.device)[:, :n]
              for n in N]
    ws_bytes = imp_nvfp4_gemm_grouped_workspace_size(M, K, N)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=x.device)
    groups = [ImpNvfp4Group(w.c_struct(), y.data_ptr(), y.stride(0)) for w, y in zip(ws, ys)]
    st = imp_nvfp4_gemm_grouped(x.data_ptr(), M, K, x.stride(0), groups,
                                None if dev_status is None else dev_status.data_ptr(),
                                workspace.data_ptr(), ws_bytes, _stream_handle(stream))
    if st != IMP_OK:
        raise ImpError(st, "imp_nvfp4_gemm_grouped")
    return ys


def gemm_chain(links: list, ys=None, dev_status=None, stream=None, workspace=None):
    """A decode chain in one call: links = [(weights, x), ...] with weights a
    list of MMA-layout tensors of one K and x a bf16 [M][K] tensor, None for
    the previous link's first output, or "swiglu" for silu(g) * u of the
    previous link's first two outputs.  Returns the outputs, one list per
    link (allocated with row strides rounded up to 8 unless given)."""
    import torch
    x0 = links[0][1]
    assert x0 is not None and x0.dtype == torch.bfloat16 and x0.dim() == 2
    M = x0.shape[0]
    if ys is None:
        ys = [[torch.empty((M, (w.rows + 7) // 8 * 8), dtype=torch.bfloat16,
                           device=x0.device)[:, :w.rows] for w in ws] for ws, _ in links]
    spec = []
    for (ws, x), yl in zip(links, ys):
        assert all(w.layout == "mma" for w in ws)
        groups = [ImpNvfp4Group(w.c_struct(), y.data_ptr(), y.stride(0)) for w, y in zip(ws, yl)]
        if x is None or isinstance(x, str):
            assert x in (None, "swiglu")
            spec.append((groups, None, 0, 1 if x == "swiglu" else 0))
        else:
            assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
            spec.append((groups, x.data_ptr(), x.stride(0)))
    cl = ChainLinks(spec)
    ws_bytes = imp_nvfp4_gemm_chain_workspace_size(M, cl)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=x0.device)
    st = imp_nvfp4_gemm_chain(M, cl, None if dev_status is None else dev_status.data_ptr(),
                              workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
    if st != IMP_OK:
        raise ImpError(st, "imp_nvfp4_gemm_chain")
    return ys


# ---- MXFP4 and FP8 weights ----------------------------------------------------------

@dataclass
class MXFP4Tensor:
    """Device MXFP4 tensor: codes uint8[rows][K/2], E8M0 scales uint8[rows][K/32]."""
    codes: "object"
    scales: "object"

    @property
    def rows(self) -> int:
        return self.codes.shape[0]

    @property
    def K(self) -> int:
        return self.codes.shape[1] * 2

    def c_struct(self) -> ImpMxfp4Tensor:
        return ImpMxfp4Tensor(self.codes.data_ptr(), self.scales.data_ptr(), self.rows, self.K)


@dataclass
class FP8Tensor:
    """Device FP8 E4M3 weight: codes uint8[rows][K], tensor_scale float32[1]."""
    codes: "object"
    tensor_scale: "object"

    @property
    def rows(self) -> int:
        return self.codes.shape[0]

    @property
    def K(self) -> int:
        return self.codes.shape[1]

    def c_struct(self) -> ImpFp8Tensor:
        return ImpFp8Tensor(self.codes.data_ptr(), self.tensor_scale.data_ptr(), self.rows, self.K)


def mxfp4_quantize(x, dev_status=None, stream=None) -> MXFP4Tensor:
    """Quantize a 2-D bf16 CUDA tensor to MXFP4 (OCP MX v1.0)."""
    import torch
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, K = x.shape
    out = MXFP4Tensor(torch.empty((rows, K // 2), dtype=torch.uint8, device=x.device),
                      torch.empty((rows, K // 32), dtype=torch.uint8, device=x.device))
    st = imp_mxfp4_quantize(x.data_ptr(), rows, K, x.stride(0), out.c_struct(),
                            None if dev_status is None else dev_status.data_ptr(),
                            _stream_handle(stream))
    if st != IMP_OK:
        raise ImpError(st, "imp_mxfp4_quantize")
    return out


def mxfp4_to_nvfp4(t: MXFP4Tensor, dev_status=None, stream=None) -> NVFP4Tensor:
    """The same values as an NVFP4 tensor (row-major) for the NVFP4 kernels."""
    import torch
    out = NVFP4Tensor(torch.empty_like(t.codes),
                      torch.empty((t.rows, t.K // 16), dtype=torch.uint8, device=t.codes.device),
                      torch.empty(1, dtype=torch.float32, device=t.codes.device))
    wsb = imp_mxfp4_to_nvfp4_workspace_size()
    ws = torch.empty(wsb, dtype=torch.uint8, device=t.codes.device)
    st = imp_mxfp4_to_nvfp4(t.c_struct(), out.c_struct(),
                            None if dev_status is None else dev_status.data_ptr(), ws.data_ptr(),
                            wsb, _stream_handle(stream))
    if st != IMP_OK:
        raise ImpError(st, "imp_mxfp4_to_nvfp4")
    return out


def fp8_quantize(x, dev_status=None, stream=None) -> FP8Tensor:
    """Quantize a 2-D bf16 CUDA tensor to FP8 E4M3 with one tensor scale."""
    import torch
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, K = x.shape
    out = FP8Tensor(torch.empty((rows, K), dtype=torch.uint8, device=x.device),
                    torch.empty(1, dtype=torch.float32, device=x.device))
    wsb = imp_fp8_quantize_workspace_size(rows, K)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=x.device)
    st = imp_fp8_quantize(x.data_ptr(), rows, K, x.stride(0), out.c_struct(),
                          None if dev_status is None else dev_status.data_ptr(), ws.data_ptr(),
                          wsb, _stream_handle(stream))
    if st != IMP_OK:
        raise ImpError(st, "imp_fp8_quantize")
    return out


def gemm_fp8(x, w: FP8Tensor, y=None, dev_status=None, stream=None, workspace=None):
    """Y = X W^T for a decode-sized bf16 X and an FP8 E4M3 weight."""
    import torch
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    N = w.rows
    if y is None:
        y = torch.empty((M, (N + 7) // 8 * 8), dtype=torch.bfloat16, device=x.device)[:, :N]
    wsb = imp_fp8_gemm_workspace_size(M, N, K)
    if workspace is None:
        workspace = torch.empty(max(wsb, 16), dtype=torch.uint8, device=x.device)
    st = imp_fp8_gemm(x.data_ptr(), M, K, x.stride(0), w.c_struct(), y.data_ptr(), y.stride(0),
                      None if dev_status is None else dev_status.data_ptr(), workspace.data_ptr(),
                      wsb, _stream_handle(stream))
    if st != IMP_OK:
        raise ImpError(st, "imp_fp8_gemm")
    return y


def gemm_swiglu(x, w_gate: NVFP4Tensor, w_up: NVFP4Tensor, h=None, h_amax=None, dev_status=None,
                stream=None, workspace=None):
    """(h, h_amax): h = silu(X Wg^T) * (X Wu^T) for a prefill-sized bf16 X and
    gate/up weights in MMA layout; h_amax = max|h| as bf16 magnitude bits
    (device int32[1])."""
    import torch
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    assert w_gate.layout == "mma" and w_up.layout == "mma"
    M, K = x.shape
    N = w_gate.rows
    if h is None:
        h = torch.empty((M, (N + 7) // 8 * 8), dtype=torch.bfloat16, device=x.device)[:, :N]
    if h_amax is None:
        h_amax = torch.zeros(1, dtype=torch.int32, device=x.device)
    wsb = imp_nvfp4_gemm_swiglu_workspace_size(M, N, K)
    if workspace is None:
        workspace = torch.empty(max(wsb, 16), dtype=torch.uint8, device=x.device)
    st = imp_nvfp4_gemm_swiglu(x.data_ptr(), M, K, x.stride(0), w_gate.c_struct(), w_up.c_struct(),
                               h.data_ptr(), h.stride(0), h_amax.data_ptr(),
                               None if dev_status is None else dev_status.data_ptr(),
                               workspace.data_ptr(), wsb, _stream_handle(stream))
    if st != IMP_OK:
        raise ImpError(st, "imp_nvfp4_gemm_swiglu")
    return h, h_amax


def quantize_mma_amax(x, amax, dev_status=None, stream=None) -> NVFP4Tensor:
    """quantize_mma with the global amax given (device int32[1], bf16 bits)."""
    import torch
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, K = x.shape
    out = NVFP4Tensor(torch.empty((rows, K // 2), dtype=torch.uint8, device=x.device),
                      torch.empty(imp_nvfp4_mma_scales_size(rows, K), dtype=torch.uint8,
                                  device=x.device),
                      torch.empty(1, dtype=torch.float32, device=x.device))
    st = imp_nvfp4_quantize_mma_amax(x.data_ptr(), rows, K, x.stride(0), amax.data_ptr(),
                                     _struct(out),
                                     None if dev_status is None else dev_status.data_ptr(),
                                     _stream_handle(stream))
    if st != IMP_OK:
        raise ImpError(st, "imp_nvfp4_quantize_mma_amax")
    return out

"""Seeded synthetic inputs for the NVFP4 linear-layer workloads.

The one input source that both sides use: the oracle (tests) and the device
path (tests, bench) read the same bf16 bytes from here.  The module draws
numbers and rounds them to bf16; it contains no quantization arithmetic.

Every value is a pure function of (seed, tensor name, row, column), so a
subset of rows can be regenerated alone (sampled parity at full size).

Recipes (one per workload; shapes are (K -> N) with Y[M,N] = X[M,K] W^T):

* ``single_1k``   M=1, 1024 -> 1024; W ~ N(0, 0.02^2); X ~ N(0,1); seed 0.
* ``decode_0p6b`` one decode step of a 0.6B-class transformer at M=1:
  q 1024->2048, k 1024->1024, v 1024->1024, o 2048->1024,
  gate 1024->3072, up 1024->3072, down 3072->1024; W ~ N(0, 0.02^2);
  X ~ N(0,1); seed 1.
* ``decode_27b``  27B-class decode at M=1: up/gate 5120->17408,
  down 17408->5120, LM head 5120->151936; W Student-t(4) scaled to std
  0.02 with 0.1 % of 16-wide blocks zeroed; X ~ N(0,1) with 1 % of the
  channels multiplied by 20; seed 2.
* ``skinny_27b``  M in {2,4,8,16}; 5120->17408 and 17408->5120; W as in
  decode_27b; X ~ N(0,1) (no outliers); seed 3.
* ``prefill_27b`` M=2048; 5120->17408 and 17408->5120; W as in decode_27b;
  X ~ N(0,1) with 1 % outlier channels x20; seed 4.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libsynth.so")
_lib = None

DIST_NORMAL = 0
DIST_STUDENT_T4 = 1


def build(force: bool = False) -> str:
    """Compile synth.c into _build/libsynth.so (plain C, any host arch)."""
    src = os.path.join(_HERE, "synth.c")
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-ffp-contract=off", src, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.synth_fill_bf16.restype = ctypes.c_int
        lib.synth_fill_bf16.argtypes = [
            ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_double, ctypes.c_double,
            ctypes.c_void_p, ctypes.c_double, ctypes.c_void_p, ctypes.c_int]
        lib.synth_pick_channels.restype = ctypes.c_int
        lib.synth_pick_channels.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64,
                                            ctypes.c_int64, ctypes.c_void_p]
        _lib = lib
    return _lib


def stream_id(name: str) -> int:
    """Stable 64-bit id of a tensor name (FNV-1a)."""
    h = 0xCBF29CE484222325
    for b in name.encode():
        h ^= b
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def fill_bf16(dist: int, seed: int, name: str, row0: int, rows: int, cols: int,
              scale: float = 1.0, zero_block_p: float = 0.0,
              outlier_mask: np.ndarray | None = None, outlier_mult: float = 1.0,
              out: np.ndarray | None = None) -> np.ndarray:
    """Rows [row0, row0+rows) of a bf16 matrix as uint16 bit patterns."""
    lib = _load()
    if out is None:
        out = np.empty((rows, cols), dtype=np.uint16)
    assert out.dtype == np.uint16 and out.shape == (rows, cols) and out.flags.c_contiguous
    mask_ptr = None
    if outlier_mask is not None:
        outlier_mask = np.ascontiguousarray(outlier_mask, dtype=np.uint8)
        assert outlier_mask.shape == (cols,)
        mask_ptr = outlier_mask.ctypes.data
    rc = lib.synth_fill_bf16(dist, seed, stream_id(name), row0, rows, cols, cols, scale,
                             zero_block_p, mask_ptr, outlier_mult, out.ctypes.data, _threads())
    if rc != 0:
        raise ValueError("synth_fill_bf16: bad arguments")
    return out


def pick_channels(seed: int, name: str, cols: int, count: int) -> np.ndarray:
    """Exactly `count` distinct channels of `cols`, as a uint8 mask."""
    lib = _load()
    mask = np.zeros(cols, dtype=np.uint8)
    if lib.synth_pick_channels(seed, stream_id(name), cols, count, mask.ctypes.data) != 0:
        raise ValueError("synth_pick_channels: bad arguments")
    return mask


@dataclass(frozen=True)
class Linear:
    """One Y[M,N] = X[M,K] W^T problem of a workload."""
    name: str
    M: int
    K: int
    N: int
    seed: int
    w_dist: int = DIST_NORMAL
    w_scale: float = 0.02
    zero_block_p: float = 0.0
    x_outlier_frac: float = 0.0
    x_outlier_mult: float = 20.0

    def weight_bf16(self, row0: int = 0, rows: int | None = None) -> np.ndarray:
        """Rows of W[N][K] (bf16 bit patterns, uint16)."""
        rows = self.N - row0 if rows is None else rows
        return fill_bf16(self.w_dist, self.seed, self.name + ".w", row0, rows, self.K,
                         scale=self.w_scale, zero_block_p=self.zero_block_p)

    def outlier_mask(self) -> np.ndarray | None:
        if self.x_outlier_frac <= 0.0:
            return None
        count = int(round(self.x_outlier_frac * self.K))
        return pick_channels(self.seed, self.name + ".x", self.K, count)

    def act_bf16(self, row0: int = 0, rows: int | None = None) -> np.ndarray:
        """Rows of X[M][K] (bf16 bit patterns, uint16)."""
        rows = self.M - row0 if rows is None else rows
        return fill_bf16(DIST_NORMAL, self.seed, self.name + ".x", row0, rows, self.K,
                         outlier_mask=self.outlier_mask(), outlier_mult=self.x_outlier_mult)

    @property
    def weight_bytes(self) -> int:
        """Bytes of the NVFP4 weight: packed codes + E4M3 block scales + fp32 scale."""
        return self.N * self.K // 2 + self.N * self.K // 16 + 4


# Student-t with nu = 4 has variance nu/(nu-2) = 2; dividing by sqrt(2)
# gives the stated standard deviation of 0.02.
_T4_SCALE = 0.02 / 2 ** 0.5


def _w27(name, M, K, N, seed, outlier_frac):
    return Linear(name, M, K, N, seed, w_dist=DIST_STUDENT_T4, w_scale=_T4_SCALE,
                  zero_block_p=0.001, x_outlier_frac=outlier_frac)


def workload(name: str) -> list[Linear]:
    """The list of linear problems of a named workload.  ``<workload>:<name>``
    selects one problem of a workload (e.g. ``decode_27b:down``)."""
    if ":" in name:
        base, part = name.split(":", 1)
        sel = [l for l in workload(base) if l.name == part]
        if not sel:
            raise KeyError(name)
        return sel
    if name == "single_1k":
        return [Linear("single", 1, 1024, 1024, 0)]
    if name == "decode_0p6b":
        shapes = [("q", 1024, 2048), ("k", 1024, 1024), ("v", 1024, 1024), ("o", 2048, 1024),
                  ("gate", 1024, 3072), ("up", 1024, 3072), ("down", 3072, 1024)]
        return [Linear(n, 1, k, nn, 1) for n, k, nn in shapes]
    if name == "decode_27b":
        return [_w27("up", 1, 5120, 17408, 2, 0.01), _w27("gate", 1, 5120, 17408, 2, 0.01),
                _w27("down", 1, 17408, 5120, 2, 0.01), _w27("lm_head", 1, 5120, 151936, 2, 0.01)]
    if name.startswith("skinny_27b"):
        ms = [2, 4, 8, 16]
        if name != "skinny_27b":
            ms = [int(name.split("_m")[-1])]
        out = []
        for m in ms:
            out += [_w27(f"up_m{m}", m, 5120, 17408, 3, 0.0), _w27(f"down_m{m}", m, 17408, 5120, 3, 0.0)]
        return out
    if name == "prefill_27b":
        return [_w27("up", 2048, 5120, 17408, 4, 0.01), _w27("down", 2048, 17408, 5120, 4, 0.01)]
    raise KeyError(name)


WORKLOADS = ["single_1k", "decode_0p6b", "decode_27b", "skinny_27b", "prefill_27b"]

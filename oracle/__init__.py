"""CPU oracle for the Q4 verify matmul -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline /
``--impl reference`` leg may import this package.  The product path (the CUDA
library under ``bit_row_speculative_gb300``) never imports, links or executes
anything here, and this package imports nothing from it.

The arithmetic lives in ``q4_oracle.c`` (plain C, fp64, -O2, no fast-math):

* ``packed_bytes(N, K)``: the "Splash engine" page's q4PackedBytes
  (section "The engine hard-codes the model"): overflow-checked
  ``(N*K/16)*9``; 0 for an unsupported shape or overflow.
* ``matmul(x, W, N, K)``: ``y[m,n] = sum_k x[m,k]*(s[n,k//64]*q[n,k]+b[n,k//64])``
  exactly up to the fp64 rounding of the running sum (increasing k), plus
  ``sum_k |x*w|`` per output for the tolerance test.
* ``glue(y, K, kind)``: the fixed stand-in for the between-layer operators of
  the chained verify pass (RMS normalisation, optionally after SwiGLU), in fp64,
  rounded once to bf16.

Every function here is pinned by ``tests/test_oracle_pins.py`` against values
that do not come from the oracle itself (hand-packed groups with closed-form
outputs, exact rational brute force, the pages' published byte totals).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD_DIR, "libq4oracle.so")

GLUE_RMSNORM = 1
GLUE_SWIGLU_RMSNORM = 2
GROUP = 64

_lock = threading.Lock()
_lib = None


def compile_oracle(src: str = _SRC, out: str = _SO, defines: tuple[str, ...] = ()) -> str:
    """Compile the C oracle into a shared library (gcc -O2, no fast-math)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", *defines, src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def build(force: bool = False) -> str:
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        compile_oracle()
    return _SO


def load_library(path: str) -> ctypes.CDLL:
    lib = ctypes.CDLL(path)
    lib.q4o_packed_bytes.restype = ctypes.c_uint64
    lib.q4o_packed_bytes.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
    lib.q4o_matmul_cols_f64.restype = ctypes.c_int
    lib.q4o_matmul_cols_f64.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64,
        ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    lib.q4o_glue_f64.restype = ctypes.c_int
    lib.q4o_glue_f64.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64,
                                 ctypes.c_int, ctypes.c_double, ctypes.c_void_p]
    lib.q4o_weight.restype = ctypes.c_double
    lib.q4o_weight.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64,
                               ctypes.c_uint64, ctypes.c_uint64]
    lib.q4o_f64_to_bf16.restype = ctypes.c_uint16
    lib.q4o_f64_to_bf16.argtypes = [ctypes.c_double]
    lib.q4o_bf16_to_f64.restype = ctypes.c_double
    lib.q4o_bf16_to_f64.argtypes = [ctypes.c_uint16]
    return lib


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
        return _lib


class Oracle:
    """Typed wrapper over one compiled oracle library (the real one, or a
    deliberately broken copy built by the mutation tests)."""

    def __init__(self, cdll: ctypes.CDLL):
        self._l = cdll

    def packed_bytes(self, N: int, K: int) -> int:
        return int(self._l.q4o_packed_bytes(N, K))

    def matmul(self, x_bits: np.ndarray, W: np.ndarray, N: int, K: int,
               cols: np.ndarray | None = None, threads: int | None = None):
        """x_bits: uint16 [M, K] bf16 bit patterns; W: uint8 packed buffer.
        Returns (y, absy): float64 [M, ncols] each."""
        x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
        W = np.ascontiguousarray(W, dtype=np.uint8)
        M = x_bits.shape[0]
        assert x_bits.shape == (M, K)
        assert W.size == self.packed_bytes(N, K)
        if cols is None:
            ncols, cptr = N, None
        else:
            cols = np.ascontiguousarray(cols, dtype=np.int64)
            ncols, cptr = cols.size, cols.ctypes.data
        y = np.zeros((M, ncols), dtype=np.float64)
        a = np.zeros((M, ncols), dtype=np.float64)
        if threads is None:
            threads = os.cpu_count() or 1
        rc = self._l.q4o_matmul_cols_f64(x_bits.ctypes.data, W.ctypes.data, M, N, K, cptr,
                                         ncols, y.ctypes.data, a.ctypes.data, threads)
        if rc != 0:
            raise ValueError(f"oracle matmul rejected arguments (rc={rc})")
        return y, a

    def weight(self, W: np.ndarray, N: int, K: int, n: int, k: int) -> float:
        W = np.ascontiguousarray(W, dtype=np.uint8)
        return float(self._l.q4o_weight(W.ctypes.data, N, K, n, k))

    def glue(self, y: np.ndarray, K: int, kind: int, eps: float = 1e-6) -> np.ndarray:
        y = np.ascontiguousarray(y, dtype=np.float32)
        M, Nprev = y.shape
        out = np.zeros((M, K), dtype=np.uint16)
        rc = self._l.q4o_glue_f64(y.ctypes.data, M, Nprev, K, kind, eps, out.ctypes.data)
        if rc != 0:
            raise ValueError(f"oracle glue rejected arguments (rc={rc})")
        return out

    def f64_to_bf16(self, v: float) -> int:
        return int(self._l.q4o_f64_to_bf16(v))

    def bf16_to_f64(self, h: int) -> float:
        return float(self._l.q4o_bf16_to_f64(h))


_default = None


def get() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(lib())
    return _default


def packed_bytes(N: int, K: int) -> int:
    return get().packed_bytes(N, K)


def matmul(x_bits, W, N, K, cols=None, threads=None):
    return get().matmul(x_bits, W, N, K, cols=cols, threads=threads)


def glue(y, K, kind, eps=1e-6):
    return get().glue(y, K, kind, eps)

"""f64 CPU checker for the affine group-wise quantized matmul (ctypes binding).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the smoke check and by
the benchmark's CPU-baseline / reference leg, never by the CUDA library.  It
shares no code with the CUDA path: its arithmetic lives in ``mxq_oracle.c``
(plain f64 loops; each function there cites the page passage it follows).

Functions take numpy arrays in the storage conventions of ``synth`` (bf16 as
uint16 bits, packed uint32 codes) and return float64 results plus the
per-element magnitude bound ``sum_k |x_k * w^_kn|`` used by the parity
tolerance.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxq_oracle.c")
_LIB = os.path.join(_HERE, "libmxq_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the checker with gcc and OpenMP (plain C, any host arch)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_threads.restype = I
            lib.oracle_unpack.argtypes = [P, I, I, I, P]
            lib.oracle_dequant.argtypes = [P, P, P, I, I, I, I, P]
            lib.oracle_qmm.argtypes = [P, P, P, P, I, I, I, I, I, P, P]
            lib.oracle_qmm.restype = I
            lib.oracle_qmv.argtypes = [P, P, P, P, I, I, I, I, P, P]
            lib.oracle_qmv.restype = I
            lib.oracle_gather_qmm.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, P, P]
            lib.oracle_gather_qmm.restype = I
            lib.oracle_points.argtypes = [P, P, P, P, P, P, I, I, I, I, I,
                                          P, P, ctypes.c_longlong, P, P]
            lib.oracle_points.restype = I
            lib.oracle_quantize.argtypes = [P, I, I, I, I, P, P, P]
            lib.oracle_qmm_kn.argtypes = [P, P, P, P, I, I, I, I, I, P, P]
            lib.oracle_qmm_kn.restype = I
            _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(np.asarray(a, dtype=dtype))
    return a, a.ctypes.data_as(ctypes.c_void_p)


def threads() -> int:
    return _load().oracle_threads()


def unpack(w, N: int, K: int, bits: int) -> np.ndarray:
    w, pw = _c(w, np.uint32)
    q = np.empty((N, K), dtype=np.uint8)
    _load().oracle_unpack(pw, N, K, bits, q.ctypes.data_as(ctypes.c_void_p))
    return q


def dequant(w, scales, biases, N: int, K: int, bits: int, group: int = 64) -> np.ndarray:
    w, pw = _c(w, np.uint32)
    s, ps = _c(scales, np.uint16)
    b, pb = _c(biases, np.uint16)
    out = np.empty((N, K), dtype=np.float64)
    _load().oracle_dequant(pw, ps, pb, N, K, bits, group, out.ctypes.data_as(ctypes.c_void_p))
    return out


def qmm(x, w, scales, biases, M: int, K: int, N: int, bits: int, group: int = 64):
    """y[M, N] and bound[M, N] in f64."""
    x, px = _c(x, np.uint16)
    w, pw = _c(w, np.uint32)
    s, ps = _c(scales, np.uint16)
    b, pb = _c(biases, np.uint16)
    y = np.empty((M, N), dtype=np.float64)
    bnd = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_qmm(px, pw, ps, pb, M, K, N, bits, group,
                            y.ctypes.data_as(ctypes.c_void_p), bnd.ctypes.data_as(ctypes.c_void_p))
    if rc:
        raise MemoryError("oracle_qmm failed")
    return y, bnd


def qmm_kn(x, w, scales, biases, M: int, K: int, N: int, bits: int, group: int = 64):
    """The [K, N] operand layout: w uint32 [K, N*bits/32] (codes along n),
    scales/biases bf16 bits [K, N/group]; y[M, N] and bound[M, N] in f64."""
    x, px = _c(x, np.uint16)
    w, pw = _c(w, np.uint32)
    s, ps = _c(scales, np.uint16)
    b, pb = _c(biases, np.uint16)
    y = np.empty((M, N), dtype=np.float64)
    bnd = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_qmm_kn(px, pw, ps, pb, M, K, N, bits, group,
                               y.ctypes.data_as(ctypes.c_void_p),
                               bnd.ctypes.data_as(ctypes.c_void_p))
    if rc:
        raise MemoryError("oracle_qmm_kn failed")
    return y, bnd


def qmv(x, w, scales, biases, K: int, N: int, bits: int, group: int = 64):
    """y[N] and bound[N] in f64 for one activation row."""
    x, px = _c(x, np.uint16)
    w, pw = _c(w, np.uint32)
    s, ps = _c(scales, np.uint16)
    b, pb = _c(biases, np.uint16)
    y = np.empty((N,), dtype=np.float64)
    bnd = np.empty((N,), dtype=np.float64)
    rc = _load().oracle_qmv(px, pw, ps, pb, K, N, bits, group,
                            y.ctypes.data_as(ctypes.c_void_p), bnd.ctypes.data_as(ctypes.c_void_p))
    if rc:
        raise MemoryError("oracle_qmv failed")
    return y, bnd


def gather_qmm(x, w, scales, biases, expert_ids, row_src, T: int, B: int, E: int,
               K: int, N: int, bits: int, group: int = 64):
    """Sorted-MoE y[B, N] and bound[B, N]; ``row_src`` None means identity."""
    x, px = _c(x, np.uint16)
    w, pw = _c(w, np.uint32)
    s, ps = _c(scales, np.uint16)
    b, pb = _c(biases, np.uint16)
    e, pe = _c(expert_ids, np.int32)
    if row_src is None:
        pr = None
    else:
        r, pr = _c(row_src, np.int32)
    y = np.empty((B, N), dtype=np.float64)
    bnd = np.empty((B, N), dtype=np.float64)
    rc = _load().oracle_gather_qmm(px, pw, ps, pb, pe, pr, T, B, E, K, N, bits, group,
                                   y.ctypes.data_as(ctypes.c_void_p),
                                   bnd.ctypes.data_as(ctypes.c_void_p))
    if rc:
        raise MemoryError("oracle_gather_qmm failed")
    return y, bnd


def points(x, w, scales, biases, rows, cols, K: int, N: int, bits: int, group: int = 64,
           expert_ids=None, row_src=None, E: int = 1):
    """Outputs (rows[i], cols[i]) only, with their bounds, for full-size
    launches checked on a sample.  Without ``expert_ids`` this is qmm/qmv."""
    x, px = _c(x, np.uint16)
    w, pw = _c(w, np.uint32)
    s, ps = _c(scales, np.uint16)
    b, pb = _c(biases, np.uint16)
    rr, prr = _c(rows, np.int64)
    cc, pcc = _c(cols, np.int64)
    pe = pr = None
    if expert_ids is not None:
        e, pe = _c(expert_ids, np.int32)
    if row_src is not None:
        r, pr = _c(row_src, np.int32)
    n = rr.shape[0]
    y = np.empty((n,), dtype=np.float64)
    bnd = np.empty((n,), dtype=np.float64)
    rc = _load().oracle_points(px, pw, ps, pb, pe, pr, E, K, N, bits, group, prr, pcc, n,
                               y.ctypes.data_as(ctypes.c_void_p),
                               bnd.ctypes.data_as(ctypes.c_void_p))
    if rc:
        raise MemoryError("oracle_points failed")
    return y, bnd


def quantize(W, bits: int, group: int = 64):
    """The affine min/max encoder, binary32 decisions: (codes uint32
    [N, K*bits/32], scales and biases as bf16 bits uint16 [N, K/group])."""
    W, pw = _c(W, np.float32)
    N, K = W.shape
    codes = np.zeros((N, K * bits // 32), np.uint32)
    scales = np.zeros((N, K // group), np.uint16)
    biases = np.zeros((N, K // group), np.uint16)
    _load().oracle_quantize(pw, N, K, bits, group, codes.ctypes.data_as(ctypes.c_void_p),
                            scales.ctypes.data_as(ctypes.c_void_p),
                            biases.ctypes.data_as(ctypes.c_void_p))
    return codes, scales, biases


def within_tolerance(y_gpu, y_ref, bound, rel: float = 8e-3, abs_: float = 1e-3):
    """Elementwise acceptance |y_gpu - y_ref| <= rel * bound + abs_; returns
    (ok mask, worst ratio of error to allowance)."""
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref)
    allow = rel * bound + abs_
    ok = err <= allow
    worst = float(np.max(err / allow)) if err.size else 0.0
    return ok, worst

"""affine_bit_matmul_gb300 — affine group-wise quantized matmul on GB300.

A thin Python binding over the C ABI of ``libmxq.so`` (declared in
``include/mxq.h``).  Every step of the computation runs in the library's
sm_103a kernels; this module only checks tensors, passes their device
pointers and the current CUDA stream, and turns status codes into
exceptions.  There is no fallback: if the library is missing or the device
is not sm_103a, the calls raise.

Storage conventions (mlxcel issue #1536, Baseline section: "affine 4-bit /
group 64"):

* ``x``: bf16 ``[M, K]`` (``[K]`` for ``qmv``);
* ``w``: int32 or uint32 ``[N, K*bits/32]`` packed codes, 4-bit codes eight per
  little-endian word (lowest k in the lowest nibble), 2-bit codes sixteen per
  word, 8-bit codes four per word; 3- and 6-bit codes continue the same
  little-endian bit stream per row and may straddle words (``bits`` in 2, 3,
  4, 6, 8);
* ``scales``, ``biases``: bf16 ``[N, K/group_size]``, one pair per group of
  ``group_size`` consecutive k (32, 64 or 128; every call defaults to 64);
* result ``y``: bf16 ``[M, N]``.
"""

from __future__ import annotations

import ctypes
import os

__all__ = [
    "lib",
    "qmv",
    "qmm",
    "qmv_kn",
    "qmm_kn",
    "gather_qmm",
    "gather_qmm_kn",
    "gather_qmm_gateup",
    "gather_workspace_bytes",
    "gather_qmm_noalloc",
    "quantize",
    "set_wait_budget",
    "NOALLOC_SCRATCH_BYTES",
    "MxqError",
    "DEV_BAD_EXPERT_ID",
    "DEV_UNSORTED_IDS",
    "DEV_BAD_ROW_SRC",
    "DEV_TIMEOUT",
    "EXPORTED_SYMBOLS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmxq.so")

MXQ_OK = 0
STATUS_NAMES = {
    0: "MXQ_OK",
    1: "MXQ_ERR_INVALID_ARG",
    2: "MXQ_ERR_MISALIGNED",
    3: "MXQ_ERR_UNSUPPORTED",
    4: "MXQ_ERR_ARCH",
    5: "MXQ_ERR_CUDA",
    6: "MXQ_ERR_WORKSPACE",
    7: "MXQ_ERR_SCRATCH_LIMIT",
}
DEV_BAD_EXPERT_ID = 0x1
DEV_UNSORTED_IDS = 0x2
DEV_BAD_ROW_SRC = 0x4
DEV_TIMEOUT = 0x8
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024  # MXQ_NOALLOC_SCRATCH_BYTES

EXPORTED_SYMBOLS = (
    "mxq_qmv",
    "mxq_qmm",
    "mxq_qmv_kn",
    "mxq_qmm_kn",
    "mxq_gather_qmm",
    "mxq_gather_qmm_kn",
    "mxq_gather_qmm_gateup",
    "mxq_gather_workspace_bytes",
    "mxq_gather_qmm_noalloc",
    "mxq_quantize",
    "mxq_status_string",
    "mxq_version",
    "mxq_debug_set_wait_budget",
)


class MxqError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s (%s)" % (what, STATUS_NAMES.get(status, status),
                                           _status_string(status)))


_lib_handle = None


def lib():
    """The loaded ``libmxq.so`` with argument types set (raises if absent)."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libmxq.so is not built; run affine_bit_matmul_gb300.build.build() "
                "(needs nvcc) before using the library")
        L = ctypes.CDLL(LIB_PATH)
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.mxq_qmv.argtypes = [P, P, P, P, P, I, I, I, I, P, P]
        L.mxq_qmv.restype = I
        L.mxq_qmm.argtypes = [P, P, P, P, P, I, I, I, I, I, P, P]
        L.mxq_qmm.restype = I
        L.mxq_qmv_kn.argtypes = [P, P, P, P, P, I, I, I, I, P, P]
        L.mxq_qmv_kn.restype = I
        L.mxq_qmm_kn.argtypes = [P, P, P, P, P, I, I, I, I, I, P, P]
        L.mxq_qmm_kn.restype = I
        L.mxq_gather_qmm.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, Z, P, P]
        L.mxq_gather_qmm.restype = I
        L.mxq_gather_qmm_kn.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, Z, P, P]
        L.mxq_gather_qmm_kn.restype = I
        L.mxq_gather_qmm_gateup.argtypes = [P, P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I,
                                             I, P, Z, P, P]
        L.mxq_gather_qmm_gateup.restype = I
        L.mxq_gather_qmm_noalloc.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, P]
        L.mxq_gather_qmm_noalloc.restype = I
        L.mxq_quantize.argtypes = [P, P, P, P, I, I, I, I, P]
        L.mxq_quantize.restype = I
        L.mxq_gather_workspace_bytes.argtypes = [I, I, I, I]
        L.mxq_gather_workspace_bytes.restype = Z
        L.mxq_status_string.argtypes = [I]
        L.mxq_status_string.restype = ctypes.c_char_p
        L.mxq_version.restype = I
        L.mxq_debug_set_wait_budget.argtypes = [ctypes.c_longlong]
        L.mxq_debug_set_wait_budget.restype = ctypes.c_longlong
        _lib_handle = L
    return _lib_handle


def _status_string(status: int) -> str:
    try:
        return lib().mxq_status_string(status).decode()
    except Exception:  # library not loadable: name only
        return STATUS_NAMES.get(status, "unknown")


def _check(status: int, what: str):
    if status != MXQ_OK:
        raise MxqError(status, what)


# ---------------------------------------------------------------- torch level

def _torch():
    import torch

    return torch


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _launch_on(device, stream):
    """The device context and raw stream handle for a call on ``device``.

    The library launches on the CUDA device that is current when it is
    called, so every wrapper makes the tensors' device current for the call;
    ``stream`` (default: that device's current stream) must belong to the
    same device, else the launch would pair one device's pointers with
    another device's stream."""
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    elif stream.device != device:
        raise ValueError("stream is on %s but the tensors are on %s" % (stream.device, device))
    return torch.cuda.device(device), ctypes.c_void_p(stream.cuda_stream)


def _require(t, name, dtypes, device=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype not in dtypes:
        raise TypeError("%s has dtype %s, expected one of %s" % (name, t.dtype, dtypes))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))


def _code_dtypes():
    torch = _torch()
    out = [torch.int32]
    if hasattr(torch, "uint32"):
        out.append(torch.uint32)
    return tuple(out)


def _check_weights(w, scales, biases, N, K, bits, device, lead=(), group_size=64):
    torch = _torch()
    _require(w, "w", _code_dtypes(), device)
    _require(scales, "scales", (torch.bfloat16,), device)
    _require(biases, "biases", (torch.bfloat16,), device)
    if tuple(w.shape) != tuple(lead) + (N, K * bits // 32):
        raise ValueError("w has shape %s, expected %s" % (tuple(w.shape), tuple(lead) + (N, K * bits // 32)))
    if group_size <= 0:
        raise ValueError("group_size must be positive")
    for t, name in ((scales, "scales"), (biases, "biases")):
        if tuple(t.shape) != tuple(lead) + (N, K // group_size):
            raise ValueError("%s has shape %s, expected %s" % (
                name, tuple(t.shape), tuple(lead) + (N, K // group_size)))


def qmv(x, w, scales, biases, bits: int, out=None, dev_status=None, stream=None,
        group_size: int = 64):
    """Decode GEMV: ``y[N] = sum_k x[k] * (s*q + b)[n, k]`` (``x`` bf16 [K]).
    ``dev_status`` (CUDA int32 [1]) receives DEV_TIMEOUT if a wait gave up."""
    torch = _torch()
    _require(x, "x", (torch.bfloat16,))
    if x.dim() != 1:
        raise ValueError("x must be 1-D [K]")
    K = x.shape[0]
    N = w.shape[0]
    _check_weights(w, scales, biases, N, K, bits, x.device, group_size=group_size)
    if out is None:
        out = torch.empty((N,), dtype=torch.bfloat16, device=x.device)
    _require(out, "out", (torch.bfloat16,), x.device)
    if dev_status is not None:
        _require(dev_status, "dev_status", (torch.int32,), x.device)
    ctx, st = _launch_on(x.device, stream)
    with ctx:
        _check(lib().mxq_qmv(_ptr(x), _ptr(w), _ptr(scales), _ptr(biases), _ptr(out), K, N, bits,
                             group_size, _ptr(dev_status), st), "mxq_qmv")
    return out


def qmv_kn(x, w, scales, biases, bits: int, out=None, dev_status=None, stream=None,
           group_size: int = 64):
    """Decode GEMV with w stored [K, N] (codes and groups along n):
    ``y[n] = sum_k x[k] * (s[k, n/G] q[k, n] + b[k, n/G])``; ``w`` int32
    [K, N*bits/32], ``scales``/``biases`` bf16 [K, N/G], ``x`` bf16 [K]."""
    torch = _torch()
    _require(x, "x", (torch.bfloat16,))
    if x.dim() != 1:
        raise ValueError("x must be 1-D [K]")
    K = x.shape[0]
    _require(w, "w", _code_dtypes(), x.device)
    _require(scales, "scales", (torch.bfloat16,), x.device)
    _require(biases, "biases", (torch.bfloat16,), x.device)
    if w.dim() != 2 or w.shape[0] != K:
        raise ValueError("w must be [K, N*bits/32]")
    N = w.shape[1] * 32 // bits
    if group_size <= 0:
        raise ValueError("group_size must be positive")
    for t, name in ((scales, "scales"), (biases, "biases")):
        if tuple(t.shape) != (K, N // group_size):
            raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape),
                                                               (K, N // group_size)))
    if out is None:
        out = torch.empty((N,), dtype=torch.bfloat16, device=x.device)
    _require(out, "out", (torch.bfloat16,), x.device)
    if dev_status is not None:
        _require(dev_status, "dev_status", (torch.int32,), x.device)
    ctx, st = _launch_on(x.device, stream)
    with ctx:
        _check(lib().mxq_qmv_kn(_ptr(x), _ptr(w), _ptr(scales), _ptr(biases), _ptr(out), K, N,
                                bits, group_size, _ptr(dev_status), st), "mxq_qmv_kn")
    return out


def qmm(x, w, scales, biases, bits: int, out=None, dev_status=None, stream=None,
        group_size: int = 64):
    """Prefill GEMM on the tensor cores: ``y[M, N] = x[M, K] . w^[N, K]^T``.

    ``dev_status`` (CUDA int32 [1]) receives DEV_TIMEOUT if a pipeline wait
    gave up.
    """
    torch = _torch()
    _require(x, "x", (torch.bfloat16,))
    if x.dim() != 2:
        raise ValueError("x must be 2-D [M, K]")
    M, K = x.shape
    N = w.shape[0]
    _check_weights(w, scales, biases, N, K, bits, x.device, group_size=group_size)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _require(out, "out", (torch.bfloat16,), x.device)
    if dev_status is not None:
        _require(dev_status, "dev_status", (torch.int32,), x.device)
    ctx, st = _launch_on(x.device, stream)
    with ctx:
        _check(lib().mxq_qmm(_ptr(x), _ptr(w), _ptr(scales), _ptr(biases), _ptr(out), M, K, N,
                             bits, group_size, _ptr(dev_status), st), "mxq_qmm")
    return out


def _check_weights_kn(w, scales, biases, K, N, bits, device, lead=(), group_size=64):
    """[K, N]-layout weights: ``w`` int32 [..., K, N*bits/32], ``scales`` and
    ``biases`` bf16 [..., K, N/G]."""
    torch = _torch()
    _require(w, "w", _code_dtypes(), device)
    _require(scales, "scales", (torch.bfloat16,), device)
    _require(biases, "biases", (torch.bfloat16,), device)
    if group_size <= 0:
        raise ValueError("group_size must be positive")
    if tuple(w.shape) != tuple(lead) + (K, N * bits // 32):
        raise ValueError("w has shape %s, expected %s" % (tuple(w.shape),
                                                          tuple(lead) + (K, N * bits // 32)))
    for t, name in ((scales, "scales"), (biases, "biases")):
        if tuple(t.shape) != tuple(lead) + (K, N // group_size):
            raise ValueError("%s has shape %s, expected %s" % (
                name, tuple(t.shape), tuple(lead) + (K, N // group_size)))


def qmm_kn(x, w, scales, biases, bits: int, out=None, dev_status=None, stream=None,
           group_size: int = 64):
    """Prefill GEMM with w stored [K, N] (codes and groups along n):
    ``y[m, n] = sum_k x[m, k] (s[k, n/G] q[k, n] + b[k, n/G])``; ``x`` bf16
    [M, K], ``w`` int32 [K, N*bits/32], ``scales``/``biases`` bf16 [K, N/G]."""
    torch = _torch()
    _require(x, "x", (torch.bfloat16,))
    if x.dim() != 2:
        raise ValueError("x must be 2-D [M, K]")
    M, K = x.shape
    if w.dim() != 2:
        raise ValueError("w must be [K, N*bits/32]")
    N = w.shape[1] * 32 // bits
    _check_weights_kn(w, scales, biases, K, N, bits, x.device, group_size=group_size)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _require(out, "out", (torch.bfloat16,), x.device)
    if tuple(out.shape) != (M, N):
        raise ValueError("out has shape %s, expected %s" % (tuple(out.shape), (M, N)))
    if dev_status is not None:
        _require(dev_status, "dev_status", (torch.int32,), x.device)
    ctx, st = _launch_on(x.device, stream)
    with ctx:
        _check(lib().mxq_qmm_kn(_ptr(x), _ptr(w), _ptr(scales), _ptr(biases), _ptr(out), M, K, N,
                                bits, group_size, _ptr(dev_status), st), "mxq_qmm_kn")
    return out


def gather_qmm_kn(x, w, scales, biases, expert_ids, row_src, bits: int, out=None, workspace=None,
                  dev_status=None, stream=None, group_size: int = 64):
    """Sorted mixture-of-experts GEMM with each expert's w stored [K, N]:
    ``w`` int32 [E, K, N*bits/32], ``scales``/``biases`` bf16 [E, K, N/G];
    sorted row r multiplies ``x[row_src[r]]`` by expert ``expert_ids[r]``."""
    torch = _torch()
    _require(x, "x", (torch.bfloat16,))
    if x.dim() != 2:
        raise ValueError("x must be 2-D [T, K]")
    T, K = x.shape
    if w.dim() != 3:
        raise ValueError("w must be [E, K, N*bits/32]")
    E = w.shape[0]
    N = w.shape[2] * 32 // bits
    _check_weights_kn(w, scales, biases, K, N, bits, x.device, lead=(E,), group_size=group_size)
    _require(expert_ids, "expert_ids", (torch.int32,), x.device)
    B = expert_ids.numel()
    if row_src is not None:
        _require(row_src, "row_src", (torch.int32,), x.device)
        if row_src.numel() != B:
            raise ValueError("row_src must have B entries")
    if out is None:
        out = torch.empty((B, N), dtype=torch.bfloat16, device=x.device)
    _require(out, "out", (torch.bfloat16,), x.device)
    if tuple(out.shape) != (B, N):
        raise ValueError("out has shape %s, expected %s" % (tuple(out.shape), (B, N)))
    if workspace is None:
        workspace = torch.empty((gather_workspace_bytes(B, E, K if row_src is not None else 0, N),),
                                dtype=torch.uint8, device=x.device)
    _require(workspace, "workspace", (torch.uint8,), x.device)
    if dev_status is not None:
        _require(dev_status, "dev_status", (torch.int32,), x.device)
    ctx, st = _launch_on(x.device, stream)
    with ctx:
        _check(lib().mxq_gather_qmm_kn(
            _ptr(x), _ptr(w), _ptr(scales), _ptr(biases), _ptr(expert_ids), _ptr(row_src),
            _ptr(out), T, B, E, K, N, bits, group_size, _ptr(workspace), workspace.numel(),
            _ptr(dev_status), st), "mxq_gather_qmm_kn")
    return out


def quantize(w, bits: int, codes=None, scales=None, biases=None, stream=None,
             group_size: int = 64):
    """Affine group-wise encoder on the GPU: float32 ``w`` [N, K] -> (codes
    int32 [N, K*bits/32], scales bf16 [N, K/G], biases bf16 [N, K/G]),
    G = ``group_size``."""
    torch = _torch()
    _require(w, "w", (torch.float32,))
    if w.dim() != 2:
        raise ValueError("w must be 2-D [N, K]")
    N, K = w.shape
    dev = w.device
    if codes is None:
        codes = torch.empty((N, K * bits // 32), dtype=torch.int32, device=dev)
    if group_size <= 0:
        raise ValueError("group_size must be positive")
    if scales is None:
        scales = torch.empty((N, K // group_size), dtype=torch.bfloat16, device=dev)
    if biases is None:
        biases = torch.empty((N, K // group_size), dtype=torch.bfloat16, device=dev)
    _check_weights(codes, scales, biases, N, K, bits, dev, group_size=group_size)
    ctx, st = _launch_on(dev, stream)
    with ctx:
        _check(lib().mxq_quantize(_ptr(w), _ptr(codes), _ptr(scales), _ptr(biases), N, K, bits,
                                  group_size, st), "mxq_quantize")
    return codes, scales, biases


def gather_workspace_bytes(B: int, E: int, K: int, N: int) -> int:
    """Workspace bytes for gather_qmm and gather_qmm_gateup; pass K = 0 when
    row_src is None."""
    return int(lib().mxq_gather_workspace_bytes(B, E, K, N))


def gather_qmm_noalloc(x, w, scales, biases, expert_ids, row_src, bits: int, out,
                       dev_status=None, stream=None, group_size: int = 64):
    """gather_qmm without any allocation: ``out`` must be given, and the
    scratch is the library's fixed MXQ_NOALLOC_SCRATCH_BYTES array (calls on
    one device must not overlap in time; see include/mxq.h)."""
    torch = _torch()
    _require(x, "x", (torch.bfloat16,))
    if x.dim() != 2:
        raise ValueError("x must be 2-D [T, K]")
    T, K = x.shape
    if w.dim() != 3:
        raise ValueError("w must be 3-D [E, N, K*bits/32]")
    E, N = w.shape[0], w.shape[1]
    _check_weights(w, scales, biases, N, K, bits, x.device, lead=(E,), group_size=group_size)
    _require(expert_ids, "expert_ids", (torch.int32,), x.device)
    B = expert_ids.numel()
    if row_src is not None:
        _require(row_src, "row_src", (torch.int32,), x.device)
        if row_src.numel() != B:
            raise ValueError("row_src must have B entries")
    _require(out, "out", (torch.bfloat16,), x.device)
    if tuple(out.shape) != (B, N):
        raise ValueError("out has shape %s, expected %s" % (tuple(out.shape), (B, N)))
    if dev_status is not None:
        _require(dev_status, "dev_status", (torch.int32,), x.device)
    ctx, st = _launch_on(x.device, stream)
    with ctx:
        _check(lib().mxq_gather_qmm_noalloc(_ptr(x), _ptr(w), _ptr(scales), _ptr(biases),
                                            _ptr(expert_ids), _ptr(row_src), _ptr(out), T, B, E, K,
                                            N, bits, group_size, _ptr(dev_status),
                                            st), "mxq_gather_qmm_noalloc")
    return out


def gather_qmm(x, w, scales, biases, expert_ids, row_src, bits: int, out=None, workspace=None,
               dev_status=None, stream=None, group_size: int = 64):
    """Sorted mixture-of-experts GEMM: sorted row r multiplies expert
    ``expert_ids[r]``'s dequantised matrix by ``x[row_src[r]]``.

    ``w`` is [E, N, K*bits/32], ``scales``/``biases`` [E, N, K/group_size],
    ``expert_ids`` int32 [B] non-decreasing, ``row_src`` int32 [B] or None
    (identity).  Returns y bf16 [B, N] in sorted row order.
    """
    torch = _torch()
    _require(x, "x", (torch.bfloat16,))
    if x.dim() != 2:
        raise ValueError("x must be 2-D [T, K]")
    T, K = x.shape
    if w.dim() != 3:
        raise ValueError("w must be 3-D [E, N, K*bits/32]")
    E, N = w.shape[0], w.shape[1]
    _check_weights(w, scales, biases, N, K, bits, x.device, lead=(E,), group_size=group_size)
    _require(expert_ids, "expert_ids", (torch.int32,), x.device)
    B = expert_ids.numel()
    if row_src is not None:
        _require(row_src, "row_src", (torch.int32,), x.device)
        if row_src.numel() != B:
            raise ValueError("row_src must have B entries")
    if out is None:
        out = torch.empty((B, N), dtype=torch.bfloat16, device=x.device)
    _require(out, "out", (torch.bfloat16,), x.device)
    if workspace is None:
        workspace = torch.empty((gather_workspace_bytes(B, E, K if row_src is not None else 0, N),),
                                dtype=torch.uint8, device=x.device)
    _require(workspace, "workspace", (torch.uint8,), x.device)
    if dev_status is not None:
        _require(dev_status, "dev_status", (torch.int32,), x.device)
    ctx, st = _launch_on(x.device, stream)
    with ctx:
        _check(lib().mxq_gather_qmm(_ptr(x), _ptr(w), _ptr(scales), _ptr(biases),
                                    _ptr(expert_ids), _ptr(row_src), _ptr(out), T, B, E, K, N,
                                    bits, group_size, _ptr(workspace), workspace.numel(),
                                    _ptr(dev_status), st), "mxq_gather_qmm")
    return out


def gather_qmm_gateup(x, w_gate, s_gate, b_gate, w_up, s_up, b_up, expert_ids, row_src,
                      bits: int, out_gate=None, out_up=None, workspace=None, dev_status=None,
                      stream=None, group_size: int = 64):
    """The gate and up projections of a mixture-of-experts layer: the same
    routed rows against two expert weight sets of one shape.  Returns
    (y_gate, y_up), each bf16 [B, N] in sorted row order; no activation
    function is applied."""
    torch = _torch()
    _require(x, "x", (torch.bfloat16,))
    if x.dim() != 2:
        raise ValueError("x must be 2-D [T, K]")
    T, K = x.shape
    if w_gate.dim() != 3 or tuple(w_up.shape) != tuple(w_gate.shape):
        raise ValueError("w_gate and w_up must both be [E, N, K*bits/32]")
    E, N = w_gate.shape[0], w_gate.shape[1]
    _check_weights(w_gate, s_gate, b_gate, N, K, bits, x.device, lead=(E,),
                   group_size=group_size)
    _check_weights(w_up, s_up, b_up, N, K, bits, x.device, lead=(E,), group_size=group_size)
    _require(expert_ids, "expert_ids", (torch.int32,), x.device)
    B = expert_ids.numel()
    if row_src is not None:
        _require(row_src, "row_src", (torch.int32,), x.device)
        if row_src.numel() != B:
            raise ValueError("row_src must have B entries")
    outs = []
    for o, name in ((out_gate, "out_gate"), (out_up, "out_up")):
        if o is None:
            o = torch.empty((B, N), dtype=torch.bfloat16, device=x.device)
        _require(o, name, (torch.bfloat16,), x.device)
        if tuple(o.shape) != (B, N):
            raise ValueError("%s has shape %s, expected %s" % (name, tuple(o.shape), (B, N)))
        outs.append(o)
    if workspace is None:
        workspace = torch.empty((gather_workspace_bytes(B, E, K if row_src is not None else 0, N),),
                                dtype=torch.uint8, device=x.device)
    _require(workspace, "workspace", (torch.uint8,), x.device)
    if dev_status is not None:
        _require(dev_status, "dev_status", (torch.int32,), x.device)
    ctx, st = _launch_on(x.device, stream)
    with ctx:
        _check(lib().mxq_gather_qmm_gateup(
            _ptr(x), _ptr(w_gate), _ptr(s_gate), _ptr(b_gate), _ptr(w_up), _ptr(s_up), _ptr(b_up),
            _ptr(expert_ids), _ptr(row_src), _ptr(outs[0]), _ptr(outs[1]), T, B, E, K, N, bits,
            group_size, _ptr(workspace), workspace.numel(), _ptr(dev_status), st),
            "mxq_gather_qmm_gateup")
    return outs[0], outs[1]


def set_wait_budget(cycles: int) -> int:
    """Testing aid: the budget, in SM clock cycles, after which an on-chip
    pipeline wait of a kernel launched from now on gives up (the call's
    ``dev_status`` then gets ``DEV_TIMEOUT`` and its output is incomplete).
    ``cycles <= 0`` restores the default of 2e9 cycles.  Returns the budget in
    force.  Waits for a CTA's own copies and MMAs keep the default, so the
    next call after a timed-out one runs normally."""
    return int(lib().mxq_debug_set_wait_budget(int(cycles)))

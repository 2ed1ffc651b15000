"""Seeded synthetic inputs for the affine group-wise quantized matmul.

This module is shared by the f64 checker in ``oracle/`` and by the CUDA
library's tests and benchmark.  It creates data only: dense weights, bf16
activations, the affine 4-/8-bit encoding of those weights (the input recipe
of the workloads: scale = (max - min)/(2^bits - 1), bias = min, both stored as
bf16, codes rounded against the stored bf16 values) and sorted mixture-of-
experts routing.  It holds none of the arithmetic of the product itself
(decoding codes, dequantising, contracting): that lives, written twice and
independently, in the CUDA kernels and in the checker.

Every array is a numpy array so that both sides can consume it without
touching a GPU.  bf16 values are carried as their raw ``uint16`` bit patterns.

Storage conventions (mlxcel "affine 4-bit / group 64" weights, issue #1536
Baseline section; packing as ``integer_subbyte<4>`` in the qmm_naive kernel
name of the same page's profile table):

* codes ``w``: uint32 ``[N, K*bits/32]`` row-major; for 4-bit, word ``j`` of
  row ``n`` holds ``q[n, 8j+i]`` in bits ``4i..4i+3`` (low nibble first); for
  8-bit, byte ``i`` (little-endian) of word ``j`` holds ``q[n, 4j+i]``;
* ``scales``, ``biases``: bf16 ``[N, K/G]``, entry ``[n, g]`` covering
  ``k in [g*G, (g+1)*G)``;
* ``x``: bf16 ``[M, K]``; ``y``: bf16 ``[M, N]``.
"""

from __future__ import annotations

import numpy as np

GROUP = 64

__all__ = [
    "GROUP",
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "dense_weights",
    "activations",
    "quantize",
    "pack_codes",
    "routing",
    "QuantizedWeight",
]


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even) and
    return the 16-bit patterns.  Inputs are finite by construction."""
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(h) -> np.ndarray:
    h = np.ascontiguousarray(np.asarray(h, dtype=np.uint16))
    return (h.astype(np.uint32) << np.uint32(16)).view(np.float32)


def dense_weights(N: int, K: int, seed: int, std: float = 0.02) -> np.ndarray:
    """W ~ N(0, std^2) as float32 [N, K]."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal((N, K), dtype=np.float32) * np.float32(std)


def activations(M: int, K: int, seed: int, std: float = 1.0) -> np.ndarray:
    """x ~ N(0, std^2), rounded to bf16, returned as uint16 bits [M, K]."""
    rng = np.random.default_rng(seed)
    return f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32) * np.float32(std))


def pack_codes(q: np.ndarray, bits: int) -> np.ndarray:
    """Pack integer codes ``q[N, K]`` (values < 2^bits) into uint32 words
    ``[N, K*bits/32]`` as one little-endian bit stream per row: code k holds
    bits [k*bits, k*bits + bits), word j bits [32j, 32j + 32)."""
    q = np.asarray(q)
    N, K = q.shape
    if (K * bits) % 32:
        raise ValueError("K * bits must be a multiple of 32")
    bitplanes = (q.astype(np.uint32)[:, :, None] >> np.arange(bits, dtype=np.uint32)) & 1
    stream = bitplanes.astype(np.uint8).reshape(N, K * bits)
    packed = np.packbits(stream, axis=1, bitorder="little")
    return packed.view("<u4").astype(np.uint32).reshape(N, K * bits // 32)


class QuantizedWeight:
    """Packed codes plus bf16 scales/biases, and the raw codes for tests."""

    def __init__(self, w, scales, biases, q, bits, group):
        self.w = w            # uint32 [N, K*bits/32]
        self.scales = scales  # uint16 (bf16 bits) [N, K/group]
        self.biases = biases  # uint16 (bf16 bits) [N, K/group]
        self.q = q            # uint8 [N, K]
        self.bits = bits
        self.group = group

    @property
    def shape(self):
        return self.q.shape


def quantize(W: np.ndarray, bits: int, group: int = GROUP) -> QuantizedWeight:
    """Affine min/max encoding of dense float weights ``W[N, K]``.

    Per (row n, group g): scale = (max - min)/(2^bits - 1) and bias = min, each
    rounded to bf16; then q = clamp(round_half_even((w - bias)/scale), 0,
    2^bits - 1) computed in float64 against the *stored* bf16 scale and bias.
    A flat group (max == min) gets scale 0 and all-zero codes.
    """
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    if K % group:
        raise ValueError("K must be a multiple of the group size")
    levels = (1 << bits) - 1
    Wg = W.reshape(N, K // group, group)
    mn = Wg.min(axis=2).astype(np.float64)
    mx = Wg.max(axis=2).astype(np.float64)
    s_bits = f32_to_bf16_bits(((mx - mn) / levels).astype(np.float32))
    b_bits = f32_to_bf16_bits(mn.astype(np.float32))
    s = bf16_bits_to_f32(s_bits).astype(np.float64)[:, :, None]
    b = bf16_bits_to_f32(b_bits).astype(np.float64)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.where(s > 0, (Wg.astype(np.float64) - b) / np.where(s > 0, s, 1.0), 0.0)
    q = np.clip(np.rint(t), 0, levels).astype(np.uint8).reshape(N, K)
    return QuantizedWeight(pack_codes(q, bits), s_bits, b_bits, q, bits, group)


def routing(T: int, E: int, top_k: int, seed: int):
    """Sorted mixture-of-experts routing.

    Each token picks ``top_k`` distinct experts uniformly at random; the
    ``T*top_k`` (token, slot) rows are stably sorted by expert id.
    Returns ``expert_ids`` (int32 [B], non-decreasing) and ``row_src``
    (int32 [B], the token whose activation row feeds sorted row r).
    """
    rng = np.random.default_rng(seed)
    choice = rng.random((T, E)).argsort(axis=1, kind="stable")[:, :top_k]
    flat_e = choice.reshape(-1).astype(np.int32)
    flat_t = np.repeat(np.arange(T, dtype=np.int32), top_k)
    order = np.argsort(flat_e, kind="stable")
    return flat_e[order].copy(), flat_t[order].copy()

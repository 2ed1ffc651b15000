"""Helpers for the GPU parity tests: move synthetic inputs to the device and
compare bf16 results with the f64 checker under the acceptance rule
|y - y_ref| <= 8e-3 * sum_k |x_k * w^_kn| + 1e-3."""

from __future__ import annotations

import numpy as np

import synth

REL_TOL = 8e-3
ABS_TOL = 1e-3


def torch():
    import torch as _t

    return _t


def bf16_dev(bits_u16, device="cuda"):
    t = torch()
    a = np.ascontiguousarray(bits_u16, dtype=np.uint16).view(np.int16)
    return t.from_numpy(a.copy()).view(t.bfloat16).to(device)


def codes_dev(w_u32, device="cuda"):
    t = torch()
    a = np.ascontiguousarray(w_u32, dtype=np.uint32).view(np.int32)
    return t.from_numpy(a.copy()).to(device)


def i32_dev(a, device="cuda"):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a, dtype=np.int32).copy()).to(device)


def to_f64(y_bf16):
    """bf16 device tensor -> float64 numpy array (exact)."""
    t = torch()
    bits = y_bf16.detach().contiguous().view(t.int16).cpu().numpy().view(np.uint16)
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def assert_close(y_gpu, y_ref, bound, what=""):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    assert y_gpu.shape == y_ref.shape, (y_gpu.shape, y_ref.shape)
    assert np.all(np.isfinite(y_gpu)), "non-finite output " + what
    err = np.abs(y_gpu - y_ref)
    allow = REL_TOL * bound + ABS_TOL
    bad = err > allow
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            "%s: %d of %d outside tolerance; first %s; worst err/allow %.3g" %
            (what, int(bad.sum()), bad.size, [(tuple(i), float(y_gpu[tuple(i)]),
                                               float(y_ref[tuple(i)])) for i in idx],
             float((err / allow).max())))
    return float((err / allow).max()) if err.size else 0.0


class DenseCase:
    """Quantized dense weight + activations on host and device."""

    def __init__(self, M, K, N, bits, seed=0, x_seed=1, group=64):
        self.M, self.K, self.N, self.bits, self.group = M, K, N, bits, group
        self.qw = synth.quantize(synth.dense_weights(N, K, seed=seed), bits, group)
        self.x = synth.activations(M, K, seed=x_seed)
        self.w_d = codes_dev(self.qw.w)
        self.s_d = bf16_dev(self.qw.scales)
        self.b_d = bf16_dev(self.qw.biases)
        self.x_d = bf16_dev(self.x)


class MoECase:
    """Sorted-MoE routing + per-expert quantized weights."""

    def __init__(self, T, E, top_k, K, N, bits, seed=0, identity_src=False, routing_seed=2,
                 x_seed=1, group=64):
        self.E, self.K, self.N, self.bits, self.group = E, K, N, bits, group
        ids, src = synth.routing(T, E, top_k, seed=routing_seed)
        self.B = ids.shape[0]
        self.ids = ids
        if identity_src:
            self.src = None
            self.T = self.B
        else:
            self.src = src
            self.T = T
        ws, ss, bs = [], [], []
        for e in range(E):
            q = synth.quantize(synth.dense_weights(N, K, seed=seed * 100003 + e), bits, group)
            ws.append(q.w)
            ss.append(q.scales)
            bs.append(q.biases)
        self.w = np.stack(ws)
        self.s = np.stack(ss)
        self.b = np.stack(bs)
        self.x = synth.activations(self.T, K, seed=x_seed)
        self.w_d = codes_dev(self.w)
        self.s_d = bf16_dev(self.s)
        self.b_d = bf16_dev(self.b)
        self.x_d = bf16_dev(self.x)
        self.ids_d = i32_dev(self.ids)
        self.src_d = i32_dev(self.src) if self.src is not None else None

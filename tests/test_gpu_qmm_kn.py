"""GPU parity of the [K, N]-layout tensor-core GEMMs (mlxcel PR #1562, What
changed: the grouped GEMM is checked in both operand layouts), through the C
ABI against the f64 checker, element by element:

* mxq_qmm_kn: the prefill shape (M=600, K=5120, N=17408) whole, every width
  and group size on ragged shapes spanning several tiles (partial M tiles, K
  not a multiple of 64, K split over clusters), M = 1 against mxq_qmv_kn,
  guard bands, run-to-run determinism;
* mxq_gather_qmm_kn: small routings and both expert shapes of the sorted-MoE
  workload (E=128, top_k=8, 573 tokens) whole, against the checker applied
  per expert; invalid ids give zero rows and the status bit."""

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import assert_close, bf16_dev, codes_dev, i32_dev, to_f64

pytestmark = pytest.mark.gpu


def _mxq():
    import affine_bit_matmul_gb300 as mxq

    return mxq


def _kn_weights(K, N, bits, group, seed):
    # synth.quantize groups along the last axis: quantizing the [K, N] matrix
    # gives codes and groups along n
    qw = synth.quantize(synth.dense_weights(K, N, seed=seed), bits, group)
    return qw.w, qw.scales, qw.biases


class KnGemm:
    def __init__(self, M, K, N, bits, group=64, seed=0, x_seed=1):
        self.M, self.K, self.N, self.bits, self.group = M, K, N, bits, group
        self.w, self.s, self.b = _kn_weights(K, N, bits, group, seed)
        self.x = synth.activations(M, K, seed=x_seed)
        self.w_d, self.s_d, self.b_d = codes_dev(self.w), bf16_dev(self.s), bf16_dev(self.b)
        self.x_d = bf16_dev(self.x)

    def run(self, **kw):
        return _mxq().qmm_kn(self.x_d, self.w_d, self.s_d, self.b_d, self.bits,
                             group_size=self.group, **kw)

    def ref(self):
        return oracle.qmm_kn(self.x, self.w, self.s, self.b, self.M, self.K, self.N, self.bits,
                             self.group)


def test_qmm_kn_prefill_full_size():
    import torch

    c = KnGemm(600, 5120, 17408, 4, seed=11, x_seed=12)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    y = c.run(dev_status=status)
    yr, bnd = c.ref()
    assert_close(to_f64(y), yr, bnd, "qmm_kn prefill")
    assert int(status.item()) == 0
    y2 = c.run()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("bits", [2, 8])
def test_qmm_kn_wide_other_widths(bits):
    c = KnGemm(128, 5120, 17408, bits, seed=13 + bits, x_seed=14)
    yr, bnd = c.ref()
    assert_close(to_f64(c.run()), yr, bnd, "qmm_kn M=128 bits=%d" % bits)


@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("M,K,N", [
    (2, 64, 128), (16, 4096, 256), (33, 200, 640), (130, 1000, 384), (257, 5120, 1280),
    (64, 8, 64), (600, 704, 2816), (320, 1024, 512),
])
def test_qmm_kn_shapes(bits, group, M, K, N):
    if N % group:
        pytest.skip("N is not a multiple of the group size")
    c = KnGemm(M, K, N, bits, group=group, seed=M + K + N + bits, x_seed=M + 3)
    yr, bnd = c.ref()
    assert_close(to_f64(c.run()), yr, bnd, "qmm_kn M=%d K=%d N=%d bits=%d G=%d" %
                 (M, K, N, bits, group))


def test_qmm_kn_single_row_is_the_gemv():
    import torch

    c = KnGemm(1, 5120, 4096, 4, seed=3)
    y = c.run()
    y1 = _mxq().qmv_kn(c.x_d[0], c.w_d, c.s_d, c.b_d, 4)
    assert torch.equal(y[0].view(torch.int16), y1.view(torch.int16))
    yr, bnd = c.ref()
    assert_close(to_f64(y), yr, bnd, "qmm_kn M=1")


def test_qmm_kn_one_hot_rows():
    # x row m = e_{k_m} selects row k_m of the dequantised matrix, every column
    K, N = 640, 512
    ks = [0, 1, 7, 8, 63, 64, 65, 127, 128, 300, 511, 639]
    c = KnGemm(len(ks), K, N, 4, seed=21)
    x = np.zeros((len(ks), K), np.uint16)
    for m, k in enumerate(ks):
        x[m, k] = 0x3F80  # bf16 1.0
    c.x = x
    c.x_d = bf16_dev(x)
    yr, bnd = c.ref()
    assert_close(to_f64(c.run()), yr, bnd, "qmm_kn one-hot rows")


def test_qmm_kn_guard_bands():
    import torch

    c = KnGemm(40, 1024, 384, 4, seed=5)
    guard = 4096
    buf = torch.full((guard + 40 * 384 + guard,), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    out = buf[guard:guard + 40 * 384].view(40, 384)
    c.run(out=out)
    torch.cuda.synchronize()
    assert torch.isnan(buf[:guard]).all() and torch.isnan(buf[guard + 40 * 384:]).all()
    yr, bnd = c.ref()
    assert_close(to_f64(out), yr, bnd, "qmm_kn guarded")


# ---------------------------------------------------------------- grouped form


class KnMoE:
    def __init__(self, T, E, top_k, K, N, bits, group=64, seed=0, identity_src=False,
                 routing_seed=2, x_seed=1):
        self.E, self.K, self.N, self.bits, self.group = E, K, N, bits, group
        ids, src = synth.routing(T, E, top_k, seed=routing_seed)
        self.ids = ids
        self.B = ids.shape[0]
        if identity_src:
            self.src, self.T = None, self.B
        else:
            self.src, self.T = src, T
        ws, ss, bs = [], [], []
        for e in range(E):
            w, s, b = _kn_weights(K, N, bits, group, seed * 100003 + e)
            ws.append(w)
            ss.append(s)
            bs.append(b)
        self.w, self.s, self.b = np.stack(ws), np.stack(ss), np.stack(bs)
        self.x = synth.activations(self.T, K, seed=x_seed)
        self.w_d, self.s_d, self.b_d = codes_dev(self.w), bf16_dev(self.s), bf16_dev(self.b)
        self.x_d = bf16_dev(self.x)
        self.ids_d = i32_dev(self.ids)
        self.src_d = i32_dev(self.src) if self.src is not None else None

    def run(self, ids_d=None, **kw):
        return _mxq().gather_qmm_kn(self.x_d, self.w_d, self.s_d, self.b_d,
                                    self.ids_d if ids_d is None else ids_d, self.src_d,
                                    self.bits, group_size=self.group, **kw)

    def ref(self, ids=None):
        """The checker's dense [K, N] GEMM of each expert over its rows; rows
        with an id outside [0, E) are zero."""
        ids = self.ids if ids is None else ids
        y = np.zeros((self.B, self.N))
        bnd = np.zeros((self.B, self.N))
        src = np.arange(self.B) if self.src is None else self.src
        for e in np.unique(ids):
            if not 0 <= e < self.E:
                continue
            rows = np.nonzero(ids == e)[0]
            ye, be = oracle.qmm_kn(self.x[src[rows]], self.w[e], self.s[e], self.b[e], len(rows),
                                   self.K, self.N, self.bits, self.group)
            y[rows] = ye
            bnd[rows] = be
        return y, bnd


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("T,E,top_k,K,N,ident", [
    (9, 4, 2, 128, 128, False), (40, 8, 3, 704, 256, False), (33, 16, 4, 256, 192, True),
    (300, 6, 2, 200, 256, False), (5, 3, 3, 64, 64, True),
])
def test_gather_kn_small(bits, T, E, top_k, K, N, ident):
    import torch

    c = KnMoE(T, E, top_k, K, N, bits, seed=T + E, identity_src=ident)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    y = c.run(dev_status=status)
    yr, bnd = c.ref()
    assert_close(to_f64(y), yr, bnd, "gather_kn T=%d E=%d bits=%d" % (T, E, bits))
    assert int(status.item()) == 0


@pytest.mark.parametrize("K,N,ident", [(2816, 704, False), (704, 2816, True)])
def test_gather_kn_workload_shapes(K, N, ident):
    # the sorted-MoE workload (573 tokens, top 8 of 128 experts), whole output
    c = KnMoE(573, 128, 8, K, N, 4, seed=1, identity_src=ident)
    yr, bnd = c.ref()
    assert_close(to_f64(c.run()), yr, bnd, "gather_kn K=%d N=%d" % (K, N))


@pytest.mark.parametrize("group", [32, 128])
def test_gather_kn_group_sizes(group):
    c = KnMoE(64, 8, 4, 512, 256, 4, group=group, seed=9)
    yr, bnd = c.ref()
    assert_close(to_f64(c.run()), yr, bnd, "gather_kn G=%d" % group)


def test_gather_kn_out_of_range_ids_zeroed_and_reported():
    import torch

    mxq = _mxq()
    c = KnMoE(40, 8, 2, 256, 128, 4, seed=4)
    ids = c.ids.copy()
    ids[-3:] = 8   # past the last expert (still non-decreasing)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = c.run(ids_d=i32_dev(ids), dev_status=status)
    assert int(status.item()) & mxq.DEV_BAD_EXPERT_ID
    yr, bnd = c.ref(ids)
    assert_close(to_f64(y), yr, bnd, "gather_kn invalid ids")
    assert not to_f64(y)[-3:].any()

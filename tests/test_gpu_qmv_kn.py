"""GPU parity of mxq_qmv_kn, the decode GEMV for the [K, N] operand layout
(codes and groups along n; mlxcel PR #1562, What changed: both operand
layouts), through the C ABI against the f64 checker: the decode shapes in
full, ragged K and small N (cluster sizes from 1 to 8), every supported
width and group size, one-hot rows, and run-to-run determinism."""

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import assert_close, bf16_dev, codes_dev, to_f64

pytestmark = pytest.mark.gpu


def _mxq():
    import affine_bit_matmul_gb300 as mxq

    return mxq


class KnCase:
    """W [K, N] quantized along n (per row k, groups of G columns)."""

    def __init__(self, K, N, bits, group=64, seed=0, x_seed=1):
        self.K, self.N, self.bits, self.group = K, N, bits, group
        # quantize W^T's rows: synth.quantize groups along the last axis, so
        # quantizing the [K, N] matrix directly gives codes and scales along n
        qw = synth.quantize(synth.dense_weights(K, N, seed=seed), bits, group)
        self.w, self.s, self.b = qw.w, qw.scales, qw.biases
        self.x = synth.activations(1, K, seed=x_seed)
        self.w_d = codes_dev(self.w)
        self.s_d = bf16_dev(self.s)
        self.b_d = bf16_dev(self.b)
        self.x_d = bf16_dev(self.x)[0]

    def ref(self):
        y, bnd = oracle.qmm_kn(self.x, self.w, self.s, self.b, 1, self.K, self.N, self.bits,
                               self.group)
        return y[0], bnd[0]

    def run(self, **kw):
        return _mxq().qmv_kn(self.x_d, self.w_d, self.s_d, self.b_d, self.bits,
                             group_size=self.group, **kw)


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("K,N", [(5120, 17408), (17408, 5120)])
def test_qmv_kn_decode_shapes(bits, K, N):
    import torch

    c = KnCase(K, N, bits, seed=K + bits)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    y = c.run(dev_status=status)
    yr, bnd = c.ref()
    assert_close(to_f64(y), yr, bnd, "qmv_kn K=%d N=%d bits=%d" % (K, N, bits))
    assert int(status.item()) == 0
    y2 = c.run()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("K,N", [(1, 128), (7, 256), (33, 64), (100, 640), (1000, 384),
                                 (4097, 1280)])
def test_qmv_kn_ragged(bits, group, K, N):
    if N % group:
        pytest.skip("N is not a multiple of the group size")
    c = KnCase(K, N, bits, group=group, seed=K * 3 + N + bits, x_seed=K + 2)
    y = c.run()
    yr, bnd = c.ref()
    assert_close(to_f64(y), yr, bnd, "qmv_kn K=%d N=%d bits=%d G=%d" % (K, N, bits, group))


def test_qmv_kn_one_hot_rows():
    # x = e_k picks row k of the dequantised matrix: every column of that row
    K, N = 300, 512
    c = KnCase(K, N, 4, seed=5)
    mxq = _mxq()
    for k in (0, 1, 31, 32, 33, 150, 299):
        x = np.zeros((1, K), np.float32)
        x[0, k] = 1.0
        xb = synth.f32_to_bf16_bits(x)
        y = mxq.qmv_kn(bf16_dev(xb)[0], c.w_d, c.s_d, c.b_d, 4)
        yr, _ = oracle.qmm_kn(xb, c.w, c.s, c.b, 1, K, N, 4)
        assert_close(to_f64(y), yr[0], np.abs(yr[0]), "one-hot row %d" % k)

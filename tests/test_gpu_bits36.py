"""GPU parity of 3- and 6-bit codes (one little-endian bit stream per row,
code k in bits [k*b, k*b + b), so codes straddle words; the bit width is a
parameter of the kernels in issue #1536, Diagnosis item 3) for every entry
point, through the C ABI, against the f64 checker: the direct-load GEMV,
the split-K and persistent tensor-core GEMMs (stages that cross the 128-byte
copy boxes), the grouped GEMM (one CTA per tile and the decode form), and
the encoder bit for bit."""

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import DenseCase, MoECase, assert_close, bf16_dev, to_f64

pytestmark = pytest.mark.gpu


def _mxq():
    import affine_bit_matmul_gb300 as mxq

    return mxq


def _ref_dense(c):
    return oracle.qmm(c.x, c.qw.w, c.qw.scales, c.qw.biases, c.M, c.K, c.N, c.bits, c.group)


@pytest.mark.parametrize("bits", [3, 6])
@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("K,N", [(5120, 1000), (17408, 96), (640, 257), (128, 33)])
def test_qmv_3_6_bit(bits, group, K, N):
    if K % group or (bits == 3 and K % 128):
        pytest.skip("K does not fit the group size or the 3-bit row rule")
    c = DenseCase(1, K, N, bits, seed=K + N + group + bits, x_seed=7, group=group)
    y = _mxq().qmv(c.x_d[0], c.w_d, c.s_d, c.b_d, bits, group_size=group)
    yr, bnd = _ref_dense(c)
    assert_close(to_f64(y), yr[0], bnd[0], "qmv %d-bit K=%d N=%d G=%d" % (bits, K, N, group))


@pytest.mark.parametrize("bits", [3, 6])
def test_qmv_3_6_bit_decode_shape(bits):
    import torch

    c = DenseCase(1, 5120, 17408, bits, seed=0, x_seed=1)
    mxq = _mxq()
    y = mxq.qmv(c.x_d[0], c.w_d, c.s_d, c.b_d, bits)
    yr, bnd = _ref_dense(c)
    assert_close(to_f64(y), yr[0], bnd[0], "qmv %d-bit decode" % bits)
    y2 = mxq.qmv(c.x_d[0], c.w_d, c.s_d, c.b_d, bits)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("bits", [3, 6])
@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("M,K,N", [
    (1, 128, 128),      # one stage; codes past the row end are never read
    (5, 704, 130),      # 6-bit only (704 % 128 != 0): K / 64 odd, a half stage
    (7, 2304, 256),     # K split over a cluster (3-bit: an even number of 64-blocks per split)
    (129, 1152, 257),   # one CTA per tile, several code slots
    (300, 640, 19456),  # persistent, 3-bit skipped (640 % 128 != 0)
    (100, 1280, 19456), # persistent
])
def test_qmm_3_6_bit(bits, group, M, K, N):
    if K % group or (bits == 3 and K % 128):
        pytest.skip("K does not fit the group size or the 3-bit row rule")
    c = DenseCase(M, K, N, bits, seed=M + K + N + group + bits, x_seed=M + 3, group=group)
    y = _mxq().qmm(c.x_d, c.w_d, c.s_d, c.b_d, bits, group_size=group)
    yr, bnd = _ref_dense(c)
    assert_close(to_f64(y), yr, bnd, "qmm %d-bit M=%d K=%d N=%d G=%d" % (bits, M, K, N, group))


@pytest.mark.parametrize("bits", [3, 6])
def test_qmm_3_6_bit_one_hot(bits):
    # x = e_k picks single weights: codes that straddle words (3-bit codes
    # 10, 21, 42, ...; 6-bit codes 5, 10, 21, ...) and stages that cross the
    # copy boxes, on the tensor path
    K, N = 768, 128
    ks = sorted({0, 1, 5, 10, 11, 21, 22, 31, 32, 42, 63, 64, 85, 127, 128, 170, 191, 255, 256,
                 383, 384, 511, 512, 639, 767})
    c = DenseCase(len(ks), K, N, bits, seed=17)
    x = np.zeros((len(ks), K), np.float32)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    y = _mxq().qmm(bf16_dev(synth.f32_to_bf16_bits(x)), c.w_d, c.s_d, c.b_d, bits)
    wh = oracle.dequant(c.qw.w, c.qw.scales, c.qw.biases, N, K, bits)
    want = np.stack([wh[:, k] for k in ks])
    assert_close(to_f64(y), want, np.abs(want), "one-hot %d-bit" % bits)


@pytest.mark.parametrize("bits", [3, 6])
def test_qmm_3_6_bit_prefill_sampled(bits):
    c = DenseCase(600, 5120, 17408, bits, seed=0, x_seed=1)
    y = _mxq().qmm(c.x_d, c.w_d, c.s_d, c.b_d, bits)
    rng = np.random.default_rng(bits)
    rows = np.concatenate([rng.integers(0, 600, 3000), [0, 599]]).astype(np.int64)
    cols = np.concatenate([rng.integers(0, 17408, 3000), [17407, 0]]).astype(np.int64)
    yr, bnd = oracle.points(c.x, c.qw.w, c.qw.scales, c.qw.biases, rows, cols, 5120, 17408, bits)
    assert_close(to_f64(y)[rows, cols], yr, bnd, "prefill %d-bit sample" % bits)


@pytest.mark.parametrize("bits", [3, 6])
@pytest.mark.parametrize("T,E,top_k,K,N,ident", [
    (40, 8, 3, 768, 200, False),   # one CTA per tile (B = 120)
    (300, 6, 2, 256, 256, True),
    (3, 16, 8, 1024, 136, False),  # decode form (B = 24)
])
def test_gather_3_6_bit(bits, T, E, top_k, K, N, ident):
    import torch

    c = MoECase(T, E, top_k, K, N, bits, seed=T + E + bits, identity_src=ident,
                routing_seed=T + 5)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    y = _mxq().gather_qmm(c.x_d, c.w_d, c.s_d, c.b_d, c.ids_d, c.src_d, bits, dev_status=status)
    yr, bnd = oracle.gather_qmm(c.x, c.w, c.s, c.b, c.ids, c.src, c.T, c.B, c.E, c.K, c.N, bits)
    assert_close(to_f64(y), yr, bnd, "gather %d-bit T=%d K=%d N=%d" % (bits, T, K, N))
    assert int(status.item()) == 0


@pytest.mark.parametrize("bits", [3, 6])
@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("N,K", [(37, 256), (129, 5120), (3, 20480)])
def test_quantize_3_6_bit_bit_exact(bits, group, N, K):
    import torch

    rng = np.random.default_rng(N + K + group + bits)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    W[0, :group] = 0.75                       # a flat group
    W[1, group:2 * group] = -0.0              # a group of negative zeros
    codes, s, b = _mxq().quantize(torch.from_numpy(W).cuda(), bits, group_size=group)
    torch.cuda.synchronize()
    co, so, bo = oracle.quantize(W, bits, group)
    assert codes.shape == (N, K * bits // 32)
    assert np.array_equal(s.view(torch.int16).cpu().numpy().view(np.uint16), so)
    assert np.array_equal(b.view(torch.int16).cpu().numpy().view(np.uint16), bo)
    assert np.array_equal(codes.cpu().numpy().view(np.uint32), co)

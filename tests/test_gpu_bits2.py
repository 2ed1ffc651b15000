"""GPU parity of 2-bit codes (sixteen per little-endian word, lowest k in the
lowest two bits; the bit width is a parameter of the kernels in issue #1536,
Diagnosis item 3) for every entry point, through the C ABI, against the f64
checker: the streaming and direct-load GEMVs, the split-K and persistent
tensor-core GEMMs, the grouped GEMM (persistent and decode forms), and the
encoder bit for bit."""

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
    return oracle.qmm(c.x, c.qw.w, c.qw.scales, c.qw.biases, c.M, c.K, c.N, 2, c.group)


@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("K,N", [
    (5120, 1000),   # streaming kernel
    (17408, 200),   # streaming kernel, long K
    (640, 257),     # direct-load kernel (K % 512 != 0)
    (64, 33),       # one group row, direct-load kernel
])
def test_qmv_2bit(group, K, N):
    if K % group:
        pytest.skip("K is not a multiple of the group size")
    c = DenseCase(1, K, N, 2, seed=K + N + group, x_seed=4, group=group)
    y = _mxq().qmv(c.x_d[0], c.w_d, c.s_d, c.b_d, 2, group_size=group)
    yr, bnd = _ref_dense(c)
    assert_close(to_f64(y), yr[0], bnd[0], "qmv 2-bit K=%d N=%d G=%d" % (K, N, group))


def test_qmv_2bit_decode_shape_and_determinism():
    import torch

    c = DenseCase(1, 5120, 17408, 2, seed=0, x_seed=1)
    mxq = _mxq()
    y = mxq.qmv(c.x_d[0], c.w_d, c.s_d, c.b_d, 2)
    yr, bnd = _ref_dense(c)
    assert_close(to_f64(y), yr[0], bnd[0], "qmv 2-bit decode")
    y2 = mxq.qmv(c.x_d[0], c.w_d, c.s_d, c.b_d, 2)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("M,K,N", [
    (1, 64, 128),       # one 64-block: a half-used stage, one code box past K
    (7, 2304, 256),     # split K over a cluster
    (129, 704, 257),    # one CTA per tile, K / 64 odd
    (300, 640, 19456),  # persistent
    (100, 1152, 19456), # persistent, two tiles per CTA in flight
])
def test_qmm_2bit(group, M, K, N):
    if K % group:
        pytest.skip("K is not a multiple of the group size")
    c = DenseCase(M, K, N, 2, seed=M + K + N + group, x_seed=M + 5, group=group)
    y = _mxq().qmm(c.x_d, c.w_d, c.s_d, c.b_d, 2, group_size=group)
    yr, bnd = _ref_dense(c)
    assert_close(to_f64(y), yr, bnd, "qmm 2-bit M=%d K=%d N=%d G=%d" % (M, K, N, group))


def test_qmm_2bit_one_hot():
    # x = e_k picks single weights: the order of the sixteen codes in a word
    # and of the words along k, on the tensor path
    K, N = 512, 128
    ks = [0, 1, 2, 3, 4, 7, 8, 15, 16, 17, 31, 32, 63, 64, 127, 128, 255, 256, 511]
    c = DenseCase(len(ks), K, N, 2, seed=13)
    x = np.zeros((len(ks), K), np.float32)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    y = _mxq().qmm(bf16_dev(synth.f32_to_bf16_bits(x)), c.w_d, c.s_d, c.b_d, 2)
    wh = oracle.dequant(c.qw.w, c.qw.scales, c.qw.biases, N, K, 2)
    want = np.stack([wh[:, k] for k in ks])
    assert_close(to_f64(y), want, np.abs(want), "one-hot 2-bit")


def test_qmm_2bit_prefill_sampled():
    c = DenseCase(600, 5120, 17408, 2, seed=0, x_seed=1)
    y = _mxq().qmm(c.x_d, c.w_d, c.s_d, c.b_d, 2)
    rng = np.random.default_rng(2)
    rows = np.concatenate([rng.integers(0, 600, 3000), [0, 599]]).astype(np.int64)
    cols = np.concatenate([rng.integers(0, 17408, 3000), [17407, 0]]).astype(np.int64)
    yr, bnd = oracle.points(c.x, c.qw.w, c.qw.scales, c.qw.biases, rows, cols, 5120, 17408, 2)
    assert_close(to_f64(y)[rows, cols], yr, bnd, "prefill 2-bit sample")


@pytest.mark.parametrize("group", [32, 64])
@pytest.mark.parametrize("T,E,top_k,K,N,ident", [
    (40, 8, 3, 768, 200, False),   # persistent grouped GEMM (B = 120)
    (300, 6, 2, 256, 256, True),
    (3, 16, 8, 1024, 136, False),  # decode form (B = 24)
])
def test_gather_2bit(group, T, E, top_k, K, N, ident):
    import torch

    c = MoECase(T, E, top_k, K, N, 2, seed=T + E + group, identity_src=ident,
                routing_seed=T + 3, group=group)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    y = _mxq().gather_qmm(c.x_d, c.w_d, c.s_d, c.b_d, c.ids_d, c.src_d, 2, dev_status=status,
                          group_size=group)
    yr, bnd = oracle.gather_qmm(c.x, c.w, c.s, c.b, c.ids, c.src, c.T, c.B, c.E, c.K, c.N, 2,
                                group)
    assert_close(to_f64(y), yr, bnd, "gather 2-bit T=%d K=%d N=%d G=%d" % (T, K, N, group))
    assert int(status.item()) == 0


def test_gather_2bit_workload_sampled():
    c = MoECase(573, 128, 8, 704, 2816, 2, seed=0, identity_src=True)
    y = to_f64(_mxq().gather_qmm(c.x_d, c.w_d, c.s_d, c.b_d, c.ids_d, c.src_d, 2))
    rng = np.random.default_rng(4)
    rows = rng.integers(0, c.B, 3000).astype(np.int64)
    cols = rng.integers(0, c.N, 3000).astype(np.int64)
    yr, bnd = oracle.points(c.x, c.w, c.s, c.b, rows, cols, c.K, c.N, 2, expert_ids=c.ids,
                            row_src=c.src, E=c.E)
    assert_close(y[rows, cols], yr, bnd, "gather 2-bit workload")


@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("N,K", [(37, 256), (129, 5120), (3, 20480)])
def test_quantize_2bit_bit_exact(group, N, K):
    import torch

    rng = np.random.default_rng(N + K + group)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    W[0, :group] = -1.5                      # a flat group
    W[1, :group] = np.tile([0.0, 1.0, 2.0, 3.0], group // 4)   # exact steps with ties absent
    codes, s, b = _mxq().quantize(torch.from_numpy(W).cuda(), 2, group_size=group)
    torch.cuda.synchronize()
    co, so, bo = oracle.quantize(W, 2, group)
    assert codes.shape == (N, K // 16)
    assert np.array_equal(s.view(torch.int16).cpu().numpy().view(np.uint16), so)
    assert np.array_equal(b.view(torch.int16).cpu().numpy().view(np.uint16), bo)
    assert np.array_equal(codes.cpu().numpy().view(np.uint32), co)

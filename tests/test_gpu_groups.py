"""GPU parity at group sizes 32 and 128 (one scale/bias pair per 32 or 128
consecutive k; issue #1536, Diagnosis item 4 treats the group size as a
parameter of the stored format) for every entry point, through the C ABI,
against the f64 checker: the streaming and direct-load GEMVs, the split-K
and persistent tensor-core GEMMs, the grouped GEMM in all three of its forms
(persistent 4-bit, one CTA per tile 8-bit, per-row decode), the encoder bit
for bit, and the argument checks that go with the group size."""

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import DenseCase, MoECase, assert_close, bf16_dev, to_f64

pytestmark = pytest.mark.gpu

GROUPS = [32, 128]


def _mxq():
    import affine_bit_matmul_gb300 as mxq

    return mxq


def _ref_dense(c):
    return oracle.qmm(c.x, c.qw.w, c.qw.scales, c.qw.biases, c.M, c.K, c.N, c.bits, c.group)


# ---------------------------------------------------------------- qmv


@pytest.mark.parametrize("group", GROUPS)
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("K,N", [
    (5120, 1000),   # streaming kernel (K % 512 == 0, K / G a multiple of 8)
    (1536, 300),    # K / 128 = 12: the direct-load kernel at G = 128
    (640, 257),     # K % 512 != 0: direct-load kernel
    (17408, 96),    # the long-K decode orientation
])
def test_qmv_group_sizes(bits, group, K, N):
    c = DenseCase(1, K, N, bits, seed=K + N + group, x_seed=3, group=group)
    y = _mxq().qmv(c.x_d[0], c.w_d, c.s_d, c.b_d, bits, group_size=group)
    yr, bnd = _ref_dense(c)
    assert_close(to_f64(y), yr[0], bnd[0], "qmv K=%d N=%d bits=%d G=%d" % (K, N, bits, group))


@pytest.mark.parametrize("group", GROUPS)
def test_qmv_group_sizes_decode_shape(group):
    # the decode projection K=5120 N=17408 at 4 bits, whole output
    c = DenseCase(1, 5120, 17408, 4, seed=1, x_seed=2, group=group)
    y = _mxq().qmv(c.x_d[0], c.w_d, c.s_d, c.b_d, 4, group_size=group)
    yr, bnd = _ref_dense(c)
    assert_close(to_f64(y), yr[0], bnd[0], "qmv decode G=%d" % group)


# ---------------------------------------------------------------- qmm


@pytest.mark.parametrize("group", GROUPS)
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M,K,N", [
    (7, 2304, 256),     # K split over a cluster in 9-block parts: not on 128-group edges
    (129, 704, 257),    # one CTA per tile; K / 64 odd (G = 32 only: 704 % 128 != 0)
    (300, 640, 19456),  # persistent, ragged M and a partly used last code slot
    (100, 1152, 19456), # persistent, one accumulator buffer per tile
])
def test_qmm_group_sizes(bits, group, M, K, N):
    if K % group:
        pytest.skip("K is not a multiple of the group size")
    c = DenseCase(M, K, N, bits, seed=M + K + N + group, x_seed=M + 2, group=group)
    y = _mxq().qmm(c.x_d, c.w_d, c.s_d, c.b_d, bits, group_size=group)
    yr, bnd = _ref_dense(c)
    assert_close(to_f64(y), yr, bnd, "qmm M=%d K=%d N=%d bits=%d G=%d" % (M, K, N, bits, group))


@pytest.mark.parametrize("group", GROUPS)
def test_qmm_group_sizes_one_hot(group):
    # x = e_k picks single dequantised weights on the tensor path: the group
    # index at every group edge of both sizes
    K, N = 512, 128
    ks = sorted({0, 1, 31, 32, 33, 63, 64, 95, 96, 127, 128, 129, 255, 256, 383, 384, 511})
    c = DenseCase(len(ks), K, N, 4, seed=9, group=group)
    x = np.zeros((len(ks), K), np.float32)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    y = _mxq().qmm(bf16_dev(synth.f32_to_bf16_bits(x)), c.w_d, c.s_d, c.b_d, 4, group_size=group)
    wh = oracle.dequant(c.qw.w, c.qw.scales, c.qw.biases, N, K, 4, group)
    want = np.stack([wh[:, k] for k in ks])
    assert_close(to_f64(y), want, np.abs(want), "one-hot G=%d" % group)


@pytest.mark.parametrize("group", GROUPS)
def test_qmm_group_sizes_prefill_sampled(group):
    # the prefill shape M=600 K=5120 N=17408 (persistent), sampled outputs
    c = DenseCase(600, 5120, 17408, 4, seed=0, x_seed=1, group=group)
    y = _mxq().qmm(c.x_d, c.w_d, c.s_d, c.b_d, 4, group_size=group)
    rng = np.random.default_rng(group)
    rows = np.concatenate([rng.integers(0, 600, 3000), [0, 599]]).astype(np.int64)
    cols = np.concatenate([rng.integers(0, 17408, 3000), [17407, 0]]).astype(np.int64)
    yr, bnd = oracle.points(c.x, c.qw.w, c.qw.scales, c.qw.biases, rows, cols, 5120, 17408, 4,
                            group)
    assert_close(to_f64(y)[rows, cols], yr, bnd, "prefill sample G=%d" % group)


# ---------------------------------------------------------------- gather


def _gather(c):
    return _mxq().gather_qmm(c.x_d, c.w_d, c.s_d, c.b_d, c.ids_d, c.src_d, c.bits,
                             group_size=c.group)


def _gather_ref(c):
    return oracle.gather_qmm(c.x, c.w, c.s, c.b, c.ids, c.src, c.T, c.B, c.E, c.K, c.N, c.bits,
                             c.group)


@pytest.mark.parametrize("group", GROUPS)
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("T,E,top_k,K,N,ident", [
    (40, 8, 3, 768, 200, False),   # tensor-core forms (B = 120 rows)
    (300, 6, 2, 256, 256, True),
    (3, 16, 8, 1024, 136, False),  # decode form (B = 24 rows)
])
def test_gather_group_sizes(bits, group, T, E, top_k, K, N, ident):
    import torch

    c = MoECase(T, E, top_k, K, N, bits, seed=T + E + group, identity_src=ident,
                routing_seed=T + 1, group=group)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    y = _mxq().gather_qmm(c.x_d, c.w_d, c.s_d, c.b_d, c.ids_d, c.src_d, bits, dev_status=status,
                          group_size=group)
    yr, bnd = _gather_ref(c)
    assert_close(to_f64(y), yr, bnd, "gather T=%d K=%d N=%d bits=%d G=%d" %
                 (T, K, N, bits, group))
    assert int(status.item()) == 0


@pytest.mark.parametrize("group", GROUPS)
def test_gather_group_sizes_workload_sampled(group):
    # the up-projection expert shape K=2816 N=704 (E=128, top_k=8, 573
    # tokens), sampled; 2816 = 22 * 128
    c = MoECase(573, 128, 8, 2816, 704, 4, seed=0, group=group)
    y = to_f64(_gather(c))
    rng = np.random.default_rng(3)
    rows = rng.integers(0, c.B, 3000).astype(np.int64)
    cols = rng.integers(0, c.N, 3000).astype(np.int64)
    yr, bnd = oracle.points(c.x, c.w, c.s, c.b, rows, cols, c.K, c.N, 4, group,
                            expert_ids=c.ids, row_src=c.src, E=c.E)
    assert_close(y[rows, cols], yr, bnd, "gather workload G=%d" % group)


def test_gather_noalloc_group_32():
    import torch

    c = MoECase(40, 8, 3, 768, 200, 4, seed=5, group=32)
    out = torch.empty((c.B, c.N), dtype=torch.bfloat16, device="cuda")
    _mxq().gather_qmm_noalloc(c.x_d, c.w_d, c.s_d, c.b_d, c.ids_d, c.src_d, 4, out,
                              group_size=32)
    yr, bnd = _gather_ref(c)
    assert_close(to_f64(out), yr, bnd, "gather noalloc G=32")


# ---------------------------------------------------------------- encoder


@pytest.mark.parametrize("group", GROUPS)
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("N,K", [(37, 256), (129, 5120), (5, 20480)])
def test_quantize_group_sizes_bit_exact(bits, group, N, K):
    import torch

    rng = np.random.default_rng(N + K + group + bits)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    W[0, :group] = 0.25                       # a flat group
    W[1, group:2 * group] = -0.0              # a group of negative zeros
    codes, s, b = _mxq().quantize(torch.from_numpy(W).cuda(), bits, group_size=group)
    torch.cuda.synchronize()
    co, so, bo = oracle.quantize(W, bits, group)
    assert tuple(s.shape) == (N, K // group)
    assert np.array_equal(s.view(torch.int16).cpu().numpy().view(np.uint16), so)
    assert np.array_equal(b.view(torch.int16).cpu().numpy().view(np.uint16), bo)
    assert np.array_equal(codes.cpu().numpy().view(np.uint32), co)


# ---------------------------------------------------------------- arguments


def test_group_size_argument_checks():
    import torch

    mxq = _mxq()
    c = DenseCase(1, 192, 64, 4, seed=1, group=32)
    # K = 192 is not a multiple of 128: refused before any launch
    s128 = torch.zeros((64, 1), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mxq.MxqError) as ei:
        mxq.qmv(c.x_d[0], c.w_d, s128, s128, 4, group_size=128)
    assert ei.value.status == 1
    for g in (16, 48, 96, 256):
        sg = torch.zeros((64, max(1, 192 // g)), dtype=torch.bfloat16, device="cuda")
        with pytest.raises((mxq.MxqError, ValueError)):
            mxq.qmv(c.x_d[0], c.w_d, sg, sg, 4, group_size=g)

"""GPU parity of mxq_qmm (tcgen05 prefill GEMM) against the f64 checker,
through the C ABI, element by element: shapes that span several tiles with
ragged M and N tails, the M sweep at K=N=5120 and the full prefill workload
(M=600, K=5120, N=17408), with repeated launches compared bit for bit."""

import numpy as np
import pytest

import oracle
from tests.gpu_util import DenseCase, assert_close, to_f64

pytestmark = pytest.mark.gpu


def _mxq():
    import affine_bit_matmul_gb300 as mxq

    return mxq


def _full_ref(case):
    return oracle.qmm(case.x, case.qw.w, case.qw.scales, case.qw.biases, case.M, case.K, case.N,
                      case.bits)


def _sample(case, y, count=3000, seed=0):
    rng = np.random.default_rng(seed)
    rows = rng.integers(0, case.M, size=count)
    cols = rng.integers(0, case.N, size=count)
    # always include the corners and the last row/col
    rows = np.concatenate([rows, [0, case.M - 1, 0, case.M - 1]]).astype(np.int64)
    cols = np.concatenate([cols, [0, case.N - 1, case.N - 1, 0]]).astype(np.int64)
    yr, bnd = oracle.points(case.x, case.qw.w, case.qw.scales, case.qw.biases, rows, cols,
                            case.K, case.N, case.bits)
    yg = to_f64(y)[rows, cols]
    return yg, yr, bnd


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M,K,N", [
    # enough tiles of <= 256 rows to fill the GPU: the persistent kernel, with
    # ragged K (a partly used last code slot; an odd number of 64-blocks),
    # ragged M and N, one or two accumulator buffers (tiles above / up to
    # 128 rows) and tiles per CTA that differ
    (300, 640, 19456), (333, 192, 19500), (129, 320, 19456), (1000, 64, 9800),
    (100, 704, 19456),
])
def test_qmm_persistent_shapes(bits, M, K, N):
    test_qmm_small(bits, M, K, N)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M,K,N", [
    (1, 64, 128), (7, 128, 128), (9, 704, 200), (16, 512, 256), (33, 1024, 130),
    (127, 704, 384), (129, 640, 257), (256, 256, 128), (257, 320, 100), (600, 704, 136),
])
def test_qmm_small(bits, M, K, N):
    case = DenseCase(M, K, N, bits, seed=M * 7 + K + N, x_seed=M + 1)
    y = _mxq().qmm(case.x_d, case.w_d, case.s_d, case.b_d, bits)
    yr, bnd = _full_ref(case)
    assert_close(to_f64(y), yr, bnd, "qmm M=%d K=%d N=%d bits=%d" % (M, K, N, bits))


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M", [1, 8, 32])
def test_qmm_sweep_small_m_full(bits, M):
    # the M sweep at K = N = 5120; small M splits K over a thread-block
    # cluster and adds the partials through distributed shared memory
    import torch

    case = DenseCase(M, 5120, 5120, bits, seed=0, x_seed=1)
    mxq = _mxq()
    y = mxq.qmm(case.x_d, case.w_d, case.s_d, case.b_d, bits)
    yr, bnd = _full_ref(case)
    assert_close(to_f64(y), yr, bnd, "qmm split M=%d bits=%d" % (M, bits))
    for _ in range(3):
        y2 = mxq.qmm(case.x_d, case.w_d, case.s_d, case.b_d, bits)
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M", [128, 600])
def test_qmm_sweep_large_m_full(bits, M):
    import torch

    case = DenseCase(M, 5120, 5120, bits, seed=0, x_seed=1)
    mxq = _mxq()
    y = mxq.qmm(case.x_d, case.w_d, case.s_d, case.b_d, bits)
    yr, bnd = _full_ref(case)
    assert_close(to_f64(y), yr, bnd, "qmm sweep M=%d bits=%d" % (M, bits))
    # repeated launches give identical bits (no race between pipeline stages)
    for _ in range(3):
        y2 = mxq.qmm(case.x_d, case.w_d, case.s_d, case.b_d, bits)
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_qmm_prefill_full_size():
    import torch

    case = DenseCase(600, 5120, 17408, 4, seed=0, x_seed=1)
    mxq = _mxq()
    y = mxq.qmm(case.x_d, case.w_d, case.s_d, case.b_d, 4)
    yr, bnd = _full_ref(case)
    assert_close(to_f64(y), yr, bnd, "qmm prefill 600x5120x17408")
    for _ in range(3):
        y2 = mxq.qmm(case.x_d, case.w_d, case.s_d, case.b_d, 4)
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_qmm_m1_matches_qmv_within_tolerance():
    case = DenseCase(1, 5120, 1024, 4, seed=5, x_seed=6)
    mxq = _mxq()
    y_mm = to_f64(mxq.qmm(case.x_d, case.w_d, case.s_d, case.b_d, 4))[0]
    y_mv = to_f64(mxq.qmv(case.x_d[0], case.w_d, case.s_d, case.b_d, 4))
    yr, bnd = _full_ref(case)
    assert_close(y_mm, yr[0], bnd[0], "qmm M=1")
    assert_close(y_mv, yr[0], bnd[0], "qmv")


def test_qmm_guard_bands_and_status():
    import torch

    M, K, N = 70, 640, 200
    case = DenseCase(M, K, N, 4, seed=11)
    guard = 8192
    buf = torch.full((guard + M * N + guard,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = buf[guard:guard + M * N].view(M, N)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    _mxq().qmm(case.x_d, case.w_d, case.s_d, case.b_d, 4, out=out, dev_status=status)
    torch.cuda.synchronize()
    assert torch.isnan(buf[:guard]).all() and torch.isnan(buf[guard + M * N:]).all()
    assert int(status.item()) == 0
    yr, bnd = _full_ref(case)
    assert_close(to_f64(out), yr, bnd, "qmm guarded")


def test_qmm_group_boundary_one_hot():
    # x = e_k rows pick single dequantised weights: checks nibble order, the
    # swizzled shared-memory layout and the group index on the tensor path
    import synth
    from tests.gpu_util import bf16_dev

    K, N = 256, 128
    ks = [0, 1, 7, 8, 9, 15, 16, 31, 63, 64, 65, 127, 128, 200, 255]
    case = DenseCase(len(ks), K, N, 4, seed=2)
    x = np.zeros((len(ks), K), np.float32)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    xb = synth.f32_to_bf16_bits(x)
    y = _mxq().qmm(bf16_dev(xb), case.w_d, case.s_d, case.b_d, 4)
    wh = oracle.dequant(case.qw.w, case.qw.scales, case.qw.biases, N, K, 4)
    # the kernel rounds w^ to bf16 once; the output is that value rounded again
    want = np.stack([wh[:, k] for k in ks])
    assert_close(to_f64(y), want, np.abs(want), "one-hot")

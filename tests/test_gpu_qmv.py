"""GPU parity of mxq_qmv (decode GEMV) against the f64 checker, element by
element, through the C ABI.  Shapes: the tiny and decode workloads (K=512
N=256; K=5120 N=17408; K=17408 N=5120) plus ragged edges."""

import numpy as np
import pytest

import oracle
from tests.gpu_util import DenseCase, assert_close, bf16_dev, to_f64

pytestmark = pytest.mark.gpu


def _run(case, out=None):
    import affine_bit_matmul_gb300 as mxq

    return mxq.qmv(case.x_d[0], case.w_d, case.s_d, case.b_d, case.bits, out=out)


def _ref(case):
    return oracle.qmv(case.x[0], case.qw.w, case.qw.scales, case.qw.biases, case.K, case.N,
                      case.bits)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("K,N", [(512, 256), (64, 1), (64, 7), (128, 17), (704, 33), (1088, 100),
                                 (1024, 16), (2048, 31), (5120, 513), (6144, 129),
                                 (1536, 77), (18432, 40), (19456, 40),
                                 # rows whose scales are not whole 16-byte units:
                                 # chunks of the streaming kernel start on 2, 4
                                 # or 8 rows
                                 (2816, 704), (704, 2816), (1088, 104), (1472, 96),
                                 (2880, 66), (320, 136)])
def test_qmv_small(bits, K, N):
    case = DenseCase(1, K, N, bits, seed=K + N, x_seed=K)
    y = _run(case)
    yr, bnd = _ref(case)
    assert_close(to_f64(y), yr, bnd, "qmv K=%d N=%d bits=%d" % (K, N, bits))


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("K,N", [(5120, 17408), (17408, 5120)])
def test_qmv_decode_full(bits, K, N):
    case = DenseCase(1, K, N, bits, seed=0, x_seed=1)
    y = _run(case)
    yr, bnd = _ref(case)
    assert_close(to_f64(y), yr, bnd, "qmv decode K=%d N=%d bits=%d" % (K, N, bits))
    # bitwise run-to-run determinism
    import torch

    y2 = _run(case)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_qmv_guard_bands_untouched():
    import torch

    case = DenseCase(1, 1024, 300, 4, seed=3)
    guard = 4096
    buf = torch.full((guard + 300 + guard,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = buf[guard:guard + 300]
    _run(case, out=out)
    torch.cuda.synchronize()
    assert torch.isnan(buf[:guard]).all() and torch.isnan(buf[guard + 300:]).all()
    yr, bnd = _ref(case)
    assert_close(to_f64(out), yr, bnd, "qmv guarded")


def test_qmv_closed_form_zero_scale():
    # s = 0, b = c: y = c * sum_k x_k (all values small integers: exact)
    import synth
    import affine_bit_matmul_gb300 as mxq
    from tests.gpu_util import codes_dev

    K, N = 1024, 64
    rng = np.random.default_rng(9)
    x = rng.integers(-4, 5, size=(1, K)).astype(np.float32)
    xb = synth.f32_to_bf16_bits(x)
    c = (np.arange(N) % 8 + 1) / 8.0
    s = np.zeros((N, K // 64), np.uint16)
    b = np.repeat(synth.f32_to_bf16_bits(c.astype(np.float32))[:, None], K // 64, axis=1)
    w = rng.integers(0, 2 ** 32, size=(N, K // 8), dtype=np.uint64).astype(np.uint32)
    y = mxq.qmv(bf16_dev(xb)[0], codes_dev(w), bf16_dev(s), bf16_dev(b), 4)
    exact = (c * x.sum()).astype(np.float32)  # exact in fp32
    want = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(exact)).astype(np.float64)
    assert np.array_equal(to_f64(y), want)


@pytest.mark.parametrize("bits", [4, 8])
def test_qmv_direct_load_path(bits):
    # scales/biases that are only 2-byte aligned, and K beyond the streaming
    # kernel's range, take the direct-load kernel: same acceptance rule
    import torch

    case = DenseCase(1, 1536, 300, bits, seed=12, x_seed=13)
    import affine_bit_matmul_gb300 as mxq

    s_off = torch.empty(case.s_d.numel() + 1, dtype=torch.bfloat16, device="cuda")[1:]
    b_off = torch.empty(case.b_d.numel() + 1, dtype=torch.bfloat16, device="cuda")[1:]
    s_off.copy_(case.s_d.view(-1))
    b_off.copy_(case.b_d.view(-1))
    y = mxq.qmv(case.x_d[0], case.w_d, s_off.view_as(case.s_d), b_off.view_as(case.b_d), bits)
    yr, bnd = _ref(case)
    assert_close(to_f64(y), yr, bnd, "qmv unaligned scales bits=%d" % bits)
    big = DenseCase(1, 32768, 96, bits, seed=14, x_seed=15)
    y = _run(big)
    yr, bnd = _ref(big)
    assert_close(to_f64(y), yr, bnd, "qmv K=32768 bits=%d" % bits)
    del torch


def test_qmv_status_word_clear():
    import torch

    case = DenseCase(1, 5120, 1000, 4, seed=16)
    import affine_bit_matmul_gb300 as mxq

    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    y = mxq.qmv(case.x_d[0], case.w_d, case.s_d, case.b_d, 4, dev_status=status)
    assert int(status.item()) == 0
    yr, bnd = _ref(case)
    assert_close(to_f64(y), yr, bnd, "qmv with status")


def _qmv_bits(case, xbits):
    import affine_bit_matmul_gb300 as mxq

    return mxq.qmv(bf16_dev(xbits.reshape(1, -1))[0], case.w_d, case.s_d, case.b_d, case.bits)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("K,N", [(5120, 256), (2048, 100), (32768, 64)])
def test_qmv_power_of_two_scale_equivariance(bits, K, N):
    # Scaling x by 2^-100 scales every exact product and every fp32 partial
    # by 2^-100 with no rounding (all values stay normal), so the result is
    # the unscaled result times 2^-100 bit for bit.  This pins the exponent
    # handling of both kernels (the streaming kernel re-bases activations
    # on their largest exponent; the direct-load kernel works in fp32).
    import synth

    case = DenseCase(1, K, N, bits, seed=21, x_seed=22)
    xf = synth.bf16_bits_to_f32(case.x[0])
    xs = synth.f32_to_bf16_bits((xf * np.float32(2.0 ** -100)).astype(np.float32))
    assert np.array_equal(synth.bf16_bits_to_f32(xs).astype(np.float64),
                          xf.astype(np.float64) * 2.0 ** -100)
    y1 = to_f64(_qmv_bits(case, case.x[0]))
    y2 = to_f64(_qmv_bits(case, xs))
    assert np.array_equal(y2, y1 * 2.0 ** -100)


@pytest.mark.parametrize("bits", [4, 8])
def test_qmv_wide_range_activations(bits):
    # activations spanning 2^-60 .. 2^20 inside every 32-value lane block,
    # with zeros, subnormal bf16 values and both signs: the streaming
    # kernel's fixed-point activations round only values more than 2^15
    # below the block's largest, far inside the acceptance rule
    import synth

    K, N = 2048, 128
    case = DenseCase(1, K, N, bits, seed=23, x_seed=24)
    rng = np.random.default_rng(25)
    mag = (1.0 + rng.random(K)) * 2.0 ** rng.integers(-60, 21, size=K)
    x = np.where(rng.random(K) < 0.5, -mag, mag)
    x[rng.random(K) < 0.1] = 0.0
    x[::97] = 2.0 ** -130  # subnormal in bf16
    xb = synth.f32_to_bf16_bits(x.astype(np.float32))
    y = to_f64(_qmv_bits(case, xb))
    yr, bnd = oracle.qmv(xb, case.qw.w, case.qw.scales, case.qw.biases, K, N, bits)
    assert_close(y, yr, bnd, "qmv wide-range x bits=%d" % bits)
    # relative check without the absolute term
    assert np.all(np.abs(y - yr) <= 8e-3 * bnd + 1e-30)


@pytest.mark.parametrize("bits", [4, 8])
def test_qmv_tiny_activations(bits):
    # every activation near 2^-110: the common scale of a lane block is a
    # subnormal float, the products and the result are still normal
    import synth

    K, N = 1024, 64
    case = DenseCase(1, K, N, bits, seed=26, x_seed=27)
    rng = np.random.default_rng(28)
    x = (rng.standard_normal(K) * 2.0 ** -110).astype(np.float32)
    x[np.abs(x) < 2.0 ** -118] = 2.0 ** -118
    xb = synth.f32_to_bf16_bits(x)
    y = to_f64(_qmv_bits(case, xb))
    yr, bnd = oracle.qmv(xb, case.qw.w, case.qw.scales, case.qw.biases, K, N, bits)
    assert np.all(np.isfinite(y))
    assert np.all(np.abs(y - yr) <= 8e-3 * bnd + 2.0 ** -140)

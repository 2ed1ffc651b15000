"""GPU parity of mxq_quantize (the affine group-64 encoder) with the oracle's
encoder: every decision is taken in binary32 on both sides, so codes, scales
and biases must match bit for bit."""

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu


def _gpu(W, bits):
    import torch

    import affine_bit_matmul_gb300 as mxq

    w = torch.from_numpy(np.ascontiguousarray(W, np.float32)).cuda()
    codes, s, b = mxq.quantize(w, bits)
    torch.cuda.synchronize()
    return (codes.cpu().numpy().view(np.uint32), s.view(torch.int16).cpu().numpy().view(np.uint16),
            b.view(torch.int16).cpu().numpy().view(np.uint16))


def _same(W, bits):
    c, s, b = _gpu(W, bits)
    co, so, bo = oracle.quantize(W, bits)
    assert np.array_equal(s, so), "scales differ"
    assert np.array_equal(b, bo), "biases differ"
    assert np.array_equal(c, co), "codes differ at %s" % (np.argwhere(c != co)[:5],)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("N,K", [(1, 64), (37, 192), (129, 5120), (17, 20480), (300, 704)])
def test_quantize_matches_oracle(bits, N, K):
    rng = np.random.default_rng(N * 7 + K)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    _same(W, bits)


@pytest.mark.parametrize("bits", [4, 8])
def test_quantize_special_groups(bits):
    rng = np.random.default_rng(5)
    N, K = 8, 512
    W = (rng.standard_normal((N, K)) * 3.0).astype(np.float32)
    W[0, :64] = 0.7                                   # flat group
    W[0, 64:128] = -0.0                               # negative zeros
    W[1, :64] = np.where(np.arange(64) % 2, 0.0, -0.0)
    W[2] *= np.float32(1e30)                          # huge
    W[3] *= np.float32(1e-30)                         # tiny (some subnormal)
    W[4, :64] = np.arange(64, dtype=np.float32)       # exact grid with ties
    W[5] = np.round(W[5] * 4) / 4                     # many repeated values
    W[6, ::2] = W[6, 1::2]                            # pairs of equal values
    _same(W, bits)


def test_quantize_then_matmul_roundtrip():
    # encode on the GPU, multiply with the GPU GEMV, compare with the oracle
    # GEMV on the oracle's encoding of the same weights
    import torch

    import affine_bit_matmul_gb300 as mxq
    import synth
    from tests.gpu_util import assert_close, bf16_dev, to_f64

    rng = np.random.default_rng(9)
    K, N = 2048, 384
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    x = synth.activations(1, K, seed=3)
    codes, s, b = mxq.quantize(torch.from_numpy(W).cuda(), 4)
    y = to_f64(mxq.qmv(bf16_dev(x)[0], codes, s, b, 4))
    co, so, bo = oracle.quantize(W, 4)
    yr, bnd = oracle.qmv(x[0], co, so, bo, K, N, 4)
    assert_close(y, yr, bnd, "quantize + qmv")

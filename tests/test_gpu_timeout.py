"""The give-up path of the kernels' bounded waits, made to run out on purpose.

Every on-chip pipeline wait gives up after a budget of SM clock cycles; the
budget is shortened here to one cycle (``set_wait_budget``), so that the
first wait of each pipeline role that is not already satisfied gives up.
Each kernel family must then (1) return, (2) report ``DEV_TIMEOUT`` in its
status word, and (3) leave the device usable: with the default budget back,
the same call again equals the result of a normal call before the timeout,
bit for bit, and matches the oracle.  Nothing here faults or hangs a GPU:
the waits are bounded, and the waits for a CTA's own copies and MMAs keep
the default budget, so no asynchronous write outlives the kernel."""

import numpy as np
import pytest

import oracle
from tests.gpu_util import DenseCase, MoECase, assert_close, to_f64

pytestmark = pytest.mark.gpu


def _mxq():
    import affine_bit_matmul_gb300 as mxq

    return mxq


@pytest.fixture
def short_budget():
    mxq = _mxq()
    try:
        yield lambda: mxq.set_wait_budget(1)
    finally:
        assert mxq.set_wait_budget(0) == 2_000_000_000


def _status():
    import torch

    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _timed_out_then_normal(run, set_short):
    """run(status) -> y.  A normal call, a call under the short budget, then a
    normal call again; returns (y before, y after, status of the short call)."""
    import torch

    mxq = _mxq()
    st = _status()
    y0 = run(st).clone()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert set_short() == 1
    st_short = _status()
    run(st_short)
    torch.cuda.synchronize()  # the call returned: no wait outlived its budget
    code = int(st_short.item())
    assert mxq.set_wait_budget(0) == 2_000_000_000
    st2 = _status()
    y1 = run(st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    return y0, y1, code


def _points(case, y, count=2000, seed=5):
    rng = np.random.default_rng(seed)
    rows = rng.integers(0, y.shape[0], size=count).astype(np.int64)
    cols = rng.integers(0, case.N, size=count).astype(np.int64)
    return rows, cols


def test_qmv_stream_timeout_then_parity(short_budget):
    mxq = _mxq()
    c = DenseCase(1, 5120, 17408, 4, seed=0, x_seed=1)
    _, y1, code = _timed_out_then_normal(
        lambda st: mxq.qmv(c.x_d[0], c.w_d, c.s_d, c.b_d, 4, dev_status=st), short_budget)
    assert code == mxq.DEV_TIMEOUT
    yr, bnd = oracle.qmv(c.x[0], c.qw.w, c.qw.scales, c.qw.biases, c.K, c.N, 4)
    assert_close(to_f64(y1), yr, bnd, "qmv after a timeout")


def test_qmm_cluster_split_timeout_then_parity(short_budget):
    # 16 rows, K = N = 2048: too few tiles for the SMs, so K is split over
    # the CTAs of a cluster (the distributed-shared-memory reduction)
    mxq = _mxq()
    c = DenseCase(16, 2048, 2048, 4, seed=2, x_seed=3)
    _, y1, code = _timed_out_then_normal(
        lambda st: mxq.qmm(c.x_d, c.w_d, c.s_d, c.b_d, 4, dev_status=st), short_budget)
    assert code == mxq.DEV_TIMEOUT
    yr, bnd = oracle.qmm(c.x, c.qw.w, c.qw.scales, c.qw.biases, c.M, c.K, c.N, 4)
    assert_close(to_f64(y1), yr, bnd, "qmm (K split) after a timeout")


@pytest.mark.parametrize("bits", [4, 8])
def test_qmm_persistent_timeout_then_parity(short_budget, bits):
    # 300 rows x 17408 outputs: 2 x 136 tiles, one persistent CTA per SM
    mxq = _mxq()
    c = DenseCase(300, 512, 17408, bits, seed=4, x_seed=5)
    _, y1, code = _timed_out_then_normal(
        lambda st: mxq.qmm(c.x_d, c.w_d, c.s_d, c.b_d, bits, dev_status=st), short_budget)
    assert code == mxq.DEV_TIMEOUT
    rows, cols = _points(c, y1)
    yr, bnd = oracle.points(c.x, c.qw.w, c.qw.scales, c.qw.biases, rows, cols, c.K, c.N, bits)
    assert_close(to_f64(y1)[rows, cols], yr, bnd, "persistent qmm after a timeout")


@pytest.mark.parametrize("bits", [4, 8])
def test_grouped_gemm_timeout_then_parity(short_budget, bits):
    # 4-bit: the compact persistent grouped kernel; 8-bit: one CTA per tile
    mxq = _mxq()
    c = MoECase(128, 16, 4, 1024, 512, bits, seed=6)
    _, y1, code = _timed_out_then_normal(
        lambda st: mxq.gather_qmm(c.x_d, c.w_d, c.s_d, c.b_d, c.ids_d, c.src_d, bits,
                                  dev_status=st), short_budget)
    assert code == mxq.DEV_TIMEOUT
    yr, bnd = oracle.gather_qmm(c.x, c.w, c.s, c.b, c.ids, c.src, c.T, c.B, c.E, c.K, c.N, bits)
    assert_close(to_f64(y1), yr, bnd, "grouped GEMM after a timeout")


def test_gateup_grouped_timeout_then_parity(short_budget):
    import torch

    mxq = _mxq()
    c = MoECase(96, 8, 4, 512, 256, 4, seed=7)
    u = MoECase(96, 8, 4, 512, 256, 4, seed=8)

    def run(st):
        g, up = mxq.gather_qmm_gateup(c.x_d, c.w_d, c.s_d, c.b_d, u.w_d, u.s_d, u.b_d, c.ids_d,
                                      c.src_d, 4, dev_status=st)
        return torch.cat([g, up], 1)

    _, y1, code = _timed_out_then_normal(run, short_budget)
    assert code == mxq.DEV_TIMEOUT
    for w, s, b, part in ((c.w, c.s, c.b, 0), (u.w, u.s, u.b, 1)):
        yr, bnd = oracle.gather_qmm(c.x, w, s, b, c.ids, c.src, c.T, c.B, c.E, c.K, c.N, 4)
        assert_close(to_f64(y1[:, part * c.N:(part + 1) * c.N]), yr, bnd,
                     "gate/up set %d after a timeout" % part)


@pytest.mark.parametrize("M,K,N", [(16, 2048, 2048), (300, 512, 4096)])
def test_qmm_kn_timeout_then_parity(short_budget, M, K, N):
    # the [K, N]-layout GEMM: with a K split over a cluster, and without
    import synth
    from tests.gpu_util import bf16_dev, codes_dev

    mxq = _mxq()
    qw = synth.quantize(synth.dense_weights(K, N, seed=M), 4, 64)
    x = synth.activations(M, K, seed=M + 1)
    w_d, s_d, b_d, x_d = codes_dev(qw.w), bf16_dev(qw.scales), bf16_dev(qw.biases), bf16_dev(x)
    _, y1, code = _timed_out_then_normal(
        lambda st: mxq.qmm_kn(x_d, w_d, s_d, b_d, 4, dev_status=st), short_budget)
    assert code == mxq.DEV_TIMEOUT
    yr, bnd = oracle.qmm_kn(x, qw.w, qw.scales, qw.biases, M, K, N, 4)
    assert_close(to_f64(y1), yr, bnd, "qmm_kn after a timeout")

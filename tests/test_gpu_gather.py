"""GPU parity of mxq_gather_qmm (sorted mixture-of-experts GEMM) against the
f64 checker through the C ABI: small routings element by element, the two
expert shapes of the workload (E=128, top_k=8, 573 tokens; K=2816 N=704 and
K=704 N=2816) on samples plus whole rows, the constant-per-expert case,
empty / single-row / all-rows experts, and invalid ids."""

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import MoECase, assert_close, bf16_dev, codes_dev, i32_dev, to_f64

pytestmark = pytest.mark.gpu


def _mxq():
    import affine_bit_matmul_gb300 as mxq

    return mxq


_SAME = object()


def _run(c, out=None, status=None, ids_d=None, src_d=_SAME):
    return _mxq().gather_qmm(c.x_d, c.w_d, c.s_d, c.b_d, c.ids_d if ids_d is None else ids_d,
                             c.src_d if src_d is _SAME else src_d, c.bits, out=out,
                             dev_status=status)


def _ref(c, ids=None, src=_SAME):
    return oracle.gather_qmm(c.x, c.w, c.s, c.b, c.ids if ids is None else ids,
                             c.src if src is _SAME else src, c.T, c.B, c.E, c.K, c.N, c.bits)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("T,E,top_k,K,N,ident", [
    (9, 4, 2, 128, 128, False), (40, 8, 3, 704, 200, False), (33, 16, 4, 256, 130, True),
    (300, 6, 2, 192, 256, False), (5, 3, 3, 64, 64, True),
])
def test_gather_small(bits, T, E, top_k, K, N, ident):
    c = MoECase(T, E, top_k, K, N, bits, seed=T + E, identity_src=ident, routing_seed=T)
    import torch

    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    y = _run(c, status=status)
    yr, bnd = _ref(c)
    assert_close(to_f64(y), yr, bnd, "gather T=%d E=%d K=%d N=%d bits=%d" % (T, E, K, N, bits))
    assert int(status.item()) == 0


def _sample_check(c, y, count=3000):
    rng = np.random.default_rng(1)
    rows = rng.integers(0, c.B, size=count).astype(np.int64)
    cols = rng.integers(0, c.N, size=count).astype(np.int64)
    yr, bnd = oracle.points(c.x, c.w, c.s, c.b, rows, cols, c.K, c.N, c.bits, expert_ids=c.ids,
                            row_src=c.src, E=c.E)
    assert_close(to_f64(y)[rows, cols], yr, bnd, "gather sample")
    # whole rows at segment starts and ends of a few experts
    yh = to_f64(y)
    for e in (0, 1, c.E // 2, c.E - 1):
        seg = np.nonzero(c.ids == e)[0]
        for r in (seg[0], seg[-1]):
            rr = np.full(c.N, r, np.int64)
            cc = np.arange(c.N, dtype=np.int64)
            yr, bnd = oracle.points(c.x, c.w, c.s, c.b, rr, cc, c.K, c.N, c.bits,
                                    expert_ids=c.ids, row_src=c.src, E=c.E)
            assert_close(yh[r], yr, bnd, "gather row %d (expert %d)" % (r, e))


@pytest.mark.parametrize("K,N,ident,bits", [(2816, 704, False, 4), (704, 2816, True, 4),
                                             (2816, 704, False, 8)])
def test_gather_workload_shapes(K, N, ident, bits):
    # the sorted-MoE workload (573 tokens, top 8 of 128 experts), every
    # element of the [4584, N] output against the f64 checker, plus bitwise
    # run-to-run determinism
    import torch

    c = MoECase(573, 128, 8, K, N, bits, seed=0, identity_src=ident)
    assert c.B == 4584
    y = _run(c)
    yr, bnd = _ref(c)
    assert_close(to_f64(y), yr, bnd, "gather workload K=%d N=%d bits=%d" % (K, N, bits))
    _sample_check(c, y, count=500)
    y2 = _run(c)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_constant_per_expert_exact():
    # w^_e[n, k] = c_{e,n} distinct per (e, n) (s = 0); x integer: every y is
    # exact, so any mis-gathered expert, source row or column shows
    T, E, top_k, K, N = 64, 12, 4, 256, 136
    ids, src = synth.routing(T, E, top_k, seed=7)
    B = T * top_k
    rng = np.random.default_rng(8)
    x = rng.integers(-4, 5, size=(T, K)).astype(np.float32)
    # (e + 1) + (n % 16)/16 is exact in bf16 and differs between experts and
    # between neighbouring columns; every partial sum stays exact in fp32
    cvals = np.array([[(e + 1) + (n % 16) / 16.0 for n in range(N)] for e in range(E)],
                     np.float32)
    cb = synth.f32_to_bf16_bits(cvals)
    assert np.array_equal(synth.bf16_bits_to_f32(cb), cvals)
    cvals = cvals.astype(np.float64)
    s = np.zeros((E, N, K // 64), np.uint16)
    b = np.repeat(cb[:, :, None], K // 64, axis=2)
    w = rng.integers(0, 2 ** 32, size=(E, N, K // 8), dtype=np.uint64).astype(np.uint32)
    y = _mxq().gather_qmm(bf16_dev(synth.f32_to_bf16_bits(x)), codes_dev(w), bf16_dev(s),
                          bf16_dev(b), i32_dev(ids), i32_dev(src), 4)
    exact = cvals[ids] * x.sum(axis=1, dtype=np.float64)[src][:, None]
    want = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(exact.astype(np.float32)))
    assert np.array_equal(to_f64(y), want.astype(np.float64))


def _custom_ids(c, ids):
    c.ids = np.asarray(ids, np.int32)
    c.ids_d = i32_dev(c.ids)
    return c


@pytest.mark.parametrize("pattern", ["empty_and_single", "one_expert_all_rows", "large_segment"])
def test_gather_segment_edges(pattern):
    T, E, K, N = 300, 5, 192, 130
    c = MoECase(T, E, 1, K, N, 4, seed=3, identity_src=True)
    if pattern == "empty_and_single":
        ids = [0] * 1 + [2] * 150 + [4] * 149   # experts 1 and 3 empty, expert 0 one row
    elif pattern == "one_expert_all_rows":
        ids = [3] * 300
    else:
        ids = [1] * 280 + [2] * 20               # a 280-row segment: two tiles
    _custom_ids(c, ids)
    y = _run(c)
    yr, bnd = _ref(c)
    assert_close(to_f64(y), yr, bnd, "gather %s" % pattern)


def test_gather_single_expert_equals_qmm():
    c = MoECase(200, 1, 1, 640, 256, 8, seed=4, identity_src=True)
    yg = to_f64(_run(c))
    import affine_bit_matmul_gb300 as mxq

    ym = to_f64(mxq.qmm(c.x_d, c.w_d[0], c.s_d[0], c.b_d[0], 8))
    yr, bnd = _ref(c)
    assert_close(yg, yr, bnd, "gather E=1")
    assert_close(ym, yr, bnd, "qmm on same rows")


def test_gather_out_of_range_ids_zeroed_and_reported():
    import torch

    T, E, K, N = 40, 4, 128, 128
    c = MoECase(T, E, 1, K, N, 4, seed=6, identity_src=True)
    ids = [-1] * 3 + [0] * 10 + [1] * 10 + [3] * 12 + [4] * 5  # -1 and 4 are invalid
    _custom_ids(c, ids)
    out = torch.full((c.B, N), 7.0, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    _run(c, out=out, status=status)
    assert int(status.item()) & _mxq().DEV_BAD_EXPERT_ID
    y = to_f64(out)
    assert np.all(y[:3] == 0) and np.all(y[-5:] == 0)
    yr, bnd = _ref(c)
    assert_close(y, yr, bnd, "gather with invalid ids")


def test_gather_unsorted_ids_zero_output_and_report():
    import torch

    T, E, K, N = 32, 4, 128, 64
    c = MoECase(T, E, 1, K, N, 4, seed=6, identity_src=True)
    _custom_ids(c, [0] * 8 + [2] * 8 + [1] * 8 + [3] * 8)
    out = torch.full((c.B, N), 7.0, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    _run(c, out=out, status=status)
    assert int(status.item()) & _mxq().DEV_UNSORTED_IDS
    assert bool((out.float() == 0).all())


def test_gather_bad_row_src_row_is_zero():
    import torch

    T, E, K, N = 20, 3, 128, 128
    c = MoECase(T, E, 2, K, N, 4, seed=9)
    src = c.src.copy()
    src[5] = T + 3
    src[11] = -2
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    y = to_f64(_run(c, status=status, src_d=i32_dev(src)))
    assert int(status.item()) & _mxq().DEV_BAD_ROW_SRC
    assert np.all(y[5] == 0) and np.all(y[11] == 0)
    good = np.ones(c.B, bool)
    good[[5, 11]] = False
    yr, bnd = _ref(c, src=np.where(good, src, 0))
    assert_close(y[good], yr[good], bnd[good], "gather with bad row_src")


# ---- decode-sized calls (at most 32 sorted rows): one GEMV per row

@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("T,K,N,ident", [(1, 2816, 704, False), (4, 704, 2816, True),
                                         (3, 2816, 704, False)])
def test_gather_decode_rows(bits, T, K, N, ident):
    # one to four tokens routed to 8 of 128 experts: whole outputs, and
    # bitwise determinism
    import torch

    c = MoECase(T, 128, 8, K, N, bits, seed=11 + T, identity_src=ident, routing_seed=5 + T)
    assert c.B <= 32
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    y = _run(c, status=status)
    yr, bnd = _ref(c)
    assert_close(to_f64(y), yr, bnd, "gather decode T=%d K=%d N=%d bits=%d" % (T, K, N, bits))
    assert int(status.item()) == 0
    y2 = _run(c)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_gather_decode_constant_per_expert_exact():
    T, E, top_k, K, N = 4, 12, 8, 256, 136
    ids, src = synth.routing(T, E, top_k, seed=7)
    rng = np.random.default_rng(8)
    x = rng.integers(-4, 5, size=(T, K)).astype(np.float32)
    cvals = np.array([[(e + 1) + (n % 16) / 16.0 for n in range(N)] for e in range(E)],
                     np.float32)
    cb = synth.f32_to_bf16_bits(cvals)
    s = np.zeros((E, N, K // 64), np.uint16)
    b = np.repeat(cb[:, :, None], K // 64, axis=2)
    w = rng.integers(0, 2 ** 32, size=(E, N, K // 8), dtype=np.uint64).astype(np.uint32)
    y = _mxq().gather_qmm(bf16_dev(synth.f32_to_bf16_bits(x)), codes_dev(w), bf16_dev(s),
                          bf16_dev(b), i32_dev(ids), i32_dev(src), 4)
    exact = cvals.astype(np.float64)[ids] * x.sum(axis=1, dtype=np.float64)[src][:, None]
    want = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(exact.astype(np.float32)))
    assert np.array_equal(to_f64(y), want.astype(np.float64))


def test_gather_decode_invalid_ids_and_sources():
    import torch

    T, E, K, N = 12, 4, 128, 128
    c = MoECase(T, E, 2, K, N, 4, seed=21)
    ids = np.sort(c.ids).copy()
    ids[0] = -1
    ids[-1] = E            # out of range at both ends
    src = c.src.copy()
    src[5] = T + 1
    c.ids = ids.astype(np.int32)
    c.ids_d = i32_dev(c.ids)
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    out = torch.full((c.B, N), 7.0, dtype=torch.bfloat16, device="cuda")
    _run(c, out=out, status=status, src_d=i32_dev(src))
    st = int(status.item())
    assert st & _mxq().DEV_BAD_EXPERT_ID and st & _mxq().DEV_BAD_ROW_SRC
    y = to_f64(out)
    assert np.all(y[0] == 0) and np.all(y[-1] == 0) and np.all(y[5] == 0)
    good = np.ones(c.B, bool)
    good[[0, 5, c.B - 1]] = False
    yr, bnd = _ref(c, ids=np.clip(ids, 0, E - 1), src=np.where(good, src, 0))
    assert_close(y[good], yr[good], bnd[good], "gather decode with invalid rows")

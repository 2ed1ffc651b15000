"""GPU parity of the few-rows shapes against the f64 checker through the C
ABI, element by element:

* mxq_qmm with 1 <= M <= 8 (every group size; K split over clusters; N not
  a multiple of the tile); M = 1 is bit for bit the GEMV;
* mxq_gather_qmm at decode sizes: one to 128 tokens routed to 8 of 128
  experts, both expert shapes of the workload, routed and identity sources,
  a hot expert, invalid ids and sources, the constant-per-expert case, and
  both GEMV forms (streaming, and direct-load when the scales are not
  16-byte aligned);
* mxq_gather_qmm_gateup (the gate and up projections of an MoE layer in one
  launch): both outputs against two separate checker calls, at decode size
  (per-row GEMVs) and at prefill size (the grouped GEMM), each bit for bit
  equal to the single-set call."""

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import DenseCase, MoECase, assert_close, bf16_dev, codes_dev, i32_dev, to_f64

pytestmark = pytest.mark.gpu


def _mxq():
    import affine_bit_matmul_gb300 as mxq

    return mxq


@pytest.mark.parametrize("group", [32, 64, 128])
@pytest.mark.parametrize("M,K,N", [(2, 256, 16), (3, 512, 17), (5, 1280, 100), (8, 5120, 5120),
                                   (8, 2048, 1000), (7, 5120, 17408), (4, 17408, 512),
                                   (8, 768, 4000)])
def test_qmm_few_rows(M, K, N, group):
    import torch

    c = DenseCase(M, K, N, 4, seed=M * 7 + K, x_seed=N, group=group)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    y = _mxq().qmm(c.x_d, c.w_d, c.s_d, c.b_d, 4, dev_status=status, group_size=group)
    yr, bnd = oracle.qmm(c.x, c.qw.w, c.qw.scales, c.qw.biases, M, K, N, 4, group)
    assert_close(to_f64(y), yr, bnd, "qmm M=%d K=%d N=%d G=%d" % (M, K, N, group))
    assert int(status.item()) == 0
    y2 = _mxq().qmm(c.x_d, c.w_d, c.s_d, c.b_d, 4, group_size=group)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_qmm_one_row_is_the_gemv():
    c = DenseCase(1, 5120, 5120, 4, seed=3, x_seed=4)
    y = _mxq().qmm(c.x_d, c.w_d, c.s_d, c.b_d, 4)
    yv = _mxq().qmv(c.x_d[0], c.w_d, c.s_d, c.b_d, 4)
    yr, bnd = oracle.qmm(c.x, c.qw.w, c.qw.scales, c.qw.biases, 1, 5120, 5120, 4)
    assert_close(to_f64(y), yr, bnd, "qmm M=1")
    import torch

    assert torch.equal(y[0].view(torch.int16), yv.view(torch.int16))


def test_qmm_few_rows_one_hot_group_edges():
    # one-hot activations pick single dequantised weights at every group edge
    # of a 4-row call (k = 63/64, 127/128 ...), with a distinct scale/bias per group
    M, K, N = 4, 512, 48
    rng = np.random.default_rng(5)
    q = rng.integers(0, 16, size=(N, K))
    w = synth.pack_codes(q, 4)
    s = synth.f32_to_bf16_bits(rng.uniform(0.5, 2.0, size=(N, K // 64)).astype(np.float32))
    b = synth.f32_to_bf16_bits(rng.uniform(-4, 4, size=(N, K // 64)).astype(np.float32))
    ks = [0, 63, 64, 127, 128, 255, 256, 511]
    for k0 in range(0, len(ks), M):
        x = np.zeros((M, K), np.float32)
        for m, k in enumerate(ks[k0:k0 + M]):
            x[m, k] = 1.0
        xb = synth.f32_to_bf16_bits(x)
        y = _mxq().qmm(bf16_dev(xb), codes_dev(w), bf16_dev(s), bf16_dev(b), 4)
        yr, bnd = oracle.qmm(xb, w, s, b, M, K, N, 4)
        assert_close(to_f64(y), yr, bnd, "one-hot rows %s" % ks[k0:k0 + M])


@pytest.mark.parametrize("T,K,N,ident", [(1, 2816, 704, False), (4, 2816, 704, False),
                                         (4, 704, 2816, True), (16, 2816, 704, False),
                                         (64, 704, 2816, True), (128, 2816, 704, False)])
def test_gather_decode_sizes(T, K, N, ident):
    # T tokens x top 8 of 128 experts: B = 8T <= 8E rows, whole outputs
    import torch

    c = MoECase(T, 128, 8, K, N, 4, seed=40 + T, identity_src=ident, routing_seed=9 + T)
    assert c.B <= 8 * 128
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    y = _mxq().gather_qmm(c.x_d, c.w_d, c.s_d, c.b_d, c.ids_d, c.src_d, 4, dev_status=status)
    yr, bnd = oracle.gather_qmm(c.x, c.w, c.s, c.b, c.ids, c.src, c.T, c.B, c.E, c.K, c.N, 4)
    assert_close(to_f64(y), yr, bnd, "gather decode T=%d K=%d N=%d" % (T, K, N))
    assert int(status.item()) == 0
    y2 = _mxq().gather_qmm(c.x_d, c.w_d, c.s_d, c.b_d, c.ids_d, c.src_d, 4)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("T,K,N,ident", [(2, 2816, 704, False), (4, 704, 2816, True)])
def test_gather_decode_direct_form(T, K, N, ident):
    # scales and biases that are not 16-byte aligned do not fit the streaming
    # GEMV: the call takes the direct-load GEMV and must agree all the same
    import torch

    c = MoECase(T, 32, 8, K, N, 4, seed=70 + T, identity_src=ident, routing_seed=71 + T)
    pad = []
    for t in (c.s_d, c.b_d):
        buf = torch.empty((t.numel() + 1,), dtype=torch.bfloat16, device="cuda")
        v = buf[1:].view(t.shape)   # 2 bytes past a 16-byte boundary
        v.copy_(t)
        pad.append(v)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    y = _mxq().gather_qmm(c.x_d, c.w_d, pad[0], pad[1], c.ids_d, c.src_d, 4, dev_status=status)
    yr, bnd = oracle.gather_qmm(c.x, c.w, c.s, c.b, c.ids, c.src, c.T, c.B, c.E, c.K, c.N, 4)
    assert_close(to_f64(y), yr, bnd, "gather decode, direct form")
    assert int(status.item()) == 0


@pytest.mark.parametrize("group", [32, 128])
def test_gather_decode_group_sizes(group):
    c = MoECase(6, 16, 4, 1024, 200, 4, seed=61, routing_seed=62, group=group)
    y = _mxq().gather_qmm(c.x_d, c.w_d, c.s_d, c.b_d, c.ids_d, c.src_d, 4, group_size=group)
    yr, bnd = oracle.gather_qmm(c.x, c.w, c.s, c.b, c.ids, c.src, c.T, c.B, c.E, c.K, c.N, 4,
                                group)
    assert_close(to_f64(y), yr, bnd, "gather decode G=%d" % group)


def test_gather_decode_hot_expert():
    # one expert takes 20 of 24 rows
    c = MoECase(24, 4, 1, 512, 130, 4, seed=63, identity_src=True)
    ids = np.array([0, 1] + [2] * 20 + [3, 3], np.int32)
    c.ids = ids
    c.ids_d = i32_dev(ids)
    y = _mxq().gather_qmm(c.x_d, c.w_d, c.s_d, c.b_d, c.ids_d, None, 4)
    yr, bnd = oracle.gather_qmm(c.x, c.w, c.s, c.b, ids, None, c.T, c.B, c.E, c.K, c.N, 4)
    assert_close(to_f64(y), yr, bnd, "gather decode hot expert")


def test_gather_decode_invalid_rows():
    import torch

    T, E, K, N = 12, 4, 256, 64
    c = MoECase(T, E, 2, K, N, 4, seed=64)
    ids = np.sort(c.ids).copy()
    ids[0] = -1
    ids[-1] = E
    src = c.src.copy()
    src[5] = T + 2
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    out = torch.full((c.B, N), 7.0, dtype=torch.bfloat16, device="cuda")
    _mxq().gather_qmm(c.x_d, c.w_d, c.s_d, c.b_d, i32_dev(ids), i32_dev(src), 4, out=out,
                      dev_status=status)
    st = int(status.item())
    assert st & _mxq().DEV_BAD_EXPERT_ID and st & _mxq().DEV_BAD_ROW_SRC
    y = to_f64(out)
    assert np.all(y[0] == 0) and np.all(y[-1] == 0) and np.all(y[5] == 0)
    good = np.ones(c.B, bool)
    good[[0, 5, c.B - 1]] = False
    yr, bnd = oracle.gather_qmm(c.x, c.w, c.s, c.b, np.clip(ids, 0, E - 1),
                                np.where(good, src, 0), c.T, c.B, c.E, c.K, c.N, 4)
    assert_close(y[good], yr[good], bnd[good], "decode gather with invalid rows")
    # unsorted ids: all zero
    out.fill_(7.0)
    bad = np.array([1, 0] + [2] * (c.B - 2), np.int32)
    _mxq().gather_qmm(c.x_d, c.w_d, c.s_d, c.b_d, i32_dev(bad), c.src_d, 4, out=out,
                      dev_status=status)
    assert int(status.item()) & _mxq().DEV_UNSORTED_IDS
    assert bool((out.float() == 0).all())


def test_gather_decode_constant_per_expert_exact():
    # s = 0, b = c_{e,n} distinct per (e, n), integer x: exact results, so a
    # mis-gathered expert, source row or column shows
    T, E, top_k, K, N = 5, 12, 8, 512, 136
    ids, src = synth.routing(T, E, top_k, seed=71)
    rng = np.random.default_rng(72)
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


def _second_set(c, seed):
    ws, ss, bs = [], [], []
    for e in range(c.E):
        q = synth.quantize(synth.dense_weights(c.N, c.K, seed=seed * 1009 + e), c.bits, c.group)
        ws.append(q.w)
        ss.append(q.scales)
        bs.append(q.biases)
    return np.stack(ws), np.stack(ss), np.stack(bs)


@pytest.mark.parametrize("bits", [4, 8, 2])
@pytest.mark.parametrize("T,K,N,ident", [(4, 2816, 704, False), (32, 704, 2816, True),
                                         (300, 256, 192, False)])
def test_gateup_matches_two_checker_calls(T, K, N, ident, bits):
    import torch

    c = MoECase(T, 64 if T < 300 else 16, 4, K, N, bits, seed=81 + T, identity_src=ident,
                routing_seed=82 + T)
    wu, su, bu = _second_set(c, 83 + T)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    yg, yu = _mxq().gather_qmm_gateup(c.x_d, c.w_d, c.s_d, c.b_d, codes_dev(wu), bf16_dev(su),
                                      bf16_dev(bu), c.ids_d, c.src_d, bits, dev_status=status)
    rg, bg = oracle.gather_qmm(c.x, c.w, c.s, c.b, c.ids, c.src, c.T, c.B, c.E, c.K, c.N, bits)
    ru, bu_ = oracle.gather_qmm(c.x, wu, su, bu, c.ids, c.src, c.T, c.B, c.E, c.K, c.N, bits)
    assert_close(to_f64(yg), rg, bg, "gate T=%d bits=%d" % (T, bits))
    assert_close(to_f64(yu), ru, bu_, "up T=%d bits=%d" % (T, bits))
    assert int(status.item()) == 0
    # each output equals the single-set call bit for bit
    y1 = _mxq().gather_qmm(c.x_d, c.w_d, c.s_d, c.b_d, c.ids_d, c.src_d, bits)
    y2 = _mxq().gather_qmm(c.x_d, codes_dev(wu), bf16_dev(su), bf16_dev(bu), c.ids_d, c.src_d, bits)
    assert torch.equal(yg.view(torch.int16), y1.view(torch.int16))
    assert torch.equal(yu.view(torch.int16), y2.view(torch.int16))


def test_gateup_invalid_ids_zero_both_outputs():
    import torch

    T, E, K, N = 40, 4, 128, 128
    c = MoECase(T, E, 1, K, N, 4, seed=91, identity_src=True)
    ids = np.array([-1] * 3 + [0] * 10 + [1] * 10 + [3] * 12 + [4] * 5, np.int32)
    c.ids = ids
    c.ids_d = i32_dev(ids)
    wu, su, bu = _second_set(c, 92)
    og = torch.full((c.B, N), 7.0, dtype=torch.bfloat16, device="cuda")
    ou = torch.full((c.B, N), 7.0, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    _mxq().gather_qmm_gateup(c.x_d, c.w_d, c.s_d, c.b_d, codes_dev(wu), bf16_dev(su),
                             bf16_dev(bu), c.ids_d, None, 4, out_gate=og, out_up=ou,
                             dev_status=status)
    assert int(status.item()) & _mxq().DEV_BAD_EXPERT_ID
    for y in (to_f64(og), to_f64(ou)):
        assert np.all(y[:3] == 0) and np.all(y[-5:] == 0)
    rg, bg = oracle.gather_qmm(c.x, c.w, c.s, c.b, ids, None, c.T, c.B, c.E, c.K, c.N, 4)
    ru, bu_ = oracle.gather_qmm(c.x, wu, su, bu, ids, None, c.T, c.B, c.E, c.K, c.N, 4)
    assert_close(to_f64(og), rg, bg, "gate with invalid ids")
    assert_close(to_f64(ou), ru, bu_, "up with invalid ids")

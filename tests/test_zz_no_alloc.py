"""mxq_gather_qmm_noalloc (the grouped GEMM with the library's fixed scratch
instead of a caller workspace) against mxq_gather_qmm on the same inputs.

Both run the same kernels, so the results must be identical bit for bit.
Two different problems go through the fixed scratch back to back, so a
second call that read anything left behind by the first would show.  The
file is named to be collected last: it must pass alone and after every
other GPU test has used the device."""

import pytest

from tests.gpu_util import MoECase

pytestmark = pytest.mark.gpu


def _both(case):
    import torch

    import affine_bit_matmul_gb300 as mxq

    ref = mxq.gather_qmm(case.x_d, case.w_d, case.s_d, case.b_d, case.ids_d, case.src_d, case.bits)
    out = torch.full_like(ref, float("nan"))
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    mxq.gather_qmm_noalloc(case.x_d, case.w_d, case.s_d, case.b_d, case.ids_d, case.src_d,
                           case.bits, out, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return ref, out


def _same(a, b):
    import torch

    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("identity", [False, True])
def test_noalloc_matches_workspace_form_twice(identity):
    # two different problems through the fixed scratch, back to back
    c1 = MoECase(T=37, E=6, top_k=3, K=320, N=200, bits=4, seed=31, identity_src=identity)
    c2 = MoECase(T=90, E=11, top_k=2, K=704, N=136, bits=8, seed=32, identity_src=identity,
                 routing_seed=5)
    for case in (c1, c2, c1):
        ref, out = _both(case)
        assert _same(ref, out)


def test_noalloc_workload_shape():
    # the sorted-MoE up projection: 573 tokens, top 8 of 128 experts,
    # K = 2816, N = 704, routed rows (scratch 24.6 MB of the 32 MiB)
    case = MoECase(T=573, E=128, top_k=8, K=2816, N=704, bits=4, seed=33)
    ref, out = _both(case)
    assert _same(ref, out)
    ref2, out2 = _both(case)
    assert _same(ref2, out2) and _same(out, out2)


def test_noalloc_against_oracle_twice():
    # the fixed-scratch form checked directly against the f64 checker, on two
    # calls in a row (the second finds the first call's scratch contents)
    import oracle
    from tests.gpu_util import assert_close, to_f64

    case = MoECase(T=70, E=9, top_k=3, K=448, N=160, bits=4, seed=34)
    yr, bnd = oracle.gather_qmm(case.x, case.w, case.s, case.b, case.ids, case.src, case.T,
                                case.B, case.E, case.K, case.N, case.bits)
    for _ in range(2):
        _, out = _both(case)
        assert_close(to_f64(out), yr, bnd, "gather_qmm_noalloc vs oracle")


def test_noalloc_decode_sized_call():
    # a decode step: 3 tokens x top 8 of 128 experts (24 sorted rows), against
    # the workspace form bit for bit and against the f64 checker
    import oracle
    from tests.gpu_util import assert_close, to_f64

    case = MoECase(T=3, E=128, top_k=8, K=2816, N=704, bits=4, seed=35, routing_seed=6)
    assert case.B <= 32
    yr, bnd = oracle.gather_qmm(case.x, case.w, case.s, case.b, case.ids, case.src, case.T,
                                case.B, case.E, case.K, case.N, case.bits)
    for _ in range(2):
        ref, out = _both(case)
        assert _same(ref, out)
        assert_close(to_f64(out), yr, bnd, "decode-sized gather_qmm_noalloc vs oracle")


def test_noalloc_refuses_oversized_request():
    import torch

    import affine_bit_matmul_gb300 as mxq

    # routed rows needing more than the fixed scratch: refused, nothing written
    T, K, N, E = 3000, 8192, 64, 2
    x = torch.zeros((T, K), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((E, N, K // 8), dtype=torch.int32, device="cuda")
    s = torch.zeros((E, N, K // 64), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((T,), dtype=torch.int32, device="cuda")
    src = torch.arange(T, dtype=torch.int32, device="cuda")
    out = torch.full((T, N), 7.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mxq.MxqError) as e:
        mxq.gather_qmm_noalloc(x, w, s, s, ids, src, 4, out)
    assert e.value.status == 7
    assert bool((out == 7.0).all())
    assert mxq.gather_workspace_bytes(T, E, K, N) > mxq.NOALLOC_SCRATCH_BYTES

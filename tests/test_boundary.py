"""Host-side tests of the C ABI (no GPU needed): the library builds, loads and
exports every function ``include/mxq.h`` declares, and argument checks
return the documented status codes before anything touches a device."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxq.h")


@pytest.fixture(scope="module")
def L():
    from affine_bit_matmul_gb300 import build

    build.build()
    import affine_bit_matmul_gb300 as mxq

    return mxq.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mxq_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("mxq_qmv", "mxq_qmm", "mxq_qmv_kn", "mxq_qmm_kn", "mxq_gather_qmm",
              "mxq_gather_qmm_kn", "mxq_gather_qmm_gateup", "mxq_gather_workspace_bytes",
              "mxq_gather_qmm_noalloc", "mxq_quantize", "mxq_status_string", "mxq_version",
              "mxq_debug_set_wait_budget"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    import affine_bit_matmul_gb300 as mxq

    for name in declared_functions():
        assert hasattr(L, name), name
        assert name in mxq.EXPORTED_SYMBOLS or name.startswith("mxq_")


def test_status_strings(L):
    for code in range(0, 8):
        s = L.mxq_status_string(code).decode()
        assert s and s != "unknown status"
    assert L.mxq_status_string(99).decode() == "unknown status"
    assert L.mxq_version() >= 100


FAKE = ctypes.c_void_p(0x10000)       # 16-byte aligned, never dereferenced
FAKE_ODD = ctypes.c_void_p(0x10008)   # 8-byte aligned only


def qmv(L, x=FAKE, w=FAKE, s=FAKE, b=FAKE, y=FAKE, K=128, N=64, bits=4, group=64, status=None):
    return L.mxq_qmv(x, w, s, b, y, K, N, bits, group, status, None)


@pytest.mark.parametrize("kw,code", [
    (dict(bits=5), 1), (dict(bits=16), 1), (dict(bits=1), 1), (dict(bits=7), 1),
    (dict(bits=3, K=192), 1), (dict(group=16), 1),
    (dict(group=48), 1), (dict(group=256), 1), (dict(group=0), 1), (dict(group=128, K=192), 1),
    (dict(group=32, K=96), 1), (dict(K=100), 1), (dict(K=0), 1), (dict(K=-64), 1), (dict(N=0), 1),
    (dict(x=None), 1), (dict(w=None), 1), (dict(s=None), 1), (dict(b=None), 1), (dict(y=None), 1),
    (dict(x=FAKE_ODD), 2), (dict(w=FAKE_ODD), 2), (dict(y=FAKE_ODD), 2),
    (dict(s=ctypes.c_void_p(0x10001)), 2), (dict(status=ctypes.c_void_p(0x10002)), 2),
])
def test_qmv_argument_checks(L, kw, code):
    assert qmv(L, **kw) == code


def qmv_kn(L, K=100, N=128, bits=4, group=64, x=FAKE, w=FAKE, y=FAKE, status=None):
    return L.mxq_qmv_kn(x, w, FAKE, FAKE, y, K, N, bits, group, status, None)


@pytest.mark.parametrize("kw,code", [
    (dict(bits=3), 3), (dict(bits=6), 3), (dict(bits=5), 1), (dict(group=16), 1),
    (dict(N=96), 1), (dict(N=0), 1), (dict(K=0), 1), (dict(N=64, group=128), 1),
    (dict(x=None), 1), (dict(w=None), 1), (dict(y=FAKE_ODD), 2), (dict(w=FAKE_ODD), 2),
    (dict(status=ctypes.c_void_p(0x10002)), 2),
])
def test_qmv_kn_argument_checks(L, kw, code):
    assert qmv_kn(L, **kw) == code


def qmm_kn(L, M=16, K=200, N=128, bits=4, group=64, x=FAKE, w=FAKE, y=FAKE, status=None):
    return L.mxq_qmm_kn(x, w, FAKE, FAKE, y, M, K, N, bits, group, status, None)


@pytest.mark.parametrize("kw,code", [
    (dict(bits=3), 3), (dict(bits=6), 3), (dict(bits=5), 1), (dict(group=16), 1),
    (dict(N=96), 1), (dict(N=0), 1), (dict(K=0), 1), (dict(M=0), 1), (dict(K=100), 1),
    (dict(N=64, group=128), 1), (dict(x=None), 1), (dict(w=None), 1), (dict(y=FAKE_ODD), 2),
    (dict(w=FAKE_ODD), 2), (dict(x=FAKE_ODD), 2), (dict(status=ctypes.c_void_p(0x10002)), 2),
])
def test_qmm_kn_argument_checks(L, kw, code):
    assert qmm_kn(L, **kw) == code


def test_qmm_kn_single_row_takes_any_k(L):
    # M = 1 is the [K, N] GEMV, which takes any K > 0: the host checks pass
    # and only the device check remains
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the GPU tests")
    assert qmm_kn(L, M=1, K=100) in (4, 5)


def gather_kn(L, T=8, B=8, E=2, K=128, N=64, bits=4, group=64, ids=FAKE, src=FAKE, ws=FAKE,
              wsb=1 << 24):
    return L.mxq_gather_qmm_kn(FAKE, FAKE, FAKE, FAKE, ids, src, FAKE, T, B, E, K, N, bits, group,
                               ws, wsb, None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(bits=3), 3), (dict(bits=6), 3), (dict(bits=7), 1), (dict(T=0), 1), (dict(B=0), 1),
    (dict(E=0), 1), (dict(K=100), 1), (dict(N=96), 1), (dict(N=64, group=128), 1),
    (dict(ids=None), 1), (dict(src=None, T=5, B=8), 1),
    (dict(ids=ctypes.c_void_p(0x10002)), 2), (dict(ws=ctypes.c_void_p(0x10080)), 2),
    (dict(ws=None), 6), (dict(wsb=16), 6),
])
def test_gather_kn_argument_checks(L, kw, code):
    assert gather_kn(L, **kw) == code


def qmm(L, M=16, K=128, N=64, bits=4, group=64, status=None, x=FAKE, y=FAKE):
    return L.mxq_qmm(x, FAKE, FAKE, FAKE, y, M, K, N, bits, group, status, None)


@pytest.mark.parametrize("kw,code", [
    (dict(M=0), 1), (dict(M=-1), 1), (dict(bits=5), 1), (dict(group=16), 1), (dict(K=96), 1),
    (dict(group=96), 1), (dict(group=128, K=320), 1),
    (dict(x=None), 1), (dict(x=FAKE_ODD), 2), (dict(y=FAKE_ODD), 2),
    (dict(status=ctypes.c_void_p(0x10002)), 2),
])
def test_qmm_argument_checks(L, kw, code):
    assert qmm(L, **kw) == code


def gather(L, T=8, B=8, E=2, K=128, N=64, bits=4, group=64, ids=FAKE, src=FAKE, ws=FAKE,
           wsb=1 << 24):
    return L.mxq_gather_qmm(FAKE, FAKE, FAKE, FAKE, ids, src, FAKE, T, B, E, K, N, bits, group,
                            ws, wsb, None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(T=0), 1), (dict(B=0), 1), (dict(E=0), 1), (dict(bits=7), 1), (dict(K=65), 1),
    (dict(bits=3, K=64), 1),
    (dict(group=64 + 32), 1), (dict(group=128, K=192), 1),
    (dict(ids=None), 1), (dict(src=None, T=5, B=8), 1),
    (dict(ids=ctypes.c_void_p(0x10002)), 2), (dict(ws=ctypes.c_void_p(0x10080)), 2),
    (dict(ws=None), 6), (dict(wsb=16), 6),
])
def test_gather_argument_checks(L, kw, code):
    assert gather(L, **kw) == code


def test_workspace_sizes(L):
    n0 = L.mxq_gather_workspace_bytes(4584, 128, 0, 704)
    # one 16-byte tile record per possible tile plus the count
    assert n0 >= (4584 // 128 + 128) * 16
    # with routed rows it also holds the sorted activation copy
    n1 = L.mxq_gather_workspace_bytes(4584, 128, 2816, 704)
    assert n1 >= n0 + 4584 * 2816 * 2
    assert L.mxq_gather_workspace_bytes(0, 4, 64, 4) == 0


def test_valid_call_without_sm103_device_reports_device_error(L):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the GPU tests")
    # arguments pass the host checks; the device check must then refuse
    assert qmv(L) in (4, 5)


def test_noalloc_scratch_limit_refused_before_device(L):
    import affine_bit_matmul_gb300 as mxq

    text = open(HEADER).read()
    m = re.search(r"#define MXQ_NOALLOC_SCRATCH_BYTES \((\d+)u \* 1024u \* 1024u\)", text)
    assert m and int(m.group(1)) * 2 ** 20 == mxq.NOALLOC_SCRATCH_BYTES
    # 100000 routed rows of K = 8192 need 1.6 GB of scratch: refused with
    # MXQ_ERR_SCRATCH_LIMIT before any device is touched (this runs on hosts
    # without a GPU too)
    rc = L.mxq_gather_qmm_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 100000, 100000, 8,
                                  8192, 64, 4, 64, None, None)
    assert rc == 7
    # without row_src only the tile table is needed: the same B fits
    need = L.mxq_gather_workspace_bytes(100000, 8, 0, 64)
    assert 0 < need <= mxq.NOALLOC_SCRATCH_BYTES
    # the routed up projection of the sorted-MoE workload fits
    assert L.mxq_gather_workspace_bytes(4584, 128, 2816, 704) <= mxq.NOALLOC_SCRATCH_BYTES


def quantize(L, w=FAKE, codes=FAKE, s=FAKE, b=FAKE, N=16, K=128, bits=4, group=64):
    return L.mxq_quantize(w, codes, s, b, N, K, bits, group, None)


@pytest.mark.parametrize("kw,code", [
    (dict(bits=5), 1), (dict(bits=3, K=64), 1), (dict(group=16), 1), (dict(group=256), 1),
    (dict(group=128, K=192), 1),
    (dict(K=100), 1), (dict(N=0), 1), (dict(w=None), 1),
    (dict(codes=None), 1), (dict(w=FAKE_ODD), 2), (dict(codes=FAKE_ODD), 2),
    (dict(s=ctypes.c_void_p(0x10001)), 2),
])
def test_quantize_argument_checks(L, kw, code):
    assert quantize(L, **kw) == code


def test_wrapper_refuses_a_stream_of_another_device():
    # every Python wrapper makes the tensors' device current for the call and
    # refuses a stream that belongs to another device (that pairing would
    # launch one device's kernels on another device's pointers); the check
    # runs before anything touches a GPU
    import torch

    import affine_bit_matmul_gb300 as mxq

    class FakeStream:
        device = torch.device("cuda", 1)
        cuda_stream = 0

    with pytest.raises(ValueError, match="stream is on cuda:1"):
        mxq._launch_on(torch.device("cuda", 0), FakeStream())


def test_bench_reference_arm_uses_the_same_config():
    # both arms of bench.py print the identical config dict
    import sys

    sys.path.insert(0, ROOT)
    import bench

    src = open(os.path.join(ROOT, "bench.py")).read()
    ref = src[src.index("def run_reference"):src.index("def run_profile")]
    assert '"config": CONFIG' in ref
    assert bench.CONFIG["workload"] == bench.WORKLOAD


def test_wait_budget_setter_clamps(L):
    # the pipeline-wait budget is host state (no device needed): values in
    # (0, default] are taken, anything else restores the default
    default = 2_000_000_000
    try:
        assert L.mxq_debug_set_wait_budget(1000) == 1000
        assert L.mxq_debug_set_wait_budget(default) == default
        assert L.mxq_debug_set_wait_budget(10 ** 12) == default
        assert L.mxq_debug_set_wait_budget(1) == 1
        assert L.mxq_debug_set_wait_budget(-5) == default
    finally:
        assert L.mxq_debug_set_wait_budget(0) == default

"""The C ABI on the host (no GPU): the library loads, exports every function
that include/qgemv.h declares, and refuses bad arguments before touching any
pointer (poison pointers that would fault if dereferenced)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qgemv.h")


@pytest.fixture(scope="module")
def qg():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "qgemv_build", os.path.join(ROOT, "weight_only_quantized_i4g_gb300", "_build.py"))
    build_script = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(build_script)
    build_script.build()
    import weight_only_quantized_i4g_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:[a-z_0-9]+\s+)+\*?\s*(q[a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_header_lists_the_entry_points():
    names = declared_functions()
    for must in ["qgemv_i4g", "qgemv_fp8b128", "qgemv_mq4v2", "qgemm_i4g", "qgemm_fp8b128", "qgemm_mq4v2",
                 "qg_workspace_bytes", "qg_gemm_workspace_bytes", "qg_device_status",
                 "qg_strerror", "qg_last_error", "qg_quantize_i4g", "qg_encode_mq4v2", "qg_fwht256",
                 "qgemv_moe", "qgemm_moe", "qgemv_q2_0", "qg_launch_count", "qgemv_i4g_noalloc",
                 "qg_selftest_wait_timeout", "qg_stamps_take", "qg_selftest_pdl_chain"]:
        assert must in names, names


def test_library_exports_every_declared_symbol(qg):
    lib = ctypes.CDLL(qg.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(qg.EXPORTED)


def test_strerror(qg):
    for code in range(0, -10, -1):
        assert qg.strerror(code).startswith("QG_")
    assert "unknown" in qg.strerror(-99)


POISON = 0xDEADBEE0     # 16-byte aligned, never mapped: a dereference would fault


def test_i4g_refusals(qg):
    P = POISON
    assert qg.qgemv_i4g(P, P, P, P, 1, 512, 256, 3, stream=0) == qg.QG_EGS
    assert "gs = 3" in qg.last_error()
    assert qg.qgemv_i4g(P, P, P, P, 1, 512, 256, 0, stream=0) == qg.QG_EGS
    assert qg.qgemv_i4g(P, P, P, P, 0, 512, 256, 64, stream=0) == qg.QG_EINVAL
    assert qg.qgemv_i4g(P, P, P, P, 1, 0, 256, 64, stream=0) == qg.QG_EINVAL
    assert qg.qgemv_i4g(P, P, P, P, 1, 512, -5, 64, stream=0) == qg.QG_EINVAL
    assert qg.qgemv_i4g(P, P, 0, P, 1, 512, 256, 64, stream=0) == qg.QG_EINVAL
    assert qg.qgemv_i4g(P + 2, P, P, P, 1, 512, 256, 64, stream=0) == qg.QG_EALIGN
    assert qg.qgemv_i4g(P, P, P, P + 1, 1, 512, 256, 64, stream=0) == qg.QG_EALIGN
    assert qg.qgemv_i4g(P, P, P, P, 1, 512, 256, 64, ws=P + 16, stream=0) == qg.QG_EALIGN


def test_i4g_noalloc_refusals(qg):
    P = POISON
    assert qg.qgemv_i4g_noalloc(P, P, P, P, 1, 512, 256, 3, stream=0) == qg.QG_EGS
    assert qg.qgemv_i4g_noalloc(P, P, 0, P, 1, 512, 256, 64, stream=0) == qg.QG_EINVAL
    assert qg.qgemv_i4g_noalloc(P + 2, P, P, P, 1, 512, 256, 64, stream=0) == qg.QG_EALIGN
    # a shape whose split-reduction scratch exceeds the fixed 4 MiB
    assert qg.qg_workspace_bytes(qg.QG_FMT_I4G, 8, 65536, 16384, 64) > (4 << 20)
    assert qg.qgemv_i4g_noalloc(P, P, P, P, 8, 65536, 16384, 64, stream=0) == qg.QG_EWORKSPACE
    assert "4194304" in qg.last_error()


def test_fp8_refusals(qg):
    P = POISON
    assert qg.qgemv_fp8b128(P, P, P, P, 1, 0, 1, stream=0) == qg.QG_EINVAL
    assert qg.qgemv_fp8b128(P, P + 1, P, P, 1, 16, 1, stream=0) == qg.QG_EALIGN
    assert qg.qgemv_fp8b128(0, P, P, P, 1, 16, 1, stream=0) == qg.QG_EINVAL


def test_mq4_refusals(qg):
    P = POISON
    assert qg.qgemv_mq4v2(P, P, P, 1, 300, 4, stream=0) == qg.QG_ESHAPE
    assert "300" in qg.last_error()
    assert qg.qgemv_mq4v2(P, P, P + 4, 1, 256, 4, stream=0) == qg.QG_EALIGN
    assert qg.qgemv_mq4v2(P, P, P, 1, 256, 0, stream=0) == qg.QG_EINVAL


def test_fp8ue8m0_refusals(qg):
    P = POISON
    assert qg.qgemv_fp8ue8m0(P, P, P, None, 1, 256, 4, stream=0) == qg.QG_EINVAL
    assert qg.qgemv_fp8ue8m0(P, P + 1, P, P + 1, 1, 256, 4, stream=0) == qg.QG_EALIGN   # x odd; scales any
    assert qg.qgemv_fp8ue8m0(P, P, P, P, 1, 256, 0, stream=0) == qg.QG_EINVAL
    assert qg.qgemm_fp8ue8m0(P, P, P, P, 0, 256, 4, stream=0) == qg.QG_EINVAL
    assert qg.qgemm_fp8ue8m0(P + 2, P, P, P, 4, 256, 4, stream=0) == qg.QG_EALIGN


def test_q2_0_refusals(qg):
    P = POISON
    assert qg.qgemv_q2_0(P, P, P, 1, 100, 4, stream=0) == qg.QG_ESHAPE
    assert "100" in qg.last_error()
    assert qg.qgemv_q2_0(P, P, P + 1, 1, 128, 4, stream=0) == qg.QG_EALIGN
    assert qg.qgemv_q2_0(P, P, None, 1, 128, 4, stream=0) == qg.QG_EINVAL
    assert qg.qgemv_q2_0(P, P, P, 0, 128, 4, stream=0) == qg.QG_EINVAL


def test_moe_refusals(qg):
    P = POISON
    moe = qg.qgemv_moe
    assert moe(4, P, P, 0, P, 4, P, 2, 9, 256, 64, 64, stream=0) == qg.QG_EINVAL      # S > 8
    assert "S = 9" in qg.last_error()
    assert moe(5, P, P, 0, P, 4, P, 2, 1, 256, 64, 64, stream=0) == qg.QG_EINVAL      # no such format
    assert moe(4, P, P, 0, P, 4, P, 2, 1, 256, 64, 7, stream=0) == qg.QG_EGS
    assert moe(44, P, P, 0, P, 4, P, 2, 1, 300, 64, 0, stream=0) == qg.QG_ESHAPE
    assert moe(4, P, P, 0, P, 0, P, 2, 1, 256, 64, 64, stream=0) == qg.QG_EINVAL      # empty table
    assert moe(4, P, P, 0, P, 4, P, -1, 1, 256, 64, 64, stream=0) == qg.QG_EINVAL     # negative slots
    assert moe(4, P, P, 0, P, 4, P, 70000, 1, 256, 64, 64, stream=0) == qg.QG_EINVAL  # grid.z limit
    assert moe(4, P, None, 0, P, 4, P, 2, 1, 256, 64, 64, stream=0) == qg.QG_EINVAL
    assert moe(4, P, P + 8, 0, P, 4, P, 2, 1, 256, 64, 64, stream=0) == qg.QG_EALIGN  # x not 16-byte aligned
    assert moe(4, P, P, 258, P, 4, P, 2, 1, 256, 64, 64, stream=0) == qg.QG_EALIGN    # 1032-byte slot stride
    assert moe(4, P, P, 100, P, 4, P, 2, 1, 256, 64, 64, stream=0) == qg.QG_EINVAL    # slots overlap
    assert moe(4, P, P, 0, P + 4, 4, P, 2, 1, 256, 64, 64, stream=0) == qg.QG_EALIGN  # table alignment
    assert moe(4, P, P, 0, P, 4, P, 0, 1, 256, 64, 64, stream=0) == qg.QG_OK          # nothing to do


def test_moe_gemm_refusals(qg):
    P = POISON
    tab = qg.expert_table([(P, P), (P, P)])
    mm = qg.qgemm_moe
    assert mm(5, P, P, tab, 2, [0], [0, 4], 1, 256, 64, 64, stream=0) == qg.QG_EINVAL      # no such format
    assert mm(4, P, P, tab, 2, [2], [0, 4], 1, 256, 64, 64, stream=0) == qg.QG_EINVAL      # expert 2 of 2
    assert "expert 2" in qg.last_error()
    assert mm(4, P, P, tab, 2, [0, 1], [0, 4, 3], 2, 256, 64, 64, stream=0) == qg.QG_EINVAL  # offsets decrease
    assert mm(4, P, P, tab, 2, [0], [-1, 4], 1, 256, 64, 64, stream=0) == qg.QG_EINVAL     # negative offset
    assert mm(4, P, P, tab, 0, [0], [0, 4], 1, 256, 64, 64, stream=0) == qg.QG_EINVAL      # empty table
    assert mm(4, P, P, tab, 2, [0], [0, 4], -1, 256, 64, 64, stream=0) == qg.QG_EINVAL     # negative groups
    assert mm(4, None, P, tab, 2, [0], [0, 4], 1, 256, 64, 64, stream=0) == qg.QG_EINVAL
    assert mm(4, P, P, tab, 2, [0, 1], [3, 3, 3], 2, 256, 64, 64, stream=0) == qg.QG_OK      # only empty groups
    assert mm(4, P, P, tab, 2, [], [0], 0, 256, 64, 64, stream=0) == qg.QG_OK


def test_gemm_and_prep_refusals(qg):
    P = POISON
    assert qg.qgemm_i4g(P, P, P, P, 0, 64, 64, 64, stream=0) == qg.QG_EINVAL
    assert qg.qgemm_i4g(P, P, P, P, 4, 64, 64, 7, stream=0) == qg.QG_EGS
    assert qg.qgemm_fp8b128(P, P, P, P, 4, 0, 64, stream=0) == qg.QG_EINVAL
    assert qg.qgemm_fp8b128(P, P, 0, P, 4, 64, 64, stream=0) == qg.QG_EINVAL
    assert qg.qgemm_fp8b128(P, P + 1, P, P, 4, 64, 64, stream=0) == qg.QG_EALIGN
    assert qg.qgemm_fp8b128(P, P, P, P + 2, 4, 64, 64, stream=0) == qg.QG_EALIGN
    assert qg.qgemm_mq4v2(P, P, P, 4, 300, 64, stream=0) == qg.QG_ESHAPE
    assert qg.qgemm_mq4v2(P, P, P + 4, 4, 256, 64, stream=0) == qg.QG_EALIGN
    assert qg.qgemm_mq4v2(P, P, P, 4, 256, 64, ws=P + 16, stream=0) == qg.QG_EALIGN
    assert qg.qgemm_mq4v2(P, P, P, 4, 256, 0, stream=0) == qg.QG_EINVAL
    assert qg.qg_quantize_i4g(P, P, P, 4, 64, 5, stream=0) == qg.QG_EGS
    assert qg.qg_encode_mq4v2(P, P, 4, 100, stream=0) == qg.QG_ESHAPE
    assert qg.qg_fwht256(P, P, P, 0, stream=0) == qg.QG_EINVAL


def test_workspace_query_is_pure(qg):
    # no split for these decode shapes of the workloads
    assert qg.qg_workspace_bytes(qg.QG_FMT_I4G, 1, 7168, 2048, 64) == 0
    assert qg.qg_workspace_bytes(qg.QG_FMT_FP8B128, 1, 16384, 7168) == 0
    assert qg.qg_workspace_bytes(qg.QG_FMT_MQ4V2, 1, 5120, 17408) == 0
    # 17408 MQ4 columns are more than one block's warps hold: the reduction
    # splits, splits * S * O floats
    n = qg.qg_workspace_bytes(qg.QG_FMT_MQ4V2, 1, 17408, 5120)
    assert n > 0 and n % (5120 * 4) == 0
    # a short-O / long-I shape splits the reduction and needs splits*S*O floats
    n = qg.qg_workspace_bytes(qg.QG_FMT_I4G, 1, 16384, 64, 64)
    assert n > 0 and n % (64 * 4) == 0
    # invalid arguments -> 0
    assert qg.qg_workspace_bytes(qg.QG_FMT_MQ4V2, 1, 300, 4) == 0
    assert qg.qg_workspace_bytes(99, 1, 256, 4) == 0


def test_gemm_workspace_query(qg):
    # tensor-core shapes of every format: counters + partial slots, 256-byte multiple
    for fmt, gs in ((qg.QG_FMT_I4G, 64), (qg.QG_FMT_FP8B128, 0), (qg.QG_FMT_MQ4V2, 0)):
        n = qg.qg_gemm_workspace_bytes(fmt, 512, 7168, 2048, gs)
        assert n > 0 and n % 256 == 0, (fmt, n)
    # shapes that run the general kernel need none
    assert qg.qg_gemm_workspace_bytes(qg.QG_FMT_I4G, 64, 1000, 256, 64) == 0
    assert qg.qg_gemm_workspace_bytes(qg.QG_FMT_FP8B128, 64, 1000, 256) == 0
    assert qg.qg_gemm_workspace_bytes(qg.QG_FMT_MQ4V2, 64, 300, 256) == 0
    assert qg.qg_gemm_workspace_bytes(qg.QG_FMT_MQ4V2, 0, 256, 256) == 0


def test_selftest_refusals(qg):
    """Bad arguments are refused on the host, before any launch."""
    lib = ctypes.CDLL(qg.LIB_PATH)
    lib.qg_selftest_wait_timeout.argtypes = [ctypes.c_int, ctypes.c_void_p]
    v = ctypes.c_int(0)
    assert lib.qg_selftest_wait_timeout(1024, None) == qg.QG_EINVAL
    assert lib.qg_selftest_wait_timeout(0, ctypes.byref(v)) == qg.QG_EINVAL
    assert lib.qg_selftest_wait_timeout((1 << 22) + 1, ctypes.byref(v)) == qg.QG_EINVAL
    assert "spin_limit" in qg.last_error()


def test_profiling_aid_refusals(qg):
    """The stamps reader refuses bad arguments, and refuses outright in the
    normal build (which records no stamps); the launch chain refuses bad
    launch shapes before any launch."""
    n0 = qg.qg_launch_count()
    lib = ctypes.CDLL(qg.LIB_PATH)
    lib.qg_stamps_take.argtypes = [ctypes.c_void_p, ctypes.c_int]
    buf = (ctypes.c_uint64 * 8)()
    assert lib.qg_stamps_take(None, 1) == qg.QG_EINVAL
    assert lib.qg_stamps_take(buf, 0) == qg.QG_EINVAL
    rc, _ = qg.qg_stamps_take(1)
    assert rc == qg.QG_EINVAL and "without stamps" in qg.last_error()
    for blocks, threads, launches in [(0, 256, 1), (65536, 256, 1), (152, 31, 1), (152, 48, 1), (152, 2048, 1),
                                      (152, 256, 0), (152, 256, 100001)]:
        assert qg.qg_selftest_pdl_chain(blocks, threads, launches, 0) == qg.QG_EINVAL
    assert "launches" in qg.last_error()
    assert qg.qg_launch_count() == n0

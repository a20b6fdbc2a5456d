"""The stamps build (-DQG_STAMPS, the profiling build behind `bench.py
--stamps`) and the launch-chain floor (needs a GPU).

In the stamps build every block of a staged or warp-MMA decode GEMV records
its timeline after the device error word.  The results must still match the
oracle, each block's stamps must come in the order the kernel passes them,
every stamping block must have run at least one row batch, and the error
word must stay clean.  The launch chain behind the floor measurement must
run and leave the error word clean too."""
import ctypes
import importlib.util
import os

import pytest

from gpu_util import compare, dev, host, i4g_inputs, mq4_inputs, orc, out, par_rows, torch, workspace

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ENTRY, WAIT, XREADY, FIRST, CONSUMED, STORED, BATCHES, GLOBAL = range(8)


@pytest.fixture(scope="module")
def qg():
    import weight_only_quantized_i4g_gb300 as m
    return m


@pytest.fixture(scope="module")
def st(qg):
    spec = importlib.util.spec_from_file_location(
        "qgemv_build", os.path.join(ROOT, "weight_only_quantized_i4g_gb300", "_build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    lib = ctypes.CDLL(b.build_stamps())
    for name, (args, res) in qg._SIGNATURES.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


def status_clean(qg, lib):
    s = ctypes.c_int(0)
    assert lib.qg_device_status(ctypes.byref(s)) == qg.QG_OK
    assert s.value == qg.QG_OK, f"device status {s.value} ({qg.strerror(s.value)})"


def check_timelines(qg, lib):
    rc, blocks = qg.qg_stamps_take(qg.STAMP_BLOCKS, lib=lib)
    assert rc == qg.QG_OK
    stamped = [b for b in blocks if b[ENTRY] != 0]
    assert stamped, "no block stamped its start"
    for b in stamped:
        assert b[BATCHES] >= 1
        assert b[ENTRY] <= b[WAIT] <= b[XREADY] <= b[FIRST] <= b[CONSUMED], b
        assert b[STORED] >= b[ENTRY] and b[GLOBAL] > 0, b
    rc, again = qg.qg_stamps_take(qg.STAMP_BLOCKS, lib=lib)
    assert rc == qg.QG_OK and all(w == 0 for b in again for w in b), "take must clear the stamps"
    return stamped


@pytest.mark.parametrize("O,I,S", [(2048, 7168, 1),    # staged kernel, one block per SM
                                   (7168, 2048, 1),    # staged kernel, several blocks per SM
                                   (300, 2048, 2)])    # warp-MMA kernel
def test_stamps_build_i4g(qg, st, O, I, S):
    gs = 64
    x, wq, sc = i4g_inputs(O, I, S, gs, tag=O + S)
    ws, nws = workspace(qg, qg.QG_FMT_I4G, S, I, O, gs)
    y = out(S, O)
    xd, wd, sd = dev(x), dev(wq), dev(sc)          # alive until the kernel has run
    s = torch().cuda.current_stream().cuda_stream
    assert st.qgemv_i4g(y.data_ptr(), xd.data_ptr(), wd.data_ptr(), sd.data_ptr(), S, I, O, gs,
                        None if ws is None else ws.data_ptr(), nws, s) == qg.QG_OK
    got = host(y, S, O)
    ref, mag = par_rows(orc().qgemv_i4g, O, x, wq, sc, S, I, O, gs)
    compare(got, ref, mag, what=f"stamps build fmt4 {O}x{I} S={S}")
    check_timelines(qg, st)
    status_clean(qg, st)


def test_stamps_build_mq4_mma(qg, st):
    O, I, S = 17408, 5120, 1          # warp-MMA kernel at one token
    x, blocks = mq4_inputs(O, I, S, tag=5)
    ws, nws = workspace(qg, qg.QG_FMT_MQ4V2, S, I, O)
    y = out(S, O)
    xd, bd = dev(x), dev(blocks)                   # alive until the kernel has run
    s = torch().cuda.current_stream().cuda_stream
    assert st.qgemv_mq4v2(y.data_ptr(), xd.data_ptr(), bd.data_ptr(), S, I, O,
                          None if ws is None else ws.data_ptr(), nws, s) == qg.QG_OK
    got = host(y, S, O)
    ref, mag = par_rows(orc().qgemv_mq4v2, O, x, blocks, S, I, O)
    compare(got, ref, mag, what="stamps build MQ4-V2 17408x5120")
    stamped = check_timelines(qg, st)
    assert sum(b[BATCHES] for b in stamped) == O // 16      # 16-row batches, every one run once
    status_clean(qg, st)


def test_pdl_chain_floor_runs(qg):
    t = torch()
    s = t.cuda.Stream()
    n0 = qg.qg_launch_count()
    assert qg.qg_selftest_pdl_chain(152, 256, 500, s.cuda_stream) == qg.QG_OK
    assert qg.qg_launch_count() - n0 == 500
    s.synchronize()
    st_word = ctypes.c_int(0)
    assert qg._lib.qg_device_status(ctypes.byref(st_word)) == qg.QG_OK and st_word.value == qg.QG_OK

"""The decode GEMVs built with index guards (-DQG_BOUNDS_CHECK; the stand-in
for a memory checker, which this GPU pool does not offer).  In that build every
global index a decode kernel forms -- a weight row and the byte range of a
unit or a staged segment inside it, a scale or header, an activation unit, an
output element -- is checked against its array; a failed guard records
QG_EBOUNDS in the device error word and skips the access.  Tiny odd shapes
through every decode path (general, direct, staged, warp-MMA, split reduction,
routed experts) must match the oracle and leave the error word clean."""
import ctypes
import importlib.util
import os

import numpy as np
import pytest

import synth
from gpu_util import compare, dev, fp8_inputs, host, i4g_inputs, mq4_inputs, orc, out, par_rows, torch, workspace

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def qg():
    import weight_only_quantized_i4g_gb300 as m
    return m


@pytest.fixture(scope="module")
def bc(qg):
    spec = importlib.util.spec_from_file_location(
        "qgemv_build", os.path.join(ROOT, "weight_only_quantized_i4g_gb300", "_build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    lib = ctypes.CDLL(b.build_bounds_check())
    for name, (args, res) in qg._SIGNATURES.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


def status_clean(qg, bc):
    st = ctypes.c_int(0)
    assert bc.qg_device_status(ctypes.byref(st)) == qg.QG_OK
    assert st.value == qg.QG_OK, f"device status {st.value} ({qg.strerror(st.value)})"


def ptr(t):
    return None if t is None else t.data_ptr()


def stream():
    return torch().cuda.current_stream().cuda_stream


@pytest.mark.parametrize("O,I,S,gs", [(37, 320, 1, 64),     # direct (ceil(I/gs) % 4 != 0)
                                      (33, 1024, 1, 64),    # staged
                                      (33, 1024, 3, 64),    # warp-MMA
                                      (5, 130, 3, 2),       # general kernel
                                      (9, 32768, 1, 64)])   # split reduction
def test_bc_i4g(qg, bc, O, I, S, gs):
    x, wq, sc = i4g_inputs(O, I, S, gs, tag=O + I)
    ws, nws = workspace(qg, qg.QG_FMT_I4G, S, I, O, gs)
    y = out(S, O)
    xd, wd, sd = dev(x), dev(wq), dev(sc)      # kept alive until the kernel has run
    qg.check(bc.qgemv_i4g(ptr(y), ptr(xd), ptr(wd), ptr(sd), S, I, O, gs, ptr(ws), nws, stream()))
    got = host(y, S, O)
    ref, mag = par_rows(orc().qgemv_i4g, O, x, wq, sc, S, I, O, gs)
    compare(got, ref, mag, what=f"bounds-checked fmt4 {O}x{I} S={S}")
    status_clean(qg, bc)


@pytest.mark.parametrize("O,I,S", [(131, 272, 1), (130, 1024, 3), (50, 203, 2), (64, 32768, 1)])
def test_bc_fp8(qg, bc, O, I, S):
    codes, scales, x = fp8_inputs(O, I, S, tag=O + I)
    ws, nws = workspace(qg, qg.QG_FMT_FP8B128, S, I, O)
    y = out(S, O)
    xd, wd, sd = dev(x), dev(codes), dev(scales)
    qg.check(bc.qgemv_fp8b128(ptr(y), ptr(xd), ptr(wd), ptr(sd), S, I, O, ptr(ws), nws, stream()))
    got = host(y, S, O)
    ref, mag = par_rows(orc().qgemv_fp8b128, O, x, codes, scales, S, I, O, step=128)
    compare(got, ref, mag, what=f"bounds-checked fp8 {O}x{I} S={S}")
    status_clean(qg, bc)


@pytest.mark.parametrize("O,I,S", [(7, 768, 5), (33, 1536, 2), (19, 512, 1), (64, 32768, 1)])
def test_bc_mq4v2(qg, bc, O, I, S):
    x, blocks = mq4_inputs(O, I, S, tag=O + I)
    ws, nws = workspace(qg, qg.QG_FMT_MQ4V2, S, I, O)
    y = out(S, O)
    xd, bd = dev(x), dev(blocks)
    qg.check(bc.qgemv_mq4v2(ptr(y), ptr(xd), ptr(bd), S, I, O, ptr(ws), nws, stream()))
    got = host(y, S, O)
    ref, mag = par_rows(orc().qgemv_mq4v2, O, x, blocks, S, I, O)
    compare(got, ref, mag, what=f"bounds-checked MQ4-V2 {O}x{I} S={S}")
    status_clean(qg, bc)


@pytest.mark.parametrize("O,I,S", [(13, 576, 1), (640, 2560, 1), (11, 1024, 3)])
def test_bc_q2_0(qg, bc, O, I, S):
    w = synth.normal(7000 + O, O * I, 0.02).reshape(O, I)
    x = synth.bf16_bits(synth.normal(7500 + O, S * I).astype(np.float32)).reshape(S, I)
    blocks = orc().encode_q2_0(w, O, I)
    ws, nws = workspace(qg, qg.QG_FMT_Q2_0, S, I, O)
    y = out(S, O)
    xd, bd = dev(x), dev(blocks)
    qg.check(bc.qgemv_q2_0(ptr(y), ptr(xd), ptr(bd), S, I, O, ptr(ws), nws, stream()))
    got = host(y, S, O)
    ref, mag = par_rows(orc().qgemv_q2_0, O, x, blocks, S, I, O)
    compare(got, ref, mag, what=f"bounds-checked Q2_0 {O}x{I} S={S}")
    status_clean(qg, bc)


@pytest.mark.parametrize("fmt", [4, 7, 44])
def test_bc_routed_experts(qg, bc, fmt):
    """Routed-expert GEMV (one staged launch over the slots): 4 experts, 5 slots, per-slot x."""
    from test_moe import activations, experts, upload_table
    O, I, S = 130, 1024, 2
    gs = 64 if fmt == 4 else 0
    ws_, ss_ = experts(fmt, 4, O, I, gs, tag=500 + fmt)
    ids = [3, 0, 2, 2, 1]
    n = len(ids)
    x = activations(fmt, n, S, I, 77)
    t = torch()
    ws_d = [dev(w) for w in ws_]
    ss_d = [None if v is None else dev(v) for v in ss_]
    table = upload_table(qg, ws_d, ss_d)
    ids_d = dev(np.asarray(ids, np.int32))
    xd = dev(x)
    y = t.full((n * S * O,), float("nan"), dtype=t.float32, device="cuda:0")
    qg.check(bc.qgemv_moe(fmt, ptr(y), ptr(xd), S * I, ptr(table), len(ws_), ptr(ids_d), n, S, I, O, gs, stream()))
    got = host(y, n * S, O)
    ref, mag = orc().qgemv_moe(fmt, x, S * I, ws_, ss_, ids, S, I, O, gs)
    compare(got, ref.reshape(-1, O), mag.reshape(-1, O), what=f"bounds-checked moe fmt={fmt}")
    status_clean(qg, bc)

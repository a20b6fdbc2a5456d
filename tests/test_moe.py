"""Routed-expert GEMV (qgemv_moe) on the GPU against the oracle (needs a GPU):
every format, shared and per-slot activations, repeated and unordered expert
ids, 1..8 tokens per slot, the routed-expert decode shapes, ids written by a
kernel just before the call, and slots that name no expert.

colibri PR #457, section 7 (the batched routed-expert path: a per-expert
pointer array, one format and group size per tensor); hipfire docs "MQ4 V2",
section 9 (MoE decode on MQ4-V2)."""
import numpy as np
import pytest

import synth
from gpu_util import TOL, compare, dev, orc, torch

pytestmark = pytest.mark.gpu

FMTS = (4, 7, 71, 44, 13, 45)


@pytest.fixture(scope="module")
def qg():
    import weight_only_quantized_i4g_gb300 as m
    return m


def experts(fmt, E, O, I, gs, tag):
    """E seeded experts of one format, packed by the oracle's encoders."""
    ws, ss = [], []
    for e in range(E):
        if fmt == 4:
            w, _ = synth.fmt4_raw(O, I, 1, tag + e)
            wq, sc = orc().quantize_i4g(w, O, I, gs)
            ws.append(wq.reshape(-1)); ss.append(sc.reshape(-1))
        elif fmt == 7:
            codes, sc, _ = synth.fmt7_raw(O, I, 1, tag + e)
            ws.append(codes.reshape(-1)); ss.append(sc.reshape(-1))
        elif fmt == 71:
            codes, _, _ = synth.fmt7_raw(O, I, 1, tag + e)
            nb = ((O + 127) // 128) * ((I + 127) // 128)
            ws.append(codes.reshape(-1)); ss.append((113 + synth.uint64(tag + e, nb) % 8).astype(np.uint8))
        else:
            w, _, d = synth.mq4_raw(O, I, 1, tag + e)
            wr = orc().fwht256(w, d)
            enc = {44: orc().encode_mq4v2, 13: orc().encode_mq4v1, 45: orc().encode_mq4c}[fmt]
            ws.append(enc(wr, O, I).reshape(-1)); ss.append(None)
    return ws, ss


def activations(fmt, n, S, I, tag):
    x = synth.normal(9000 + tag, n * S * I).astype(np.float32)
    return x if fmt == 4 else synth.bf16_bits(x)


def upload_table(qg, ws_dev, ss_dev):
    t = torch()
    raw = qg.expert_table(list(zip(ws_dev, ss_dev)))
    return t.frombuffer(bytearray(raw), dtype=t.uint8).to("cuda:0")


def run(qg, fmt, ws, ss, ids, x, x_stride, S, I, O, gs, keep=None):
    t = torch()
    ws_d = [dev(w) for w in ws]
    ss_d = [None if s is None else dev(s) for s in ss]
    table = upload_table(qg, ws_d, ss_d)
    ids_d = dev(np.asarray(ids, np.int32))
    xd = dev(x)
    n = len(ids)
    y = t.full((n * S * O,), float("nan"), dtype=t.float32, device="cuda:0")
    qg.check(qg.qgemv_moe(fmt, y, xd, x_stride, table, len(ws), ids_d, n, S, I, O, gs))
    t.cuda.synchronize()
    if keep is not None:
        keep.extend([ws_d, ss_d, table, ids_d, xd])
    return y.cpu().numpy().astype(np.float64).reshape(n, S, O)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("S", [1, 2, 5, 8])
@pytest.mark.parametrize("shared", [True, False])
def test_moe_small(qg, fmt, S, shared):
    O, I, gs = (300, 1024, 64) if fmt not in (7, 71) else (300, 1040, 0)
    ws, ss = experts(fmt, 6, O, I, gs, tag=100 * fmt + S)
    ids = [3, 0, 3, 5, 1]
    n_x = 1 if shared else len(ids)
    x = activations(fmt, n_x, S, I, S)
    stride = 0 if shared else S * I
    y = run(qg, fmt, ws, ss, ids, x, stride, S, I, O, gs)
    ref, mag = orc().qgemv_moe(fmt, x, stride, ws, ss, ids, S, I, O, gs)
    compare(y.reshape(-1, O), ref.reshape(-1, O), mag.reshape(-1, O), what=f"moe fmt={fmt} S={S}")


ROUTED = [(4, 2048, 7168, 64, True), (4, 7168, 2048, 64, False), (44, 2048, 7168, 0, True),
          (7, 2048, 7168, 0, True)]


@pytest.mark.parametrize("fmt,O,I,gs,shared", ROUTED)
def test_moe_routed_decode_shapes(qg, fmt, O, I, gs, shared):
    """Eight routed slots of the routed-expert decode shapes (gate/up read one
    token's x, down one x per slot), 16 experts in the table."""
    E, S = 16, 1
    ws, ss = experts(fmt, E, O, I, gs, tag=7 * O)
    ids = [11, 2, 7, 2, 15, 0, 9, 4]
    n_x = 1 if shared else len(ids)
    x = activations(fmt, n_x, S, I, O)
    stride = 0 if shared else S * I
    y = run(qg, fmt, ws, ss, ids, x, stride, S, I, O, gs)
    ref, mag = orc().qgemv_moe(fmt, x, stride, ws, ss, ids, S, I, O, gs)
    compare(y.reshape(-1, O), ref.reshape(-1, O), mag.reshape(-1, O), what=f"moe fmt={fmt} {O}x{I}")


def test_moe_ids_from_a_kernel(qg):
    """The ids are written by a kernel enqueued just before the call on the
    same stream (a stand-in for a router); the call must read them after it."""
    t = torch()
    fmt, O, I, gs, S = 4, 512, 2048, 64, 1
    ws, ss = experts(fmt, 8, O, I, gs, tag=500)
    ws_d = [dev(w) for w in ws]
    ss_d = [dev(s) for s in ss]
    table = upload_table(qg, ws_d, ss_d)
    x = activations(fmt, 1, S, I, 3)
    xd = dev(x)
    scores = t.tensor([0.1, 0.9, 0.3, 0.8, 0.2, 0.7, 0.4, 0.6], device="cuda:0")
    st = t.cuda.Stream()
    y = t.empty(4 * O, dtype=t.float32, device="cuda:0")
    with t.cuda.stream(st):
        ids_d = t.empty(4, dtype=t.int32, device="cuda:0")
        t.cuda._sleep(2_000_000)                       # keep the stream busy so a racing read would see stale ids
        ids_d.copy_(t.topk(scores, 4).indices.to(t.int32))
        qg.check(qg.qgemv_moe(fmt, y, xd, 0, table, 8, ids_d, 4, S, I, O, gs, stream=st))
    st.synchronize()
    ids = [1, 3, 5, 7]
    ref, mag = orc().qgemv_moe(fmt, x, 0, ws, ss, ids, S, I, O, gs)
    compare(y.cpu().numpy().astype(np.float64).reshape(-1, O), ref.reshape(-1, O), mag.reshape(-1, O),
            what="moe ids from a kernel")


def test_moe_bad_slots(qg):
    """Ids outside the table and a misaligned expert: those slots are NaN, the
    others exact, and the device error word says QG_EEXPERT (then clears)."""
    fmt, O, I, gs, S = 44, 200, 512, 0, 2
    ws, ss = experts(fmt, 3, O, I, gs, tag=600)
    t = torch()
    ws_d = [dev(w) for w in ws]
    pad = t.zeros(ws_d[2].numel() + 16, dtype=t.uint8, device="cuda:0")
    pad[1:1 + ws_d[2].numel()].copy_(ws_d[2])
    table = upload_table(qg, [ws_d[0], ws_d[1], pad.data_ptr() + 1], [None, None, None])
    ids = [0, -1, 2, 3, 1]
    x = activations(fmt, 1, S, I, 4)
    xd = dev(x)
    ids_d = dev(np.asarray(ids, np.int32))
    y = t.zeros(len(ids) * S * O, dtype=t.float32, device="cuda:0")
    assert qg.qg_device_status() == (0, 0)
    qg.check(qg.qgemv_moe(fmt, y, xd, 0, table, 3, ids_d, len(ids), S, I, O, gs))
    rc, status = qg.qg_device_status()
    assert rc == 0 and status == qg.QG_EEXPERT
    assert qg.qg_device_status() == (0, 0)
    yh = y.cpu().numpy().astype(np.float64).reshape(len(ids), S, O)
    assert np.isnan(yh[1]).all() and np.isnan(yh[2]).all() and np.isnan(yh[3]).all()
    ref, mag = orc().qgemv_moe(fmt, x, 0, ws, ss, [0, 1], S, I, O, gs)
    compare(yh[[0, 4]].reshape(-1, O), ref.reshape(-1, O), mag.reshape(-1, O), what="moe good slots")


def test_moe_no_slots(qg):
    t = torch()
    y = t.full((8,), 7.0, device="cuda:0")
    assert qg.qgemv_moe(4, y, y, 0, y, 1, y, 0, 1, 64, 4, 64) == qg.QG_OK
    assert (y.cpu() == 7.0).all()


# ----------------------------------------------------------------------------
# routed-expert prefill GEMM (qgemm_moe)
# ----------------------------------------------------------------------------

GEMM_FMTS = (4, 7, 71, 44, 13, 45)


@pytest.mark.parametrize("fmt", GEMM_FMTS)
def test_moe_gemm_groups(qg, fmt):
    """Five groups of 0, 1, 70, 130 and 257 token rows (tensor-core tiles of
    several sizes and a ragged tail), experts repeated and out of order; the
    rows before the first group are left alone."""
    t = torch()
    O, I, gs = (256, 1024, 64) if fmt not in (7, 71) else (260, 1024, 0)
    ws, ss = experts(fmt, 4, O, I, gs, tag=900 + fmt)
    ge = [2, 0, 3, 0, 1]
    off = [5, 5, 6, 76, 206, 463]
    M = off[-1]
    x = synth.normal(950 + fmt, M * I).astype(np.float32)
    xb = synth.bf16_bits(x).reshape(M, I)
    ws_d = [dev(w) for w in ws]
    ss_d = [None if s is None else dev(s) for s in ss]
    table = qg.expert_table(list(zip(ws_d, ss_d)))
    n = qg.qg_moe_gemm_workspace_bytes(fmt, off, len(ge), I, O, gs)
    buf = t.empty(max(n, 1), dtype=t.uint8, device="cuda:0")
    Y = t.full((M * O,), float("nan"), dtype=t.float32, device="cuda:0")
    qg.check(qg.qgemm_moe(fmt, Y, dev(xb), table, 4, ge, off, len(ge), I, O, gs, buf, n))
    Yh = Y.cpu().numpy().astype(np.float64).reshape(M, O)
    assert np.isnan(Yh[:5]).all()
    ref, mag = orc().qgemm_moe(fmt, xb, ws, ss, ge, off, I, O, gs)
    compare(Yh[5:], ref[5:], mag[5:], what=f"moe gemm fmt={fmt}")


def test_moe_gemm_general_kernel_rows(qg):
    """I not a multiple of 64: every group takes the general kernel."""
    t = torch()
    fmt, O, I, gs = 4, 96, 200, 40
    ws, ss = experts(fmt, 3, O, I, gs, tag=990)
    ge, off = [1, 2, 1], [0, 9, 10, 40]
    M = off[-1]
    xb = synth.bf16_bits(synth.normal(991, M * I).astype(np.float32)).reshape(M, I)
    ws_d = [dev(w) for w in ws]                   # kept alive until the call has run
    ss_d = [dev(s) for s in ss]
    table = qg.expert_table(list(zip(ws_d, ss_d)))
    Y = t.full((M * O,), float("nan"), dtype=t.float32, device="cuda:0")
    assert qg.qg_moe_gemm_workspace_bytes(fmt, off, len(ge), I, O, gs) == 0
    qg.check(qg.qgemm_moe(fmt, Y, dev(xb), table, 3, ge, off, len(ge), I, O, gs))
    ref, mag = orc().qgemm_moe(fmt, xb, ws, ss, ge, off, I, O, gs)
    compare(Y.cpu().numpy().astype(np.float64).reshape(M, O), ref, mag, what="moe gemm general")


def run_moe_gemm(qg, fmt, ws, ss, ge, off, I, O, gs, xb, keep_w=None):
    t = torch()
    M = off[-1]
    ws_d = keep_w if keep_w is not None else [dev(w) for w in ws]
    ss_d = [None if s is None else dev(s) for s in ss]
    table = qg.expert_table(list(zip(ws_d, ss_d)))
    n = qg.qg_moe_gemm_workspace_bytes(fmt, off, len(ge), I, O, gs)
    buf = t.empty(max(n, 1), dtype=t.uint8, device="cuda:0")
    Y = t.full((M * O,), float("nan"), dtype=t.float32, device="cuda:0")
    qg.check(qg.qgemm_moe(fmt, Y, dev(xb), table, len(ws), ge, off, len(ge), I, O, gs, buf, n))
    return Y.cpu().numpy().astype(np.float64).reshape(M, O)


@pytest.mark.parametrize("fmt", [4, 44])
def test_moe_gemm_many_groups(qg, fmt):
    """70 non-empty groups (two grouped launches: 64 + 6) of 1..40 rows, four
    empty groups in between."""
    O, I, gs = 256, 512, 64
    ws, ss = experts(fmt, 8, O, I, gs, tag=1200 + fmt)
    sizes = [int(v) for v in (1 + synth.uint64(1300 + fmt, 74) % 40)]
    for g in (5, 30, 31, 60):
        sizes[g] = 0
    off = [0]
    for c in sizes:
        off.append(off[-1] + c)
    ge = [int(v) for v in synth.uint64(1400 + fmt, 74) % 8]
    M = off[-1]
    xb = synth.bf16_bits(synth.normal(1500 + fmt, M * I).astype(np.float32)).reshape(M, I)
    Y = run_moe_gemm(qg, fmt, ws, ss, ge, off, I, O, gs, xb)
    ref, mag = orc().qgemm_moe(fmt, xb, ws, ss, ge, off, I, O, gs)
    compare(Y, ref, mag, what=f"moe gemm 74 groups fmt={fmt}")


def test_moe_gemm_misaligned_expert_falls_back(qg):
    """An expert's weights 8 bytes off a 16-byte line: that chunk runs group by
    group (the fmt=7 tensor-core kernel needs 16-byte aligned codes; the
    general kernel takes it), still exact."""
    t = torch()
    fmt, O, I, gs = 7, 130, 512, 0
    ws, ss = experts(fmt, 2, O, I, gs, tag=1600)
    w0 = dev(ws[0])
    padded = t.zeros(ws[1].size + 16, dtype=t.uint8, device="cuda:0")
    padded[8:8 + ws[1].size].copy_(dev(ws[1]))
    ge, off = [0, 1, 0], [0, 70, 140, 150]
    M = off[-1]
    xb = synth.bf16_bits(synth.normal(1601, M * I).astype(np.float32)).reshape(M, I)
    Y = run_moe_gemm(qg, fmt, ws, ss, ge, off, I, O, gs, xb, keep_w=[w0, padded.data_ptr() + 8])
    ref, mag = orc().qgemm_moe(fmt, xb, ws, ss, ge, off, I, O, gs)
    compare(Y, ref, mag, what="moe gemm fallback")
    del padded

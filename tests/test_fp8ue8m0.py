"""fmt=7 with UE8M0 block scales on the GPU against the oracle (needs a GPU):
the decode GEMV on the fmt=7 decode shapes, batches, block edges, the split
reduction and the general kernel; every exponent byte through the kernel bit
for bit; the prefill GEMM (tensor-core and general kernels) with its
dequantized operand pinned bit for bit.

colibri PR #528, section "Design": the e4m3 weight geometry of fmt=7 with one
UE8M0 byte per 128x128 block, a power-of-two exponent (2^(e - 127))."""
import numpy as np
import pytest

import synth
from gpu_util import compare, dev, host, orc, out, par_rows, torch, workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qg():
    import weight_only_quantized_i4g_gb300 as m
    return m


def inputs(O, I, S, tag):
    """The fmt=7 recipe (uniform codes without the NaN codes, bf16 N(0,1) x)
    with UE8M0 exponents drawn uniformly from [113, 120] (scales 2^-14..2^-7,
    the f32 recipe's 1e-4..1e-2)."""
    codes, _, x = synth.fmt7_raw(O, I, S, tag)
    nbo, nbi = (O + 127) // 128, (I + 127) // 128
    e = (113 + synth.uint64(4000 + tag, nbo * nbi) % 8).astype(np.uint8)
    return codes, e, x


def run(qg, x, codes, e, S, I, O, x_offset=0):
    ws, nws = workspace(qg, qg.QG_FMT_FP8UE8M0, S, I, O)
    y = out(S, O)
    if x_offset:
        xd = dev(np.concatenate([np.zeros(x_offset, np.uint16), x.reshape(-1)]))[x_offset:]
    else:
        xd = dev(x)
    qg.check(qg.qgemv_fp8ue8m0(y, xd, dev(codes), dev(e), S, I, O, ws, nws))
    return host(y, S, O)


SHAPES = [(7168, 16384, 1), (24576, 7168, 1), (2048, 6144, 4), (130, 200, 2), (129, 128, 1), (128, 129, 1),
          (300, 1024, 8), (7, 2048, 3)]


@pytest.mark.parametrize("O,I,S", SHAPES)
def test_gemv_shapes(qg, O, I, S):
    codes, e, x = inputs(O, I, S, O + I + S)
    y = run(qg, x, codes, e, S, I, O)
    ref, mag = par_rows(orc().qgemv_fp8ue8m0, O, x, codes, e, S, I, O, step=128)
    compare(y, ref, mag, what=f"fp8ue8m0 {O}x{I} S={S}")
    compare(y, ref, mag, tol=1e-4, what="fp8ue8m0 page bar 1e-4")


def test_gemv_every_exponent_bit_exact(qg):
    """Row block b (128 rows) has exponent byte b; row r holds code 0x38
    (+1.0) in column 0 and x = e_0: y[r] = 2^(b - 127) bit for bit, from
    2^-127 (an f32 subnormal) to 2^127, and NaN for byte 255."""
    O, I, S = 128 * 256, 16, 1
    codes = np.zeros((O, I), np.uint8)
    codes[:, 0] = 0x38
    e = np.arange(256, dtype=np.uint8)
    x = np.zeros((S, I), np.float32)
    x[0, 0] = 1.0
    y = run(qg, synth.bf16_bits(x).reshape(S, I), codes, e, S, I, O)[0]
    want = np.array([orc().e8m0_value(b // 128) for b in range(O)])
    assert np.array_equal(np.isnan(y), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(y[ok].astype(np.float32).view(np.uint32), want[ok].astype(np.float32).view(np.uint32))


def test_gemv_split_and_general(qg):
    O, I, S = 64, 32768, 1
    assert qg.qg_workspace_bytes(qg.QG_FMT_FP8UE8M0, S, I, O) > 0
    codes, e, x = inputs(O, I, S, 21)
    y = run(qg, x, codes, e, S, I, O)
    ref, mag = par_rows(orc().qgemv_fp8ue8m0, O, x, codes, e, S, I, O, step=128)
    compare(y, ref, mag, what="fp8ue8m0 split")
    O, I, S = 50, 203, 2               # I % 16 != 0: general kernel
    codes, e, x = inputs(O, I, S, 22)
    y = run(qg, x, codes, e, S, I, O)
    ref, mag = par_rows(orc().qgemv_fp8ue8m0, O, x, codes, e, S, I, O, step=128)
    compare(y, ref, mag, what="fp8ue8m0 general")
    O, I, S = 300, 1024, 2             # x not 16-byte aligned: direct kernel
    codes, e, x = inputs(O, I, S, 23)
    y = run(qg, x, codes, e, S, I, O, x_offset=1)
    ref, mag = par_rows(orc().qgemv_fp8ue8m0, O, x, codes, e, S, I, O, step=128)
    compare(y, ref, mag, what="fp8ue8m0 direct")


def run_gemm(qg, X, codes, e, M, I, O, x_offset=0):
    t = torch()
    Y = out(M, O)
    n = 0 if x_offset else qg.qg_gemm_workspace_bytes(qg.QG_FMT_FP8UE8M0, M, I, O, 0)
    buf = t.empty(n, dtype=t.uint8, device="cuda:0") if n else None
    if buf is not None:
        buf.fill_(0xA5)
    if x_offset:
        xd = dev(np.concatenate([np.zeros(x_offset, np.uint16), X.reshape(-1)]))[x_offset:]
    else:
        xd = dev(X)
    qg.check(qg.qgemm_fp8ue8m0(Y, xd, dev(codes), dev(e), M, I, O, buf, n))
    return host(Y, M, O)


@pytest.mark.parametrize("M,I,O", [(1, 128, 1), (70, 512, 130), (257, 2048, 384), (33, 320, 200), (512, 1024, 1024)])
def test_gemm_shapes(qg, M, I, O):
    codes, e, X = inputs(O, I, M, M + 3 * I + O)
    Y = run_gemm(qg, X, codes, e, M, I, O)
    ref, mag = par_rows(orc().qgemv_fp8ue8m0, O, X, codes, e, M, I, O, step=128)
    compare(Y, ref, mag, what=f"fp8ue8m0 gemm {M}x{I}x{O}")


def test_gemm_general_kernel(qg):
    M, I, O = 20, 512, 200
    codes, e, X = inputs(O, I, M, 31)
    Y = run_gemm(qg, X, codes, e, M, I, O, x_offset=1)
    ref, mag = par_rows(orc().qgemv_fp8ue8m0, O, X, codes, e, M, I, O, step=128)
    compare(Y, ref, mag, what="fp8ue8m0 gemm general")


def test_gemm_dequant_bits(qg):
    """With X = e_0 the GEMM returns weight 0 of each row: every e4m3 code
    (row r holds code r % 256) times its block's power of two, exact in f32 and
    in 11 bits; NaN for the NaN codes."""
    M, I, O = 1, 256, 512
    codes = np.zeros((O, I), np.uint8)
    codes[:, 0] = (np.arange(O) % 256).astype(np.uint8)
    e = np.array([100, 102, 127, 125, 130, 131, 118, 116], np.uint8)   # [4 row blocks, 2 column blocks]
    x = np.zeros((M, I), np.float32)
    x[:, 0] = 1.0
    Y = run_gemm(qg, synth.bf16_bits(x).reshape(M, I), codes, e, M, I, O)[0]
    want = np.array([orc().e4m3_value(o % 256) * orc().e8m0_value(int(e[(o // 128) * 2])) for o in range(O)])
    assert np.array_equal(np.isnan(Y), np.isnan(want))
    ok = ~np.isnan(want)
    w32 = np.where(want[ok] == 0.0, 0.0, want[ok]).astype(np.float32)
    assert np.array_equal(Y[ok].astype(np.float32).view(np.uint32), w32.view(np.uint32))

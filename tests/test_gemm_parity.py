"""Batched-prefill dequant-GEMMs of the three formats against the oracle
(needs a GPU).

Small shapes and the fmt=4 M=512 prefill workloads are compared in full;
the fmt=7 and MQ4-V2 GEMMs on their decode shapes at M=512 on a seeded
sample of token rows (every output column of those rows).  The
fmt=7 and MQ4-V2 GEMMs compute the same sums as their GEMVs over M tokens,
so the oracle's GEMV functions with S = M are their references."""
import numpy as np
import pytest

import synth
from gpu_util import compare, dev, fp8_inputs, host, mq4_inputs, orc, out, par_rows, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qg():
    import weight_only_quantized_i4g_gb300 as m
    return m


def gemm_inputs(M, I, O, gs, tag):
    w, _ = synth.fmt4_raw(O, I, 1, 4000 + tag)
    X = synth.bf16_bits(synth.normal(5000 + tag, M * I)).reshape(M, I)
    wq, sc = orc().quantize_i4g(w, O, I, gs)
    return X, wq, sc


def gemm_workspace(qg, M, I, O, gs):
    import torch
    n = qg.qg_gemm_workspace_bytes(qg.QG_FMT_I4G, M, I, O, gs)
    return (torch.empty(n, dtype=torch.uint8, device="cuda:0") if n else None), n


def run_gemm(qg, X, wq, sc, M, I, O, gs, ws=None):
    Y = out(M, O)
    if ws is None:
        ws = gemm_workspace(qg, M, I, O, gs)
    buf, n = ws
    if buf is not None:
        buf.fill_(0xA5)             # stale contents must not matter
    qg.check(qg.qgemm_i4g(Y, dev(X), dev(wq), dev(sc), M, I, O, gs, buf, n))
    return host(Y, M, O)


# Shapes with I % 64 == 0 and gs % 32 == 0 take the tensor-core kernel:
# ragged M and O tails, gs 32/64/96/128/256, a last K step of 64 (I % 128 ==
# 64), tiles whose K range is split over many blocks (few tiles) and whole
# tiles.
TC_SHAPES = [(1, 64, 1, 64), (64, 6144, 2048, 64), (70, 512, 130, 32), (128, 1024, 256, 128),
             (257, 2048, 384, 64), (129, 768, 33, 96), (300, 4096, 520, 256), (16, 128, 4, 64),
             (512, 1024, 1024, 64), (200, 8192, 16, 64), (33, 320, 200, 64), (7, 192, 130, 32),
             (96, 448, 64, 32)]


@pytest.mark.parametrize("M,I,O,gs", TC_SHAPES + [(5, 200, 33, 64), (3, 201, 7, 64), (40, 96, 24, 48)])
def test_gemm_small(qg, M, I, O, gs):
    X, wq, sc = gemm_inputs(M, I, O, gs, M + I + O)
    Y = run_gemm(qg, X, wq, sc, M, I, O, gs)
    ref, mag = par_rows(orc().qgemm_i4g, O, X, wq, sc, M, I, O, gs)
    compare(Y, ref, mag, what=f"gemm {M}x{I}x{O}")


@pytest.mark.parametrize("O", [7168, 2048])
def test_gemm_prefill_workload_full(qg, O):
    """The M=512 prefill workloads in full, in the launch shape the bench times
    (7168x7168: whole tiles per block; 2048x7168: K ranges split over the SMs),
    every one of the 512 x O outputs against the oracle (colibri PR #457,
    section 4: the large-batch GEMM computes the grouped product of section 3
    for every token row)."""
    M, I, gs = 512, 7168, 64
    X, wq, sc = gemm_inputs(M, I, O, gs, O)
    Y = run_gemm(qg, X, wq, sc, M, I, O, gs)
    ref, mag = par_rows(orc().qgemm_i4g, O, X, wq, sc, M, I, O, gs)
    compare(Y, ref, mag, what=f"gemm prefill {M}x{I}x{O}")


def test_gemm_tc_needs_workspace(qg):
    M, I, O, gs = 64, 1024, 256, 64
    assert qg.qg_gemm_workspace_bytes(qg.QG_FMT_I4G, M, I, O, gs) > 0
    assert qg.qg_gemm_workspace_bytes(qg.QG_FMT_I4G, M, 1000, O, gs) == 0      # general kernel
    X, wq, sc = gemm_inputs(M, I, O, gs, 9)
    Y = out(M, O)
    assert qg.qgemm_i4g(Y, dev(X), dev(wq), dev(sc), M, I, O, gs) == qg.QG_EWORKSPACE


def test_gemm_tc_repeatable(qg):
    """Split tiles are summed in contributor order: two calls agree bit for bit."""
    M, I, O, gs = 96, 7168, 512, 64
    X, wq, sc = gemm_inputs(M, I, O, gs, 11)
    ws = gemm_workspace(qg, M, I, O, gs)
    Y1 = run_gemm(qg, X, wq, sc, M, I, O, gs, ws)
    Y2 = run_gemm(qg, X, wq, sc, M, I, O, gs, ws)
    assert np.array_equal(Y1, Y2)
    ref, mag = par_rows(orc().qgemm_i4g, O, X, wq, sc, M, I, O, gs)
    compare(Y1, ref, mag, what="gemm repeatable")


# ----------------------------------------------------------------------------
# Dequantized values through the tensor-core path: with X = e_0 and every
# weight but column 0 zero, Y[0, o] is the fp16 operand itself, unscaled (one
# product by a power of two, then sums of zeros, then the exact power-of-two
# store scaling), so it must equal the weight rounded once to f32 and then to
# 11 significant bits (nearest even), bit for bit.
# ----------------------------------------------------------------------------

def f32_then_11_bits(v):
    v = np.asarray(v, np.float64).astype(np.float32).astype(np.float64)
    m, e = np.frexp(v)                      # v = m * 2^e, |m| in [0.5, 1)
    return np.ldexp(np.round(np.ldexp(m, 11)), e - 11)   # np.round: ties to even


def unit_x(M, I):
    x = np.zeros((M, I), np.float32)
    x[:, 0] = 1.0
    return synth.bf16_bits(x).reshape(M, I)


def assert_bits(y, ref, what):
    y = np.asarray(y, np.float32)
    ref = np.asarray(ref, np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(y), nan), what
    ref = np.where(ref == 0.0, np.float32(0.0), ref)          # 0 + -0 = +0
    assert np.array_equal(y[~nan].view(np.uint32), ref[~nan].view(np.uint32)), what


def test_gemm_i4g_tc_dequant_bits(qg):
    """Every nibble with scales spanning many binades across rows; within a
    row the other group's scale is up to 2^20 larger or smaller (the row's
    power of two follows the larger one; weights within 2^29 of the row
    bound stay in fp16's normal range)."""
    M, I, O, gs = 2, 128, 256, 64
    wq = np.full((O, I // 2), 0x88, np.uint8)
    wq[:, 0] = (np.arange(O) % 16).astype(np.uint8) | 0x80
    sc = np.empty((O, I // gs), np.float32)
    sc[:, 0] = synth.log_uniform(77, O, 1e-6, 1e3)
    sc[:, 1] = sc[:, 0] * synth.log_uniform(78, O, 2.0 ** -20, 2.0 ** 20)
    Y = run_gemm(qg, unit_x(M, I), wq, sc, M, I, O, gs)
    ref = f32_then_11_bits((np.arange(O) % 16 - 8) * sc[:, 0].astype(np.float64))
    assert_bits(Y[0], ref, "fmt4 dequant")
    assert_bits(Y[1], ref, "fmt4 dequant row 1")


def fp8_workspace(qg, M, I, O):
    n = qg.qg_gemm_workspace_bytes(qg.QG_FMT_FP8B128, M, I, O, 0)
    return (torch().empty(n, dtype=torch().uint8, device="cuda:0") if n else None), n


def run_gemm_fp8(qg, X, codes, scales, M, I, O, ws=None, x_offset=0):
    Y = out(M, O)
    buf, n = ws if ws is not None else fp8_workspace(qg, M, I, O)
    if buf is not None:
        buf.fill_(0xA5)
    if x_offset:
        xd = dev(np.concatenate([np.zeros(x_offset, np.uint16), X.reshape(-1)]))
        xp = xd[x_offset:]
    else:
        xp = dev(X)
    qg.check(qg.qgemm_fp8b128(Y, xp, dev(codes), dev(scales), M, I, O, buf, n))
    return host(Y, M, O)


def test_gemm_fp8_all_256_codes(qg):
    """Row r holds code r in column 0; with scale 1 the bf16 weight is the
    E4M3-FN value itself (exact in bf16); NaN codes give NaN."""
    M, I, O = 3, 128, 256
    codes = np.zeros((O, I), np.uint8)
    codes[:, 0] = np.arange(256, dtype=np.uint8)
    scales = np.ones((2, 1), np.float32)
    Y = run_gemm_fp8(qg, unit_x(M, I), codes, scales, M, I, O)
    ref = np.array([orc().e4m3_value(c) for c in range(256)])
    assert set(np.nonzero(np.isnan(ref))[0].tolist()) == {0x7F, 0xFF}
    for m in range(M):
        assert_bits(Y[m], ref, f"fp8 codes row {m}")


def test_gemm_fp8_scaled_bits(qg):
    """code * scale rounded once to f32, then to bf16."""
    M, I, O = 1, 256, 384
    codes = np.zeros((O, I), np.uint8)
    codes[:, 0] = synth.bytes_excluding(5, O)
    scales = synth.log_uniform(6, 3 * 2, 1e-4, 1e-2).reshape(3, 2)
    Y = run_gemm_fp8(qg, unit_x(M, I), codes, scales, M, I, O)
    val = np.array([orc().e4m3_value(int(c)) for c in codes[:, 0]])
    ref = f32_then_11_bits(val * scales[np.arange(O) // 128, 0].astype(np.float64))
    assert_bits(Y[0], ref, "fp8 scaled")


# Tensor-core shapes (I % 64 == 0): ragged M and O, a last K step of 64, split
# and whole tiles; then general-kernel shapes.
FP8_GEMM_SHAPES = [(1, 64, 1), (64, 6144, 2048), (70, 512, 130), (257, 2048, 384), (129, 768, 33),
                   (33, 320, 200), (7, 192, 130), (200, 8192, 16), (512, 1024, 1024), (96, 448, 64),
                   (5, 200, 33), (3, 201, 7), (40, 96, 24)]


@pytest.mark.parametrize("M,I,O", FP8_GEMM_SHAPES)
def test_gemm_fp8_small(qg, M, I, O):
    codes, scales, X = fp8_inputs(O, I, M, tag=M + I + O)
    Y = run_gemm_fp8(qg, X, codes, scales, M, I, O)
    ref, mag = par_rows(orc().qgemv_fp8b128, O, X, codes, scales, M, I, O, step=128)
    compare(Y, ref, mag, what=f"fp8 gemm {M}x{I}x{O}")


def test_gemm_fp8_unaligned_x_general_kernel(qg):
    M, I, O = 20, 512, 200
    codes, scales, X = fp8_inputs(O, I, M, tag=31)
    Y = run_gemm_fp8(qg, X, codes, scales, M, I, O, ws=(None, 0), x_offset=1)
    ref, mag = par_rows(orc().qgemv_fp8b128, O, X, codes, scales, M, I, O, step=128)
    compare(Y, ref, mag, what="fp8 gemm general")


def test_gemm_fp8_nan_columns(qg):
    M, I, O = 40, 1024, 300
    codes, scales, X = fp8_inputs(O, I, M, tag=32)
    codes[7, 100] = 0x7F
    codes[129, 1000] = 0xFF
    Y = run_gemm_fp8(qg, X, codes, scales, M, I, O)
    ref, mag = par_rows(orc().qgemv_fp8b128, O, X, codes, scales, M, I, O, step=128)
    compare(Y, ref, mag, what="fp8 gemm NaN")
    assert set(np.nonzero(np.isnan(Y).all(axis=0))[0].tolist()) == {7, 129}


@pytest.mark.parametrize("O,I", [(24576, 7168), (7168, 16384)])
def test_gemm_fp8_prefill_sampled(qg, O, I):
    M = 512
    codes, scales, X = fp8_inputs(O, I, M, tag=O)
    Y = run_gemm_fp8(qg, X, codes, scales, M, I, O)
    rows = np.sort(np.random.default_rng(O).choice(M, 6, replace=False))
    ref, mag = par_rows(orc().qgemv_fp8b128, O, np.ascontiguousarray(X[rows]), codes, scales, len(rows), I, O,
                        step=128)
    compare(Y[rows], ref, mag, what=f"fp8 gemm prefill {O}x{I}")


def test_gemm_fp8_repeatable(qg):
    M, I, O = 96, 7168, 512
    codes, scales, X = fp8_inputs(O, I, M, tag=33)
    ws = fp8_workspace(qg, M, I, O)
    Y1 = run_gemm_fp8(qg, X, codes, scales, M, I, O, ws)
    Y2 = run_gemm_fp8(qg, X, codes, scales, M, I, O, ws)
    assert np.array_equal(Y1, Y2)


def mq4_workspace(qg, M, I, O):
    n = qg.qg_gemm_workspace_bytes(qg.QG_FMT_MQ4V2, M, I, O, 0)
    return (torch().empty(n, dtype=torch().uint8, device="cuda:0") if n else None), n


def run_gemm_mq4(qg, X, blocks, M, I, O, ws=None, x_offset=0):
    Y = out(M, O)
    buf, n = ws if ws is not None else mq4_workspace(qg, M, I, O)
    if buf is not None:
        buf.fill_(0xA5)
    if x_offset:
        xd = dev(np.concatenate([np.zeros(x_offset, np.uint16), X.reshape(-1)]))
        xp = xd[x_offset:]
    else:
        xp = dev(X)
    qg.check(qg.qgemm_mq4v2(Y, xp, dev(blocks), M, I, O, buf, n))
    return host(Y, M, O)


def test_gemm_mq4_dequant_bits(qg):
    """q * scale + zero rounded once to f32 (fused), then to bf16, for every
    q and both halves of a block, with encoder-made headers."""
    M, I, O = 1, 256, 256
    X, blocks = mq4_inputs(O, I, M, tag=41)
    blocks = blocks.reshape(O, 136).copy()
    X = unit_x(M, I)
    # weight 0 of each row: nibble = o % 16 (the other weights keep their codes
    # but meet x = 0)
    blocks[:, 8] = (blocks[:, 8] & 0xF0) | (np.arange(O) % 16).astype(np.uint8)
    Y = run_gemm_mq4(qg, X, blocks, M, I, O)
    hdr = blocks[:, 0:4].copy().view(np.uint32)[:, 0]
    sc = np.array([orc().f16_value(int(h) & 0xFFFF) for h in hdr])
    ze = np.array([orc().f16_value(int(h) >> 16) for h in hdr])
    ref = f32_then_11_bits((np.arange(O) % 16) * sc + ze)
    assert_bits(Y[0], ref, "mq4 dequant")


MQ4_GEMM_SHAPES = [(1, 256, 1), (70, 512, 130), (257, 2048, 384), (129, 768, 33), (33, 1280, 200),
                   (7, 256, 130), (200, 8192, 16), (512, 1024, 1024), (64, 5120, 1024)]


@pytest.mark.parametrize("M,I,O", MQ4_GEMM_SHAPES)
def test_gemm_mq4_small(qg, M, I, O):
    X, blocks = mq4_inputs(O, I, M, tag=M + I + O)
    Y = run_gemm_mq4(qg, X, blocks, M, I, O)
    ref, mag = par_rows(orc().qgemv_mq4v2, O, X, blocks, M, I, O)
    compare(Y, ref, mag, what=f"mq4 gemm {M}x{I}x{O}")


def test_gemm_mq4_unaligned_x_general_kernel(qg):
    M, I, O = 20, 512, 200
    X, blocks = mq4_inputs(O, I, M, tag=42)
    Y = run_gemm_mq4(qg, X, blocks, M, I, O, ws=(None, 0), x_offset=1)
    ref, mag = par_rows(orc().qgemv_mq4v2, O, X, blocks, M, I, O)
    compare(Y, ref, mag, what="mq4 gemm general")


@pytest.mark.parametrize("O,I", [(5120, 17408), (17408, 5120)])
def test_gemm_mq4_prefill_sampled(qg, O, I):
    M = 512
    X, blocks = mq4_inputs(O, I, M, tag=O)
    Y = run_gemm_mq4(qg, X, blocks, M, I, O)
    rows = np.sort(np.random.default_rng(O).choice(M, 6, replace=False))
    ref, mag = par_rows(orc().qgemv_mq4v2, O, np.ascontiguousarray(X[rows]), blocks, len(rows), I, O)
    compare(Y[rows], ref, mag, what=f"mq4 gemm prefill {O}x{I}")


def test_gemm_mq4_repeatable(qg):
    M, I, O = 96, 5120, 512
    X, blocks = mq4_inputs(O, I, M, tag=43)
    ws = mq4_workspace(qg, M, I, O)
    Y1 = run_gemm_mq4(qg, X, blocks, M, I, O, ws)
    Y2 = run_gemm_mq4(qg, X, blocks, M, I, O, ws)
    assert np.array_equal(Y1, Y2)


# ----------------------------------------------------------------------------
# Range: the tensor-core path keeps fp16 operands in range with a power of
# two per token row and per weight row; rows spanning many binades must
# still meet the bound.
# ----------------------------------------------------------------------------

ROW_POW2 = np.array([-50, -33, -20, -1, 0, 7, 20, 33, 50], np.float64)


def scaled_rows(X_bits, pows):
    x = synth.bf16_to_f32(X_bits).astype(np.float64)
    x *= np.exp2(pows[np.arange(x.shape[0]) % len(pows)])[:, None]
    return synth.bf16_bits(x.astype(np.float32)).reshape(X_bits.shape)


def test_gemm_i4g_rows_across_binades(qg):
    M, I, O, gs = 18, 512, 260, 64
    X, wq, sc = gemm_inputs(M, I, O, gs, 51)
    X = scaled_rows(X, ROW_POW2)
    sc = (sc.astype(np.float64) * np.exp2(ROW_POW2[np.arange(O) % len(ROW_POW2)])[:, None]).astype(np.float32)
    Y = run_gemm(qg, X, wq, sc, M, I, O, gs)
    ref, mag = par_rows(orc().qgemm_i4g, O, X, wq, sc, M, I, O, gs)
    compare(Y, ref, mag, what="fmt4 gemm rows across binades")


def test_gemm_fp8_rows_across_binades(qg):
    M, I, O = 18, 512, 384
    codes, scales, X = fp8_inputs(O, I, M, tag=52)
    X = scaled_rows(X, ROW_POW2)
    scales = (scales.astype(np.float64) * np.exp2(np.array([-40.0, 0.0, 40.0]))[:, None]).astype(np.float32)
    Y = run_gemm_fp8(qg, X, codes, scales, M, I, O)
    ref, mag = par_rows(orc().qgemv_fp8b128, O, X, codes, scales, M, I, O, step=128)
    compare(Y, ref, mag, what="fp8 gemm rows across binades")


def test_gemm_mq4_rows_across_binades(qg):
    M, I, O = 18, 512, 200
    X, blocks = mq4_inputs(O, I, M, tag=53)
    X = scaled_rows(X, ROW_POW2)
    Y = run_gemm_mq4(qg, X, blocks, M, I, O)
    ref, mag = par_rows(orc().qgemv_mq4v2, O, X, blocks, M, I, O)
    compare(Y, ref, mag, what="mq4 gemm rows across binades")


def test_gemm_nonfinite_x_propagates(qg):
    """An inf or NaN activation makes its token row's outputs non-finite,
    as in the oracle (the row's power of two comes from its finite values)."""
    M, I, O, gs = 6, 256, 130, 64
    X, wq, sc = gemm_inputs(M, I, O, gs, 54)
    X = X.copy()
    X[1, 17] = 0x7FC0          # NaN
    X[4, 200] = 0x7F80         # +inf
    Y = run_gemm(qg, X, wq, sc, M, I, O, gs)
    ref, mag = par_rows(orc().qgemm_i4g, O, X, wq, sc, M, I, O, gs)
    assert np.array_equal(np.isnan(Y), np.isnan(ref))
    assert np.array_equal(np.isinf(Y), np.isinf(ref))
    fin = np.isfinite(ref)
    compare(Y[fin], ref[fin], mag[fin], what="gemm finite rows")

"""GPU decode GEMVs against the CPU oracle, element by element (needs a GPU).

Shapes follow the pages' test matrices (colibri #457 section 5, colibri #528
"Metal validation record", hipfire MQ4 V2 section 1e) plus the decode
workloads at full size, ragged tails, every S up to 8 and beyond, the
split-reduction path and the general (unaligned) kernels."""
import numpy as np
import pytest

import synth
from gpu_util import (compare, dev, fp8_inputs, host, i4g_inputs, mq4_inputs, orc, out, par_rows,
                      torch, workspace)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qg():
    import weight_only_quantized_i4g_gb300 as m
    return m


# ----------------------------------------------------------------------------
# fmt=4 grouped int4
# ----------------------------------------------------------------------------

def run_i4g(qg, x, wq, sc, S, I, O, gs, w_offset=0):
    t = torch()
    wd = dev(wq)
    if w_offset:
        buf = t.zeros(wd.numel() + 16, dtype=t.uint8, device=wd.device)
        buf[w_offset:w_offset + wd.numel()] = wd.reshape(-1)
        wd = buf[w_offset:]
    ws, nws = workspace(qg, qg.QG_FMT_I4G, S, I, O, gs)
    y = out(S, O)
    qg.check(qg.qgemv_i4g(y, dev(x), wd, dev(sc), S, I, O, gs, ws, nws))
    return host(y, S, O)


I4G_SHAPES = [
    # (O, I, gs, S, outlier)
    (256, 512, 64, 1, False),      # tiny decode workload
    (2048, 7168, 64, 1, False),    # routed-expert decode shapes, batch 1 and 4
    (2048, 7168, 64, 4, False),
    (7168, 2048, 64, 1, False),
    (7168, 2048, 64, 4, False),
    (2048, 6144, 64, 1, False),    # the page's gate/up and down shapes
    (6144, 2048, 64, 4, False),
    (3, 200, 64, 2, False),        # I not a multiple of gs
    (3, 201, 64, 3, False),        # odd I: nibble tail
    (5, 64, 64, 1, False),         # one group
    (5, 40, 64, 4, False),         # one partial group
    (33, 512, 64, 1, True),        # outlier activation 50.0
    (17, 201, 64, 2, True),
    (1, 7168, 64, 1, False),       # single row
    (1001, 1024, 64, 1, False),    # ragged last row batch
]


@pytest.mark.parametrize("O,I,gs,S,outlier", I4G_SHAPES)
def test_i4g_shapes(qg, O, I, gs, S, outlier):
    x, wq, sc = i4g_inputs(O, I, S, gs, tag=O + I, outlier=outlier)
    y = run_i4g(qg, x, wq, sc, S, I, O, gs)
    ref, mag = par_rows(orc().qgemv_i4g, O, x, wq, sc, S, I, O, gs)
    compare(y, ref, mag, what=f"i4g {O}x{I} gs={gs} S={S}")
    compare(y, ref, mag, tol=1e-4, what="i4g page bar 1e-4")


@pytest.mark.parametrize("gs", [16, 32, 48, 64, 96, 128, 192, 256])
def test_i4g_group_sizes(qg, gs):
    O, I, S = 129, 768, 2
    x, wq, sc = i4g_inputs(O, I, S, gs, tag=gs)
    y = run_i4g(qg, x, wq, sc, S, I, O, gs)
    ref, mag = par_rows(orc().qgemv_i4g, O, x, wq, sc, S, I, O, gs)
    compare(y, ref, mag, what=f"i4g gs={gs}")


@pytest.mark.parametrize("S", [1, 2, 3, 4, 5, 6, 7, 8, 9, 13, 17])
def test_i4g_batch(qg, S):
    O, I, gs = 300, 1024, 64
    x, wq, sc = i4g_inputs(O, I, S, gs, tag=S)
    y = run_i4g(qg, x, wq, sc, S, I, O, gs)
    ref, mag = par_rows(orc().qgemv_i4g, O, x, wq, sc, S, I, O, gs)
    compare(y, ref, mag, what=f"i4g S={S}")


@pytest.mark.parametrize("O,I,S", [(64, 16384, 1), (16, 8192, 3), (100, 4096, 8), (8, 32768, 1),
                                   (3, 65536, 1)])
def test_i4g_split_reduction(qg, O, I, S):
    gs = 64
    assert qg.qg_workspace_bytes(qg.QG_FMT_I4G, S, I, O, gs) > 0
    x, wq, sc = i4g_inputs(O, I, S, gs, tag=7)
    y = run_i4g(qg, x, wq, sc, S, I, O, gs)
    ref, mag = par_rows(orc().qgemv_i4g, O, x, wq, sc, S, I, O, gs)
    compare(y, ref, mag, what=f"i4g split {O}x{I}")


def test_i4g_missing_workspace_refused(qg):
    O, I, S, gs = 3, 65536, 1, 64          # rows too long for one block on every path
    x, wq, sc = i4g_inputs(O, I, S, gs)
    y = out(S, O)
    rc = qg.qgemv_i4g(y, dev(x), dev(wq), dev(sc), S, I, O, gs, None, 0)
    assert rc == qg.QG_EWORKSPACE


def test_i4g_unaligned_weights(qg):
    O, I, S, gs = 77, 1024, 2, 64
    x, wq, sc = i4g_inputs(O, I, S, gs, tag=9)
    y = run_i4g(qg, x, wq, sc, S, I, O, gs, w_offset=3)
    ref, mag = par_rows(orc().qgemv_i4g, O, x, wq, sc, S, I, O, gs)
    compare(y, ref, mag, what="i4g unaligned")


def test_i4g_pad_nibble_never_read(qg):
    O, I, S, gs = 9, 201, 1, 64
    x, wq, sc = i4g_inputs(O, I, S, gs, tag=4)
    poisoned = wq.copy()
    poisoned[:, -1] |= 0xF0
    y = run_i4g(qg, x, poisoned, sc, S, I, O, gs)
    ref, mag = par_rows(orc().qgemv_i4g, O, x, wq, sc, S, I, O, gs)
    compare(y, ref, mag, what="i4g pad nibble")


# ----------------------------------------------------------------------------
# fmt=7 FP8-e4m3 b128
# ----------------------------------------------------------------------------

def run_fp8(qg, x, codes, scales, S, I, O):
    ws, nws = workspace(qg, qg.QG_FMT_FP8B128, S, I, O)
    y = out(S, O)
    qg.check(qg.qgemv_fp8b128(y, dev(x), dev(codes), dev(scales), S, I, O, ws, nws))
    return host(y, S, O)


def test_fp8_all_256_codes_through_the_kernel(qg):
    """Row r holds code r in column 0 (zeros elsewhere), x = e_0, scale 1:
    y[r] must be the E4M3-FN value of code r, bit for bit (NaN for 0x7F/0xFF).
    The sign of a zero cannot survive a sum that starts at +0 (0 + -0 = +0),
    so both zero codes must read +0."""
    O, I, S = 256, 16, 1
    codes = np.zeros((O, I), np.uint8)
    codes[:, 0] = np.arange(256, dtype=np.uint8)
    scales = np.ones((2, 1), np.float32)
    x = np.zeros((1, I), np.float32)
    x[0, 0] = 1.0
    xb = synth.bf16_bits(x)
    y = run_fp8(qg, xb, codes, scales, S, I, O)[0]
    ref = np.array([orc().e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(y), nan)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    ref = np.where(ref == 0.0, 0.0, ref)          # -0 -> +0
    assert np.array_equal(y[~nan].astype(np.float32).view(np.uint32),
                          ref[~nan].astype(np.float32).view(np.uint32))


FP8_SHAPES = [
    (7168, 16384, 1),     # o_proj-like decode shape
    (24576, 7168, 1),
    (2048, 6144, 1),      # the page's spec shapes
    (6144, 2048, 1),
    (2048, 6144, 4),
    (130, 200, 2),        # block edges
    (129, 128, 1),
    (128, 129, 1),
    (1, 1, 1),            # 1x1
    (384, 6144, 3),       # non-square block grid 3 x 48
    (1000, 2048, 2),      # ragged row batch
]


@pytest.mark.parametrize("O,I,S", FP8_SHAPES)
def test_fp8_shapes(qg, O, I, S):
    codes, scales, x = fp8_inputs(O, I, S, tag=O + I)
    y = run_fp8(qg, x, codes, scales, S, I, O)
    ref, mag = par_rows(orc().qgemv_fp8b128, O, x, codes, scales, S, I, O, step=128)
    compare(y, ref, mag, what=f"fp8 {O}x{I} S={S}")
    compare(y, ref, mag, tol=1e-4, what="fp8 page bar 1e-4")


@pytest.mark.parametrize("S", [1, 2, 3, 4, 5, 6, 7, 8, 9])
def test_fp8_batch(qg, S):
    O, I = 260, 1024
    codes, scales, x = fp8_inputs(O, I, S, tag=S)
    y = run_fp8(qg, x, codes, scales, S, I, O)
    ref, mag = par_rows(orc().qgemv_fp8b128, O, x, codes, scales, S, I, O, step=128)
    compare(y, ref, mag, what=f"fp8 S={S}")


@pytest.mark.parametrize("span", [0, 40, 120])
def test_fp8_activation_range(qg, span):
    """Batch-1 activations whose magnitudes span 2^-span .. 2^span (the
    one-token kernel carries x as fp16 scaled by a power of two per thread)."""
    O, I, S = 384, 4096, 1
    codes, scales, _ = fp8_inputs(O, I, S, tag=300 + span)
    x = (synth.normal(9300 + span, I) * np.exp2(span * (2 * synth.uniform(9350 + span, I) - 1))).astype(np.float32)
    xb = synth.bf16_bits(x).reshape(S, I)
    y = run_fp8(qg, xb, codes, scales, S, I, O)
    ref, mag = par_rows(orc().qgemv_fp8b128, O, xb, codes, scales, S, I, O, step=128)
    compare(y, ref, mag, what=f"fp8 x span 2^{span}")


def test_fp8_nan_rows(qg):
    O, I, S = 130, 256, 2
    codes, scales, x = fp8_inputs(O, I, S, tag=11)
    codes[7, 100] = 0x7F
    codes[129, 3] = 0xFF
    y = run_fp8(qg, x, codes, scales, S, I, O)
    ref, mag = par_rows(orc().qgemv_fp8b128, O, x, codes, scales, S, I, O, step=128)
    compare(y, ref, mag, what="fp8 NaN rows")
    assert set(np.nonzero(np.isnan(y[0]))[0].tolist()) == {7, 129}


@pytest.mark.parametrize("O,I,S", [(64, 32768, 1), (32, 8192, 5)])
def test_fp8_split_reduction(qg, O, I, S):
    assert qg.qg_workspace_bytes(qg.QG_FMT_FP8B128, S, I, O) > 0
    codes, scales, x = fp8_inputs(O, I, S, tag=12)
    y = run_fp8(qg, x, codes, scales, S, I, O)
    ref, mag = par_rows(orc().qgemv_fp8b128, O, x, codes, scales, S, I, O, step=128)
    compare(y, ref, mag, what="fp8 split")


def test_fp8_unaligned_general_kernel(qg):
    O, I, S = 50, 200 + 3, 2          # I % 16 != 0 -> general kernel
    codes, scales, x = fp8_inputs(O, I, S, tag=13)
    y = run_fp8(qg, x, codes, scales, S, I, O)
    ref, mag = par_rows(orc().qgemv_fp8b128, O, x, codes, scales, S, I, O, step=128)
    compare(y, ref, mag, what="fp8 general")


# ----------------------------------------------------------------------------
# MQ4-V2
# ----------------------------------------------------------------------------

def run_mq4(qg, x, blocks, S, I, O):
    ws, nws = workspace(qg, qg.QG_FMT_MQ4V2, S, I, O)
    y = out(S, O)
    qg.check(qg.qgemv_mq4v2(y, dev(x), dev(blocks), S, I, O, ws, nws))
    return host(y, S, O)


MQ4_SHAPES = [
    (5120, 17408, 1),     # decode shapes, batch 1 and 8
    (5120, 17408, 8),
    (17408, 5120, 1),
    (17408, 5120, 8),
    (1, 256, 1),          # one block
    (3, 512, 2),
    (7, 768, 5),          # odd number of blocks per row (8-byte aligned rows)
    (1000, 4096, 3),
    (64, 32768, 1),       # long rows: split reduction
]


@pytest.mark.parametrize("O,I,S", MQ4_SHAPES)
def test_mq4_shapes(qg, O, I, S):
    x, blocks = mq4_inputs(O, I, S, tag=O + I)
    y = run_mq4(qg, x, blocks, S, I, O)
    ref, mag = par_rows(orc().qgemv_mq4v2, O, x, blocks, S, I, O)
    compare(y, ref, mag, what=f"mq4 {O}x{I} S={S}")


@pytest.mark.parametrize("S", [1, 2, 3, 4, 5, 6, 7, 8, 9])
def test_mq4_batch(qg, S):
    O, I = 200, 1280
    x, blocks = mq4_inputs(O, I, S, tag=S)
    y = run_mq4(qg, x, blocks, S, I, O)
    ref, mag = par_rows(orc().qgemv_mq4v2, O, x, blocks, S, I, O)
    compare(y, ref, mag, what=f"mq4 S={S}")


def test_mq4_distinct_half_headers(qg):
    """Clearly different (scale, zero) per half catch a wrong half predicate,
    a swapped header field, a +4 payload offset or a 132-byte stride."""
    rng = np.random.default_rng(5)
    O, I, S = 33, 1536, 2
    nb = I // 256
    blocks = rng.integers(0, 256, (O, nb, 136), dtype=np.uint8)
    hv = (rng.uniform(0.5, 2.0, (O, nb, 4)) * [1e-2, 1, 1e-2, -1]).astype(np.float16)
    blocks[:, :, 0:8] = hv.view(np.uint8).reshape(O, nb, 8)
    x = synth.bf16_bits(rng.standard_normal(S * I).astype(np.float32)).reshape(S, I)
    y = run_mq4(qg, x, blocks, S, I, O)
    ref, mag = par_rows(orc().qgemv_mq4v2, O, x, blocks, S, I, O)
    compare(y, ref, mag, what="mq4 distinct halves")


def test_mq4_equal_halves_constant(qg):
    """Equal half headers, all-equal nibbles: y = (q*s + z) * sum(x) per row."""
    O, I, S = 4, 512, 1
    blocks = np.zeros((O, I // 256, 136), np.uint8)
    s16, z16 = np.float16(0.125), np.float16(-0.5)
    pair = np.array([s16, z16], np.float16).view(np.uint8)
    blocks[:, :, 0:4] = pair
    blocks[:, :, 4:8] = pair
    blocks[:, :, 8:] = 0x33                      # q = 3 everywhere
    x = np.zeros((S, I), np.float32)
    x[0, :] = np.arange(I) % 7 - 3               # small integers: exact sums
    y = run_mq4(qg, synth.bf16_bits(x), blocks, S, I, O)
    want = (3 * 0.125 - 0.5) * float(x.sum())
    assert np.all(y == want), (y, want)


def test_device_status_clean_after_staged_calls(qg):
    """No staged-kernel barrier wait gave up in any call above (or in this one)."""
    O, I, S, gs = 2048, 7168, 1, 64
    x, wq, sc = i4g_inputs(O, I, S, gs, tag=99)
    run_i4g(qg, x, wq, sc, S, I, O, gs)
    rc, status = qg.qg_device_status()
    assert rc == qg.QG_OK and status == qg.QG_OK, (rc, status, qg.last_error())

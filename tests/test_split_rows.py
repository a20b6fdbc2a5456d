"""Rows split into column segments across blocks (needs a GPU).

Rows longer than one block's warps cover split into column segments along
grid.y; each segment writes its partial sums to the caller's workspace and a
second kernel adds them in segment order.  These cases cover ragged last
batches, odd token counts, many batches per block, 2- to 9-segment splits on
the warp-MMA kernel (from two tokens on) and the staged kernel (one token),
and repeatability.  Every output is compared with the oracle element by
element."""
import numpy as np
import pytest

from gpu_util import compare, dev, host, i4g_inputs, mq4_inputs, orc, out, par_rows, workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qg():
    import weight_only_quantized_i4g_gb300 as m
    return m


def mq4_call(qg, x, blocks, S, I, O):
    ws, nws = workspace(qg, qg.QG_FMT_MQ4V2, S, I, O)
    y = out(S, O)
    rc = qg.qgemv_mq4v2(y, dev(x), dev(blocks), S, I, O, ws, nws)
    return rc, y


# (O, I, S): on the warp-MMA kernel (two tokens on) segments = ceil(I / 64 /
# 120) for MQ4-V2 (15 consumer warps of 8 spans of 64 weights), rounded to
# whole pairs of 256-weight blocks; at one token the staged kernel splits
MQ4_SPLIT = [
    (1000, 17408, 1),    # staged split, ragged last batch (1000 = 62 x 16 + 8)
    (333, 17408, 5),     # 3 segments, odd token count, ragged
    (5120, 17408, 3),    # 3 segments, many batches per block
    (24, 9216, 2),       # 2 segments, two batches of which one is ragged
    (70, 61440, 1),      # staged split of long rows
    (17, 61440, 8),      # 8 segments at eight tokens
    (40, 65536, 2),      # 9 segments
]


@pytest.mark.parametrize("O,I,S", MQ4_SPLIT)
def test_mq4_split_rows(qg, O, I, S):
    x, blocks = mq4_inputs(O, I, S, tag=O + 3 * I + S)
    rc, y = mq4_call(qg, x, blocks, S, I, O)
    qg.check(rc)
    ref, mag = par_rows(orc().qgemv_mq4v2, O, x, blocks, S, I, O)
    compare(host(y, S, O), ref, mag, what=f"mq4 split {O}x{I} S={S}")


def test_mq4_split_repeatable(qg):
    """The segments are added in a fixed order: two calls agree bit for bit."""
    O, I, S = 777, 17408, 4
    x, blocks = mq4_inputs(O, I, S, tag=21)
    xd, bd = dev(x), dev(blocks)
    ws, nws = workspace(qg, qg.QG_FMT_MQ4V2, S, I, O)
    ys = []
    for _ in range(2):
        y = out(S, O)
        qg.check(qg.qgemv_mq4v2(y, xd, bd, S, I, O, ws, nws))
        ys.append(host(y, S, O))
    assert np.array_equal(ys[0], ys[1])


# fmt=4 on the warp-MMA kernel from two tokens on: 14 consumer warps of 8 spans
I4G_SPLIT = [
    (77, 8192, 2),       # 2 segments, ragged
    (300, 16384, 4),     # 3 segments
    (1000, 16384, 3),    # 3 segments, many batches, ragged
]


@pytest.mark.parametrize("O,I,S", I4G_SPLIT)
def test_i4g_split_rows(qg, O, I, S):
    gs = 64
    x, wq, sc = i4g_inputs(O, I, S, gs, tag=O + I + S)
    ws, nws = workspace(qg, qg.QG_FMT_I4G, S, I, O, gs)
    y = out(S, O)
    qg.check(qg.qgemv_i4g(y, dev(x), dev(wq), dev(sc), S, I, O, gs, ws, nws))
    ref, mag = par_rows(orc().qgemv_i4g, O, x, wq, sc, S, I, O, gs)
    compare(host(y, S, O), ref, mag, what=f"i4g split {O}x{I} S={S}")
    compare(host(y, S, O), ref, mag, tol=1e-4, what="i4g split, page bar 1e-4")


def test_mq4v1_split_rows(qg):
    """The one-header MQ4 layout runs the same kernel templates."""
    O, I, S = 129, 17408, 2
    rng = np.random.default_rng(4)
    w = rng.standard_normal((O, I)) * 0.02
    blocks = orc().encode_mq4v1(w, O, I)
    import synth
    x = synth.bf16_bits(rng.standard_normal(S * I).astype(np.float32)).reshape(S, I)
    ws, nws = workspace(qg, qg.QG_FMT_MQ4V1, S, I, O)
    y = out(S, O)
    qg.check(qg.qgemv_mq4v1(y, dev(x), dev(blocks), S, I, O, ws, nws))
    ref, mag = par_rows(orc().qgemv_mq4v1, O, x, blocks, S, I, O)
    compare(host(y, S, O), ref, mag, what="mq4v1 split")

"""Q2_0 decode GEMV on the GPU against the oracle (needs a GPU): the routed-
expert shapes the strata review checks (gate/up 2560 rows, down 640), a
routed-expert shape of the fmt=4 configs, batches 1..9, single blocks and
every code through the kernel.

strata review, "convert_k256_q2_0.cpp vs ref_quant.cpp" (2.5): 64 weights in
18 bytes, fp16 d and 2-bit codes, w = (code - 1) * d."""
import numpy as np
import pytest

import synth
from gpu_util import compare, dev, host, orc, out, par_rows, workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qg():
    import weight_only_quantized_i4g_gb300 as m
    return m


def inputs(O, I, S, tag):
    w = synth.normal(7000 + tag, O * I, 0.02).reshape(O, I)
    x = synth.normal(7500 + tag, S * I).astype(np.float32)
    return synth.bf16_bits(x).reshape(S, I), orc().encode_q2_0(w, O, I)


def run(qg, x, blocks, S, I, O):
    ws, nws = workspace(qg, qg.QG_FMT_Q2_0, S, I, O)
    y = out(S, O)
    qg.check(qg.qgemv_q2_0(y, dev(x), dev(blocks), S, I, O, ws, nws))
    return host(y, S, O)


SHAPES = [(640, 2560, 1), (2560, 640, 1), (2048, 7168, 1), (7168, 2048, 1), (1, 64, 1), (3, 192, 2), (130, 1280, 5),
          (64, 65536, 1)]


@pytest.mark.parametrize("O,I,S", SHAPES)
def test_q2_0_shapes(qg, O, I, S):
    x, blocks = inputs(O, I, S, O + I + S)
    y = run(qg, x, blocks, S, I, O)
    ref, mag = par_rows(orc().qgemv_q2_0, O, x, blocks, S, I, O)
    compare(y, ref, mag, what=f"q2_0 {O}x{I} S={S}")


@pytest.mark.parametrize("S", [1, 2, 3, 4, 5, 6, 7, 8, 9])
def test_q2_0_batch(qg, S):
    O, I = 200, 2560
    x, blocks = inputs(O, I, S, 40 + S)
    y = run(qg, x, blocks, S, I, O)
    ref, mag = par_rows(orc().qgemv_q2_0, O, x, blocks, S, I, O)
    compare(y, ref, mag, what=f"q2_0 S={S}")


def test_q2_0_every_code_and_position(qg):
    """Row r: weight (r % 64) of its block holds code (r // 64) % 4, every other
    code is 1 (weight 0), d = 2^-(r % 7); x = ones: y[r] = (code - 1) * d exactly."""
    O, I = 256, 64
    blocks = np.zeros((O, 18), np.uint8)
    blocks[:, 2:] = 0x55
    for r in range(O):
        e, c = r % 64, (r // 64) % 4
        byte = 2 + e // 4
        blocks[r, byte] = (int(blocks[r, byte]) & (0xFF ^ (3 << (2 * (e % 4))))) | (c << (2 * (e % 4)))
        blocks[r, 0:2] = np.array([2.0 ** -(r % 7)], np.float16).view(np.uint8)
    x = synth.bf16_bits(np.ones(I, np.float32)).reshape(1, I)
    y = run(qg, x, blocks, 1, I, O)[0]
    want = np.array([((r // 64) % 4 - 1) * 2.0 ** -(r % 7) for r in range(O)])
    assert np.array_equal(y, want)


def test_q2_0_staged_every_code_and_position(qg):
    """The staged kernel (one token, I a multiple of 512): row r holds code
    (r // 512) % 4 at weight r % 512 of its row, code 1 (weight 0) elsewhere,
    d = 2^-(r % 5) in every block; x = ones: y[r] = (code - 1) * d exactly."""
    O, I = 2048, 512
    blocks = np.zeros((O, I // 64, 18), np.uint8)
    blocks[:, :, 2:] = 0x55
    for r in range(O):
        blocks[r, :, 0:2] = np.array([2.0 ** -(r % 5)], np.float16).view(np.uint8)
        e, c = r % I, (r // I) % 4
        b, byte = e // 64, 2 + (e % 64) // 4
        sh = 2 * (e % 4)
        blocks[r, b, byte] = (int(blocks[r, b, byte]) & (0xFF ^ (3 << sh))) | (c << sh)
    blocks = blocks.reshape(O, -1)
    x = synth.bf16_bits(np.ones(I, np.float32)).reshape(1, I)
    y = run(qg, x, blocks, 1, I, O)[0]
    want = np.array([((r // I) % 4 - 1) * 2.0 ** -(r % 5) for r in range(O)])
    assert np.array_equal(y, want)


@pytest.mark.parametrize("span", [0, 40, 120])
def test_q2_0_activation_range(qg, span):
    """Activations whose magnitudes span 2^-span .. 2^span (the staged kernel
    rescales x by a power of two per thread before its fp16 products)."""
    O, I, S = 512, 4096, 1
    x = (synth.normal(9100 + span, I) * np.exp2(span * (2 * synth.uniform(9150 + span, I) - 1))).astype(np.float32)
    xb = synth.bf16_bits(x).reshape(S, I)
    w = synth.normal(9200 + span, O * I, 0.02).reshape(O, I)
    blocks = orc().encode_q2_0(w, O, I)
    y = run(qg, xb, blocks, S, I, O)
    ref, mag = par_rows(orc().qgemv_q2_0, O, xb, blocks, S, I, O)
    compare(y, ref, mag, what=f"q2_0 x span 2^{span}")

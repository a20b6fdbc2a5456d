"""Device weight preparation against the oracle (needs a GPU): the fmt=4
quantizer and the MQ4-V2 encoder bit for bit, the FWHT-256 rotation within
binary32 rounding of the oracle's double-precision transform."""
import numpy as np
import pytest

import synth
from gpu_util import dev, orc, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qg():
    import weight_only_quantized_i4g_gb300 as m
    return m


@pytest.mark.parametrize("O,I,gs", [(2048, 7168, 64), (7168, 2048, 64), (7, 201, 64), (5, 40, 16),
                                    (3, 999, 48), (64, 512, 256)])
def test_quantize_i4g_bit_exact(qg, O, I, gs):
    t = torch()
    w = synth.normal(100 + I, O * I, 0.02).reshape(O, I)
    w[0, :min(gs, I)] = 0.0                      # an all-zero group
    if I > 2 * gs:
        w[1, gs:2 * gs] = 0.5                    # a constant group
    rb, ng = (I + 1) // 2, (I + gs - 1) // gs
    wq = t.full((O * rb,), 0xAB, dtype=t.uint8, device="cuda")
    sc = t.full((O * ng,), float("nan"), dtype=t.float32, device="cuda")
    qg.check(qg.qg_quantize_i4g(wq, sc, dev(w), O, I, gs))
    t.cuda.synchronize()
    ref_q, ref_s = orc().quantize_i4g(w, O, I, gs)
    assert np.array_equal(wq.cpu().numpy().reshape(O, rb), ref_q)
    assert np.array_equal(sc.cpu().numpy().reshape(O, ng).view(np.uint32), ref_s.view(np.uint32))


@pytest.mark.parametrize("O,I", [(64, 17408), (17, 5120), (3, 256)])
def test_encode_mq4v2_bit_exact(qg, O, I):
    t = torch()
    w = synth.normal(200 + I, O * I, 0.02).reshape(O, I)
    w[0, 0:128] = 0.0123                         # a constant half
    w[1, 128:256] = np.float32(1e-9) * np.arange(128, dtype=np.float32)   # fp16 step rounds to 0
    blocks = t.full((O * (I // 256) * 136,), 0xCD, dtype=t.uint8, device="cuda")
    qg.check(qg.qg_encode_mq4v2(blocks, dev(w), O, I))
    t.cuda.synchronize()
    ref = orc().encode_mq4v2(w, O, I)
    got = blocks.cpu().numpy().reshape(O, -1)
    assert np.array_equal(got, ref)


def test_fwht256_matches_oracle(qg):
    t = torch()
    n = 1024
    v = synth.normal(300, 256 * n)
    d = synth.signs(synth.SIGN_SEED, 256)
    outd = t.empty(256 * n, dtype=t.float32, device="cuda")
    qg.check(qg.qg_fwht256(outd, dev(v), dev(d), n))
    t.cuda.synchronize()
    ref = orc().fwht256(v, d).reshape(n, 256).astype(np.float64)
    got = outd.cpu().numpy().reshape(n, 256).astype(np.float64)
    norms = np.linalg.norm(v.reshape(n, 256).astype(np.float64), axis=1, keepdims=True)
    assert np.max(np.abs(got - ref) / norms) < 2e-6
    # in place
    vd = dev(v)
    qg.check(qg.qg_fwht256(vd, vd, dev(d), n))
    t.cuda.synchronize()
    assert np.array_equal(vd.cpu().numpy(), outd.cpu().numpy())

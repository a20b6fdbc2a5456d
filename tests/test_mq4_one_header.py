"""MQ4 v1 (hipfire qt=13) and MQ4C pad (qt=45) on the GPU against the oracle
(needs a GPU): decode GEMV at the MQ4-V2 decode shapes, batches 1..9, the
direct path (x not 16-byte aligned) and the split reduction; the tensor-core
prefill GEMM and its general kernel; the device encoders bit for bit.

Both formats keep the MQ4-V2 block (136 B per 256 weights, nibbles at
[8,136)) with one header for the block: v1 f32 scale and zero, pad fp16
scale and zero then four zero bytes (hipfire "MQ4 V2", sections 1b, 1e)."""
import numpy as np
import pytest

import synth
from gpu_util import compare, dev, host, orc, out, par_rows, torch, workspace

pytestmark = pytest.mark.gpu

FORMATS = ("v1", "c")


@pytest.fixture(scope="module")
def qg():
    import weight_only_quantized_i4g_gb300 as m
    return m


def fmt_id(qg, f):
    return qg.QG_FMT_MQ4V1 if f == "v1" else qg.QG_FMT_MQ4C


def inputs(f, O, I, S, tag):
    w, x, d = synth.mq4_raw(O, I, S, tag)
    wr = orc().fwht256(w, d)
    xr = orc().fwht256(x, d)
    enc = orc().encode_mq4v1 if f == "v1" else orc().encode_mq4c
    return synth.bf16_bits(xr).reshape(S, I), enc(wr, O, I)


def oracle_gemv(f):
    return orc().qgemv_mq4v1 if f == "v1" else orc().qgemv_mq4c


def run_gemv(qg, f, x, blocks, S, I, O, x_offset=0):
    ws, nws = workspace(qg, fmt_id(qg, f), S, I, O)
    y = out(S, O)
    if x_offset:
        xd = dev(np.concatenate([np.zeros(x_offset, np.uint16), x.reshape(-1)]))[x_offset:]
    else:
        xd = dev(x)
    fn = qg.qgemv_mq4v1 if f == "v1" else qg.qgemv_mq4c
    qg.check(fn(y, xd, dev(blocks), S, I, O, ws, nws))
    return host(y, S, O)


SHAPES = [(5120, 17408, 1), (17408, 5120, 1), (17408, 5120, 8), (1, 256, 1), (7, 768, 5), (1000, 4096, 3),
          (64, 32768, 1)]


@pytest.mark.parametrize("f", FORMATS)
@pytest.mark.parametrize("O,I,S", SHAPES)
def test_gemv_shapes(qg, f, O, I, S):
    x, blocks = inputs(f, O, I, S, O + I + S)
    y = run_gemv(qg, f, x, blocks, S, I, O)
    ref, mag = par_rows(oracle_gemv(f), O, x, blocks, S, I, O)
    compare(y, ref, mag, what=f"mq4{f} {O}x{I} S={S}")


@pytest.mark.parametrize("f", FORMATS)
@pytest.mark.parametrize("S", [1, 2, 3, 4, 5, 6, 7, 8, 9])
def test_gemv_batch(qg, f, S):
    O, I = 200, 1280
    x, blocks = inputs(f, O, I, S, 60 + S)
    y = run_gemv(qg, f, x, blocks, S, I, O)
    ref, mag = par_rows(oracle_gemv(f), O, x, blocks, S, I, O)
    compare(y, ref, mag, what=f"mq4{f} S={S}")


@pytest.mark.parametrize("f", FORMATS)
def test_gemv_direct_path(qg, f):
    """x not 16-byte aligned: the direct (global-load) kernel."""
    O, I, S = 300, 2048, 2
    x, blocks = inputs(f, O, I, S, 70)
    y = run_gemv(qg, f, x, blocks, S, I, O, x_offset=1)
    ref, mag = par_rows(oracle_gemv(f), O, x, blocks, S, I, O)
    compare(y, ref, mag, what=f"mq4{f} direct")


@pytest.mark.parametrize("f", FORMATS)
def test_gemv_distinct_block_headers(qg, f):
    """Random payload and a clearly different header per block catch a
    per-half header read, swapped fields, a +4 payload offset or a 132-byte
    stride."""
    rng = np.random.default_rng(71)
    O, I, S = 33, 1536, 2
    nb = I // 256
    blocks = rng.integers(0, 256, (O, nb, 136), dtype=np.uint8)
    s = rng.uniform(1e-3, 1e-2, (O, nb))
    z = rng.uniform(-0.1, 0.1, (O, nb))
    if f == "v1":
        blocks[:, :, 0:8] = np.stack([s, z], -1).astype("<f4").view(np.uint8).reshape(O, nb, 8)
    else:
        blocks[:, :, 0:4] = np.stack([s, z], -1).astype(np.float16).view(np.uint8).reshape(O, nb, 4)
        blocks[:, :, 4:8] = 0
    x = synth.bf16_bits(rng.standard_normal(S * I).astype(np.float32)).reshape(S, I)
    y = run_gemv(qg, f, x, blocks, S, I, O)
    ref, mag = par_rows(oracle_gemv(f), O, x, blocks, S, I, O)
    compare(y, ref, mag, what=f"mq4{f} distinct headers")


def gemm_ws(qg, f, M, I, O):
    n = qg.qg_gemm_workspace_bytes(fmt_id(qg, f), M, I, O, 0)
    return (torch().empty(n, dtype=torch().uint8, device="cuda:0") if n else None), n


def run_gemm(qg, f, X, blocks, M, I, O, x_offset=0):
    Y = out(M, O)
    buf, n = gemm_ws(qg, f, M, I, O) if not x_offset else (None, 0)
    if buf is not None:
        buf.fill_(0xA5)
    if x_offset:
        xd = dev(np.concatenate([np.zeros(x_offset, np.uint16), X.reshape(-1)]))[x_offset:]
    else:
        xd = dev(X)
    fn = qg.qgemm_mq4v1 if f == "v1" else qg.qgemm_mq4c
    qg.check(fn(Y, xd, dev(blocks), M, I, O, buf, n))
    return host(Y, M, O)


GEMM_SHAPES = [(1, 256, 1), (70, 512, 130), (257, 2048, 384), (129, 768, 33), (512, 1024, 1024), (64, 5120, 1024)]


@pytest.mark.parametrize("f", FORMATS)
@pytest.mark.parametrize("M,I,O", GEMM_SHAPES)
def test_gemm_shapes(qg, f, M, I, O):
    X, blocks = inputs(f, O, I, M, M + I + O)
    Y = run_gemm(qg, f, X, blocks, M, I, O)
    ref, mag = par_rows(oracle_gemv(f), O, X, blocks, M, I, O)
    compare(Y, ref, mag, what=f"mq4{f} gemm {M}x{I}x{O}")


@pytest.mark.parametrize("f", FORMATS)
def test_gemm_general_kernel(qg, f):
    M, I, O = 20, 512, 200
    X, blocks = inputs(f, O, I, M, 72)
    Y = run_gemm(qg, f, X, blocks, M, I, O, x_offset=1)
    ref, mag = par_rows(oracle_gemv(f), O, X, blocks, M, I, O)
    compare(Y, ref, mag, what=f"mq4{f} gemm general")


@pytest.mark.parametrize("f", FORMATS)
def test_gemm_dequant_bits(qg, f):
    """With X = e_0 the GEMM returns weight 0 of each row, formed in f32 with
    one rounding and rounded to 11 significant bits."""
    M, I, O = 1, 256, 256
    X, blocks = inputs(f, O, I, M, 73)
    blocks = blocks.reshape(O, 136).copy()
    blocks[:, 8] = (blocks[:, 8] & 0xF0) | (np.arange(O) % 16).astype(np.uint8)
    x = np.zeros((M, I), np.float32)
    x[:, 0] = 1.0
    Y = run_gemm(qg, f, synth.bf16_bits(x).reshape(M, I), blocks, M, I, O)
    w = np.array([(orc().mq4v1_weight if f == "v1" else orc().mq4c_weight)(blocks[o], 0) for o in range(O)])
    v = w.astype(np.float32).astype(np.float64)
    m, e = np.frexp(v)
    ref = np.ldexp(np.round(np.ldexp(m, 11)), e - 11)
    ref = np.where(ref == 0.0, 0.0, ref)
    assert np.array_equal(Y[0].astype(np.float32).view(np.uint32), ref.astype(np.float32).view(np.uint32))


@pytest.mark.parametrize("f", FORMATS)
@pytest.mark.parametrize("O,I", [(7, 256), (64, 2048), (300, 5120)])
def test_encoder_bit_exact(qg, f, O, I):
    w = synth.normal(80 + O, O * I, 0.02).reshape(O, I)
    w[0, 0:256] = 0.0123                       # a constant block
    blocks = torch().empty(O * (I // 256) * 136, dtype=torch().uint8, device="cuda:0")
    enc = qg.qg_encode_mq4v1 if f == "v1" else qg.qg_encode_mq4c
    qg.check(enc(blocks, dev(w), O, I))
    got = host_u8(blocks)
    ref = (orc().encode_mq4v1 if f == "v1" else orc().encode_mq4c)(w, O, I).reshape(-1)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} bytes differ"


def host_u8(t):
    torch().cuda.synchronize()
    return t.cpu().numpy()

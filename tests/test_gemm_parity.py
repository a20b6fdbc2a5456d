"""fmt=4 batched-prefill dequant-GEMM against the oracle (needs a GPU).

Small shapes are compared in full; the M=512 prefill workloads are compared
on a seeded sample of token rows (every output column of those rows)."""
import numpy as np
import pytest

import synth
from gpu_util import compare, dev, host, orc, out, par_rows

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
def test_gemm_prefill_workload_sampled(qg, O):
    M, I, gs = 512, 7168, 64
    X, wq, sc = gemm_inputs(M, I, O, gs, O)
    Y = run_gemm(qg, X, wq, sc, M, I, O, gs)
    rows = np.sort(np.random.default_rng(O).choice(M, 12, replace=False))
    ref, mag = par_rows(orc().qgemm_i4g, O, np.ascontiguousarray(X[rows]), wq, sc, len(rows), I, O, gs)
    compare(Y[rows], ref, mag, what=f"gemm prefill O={O}")


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

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


def run_gemm(qg, X, wq, sc, M, I, O, gs):
    Y = out(M, O)
    qg.check(qg.qgemm_i4g(Y, dev(X), dev(wq), dev(sc), M, I, O, gs))
    return host(Y, M, O)


@pytest.mark.parametrize("M,I,O,gs", [(1, 64, 1, 64), (5, 200, 33, 64), (64, 6144, 2048, 64),
                                      (70, 512, 130, 32), (3, 201, 7, 64), (128, 1024, 256, 128),
                                      (257, 2048, 384, 64)])
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

"""Helpers of the GPU parity tests: inputs built on the CPU with the seeded
generators and the oracle's encoders, uploaded, run through the C ABI, and
compared with the oracle element by element."""
from __future__ import annotations

import numpy as np

import oracle
import synth

DEV = "cuda:0"
TOL = 1e-3          # |y - y_ref| <= TOL * sum_i |w_i x_i| per output element


def torch():
    import torch as t
    return t


def dev(a: np.ndarray):
    """numpy -> device tensor (uint16 travels as int16 bits)."""
    t = torch()
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return t.from_numpy(a.copy()).to(DEV)


def workspace(qg, fmt, S, I, O, gs=0):
    t = torch()
    n = qg.qg_workspace_bytes(fmt, S, I, O, gs)
    return (t.empty(n, dtype=t.uint8, device=DEV) if n else None), n


def out(S, O):
    t = torch()
    y = t.empty(S * O, dtype=t.float32, device=DEV)
    y.fill_(float("nan"))           # every element must be overwritten
    return y


def host(y, S, O):
    torch().cuda.synchronize()
    return y.cpu().numpy().astype(np.float64).reshape(S, O)


def compare(y, ref, mag, tol=TOL, what=""):
    """Element-wise check against the oracle; NaN exactly where the oracle has
    NaN.  Returns the worst |err| / mag."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    nan_ref = np.isnan(ref)
    assert np.array_equal(np.isnan(y), nan_ref), f"{what}: NaN pattern differs"
    ok = ~nan_ref
    err = np.abs(y[ok] - ref[ok])
    m = np.asarray(mag, np.float64)[ok]
    bad = err > tol * m
    ratio = float(np.max(err / np.maximum(m, 1e-300))) if err.size else 0.0
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {err.size} outputs outside {tol} * sum|wx|; "
                           f"worst ratio {ratio:.3g}")
    return ratio


_ORC = None


def orc():
    global _ORC
    if _ORC is None:
        _ORC = oracle.Oracle()
    return _ORC


# ----------------------------------------------------------------------------
# inputs
# ----------------------------------------------------------------------------

def i4g_inputs(O, I, S, gs, tag=0, outlier=False):
    w, x = synth.fmt4_raw(O, I, S, tag)
    if outlier:
        x[0, min(5, I - 1)] = 50.0
    wq, sc = orc().quantize_i4g(w, O, I, gs)
    return x, wq, sc


def fp8_inputs(O, I, S, tag=2):
    return synth.fmt7_raw(O, I, S, tag)


def mq4_inputs(O, I, S, tag=3):
    w, x, d = synth.mq4_raw(O, I, S, tag)
    wr = orc().fwht256(w, d)
    xr = orc().fwht256(x, d)
    blocks = orc().encode_mq4v2(wr, O, I)
    return synth.bf16_bits(xr).reshape(S, I), blocks


def par_rows(method, O, *args, step=1, **kw):
    """Run an oracle GEMV method over row slices on all host cores (ctypes
    releases the GIL) and stitch the (y, mag) slices back together."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    n = max(1, os.cpu_count() or 1)
    chunk = max(step, -(-O // n))
    chunk = -(-chunk // step) * step
    bounds = [(o0, min(O, o0 + chunk)) for o0 in range(0, O, chunk)]
    with ThreadPoolExecutor(n) as ex:
        parts = list(ex.map(lambda b: method(*args, rows=b, **kw), bounds))
    return (np.concatenate([p[0] for p in parts], axis=1),
            np.concatenate([p[1] for p in parts], axis=1))

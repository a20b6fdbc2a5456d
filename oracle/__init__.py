"""CPU oracle for the weight-only quantized GEMV formats -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, double accumulation); this
module only compiles it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off: no fused multiply-add contraction, so the binary32 steps of
# the encoders round exactly as written on every host architecture.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-Wall", "-Wextra", "-Werror"]


def build(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``src`` into the shared library ``out`` with gcc."""
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def _declare(lib):
    P = ctypes.c_void_p
    i = ctypes.c_int
    z = ctypes.c_size_t
    lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_value.restype = ctypes.c_double
    lib.oracle_f16_value.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_value.restype = ctypes.c_double
    lib.oracle_f16_from_f32.argtypes = [ctypes.c_float]
    lib.oracle_f16_from_f32.restype = ctypes.c_uint16
    lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_value.restype = ctypes.c_double
    lib.oracle_qgemv_i4g.argtypes = [P, P, P, P, P, i, i, i, i]
    lib.oracle_qgemm_i4g.argtypes = [P, P, P, P, P, i, i, i, i]
    lib.oracle_quantize_i4g.argtypes = [P, P, P, i, i, i]
    lib.oracle_qgemv_fp8b128.argtypes = [P, P, P, P, P, i, i, i]
    lib.oracle_e8m0_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e8m0_value.restype = ctypes.c_double
    lib.oracle_qgemv_fp8ue8m0.argtypes = [P, P, P, P, P, i, i, i]
    lib.oracle_mq4v2_weight.argtypes = [P, i]
    lib.oracle_mq4v2_weight.restype = ctypes.c_double
    lib.oracle_qgemv_mq4v2.argtypes = [P, P, P, P, i, i, i]
    lib.oracle_encode_mq4v2.argtypes = [P, P, i, i]
    lib.oracle_mq4v1_weight.argtypes = [P, i]
    lib.oracle_mq4v1_weight.restype = ctypes.c_double
    lib.oracle_mq4c_weight.argtypes = [P, i]
    lib.oracle_mq4c_weight.restype = ctypes.c_double
    lib.oracle_qgemv_mq4v1.argtypes = [P, P, P, P, i, i, i]
    lib.oracle_qgemv_mq4c.argtypes = [P, P, P, P, i, i, i]
    lib.oracle_encode_mq4v1.argtypes = [P, P, i, i]
    lib.oracle_encode_mq4c.argtypes = [P, P, i, i]
    lib.oracle_qgemv_moe.argtypes = [i, P, P, P, z, P, P, i, P, i, i, i, i, i]
    lib.oracle_q2_0_weight.argtypes = [P, i]
    lib.oracle_q2_0_weight.restype = ctypes.c_double
    lib.oracle_qgemv_q2_0.argtypes = [P, P, P, P, i, i, i]
    lib.oracle_encode_q2_0.argtypes = [P, P, i, i]
    lib.oracle_qgemm_moe.argtypes = [i, P, P, P, P, P, i, P, P, i, i, i, i]
    lib.oracle_fwht256.argtypes = [P, P, P, z]
    lib.oracle_ifwht256.argtypes = [P, P, P, z]
    return lib


def load(path: str | None = None):
    """Return the ctypes handle of the oracle library, building it if needed.

    ``path`` loads a specific build (the mutation tests compile altered copies
    of ``oracle.c`` to show that the pins catch plausible mistakes).
    """
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            stale = (not os.path.exists(_LIB_PATH) or
                     os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
            if stale:
                build()
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """numpy front end over one build of ``oracle.c``."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load()

    # scalar formats -------------------------------------------------------
    def e4m3_value(self, code: int) -> float:
        return self.lib.oracle_e4m3_value(code)

    def f16_value(self, bits: int) -> float:
        return self.lib.oracle_f16_value(bits)

    def f16_from_f32(self, v: float) -> int:
        return self.lib.oracle_f16_from_f32(v)

    def bf16_value(self, bits: int) -> float:
        return self.lib.oracle_bf16_value(bits)

    # fmt=4 ------------------------------------------------------------------
    def qgemv_i4g(self, x, w, scales, S, I, O, gs, rows=None):
        """y, mag (float64 [S, O]); ``rows`` = (o0, o1) restricts to a row slice."""
        x = np.ascontiguousarray(x, np.float32)
        w = np.ascontiguousarray(w, np.uint8)
        scales = np.ascontiguousarray(scales, np.float32)
        o0, o1 = rows if rows is not None else (0, O)
        rb = (I + 1) // 2
        ng = (I + gs - 1) // gs
        ws = np.ascontiguousarray(w.reshape(O, rb)[o0:o1])
        ss = np.ascontiguousarray(scales.reshape(O, ng)[o0:o1])
        n = o1 - o0
        y = np.empty((S, n), np.float64)
        mag = np.empty((S, n), np.float64)
        self.lib.oracle_qgemv_i4g(_p(y), _p(mag), _p(x), _p(ws), _p(ss), S, I, n, gs)
        return y, mag

    def qgemm_i4g(self, X_bf16, w, scales, M, I, O, gs, rows=None):
        X = np.ascontiguousarray(X_bf16, np.uint16)
        w = np.ascontiguousarray(w, np.uint8)
        scales = np.ascontiguousarray(scales, np.float32)
        o0, o1 = rows if rows is not None else (0, O)
        rb = (I + 1) // 2
        ng = (I + gs - 1) // gs
        ws = np.ascontiguousarray(w.reshape(O, rb)[o0:o1])
        ss = np.ascontiguousarray(scales.reshape(O, ng)[o0:o1])
        n = o1 - o0
        Y = np.empty((M, n), np.float64)
        mag = np.empty((M, n), np.float64)
        self.lib.oracle_qgemm_i4g(_p(Y), _p(mag), _p(X), _p(ws), _p(ss), M, I, n, gs)
        return Y, mag

    def quantize_i4g(self, w, O, I, gs):
        w = np.ascontiguousarray(w, np.float32)
        rb = (I + 1) // 2
        ng = (I + gs - 1) // gs
        wq = np.empty((O, rb), np.uint8)
        sc = np.empty((O, ng), np.float32)
        self.lib.oracle_quantize_i4g(_p(wq), _p(sc), _p(w), O, I, gs)
        return wq, sc

    # fmt=7 ------------------------------------------------------------------
    def qgemv_fp8b128(self, x_bf16, w, scale_inv, S, I, O, rows=None):
        """``rows`` = (o0, o1) with o0 a multiple of 128 restricts to a row slice."""
        x = np.ascontiguousarray(x_bf16, np.uint16)
        w = np.ascontiguousarray(w, np.uint8)
        scale_inv = np.ascontiguousarray(scale_inv, np.float32)
        o0, o1 = rows if rows is not None else (0, O)
        assert o0 % 128 == 0
        nbi = (I + 127) // 128
        nbo = (O + 127) // 128
        ws = np.ascontiguousarray(w.reshape(O, I)[o0:o1])
        ss = np.ascontiguousarray(scale_inv.reshape(nbo, nbi)[o0 // 128:])
        n = o1 - o0
        y = np.empty((S, n), np.float64)
        mag = np.empty((S, n), np.float64)
        self.lib.oracle_qgemv_fp8b128(_p(y), _p(mag), _p(x), _p(ws), _p(ss), S, I, n)
        return y, mag

    # fmt=7 with UE8M0 scales ---------------------------------------------------
    def e8m0_value(self, code: int) -> float:
        return self.lib.oracle_e8m0_value(code)

    def qgemv_fp8ue8m0(self, x_bf16, w, scale_e8m0, S, I, O, rows=None):
        """``rows`` = (o0, o1) with o0 a multiple of 128 restricts to a row slice."""
        x = np.ascontiguousarray(x_bf16, np.uint16)
        w = np.ascontiguousarray(w, np.uint8)
        sc = np.ascontiguousarray(scale_e8m0, np.uint8)
        o0, o1 = rows if rows is not None else (0, O)
        assert o0 % 128 == 0
        nbi = (I + 127) // 128
        nbo = (O + 127) // 128
        ws = np.ascontiguousarray(w.reshape(O, I)[o0:o1])
        ss = np.ascontiguousarray(sc.reshape(nbo, nbi)[o0 // 128:])
        n = o1 - o0
        y = np.empty((S, n), np.float64)
        mag = np.empty((S, n), np.float64)
        self.lib.oracle_qgemv_fp8ue8m0(_p(y), _p(mag), _p(x), _p(ws), _p(ss), S, I, n)
        return y, mag

    # MQ4-V2 -----------------------------------------------------------------
    def mq4v2_weight(self, block: np.ndarray, j: int) -> float:
        block = np.ascontiguousarray(block, np.uint8)
        return self.lib.oracle_mq4v2_weight(_p(block), j)

    def qgemv_mq4v2(self, x_bf16, blocks, S, I, O, rows=None):
        x = np.ascontiguousarray(x_bf16, np.uint16)
        blocks = np.ascontiguousarray(blocks, np.uint8)
        o0, o1 = rows if rows is not None else (0, O)
        rowbytes = (I // 256) * 136
        bs = np.ascontiguousarray(blocks.reshape(O, rowbytes)[o0:o1])
        n = o1 - o0
        y = np.empty((S, n), np.float64)
        mag = np.empty((S, n), np.float64)
        self.lib.oracle_qgemv_mq4v2(_p(y), _p(mag), _p(x), _p(bs), S, I, n)
        return y, mag

    def encode_mq4v2(self, w, O, I):
        w = np.ascontiguousarray(w, np.float32)
        blocks = np.empty((O, (I // 256) * 136), np.uint8)
        self.lib.oracle_encode_mq4v2(_p(blocks), _p(w), O, I)
        return blocks

    # MQ4 v1 (qt=13) and MQ4C pad (qt=45) ------------------------------------
    def mq4v1_weight(self, block: np.ndarray, j: int) -> float:
        block = np.ascontiguousarray(block, np.uint8)
        return self.lib.oracle_mq4v1_weight(_p(block), j)

    def mq4c_weight(self, block: np.ndarray, j: int) -> float:
        block = np.ascontiguousarray(block, np.uint8)
        return self.lib.oracle_mq4c_weight(_p(block), j)

    def _qgemv_one_header(self, fn, x_bf16, blocks, S, I, O, rows=None):
        x = np.ascontiguousarray(x_bf16, np.uint16)
        blocks = np.ascontiguousarray(blocks, np.uint8)
        o0, o1 = rows if rows is not None else (0, O)
        rowbytes = (I // 256) * 136
        bs = np.ascontiguousarray(blocks.reshape(O, rowbytes)[o0:o1])
        n = o1 - o0
        y = np.empty((S, n), np.float64)
        mag = np.empty((S, n), np.float64)
        fn(_p(y), _p(mag), _p(x), _p(bs), S, I, n)
        return y, mag

    def qgemv_mq4v1(self, x_bf16, blocks, S, I, O, rows=None):
        return self._qgemv_one_header(self.lib.oracle_qgemv_mq4v1, x_bf16, blocks, S, I, O, rows)

    def qgemv_mq4c(self, x_bf16, blocks, S, I, O, rows=None):
        return self._qgemv_one_header(self.lib.oracle_qgemv_mq4c, x_bf16, blocks, S, I, O, rows)

    def encode_mq4v1(self, w, O, I):
        w = np.ascontiguousarray(w, np.float32)
        blocks = np.empty((O, (I // 256) * 136), np.uint8)
        self.lib.oracle_encode_mq4v1(_p(blocks), _p(w), O, I)
        return blocks

    def encode_mq4c(self, w, O, I):
        w = np.ascontiguousarray(w, np.float32)
        blocks = np.empty((O, (I // 256) * 136), np.uint8)
        self.lib.oracle_encode_mq4c(_p(blocks), _p(w), O, I)
        return blocks

    # Q2_0 -------------------------------------------------------------------
    def q2_0_weight(self, block: np.ndarray, e: int) -> float:
        block = np.ascontiguousarray(block, np.uint8)
        return self.lib.oracle_q2_0_weight(_p(block), e)

    def qgemv_q2_0(self, x_bf16, blocks, S, I, O, rows=None):
        x = np.ascontiguousarray(x_bf16, np.uint16)
        blocks = np.ascontiguousarray(blocks, np.uint8)
        o0, o1 = rows if rows is not None else (0, O)
        rowbytes = (I // 64) * 18
        bs = np.ascontiguousarray(blocks.reshape(O, rowbytes)[o0:o1])
        n = o1 - o0
        y = np.empty((S, n), np.float64)
        mag = np.empty((S, n), np.float64)
        self.lib.oracle_qgemv_q2_0(_p(y), _p(mag), _p(x), _p(bs), S, I, n)
        return y, mag

    def encode_q2_0(self, w, O, I):
        w = np.ascontiguousarray(w, np.float32)
        blocks = np.empty((O, (I // 64) * 18), np.uint8)
        self.lib.oracle_encode_q2_0(_p(blocks), _p(w), O, I)
        return blocks

    # routed experts -----------------------------------------------------------
    def qgemv_moe(self, fmt, x, x_slot_stride, weights, scales, ids, S, I, O, gs=0):
        """y, mag (float64 [n_slots, S, O]).  ``weights`` / ``scales`` are
        per-expert numpy arrays (scales None for the MQ4 formats); ``x`` is f32
        for fmt=4 and bf16 bits otherwise."""
        x = np.ascontiguousarray(x, np.float32 if fmt == 4 else np.uint16)
        ws = [np.ascontiguousarray(w, np.uint8) for w in weights]
        sdt = np.uint8 if fmt == 71 else np.float32       # UE8M0 scales are bytes
        ss = [None if sc is None else np.ascontiguousarray(sc, sdt) for sc in scales]
        ids = np.ascontiguousarray(ids, np.int32)
        n = len(ids)
        wp = (ctypes.c_void_p * len(ws))(*[w.ctypes.data for w in ws])
        sp = (ctypes.c_void_p * len(ss))(*[0 if sc is None else sc.ctypes.data for sc in ss])
        y = np.empty((n, S, O), np.float64)
        mag = np.empty((n, S, O), np.float64)
        self.lib.oracle_qgemv_moe(fmt, _p(y), _p(mag), _p(x), x_slot_stride, ctypes.cast(wp, ctypes.c_void_p),
                                  ctypes.cast(sp, ctypes.c_void_p), len(ws), _p(ids), n, S, I, O, gs)
        return y, mag

    def qgemm_moe(self, fmt, X_bf16, weights, scales, group_expert, offsets, I, O, gs=0):
        """Y, mag (float64 [M, O], M = offsets[-1]; rows no group covers are NaN)."""
        X = np.ascontiguousarray(X_bf16, np.uint16)
        ws = [np.ascontiguousarray(w, np.uint8) for w in weights]
        sdt = np.uint8 if fmt == 71 else np.float32
        ss = [None if sc is None else np.ascontiguousarray(sc, sdt) for sc in scales]
        ge = np.ascontiguousarray(group_expert, np.int32)
        off = np.ascontiguousarray(offsets, np.int32)
        M = int(off[-1])
        wp = (ctypes.c_void_p * len(ws))(*[w.ctypes.data for w in ws])
        sp = (ctypes.c_void_p * len(ss))(*[0 if sc is None else sc.ctypes.data for sc in ss])
        Y = np.full((M, O), np.nan)
        mag = np.full((M, O), np.nan)
        self.lib.oracle_qgemm_moe(fmt, _p(Y), _p(mag), _p(X), ctypes.cast(wp, ctypes.c_void_p),
                                  ctypes.cast(sp, ctypes.c_void_p), len(ws), _p(ge), _p(off), len(ge), I, O, gs)
        return Y, mag

    # FWHT -------------------------------------------------------------------
    def fwht256(self, v, signs):
        v = np.ascontiguousarray(v, np.float32)
        signs = np.ascontiguousarray(signs, np.int8)
        assert v.size % 256 == 0 and signs.size == 256
        out = np.empty_like(v)
        self.lib.oracle_fwht256(_p(out), _p(v), _p(signs), v.size // 256)
        return out

    def ifwht256(self, v, signs):
        v = np.ascontiguousarray(v, np.float32)
        signs = np.ascontiguousarray(signs, np.int8)
        out = np.empty_like(v)
        self.lib.oracle_ifwht256(_p(out), _p(v), _p(signs), v.size // 256)
        return out

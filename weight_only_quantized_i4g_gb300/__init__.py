"""Python binding of libqgemv (weight-only quantized GEMV / GEMM for GB300).

Argument marshalling only: each function takes the same arguments as the C
entry point of the same name in ``include/qgemv.h`` -- device pointers given
as ``torch.Tensor`` (its ``data_ptr()``) or plain integers, sizes as ints, a
CUDA stream as a ``torch.cuda.Stream``, a raw handle or None (the current
torch stream) -- and returns the C status code.  ``check(rc)`` turns a
non-zero status into ``QGError``.  Every computation runs in the CUDA library;
importing this package fails if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqgemv.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        "libqgemv.so is not built; run `python -c 'import __graft_entry__ as g; g.build()'` "
        "(or `python weight_only_quantized_i4g_gb300/_build.py`)")

_lib = ctypes.CDLL(LIB_PATH)

QG_OK, QG_EINVAL, QG_EGS, QG_ESHAPE, QG_EALIGN, QG_EWORKSPACE, QG_ECUDA, QG_ETIMEOUT, QG_EEXPERT, QG_EBOUNDS = (
    0, -1, -2, -3, -4, -5, -6, -7, -8, -9)
QG_FMT_I4G, QG_FMT_FP8B128, QG_FMT_FP8UE8M0, QG_FMT_MQ4V1, QG_FMT_MQ4V2, QG_FMT_MQ4C, QG_FMT_Q2_0 = (
    4, 7, 71, 13, 44, 45, 20)

_P = ctypes.c_void_p
_I = ctypes.c_int
_Z = ctypes.c_size_t

_SIGNATURES = {
    "qg_strerror": ([_I], ctypes.c_char_p),
    "qg_last_error": ([], ctypes.c_char_p),
    "qg_workspace_bytes": ([_I, _I, _I, _I, _I], _Z),
    "qg_gemm_workspace_bytes": ([_I, _I, _I, _I, _I], _Z),
    "qg_device_status": ([ctypes.POINTER(_I)], _I),
    "qg_launch_count": ([], ctypes.c_ulonglong),
    "qg_selftest_wait_timeout": ([_I, ctypes.POINTER(_I)], _I),
    "qg_stamps_take": ([ctypes.POINTER(ctypes.c_uint64), _I], _I),
    "qg_selftest_pdl_chain": ([_I, _I, _I, _P], _I),
    "qgemv_i4g": ([_P, _P, _P, _P, _I, _I, _I, _I, _P, _Z, _P], _I),
    "qgemv_i4g_noalloc": ([_P, _P, _P, _P, _I, _I, _I, _I, _P], _I),
    "qgemv_fp8b128": ([_P, _P, _P, _P, _I, _I, _I, _P, _Z, _P], _I),
    "qgemv_mq4v2": ([_P, _P, _P, _I, _I, _I, _P, _Z, _P], _I),
    "qgemm_i4g": ([_P, _P, _P, _P, _I, _I, _I, _I, _P, _Z, _P], _I),
    "qgemm_fp8b128": ([_P, _P, _P, _P, _I, _I, _I, _P, _Z, _P], _I),
    "qgemm_mq4v2": ([_P, _P, _P, _I, _I, _I, _P, _Z, _P], _I),
    "qgemv_mq4v1": ([_P, _P, _P, _I, _I, _I, _P, _Z, _P], _I),
    "qgemv_mq4c": ([_P, _P, _P, _I, _I, _I, _P, _Z, _P], _I),
    "qgemm_mq4v1": ([_P, _P, _P, _I, _I, _I, _P, _Z, _P], _I),
    "qgemm_mq4c": ([_P, _P, _P, _I, _I, _I, _P, _Z, _P], _I),
    "qgemv_q2_0": ([_P, _P, _P, _I, _I, _I, _P, _Z, _P], _I),
    "qgemv_fp8ue8m0": ([_P, _P, _P, _P, _I, _I, _I, _P, _Z, _P], _I),
    "qgemm_fp8ue8m0": ([_P, _P, _P, _P, _I, _I, _I, _P, _Z, _P], _I),
    "qgemv_moe": ([_I, _P, _P, _Z, _P, _I, _P, _I, _I, _I, _I, _I, _P], _I),
    "qgemm_moe": ([_I, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _Z, _P], _I),
    "qg_moe_gemm_workspace_bytes": ([_I, _P, _I, _I, _I, _I], _Z),
    "qg_encode_mq4v1": ([_P, _P, _I, _I, _P], _I),
    "qg_encode_mq4c": ([_P, _P, _I, _I, _P], _I),
    "qg_quantize_i4g": ([_P, _P, _P, _I, _I, _I, _P], _I),
    "qg_encode_mq4v2": ([_P, _P, _I, _I, _P], _I),
    "qg_fwht256": ([_P, _P, _P, _Z, _P], _I),
}
for _name, (_args, _res) in _SIGNATURES.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res

EXPORTED = tuple(_SIGNATURES)


class QGError(RuntimeError):
    def __init__(self, status: int):
        self.status = status
        super().__init__(f"{strerror(status)} -- {last_error()}")


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def strerror(status: int) -> str:
    return _lib.qg_strerror(status).decode()


def last_error() -> str:
    return _lib.qg_last_error().decode()


def check(rc: int) -> None:
    if rc != QG_OK:
        raise QGError(rc)


def qg_device_status() -> tuple[int, int]:
    """(return code, device status) of the current device; clears the status."""
    st = _I(0)
    rc = _lib.qg_device_status(ctypes.byref(st))
    return rc, st.value


def qg_launch_count() -> int:
    """Kernels the library has launched in this process."""
    return _lib.qg_launch_count()


def qg_selftest_wait_timeout(spin_limit: int) -> tuple[int, int]:
    """(status, observed bits) of the failure-path test aid."""
    v = _I(0)
    rc = _lib.qg_selftest_wait_timeout(spin_limit, ctypes.byref(v))
    return rc, v.value


STAMP_SLOTS = 8        # words per block of qg_stamps_take
STAMP_BLOCKS = 2048    # blocks it records


def qg_stamps_take(max_blocks: int = STAMP_BLOCKS, lib=None):
    """(status, list of per-block 8-word lists) from qg_stamps_take of `lib`
    (a ctypes handle of the stamps build; this package's library refuses)."""
    lib = lib if lib is not None else _lib
    buf = (ctypes.c_uint64 * (STAMP_SLOTS * max_blocks))()
    f = lib.qg_stamps_take
    f.argtypes = [ctypes.POINTER(ctypes.c_uint64), _I]
    f.restype = _I
    rc = f(buf, max_blocks)
    words = list(buf)
    return rc, [words[STAMP_SLOTS * b:STAMP_SLOTS * (b + 1)] for b in range(max_blocks)]


def qg_selftest_pdl_chain(blocks: int, threads: int, launches: int, stream=None) -> int:
    return _lib.qg_selftest_pdl_chain(blocks, threads, launches, _stream(stream))


def qg_workspace_bytes(fmt: int, S: int, I: int, O: int, gs: int = 0) -> int:
    return _lib.qg_workspace_bytes(fmt, S, I, O, gs)


def qg_gemm_workspace_bytes(fmt: int, M: int, I: int, O: int, gs: int = 0) -> int:
    return _lib.qg_gemm_workspace_bytes(fmt, M, I, O, gs)


def qgemv_i4g(y, x, w, scales, S, I, O, gs, ws=None, ws_bytes=0, stream=None) -> int:
    return _lib.qgemv_i4g(_ptr(y), _ptr(x), _ptr(w), _ptr(scales), S, I, O, gs, _ptr(ws), ws_bytes,
                          _stream(stream))


def qgemv_i4g_noalloc(y, x, w, scales, S, I, O, gs, stream=None) -> int:
    return _lib.qgemv_i4g_noalloc(_ptr(y), _ptr(x), _ptr(w), _ptr(scales), S, I, O, gs, _stream(stream))


def qgemv_q2_0(y, x, blocks, S, I, O, ws=None, ws_bytes=0, stream=None) -> int:
    return _lib.qgemv_q2_0(_ptr(y), _ptr(x), _ptr(blocks), S, I, O, _ptr(ws), ws_bytes, _stream(stream))


def qgemv_fp8ue8m0(y, x, w, scale_e8m0, S, I, O, ws=None, ws_bytes=0, stream=None) -> int:
    return _lib.qgemv_fp8ue8m0(_ptr(y), _ptr(x), _ptr(w), _ptr(scale_e8m0), S, I, O, _ptr(ws), ws_bytes,
                               _stream(stream))


def qgemm_fp8ue8m0(Y, X, w, scale_e8m0, M, I, O, ws=None, ws_bytes=0, stream=None) -> int:
    return _lib.qgemm_fp8ue8m0(_ptr(Y), _ptr(X), _ptr(w), _ptr(scale_e8m0), M, I, O, _ptr(ws), ws_bytes,
                               _stream(stream))


def qgemv_moe(fmt, y, x, x_slot_stride, experts, n_experts, ids, n_slots, S, I, O, gs=0, stream=None) -> int:
    """Routed-expert GEMV; `experts` is a device array of qg_expert {w, scales}
    pointer pairs (see ``expert_table``), `ids` a device int32 array."""
    return _lib.qgemv_moe(fmt, _ptr(y), _ptr(x), x_slot_stride, _ptr(experts), n_experts, _ptr(ids), n_slots,
                          S, I, O, gs, _stream(stream))


def qgemm_moe(fmt, Y, X, experts, n_experts, group_expert, group_offsets, n_groups, I, O, gs=0, ws=None,
              ws_bytes=0, stream=None) -> int:
    """Routed-expert prefill GEMM.  ``experts`` (bytes from ``expert_table``),
    ``group_expert`` and ``group_offsets`` (int sequences) are host data."""
    import array
    ge = array.array("i", [int(v) for v in group_expert])
    off = array.array("i", [int(v) for v in group_offsets])
    ex = ctypes.create_string_buffer(bytes(experts), len(experts)) if experts is not None else None
    return _lib.qgemm_moe(fmt, _ptr(Y), _ptr(X), ctypes.addressof(ex) if ex is not None else None, n_experts,
                          ge.buffer_info()[0] if len(ge) else None, off.buffer_info()[0] if len(off) else None,
                          n_groups, I, O, gs, _ptr(ws), ws_bytes, _stream(stream))


def qg_moe_gemm_workspace_bytes(fmt, group_offsets, n_groups, I, O, gs=0) -> int:
    import array
    off = array.array("i", [int(v) for v in group_offsets])
    return _lib.qg_moe_gemm_workspace_bytes(fmt, off.buffer_info()[0] if len(off) else None, n_groups, I, O, gs)


def expert_table(pairs):
    """Host bytes of a qg_expert array: one (weights, scales) pair of device
    pointers (tensors, ints or None) per expert, two little-endian uint64
    each.  Upload them to device memory to pass to qgemv_moe."""
    import struct
    return b"".join(struct.pack("<QQ", _ptr(w) or 0, _ptr(sc) or 0) for w, sc in pairs)


def qgemv_fp8b128(y, x, w, scale_inv, S, I, O, ws=None, ws_bytes=0, stream=None) -> int:
    return _lib.qgemv_fp8b128(_ptr(y), _ptr(x), _ptr(w), _ptr(scale_inv), S, I, O, _ptr(ws), ws_bytes,
                              _stream(stream))


def qgemv_mq4v2(y, x, blocks, S, I, O, ws=None, ws_bytes=0, stream=None) -> int:
    return _lib.qgemv_mq4v2(_ptr(y), _ptr(x), _ptr(blocks), S, I, O, _ptr(ws), ws_bytes, _stream(stream))


def qgemm_i4g(Y, X, w, scales, M, I, O, gs, ws=None, ws_bytes=0, stream=None) -> int:
    return _lib.qgemm_i4g(_ptr(Y), _ptr(X), _ptr(w), _ptr(scales), M, I, O, gs, _ptr(ws), ws_bytes,
                          _stream(stream))


def qgemm_fp8b128(Y, X, w, scale_inv, M, I, O, ws=None, ws_bytes=0, stream=None) -> int:
    return _lib.qgemm_fp8b128(_ptr(Y), _ptr(X), _ptr(w), _ptr(scale_inv), M, I, O, _ptr(ws), ws_bytes,
                              _stream(stream))


def qgemm_mq4v2(Y, X, blocks, M, I, O, ws=None, ws_bytes=0, stream=None) -> int:
    return _lib.qgemm_mq4v2(_ptr(Y), _ptr(X), _ptr(blocks), M, I, O, _ptr(ws), ws_bytes, _stream(stream))


def qgemv_mq4v1(y, x, blocks, S, I, O, ws=None, ws_bytes=0, stream=None) -> int:
    return _lib.qgemv_mq4v1(_ptr(y), _ptr(x), _ptr(blocks), S, I, O, _ptr(ws), ws_bytes, _stream(stream))


def qgemv_mq4c(y, x, blocks, S, I, O, ws=None, ws_bytes=0, stream=None) -> int:
    return _lib.qgemv_mq4c(_ptr(y), _ptr(x), _ptr(blocks), S, I, O, _ptr(ws), ws_bytes, _stream(stream))


def qgemm_mq4v1(Y, X, blocks, M, I, O, ws=None, ws_bytes=0, stream=None) -> int:
    return _lib.qgemm_mq4v1(_ptr(Y), _ptr(X), _ptr(blocks), M, I, O, _ptr(ws), ws_bytes, _stream(stream))


def qgemm_mq4c(Y, X, blocks, M, I, O, ws=None, ws_bytes=0, stream=None) -> int:
    return _lib.qgemm_mq4c(_ptr(Y), _ptr(X), _ptr(blocks), M, I, O, _ptr(ws), ws_bytes, _stream(stream))


def qg_encode_mq4v1(blocks, w, O, I, stream=None) -> int:
    return _lib.qg_encode_mq4v1(_ptr(blocks), _ptr(w), O, I, _stream(stream))


def qg_encode_mq4c(blocks, w, O, I, stream=None) -> int:
    return _lib.qg_encode_mq4c(_ptr(blocks), _ptr(w), O, I, _stream(stream))


def qg_quantize_i4g(wq, scales, w, O, I, gs, stream=None) -> int:
    return _lib.qg_quantize_i4g(_ptr(wq), _ptr(scales), _ptr(w), O, I, gs, _stream(stream))


def qg_encode_mq4v2(blocks, w, O, I, stream=None) -> int:
    return _lib.qg_encode_mq4v2(_ptr(blocks), _ptr(w), O, I, _stream(stream))


def qg_fwht256(out, inp, signs, n_blocks, stream=None) -> int:
    return _lib.qg_fwht256(_ptr(out), _ptr(inp), _ptr(signs), n_blocks, _stream(stream))

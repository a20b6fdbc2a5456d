"""Child process of test_zz_no_alloc.py: qgemv_i4g_noalloc, then
cudaDeviceReset, then qgemv_i4g_noalloc and qgemv_i4g again, each output
compared with the oracle.

A reset destroys the context and every allocation in it (torch's included),
so this process holds its buffers through the CUDA runtime directly and never
imports torch.  After the reset the runtime makes a new context, in which the
library's scratch array and error word have new device addresses; a library
that kept the old ones would write through stale pointers.  Exits non-zero on
any mismatch or error."""
import ctypes
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import weight_only_quantized_i4g_gb300 as qg  # noqa: E402  (loads libqgemv.so and its libcudart)
from gpu_util import TOL, i4g_inputs, orc  # noqa: E402

rt = ctypes.CDLL("libcudart.so.13")        # the runtime libqgemv.so is linked against
rt.cudaMalloc.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t]
rt.cudaFree.argtypes = [ctypes.c_void_p]
rt.cudaMemcpy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
H2D, D2H = 1, 2


def ok(e, what):
    if e != 0:
        raise SystemExit(f"{what}: cudaError {e}")


def upload(a):
    a = np.ascontiguousarray(a)
    p = ctypes.c_void_p()
    ok(rt.cudaMalloc(ctypes.byref(p), a.nbytes), "cudaMalloc")
    ok(rt.cudaMemcpy(p, a.ctypes.data, a.nbytes, H2D), "cudaMemcpy H2D")
    return p.value


def run(entry, O, I, S, gs, tag):
    x, wq, sc = i4g_inputs(O, I, S, gs, tag=tag)
    want, mag = orc().qgemv_i4g(x, wq, sc, S, I, O, gs)
    bufs = [upload(x), upload(wq), upload(sc)]
    yp = ctypes.c_void_p()
    ok(rt.cudaMalloc(ctypes.byref(yp), S * O * 4), "cudaMalloc y")
    if entry == "noalloc":
        rc = qg.qgemv_i4g_noalloc(yp.value, bufs[0], bufs[1], bufs[2], S, I, O, gs, 0)
    else:
        n = qg.qg_workspace_bytes(qg.QG_FMT_I4G, S, I, O, gs)
        wsp = ctypes.c_void_p()
        ok(rt.cudaMalloc(ctypes.byref(wsp), n), "cudaMalloc ws")
        bufs.append(wsp.value)
        rc = qg.qgemv_i4g(yp.value, bufs[0], bufs[1], bufs[2], S, I, O, gs, wsp.value, n, 0)
    qg.check(rc)
    ok(rt.cudaDeviceSynchronize(), "cudaDeviceSynchronize")
    got = np.empty(S * O, np.float32)
    ok(rt.cudaMemcpy(got.ctypes.data, yp, S * O * 4, D2H), "cudaMemcpy D2H")
    for p in bufs + [yp.value]:
        ok(rt.cudaFree(ctypes.c_void_p(p)), "cudaFree")
    err = np.abs(got.reshape(S, O).astype(np.float64) - want)
    ratio = float(np.max(err / mag))
    if not np.all(err <= TOL * mag):
        raise SystemExit(f"{entry} tag {tag}: worst |err|/sum|wx| {ratio:.3g} above {TOL}")
    print(f"{entry} tag {tag}: worst |err|/sum|wx| {ratio:.2e}")


def main():
    O, I, S, gs = 64, 16384, 2, 64     # splits the reduction: the scratch array is used
    run("noalloc", O, I, S, gs, tag=501)
    ok(rt.cudaDeviceReset(), "cudaDeviceReset")
    run("noalloc", O, I, S, gs, tag=502)
    run("noalloc", O, I, S, gs, tag=503)
    run("workspace", O, I, S, gs, tag=504)
    rc, status = qg.qg_device_status()
    if rc != qg.QG_OK or status != qg.QG_OK:
        raise SystemExit(f"qg_device_status after the reset: rc {rc}, status {status}")
    print("ok")


if __name__ == "__main__":
    main()

"""The kernels' failure path on the GPU, made to run without a fault.

Every barrier wait of the staging pipeline is bounded; one that gives up
records QG_ETIMEOUT in the per-device error word, ends the block's other
waits, lands the copies it issued and leaves (fp8 page, colibri PR #528,
validation: failures are loud).  qg_selftest_wait_timeout runs that pipeline
with a batch that is never issued and a short poll limit; the test checks
what the block saw, that qg_device_status reports and clears the timeout,
that the call returns promptly, and that the context still computes
correctly afterwards."""
import time

import pytest

from gpu_util import compare, dev, host, i4g_inputs, orc, out, par_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qg():
    import weight_only_quantized_i4g_gb300 as m
    return m


def test_wait_timeout_is_reported_and_cleared(qg):
    rc, status = qg.qg_device_status()
    assert rc == qg.QG_OK and status == qg.QG_OK, "error word not clean before the test"
    t0 = time.perf_counter()
    rc, seen = qg.qg_selftest_wait_timeout(4096)
    dt = time.perf_counter() - t0
    assert rc == qg.QG_OK, qg.last_error()
    assert seen == 7, f"observed bits {seen:#x}: 1 consumer gave up, 2 producer ended on abort, 4 copy landed"
    assert dt < 5.0, f"a 4096-poll wait took {dt:.2f} s"
    rc, status = qg.qg_device_status()
    assert rc == qg.QG_OK and status == qg.QG_ETIMEOUT, (rc, status)
    rc, status = qg.qg_device_status()          # read once, then cleared
    assert rc == qg.QG_OK and status == qg.QG_OK, (rc, status)


def test_context_usable_after_timeout(qg):
    rc, _ = qg.qg_selftest_wait_timeout(1024)
    assert rc == qg.QG_OK
    qg.qg_device_status()
    O, I, S, gs = 512, 2048, 1, 64
    x, wq, sc = i4g_inputs(O, I, S, gs, tag=77)
    y = out(S, O)
    qg.check(qg.qgemv_i4g(y, dev(x), dev(wq), dev(sc), S, I, O, gs))
    got = host(y, S, O)
    ref, mag = par_rows(orc().qgemv_i4g, O, x, wq, sc, S, I, O, gs)
    compare(got, ref, mag, what="fmt4 after a timed-out wait")
    rc, status = qg.qg_device_status()
    assert rc == qg.QG_OK and status == qg.QG_OK

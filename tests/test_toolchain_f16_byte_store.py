"""A toolchain observation behind the encoders' 32-bit stores, reproduced.

tests/f16_byte_store_repro.cu stores the low byte of an fp16 conversion
result with an 8-bit store in four forms.  On nvcc 13.0 for sm_103a (at any
optimisation level, and from JIT-compiled compute_100 PTX), the form that
stores the .b16 register written by cvt.rn.f16.f32 directly with
st.global.b8 -- which is what the C++ expression
(uint8_t)(__half_as_ushort(__float2half_rn(v)) & 0xFF) compiles to -- was
measured to store 0 in place of every nonzero byte, while widening the value
first (cvt.u32.u16, or a move to a .u16 register) stores it correctly.  The
library's encoders therefore assemble and store whole 32-bit words.  This
test requires the widened forms to be right and reports what the direct
forms did (a later toolchain may store them correctly too)."""
import os
import re
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_f16_low_byte_stores(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / "f16_byte_store_repro")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", exe,
                    os.path.join(HERE, "f16_byte_store_repro.cu")], check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    forms = {int(m.group(1)): (m.group(2), int(m.group(3)), int(m.group(4)))
             for m in re.finditer(r"form (\d): (.+?) wrong (\d+) zero (\d+)", r.stdout)}
    assert sorted(forms) == [0, 1, 2, 3], r.stdout
    for f in (1, 2):
        err, wrong, _ = forms[f]
        assert err == "no error" and wrong == 0, f"widened form {f}: {r.stdout}"
    nonzero = int(re.search(r"reference low bytes nonzero (\d+)", r.stdout).group(1))
    assert nonzero > 0
    print(f"direct 8-bit stores of the fp16 result: form 0 wrong {forms[0][1]} (zero {forms[0][2]}), "
          f"form 3 wrong {forms[3][1]} (zero {forms[3][2]}) of {nonzero} nonzero bytes")

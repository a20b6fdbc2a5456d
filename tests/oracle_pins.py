"""Pins for the CPU oracle: checks against what the pages and mathematics fix.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with something other than itself:

* values the pages define, written out by hand in ``tests/golden/``;
* library routines that implement the same number formats independently
  (``torch.float8_e4m3fn``, numpy ``float16``, torch ``bfloat16``,
  ``scipy.linalg.hadamard``, ``numpy.matmul`` on an explicitly dequantized
  matrix built with vectorised numpy from the layout description);
* closed forms, invariants and special cases (single group, equal half
  headers, lattice weights, orthonormality, exact extremes).

``test_oracle_mutations.py`` compiles altered copies of ``oracle.c`` and
checks that every plausible mistake fails at least one pin.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _close(a, b, mag, rtol=1e-12, what=""):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    err = np.abs(a - b)
    bound = rtol * np.maximum(np.asarray(mag, np.float64), 1e-300)
    bad = ~(err <= bound)
    if bad.any():
        with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
            worst = np.nanmax(err / bound)
        raise AssertionError(f"{what}: {bad.sum()} mismatches, worst {worst:.3g}x bound")


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def pin_e4m3_golden(orc):
    g = _golden("e4m3_spot.json")
    for code_s, want in g["codes"].items():
        code = int(code_s, 16)
        got = orc.e4m3_value(code)
        if want == "nan":
            assert math.isnan(got), (code_s, got)
        elif want == "-0.0":
            assert got == 0.0 and math.copysign(1.0, got) < 0, (code_s, got)
        else:
            assert got == want, (code_s, got, want)


def pin_e4m3_vs_torch(orc):
    import torch
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([orc.e4m3_value(c) for c in range(256)])
    nan_ref, nan_got = np.isnan(ref), np.isnan(got)
    assert np.array_equal(nan_ref, nan_got)
    assert set(np.nonzero(nan_got)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ref[~nan_ref], got[~nan_got])
    assert np.array_equal(np.signbit(ref[~nan_ref]), np.signbit(got[~nan_got]))


def pin_e4m3_structure(orc):
    vals = [orc.e4m3_value(c) for c in range(256)]
    # the 14 non-zero subnormals (exponent field 0) are m * 2^-9, both signs
    for m in range(1, 8):
        assert vals[m] == m * 2.0 ** -9 and vals[0x80 | m] == -m * 2.0 ** -9
    # positive codes are strictly increasing up to the largest finite value
    pos = vals[0:0x7F]
    assert all(a < b for a, b in zip(pos, pos[1:]))
    assert pos[-1] == 448.0
    # sign symmetry
    for c in range(0x7F):
        assert vals[0x80 | c] == -vals[c] or (c == 0 and vals[0x80] == 0.0)


def pin_f16_decode_vs_numpy(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.f16_value(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))


def pin_f16_encode_vs_numpy(orc):
    rng = np.random.default_rng(7)
    # every f16 value, every midpoint between neighbours (ties), their float32
    # neighbours, random magnitudes across the whole range, and overflow
    f16 = np.arange(0, 0x7C00, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)
    mids = ((f16[:-1] + f16[1:]) / 2).astype(np.float32)
    near = np.concatenate([np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(np.inf))])
    rnd = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 12, 20000))).astype(np.float32)
    edge = np.array([0.0, -0.0, 65504, 65519.99, 65520, 70000, 1e30, 2.0 ** -24, 2.0 ** -25,
                     2.0 ** -25 * 1.0000001, 2.0 ** -14, 2.0 ** -14 * (1 - 2 ** -12)], np.float32)
    vals = np.concatenate([f16.astype(np.float32), mids, near, rnd, -rnd, edge, -edge])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([orc.f16_from_f32(float(v)) for v in vals], np.uint16)
    bad = np.nonzero(ref != got)[0]
    assert bad.size == 0, [(float(vals[i]), hex(ref[i]), hex(got[i])) for i in bad[:5]]


def pin_bf16_decode_vs_torch(orc):
    import torch
    bits = np.arange(0, 65536, 97, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([orc.bf16_value(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


# ---------------------------------------------------------------------------
# fmt=4 grouped int4
# ---------------------------------------------------------------------------

def _dequant_i4g_numpy(w, scales, O, I, gs):
    """Explicit dequantization from the layout description (vectorised)."""
    rb = (I + 1) // 2
    b = np.asarray(w, np.uint8).reshape(O, rb)
    nib = np.stack([b & 0xF, b >> 4], axis=-1).reshape(O, 2 * rb)[:, :I].astype(np.float64) - 8.0
    ng = (I + gs - 1) // gs
    sc = np.repeat(np.asarray(scales, np.float32).reshape(O, ng).astype(np.float64), gs, axis=1)[:, :I]
    return nib * sc


def pin_i4g_golden(orc):
    g = _golden("i4g_hand.json")
    y, mag = orc.qgemv_i4g(np.array(g["x"], np.float32), np.array(g["w"], np.uint8),
                           np.array(g["scales"], np.float32), 1, g["I"], g["O"], g["gs"])
    assert np.array_equal(y[0], g["y"]), (y, g["y"])
    assert np.array_equal(mag[0], g["mag"]), (mag, g["mag"])


def pin_i4g_bruteforce(orc):
    """Tiny shapes, every gs of the loader's list: oracle == dequantize + matmul."""
    rng = np.random.default_rng(11)
    for O in (1, 2, 3):
        for I in (1, 2, 39, 40, 63, 64, 65, 200, 201, 512):
            for gs in (16, 32, 48, 64, 96, 128, 192, 256):
                rb, ng = (I + 1) // 2, (I + gs - 1) // gs
                w = rng.integers(0, 256, O * rb, dtype=np.uint8)
                sc = rng.uniform(-2, 2, O * ng).astype(np.float32)
                S = 2
                x = rng.standard_normal(S * I).astype(np.float32)
                y, mag = orc.qgemv_i4g(x, w, sc, S, I, O, gs)
                W = _dequant_i4g_numpy(w, sc, O, I, gs)
                ref = x.reshape(S, I).astype(np.float64) @ W.T
                refmag = np.abs(x.reshape(S, I).astype(np.float64)) @ np.abs(W).T
                _close(y, ref, refmag, what=f"i4g O={O} I={I} gs={gs}")
                _close(mag, refmag, refmag, what="i4g mag")


def pin_i4g_gemm_bruteforce(orc):
    """Batched prefill (colibri PR #457, section 4: the large-batch path computes
    the grouped product of section 3 for every token row): Y and the tolerance
    denominator mag = sum |w x| against numpy dequantize + matmul with bf16
    activations, tiny shapes, every gs of the loader's list, odd I."""
    rng = np.random.default_rng(13)
    for O in (1, 3):
        for I in (1, 39, 64, 65, 201, 512):
            for gs in (16, 32, 48, 64, 96, 128, 192, 256):
                rb, ng = (I + 1) // 2, (I + gs - 1) // gs
                w = rng.integers(0, 256, O * rb, dtype=np.uint8)
                sc = rng.uniform(-2, 2, O * ng).astype(np.float32)
                M = 3
                xb = synth.bf16_bits(rng.standard_normal(M * I).astype(np.float32))
                Y, mag = orc.qgemm_i4g(xb, w, sc, M, I, O, gs)
                W = _dequant_i4g_numpy(w, sc, O, I, gs)
                X = synth.bf16_to_f32(xb).reshape(M, I).astype(np.float64)
                refmag = np.abs(X) @ np.abs(W).T
                _close(Y, X @ W.T, refmag, what=f"i4g gemm O={O} I={I} gs={gs}")
                _close(mag, refmag, refmag, what=f"i4g gemm mag O={O} I={I} gs={gs}")


def pin_i4g_single_group(orc):
    """gs >= I: one scale per row, y = scale * sum (n-8) x (the per-row form)."""
    rng = np.random.default_rng(12)
    O, I, gs = 5, 40, 64
    rb = (I + 1) // 2
    w = rng.integers(0, 256, O * rb, dtype=np.uint8)
    sc = rng.uniform(0.1, 1, O).astype(np.float32)
    x = rng.integers(-4, 5, I).astype(np.float32)          # small integers: exact sums
    y, _ = orc.qgemv_i4g(x, w, sc, 1, I, O, gs)
    b = w.reshape(O, rb)
    for o in range(O):
        ints = []
        for byte in b[o]:
            ints += [int(byte) % 16 - 8, int(byte) // 16 - 8]
        dot = sum(q * int(v) for q, v in zip(ints[:I], x))   # exact integer dot
        assert y[0, o] == float(sc[o]) * dot, (o, y[0, o], float(sc[o]) * dot)


def pin_i4g_pad_nibble_ignored(orc):
    """Odd I: the unused high nibble of the last byte never contributes."""
    rng = np.random.default_rng(13)
    O, I, gs = 3, 201, 64
    rb, ng = (I + 1) // 2, (I + gs - 1) // gs
    w = rng.integers(0, 256, (O, rb), dtype=np.uint8)
    sc = rng.uniform(-1, 1, O * ng).astype(np.float32)
    x = rng.standard_normal(I).astype(np.float32)
    w0 = w.copy(); w0[:, -1] &= 0x0F
    w1 = w.copy(); w1[:, -1] |= 0xF0
    y0, _ = orc.qgemv_i4g(x, w0, sc, 1, I, O, gs)
    y1, _ = orc.qgemv_i4g(x, w1, sc, 1, I, O, gs)
    assert np.array_equal(y0, y1)


def pin_i4g_basis(orc):
    """x = e_i picks exactly column i of the dequantized matrix."""
    O, I, gs = 2, 8, 4
    # nibbles chosen so every element is a distinct value
    q = np.array([[-8, -7, -6, -5, -4, -3, -2, -1], [0, 1, 2, 3, 4, 5, 6, 7]])
    nib = (q + 8).astype(np.uint8)
    w = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    sc = np.array([[1.0, 10.0], [100.0, 1000.0]], np.float32)
    for i in range(I):
        x = np.zeros(I, np.float32); x[i] = 1.0
        y, _ = orc.qgemv_i4g(x, w, sc, 1, I, O, gs)
        want = [q[0, i] * sc[0, i // gs], q[1, i] * sc[1, i // gs]]
        assert np.array_equal(y[0], want), (i, y[0], want)


def pin_quantizer_invariants(orc):
    """The symmetric quantizer: extremes code to +-7 exactly, zero groups are
    (scale 0, nibble 8), every weight lies within half a step of its code,
    and odd I pads the last high nibble with 8."""
    O, I, gs = 4, 201, 64
    w = synth.normal(5, O * I, 0.02).reshape(O, I)
    w[1, 64:128] = 0.0                       # an all-zero group
    wq, sc = orc.quantize_i4g(w, O, I, gs)
    ng = (I + gs - 1) // gs
    assert wq.shape == (O, (I + 1) // 2) and sc.shape == (O, ng)
    nib = np.stack([wq & 0xF, wq >> 4], -1).reshape(O, -1)
    assert np.all(nib[:, I:] == 8)            # pad nibble
    q = nib[:, :I].astype(np.int64) - 8
    for o in range(O):
        for g in range(ng):
            seg = slice(g * gs, min(I, (g + 1) * gs))
            a = np.abs(w[o, seg])
            if a.max() == 0:
                assert sc[o, g] == 0 and np.all(q[o, seg] == 0)
                continue
            assert sc[o, g] == np.float32(a.max()) / np.float32(7.0)
            k = int(np.argmax(a))
            assert q[o, seg][k] == (7 if w[o, seg][k] > 0 else -7)
            err = np.abs(w[o, seg].astype(np.float64) - q[o, seg] * np.float64(sc[o, g]))
            assert np.all(err <= 0.5 * np.float64(sc[o, g]) * (1 + 1e-6))


# ---------------------------------------------------------------------------
# fmt=7 FP8-e4m3, 128x128 block scales
# ---------------------------------------------------------------------------

def _dequant_fp8_numpy(codes, scales, O, I):
    import torch
    dec = torch.from_numpy(np.asarray(codes, np.uint8).reshape(O, I).copy()).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()
    nbo, nbi = (O + 127) // 128, (I + 127) // 128
    sc = np.kron(np.asarray(scales, np.float32).reshape(nbo, nbi).astype(np.float64),
                 np.ones((128, 128)))[:O, :I]
    return dec * sc


def pin_fp8_golden(orc):
    g = _golden("fp8b128_hand.json")
    for case in g["cases"]:
        O, I = case["O"], case["I"]
        codes = (np.full(O * I, case["fill"], np.uint8) if case["codes"] is None
                 else np.array(case["codes"], np.uint8))
        x = (np.ones(I, np.float32) if case["x"] == "ones" else np.array(case["x"], np.float32))
        y, mag = orc.qgemv_fp8b128(synth.bf16_bits(x), codes, np.array(case["scales"], np.float32),
                                   1, I, O)
        if "y" in case:
            assert np.array_equal(y[0], case["y"]) and np.array_equal(mag[0], case["mag"]), (y, mag)
        for r, v in case.get("y_rows", {}).items():
            assert y[0, int(r)] == v, (case["name"], r, y[0, int(r)], v)


def pin_fp8_bruteforce(orc):
    """Edge shapes, the non-square nblkO=3 x nblkI=48 grid, S=4."""
    rng = np.random.default_rng(21)
    for (O, I, S) in [(1, 1, 1), (130, 200, 2), (129, 128, 1), (128, 129, 1), (384, 6144, 3),
                      (5, 300, 4)]:
        codes = synth.bytes_excluding(int(rng.integers(1 << 30)), O * I)
        nbo, nbi = (O + 127) // 128, (I + 127) // 128
        sc = synth.log_uniform(int(rng.integers(1 << 30)), nbo * nbi, 1e-4, 1e-2)
        xb = synth.bf16_bits(rng.standard_normal(S * I).astype(np.float32))
        y, mag = orc.qgemv_fp8b128(xb, codes, sc, S, I, O)
        W = _dequant_fp8_numpy(codes, sc, O, I)
        X = synth.bf16_to_f32(xb).reshape(S, I).astype(np.float64)
        _close(y, X @ W.T, np.abs(X) @ np.abs(W).T, what=f"fp8 O={O} I={I}")
        _close(mag, np.abs(X) @ np.abs(W).T, np.abs(X) @ np.abs(W).T, what=f"fp8 mag O={O} I={I}")


def pin_e8m0_vs_torch(orc):
    """All 256 UE8M0 bytes against torch.float8_e8m0fnu (an independent
    implementation of the OCP E8M0 type): 2^(e-127), 255 is NaN."""
    import torch
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    got = np.array([orc.e8m0_value(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref)) and np.isnan(got[255]) and np.isnan(got).sum() == 1
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert got[127] == 1.0 and got[0] == 2.0 ** -127 and got[254] == 2.0 ** 127


def pin_fp8ue8m0_golden(orc):
    g = _golden("fp8ue8m0_hand.json")
    for c in g["cases"]:
        O, I = c["O"], c["I"]
        codes = np.full(O * I, c["fill"], np.uint8) if c["codes"] is None else np.array(c["codes"], np.uint8)
        x = np.ones(I, np.float32) if c["x"] == "ones" else np.array(c["x"], np.float32)
        xb = synth.bf16_bits(x)
        if "scale_cases" in c:
            for byte, want in c["scale_cases"]:
                y, _ = orc.qgemv_fp8ue8m0(xb, codes, np.array([byte], np.uint8), 1, I, O)
                assert (np.isnan(y[0, 0]) if want == "nan" else y[0, 0] == want), (byte, y)
            continue
        y, mag = orc.qgemv_fp8ue8m0(xb, codes, np.array(c["scales"], np.uint8), 1, I, O)
        if "y" in c:
            assert np.array_equal(y[0], c["y"]) and np.array_equal(mag[0], c["mag"]), (y, mag)
        for row, want in c.get("y_rows", {}).items():
            assert y[0, int(row)] == want, (row, y[0, int(row)], want)


def pin_fp8ue8m0_bruteforce(orc):
    """Edge shapes and every exponent byte but NaN: oracle == numpy dequantize
    (e4m3 via torch, 2.0 ** (e - 127)) + matmul; and the same codes with the
    equivalent f32 scales give the fmt=7 f32 result exactly."""
    rng = np.random.default_rng(23)
    for (O, I, S) in [(1, 1, 1), (130, 200, 2), (129, 128, 1), (384, 6144, 3), (5, 300, 4)]:
        codes = synth.bytes_excluding(int(rng.integers(1 << 30)), O * I)
        nbo, nbi = (O + 127) // 128, (I + 127) // 128
        eb = rng.integers(100, 150, nbo * nbi).astype(np.uint8)
        xb = synth.bf16_bits(rng.standard_normal(S * I).astype(np.float32))
        y, mag = orc.qgemv_fp8ue8m0(xb, codes, eb, S, I, O)
        f32 = (2.0 ** (eb.astype(np.float64) - 127)).astype(np.float32)
        W = _dequant_fp8_numpy(codes, f32, O, I)
        X = synth.bf16_to_f32(xb).reshape(S, I).astype(np.float64)
        _close(y, X @ W.T, np.abs(X) @ np.abs(W).T, what=f"fp8ue8m0 O={O} I={I}")
        _close(mag, np.abs(X) @ np.abs(W).T, np.abs(X) @ np.abs(W).T, what=f"fp8ue8m0 mag O={O} I={I}")
        y2, _ = orc.qgemv_fp8b128(xb, codes, f32, S, I, O)
        assert np.array_equal(y, y2)


def pin_fp8_nan_rows(orc):
    """A NaN code poisons exactly its own output row."""
    O, I = 130, 130
    codes = synth.bytes_excluding(3, O * I).reshape(O, I)
    codes[7, 100] = 0x7F
    codes[129, 3] = 0xFF
    sc = synth.log_uniform(4, 4, 1e-4, 1e-2)
    xb = synth.bf16_bits(synth.normal(5, I))
    y, _ = orc.qgemv_fp8b128(xb, codes, sc, 1, I, O)
    nan_rows = set(np.nonzero(np.isnan(y[0]))[0].tolist())
    assert nan_rows == {7, 129}, nan_rows


def pin_fp8_dequant_exact_130(orc):
    """Bit-exact decode at every position of a 130x130 partial-block tensor:
    x = e_i returns column i of the dequantized matrix exactly."""
    O = I = 130
    codes = synth.bytes_excluding(8, O * I).reshape(O, I)
    sc = synth.log_uniform(9, 4, 1e-4, 1e-2)
    W = _dequant_fp8_numpy(codes, sc, O, I)
    for i in range(I):
        x = np.zeros(I, np.float32); x[i] = 1.0
        y, _ = orc.qgemv_fp8b128(synth.bf16_bits(x), codes, sc, 1, I, O)
        assert np.array_equal(y[0], W[:, i]), i


# ---------------------------------------------------------------------------
# MQ4-V2
# ---------------------------------------------------------------------------

def _dequant_mq4v2_numpy(blocks, O, I):
    """Dequantize from the byte layout with numpy views (vectorised)."""
    nb = I // 256
    b = np.asarray(blocks, np.uint8).reshape(O, nb, 136)
    hdr = np.ascontiguousarray(b[:, :, 0:8]).view("<u2").reshape(O, nb, 4).view(np.float16)
    scale = hdr[:, :, 0::2].astype(np.float64)      # [O, nb, 2]
    zero = hdr[:, :, 1::2].astype(np.float64)
    pay = b[:, :, 8:136]
    q = np.stack([pay & 0xF, pay >> 4], -1).reshape(O, nb, 256).astype(np.float64)
    h = (np.arange(256) >= 128).astype(np.int64)
    return (q * scale[:, :, h] + zero[:, :, h]).reshape(O, I)


def _dequant_mq4v1_numpy(blocks, O, I):
    """The v1 (qt=1/13) reading: f32 scale at +0 and f32 zero at +4 for all 256."""
    nb = I // 256
    b = np.asarray(blocks, np.uint8).reshape(O, nb, 136)
    hdr = np.ascontiguousarray(b[:, :, 0:8]).view("<f4").reshape(O, nb, 2).astype(np.float64)
    pay = b[:, :, 8:136]
    q = np.stack([pay & 0xF, pay >> 4], -1).reshape(O, nb, 256).astype(np.float64)
    return (q * hdr[:, :, 0:1] + hdr[:, :, 1:2]).reshape(O, I)


def pin_mq4v2_golden(orc):
    g = _golden("mq4v2_hand.json")
    blk = np.array(g["header"] + [g["payload_byte"]] * 128, np.uint8)
    assert blk.size == 136
    for j, v in g["weights"].items():
        assert orc.mq4v2_weight(blk, int(j)) == v, (j, orc.mq4v2_weight(blk, int(j)), v)
    x = synth.bf16_bits(np.ones(256, np.float32))
    y, mag = orc.qgemv_mq4v2(x, blk, 1, 256, 1)
    assert y[0, 0] == g["y_ones"] and mag[0, 0] == g["mag_ones"], (y, mag)


def pin_mq4v2_size_and_bruteforce(orc):
    """136 B per 256 weights; oracle GEMV == numpy dequantize + matmul with
    distinct random headers per half (discriminates the half predicate) over
    several blocks and rows (discriminates stride and payload offset)."""
    rng = np.random.default_rng(31)
    for (O, I, S) in [(1, 256, 1), (3, 512, 2), (4, 1280, 3), (2, 768, 8)]:
        w = synth.normal(int(rng.integers(1 << 30)), O * I, 0.02)
        blocks = orc.encode_mq4v2(w, O, I)
        assert blocks.size == 136 * O * I // 256
        # scramble the headers so each half has its own, clearly distinct pair
        hb = blocks.reshape(O, I // 256, 136)
        hv = (rng.uniform(0.5, 2.0, (O, I // 256, 4)) * [1e-2, 1, 1e-2, -1]).astype(np.float16)
        hb[:, :, 0:8] = hv.view(np.uint8).reshape(O, I // 256, 8)
        xb = synth.bf16_bits(rng.standard_normal(S * I).astype(np.float32))
        y, mag = orc.qgemv_mq4v2(xb, blocks, S, I, O)
        W = _dequant_mq4v2_numpy(blocks, O, I)
        X = synth.bf16_to_f32(xb).reshape(S, I).astype(np.float64)
        _close(y, X @ W.T, np.abs(X) @ np.abs(W).T, what=f"mq4v2 O={O} I={I}")
        _close(mag, np.abs(X) @ np.abs(W).T, np.abs(X) @ np.abs(W).T, what=f"mq4v2 mag O={O} I={I}")


def pin_mq4v2_equal_halves_match_v1(orc):
    """Equal half headers make v2 numerically identical to v1 on the same
    nibbles (hipfire MQ4 V2 section 1e)."""
    rng = np.random.default_rng(32)
    O, I = 3, 768
    nb = I // 256
    pay = rng.integers(0, 256, (O, nb, 128), dtype=np.uint8)
    s16 = rng.uniform(1e-3, 1e-2, (O, nb)).astype(np.float16)
    z16 = rng.uniform(-0.1, 0.0, (O, nb)).astype(np.float16)
    v2 = np.zeros((O, nb, 136), np.uint8)
    v1 = np.zeros((O, nb, 136), np.uint8)
    pair = np.stack([s16, z16], -1).view(np.uint8).reshape(O, nb, 4)
    v2[:, :, 0:4] = pair
    v2[:, :, 4:8] = pair
    v2[:, :, 8:] = pay
    f32 = np.stack([s16.astype(np.float32), z16.astype(np.float32)], -1)
    v1[:, :, 0:8] = f32.view(np.uint8).reshape(O, nb, 8)
    v1[:, :, 8:] = pay
    W1 = _dequant_mq4v1_numpy(v1, O, I)
    for o in range(O):
        for j in range(0, I, 37):
            assert orc.mq4v2_weight(v2[o, j // 256], j % 256) == W1[o, j]
    x = synth.bf16_bits(rng.standard_normal(I).astype(np.float32))
    y, mag = orc.qgemv_mq4v2(x, v2, 1, I, O)
    X = synth.bf16_to_f32(x).astype(np.float64)
    _close(y[0], W1 @ X, np.abs(W1) @ np.abs(X), what="v2 == v1")


def pin_mq4v2_constant_half(orc):
    """A constant half stores scale 0 and decodes to exactly f16(lo)."""
    w = np.full((1, 256), 0.0123, np.float32)
    w[0, 128:] = synth.normal(3, 128, 0.02)
    blk = orc.encode_mq4v2(w, 1, 256)[0]
    want = float(np.float16(np.float32(0.0123)))
    assert blk[0:2].view("<u2")[0] == 0
    for j in range(128):
        assert orc.mq4v2_weight(blk, j) == want


def pin_mq4v2_lattice_roundtrip(orc):
    """Weights on the fp16 lattice z + k*s (k = 0..15 in each half, both ends
    present) round-trip bit-exactly through encode -> decode."""
    rng = np.random.default_rng(33)
    for _ in range(20):
        w = np.zeros(256, np.float32)
        for h in range(2):
            s = float(np.float16(2.0 ** int(rng.integers(-10, -3))))   # power of two: exact steps
            z = float(np.float16(rng.uniform(-0.5, 0.5)))
            k = rng.integers(0, 16, 128)
            k[0], k[1] = 0, 15
            rng.shuffle(k)
            w[128 * h:128 * h + 128] = (z + k * s)
        blk = orc.encode_mq4v2(w.reshape(1, 256), 1, 256)[0]
        dec = np.array([orc.mq4v2_weight(blk, j) for j in range(256)])
        assert np.array_equal(dec, w.astype(np.float64))


def pin_mq4v2_nearest_decoded_level(orc):
    """Each weight is coded to the nearest level of the grid the decoder will
    actually use (the fp16-rounded scale and zero), except where clamped at
    either end: the encoder quantizes against the round-tripped header."""
    O, I = 16, 2048
    w = synth.normal(35, O * I, 0.02).reshape(O, I)
    blocks = orc.encode_mq4v2(w, O, I).reshape(O, I // 256, 136)
    hdr = np.ascontiguousarray(blocks[:, :, 0:8]).view("<u2").view(np.float16).astype(np.float64)
    pay = blocks[:, :, 8:]
    q = np.stack([pay & 0xF, pay >> 4], -1).reshape(O, I // 256, 256).astype(np.float64)
    h = (np.arange(256) >= 128).astype(np.int64)
    st = hdr[:, :, 0::2][:, :, h]
    z = hdr[:, :, 1::2][:, :, h]
    src = w.reshape(O, I // 256, 256).astype(np.float64)
    rec = q * st + z
    err = np.abs(src - rec)
    clamped = ((q == 0) & (src < z)) | ((q == 15) & (src > z + 15 * st))
    bound = 0.5 * st + 2.0 ** -21 * (np.abs(src - z) + st)
    bad = ~clamped & ~(err <= bound)
    assert not bad.any(), f"{bad.sum()} weights not on their nearest decoded level"


def pin_mq4v2_extremes(orc):
    """Min/max fit: the smallest weight of a half codes to 0 and the largest
    to 15; reconstruction of both within the fp16 header rounding bound."""
    O, I = 8, 1024
    w = synth.normal(34, O * I, 0.02).reshape(O, I)
    blocks = orc.encode_mq4v2(w, O, I).reshape(O, I // 256, 136)
    W = _dequant_mq4v2_numpy(blocks, O, I)
    for o in range(O):
        for b in range(I // 256):
            pay = blocks[o, b, 8:]
            q = np.stack([pay & 0xF, pay >> 4], -1).reshape(256)
            for h in range(2):
                seg = slice(256 * b + 128 * h, 256 * b + 128 * h + 128)
                src = w[o, seg].astype(np.float64)
                lo, hi = src.min(), src.max()
                qq = q[128 * h:128 * h + 128]
                assert qq[np.argmin(src)] == 0 and qq[np.argmax(src)] == 15
                step = (hi - lo) / 15
                bound = 2.0 ** -11 * (abs(lo) + 15 * step) + 2.0 ** -24
                rec = W[o, seg]
                assert abs(rec[np.argmin(src)] - lo) <= bound
                assert abs(rec[np.argmax(src)] - hi) <= bound


# ---------------------------------------------------------------------------
# MQ4 v1 (qt=13) and MQ4C pad (qt=45): one header per 256-weight block
# ---------------------------------------------------------------------------

def _dequant_mq4c_numpy(blocks, O, I):
    """The pad reading: fp16 scale at +0, fp16 zero at +2, for all 256."""
    nb = I // 256
    b = np.asarray(blocks, np.uint8).reshape(O, nb, 136)
    hdr = np.ascontiguousarray(b[:, :, 0:4]).view("<u2").view(np.float16).reshape(O, nb, 2)
    hdr = hdr.astype(np.float64)
    pay = b[:, :, 8:136]
    q = np.stack([pay & 0xF, pay >> 4], -1).reshape(O, nb, 256).astype(np.float64)
    return (q * hdr[:, :, 0:1] + hdr[:, :, 1:2]).reshape(O, I)


def _golden_one_header(orc, name, weight_fn, gemv_fn):
    g = _golden(name)
    blk = np.array(g["header"] + [g["payload_byte"]] * 128, np.uint8)
    assert blk.size == 136
    for j, v in g["weights"].items():
        assert weight_fn(blk, int(j)) == v, (name, j, weight_fn(blk, int(j)), v)
    x = synth.bf16_bits(np.ones(256, np.float32))
    y, mag = gemv_fn(x, blk, 1, 256, 1)
    assert y[0, 0] == g["y_ones"] and mag[0, 0] == g["mag_ones"], (name, y, mag)


def pin_mq4v1_golden(orc):
    _golden_one_header(orc, "mq4v1_hand.json", orc.mq4v1_weight, orc.qgemv_mq4v1)


def pin_mq4c_golden(orc):
    _golden_one_header(orc, "mq4c_hand.json", orc.mq4c_weight, orc.qgemv_mq4c)


def pin_mq4_one_header_bruteforce(orc):
    """Oracle GEMVs == numpy dequantize + matmul, with a distinct random header
    per block over several blocks and rows (discriminates stride, header
    position and field order) and a payload whose first bytes differ from the
    pad (a decoder reading the payload at +4 picks up the zero pad)."""
    rng = np.random.default_rng(41)
    for (O, I, S) in [(1, 256, 1), (3, 512, 2), (4, 1280, 3)]:
        nb = I // 256
        pay = rng.integers(0, 256, (O, nb, 128), dtype=np.uint8)
        pay[:, :, 0:4] = 0xFF
        s = rng.uniform(1e-3, 1e-2, (O, nb))
        z = rng.uniform(-0.1, 0.1, (O, nb))
        v1 = np.zeros((O, nb, 136), np.uint8)
        v1[:, :, 0:8] = np.stack([s, z], -1).astype("<f4").view(np.uint8).reshape(O, nb, 8)
        v1[:, :, 8:] = pay
        c = np.zeros((O, nb, 136), np.uint8)
        c[:, :, 0:4] = np.stack([s, z], -1).astype(np.float16).view(np.uint8).reshape(O, nb, 4)
        c[:, :, 8:] = pay
        xb = synth.bf16_bits(rng.standard_normal(S * I).astype(np.float32))
        X = synth.bf16_to_f32(xb).reshape(S, I).astype(np.float64)
        for blocks, fn, ref in ((v1, orc.qgemv_mq4v1, _dequant_mq4v1_numpy),
                                (c, orc.qgemv_mq4c, _dequant_mq4c_numpy)):
            y, mag = fn(xb, blocks, S, I, O)
            W = ref(blocks, O, I)
            _close(y, X @ W.T, np.abs(X) @ np.abs(W).T, what=f"one-header O={O} I={I}")
            _close(mag, np.abs(X) @ np.abs(W).T, np.abs(X) @ np.abs(W).T, what=f"one-header mag O={O} I={I}")


def pin_mq4_three_layouts_agree(orc):
    """The same fp16-representable scale and zero in each layout (v2 with
    equal half headers, v1 as f32, pad as fp16) decode the same nibbles to
    identical weights (hipfire MQ4 V2 section 1e)."""
    rng = np.random.default_rng(42)
    O, I = 2, 512
    nb = I // 256
    pay = rng.integers(0, 256, (O, nb, 128), dtype=np.uint8)
    s16 = rng.uniform(1e-3, 1e-2, (O, nb)).astype(np.float16)
    z16 = rng.uniform(-0.1, 0.1, (O, nb)).astype(np.float16)
    pair = np.stack([s16, z16], -1).view(np.uint8).reshape(O, nb, 4)
    v2 = np.zeros((O, nb, 136), np.uint8)
    v2[:, :, 0:4] = pair
    v2[:, :, 4:8] = pair
    v2[:, :, 8:] = pay
    c = np.zeros((O, nb, 136), np.uint8)
    c[:, :, 0:4] = pair
    c[:, :, 8:] = pay
    v1 = np.zeros((O, nb, 136), np.uint8)
    v1[:, :, 0:8] = np.stack([s16.astype(np.float32), z16.astype(np.float32)], -1).view(np.uint8).reshape(O, nb, 8)
    v1[:, :, 8:] = pay
    for o in range(O):
        for b in range(nb):
            for j in range(256):
                a = orc.mq4v2_weight(v2[o, b], j)
                assert orc.mq4v1_weight(v1[o, b], j) == a and orc.mq4c_weight(c[o, b], j) == a


def _one_header_encoder_checks(orc, encode, decode_np, fp16):
    O, I = 8, 1024
    w = synth.normal(43, O * I, 0.02).reshape(O, I)
    blocks = encode(w, O, I)
    assert blocks.size == 136 * O * I // 256
    b = blocks.reshape(O, I // 256, 136)
    if fp16:
        assert not b[:, :, 4:8].any(), "pad bytes must be zero"
    W = decode_np(blocks, O, I)
    for o in range(O):
        for k in range(I // 256):
            src = w[o, 256 * k:256 * k + 256].astype(np.float64)
            pay = b[o, k, 8:]
            q = np.stack([pay & 0xF, pay >> 4], -1).reshape(256)
            assert q[np.argmin(src)] == 0 and q[np.argmax(src)] == 15
            lo, hi = src.min(), src.max()
            step = (hi - lo) / 15
            hb = (2.0 ** -11 if fp16 else 2.0 ** -23) * (abs(lo) + 15 * step) + 2.0 ** -24
            rec = W[o, 256 * k:256 * k + 256]
            assert abs(rec[np.argmin(src)] - lo) <= hb and abs(rec[np.argmax(src)] - hi) <= hb
            # every weight within half a step (plus header rounding) of its code
            assert np.all(np.abs(rec - src) <= 0.5 * step * (1 + 2.0 ** -9) + hb)
    # a constant block stores scale 0 and decodes to its value (rounded to the header type)
    wc = np.full((1, 256), 0.0123, np.float32)
    bc = encode(wc, 1, 256)[0]
    want = float(np.float16(np.float32(0.0123))) if fp16 else float(np.float32(0.0123))
    assert not bc[8:].any()
    for j in (0, 1, 255):
        assert (orc.mq4c_weight if fp16 else orc.mq4v1_weight)(bc, j) == want


def pin_mq4v1_encoder(orc):
    _one_header_encoder_checks(orc, orc.encode_mq4v1, _dequant_mq4v1_numpy, fp16=False)


def pin_mq4c_encoder(orc):
    _one_header_encoder_checks(orc, orc.encode_mq4c, _dequant_mq4c_numpy, fp16=True)


# ---------------------------------------------------------------------------
# FWHT rotation
# ---------------------------------------------------------------------------

def _dequant_q2_0_numpy(blocks, O, I):
    """numpy decode of Q2_0 rows from the layout description."""
    nb = I // 64
    b = np.asarray(blocks, np.uint8).reshape(O, nb, 18)
    d = b[:, :, 0:2].copy().view(np.float16)[:, :, 0].astype(np.float64)          # [O, nb]
    qs = b[:, :, 2:18].astype(np.int64)                                            # [O, nb, 16]
    codes = np.stack([(qs >> (2 * k)) & 3 for k in range(4)], axis=-1).reshape(O, nb, 64)   # element 4j + k
    return ((codes - 1) * d[:, :, None]).reshape(O, I)


def pin_q2_0_golden(orc):
    g = _golden("q2_0_hand.json")
    for c in g["cases"]:
        I = c["I"]
        blocks = np.zeros(I // 64 * 18, np.uint8)
        if "d_bits" in c:
            blocks[0:2] = np.array([c["d_bits"]], np.uint16).view(np.uint8)
            blocks[2:18] = c["fill"]
            for k, v in c["codes"].items():
                blocks[2 + int(k)] = v
        else:
            blocks[2:18] = 0x55                                   # block 0: weights 0
            blocks[18:20] = np.array([c["block1_d_bits"]], np.uint16).view(np.uint8)
            for k, v in c["block1_codes"].items():
                blocks[18 + 2 + int(k)] = v
        x = np.zeros(I, np.float32)
        for k, v in c["x"].items():
            x[int(k)] = v
        y, mag = orc.qgemv_q2_0(synth.bf16_bits(x), blocks, 1, I, 1)
        assert y[0, 0] == c["y"] and mag[0, 0] == c["mag"], (c["name"], y, mag)


def pin_q2_0_size_and_bruteforce(orc):
    """18 bytes per 64 weights; oracle GEMV == numpy decode + matmul on random
    codes and fp16 d over several blocks and rows."""
    rng = np.random.default_rng(61)
    for (O, I, S) in [(1, 64, 1), (3, 128, 2), (4, 640, 3), (2, 2560, 8)]:
        w = synth.normal(int(rng.integers(1 << 30)), O * I, 0.02)
        blocks = orc.encode_q2_0(w, O, I)
        assert blocks.size == 18 * O * I // 64
        b = blocks.reshape(O, I // 64, 18)
        b[:, :, 2:] = rng.integers(0, 256, (O, I // 64, 16), dtype=np.uint8)
        b[:, :, 0:2] = rng.uniform(1e-3, 1e-1, (O, I // 64, 1)).astype(np.float16).view(np.uint8)
        xb = synth.bf16_bits(rng.standard_normal(S * I).astype(np.float32))
        y, mag = orc.qgemv_q2_0(xb, blocks, S, I, O)
        W = _dequant_q2_0_numpy(blocks, O, I)
        X = synth.bf16_to_f32(xb).reshape(S, I).astype(np.float64)
        _close(y, X @ W.T, np.abs(X) @ np.abs(W).T, what=f"q2_0 O={O} I={I}")
        _close(mag, np.abs(X) @ np.abs(W).T, np.abs(X) @ np.abs(W).T, what=f"q2_0 mag O={O} I={I}")


def pin_q2_0_encoder(orc):
    """Codes on the grid; a block whose weights are (c - 1) * d with an
    fp16-exact d and at least one code 3 round-trips bit-exactly (amax = 2d is
    the first candidate, SSE 0); an all-zero block stores d = 0, codes 1; the
    stored codes give the smallest SSE of the nine candidates (recomputed here
    with numpy)."""
    rng = np.random.default_rng(62)
    O, I = 3, 192
    d = np.array([0.25, 0.0625, 1.5], np.float16).astype(np.float32)
    codes = rng.integers(0, 4, (O, I)).astype(np.int64)
    codes[:, ::64] = 3
    w = ((codes - 1) * d[:, None]).astype(np.float32)
    blocks = orc.encode_q2_0(w, O, I)
    assert np.array_equal(_dequant_q2_0_numpy(blocks, O, I), w.astype(np.float64))
    z = orc.encode_q2_0(np.zeros((1, 64), np.float32), 1, 64)
    assert z[0, 0] == 0 and z[0, 1] == 0 and (z[0, 2:] == 0x55).all()
    w = synth.normal(63, 8 * 256, 0.02).reshape(8, 256)
    blocks = orc.encode_q2_0(w, 8, 256)
    W = _dequant_q2_0_numpy(blocks, 8, 256)
    vb = w.reshape(8, 4, 64).astype(np.float32)
    for o in range(8):
        for b in range(4):
            v = vb[o, b]
            amax = np.float32(np.abs(v).max())
            sses = []
            for k in range(9):
                dk = np.float32(amax * np.float32(np.float32(0.5) + np.float32(k) / np.float32(16)))
                c = np.clip(np.rint(v / dk) + 1, 0, 3)
                sses.append(float(((v.astype(np.float64) - (c - 1) * np.float64(dk)) ** 2).sum()))
            best = int(np.argmin(sses))
            dk = np.float32(amax * np.float32(np.float32(0.5) + np.float32(best) / np.float32(16)))
            want_codes = np.clip(np.rint(v / dk) + 1, 0, 3).astype(np.int64)
            got = blocks.reshape(8, 4, 18)[o, b]
            got_codes = np.stack([(got[2:].astype(np.int64) >> (2 * k)) & 3 for k in range(4)], -1).reshape(64)
            assert np.array_equal(got_codes, want_codes), (o, b)
            assert got[0:2].copy().view(np.float16)[0] == np.float16(dk)


def _moe_experts(rng, fmt, n_experts, O, I, gs):
    """Random experts of one format: (weights, scales, numpy dequantizer)."""
    ws, ss, deq = [], [], []
    for _ in range(n_experts):
        if fmt == 4:
            rb, ng = (I + 1) // 2, (I + gs - 1) // gs
            w = rng.integers(0, 256, O * rb, dtype=np.uint8)
            sc = rng.uniform(-2, 2, O * ng).astype(np.float32)
            deq.append(_dequant_i4g_numpy(w, sc, O, I, gs))
        elif fmt in (7, 71):
            w = synth.bytes_excluding(int(rng.integers(1 << 30)), O * I)
            nbo, nbi = (O + 127) // 128, (I + 127) // 128
            if fmt == 7:
                sc = synth.log_uniform(int(rng.integers(1 << 30)), nbo * nbi, 1e-4, 1e-2)
                deq.append(_dequant_fp8_numpy(w, sc, O, I))
            else:
                sc = rng.integers(110, 125, nbo * nbi).astype(np.uint8)
                deq.append(_dequant_fp8_numpy(w, (2.0 ** (sc.astype(np.float64) - 127)).astype(np.float32), O, I))
        else:
            nb = I // 256
            w = rng.integers(0, 256, (O, nb, 136), dtype=np.uint8)
            hs = rng.uniform(1e-3, 1e-2, (O, nb, 2))
            hz = rng.uniform(-0.1, 0.1, (O, nb, 2))
            if fmt == 44:
                w[:, :, 0:8] = np.stack([hs[..., 0], hz[..., 0], hs[..., 1], hz[..., 1]], -1).astype(
                    np.float16).view(np.uint8).reshape(O, nb, 8)
                deq.append(_dequant_mq4v2_numpy(w, O, I))
            elif fmt == 13:
                w[:, :, 0:8] = np.stack([hs[..., 0], hz[..., 0]], -1).astype("<f4").view(np.uint8).reshape(O, nb, 8)
                deq.append(_dequant_mq4v1_numpy(w, O, I))
            else:
                w[:, :, 0:4] = np.stack([hs[..., 0], hz[..., 0]], -1).astype(np.float16).view(np.uint8).reshape(
                    O, nb, 4)
                w[:, :, 4:8] = 0
                deq.append(_dequant_mq4c_numpy(w, O, I))
            sc = None
        ws.append(w)
        ss.append(sc)
    return ws, ss, deq


def pin_moe_bruteforce(orc):
    """Routed experts == numpy dequantize + matmul slot by slot, every format,
    with repeated ids, ids out of order, a shared x and one x per slot; a slot
    whose id names no expert is NaN."""
    rng = np.random.default_rng(51)
    for fmt, (O, I, gs) in ((4, (3, 200, 64)), (7, (130, 260, 0)), (71, (130, 260, 0)), (44, (3, 512, 0)),
                            (13, (2, 768, 0)), (45, (2, 512, 0))):
        E = 4
        ws, ss, deq = _moe_experts(rng, fmt, E, O, I, gs)
        ids = np.array([2, 0, 2, 3, 1], np.int32)
        S = 2
        for shared in (True, False):
            n_x = 1 if shared else len(ids)
            xf = rng.standard_normal(n_x * S * I).astype(np.float32)
            xin = xf if fmt == 4 else synth.bf16_bits(xf)
            X = (xf if fmt == 4 else synth.bf16_to_f32(xin)).reshape(n_x, S, I).astype(np.float64)
            y, mag = orc.qgemv_moe(fmt, xin, 0 if shared else S * I, ws, ss, ids, S, I, O, gs)
            assert y.shape == (len(ids), S, O)
            for r, e in enumerate(ids):
                Xr = X[0 if shared else r]
                _close(y[r], Xr @ deq[e].T, np.abs(Xr) @ np.abs(deq[e]).T, what=f"moe fmt={fmt} slot {r}")
                _close(mag[r], np.abs(Xr) @ np.abs(deq[e]).T, np.abs(Xr) @ np.abs(deq[e]).T, what="moe mag")
        bad = np.array([1, -1, E], np.int32)
        y, mag = orc.qgemv_moe(fmt, xin, 0, ws, ss, bad, S, I, O, gs)
        assert not np.isnan(y[0]).any() and np.isnan(y[1]).all() and np.isnan(y[2]).all()


def pin_moe_permutation(orc):
    """Permuting the slots (ids with their x rows) permutes the outputs."""
    rng = np.random.default_rng(52)
    O, I, gs, S = 4, 128, 32, 1
    ws, ss, _ = _moe_experts(rng, 4, 5, O, I, gs)
    ids = np.array([4, 1, 0, 3], np.int32)
    x = rng.standard_normal((4, S, I)).astype(np.float32)
    y, _ = orc.qgemv_moe(4, x, S * I, ws, ss, ids, S, I, O, gs)
    perm = np.array([2, 0, 3, 1])
    yp, _ = orc.qgemv_moe(4, x[perm], S * I, ws, ss, ids[perm], S, I, O, gs)
    assert np.array_equal(yp, y[perm])


def pin_moe_gemm_bruteforce(orc):
    """Routed-expert prefill == numpy dequantize + matmul group by group, every
    format, with an empty group, a repeated expert and groups out of expert
    order; rows of the token-sorted X map to the same rows of Y."""
    rng = np.random.default_rng(53)
    for fmt, (O, I, gs) in ((4, (3, 200, 64)), (7, (130, 260, 0)), (71, (130, 260, 0)), (44, (3, 512, 0)),
                            (13, (2, 768, 0)), (45, (2, 512, 0))):
        ws, ss, deq = _moe_experts(rng, fmt, 4, O, I, gs)
        ge = np.array([2, 0, 3, 2], np.int32)
        off = np.array([0, 3, 3, 8, 9], np.int32)          # group 1 is empty
        M = int(off[-1])
        xf = rng.standard_normal(M * I).astype(np.float32)
        xb = synth.bf16_bits(xf)
        X = synth.bf16_to_f32(xb).reshape(M, I).astype(np.float64)
        Y, mag = orc.qgemm_moe(fmt, xb, ws, ss, ge, off, I, O, gs)
        for g, e in enumerate(ge):
            r = slice(off[g], off[g + 1])
            _close(Y[r], X[r] @ deq[e].T, np.abs(X[r]) @ np.abs(deq[e]).T, what=f"moe gemm fmt={fmt} group {g}")
            _close(mag[r], np.abs(X[r]) @ np.abs(deq[e]).T, np.abs(X[r]) @ np.abs(deq[e]).T,
                   what=f"moe gemm mag fmt={fmt} group {g}")
        assert not np.isnan(Y).any()


def pin_fwht_vs_scipy(orc):
    from scipy.linalg import hadamard
    H = hadamard(256).astype(np.float64)
    d = synth.signs(42, 256)
    # the transform of the basis vectors is the matrix H diag(d) / 16
    basis = np.eye(256, dtype=np.float32)
    M = orc.fwht256(basis, d).reshape(256, 256).T.astype(np.float64)
    assert np.array_equal(M, H * d[None, :] / 16.0)
    assert np.allclose(M @ M.T, np.eye(256), atol=1e-15)


def pin_fwht_inverse_and_dot(orc):
    d = synth.signs(42, 256)
    v = synth.normal(6, 256 * 8)
    u = synth.normal(7, 256 * 8)
    rv = orc.fwht256(v, d)
    back = orc.ifwht256(rv, d)
    assert np.max(np.abs(back - v)) <= 4e-7 * np.max(np.abs(v))
    ru = orc.fwht256(u, d)
    for b in range(8):
        sl = slice(256 * b, 256 * b + 256)
        a = float(np.dot(u[sl].astype(np.float64), v[sl].astype(np.float64)))
        r = float(np.dot(ru[sl].astype(np.float64), rv[sl].astype(np.float64)))
        assert abs(a - r) <= 1e-5 * float(np.linalg.norm(u[sl]) * np.linalg.norm(v[sl]))


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]

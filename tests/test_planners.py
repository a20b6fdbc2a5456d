"""The launch plans of the staged and warp-MMA decode GEMVs (O x I x S: 15 x
22 x 8, every format, up to 2^24 rows and 2^22 columns) and of the
tensor-core prefill GEMM (M x I x O: 11 x 22 x 15, and 200 routed-expert
calls of seeded group sizes), checked on the CPU.

tests/planner_dump.cu calls the library's own planners (host code, linked
against libqgemv.so; without a GPU they plan for 152 SMs) and prints every
plan they return.  Each plan's shared-memory layout must fit the per-block
limit and the share of an SM its block count was sized for, keep every
region 16-byte aligned for the bulk copies and 8-byte aligned for the
mbarriers, keep its regions apart (ring slots, side data, partial sums,
barriers; the activations inside the last ring slots), cover every row and
every column of the matrix once, respect the kernels' static limits, and,
where it splits rows over blocks, get at least its workspace from
qg_workspace_bytes.  A
prefill plan's tiles must cover the output, its blocks split the (tile, K
step) units without going past the SMs, and its workspace regions (tile
counters, partial slots when a tile's K range is shared, token scales,
weight-row exponents, the fp16 copy of X) must be 256-byte aligned, in order
and large enough."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "weight_only_quantized_i4g_gb300")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

SMEM_BLOCK = 232448        # the kernels' dynamic shared-memory limit (227 KB)
SMEM_SM = 233472           # shared memory of an SM (228 KB), 1 KB of it per block reserved


def cdiv(a, b):
    return -(-a // b)


def next_pow2(n):
    p = 1
    while p < n:
        p *= 2
    return p


@pytest.fixture(scope="module")
def plans(tmp_path_factory):
    lib = os.path.join(PKG, "libqgemv.so")
    if not os.path.exists(lib):
        pytest.fail("libqgemv.so is not built")
    if not (os.path.exists(NVCC) or shutil.which("nvcc")):
        pytest.skip("nvcc not available")
    d = tmp_path_factory.mktemp("planner")
    exe = str(d / "planner_dump")
    cmd = [NVCC, "-std=c++17", "--expt-relaxed-constexpr", "-gencode", "arch=compute_103a,code=sm_103a",
           "-I", os.path.join(PKG, "csrc"), "-I", os.path.join(ROOT, "include"), "-o", exe,
           os.path.join(ROOT, "tests", "planner_dump.cu"), "-L", PKG, "-l:libqgemv.so",
           "-Xlinker", "-rpath," + PKG]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    rows = [ln.split(",") for ln in r.stdout.splitlines() if ln]
    assert len(rows) > 1000
    return rows


# per format: bytes of a staged row, side-data bytes per row, bytes per
# activation, the warp-MMA kernel's consumer-warp limit and partial-sum stride
ROW = {"i4g": lambda I: I // 2, "mq4": lambda I: (I // 256) * 136, "fp8": lambda I: I}
SIDE = {"i4g": lambda I: cdiv(I, 64) * 4, "mq4": lambda I: 0, "fp8": lambda I: 0}
XELEM = {"i4g": 4, "mq4": 2}
MMA_WARPS = {"i4g": 14, "mq4": 15}
RED_STRIDE = {"i4g": 4, "mq4": 8}


def test_mma_plans(plans):
    n = 0
    for r in plans:
        if r[0] != "mma":
            continue
        fmt = r[1]
        S, I, O, nc, splits, per_sm, nsp, sps, nrowb, nst, x_slots = map(int, r[2:13])
        pitch, stage_w, stage_a, red_off, bar_off, x_stride, total = map(int, r[13:20])
        what = f"mma {fmt} S={S} I={I} O={O}: {r[4:]}"
        n += 1
        # coverage: 16-row batches, 64-weight spans, segments of whole 8-span granules
        assert nrowb == cdiv(O, 16), what
        assert nsp == I // 64 and sps * splits >= nsp and sps * (splits - 1) < nsp, what
        assert splits == 1 or sps % 8 == 0, what
        assert 1 <= nc <= MMA_WARPS[fmt] and nc * 8 >= sps, what
        # ring: at least one slot beside the activations, which fit their slots
        assert nst >= 2 and 1 <= x_slots < nst, what
        assert S * x_stride <= x_slots * stage_w, what
        assert x_stride % 16 == 0 and x_stride >= sps * 64 * XELEM[fmt], what
        # four groups of four rows per slot, 32 mod 128 bytes apart, each group holding four row segments
        seg_lo = ROW[fmt](I) if splits == 1 else cdiv(ROW[fmt](I), splits)
        assert pitch % 128 == 32 and stage_w == 4 * pitch and pitch >= 4 * seg_lo, what
        assert stage_a % 128 == 0 and stage_a >= 16 * SIDE[fmt](I), what
        # regions in order, aligned, within the limits
        red = nc * 16 * RED_STRIDE[fmt] * 4
        assert red_off == nst * (stage_w + stage_a), what
        assert bar_off == red_off + 2 * nst * red and bar_off % 16 == 0, what
        assert total == bar_off + 16 * nst + 16, what
        assert total <= SMEM_BLOCK and per_sm >= 1 and total <= SMEM_SM // per_sm - 1024, what
        # a split writes its segments' sums to the caller's workspace: the size query covers it
        if splits > 1:
            assert int(r[20]) >= splits * S * O * 4, what
    assert n > 500


def test_tma_plans(plans):
    n = 0
    for r in plans:
        if r[0] != "tma":
            continue
        fmt = r[1]
        S, I, O, rb, units, U, nc, splits, ups, nrowb, nst, per_sm = map(int, r[2:14])
        stage_w, stage_a, red_off, bar_off, total = map(int, r[14:19])
        what = f"tma {fmt} S={S} I={I} O={O}: {r[4:]}"
        n += 1
        # batches the kernel compiles (RB * S <= 32 partial sums per batch)
        assert rb in (2, 4, 8) and rb * S <= 32, what
        assert nrowb == cdiv(O, rb), what
        # every unit of a row has a thread: column segments cover the row once
        assert ups * splits >= units and ups * (splits - 1) < units, what
        assert 1 <= U <= 3 and 1 <= nc <= 17 and nc * 32 * U >= ups, what
        # ring of 2..6 slots, regions in order and aligned
        row = ROW[fmt](I)
        seg_lo = row if splits == 1 else cdiv(row, splits)
        assert 2 <= nst <= 6, what
        assert stage_w % 128 == 0 and stage_w >= rb * seg_lo, what
        assert stage_a % 128 == 0 and stage_a >= rb * SIDE[fmt](I), what
        assert red_off == nst * (stage_w + stage_a), what
        assert bar_off >= red_off + nst * nc * next_pow2(rb * S) * 4 and bar_off % 16 == 0, what
        assert total == bar_off + 16 * nst, what
        assert total <= SMEM_BLOCK and per_sm >= 1 and total <= SMEM_SM // per_sm - 1024, what
        # a split writes its segments' sums to the caller's workspace: the size query covers it
        if splits > 1:
            assert int(r[19]) >= splits * S * O * 4, what
    assert n > 2000


def test_decode_shapes_are_planned(plans):
    """The decode workloads' shapes get a plan on the paths they run."""
    have = {(r[0], r[1], int(r[2]), int(r[3]), int(r[4])) for r in plans if r[0] in ("mma", "tma")}
    for key in [("tma", "i4g", 1, 7168, 2048), ("tma", "i4g", 1, 2048, 7168), ("tma", "fp8", 1, 16384, 7168),
                ("tma", "fp8", 1, 7168, 24576), ("tma", "mq4", 1, 17408, 5120), ("mma", "mq4", 1, 5120, 17408),
                ("mma", "mq4", 8, 5120, 17408), ("mma", "mq4", 8, 17408, 5120), ("mma", "i4g", 4, 2048, 7168),
                ("mma", "i4g", 4, 7168, 2048)]:
        assert key in have, key


GEMM_BT = (256, 128, 64)


def check_gemm(r, grouped, tiles=None):
    M, I, O, n, tile, bt, MB, NB, Kt, P = map(int, r[1:11])
    T, U, counter, xscale, wexp, xh, ws = map(int, r[11:18])
    what = f"{r[0]} M={M} I={I} O={O} groups={n}: {r[5:]}"
    assert bt == GEMM_BT[tile], what
    assert NB == cdiv(O, 128) and Kt == cdiv(I, 128), what
    if grouped:
        assert T == tiles, what                      # every group's token blocks times the output tiles
    else:
        assert MB == cdiv(M, bt) and T == MB * NB, what
    assert U == T * Kt and 1 <= P <= min(U, 152), what
    split = not (U % P == 0 and (U // P) % Kt == 0)
    for off in (counter, xscale, wexp, xh, ws):
        assert off % 256 == 0, what
    assert counter >= 4 * T, what
    assert xscale >= counter + (2 * P * 128 * bt * 4 if split else 0), what
    assert wexp - xscale >= (cdiv(M, 256) + (1 if grouped else 0)) * 256 * 4, what
    assert xh - wexp >= (n if grouped else 1) * O * 4, what
    assert ws - xh >= M * I * 2, what


def test_gemm_plans(plans):
    n = 0
    for r in plans:
        if r[0] == "gemm":
            check_gemm(r, False)
            n += 1
    assert n > 2000


def test_grouped_gemm_plans(plans):
    n = 0
    for r, nxt in zip(plans, plans[1:]):
        if r[0] == "ggemm":
            assert nxt[0] == "gtiles"
            check_gemm(r, True, int(nxt[1]))
            n += 1
    assert n == 200

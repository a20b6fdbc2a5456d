// planner_dump.cu -- prints the launch plans the decode GEMVs and the
// tensor-core prefill GEMM would choose for a sweep of shapes and token
// counts: host code only, linked against libqgemv.so, no GPU needed (the
// planners assume 152 SMs without a device).  One CSV line per plan;
// tests/test_planners.py checks each plan's layout.
#include <cstdio>
#include <vector>

#include "gemv_fp8.cuh"
#include "gemv_mma.cuh"
#include "gemv_mq4.cuh"
#include "gemv_tma.cuh"
#include "gemm_tc.cuh"
#include "../../include/qgemv.h"

namespace qg {
bool plan_i4g_mma(int S, int I, int O, int gs, MmaPlan *pl);   // gemv_i4g.cu
bool plan_i4g_tma(int S, int I, int O, int gs, TmaPlan *pl);
}  // namespace qg

using namespace qg;

// the workspace the C ABI asks callers for at this shape (last field)
static size_t ws_query(const char *fmt, int S, int I, int O) {
    const int id = fmt[0] == 'i' ? QG_FMT_I4G : fmt[0] == 'm' ? QG_FMT_MQ4V2 : QG_FMT_FP8B128;
    return qg_workspace_bytes(id, S, I, O, 64);
}

static void dump_mma(const char *fmt, int S, int I, int O, const MmaPlan &p) {
    printf("mma,%s,%d,%d,%d,%d,%d,%d,%d,%d,%d,%d,%d,%u,%u,%u,%u,%u,%u,%u,%zu\n", fmt, S, I, O, p.nc, p.splits,
           p.per_sm, p.G.nsp, p.G.sps, p.G.nrowb, p.G.nst, p.G.x_slots, p.L.group_pitch, p.L.stage_w, p.L.stage_a,
           p.L.red_off, p.L.bar_off, p.L.x_stride, p.L.total, ws_query(fmt, S, I, O));
}

static void dump_tma(const char *fmt, int S, int I, int O, const TmaPlan &p) {
    printf("tma,%s,%d,%d,%d,%d,%d,%d,%d,%d,%d,%d,%d,%d,%u,%u,%u,%u,%u,%zu\n", fmt, S, I, O, p.rb, p.units, p.U, p.nc,
           p.splits, p.units_per_split, p.nrowb, p.nst, p.per_sm, p.L.stage_w, p.L.stage_a, p.L.red_off, p.L.bar_off,
           p.L.total, ws_query(fmt, S, I, O));
}

static void dump_gemm(const char *kind, int M, int I, int O, int n, const tc::Plan &p) {
    printf("%s,%d,%d,%d,%d,%d,%d,%d,%d,%d,%d,%lld,%lld,%zu,%zu,%zu,%zu,%zu\n", kind, M, I, O, n, p.tile, p.bt, p.MB,
           p.NB, p.Kt, p.P, p.T, p.U, p.counter_bytes, p.xscale_off, p.wexp_off, p.xh_off, p.ws_bytes);
}

// SplitMix64 (for the seeded group sizes)
static unsigned long long mix(unsigned long long &s) {
    unsigned long long z = (s += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

int main() {
    const int Is[] = {256, 512, 768, 1024, 1280, 2048, 2560, 4096, 5120, 6144, 7168, 8192, 9216,
                      12288, 16384, 17408, 24576, 32768, 61440, 65536, 1 << 20, 1 << 22};
    const int Os[] = {1, 7, 16, 33, 100, 640, 1000, 2048, 2560, 5120, 7168, 17408, 24576, 1 << 20, 1 << 24};
    for (int S = 1; S <= 8; ++S)
        for (int I : Is)
            for (int O : Os) {
                MmaPlan mp;
                TmaPlan tp;
                if (mq4::mq4_mma_plan(S, I, O, &mp)) dump_mma("mq4", S, I, O, mp);
                if (mq4::mq4_tma_plan(S, I, O, &tp)) dump_tma("mq4", S, I, O, tp);
                if (S <= 4 && plan_i4g_mma(S, I, O, 64, &mp)) dump_mma("i4g", S, I, O, mp);
                if (plan_i4g_tma(S, I, O, 64, &tp)) dump_tma("i4g", S, I, O, tp);
                if (fp8_tma_plan(S, I, O, &tp)) dump_tma("fp8", S, I, O, tp);
            }
    // prefill GEMM: one matrix, and routed-expert groups of seeded sizes
    const int Ms[] = {1, 7, 64, 100, 128, 200, 256, 512, 1000, 2048, 4096};
    for (int M : Ms)
        for (int I : Is)
            for (int O : Os) dump_gemm("gemm", M, I, O, 0, tc::choose_plan(M, I, O));
    unsigned long long seed = 7;
    for (int trial = 0; trial < 200; ++trial) {
        const int n = 1 + (int)(mix(seed) % 64);
        std::vector<int> rows(n);
        int M = 0;
        for (int g = 0; g < n; ++g) {
            rows[g] = 1 + (int)(mix(seed) % 300);
            M += rows[g];
        }
        const int I = Is[mix(seed) % (sizeof(Is) / sizeof(Is[0]))];
        const int O = Os[mix(seed) % (sizeof(Os) / sizeof(Os[0]))];
        const tc::Plan p = tc::group_plan(rows.data(), n, M, I, O);
        long long tiles = 0;
        for (int g = 0; g < n; ++g) tiles += (long long)((rows[g] + p.bt - 1) / p.bt) * p.NB;
        dump_gemm("ggemm", M, I, O, n, p);
        printf("gtiles,%lld\n", tiles);
    }
    return 0;
}

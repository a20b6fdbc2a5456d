// gemv_mma.cuh -- decode GEMV of the 4-bit formats on the warp-level MMA
// (mma.sync.m16n8k16, fp16 operands, f32 accumulators).
//
// At 4 bits per weight an SM has to retire about 33 weights per clock to
// keep up with HBM.  Decoding and multiplying each weight on the CUDA cores
// costs several issued instructions per weight, which leaves those kernels
// bound by instruction issue well below the copy rate.  Here the nibbles
// become fp16 operands with one logic op per two weights and one MMA forms
// 2048 products per warp instruction; the N = 8 columns of the MMA carry the
// tokens (up to 8 bf16 activation rows, or 4 f32 rows split into an fp16
// high and low part), so a batch of tokens costs the same per weight as one.
//
// Operands.  A word w of eight nibbles n0..n7 (bits 4k, element c+k) gives
//   P0 = w & 0x000F000F          fp16 pair (n0, n4) * 2^-24
//   P1 = w & 0x00F000F0          fp16 pair (n1, n5) * 2^-20
//   P2 = (w >> 8) & 0x000F000F   fp16 pair (n2, n6) * 2^-24
//   P3 = (w >> 8) & 0x00F000F0   fp16 pair (n3, n7) * 2^-20
// (the bit patterns n and 16 n read as fp16 are the subnormals n 2^-24 and
// n 2^-20, exactly).  The activations are held as fp16 B fragments in the
// same element order, scaled by 2^(14 - F) at the 2^-24 positions and by
// 2^(10 - F) at the 2^-20 ones, F = the exponent of the largest finite |x|
// of that token in the warp's slice, so every product is n x 2^(-10 - F)
// exactly and every scaled activation stays below 2^15.
//
// Fragment layout (m16n8k16, lane = 4 g + t): A registers {A[g][2t..2t+1],
// A[g+8][2t..2t+1], A[g][2t+8..2t+9], A[g+8][2t+8..2t+9]}, B registers
// {B[2t..2t+1][g], B[2t+8..2t+9][g]}, D {D[g][2t..2t+1], D[g+8][2t..2t+1]}.
// Lane (g, t) loads the two words of rows g and g+8 at the span's byte
// 8 t (a span = 64 consecutive weights of a row, 32 bytes); the MMA of word
// j and half h takes (P(2h), P(2h), P(2h+1), P(2h+1)) of rows (g, g+8, g,
// g+8), so its 16 k indices are the span's elements 16 t + 8 j + 2 h +
// {0, 4, 1, 5} over t.  The B fragment of lane (g, t) holds column g's
// activations at exactly those elements.  The order inside the MMA's sum is
// arbitrary; only the pairing of A and B matters.
//
// Per scale unit (fmt=4: one span, inside one group; MQ4: two spans, one
// half-block with its own scale and zero) the D fragment is the unit's
// sum(q x) for rows g, g+8 and the lane's two columns:
//   fmt=4  D starts at -8 sum(x) (C operand), so D = sum((n - 8) x) and
//          acc += scale * D
//   MQ4    acc += scale * D + zero * sum(x)
// sum(x) per unit and column comes from the same MMA with A = the constant
// pattern (2^-24, 2^-20), i.e. from the very fp16 values the products use.
//
// Block = 1 producer warp + NC consumer warps.  Consumer warp w owns the
// spans [w NS, w NS + NS) of the block's column segment, with their B
// fragments in registers for the whole kernel.  The producer streams batches
// of RB rows (whole rows, or the segment of a column split) into a ring of
// shared-memory slots with one 1-D bulk copy per row; rows sit at a stride
// of 32 modulo 128 bytes so the 8-byte loads of a half-warp (rows g..g+3)
// hit distinct banks.  Per batch each consumer warp leaves per-(row,
// column) partial sums of its spans in shared memory and the producer adds
// the NC partials of each output.  Every wait is bounded.
#pragma once

#include "common.cuh"
#include "gemv_tma.cuh"
#include "launch.h"
#include "pipeline.cuh"

namespace qg {

// D += A B, m16n8k16, fp16 inputs, f32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (lo, hi) -> fp16 pair, round to nearest even; lo in the low half.
__device__ __forceinline__ uint32_t f16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// fp16 pair -> the two values in f32 (exact)
__device__ __forceinline__ float2 f16x2_to_f32(uint32_t v) {
    float a, b;
    asm("{.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;}"
        : "=f"(a), "=f"(b)
        : "r"(v));
    return make_float2(a, b);
}

// f32 -> nearest fp16 -> f32
__device__ __forceinline__ float f16_round(float v) {
    float r;
    asm("{.reg .f16 h;\n\tcvt.rn.f16.f32 h, %1;\n\tcvt.f32.f16 %0, h;}" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ uint2 lds_u32x2(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}

// 2^k for k in [-252, 252] as two f32 factors (each a normal power of two).
struct Pow2Split { float a, b; };
__device__ __forceinline__ Pow2Split pow2_split(int k) { return Pow2Split{pow2i(k >> 1), pow2i(k - (k >> 1))}; }

// ---------------------------------------------------------------------------
// Formats.  A format F supplies:
//   kHiLo           true: column n carries token n/2, part n%2 (fp16 high /
//                   low half of an f32 activation); false: column n = token n
//   kSpansPerUnit   spans (64 weights) per scale unit
//   Params          as the staged kernels' (x, weights, scales, I, O, ...)
//   row_bytes, aux_row_bytes, w_src, a_src
//   span_byte(sp)           byte offset of span sp in a row (sp a split boundary)
//   span_off(sp_local)      byte offset of span sp_local in a staged segment
//   kXWords, x_src(p, tok, col), abs_max8(w), pair(w, i)
//                   eight activations are kXWords 32-bit words; where row
//                   tok's activations from column col start; the largest |x|
//                   of eight (as f32); elements (2i, 2i+1) as an f32 pair
//   side_off(sp_abs0, sp_local0, u) where unit u of a warp sits (sp_abs0 and
//                   sp_local0: the warp's first span in the row and in the
//                   staged segment, both multiples of 8)
//   Side, side(row_w, row_a, off)   side data of (row, unit)
//   kNeg8           D starts at -8 sum(x) (fmt=4's offset nibbles)
//   kMaxConsumerWarps  consumer warps of a block (the register budget)
//   kRedStride      floats per (warp, batch row) of the partial sums: the
//                   most tokens one launch carries (4 with kHiLo, else 8)
//   kFenceUnits     keep each unit's shared loads after the previous unit
//                   (register pressure)
//   apply(acc, d, s0, s1, X)        fold a unit's D into the accumulators
// ---------------------------------------------------------------------------

struct MmaLayout {
    uint32_t group_pitch;  // bytes between the staged groups of four rows (32 mod 128)
    uint32_t stage_w;      // bytes per ring slot, weights
    uint32_t stage_a;      // bytes per ring slot, side data
    uint32_t red_off;      // partial sums: [pass parity][slot][warp][RB][F::kRedStride] floats
    uint32_t bar_off;      // full[nst], empty[nst], x_full, x_free
    uint32_t x_stride;     // bytes between the staged activation rows
    uint32_t total;
};

struct MmaGrid {
    int nsp;               // spans per row
    int sps;               // spans per column split
    int nrowb;             // row batches
    int nst;               // ring slots
    int x_slots;           // trailing slots that hold the activations first
    int S;                 // tokens (<= 8, or <= 4 with kHiLo)
};

template <int XW>
__device__ __forceinline__ void lds_xwords(uint32_t a, uint32_t (&w)[XW]) {
    static_assert(XW == 4 || XW == 8, "eight bf16 or eight f32 activations");
#pragma unroll
    for (int v = 0; v < XW / 4; ++v)
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(w[4 * v]), "=r"(w[4 * v + 1]), "=r"(w[4 * v + 2]), "=r"(w[4 * v + 3])
                     : "r"(a + 16u * v));
}

// Rows of a batch in shared memory: four groups of four consecutive rows
// (one bulk copy each), groups `pitch` bytes apart (32 mod 128), rows of a
// group seg bytes apart.  MMA row m (lane group g = m % 8 of rows g, g + 8)
// takes batch row 4 (m % 4) + m / 4: the rows a half-warp loads at once (g
// = 0..3 or 4..7) lie in the four different groups, so their 8-byte loads at
// one offset fall in distinct banks whatever the row length.
__host__ __device__ __forceinline__ int batch_row(int m) { return 4 * (m & 3) + ((m >> 2) & 3); }
__host__ __device__ __forceinline__ uint32_t staged_row_off(int r, uint32_t pitch, uint32_t seg) {
    return (uint32_t)(r >> 2) * pitch + (uint32_t)(r & 3) * seg;
}

// NS spans per consumer warp, RB = 16 rows per batch.
template <class F, int NS, int RB>
__device__ __forceinline__ void gemv_mma_body(const typename F::Params &p, float *__restrict__ out, const MmaGrid &G,
                                              const MmaLayout &L, int *err) {
    static_assert(RB == 16, "one MMA row tile per batch");
    static_assert(NS % F::kSpansPerUnit == 0, "a warp's slice holds whole scale units");
    constexpr int NU = NS / F::kSpansPerUnit;      // scale units per warp
    constexpr int XW = F::kXWords;                 // 32-bit words per 8 activations
    constexpr uint32_t kXElem = 4u * XW / 8u;      // bytes per activation
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nc = (blockDim.x >> 5) - 1;
    const int nst = G.nst, nxs = G.x_slots;
    uint8_t *stage_w = smem;
    uint8_t *stage_a = smem + (size_t)nst * L.stage_w;
    uint8_t *xstage = smem + (size_t)(nst - nxs) * L.stage_w;   // the activations, then ring slots again
    float *red = reinterpret_cast<float *>(smem + L.red_off);
    constexpr int RS = F::kRedStride;
    static_assert(RS >= (F::kHiLo ? 4 : 8), "a batch row holds every token's partial sum");
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    uint64_t *empty = full + nst;
    uint64_t *x_full = empty + nst, *x_free = x_full + 1;

    const int Gx = gridDim.x, b = blockIdx.x;
    const int split = blockIdx.y, nsplit = gridDim.y;
    const int n_my = b < G.nrowb ? (G.nrowb - b + Gx - 1) / Gx : 0;
    const int sp_begin = split * G.sps;
    const int sp_end = min(G.nsp, sp_begin + G.sps);
    const uint32_t seg_col = nsplit == 1 ? 0u : F::span_byte(sp_begin);
    const uint32_t seg_bytes = nsplit == 1 ? F::row_bytes(p) : F::span_byte(sp_end) - seg_col;
    const uint32_t arowbytes = F::aux_row_bytes(p);
    const uint32_t xseg_bytes = (uint32_t)(sp_end - sp_begin) * 64u * kXElem;
    const int S = G.S;
    // Batch k into its slot (producer warp): lane 0 arms the slot's barrier
    // with the batch's bytes; lanes 0..3 copy four whole rows each (one bulk
    // copy issue costs about as much as a few kilobytes of transfer), or with
    // a column split lane r copies row r's segment; the last lane copies the
    // side data.
    auto issue = [&](int k) {
        const int slot = k % nst;
        const int o0 = (b + k * Gx) * RB;
        const int rows = min(RB, p.O - o0);
        // the batch's rows lie inside the matrix and the segment inside a row
        // (bounds-checking build); a refused batch is armed with no bytes
        const bool in = qg_guard(o0 >= 0 && rows >= 1 && o0 + rows <= p.O && seg_col + seg_bytes <= F::row_bytes(p),
                                 err);
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], in ? (uint32_t)rows * (seg_bytes + arowbytes) : 0u);
        __syncwarp();
        if (!in) return;
        uint8_t *dw = stage_w + (size_t)slot * L.stage_w;
        if (nsplit == 1) {
            // whole rows: four consecutive rows are consecutive in memory
            const int n4 = min(4, rows - 4 * lane);
            if (lane < 4 && n4 > 0)
                bulk_copy_g2s(dw + (size_t)lane * L.group_pitch, F::w_src(p, o0 + 4 * lane, 0u), (uint32_t)n4 * seg_bytes,
                              &full[slot]);
        } else {
            for (int r = lane; r < rows; r += 32)
                bulk_copy_g2s(dw + staged_row_off(r, L.group_pitch, seg_bytes), F::w_src(p, o0 + r, seg_col), seg_bytes,
                              &full[slot]);
        }
        if (arowbytes && lane == 31)
            bulk_copy_g2s(stage_a + (size_t)slot * L.stage_a, F::a_src(p, o0), (uint32_t)rows * arowbytes,
                          &full[slot]);
    };
    // The producer warp sets up the barriers and streams in the first batch
    // (the weights do not depend on the previous kernel on the stream) before
    // the block barrier; the consumers see the barriers after it.
    const int first = min(nst, n_my), nw0 = min(nst - nxs, first);
    if (warp == 0) {
        if (lane == 0) {
            qg_stamp_entry(err);
            griddep_launch_dependents();
            for (int s = 0; s < nst; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], (uint32_t)nc);
            }
            mbar_init(x_full, 1);
            mbar_init(x_free, (uint32_t)nc);
            mbar_fence_init();
        }
        __syncwarp();
        if (nw0 > 0) issue(0);
    }
    __syncthreads();

    if (warp == 0) {
        // ------------------------------- producer -------------------------------
        // Lands every copy this warp issued (batches below `issued`, and the
        // activations) before the warp leaves after a wait that gave up.
        auto drain = [&](int k, int issued) {
            if (lane == 0) {
                raise_device_error(err, kErrTimeout);
                (void)mbar_wait(x_full, 0u);
                for (int j = k; j < issued; ++j) (void)mbar_wait(&full[j % nst], (uint32_t)(j / nst) & 1u);
            }
        };
        // The activations (x may be the previous kernel's output) come after
        // the wait for it, ahead of the other free slots' weight copies,
        // because the consumers need them before any batch.
        griddep_wait();
        if (lane == 0) qg_stamp(err, kStWaitDone);
        if (lane == 0) mbar_arrive_expect_tx(x_full, (uint32_t)S * xseg_bytes);
        __syncwarp();
        for (int s = lane; s < S; s += 32)
            if (qg_guard((long)sp_begin * 64 + (long)(xseg_bytes / kXElem) <= (long)p.I, err))
                bulk_copy_g2s(xstage + (size_t)s * L.x_stride, F::x_src(p, s, sp_begin * 64), xseg_bytes, x_full);
        for (int k = 1; k < nw0; ++k) issue(k);
        // The slots under the activations, once every consumer has its fragments.
        if (nw0 < first) {
            if (!mbar_wait(x_free, 0u)) {
                drain(0, nw0);
                return;
            }
            for (int k = nw0; k < first; ++k) issue(k);
        }
        // This lane's outputs of a batch: (row, token) i = lane + 32 v, v < 4.
        int ri[4], si[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int i = lane + 32 * v;
            ri[v] = i < RB * S ? i / S : -1;
            si[v] = i < RB * S ? i - (i / S) * S : 0;
        }
        for (int k = 0; k < n_my; ++k) {
            const int slot = k % nst;
            if (!mbar_wait(&empty[slot], (uint32_t)(k / nst) & 1u)) {
                drain(k, min(k + nst, n_my));
                return;
            }
            // The slot's weights are consumed: refill it first.  The partial
            // sums of batch k sit in the half of the partial area for its
            // pass parity, which batch k + nst does not write.
            if (k + nst < n_my) issue(k + nst);
            const int o0 = (b + k * Gx) * RB;
            const float *rs = red + (size_t)((((k / nst) & 1) * nst + slot) * nc) * RB * RS;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int w = 0; w < nc; ++w)
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    if (ri[v] >= 0) acc[v] += rs[((size_t)w * RB + ri[v]) * RS + si[v]];
#pragma unroll
            for (int v = 0; v < 4; ++v)
                if (ri[v] >= 0 && o0 + ri[v] < p.O && qg_guard(split < nsplit && si[v] < S, err))
                    out[((size_t)split * S + si[v]) * p.O + o0 + ri[v]] = acc[v];
            __syncwarp();
        }
        if (lane == 0) {
            qg_stamp(err, kStStored);
            qg_stamp_put(err, kStBatches, (unsigned long long)n_my);
        }
        return;
    }

    // ------------------------------- consumers ----------------------------------
    // Everything a consumer reads is in shared memory (the producer waits for
    // the previous kernel before it copies the activations).
    const int cw = warp - 1;
    const int g = lane >> 2, t = lane & 3;
    const int sl0 = cw * NS;                                   // first span of this warp, local to the segment
    const int nsw = max(0, min(NS, (sp_end - sp_begin) - sl0));  // spans this warp owns
    // column g of the MMA: token and part (high / low half) it carries
    const int tok = F::kHiLo ? (g >> 1) : g;
    const bool lo_part = F::kHiLo && (g & 1);
    const bool has_tok = tok < S;
    if (!mbar_wait(x_full, 0u)) {
        if (lane == 0) raise_device_error(err, kErrTimeout);
        return;
    }
    if (tid == 32) qg_stamp(err, kStXReady);
    // Setup.  The staged activations of this warp's spans are entries of
    // eight (span sp, word j, lane t: elements 16 t + 8 j .. +7 of the span)
    // per token.  All 32 lanes share the work of scaling them to fp16 in
    // place, entry by entry; then lane (g, t) loads its B fragments.
    const uint32_t x0 = smem_addr(xstage);
    const int per_tok = 8 * nsw;                               // entries per token
    auto xentry = [&](int s, int sp, int j, int tt) {
        return x0 + (uint32_t)s * L.x_stride + (uint32_t)((sl0 + sp) * 64 + 16 * tt + 8 * j) * kXElem;
    };
    // Largest |x| per token over the warp's spans -> F (a NaN or an infinity
    // makes F large; such a token's outputs are NaN either way).  The lanes
    // split into groups of LPT, one group per token; lane r of a group takes
    // the token's entries r, r + LPT, ...
    const int S2 = S <= 1 ? 1 : S <= 2 ? 2 : S <= 4 ? 4 : 8;
    const int LPT = 32 / S2;
    const int my_s = lane / LPT, r0 = lane - my_s * LPT;
    const bool my_ok = my_s < S;
    float m = 0.f;
#pragma unroll 4
    for (int r = r0; r < (my_ok ? per_tok : 0); r += LPT) {
        uint32_t w[XW];
        lds_xwords<XW>(xentry(my_s, r >> 3, (r >> 2) & 1, r & 3), w);
        m = fmaxf(m, F::abs_max8(w));
    }
    for (int d = LPT >> 1; d >= 1; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, d));
    int Fs = (int)((__float_as_uint(m) >> 23) & 0xFF) - 127;   // m < 2^(Fs + 1)
    if (Fs < -126) Fs = -126;
    // this lane's column (token tok) and its two D columns (tokens 2t, 2t+1,
    // or token t twice with split activations); absent tokens read lane 0
    const int Fmine = __shfl_sync(0xFFFFFFFFu, Fs, has_tok ? tok * LPT : 0);
    const int cd0 = F::kHiLo ? t : 2 * t, cd1 = F::kHiLo ? t : 2 * t + 1;
    const int Fd0 = __shfl_sync(0xFFFFFFFFu, Fs, cd0 < S ? cd0 * LPT : 0);
    const int Fd1 = __shfl_sync(0xFFFFFFFFu, Fs, cd1 < S ? cd1 * LPT : 0);
    // each entry's four fp16 pairs (x0, x4), (x1, x5), (x2, x6), (x3, x7) times
    // (2^(14-F), 2^(10-F)) (elements 0, 2, 4, 6 pair with 2^-24 nibbles, 1, 3,
    // 5, 7 with 2^-20 ones), over the entry's first 16 bytes; with split
    // activations the rounding remainders, in fp16, over the next 16
    {
        const bool one_factor = Fs >= -113;   // 2^(14-F) a single f32 factor
        const Pow2Split k24 = pow2_split(14 - Fs), k20 = pow2_split(10 - Fs);
        const uint64_t kmul = one_factor ? pack2(pow2i(14 - Fs), pow2i(10 - Fs)) : pack2(k24.a, k20.a);
        const uint64_t kmul2 = pack2(k24.b, k20.b);
#pragma unroll 2
        for (int r = r0; r < (my_ok ? per_tok : 0); r += LPT) {
            const uint32_t a = xentry(my_s, r >> 3, (r >> 2) & 1, r & 3);
            uint32_t w[XW];
            lds_xwords<XW>(a, w);
            uint64_t v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[i] = fmul2(F::pair(w, i), kmul);
                if (!one_factor) v[i] = fmul2(v[i], kmul2);
            }
            uint32_t h[4], l[4];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float2 e = unpack2(v[i]), c = unpack2(v[i + 2]);
                h[2 * i] = f16x2_rn(e.x, c.x);
                h[2 * i + 1] = f16x2_rn(e.y, c.y);
                if constexpr (F::kHiLo) {
                    const float2 e0 = f16x2_to_f32(h[2 * i]), e1 = f16x2_to_f32(h[2 * i + 1]);
                    l[2 * i] = f16x2_rn(e.x - e0.x, c.x - e0.y);
                    l[2 * i + 1] = f16x2_rn(e.y - e1.x, c.y - e1.y);
                }
            }
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(h[0]), "r"(h[1]), "r"(h[2]),
                         "r"(h[3])
                         : "memory");
            if constexpr (F::kHiLo)
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a + 16u), "r"(l[0]), "r"(l[1]),
                             "r"(l[2]), "r"(l[3])
                             : "memory");
        }
    }
    (void)Fmine;
    __syncwarp();
    // B fragments bf[sp][j][h][0..1] = pairs (2h, 2h+1) of lane (g, t)'s entry (sp, j)
    const uint32_t part_off = lo_part ? 16u : 0u;
    uint32_t bf[NS][2][2][2];
#pragma unroll
    for (int sp = 0; sp < NS; ++sp)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            uint32_t h[4] = {0u, 0u, 0u, 0u};
            if (has_tok && sp < nsw)
                asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
                             : "r"(xentry(tok, sp, j, t) + part_off)
                             : "memory");
            bf[sp][j][0][0] = h[0];
            bf[sp][j][0][1] = h[1];
            bf[sp][j][1][0] = h[2];
            bf[sp][j][1][1] = h[3];
        }
    // The activations' slots go back to the ring.
    __syncwarp();
    if (lane == 0) mbar_arrive(x_free);
    // Per unit and column: sum of the activations as the MMA sees them (A =
    // the nibble pattern of 1, i.e. 2^-24 and 2^-20); the units' chains
    // interleave.
    float X[NU][2];
    {
        float d[NU][4];
#pragma unroll
        for (int u = 0; u < NU; ++u) d[u][0] = d[u][1] = d[u][2] = d[u][3] = 0.f;
#pragma unroll
        for (int q = 0; q < F::kSpansPerUnit; ++q)
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int u = 0; u < NU; ++u) {
                        const int sp = u * F::kSpansPerUnit + q;
                        mma_16816(d[u], 0x00010001u, 0x00010001u, 0x00100010u, 0x00100010u, bf[sp][j][h][0],
                                  bf[sp][j][h][1]);
                    }
#pragma unroll
        for (int u = 0; u < NU; ++u) {
            if constexpr (F::kHiLo) {
                // the two columns of a token are added at the end: one start
                // value (-8 times the token's whole sum) on the high column
                // serves both
                X[u][0] = F::kNeg8 ? -8.f * (d[u][0] + d[u][1]) : d[u][0] + d[u][1];
                X[u][1] = 0.f;
            } else {
                X[u][0] = F::kNeg8 ? -8.f * d[u][0] : d[u][0];
                X[u][1] = F::kNeg8 ? -8.f * d[u][1] : d[u][1];
            }
        }
    }

    // 2^(10 + F) of the lane's two D columns, to undo the scaling
    const Pow2Split u0 = pow2_split(10 + Fd0), u1 = pow2_split(10 + Fd1);

    const uint32_t sw0 = smem_addr(stage_w), sa0 = smem_addr(stage_a);
    float *redw = red + (size_t)cw * RB * RS;
    // MMA rows g and g + 8 of this lane: batch rows batch_row(g), batch_row(g + 8)
    const int row_lo = batch_row(g), row_hi = batch_row(g + 8);
    const uint32_t rw_lo = staged_row_off(row_lo, L.group_pitch, seg_bytes);
    const uint32_t rw_hi = staged_row_off(row_hi, L.group_pitch, seg_bytes);
    const uint32_t ra_lo = (uint32_t)row_lo * arowbytes, ra_hi = (uint32_t)row_hi * arowbytes;

    for (int k = 0; k < n_my; ++k) {
        const int slot = k % nst;
        if (!mbar_wait(&full[slot], (uint32_t)(k / nst) & 1u)) {
            if (lane == 0) raise_device_error(err, kErrTimeout);
            return;
        }
        if (tid == 32 && k == 0) qg_stamp(err, kStFirstBatch);
        const uint32_t swb = sw0 + (uint32_t)slot * L.stage_w;
        const uint32_t sab = sa0 + (uint32_t)slot * L.stage_a;
        float *rslot = redw + (size_t)((((k / nst) & 1) * nst + slot) * nc) * RB * RS;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int u = 0; u < NU; ++u) {
            if (u * F::kSpansPerUnit < nsw) {
                const uint32_t so = F::side_off(sp_begin + sl0, sl0, u);
                const typename F::Side s0 = F::side(swb + rw_lo, sab + ra_lo, so);
                const typename F::Side s1 = F::side(swb + rw_hi, sab + ra_hi, so);
                float d[4];
                d[0] = d[2] = F::kNeg8 ? X[u][0] : 0.f;
                d[1] = d[3] = F::kNeg8 ? X[u][1] : 0.f;
#pragma unroll
                for (int q = 0; q < F::kSpansPerUnit; ++q) {
                    const int sp = u * F::kSpansPerUnit + q;
                    const uint32_t off = F::span_off(sl0 + sp) + 8u * (uint32_t)t;
                    const uint2 wa = lds_u32x2(swb + rw_lo + off), wb = lds_u32x2(swb + rw_hi + off);
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const uint32_t a = j ? wa.y : wa.x, c = j ? wb.y : wb.x;
                        const uint32_t a8 = a >> 8, c8 = c >> 8;
                        mma_16816(d, a & 0x000F000Fu, c & 0x000F000Fu, a & 0x00F000F0u, c & 0x00F000F0u,
                                  bf[sp][j][0][0], bf[sp][j][0][1]);
                        mma_16816(d, a8 & 0x000F000Fu, c8 & 0x000F000Fu, a8 & 0x00F000F0u, c8 & 0x00F000F0u,
                                  bf[sp][j][1][0], bf[sp][j][1][1]);
                    }
                }
                F::apply(acc, d, s0, s1, X[u]);
                if constexpr (F::kFenceUnits) asm volatile("" ::: "memory");
            }
        }
        // partial sums of this warp's spans, unscaled, per (batch row, token)
        if constexpr (F::kHiLo) {
            if (t < S) {
                rslot[(size_t)row_lo * RS + t] = (acc[0] + acc[1]) * u0.a * u0.b;
                rslot[(size_t)row_hi * RS + t] = (acc[2] + acc[3]) * u0.a * u0.b;
            }
        } else {
            if (2 * t < S) {
                rslot[(size_t)row_lo * RS + 2 * t] = acc[0] * u0.a * u0.b;
                rslot[(size_t)row_hi * RS + 2 * t] = acc[2] * u0.a * u0.b;
            }
            if (2 * t + 1 < S) {
                rslot[(size_t)row_lo * RS + 2 * t + 1] = acc[1] * u1.a * u1.b;
                rslot[(size_t)row_hi * RS + 2 * t + 1] = acc[3] * u1.a * u1.b;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }
    if (tid == 32) qg_stamp(err, kStConsumed);
}

// One block per SM of at most F::kMaxConsumerWarps + 1 warps: the B
// fragments of a warp's 512 columns take 64 registers a thread.
template <class F, int NS, int RB>
__global__ void __launch_bounds__(32 * (F::kMaxConsumerWarps + 1), 1)
gemv_mma_kernel(const typename F::Params p, float *__restrict__ out, MmaGrid G, MmaLayout L, int *err) {
    gemv_mma_body<F, NS, RB>(p, out, G, L, err);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
constexpr int kMmaSpansPerWarp = 8;      // 512 weights of a row per consumer warp

struct MmaPlan {
    MmaGrid G;
    MmaLayout L;
    int nc;          // consumer warps
    int splits;
    int per_sm;      // blocks per SM the ring was sized for
};

// Plan for rows of nsp spans (64 weights each), `granule` spans per column
// split boundary, rowbytes / arowbytes staged per row (whole row), xelem
// bytes per activation, red_stride = the format's kRedStride, and
// span_bytes(sp) the byte offset of span sp.
// False if the shape does not fit.
template <class SpanBytes>
bool mma_plan(int nsp, int granule, uint32_t rowbytes, uint32_t arowbytes, uint32_t xelem, int S, int O, int RB,
              int max_warps, int red_stride, SpanBytes span_bytes, MmaPlan *pl) {
    if (nsp < 1 || RB != 16) return false;
    int splits = (nsp + kMmaSpansPerWarp * max_warps - 1) / (kMmaSpansPerWarp * max_warps);
    int sps = (nsp + splits - 1) / splits;
    sps = (sps + granule - 1) / granule * granule;
    splits = (nsp + sps - 1) / sps;
    if (splits == 1) sps = nsp;
    const int nc = (sps + kMmaSpansPerWarp - 1) / kMmaSpansPerWarp;
    if (nc > max_warps) return false;
    // the largest staged segment
    uint32_t seg = rowbytes;
    if (splits > 1) {
        seg = 0;
        for (int s = 0; s < splits; ++s) {
            const int b0 = s * sps, b1 = std::min(nsp, b0 + sps);
            const uint32_t n = span_bytes(b1) - span_bytes(b0);
            if (n % 16 != 0) return false;
            seg = std::max(seg, n);
        }
    }
    if (seg % 16 != 0 || rowbytes % 16 != 0 || arowbytes % 16 != 0) return false;
    const uint32_t pitch = (uint32_t)(((4u * seg + 96u + 127u) / 128u) * 128u) - 96u;   // >= 4 seg, 32 mod 128
    const uint32_t stage_w = 4u * pitch;                      // RB = 16 rows
    // the activations of the widest segment, S rows
    const uint32_t xseg = (uint32_t)sps * 64u * xelem;
    const uint32_t x_stride = (xseg + 127u) / 128u * 128u + 16u;
    const int x_slots = (int)(((uint32_t)S * x_stride + stage_w - 1) / stage_w);
    const uint32_t stage_a = (uint32_t)(((RB * arowbytes) + 127u) / 128u * 128u);
    const uint32_t red = (uint32_t)nc * RB * (uint32_t)red_stride * 4u;
    const uint32_t per_slot = stage_w + stage_a + 2u * red + 16u;   // + x_full, x_free below
    // about 16 consumer warps per SM; as many slots (2..6) as fit
    int per_sm = std::max(1, 16 / nc);
    int nst = 0;
    for (; per_sm >= 1; --per_sm) {
        long budget = 233472L / per_sm - 1024;
        if (budget > 232448) budget = 232448;
        budget -= 16;
        nst = (int)std::min<long>(6, budget / per_slot);
        if (nst >= 2 && nst - x_slots >= 1) break;   // a slot left beside the activations
    }
    if (nst < 2 || nst - x_slots < 1) return false;
    pl->nc = nc;
    pl->splits = splits;
    pl->per_sm = per_sm;
    pl->G.nsp = nsp;
    pl->G.sps = sps;
    pl->G.nrowb = (O + RB - 1) / RB;
    pl->G.nst = nst;
    pl->G.x_slots = x_slots;
    pl->G.S = S;
    pl->L.group_pitch = pitch;
    pl->L.stage_w = stage_w;
    pl->L.stage_a = stage_a;
    pl->L.red_off = (uint32_t)nst * (stage_w + stage_a);
    pl->L.bar_off = pl->L.red_off + 2u * (uint32_t)nst * red;
    pl->L.x_stride = x_stride;
    pl->L.total = pl->L.bar_off + 16u * (uint32_t)nst + 16u;
    return true;
}

template <class F, int NS, int RB>
void launch_mma(const typename F::Params &p, float *out, const MmaPlan &pl, cudaStream_t st) {
    auto kern = gemv_mma_kernel<F, NS, RB>;
    set_max_dynamic_smem(reinterpret_cast<const void *>(kern), 232448);
    const int threads = 32 * (pl.nc + 1);
    int per_sm = 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, pl.L.total) != cudaSuccess ||
        per_sm < 1) {
        cudaGetLastError();
        per_sm = 1;
    }
    long resident = (long)num_sms() * per_sm / pl.splits;
    if (resident < 1) resident = 1;
    const int grid_x = pl.G.nrowb < resident ? pl.G.nrowb : (int)resident;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_x, pl.splits, 1);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = pl.L.total;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, kern, p, out, pl.G, pl.L, device_error_word());
    count_launch();
}

}  // namespace qg

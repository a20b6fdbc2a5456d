// streamk.h -- how the tensor-core prefill GEMM splits its work over the
// resident thread blocks ("stream-K"): the (output tile, K step) units of the
// whole problem are laid end to end, tile by tile, and block c of P takes the
// contiguous range [c*U/P, (c+1)*U/P).  A tile whose K steps fall into more
// than one block's range is reduced through per-block partial slots; the
// block that arrives last at the tile's counter sums the slots in contributor
// order and writes the output.
//
// Plain integer functions, compiled for the host too, so that the
// partition can be checked exhaustively on the CPU.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define QG_HD __host__ __device__ __forceinline__
#else
#define QG_HD inline
#endif

namespace qg {
namespace sk {

// First unit of block c:  floor(c * U / P).
QG_HD int64_t range_begin(int64_t c, int64_t U, int64_t P) { return c * U / P; }

// The block whose range holds unit u: the largest c with floor(c*U/P) <= u,
// which is floor(((u + 1) * P - 1) / U).
QG_HD int64_t owner(int64_t u, int64_t U, int64_t P) { return ((u + 1) * P - 1) / U; }

// Blocks that hold at least one K step of tile t (Kt steps per tile):
// [first_contributor, last_contributor].
QG_HD int64_t first_contributor(int64_t t, int64_t Kt, int64_t U, int64_t P) { return owner(t * Kt, U, P); }
QG_HD int64_t last_contributor(int64_t t, int64_t Kt, int64_t U, int64_t P) {
    return owner(t * Kt + Kt - 1, U, P);
}

// Partial slot that block c uses for tile t: every block has two, slot 0 for
// the tile its range starts in and slot 1 for the tile its range ends in (a
// range that starts and ends in the same tile uses slot 0).  Tiles strictly
// inside a range are whole and need no slot.
QG_HD int64_t partial_slot(int64_t c, int64_t t, int64_t Kt, int64_t U, int64_t P) {
    return 2 * c + ((range_begin(c, U, P) / Kt == t) ? 0 : 1);
}

}  // namespace sk
}  // namespace qg

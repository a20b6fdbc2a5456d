// abi.cu -- the extern "C" entry points of libqgemv (declared in
// include/qgemv.h).  Every argument is checked here, on the host, before any
// pointer is dereferenced or any kernel is enqueued; a refused call returns a
// negative status and records which condition failed (qg_last_error).
#include <limits.h>
#include <stdint.h>

#include "../../include/qgemv.h"
#include "launch.h"

namespace qg {
const char *error_detail();
int run_gemm_i4g_general(float *Y, const uint16_t *X, const uint8_t *w, const float *scales, int M, int I,
                         int O, int gs, cudaStream_t st);
int run_gemm_i4g_tc(float *Y, const uint16_t *X, const uint8_t *w, const float *scales, int M, int I, int O,
                    int gs, void *ws, size_t ws_bytes, cudaStream_t st, bool *taken);
size_t ws_gemm_i4g(int M, int I, int O, int gs);
int run_gemm_fp8b128_general(float *Y, const uint16_t *X, const uint8_t *w, const float *scale_inv, int M,
                             int I, int O, cudaStream_t st);
int run_gemm_fp8b128_tc(float *Y, const uint16_t *X, const uint8_t *w, const float *scale_inv, int M, int I,
                        int O, void *ws, size_t ws_bytes, cudaStream_t st, bool *taken);
size_t ws_gemm_fp8b128(int M, int I, int O);
int run_gemm_fp8ue8m0_general(float *Y, const uint16_t *X, const uint8_t *w, const uint8_t *scale_e8m0, int M,
                              int I, int O, cudaStream_t st);
int run_gemm_fp8ue8m0_tc(float *Y, const uint16_t *X, const uint8_t *w, const uint8_t *scale_e8m0, int M, int I,
                         int O, void *ws, size_t ws_bytes, cudaStream_t st, bool *taken);
size_t ws_gemm_fp8ue8m0(int M, int I, int O);
int run_gemm_mq4v2_general(float *Y, const uint16_t *X, const uint8_t *blocks, int M, int I, int O,
                           cudaStream_t st);
int run_gemm_mq4v2_tc(float *Y, const uint16_t *X, const uint8_t *blocks, int M, int I, int O, void *ws,
                      size_t ws_bytes, cudaStream_t st, bool *taken);
size_t ws_gemm_mq4v2(int M, int I, int O);
int run_gemm_mq4v1_general(float *Y, const uint16_t *X, const uint8_t *blocks, int M, int I, int O,
                           cudaStream_t st);
int run_gemm_mq4v1_tc(float *Y, const uint16_t *X, const uint8_t *blocks, int M, int I, int O, void *ws,
                      size_t ws_bytes, cudaStream_t st, bool *taken);
size_t ws_gemm_mq4v1(int M, int I, int O);
int run_gemm_mq4c_general(float *Y, const uint16_t *X, const uint8_t *blocks, int M, int I, int O,
                          cudaStream_t st);
int run_gemm_mq4c_tc(float *Y, const uint16_t *X, const uint8_t *blocks, int M, int I, int O, void *ws,
                     size_t ws_bytes, cudaStream_t st, bool *taken);
size_t ws_gemm_mq4c(int M, int I, int O);
}  // namespace qg

using namespace qg;

namespace {

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

#define QG_REFUSE(code, ...)              \
    do {                                  \
        set_error_detail(__VA_ARGS__);    \
        return (code);                    \
    } while (0)

// Common checks of the shape arguments.
int check_dims(const char *fn, const char *sname, int S, int I, int O) {
    if (S < 1) QG_REFUSE(kEInval, "%s: %s = %d, must be >= 1", fn, sname, S);
    if (I < 1) QG_REFUSE(kEInval, "%s: I = %d, must be >= 1", fn, I);
    if (O < 1) QG_REFUSE(kEInval, "%s: O = %d, must be >= 1", fn, O);
    return kOk;
}

int check_gs(const char *fn, int gs) {
    if (gs < 2 || (gs & 1)) QG_REFUSE(kEGs, "%s: gs = %d, must be even and >= 2", fn, gs);
    return kOk;
}

cudaStream_t as_stream(qg_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// One grouped tensor-core launch for the non-empty groups g0 .. g1 (at most
// kMoeGroupsPerLaunch), rows [lo, hi) of X and Y; *taken false when the
// shapes or pointers do not suit it.
int moe_gemm_chunk_tc(int fmt, float *Y, const uint16_t *X, const qg_expert *experts, const int *ge,
                             const int *off, const int *idx, int n, int I, int O, int gs, void *ws, size_t ws_bytes,
                             cudaStream_t st, bool *taken) {
    int row0[kMoeGroupsPerLaunch], rows[kMoeGroupsPerLaunch];
    const uint8_t *w[kMoeGroupsPerLaunch];
    const float *sc[kMoeGroupsPerLaunch];
    const int lo = off[idx[0]], hi = off[idx[n - 1] + 1];
    for (int i = 0; i < n; ++i) {
        const int g = idx[i];
        row0[i] = off[g] - lo;
        rows[i] = off[g + 1] - off[g];
        w[i] = static_cast<const uint8_t *>(experts[ge[g]].w);
        sc[i] = experts[ge[g]].scales;
    }
    float *Yc = Y + (size_t)lo * O;
    const uint16_t *Xc = X + (size_t)lo * I;
    const int M = hi - lo;
    switch (fmt) {
        case QG_FMT_I4G:
            return run_gemm_moe_i4g_tc(Yc, Xc, row0, rows, w, sc, n, M, I, O, gs, ws, ws_bytes, st, taken);
        case QG_FMT_FP8B128:
            return run_gemm_moe_fp8b128_tc(Yc, Xc, row0, rows, w, sc, n, M, I, O, ws, ws_bytes, st, taken);
        case QG_FMT_FP8UE8M0:
            return run_gemm_moe_fp8ue8m0_tc(Yc, Xc, row0, rows, w, sc, n, M, I, O, ws, ws_bytes, st, taken);
        case QG_FMT_MQ4V2: return run_gemm_moe_mq4v2_tc(Yc, Xc, row0, rows, w, n, M, I, O, ws, ws_bytes, st, taken);
        case QG_FMT_MQ4V1: return run_gemm_moe_mq4v1_tc(Yc, Xc, row0, rows, w, n, M, I, O, ws, ws_bytes, st, taken);
        default: return run_gemm_moe_mq4c_tc(Yc, Xc, row0, rows, w, n, M, I, O, ws, ws_bytes, st, taken);
    }
}

size_t moe_chunk_ws(int fmt, const int *off, const int *idx, int n, int I, int O, int gs) {
    int rows[kMoeGroupsPerLaunch];
    for (int i = 0; i < n; ++i) rows[i] = off[idx[i] + 1] - off[idx[i]];
    const int M = off[idx[n - 1] + 1] - off[idx[0]];
    switch (fmt) {
        case QG_FMT_I4G: return ws_gemm_moe_i4g(rows, n, M, I, O, gs);
        case QG_FMT_FP8B128:
        case QG_FMT_FP8UE8M0: return ws_gemm_moe_fp8(rows, n, M, I, O);
        default: return ws_gemm_moe_mq4(rows, n, M, I, O);
    }
}

bool moe_fmt_ok(int fmt) {
    return fmt == QG_FMT_I4G || fmt == QG_FMT_FP8B128 || fmt == QG_FMT_FP8UE8M0 || fmt == QG_FMT_MQ4V2 ||
           fmt == QG_FMT_MQ4V1 || fmt == QG_FMT_MQ4C;
}

// Calls fn(idx, n) for the non-empty groups in chunks of at most
// kMoeGroupsPerLaunch; stops at the first non-zero return.
template <class Fn>
int for_each_moe_chunk(const int *off, int n_groups, Fn fn) {
    int idx[kMoeGroupsPerLaunch], n = 0;
    for (int g = 0; g < n_groups; ++g) {
        if (off[g + 1] == off[g]) continue;
        idx[n++] = g;
        if (n == kMoeGroupsPerLaunch) {
            const int rc = fn(idx, n);
            if (rc) return rc;
            n = 0;
        }
    }
    return n ? fn(idx, n) : 0;
}

}  // namespace

extern "C" {

const char *qg_strerror(int status) {
    switch (status) {
        case QG_OK: return "QG_OK: success";
        case QG_EINVAL: return "QG_EINVAL: null pointer, non-positive size or size overflow";
        case QG_EGS: return "QG_EGS: group size must be even and >= 2";
        case QG_ESHAPE: return "QG_ESHAPE: shape not supported by the format (MQ4-V2 needs I % 256 == 0)";
        case QG_EALIGN: return "QG_EALIGN: pointer misaligned for its element type";
        case QG_EWORKSPACE: return "QG_EWORKSPACE: workspace missing or smaller than qg_workspace_bytes()";
        case QG_ECUDA: return "QG_ECUDA: CUDA runtime error";
        case QG_ETIMEOUT: return "QG_ETIMEOUT: a kernel gave up waiting on a barrier";
        case QG_EEXPERT: return "QG_EEXPERT: a routed slot named a missing expert or one with misaligned weights";
        case QG_EBOUNDS: return "QG_EBOUNDS: a kernel formed an index outside its arrays (bounds-checking build)";
        default: return "unknown qg_status";
    }
}

const char *qg_last_error(void) { return error_detail(); }

unsigned long long qg_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int qg_stamps_take(uint64_t *host, int max_blocks) {
    if (host == nullptr || max_blocks < 1) {
        set_error_detail("qg_stamps_take: host must be non-NULL and max_blocks >= 1 (got %d)", max_blocks);
        return kEInval;
    }
    return stamps_take(reinterpret_cast<unsigned long long *>(host), max_blocks);
}

int qg_device_status(int *status) {
    if (!status) QG_REFUSE(kEInval, "qg_device_status: status must be non-NULL");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        set_error_detail("qg_device_status: %s", cudaGetErrorString(e));
        return kECuda;
    }
    return read_device_error(status);
}

size_t qg_workspace_bytes(int fmt, int S, int I, int O, int gs) {
    if (S < 1 || I < 1 || O < 1) return 0;
    switch (fmt) {
        case QG_FMT_I4G: return (gs >= 2 && !(gs & 1)) ? ws_i4g(S, I, O, gs) : 0;
        case QG_FMT_FP8B128: return ws_fp8b128(S, I, O);
        case QG_FMT_FP8UE8M0: return ws_fp8ue8m0(S, I, O);
        case QG_FMT_MQ4V2: return (I % 256 == 0) ? ws_mq4v2(S, I, O) : 0;
        case QG_FMT_MQ4V1: return (I % 256 == 0) ? ws_mq4v1(S, I, O) : 0;
        case QG_FMT_MQ4C: return (I % 256 == 0) ? ws_mq4c(S, I, O) : 0;
        case QG_FMT_Q2_0: return (I % 64 == 0) ? ws_q2_0(S, I, O) : 0;
        default: return 0;
    }
}

size_t qg_gemm_workspace_bytes(int fmt, int M, int I, int O, int gs) {
    if (M < 1 || I < 1 || O < 1) return 0;
    switch (fmt) {
        case QG_FMT_I4G: return (gs >= 2 && !(gs & 1)) ? ws_gemm_i4g(M, I, O, gs) : 0;
        case QG_FMT_FP8B128: return ws_gemm_fp8b128(M, I, O);
        case QG_FMT_FP8UE8M0: return ws_gemm_fp8ue8m0(M, I, O);
        case QG_FMT_MQ4V2: return ws_gemm_mq4v2(M, I, O);
        case QG_FMT_MQ4V1: return ws_gemm_mq4v1(M, I, O);
        case QG_FMT_MQ4C: return ws_gemm_mq4c(M, I, O);
        default: return 0;
    }
}

int qgemv_i4g(float *y, const float *x, const uint8_t *w, const float *scales, int S, int I, int O, int gs,
              void *ws, size_t ws_bytes, qg_stream_t stream) {
    const char *fn = "qgemv_i4g";
    int rc = check_dims(fn, "S", S, I, O);
    if (rc) return rc;
    if ((rc = check_gs(fn, gs))) return rc;
    if (!y || !x || !w || !scales) QG_REFUSE(kEInval, "%s: y, x, w and scales must be non-NULL", fn);
    if (!aligned(y, 4) || !aligned(x, 4) || !aligned(scales, 4))
        QG_REFUSE(kEAlign, "%s: y, x and scales must be 4-byte aligned", fn);
    if (ws && !aligned(ws, 256)) QG_REFUSE(kEAlign, "%s: workspace must be 256-byte aligned", fn);
    cudaGetLastError();
    return run_gemv_i4g(y, x, w, scales, S, I, O, gs, ws, ws_bytes, as_stream(stream));
}

int qgemv_fp8b128(float *y, const uint16_t *x, const uint8_t *w, const float *scale_inv, int S, int I, int O,
                  void *ws, size_t ws_bytes, qg_stream_t stream) {
    const char *fn = "qgemv_fp8b128";
    int rc = check_dims(fn, "S", S, I, O);
    if (rc) return rc;
    if (!y || !x || !w || !scale_inv) QG_REFUSE(kEInval, "%s: y, x, w and scale_inv must be non-NULL", fn);
    if (!aligned(y, 4) || !aligned(x, 2) || !aligned(scale_inv, 4))
        QG_REFUSE(kEAlign, "%s: y and scale_inv must be 4-byte and x 2-byte aligned", fn);
    if (ws && !aligned(ws, 256)) QG_REFUSE(kEAlign, "%s: workspace must be 256-byte aligned", fn);
    cudaGetLastError();
    return run_gemv_fp8b128(y, x, w, scale_inv, S, I, O, ws, ws_bytes, as_stream(stream));
}

int qgemv_q2_0(float *y, const uint16_t *x, const uint8_t *blocks, int S, int I, int O, void *ws, size_t ws_bytes,
               qg_stream_t stream) {
    const char *fn = "qgemv_q2_0";
    int rc = check_dims(fn, "S", S, I, O);
    if (rc) return rc;
    if (I % 64) QG_REFUSE(kEShape, "%s: I = %d is not a multiple of 64", fn, I);
    if (!y || !x || !blocks) QG_REFUSE(kEInval, "%s: y, x and blocks must be non-NULL", fn);
    if (!aligned(y, 4) || !aligned(x, 2) || !aligned(blocks, 2))
        QG_REFUSE(kEAlign, "%s: y must be 4-byte, x and blocks 2-byte aligned", fn);
    if (ws && !aligned(ws, 256)) QG_REFUSE(kEAlign, "%s: workspace must be 256-byte aligned", fn);
    cudaGetLastError();
    return run_gemv_q2_0(y, x, blocks, S, I, O, ws, ws_bytes, as_stream(stream));
}

int qgemv_fp8ue8m0(float *y, const uint16_t *x, const uint8_t *w, const uint8_t *scale_e8m0, int S, int I, int O,
                   void *ws, size_t ws_bytes, qg_stream_t stream) {
    const char *fn = "qgemv_fp8ue8m0";
    int rc = check_dims(fn, "S", S, I, O);
    if (rc) return rc;
    if (!y || !x || !w || !scale_e8m0) QG_REFUSE(kEInval, "%s: y, x, w and scale_e8m0 must be non-NULL", fn);
    if (!aligned(y, 4) || !aligned(x, 2)) QG_REFUSE(kEAlign, "%s: y must be 4-byte and x 2-byte aligned", fn);
    if (ws && !aligned(ws, 256)) QG_REFUSE(kEAlign, "%s: workspace must be 256-byte aligned", fn);
    cudaGetLastError();
    return run_gemv_fp8ue8m0(y, x, w, scale_e8m0, S, I, O, ws, ws_bytes, as_stream(stream));
}

size_t qg_moe_gemm_workspace_bytes(int fmt, const int *group_offsets, int n_groups, int I, int O, int gs) {
    if (!moe_fmt_ok(fmt) || n_groups < 1 || !group_offsets || I < 1 || O < 1) return 0;
    if (fmt == QG_FMT_I4G && (gs < 2 || (gs & 1))) return 0;
    for (int g = 0; g < n_groups; ++g)
        if (group_offsets[g] < 0 || group_offsets[g + 1] < group_offsets[g]) return 0;
    size_t need = 0;
    // the grouped launches, and the group-by-group calls taken when pointers do not suit them
    for_each_moe_chunk(group_offsets, n_groups, [&](const int *idx, int n) {
        const size_t c = moe_chunk_ws(fmt, group_offsets, idx, n, I, O, gs);
        if (c > need) need = c;
        for (int i = 0; i < n; ++i) {
            const size_t s1 = qg_gemm_workspace_bytes(fmt, group_offsets[idx[i] + 1] - group_offsets[idx[i]], I, O, gs);
            if (s1 > need) need = s1;
        }
        return 0;
    });
    return need;
}

int qgemm_moe(int fmt, float *Y, const uint16_t *X, const qg_expert *experts, int n_experts,
              const int *group_expert, const int *group_offsets, int n_groups, int I, int O, int gs, void *ws,
              size_t ws_bytes, qg_stream_t stream) {
    const char *fn = "qgemm_moe";
    if (!moe_fmt_ok(fmt)) QG_REFUSE(kEInval, "%s: unknown format id %d", fn, fmt);
    if (n_groups < 0) QG_REFUSE(kEInval, "%s: n_groups = %d, must be >= 0", fn, n_groups);
    if (n_groups == 0) return kOk;
    if (!experts || !group_expert || !group_offsets)
        QG_REFUSE(kEInval, "%s: experts, group_expert and group_offsets must be non-NULL", fn);
    if (n_experts < 1) QG_REFUSE(kEInval, "%s: n_experts = %d, must be >= 1", fn, n_experts);
    if (I < 1 || O < 1) QG_REFUSE(kEInval, "%s: I = %d and O = %d must be >= 1", fn, I, O);
    if (fmt == QG_FMT_I4G && check_gs(fn, gs)) return kEGs;
    if ((fmt == QG_FMT_MQ4V2 || fmt == QG_FMT_MQ4V1 || fmt == QG_FMT_MQ4C) && I % 256)
        QG_REFUSE(kEShape, "%s: I = %d is not a multiple of 256", fn, I);
    if (group_offsets[0] < 0) QG_REFUSE(kEInval, "%s: group_offsets[0] = %d is negative", fn, group_offsets[0]);
    int m_max = 0;
    for (int g = 0; g < n_groups; ++g) {
        const int m = group_offsets[g + 1] - group_offsets[g];
        if (m < 0) QG_REFUSE(kEInval, "%s: group_offsets decrease at group %d", fn, g);
        if (group_expert[g] < 0 || group_expert[g] >= n_experts)
            QG_REFUSE(kEInval, "%s: group %d names expert %d of %d", fn, g, group_expert[g], n_experts);
        if (m > m_max) m_max = m;
    }
    if (m_max == 0) return kOk;
    if (!Y || !X) QG_REFUSE(kEInval, "%s: Y and X must be non-NULL", fn);
    const size_t need = qg_moe_gemm_workspace_bytes(fmt, group_offsets, n_groups, I, O, gs);
    if (need > 0 && (ws == nullptr || ws_bytes < need))
        QG_REFUSE(kEWorkspace, "%s: needs a workspace of %zu bytes (qg_moe_gemm_workspace_bytes; got %zu)", fn, need,
                  ws == nullptr ? (size_t)0 : ws_bytes);
    if (ws && !aligned(ws, 256)) QG_REFUSE(kEAlign, "%s: workspace must be 256-byte aligned", fn);
    cudaGetLastError();
    const cudaStream_t st = as_stream(stream);
    // up to kMoeGroupsPerLaunch groups per tensor-core launch; group by group
    // through the format's GEMM entry point when the chunk does not suit it
    return for_each_moe_chunk(group_offsets, n_groups, [&](const int *idx, int n) {
        bool taken = false;
        int rc = moe_gemm_chunk_tc(fmt, Y, X, experts, group_expert, group_offsets, idx, n, I, O, gs, ws, ws_bytes,
                                   st, &taken);
        if (taken) return rc == kOk ? check_launch(fn) : rc;
        for (int i = 0; i < n; ++i) {
            const int g = idx[i];
            const int m = group_offsets[g + 1] - group_offsets[g];
            const qg_expert e = experts[group_expert[g]];
            float *Yg = Y + (size_t)group_offsets[g] * O;
            const uint16_t *Xg = X + (size_t)group_offsets[g] * I;
            const uint8_t *w = static_cast<const uint8_t *>(e.w);
            switch (fmt) {
                case QG_FMT_I4G: rc = qgemm_i4g(Yg, Xg, w, e.scales, m, I, O, gs, ws, ws_bytes, stream); break;
                case QG_FMT_FP8B128: rc = qgemm_fp8b128(Yg, Xg, w, e.scales, m, I, O, ws, ws_bytes, stream); break;
                case QG_FMT_FP8UE8M0:
                    rc = qgemm_fp8ue8m0(Yg, Xg, w, reinterpret_cast<const uint8_t *>(e.scales), m, I, O, ws, ws_bytes,
                                        stream);
                    break;
                case QG_FMT_MQ4V2: rc = qgemm_mq4v2(Yg, Xg, w, m, I, O, ws, ws_bytes, stream); break;
                case QG_FMT_MQ4V1: rc = qgemm_mq4v1(Yg, Xg, w, m, I, O, ws, ws_bytes, stream); break;
                default: rc = qgemm_mq4c(Yg, Xg, w, m, I, O, ws, ws_bytes, stream); break;
            }
            if (rc != kOk) return rc;   // qg_last_error names the group's failed condition
        }
        return (int)kOk;
    });
}

int qgemv_moe(int fmt, float *y, const void *x, size_t x_slot_stride, const qg_expert *experts, int n_experts,
              const int *ids, int n_slots, int S, int I, int O, int gs, qg_stream_t stream) {
    const char *fn = "qgemv_moe";
    int rc = check_dims(fn, "S", S, I, O);
    if (rc) return rc;
    if (fmt != QG_FMT_I4G && fmt != QG_FMT_FP8B128 && fmt != QG_FMT_FP8UE8M0 && fmt != QG_FMT_MQ4V2 &&
        fmt != QG_FMT_MQ4V1 && fmt != QG_FMT_MQ4C)
        QG_REFUSE(kEInval, "%s: unknown format id %d", fn, fmt);
    if (fmt == QG_FMT_I4G && (rc = check_gs(fn, gs))) return rc;
    if ((fmt == QG_FMT_MQ4V2 || fmt == QG_FMT_MQ4V1 || fmt == QG_FMT_MQ4C) && I % 256)
        QG_REFUSE(kEShape, "%s: I = %d is not a multiple of 256", fn, I);
    if (S > 8) QG_REFUSE(kEInval, "%s: S = %d tokens per slot, must be <= 8", fn, S);
    if (n_slots < 0 || n_slots > 65535) QG_REFUSE(kEInval, "%s: n_slots = %d, must be in [0, 65535]", fn, n_slots);
    if (n_experts < 1) QG_REFUSE(kEInval, "%s: n_experts = %d, must be >= 1", fn, n_experts);
    if (n_slots == 0) return kOk;
    if (!y || !x || !experts || !ids) QG_REFUSE(kEInval, "%s: y, x, experts and ids must be non-NULL", fn);
    const size_t esz = fmt == QG_FMT_I4G ? 4 : 2;
    if (x_slot_stride != 0 && x_slot_stride < (size_t)S * I)
        QG_REFUSE(kEInval, "%s: x_slot_stride = %zu is below S * I = %zu (slots would overlap)", fn, x_slot_stride,
                  (size_t)S * I);
    if ((size_t)n_slots * S * O > (size_t)INT_MAX * 64 || x_slot_stride > (size_t)INT_MAX * 64)
        QG_REFUSE(kEInval, "%s: sizes overflow", fn);
    if (!aligned(y, 4) || !aligned(ids, 4) || !aligned(experts, 8))
        QG_REFUSE(kEAlign, "%s: y and ids must be 4-byte and experts 8-byte aligned", fn);
    if (!aligned(x, 16) || (x_slot_stride * esz) % 16)
        QG_REFUSE(kEAlign, "%s: x and every slot's x (x_slot_stride * %zu bytes) must be 16-byte aligned", fn, esz);
    cudaGetLastError();
    const cudaStream_t st = as_stream(stream);
    switch (fmt) {
        case QG_FMT_I4G:
            return run_gemv_moe_i4g(y, static_cast<const float *>(x), x_slot_stride, experts, n_experts, ids,
                                    n_slots, S, I, O, gs, st);
        case QG_FMT_FP8UE8M0:
            return run_gemv_moe_fp8ue8m0(y, static_cast<const uint16_t *>(x), x_slot_stride, experts, n_experts,
                                         ids, n_slots, S, I, O, st);
        case QG_FMT_FP8B128:
            return run_gemv_moe_fp8b128(y, static_cast<const uint16_t *>(x), x_slot_stride, experts, n_experts,
                                        ids, n_slots, S, I, O, st);
        case QG_FMT_MQ4V2:
            return run_gemv_moe_mq4v2(y, static_cast<const uint16_t *>(x), x_slot_stride, experts, n_experts,
                                      ids, n_slots, S, I, O, st);
        case QG_FMT_MQ4V1:
            return run_gemv_moe_mq4v1(y, static_cast<const uint16_t *>(x), x_slot_stride, experts, n_experts,
                                      ids, n_slots, S, I, O, st);
        default:
            return run_gemv_moe_mq4c(y, static_cast<const uint16_t *>(x), x_slot_stride, experts, n_experts,
                                     ids, n_slots, S, I, O, st);
    }
}

}  // extern "C"

namespace {

typedef int (*Mq4GemvFn)(float *, const uint16_t *, const uint8_t *, int, int, int, void *, size_t, cudaStream_t);
typedef int (*Mq4GemmTcFn)(float *, const uint16_t *, const uint8_t *, int, int, int, void *, size_t,
                           cudaStream_t, bool *);
typedef int (*Mq4GemmGenFn)(float *, const uint16_t *, const uint8_t *, int, int, int, cudaStream_t);

// Checks shared by the three 136-byte MQ4 formats (the same block geometry).
int check_mq4(const char *fn, const char *sname, int S, int I, int O, const void *y, const void *x,
              const void *blocks, const void *ws) {
    int rc = check_dims(fn, sname, S, I, O);
    if (rc) return rc;
    if (I % 256) QG_REFUSE(kEShape, "%s: I = %d is not a multiple of 256", fn, I);
    if (!y || !x || !blocks) QG_REFUSE(kEInval, "%s: output, activations and blocks must be non-NULL", fn);
    if (!aligned(y, 4) || !aligned(x, 2) || !aligned(blocks, 8))
        QG_REFUSE(kEAlign, "%s: the output must be 4-byte, the activations 2-byte and blocks 8-byte aligned", fn);
    if (ws && !aligned(ws, 256)) QG_REFUSE(kEAlign, "%s: workspace must be 256-byte aligned", fn);
    return kOk;
}

int mq4_gemv(const char *fn, Mq4GemvFn run, float *y, const uint16_t *x, const uint8_t *blocks, int S, int I,
             int O, void *ws, size_t ws_bytes, qg_stream_t stream) {
    const int rc = check_mq4(fn, "S", S, I, O, y, x, blocks, ws);
    if (rc) return rc;
    cudaGetLastError();
    return run(y, x, blocks, S, I, O, ws, ws_bytes, as_stream(stream));
}

int mq4_gemm(const char *fn, Mq4GemmTcFn tc, Mq4GemmGenFn gen, float *Y, const uint16_t *X,
             const uint8_t *blocks, int M, int I, int O, void *ws, size_t ws_bytes, qg_stream_t stream) {
    int rc = check_mq4(fn, "M", M, I, O, Y, X, blocks, ws);
    if (rc) return rc;
    cudaGetLastError();
    bool taken = false;
    rc = tc(Y, X, blocks, M, I, O, ws, ws_bytes, as_stream(stream), &taken);
    if (taken) return rc;
    return gen(Y, X, blocks, M, I, O, as_stream(stream));
}

}  // namespace

extern "C" {

int qgemv_mq4v2(float *y, const uint16_t *x, const uint8_t *blocks, int S, int I, int O, void *ws,
                size_t ws_bytes, qg_stream_t stream) {
    return mq4_gemv("qgemv_mq4v2", run_gemv_mq4v2, y, x, blocks, S, I, O, ws, ws_bytes, stream);
}

int qgemv_mq4v1(float *y, const uint16_t *x, const uint8_t *blocks, int S, int I, int O, void *ws,
                size_t ws_bytes, qg_stream_t stream) {
    return mq4_gemv("qgemv_mq4v1", run_gemv_mq4v1, y, x, blocks, S, I, O, ws, ws_bytes, stream);
}

int qgemv_mq4c(float *y, const uint16_t *x, const uint8_t *blocks, int S, int I, int O, void *ws,
               size_t ws_bytes, qg_stream_t stream) {
    return mq4_gemv("qgemv_mq4c", run_gemv_mq4c, y, x, blocks, S, I, O, ws, ws_bytes, stream);
}

int qgemm_i4g(float *Y, const uint16_t *X, const uint8_t *w, const float *scales, int M, int I, int O, int gs,
              void *ws, size_t ws_bytes, qg_stream_t stream) {
    const char *fn = "qgemm_i4g";
    int rc = check_dims(fn, "M", M, I, O);
    if (rc) return rc;
    if ((rc = check_gs(fn, gs))) return rc;
    if (!Y || !X || !w || !scales) QG_REFUSE(kEInval, "%s: Y, X, w and scales must be non-NULL", fn);
    if (!aligned(Y, 4) || !aligned(X, 2) || !aligned(scales, 4))
        QG_REFUSE(kEAlign, "%s: Y and scales must be 4-byte and X 2-byte aligned", fn);
    if (ws && !aligned(ws, 256)) QG_REFUSE(kEAlign, "%s: workspace must be 256-byte aligned", fn);
    cudaGetLastError();
    bool taken = false;
    rc = run_gemm_i4g_tc(Y, X, w, scales, M, I, O, gs, ws, ws_bytes, as_stream(stream), &taken);
    if (taken) return rc;
    return run_gemm_i4g_general(Y, X, w, scales, M, I, O, gs, as_stream(stream));
}

int qgemm_fp8b128(float *Y, const uint16_t *X, const uint8_t *w, const float *scale_inv, int M, int I, int O,
                  void *ws, size_t ws_bytes, qg_stream_t stream) {
    const char *fn = "qgemm_fp8b128";
    int rc = check_dims(fn, "M", M, I, O);
    if (rc) return rc;
    if (!Y || !X || !w || !scale_inv) QG_REFUSE(kEInval, "%s: Y, X, w and scale_inv must be non-NULL", fn);
    if (!aligned(Y, 4) || !aligned(X, 2) || !aligned(scale_inv, 4))
        QG_REFUSE(kEAlign, "%s: Y and scale_inv must be 4-byte and X 2-byte aligned", fn);
    if (ws && !aligned(ws, 256)) QG_REFUSE(kEAlign, "%s: workspace must be 256-byte aligned", fn);
    cudaGetLastError();
    bool taken = false;
    rc = run_gemm_fp8b128_tc(Y, X, w, scale_inv, M, I, O, ws, ws_bytes, as_stream(stream), &taken);
    if (taken) return rc;
    return run_gemm_fp8b128_general(Y, X, w, scale_inv, M, I, O, as_stream(stream));
}

int qgemm_fp8ue8m0(float *Y, const uint16_t *X, const uint8_t *w, const uint8_t *scale_e8m0, int M, int I, int O,
                   void *ws, size_t ws_bytes, qg_stream_t stream) {
    const char *fn = "qgemm_fp8ue8m0";
    int rc = check_dims(fn, "M", M, I, O);
    if (rc) return rc;
    if (!Y || !X || !w || !scale_e8m0) QG_REFUSE(kEInval, "%s: Y, X, w and scale_e8m0 must be non-NULL", fn);
    if (!aligned(Y, 4) || !aligned(X, 2)) QG_REFUSE(kEAlign, "%s: Y must be 4-byte and X 2-byte aligned", fn);
    if (ws && !aligned(ws, 256)) QG_REFUSE(kEAlign, "%s: workspace must be 256-byte aligned", fn);
    cudaGetLastError();
    bool taken = false;
    rc = run_gemm_fp8ue8m0_tc(Y, X, w, scale_e8m0, M, I, O, ws, ws_bytes, as_stream(stream), &taken);
    if (taken) return rc;
    return run_gemm_fp8ue8m0_general(Y, X, w, scale_e8m0, M, I, O, as_stream(stream));
}

int qgemm_mq4v2(float *Y, const uint16_t *X, const uint8_t *blocks, int M, int I, int O, void *ws,
                size_t ws_bytes, qg_stream_t stream) {
    return mq4_gemm("qgemm_mq4v2", run_gemm_mq4v2_tc, run_gemm_mq4v2_general, Y, X, blocks, M, I, O, ws,
                    ws_bytes, stream);
}

int qgemm_mq4v1(float *Y, const uint16_t *X, const uint8_t *blocks, int M, int I, int O, void *ws,
                size_t ws_bytes, qg_stream_t stream) {
    return mq4_gemm("qgemm_mq4v1", run_gemm_mq4v1_tc, run_gemm_mq4v1_general, Y, X, blocks, M, I, O, ws,
                    ws_bytes, stream);
}

int qgemm_mq4c(float *Y, const uint16_t *X, const uint8_t *blocks, int M, int I, int O, void *ws,
               size_t ws_bytes, qg_stream_t stream) {
    return mq4_gemm("qgemm_mq4c", run_gemm_mq4c_tc, run_gemm_mq4c_general, Y, X, blocks, M, I, O, ws,
                    ws_bytes, stream);
}

int qg_quantize_i4g(uint8_t *wq, float *scales, const float *w, int O, int I, int gs, qg_stream_t stream) {
    const char *fn = "qg_quantize_i4g";
    int rc = check_dims(fn, "O", 1, I, O);
    if (rc) return rc;
    if ((rc = check_gs(fn, gs))) return rc;
    if (!wq || !scales || !w) QG_REFUSE(kEInval, "%s: wq, scales and w must be non-NULL", fn);
    if (!aligned(scales, 4) || !aligned(w, 4)) QG_REFUSE(kEAlign, "%s: scales and w must be 4-byte aligned", fn);
    cudaGetLastError();
    return run_quantize_i4g(wq, scales, w, O, I, gs, as_stream(stream));
}

int qg_encode_mq4v2(uint8_t *blocks, const float *w, int O, int I, qg_stream_t stream) {
    const char *fn = "qg_encode_mq4v2";
    int rc = check_dims(fn, "O", 1, I, O);
    if (rc) return rc;
    if (I % 256) QG_REFUSE(kEShape, "%s: I = %d is not a multiple of 256", fn, I);
    if (!blocks || !w) QG_REFUSE(kEInval, "%s: blocks and w must be non-NULL", fn);
    if (!aligned(w, 4) || !aligned(blocks, 8))
        QG_REFUSE(kEAlign, "%s: w must be 4-byte and blocks 8-byte aligned", fn);
    cudaGetLastError();
    return run_encode_mq4v2(blocks, w, O, I, as_stream(stream));
}

static int encode_mq4_one_header(const char *fn, uint8_t *blocks, const float *w, int O, int I, bool fp16,
                                 qg_stream_t stream) {
    int rc = check_dims(fn, "O", 1, I, O);
    if (rc) return rc;
    if (I % 256) QG_REFUSE(kEShape, "%s: I = %d is not a multiple of 256", fn, I);
    if (!blocks || !w) QG_REFUSE(kEInval, "%s: blocks and w must be non-NULL", fn);
    if (!aligned(w, 4) || !aligned(blocks, 8))
        QG_REFUSE(kEAlign, "%s: w must be 4-byte and blocks 8-byte aligned", fn);
    cudaGetLastError();
    return run_encode_mq4_one_header(blocks, w, O, I, fp16, as_stream(stream));
}

int qg_encode_mq4v1(uint8_t *blocks, const float *w, int O, int I, qg_stream_t stream) {
    return encode_mq4_one_header("qg_encode_mq4v1", blocks, w, O, I, false, stream);
}

int qg_encode_mq4c(uint8_t *blocks, const float *w, int O, int I, qg_stream_t stream) {
    return encode_mq4_one_header("qg_encode_mq4c", blocks, w, O, I, true, stream);
}

int qg_fwht256(float *out, const float *in, const int8_t *signs, size_t n_blocks, qg_stream_t stream) {
    const char *fn = "qg_fwht256";
    if (n_blocks < 1) QG_REFUSE(kEInval, "%s: n_blocks must be >= 1", fn);
    if (n_blocks > ((size_t)1 << 40)) QG_REFUSE(kEInval, "%s: n_blocks too large", fn);
    if (!out || !in || !signs) QG_REFUSE(kEInval, "%s: out, in and signs must be non-NULL", fn);
    if (!aligned(out, 4) || !aligned(in, 4)) QG_REFUSE(kEAlign, "%s: out and in must be 4-byte aligned", fn);
    cudaGetLastError();
    return run_fwht256(out, in, signs, n_blocks, as_stream(stream));
}

}  // extern "C"

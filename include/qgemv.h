/*
 * qgemv.h -- C ABI of libqgemv: dequantize-fused weight-only quantized GEMV
 * (decode, a handful of tokens) and dequant-GEMM (batched prefill) for three
 * packed weight formats, on one NVIDIA GB300 (sm_103a).
 *
 * Sources of each format's definition (page title, section):
 *   fmt=4  grouped int4     colibri PR #457 "metal: grouped-int4 (fmt=4) GEMV
 *                           support + two latent fmt=4 fixes", sections 3, 4, 11
 *   fmt=7  FP8-e4m3 b128    colibri PR #528 "fmt=7: fp8-e4m3-b128 passthrough
 *                           weight format", section "Design"
 *   MQ4-V2 (qt=44)          hipfire docs "MQ4 V2", sections 2, 3, 4
 *   MQ4 v1 (qt=13),         hipfire docs "MQ4 V2", sections 1b, 1c, 1e
 *   MQ4C pad (qt=45)
 *   Q2_0                    strata review, "convert_k256_q2_0.cpp vs
 *                           ref_quant.cpp" (2.5)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All data pointers are DEVICE pointers owned by the caller.  The library
 *   allocates no device memory and never frees anything.  Its only state is
 *   one 4-byte error word per device (see qg_device_status; in the stamps
 *   build, libqgemv_stamps.so, followed by the timeline stamps of
 *   qg_stamps_take) and host-side per-device caches (SM count, that word's
 *   address, kernel attributes).
 * - Calls are asynchronous on `stream` (0 = legacy default stream).  No call
 *   synchronises the host.  Outputs are fully overwritten, never accumulated.
 * - A call's kernels may start while the previous kernel on `stream` is still
 *   running (programmatic dependent launch) and stream the weights, scales
 *   and the expert table's matrices into shared memory before they wait for
 *   it; activations, routing ids and workspace are read, and outputs
 *   written, only after that kernel has completed.  So weights that a kernel
 *   writes (qg_encode_* included) must not come from the kernel just before
 *   the call on `stream`: put another kernel, an event wait or a host
 *   synchronisation between them.
 * - Activations x are row-major [S, I]; outputs y are row-major f32 [S, O]
 *   (y[s*O + o]).  bf16 activations are passed as their raw 16-bit patterns.
 * - Every argument is validated on the host BEFORE any pointer is touched or
 *   any kernel is launched.  A refused call returns a negative qg_status and
 *   launches nothing; qg_last_error() names the failed condition.  There is
 *   no CPU fallback and no silent format conversion: a shape or alignment the
 *   fast kernels cannot take runs a general (slower) kernel of the same
 *   format, which is still exact to the same tolerance.
 * - Accumulation is f32.  Results match the exact (f64) value of the
 *   definition within 1e-3 * sum_i |w_i * x_i| per output element; NaN
 *   weights or activations propagate to their output element.
 * - Workspace: a call that splits the reduction dimension across thread
 *   blocks needs a caller-provided scratch buffer of qg_workspace_bytes()
 *   bytes (256-byte aligned).  When that function returns 0, ws may be NULL.
 *   Passing a smaller workspace than required returns QG_EWORKSPACE.
 *   Two calls in flight at the same time must not share a workspace.
 */
#ifndef QGEMV_H
#define QGEMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so that this header does not
 * require the CUDA headers. */
typedef struct CUstream_st *qg_stream_t;

typedef enum {
    QG_OK = 0,
    QG_EINVAL = -1,      /* NULL pointer, S/M/I/O < 1, or a size overflows  */
    QG_EGS = -2,         /* fmt=4 group size odd or < 2                      */
    QG_ESHAPE = -3,      /* MQ4-V2 with I % 256 != 0                         */
    QG_EALIGN = -4,      /* pointer misaligned for its element type          */
    QG_EWORKSPACE = -5,  /* workspace NULL or smaller than required          */
    QG_ECUDA = -6,       /* CUDA runtime error (no device, launch failure)   */
    QG_ETIMEOUT = -7,    /* a kernel gave up waiting (see qg_device_status)  */
    QG_EEXPERT = -8,     /* qgemv_moe: a slot's expert id was out of range   */
                         /* or its weights misaligned (qg_device_status)     */
    QG_EBOUNDS = -9      /* bounds-checking build only: a kernel formed an   */
                         /* index outside its arrays and skipped the access  */
                         /* (qg_device_status; never raised by libqgemv.so)  */
} qg_status;

/* Static name of a status code ("QG_EGS: ..."). Never NULL. */
const char *qg_strerror(int status);

/* Detail of the last refusal or CUDA error on the calling host thread
 * (which argument, which condition, or the CUDA error string).  The pointer
 * stays valid until the next call on the same thread. */
const char *qg_last_error(void);

/* Kernel-side status of the current device.  Kernels that stage weights
 * through shared memory wait on hardware barriers; every such wait is bounded
 * and, if it ever gives up (which no valid call does), the kernel stops early
 * and records QG_ETIMEOUT in a per-device error word instead of hanging the
 * GPU.  qgemv_moe records QG_EEXPERT there for a slot whose expert it cannot
 * read (its arguments live in device memory, out of the host's reach).  This call synchronizes the device, stores that word (QG_OK when
 * clean) in *status and clears it.  Returns QG_OK, QG_EINVAL for a NULL
 * status, or QG_ECUDA. */
int qg_device_status(int *status);

/* Number of kernels this library has launched in this process, over all
 * devices and threads (every entry point counts the launches it enqueues:
 * one per GEMV, plus one for a split reduction's summing pass; two per
 * tensor-core GEMM).  For profiling and launch accounting; the pages have no
 * counterpart.  Never fails. */
unsigned long long qg_launch_count(void);

/* Test aid for the failure path above (no counterpart in the pages, whose
 * fp8 page asks that failures be loud and every refusal name its condition).
 * Runs one block of the staging pipeline on the current device in which a
 * consumer waits for a batch that is never issued: its bounded wait gives up
 * after spin_limit polls (1 .. 4194304, the kernels' own limit) instead of
 * 4194304, records QG_ETIMEOUT in the device error word and ends the other
 * wait of the block, whose producer first lands the copy it issued.
 * Synchronizes the device; *observed receives what the block saw (bit 0: the
 * consumer gave up on the missing batch; bit 1: the producer's wait ended on
 * the block's abort flag; bit 2: the issued copy landed before the block
 * exited), and the error word is left for qg_device_status to read.
 * Nothing faults and the context stays usable.  Returns QG_OK, QG_EINVAL
 * (NULL observed or spin_limit out of range) or QG_ECUDA. */
int qg_selftest_wait_timeout(int spin_limit, int *observed);

/* Profiling aids (no counterpart in the pages).
 *
 * qg_stamps_take: in the stamps build of this library (libqgemv_stamps.so,
 * built with `_build.py --stamps`), every block of a staged or warp-MMA
 * decode GEMV records its timeline: 8 words per block b (b < 2048, b =
 * blockIdx.x + gridDim.x * blockIdx.y), in order the SM clock (clock64) at
 * the block's start, when its wait for the previous kernel on the stream
 * returned, when its activations were ready, when its first row batch had
 * landed (warp-MMA kernel: after the activation setup), when its consumers
 * had finished its last batch and when its last output was stored; then the
 * number of row batches it ran and the global timer (ns) at its start.
 * Later calls overwrite earlier ones block by block.  Synchronizes the
 * device, copies min(max_blocks, 2048) blocks' words to `host` (8 uint64 per
 * block) and zeroes them on the device.  Returns QG_OK, QG_EINVAL (NULL host,
 * max_blocks < 1, or a library built without stamps) or QG_ECUDA.
 *
 * qg_selftest_pdl_chain: enqueues `launches` launches (1 .. 100000) of an
 * empty kernel of `blocks` x `threads` threads (1 .. 65535, 32 .. 1024 and a
 * multiple of 32) on `stream` with programmatic stream serialization, the
 * launch mode of every GEMV here; each launch lets the next start early,
 * waits for the previous one and adds one to a device word.  Its time per
 * launch is the floor under any of these kernels that waits for its
 * predecessor.  Returns QG_OK, QG_EINVAL or QG_ECUDA; asynchronous. */
int qg_stamps_take(uint64_t *host, int max_blocks);
int qg_selftest_pdl_chain(int blocks, int threads, int launches, qg_stream_t stream);

/* Format ids for qg_workspace_bytes. */
enum {
    QG_FMT_I4G = 4,         /* grouped int4 (fmt=4)                            */
    QG_FMT_FP8B128 = 7,     /* FP8-e4m3, 128x128 f32 block scales (fmt=7)      */
    QG_FMT_FP8UE8M0 = 71,   /* FP8-e4m3, 128x128 UE8M0 block scales (fmt=7 with */
                            /* the page's second scale encoding; a library id) */
    QG_FMT_MQ4V1 = 13,      /* MQ4 v1 (qt=13)                                  */
    QG_FMT_MQ4V2 = 44,      /* MQ4-V2 (qt=44)                                  */
    QG_FMT_MQ4C = 45,       /* MQ4C pad (qt=45)                                */
    QG_FMT_Q2_0 = 20        /* Q2_0 codec, 2.25 bits per weight (a library id) */
};

/* Bytes of workspace that the GEMV entry point of format `fmt` needs for
 * this shape on the current device (0 when the call does not split the
 * reduction).  Returns 0 for invalid arguments (the call itself then
 * refuses).  `gs` is only read for fmt=4. */
size_t qg_workspace_bytes(int fmt, int S, int I, int O, int gs);

/* Bytes of workspace that the batched-prefill GEMM entry point of format
 * `fmt` (qgemm_i4g, qgemm_fp8b128, qgemm_mq4v2) needs for an M x I x O call
 * on the current device: the fp16 copy of X (2*M*I bytes), one exponent per
 * token row and per weight row, tile counters, and, when tiles' K ranges
 * are shared by several blocks, two f32 partial-sum slots of up to
 * 128 x 256 per thread block.  0 when the shape runs the general kernel (no
 * workspace) or the arguments are invalid.  `gs` is only read for fmt=4. */
size_t qg_gemm_workspace_bytes(int fmt, int M, int I, int O, int gs);

/* ------------------------------------------------------------------------ */
/* fmt=4 grouped int4, decode GEMV                                          */
/* colibri PR #457, section 3 (per-group scale folded into the sum) and     */
/* section 11 (packed layout shared with the CUDA tier).                    */
/*                                                                          */
/*   w      uint8 [O, (I+1)/2]: element i of row o is in byte i/2 of the    */
/*          row, low nibble for even i, high nibble for odd i; the stored   */
/*          nibble n means the integer n - 8.  For odd I the last high      */
/*          nibble of each row is never read.                               */
/*   scales f32 [O, ceil(I/gs)]: element i uses scales[o*ceil(I/gs) + i/gs] */
/*   x      f32 [S, I]                                                      */
/*   y      f32 [S, O]:  y[s,o] = sum_i (n(o,i) - 8) * scales[o, i/gs] * x[s,i] */
/*   gs     any even group size >= 2 (16..256 are the loader's values)      */
/*   S      any >= 1 (the weights are streamed once per group of up to 8    */
/*          activation rows)                                                */
/* Alignment: x, y, scales 4-byte aligned.  The fastest path also wants     */
/* w and x 16-byte aligned, I % 32 == 0 and gs % 32 == 0.                   */
/* ------------------------------------------------------------------------ */
int qgemv_i4g(float *y, const float *x, const uint8_t *w, const float *scales,
              int S, int I, int O, int gs, void *ws, size_t ws_bytes, qg_stream_t stream);

/* qgemv_i4g for callers that cannot allocate device memory.  The pages have
 * no counterpart: this is a library convenience.  Same arguments, layout,
 * results and errors as qgemv_i4g, minus the workspace: a shape whose
 * reduction is split across thread blocks takes its scratch from a fixed
 * 4 MiB array inside the library instead of a caller buffer.  Meant for
 * engines whose device memory is planned once at start-up by their own
 * allocator, and for host code that must not call cudaMalloc on the decode
 * path (it can wait for the whole device).  Shapes needing more than 4 MiB
 * of scratch (qg_workspace_bytes(QG_FMT_I4G, ...) > 4 MiB) are refused with
 * QG_EWORKSPACE.  The first call in a CUDA context (the device's primary
 * context, a new one after cudaDeviceReset, or a driver-API context of the
 * caller's) looks up the array's device address there
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * Every call on a device shares the array and leaves its contents
 * behind; calls whose kernels may run at the same time (different streams or
 * host threads) race on it and must be ordered by the caller.  Allocates
 * nothing; every GPU that loads the library holds the 4 MiB until exit. */
int qgemv_i4g_noalloc(float *y, const float *x, const uint8_t *w, const float *scales,
                      int S, int I, int O, int gs, qg_stream_t stream);

/* ------------------------------------------------------------------------ */
/* fmt=7 FP8-e4m3 with 128x128 block scales, decode GEMV                    */
/* colibri PR #528, section "Design".                                       */
/*                                                                          */
/*   w         uint8 [O, I]: raw OCP E4M3-FN codes (bias 7; the only NaN    */
/*             codes are 0x7F and 0xFF; no infinities; subnormals valid)    */
/*   scale_inv f32 [ceil(O/128), ceil(I/128)], row-major block order:       */
/*             W[o,i] = e4m3(w[o*I+i]) * scale_inv[(o/128)*ceil(I/128) + i/128] */
/*             (multiply, not divide; partial edge blocks indexed the same) */
/*   x         bf16 bits [S, I]                                             */
/*   y         f32 [S, O] = x . W^T; a NaN weight makes its row NaN         */
/* Alignment: x 2-byte, y and scale_inv 4-byte aligned.  The fastest path   */
/* also wants w and x 16-byte aligned and I % 16 == 0.                      */
/* ------------------------------------------------------------------------ */
int qgemv_fp8b128(float *y, const uint16_t *x, const uint8_t *w, const float *scale_inv,
                  int S, int I, int O, void *ws, size_t ws_bytes, qg_stream_t stream);

/* ------------------------------------------------------------------------ */
/* fmt=7 with UE8M0 block scales, decode GEMV                               */
/* colibri PR #528, section "Design": the scale encoding is a property of   */
/* the format; DeepSeek-V4 ships the same e4m3 weight geometry with UE8M0   */
/* scales, one byte per 128x128 block holding a power-of-two exponent.      */
/*                                                                          */
/*   w           e4m3 [O, I] as for qgemv_fp8b128                           */
/*   scale_e8m0  uint8 [ceil(O/128), ceil(I/128)]: byte e means 2^(e - 127) */
/*               (OCP MX E8M0; e = 255 is NaN and poisons its block)        */
/*   y[s,o] = sum_i e4m3(w[o,i]) * 2^(scale_e8m0[o/128, i/128] - 127) * x[s,i] */
/* Everything else (x, y, workspace, alignment, paths) as qgemv_fp8b128,    */
/* except that scale_e8m0 needs no alignment.                               */
/* ------------------------------------------------------------------------ */
int qgemv_fp8ue8m0(float *y, const uint16_t *x, const uint8_t *w, const uint8_t *scale_e8m0,
                   int S, int I, int O, void *ws, size_t ws_bytes, qg_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Q2_0 codec, decode GEMV                                                  */
/* strata review, "convert_k256_q2_0.cpp vs ref_quant.cpp" (2.5): the ggml  */
/* Q2_0 layout of the routed experts it checks.                             */
/*                                                                          */
/*   blocks  uint8 [O, I/64 * 18]: each 64-weight block is an fp16 d (bytes  */
/*           0-1, little-endian) and 16 bytes of 2-bit codes; weight e of   */
/*           the block sits in byte 2 + e/4 at bit 2*(e%4)                  */
/*   x       bf16 [S, I];  y  f32 [S, O]                                    */
/*   y[s,o] = sum_i (code(o,i) - 1) * d(o, i/64) * x[s,i]                    */
/*   I       multiple of 64 (else QG_ESHAPE); S any >= 1                     */
/* Alignment: y 4-byte, x and blocks 2-byte.  Workspace: qg_workspace_bytes */
/* (QG_FMT_Q2_0, ...) when the row is split across thread blocks.           */
/* ------------------------------------------------------------------------ */
int qgemv_q2_0(float *y, const uint16_t *x, const uint8_t *blocks, int S, int I, int O,
               void *ws, size_t ws_bytes, qg_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Routed experts: many decode GEMVs of one format and shape in one launch  */
/* colibri PR #457, section 7 (fmt=4 is mostly an expert format; the        */
/* batched routed-expert path takes a per-expert pointer array and one      */
/* format and group size per tensor) and hipfire docs "MQ4 V2", section 9   */
/* (MoE decode on MQ4-V2).                                                  */
/*                                                                          */
/*   experts  DEVICE array [n_experts] of qg_expert: each expert's packed   */
/*            weights `w` and, for fmt=4 and fmt=7, its `scales` (NULL for  */
/*            the MQ4 formats), laid out exactly as the single-matrix entry */
/*            point of `fmt` takes them, all experts with the same O x I    */
/*            (and gs for fmt=4)                                            */
/*   ids      DEVICE int32 [n_slots]: slot r uses expert ids[r]; the same   */
/*            expert may appear in several slots                            */
/*   x        DEVICE [n_slots or 1][S, I] activations, f32 for fmt=4 and    */
/*            bf16 otherwise: slot r reads x + r * x_slot_stride (elements; */
/*            0 = every slot reads the same x, e.g. gate and up projections */
/*            of one token)                                                 */
/*   y        DEVICE f32 [n_slots][S, O]: y[r][s][o] = sum_i                */
/*            W_{ids[r]}[o, i] * x_r[s, i] with the format's dequantization */
/*   fmt      QG_FMT_I4G, QG_FMT_FP8B128, QG_FMT_FP8UE8M0 (scales are then  */
/*            the UE8M0 bytes), QG_FMT_MQ4V2, QG_FMT_MQ4V1 or QG_FMT_MQ4C;  */
/*            gs is read for fmt=4 only                                     */
/*   S        tokens per slot, 1..8 (decode)                                */
/* experts and ids may be written by earlier kernels on `stream` (a        */
/* router): the kernel reads them after those kernels finish.  n_slots = 0 */
/* returns QG_OK and launches nothing.  Needs x 16-byte aligned (and        */
/* x_slot_stride a whole number of 16-byte lines), each expert's w 16-byte */
/* aligned (fmt=4 scales too; fmt=7 f32 scales 4-byte), and rows short enough */
/* for one thread block (fmt=4: I % 32 == 0, gs % 32 == 0, ceil(I/gs) % 4  */
/* == 0; fmt=7: I % 16 == 0; MQ4: I/256 even), else QG_ESHAPE / QG_EALIGN. */
/* A slot whose id is outside [0, n_experts) or whose expert pointers are  */
/* NULL or misaligned is not computed: its outputs are set to NaN and the   */
/* device error word records QG_EEXPERT (see qg_device_status).  No        */
/* workspace.                                                               */
/* ------------------------------------------------------------------------ */
typedef struct {
    const void *w;
    const float *scales;
} qg_expert;

int qgemv_moe(int fmt, float *y, const void *x, size_t x_slot_stride,
              const qg_expert *experts, int n_experts, const int *ids, int n_slots,
              int S, int I, int O, int gs, qg_stream_t stream);

/* Routed experts, batched prefill: the tokens of a prompt sorted by routed
 * expert (colibri PR #457, section 7; hipfire docs "MQ4 V2", section 9: the
 * grouped MoE prefill).  Group g multiplies rows [group_offsets[g],
 * group_offsets[g+1]) of X by expert experts[group_expert[g]] into the same
 * rows of Y, each group as one call of the format's prefill GEMM (qgemm_i4g,
 * qgemm_fp8b128, qgemm_fp8ue8m0, qgemm_mq4v2, qgemm_mq4v1, qgemm_mq4c; same
 * layouts, precision and paths), one after another on `stream`.
 *   experts        HOST array [n_experts] of qg_expert (device pointers)
 *   group_expert   HOST int32 [n_groups], each in [0, n_experts)
 *   group_offsets  HOST int32 [n_groups + 1], non-decreasing, >= 0 (a group
 *                  may be empty; rows outside every group are not written)
 *   X, Y           DEVICE bf16 [M, I] and f32 [M, O], M >= group_offsets[n_groups]
 *   ws             qg_moe_gemm_workspace_bytes(fmt, group_offsets, n_groups,
 *                  I, O, gs) bytes, 256-byte aligned
 * Up to 64 non-empty groups run as ONE tensor-core launch (every group's
 * token blocks times the output tiles form one range of tiles, each tile
 * dequantizing its group's weights); a chunk whose shapes or pointers the
 * tensor-core kernel cannot take runs group by group through the format's
 * GEMM entry point instead.  The group sizes decide the launches, so they
 * are host data here (a router's counts are read back once per prompt).
 * Errors: QG_EINVAL for a bad format, group table or size; QG_EGS /
 * QG_ESHAPE as the format's GEMM; QG_EWORKSPACE; otherwise the first failing
 * group's status from its GEMM (qg_last_error names it). */
/* Workspace of qgemm_moe for these groups (host group_offsets [n_groups+1]);
 * 0 for invalid arguments. */
size_t qg_moe_gemm_workspace_bytes(int fmt, const int *group_offsets, int n_groups, int I, int O, int gs);

int qgemm_moe(int fmt, float *Y, const uint16_t *X, const qg_expert *experts, int n_experts,
              const int *group_expert, const int *group_offsets, int n_groups,
              int I, int O, int gs, void *ws, size_t ws_bytes, qg_stream_t stream);

/* ------------------------------------------------------------------------ */
/* MQ4-V2 (hipfire qt=44), decode GEMV                                      */
/* hipfire "MQ4 V2", section 2 (layout) and section 4 (decoder).            */
/*                                                                          */
/*   blocks uint8 [O, I/256, 136]: per 256 weights, little-endian           */
/*          [0,4)   fp16 scale (low 16 bits) and fp16 zero (high 16 bits)   */
/*                  of weights 0..127                                       */
/*          [4,8)   the same for weights 128..255                           */
/*          [8,136) nibbles: weight j in payload byte j/2, low nibble for   */
/*                  even j                                                  */
/*          w_j = q_j * scale[h] + zero[h], h = (j >= 128)                  */
/*   x      bf16 bits [S, I];  y f32 [S, O]                                 */
/*   I      multiple of 256 (else QG_ESHAPE)                                */
/* Alignment: blocks 8-byte, x 2-byte, y 4-byte aligned.  The fastest path  */
/* also wants x 16-byte aligned.                                            */
/* ------------------------------------------------------------------------ */
int qgemv_mq4v2(float *y, const uint16_t *x, const uint8_t *blocks,
                int S, int I, int O, void *ws, size_t ws_bytes, qg_stream_t stream);

/* ------------------------------------------------------------------------ */
/* MQ4 v1 (hipfire qt=13) and MQ4C pad (hipfire qt=45), decode GEMV        */
/* hipfire "MQ4 V2", sections 1b and 1e: the MQ4-V2 block geometry (136 B  */
/* per 256 weights, nibbles at [8,136), weight j in payload byte j/2, low   */
/* nibble for even j) with ONE header for all 256 weights of the block:     */
/*   qgemv_mq4v1: [0,4) f32 scale, [4,8) f32 zero                           */
/*   qgemv_mq4c:  [0,2) fp16 scale, [2,4) fp16 zero, [4,8) zero bytes       */
/*   w_j = q_j * scale + zero.  Arguments, alignment, workspace            */
/*   (qg_workspace_bytes with QG_FMT_MQ4V1 / QG_FMT_MQ4C), errors and      */
/*   precision exactly as qgemv_mq4v2.                                      */
/* ------------------------------------------------------------------------ */
int qgemv_mq4v1(float *y, const uint16_t *x, const uint8_t *blocks,
                int S, int I, int O, void *ws, size_t ws_bytes, qg_stream_t stream);
int qgemv_mq4c(float *y, const uint16_t *x, const uint8_t *blocks,
               int S, int I, int O, void *ws, size_t ws_bytes, qg_stream_t stream);

/* ------------------------------------------------------------------------ */
/* fmt=4 batched prefill dequant-GEMM on the tensor cores                   */
/* colibri PR #457, section 4 (the large-batch GEMM path takes the same     */
/* grouped layout as the GEMV).                                             */
/*                                                                          */
/*   Y[M, O] f32 = X[M, I] (bf16 bits) . W^T, W as in qgemv_i4g.  The      */
/*   tensor-core path contracts fp16 operands with f32 accumulation: each   */
/*   weight (n-8)*scale is formed in f32 and rounded to 11 significant bits */
/*   (nearest even), X is exact; powers of two per weight row and per token */
/*   row keep both in fp16's range and are undone exactly at the store.     */
/*   Every output is within 2^-11 (plus f32 summation error) of             */
/*   sum_i |w_i x_i|, for elements of X within 2^29 of their row's largest  */
/*   finite |x| and weights within 2^29 of their row's bound                */
/*   (8 max_g |scale_g|).                                                   */
/*   Any M >= 1.  The tensor-core path takes I % 64 == 0, gs % 32 == 0 and  */
/*   16-byte aligned X and w, and needs a 256-byte aligned workspace of     */
/*   qg_gemm_workspace_bytes(QG_FMT_I4G, M, I, O, gs) bytes (QG_EWORKSPACE  */
/*   otherwise: it holds the fp16 copy of X, 2*M*I bytes, plus per-row      */
/*   exponents and the split-tile scratch); other shapes run a general      */
/*   CUDA-core kernel with f32 weights and ignore ws.                       */
/*   The work is split evenly over one thread block per SM; a tile shared   */
/*   by several blocks is summed in a fixed order, so repeated calls give   */
/*   identical results.                                                     */
/* ------------------------------------------------------------------------ */
int qgemm_i4g(float *Y, const uint16_t *X, const uint8_t *w, const float *scales,
              int M, int I, int O, int gs, void *ws, size_t ws_bytes, qg_stream_t stream);

/* ------------------------------------------------------------------------ */
/* fmt=7 batched prefill dequant-GEMM on the tensor cores                   */
/* colibri PR #528, section "Design" (the same block-scaled product as the  */
/* GEMV, over M tokens).                                                    */
/*                                                                          */
/*   Y[M, O] f32 = X[M, I] (bf16 bits) . W^T, w and scale_inv as in         */
/*   qgemv_fp8b128.  Each weight e4m3(code) * scale is formed in f32 and    */
/*   rounded to fp16 as in qgemm_i4g (row bound 448 max_k |scale_inv|).     */
/*   A NaN code makes its output column Y[:, o] NaN.                        */
/*   Any M >= 1.  The tensor-core path takes I % 64 == 0 and 16-byte        */
/*   aligned X and w, and needs a 256-byte aligned workspace of             */
/*   qg_gemm_workspace_bytes(QG_FMT_FP8B128, M, I, O, 0) bytes              */
/*   (QG_EWORKSPACE otherwise); other shapes run a general CUDA-core kernel */
/*   and ignore ws.  Deterministic like qgemm_i4g.                          */
/* ------------------------------------------------------------------------ */
int qgemm_fp8b128(float *Y, const uint16_t *X, const uint8_t *w, const float *scale_inv,
                  int M, int I, int O, void *ws, size_t ws_bytes, qg_stream_t stream);

/* qgemm_fp8b128 with UE8M0 block scales (the byte e means 2^(e - 127), see  */
/* qgemv_fp8ue8m0): same X, Y, workspace (qg_gemm_workspace_bytes with      */
/* QG_FMT_FP8UE8M0), paths, precision and errors as qgemm_fp8b128.          */
int qgemm_fp8ue8m0(float *Y, const uint16_t *X, const uint8_t *w, const uint8_t *scale_e8m0,
                   int M, int I, int O, void *ws, size_t ws_bytes, qg_stream_t stream);

/* ------------------------------------------------------------------------ */
/* MQ4-V2 batched prefill dequant-GEMM on the tensor cores                  */
/* hipfire "MQ4 V2", sections 2 and 4 (the same decoder as the GEMV, over   */
/* M tokens).                                                               */
/*                                                                          */
/*   Y[M, O] f32 = X[M, I] (bf16 bits) . W^T, blocks as in qgemv_mq4v2.     */
/*   Each weight q * scale + zero is formed in f32 with one rounding (fused */
/*   multiply-add) and rounded to fp16 as in qgemm_i4g (row bound           */
/*   max_h |zero_h| + 15 |scale_h|); f32 accumulation.                      */
/*   I % 256 == 0 (else QG_ESHAPE); blocks 8-byte, X 2-byte, Y 4-byte       */
/*   aligned.  A 16-byte aligned X takes the tensor-core path, which needs  */
/*   a 256-byte aligned workspace of                                        */
/*   qg_gemm_workspace_bytes(QG_FMT_MQ4V2, M, I, O, 0) bytes (QG_EWORKSPACE */
/*   otherwise); other X run a general CUDA-core kernel and ignore ws.      */
/*   Deterministic like qgemm_i4g.                                          */
/* ------------------------------------------------------------------------ */
int qgemm_mq4v2(float *Y, const uint16_t *X, const uint8_t *blocks,
                int M, int I, int O, void *ws, size_t ws_bytes, qg_stream_t stream);

/* ------------------------------------------------------------------------ */
/* MQ4 v1 and MQ4C pad batched prefill dequant-GEMM on the tensor cores     */
/* The same contract as qgemm_mq4v2 (fp16 operands with powers of two, the */
/* row bound max over the row's blocks of |zero| + 15 |scale|), with the     */
/* formats of qgemv_mq4v1 / qgemv_mq4c; workspace from                      */
/* qg_gemm_workspace_bytes with QG_FMT_MQ4V1 / QG_FMT_MQ4C.                 */
/* ------------------------------------------------------------------------ */
int qgemm_mq4v1(float *Y, const uint16_t *X, const uint8_t *blocks,
                int M, int I, int O, void *ws, size_t ws_bytes, qg_stream_t stream);
int qgemm_mq4c(float *Y, const uint16_t *X, const uint8_t *blocks,
               int M, int I, int O, void *ws, size_t ws_bytes, qg_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Weight preparation on the device (not on the decode path)                */
/* ------------------------------------------------------------------------ */

/* Symmetric per-group int4 quantizer producing fmt=4 (the reading used for
 * the grouped-int4 checkpoints): scale_g = max|w| / 7 (binary32 division),
 * q = clamp(rint(w / scale_g), -8, 7) stored as q + 8; an all-zero group
 * stores scale 0 and nibbles 8; for odd I the unused last high nibble is 8.
 *   w  f32 [O, I] (device);  wq uint8 [O, (I+1)/2];  scales f32 [O, ceil(I/gs)] */
int qg_quantize_i4g(uint8_t *wq, float *scales, const float *w, int O, int I, int gs,
                    qg_stream_t stream);

/* MQ4-V2 encoder, hipfire "MQ4 V2" section 3: per 128-weight half,
 * step = (max - min) / 15 in binary32, scale = fp16(step), zero = fp16(min),
 * q = clamp(rint((w - f32(zero)) / f32(scale)), 0, 15) against the
 * round-tripped header; a constant half (or one whose fp16 step rounds to 0)
 * stores scale 0 and q = 0.
 *   w f32 [O, I] (device, 4-byte aligned), I % 256 == 0;
 *   blocks uint8 [O, I/256, 136] (device, 8-byte aligned) */
int qg_encode_mq4v2(uint8_t *blocks, const float *w, int O, int I, qg_stream_t stream);

/* MQ4 v1 and MQ4C pad encoders: the MQ4 rule (levels uniform over the
 * block's [min, max], hipfire "MQ4 V2" section 1c) over each 256-weight
 * block: step = (max - min) / 15 in binary32; v1 stores scale = step and
 * zero = min as f32; pad stores fp16(step), fp16(min) and four zero bytes and
 * quantizes against the round-tripped values; q = clamp(rint((w - zero) /
 * scale), 0, 15); a constant block (or a zero stored step) stores scale 0
 * and q = 0.  Same arguments and errors as qg_encode_mq4v2. */
int qg_encode_mq4v1(uint8_t *blocks, const float *w, int O, int I, qg_stream_t stream);
int qg_encode_mq4c(uint8_t *blocks, const float *w, int O, int I, qg_stream_t stream);

/* Signed Walsh-Hadamard rotation of 256-element blocks (hipfire "MQ4 V2"
 * sections 1 and 3: the MQ line rotates weights and activations with the
 * same seeded sign-FWHT): out_b = H_256 (signs . in_b) / 16, H_256 the
 * Sylvester Hadamard matrix in natural order, signs int8 +-1 [256].
 *   in, out f32 [n_blocks, 256] (device; may alias) */
int qg_fwht256(float *out, const float *in, const int8_t *signs, size_t n_blocks,
               qg_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* QGEMV_H */

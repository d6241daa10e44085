/*
 * qoq.h -- C ABI of the GB300 (sm_103a) W4A8 GEMM library (libqoq.so).
 *
 * The library computes the hot path of the QoQ / QServe method: a GEMM whose
 * weights are 4-bit under progressive group quantization and whose
 * activations are 8-bit per-token, with an fp16 output:
 *
 *   O[m,n] = s_x[m] * s_w[n] * sum_k Qx[m,k] * (q4[n,k] - z[n,k/128]) * s_g[n,k/128]
 *
 * Page references (web pages on QServe / QoQ):
 *   [QS-summary] "QServe: W4A8KV4 Quantization and System Co-design for
 *                Efficient LLM Serving" (papercache.org summary).
 *   [QS-review]  "QServe：把 W4A8KV4 的理论收益做成实测吞吐的量化—系统协同设计"
 *                (zenmind.me review).
 *
 * Conventions for every entry point:
 *  - Every tensor pointer is DEVICE memory owned by the caller; the library
 *    never allocates, frees or synchronizes the device (except
 *    qoq_workspace_status and qoq_noalloc_status, which synchronize the
 *    given stream).
 *  - fp16 tensors are passed as uint16_t IEEE binary16 bit patterns.
 *  - Matrices are row-major and dense: X, Qx [M][K]; W, q4 [N][K]; O [M][N].
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and runs asynchronously.  Calls are stateless and thread-safe
 *    as long as concurrent GEMMs use distinct workspaces.
 *  - Arguments are validated before any launch; on a validation error
 *    nothing is enqueued.  Errors never throw across the ABI.
 *  - Return value: a qoq_status code.
 */
#ifndef QOQ_H_
#define QOQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *qoq_stream_t; /* same type as cudaStream_t */

typedef enum {
    QOQ_OK = 0,
    QOQ_ERR_INVALID_ARG = 1, /* null pointer, non-positive size */
    QOQ_ERR_UNSUPPORTED = 2, /* N or K not a multiple of 128, group not 0/128 */
    QOQ_ERR_MISALIGNED = 3,  /* a pointer breaks the alignment stated below */
    QOQ_ERR_WORKSPACE = 4,   /* workspace smaller than qoq_gemm_workspace_bytes */
    QOQ_ERR_CUDA = 5,        /* a CUDA launch / runtime call failed */
    QOQ_ERR_TIMEOUT = 6,     /* a device-side bounded wait expired (status word) */
    QOQ_ERR_DEVICE = 7       /* packed weights do not match the call or hold illegal codes */
} qoq_status;

/* Human-readable name of a status code (static string, never NULL). */
const char *qoq_status_string(int status);

/* Library / packed-format version (packed buffers carry it in their header). */
int qoq_version(void);

/*
 * qoq_bounds_checked -- 1 when this library is the bounds-check build
 * (compiled with QOQ_DEBUG_BOUNDS; the Python binding loads it when the
 * environment sets QOQ_DEBUG=1), else 0.  In that build every GEMM kernel
 * (all three paths) tests, before the access, each weight-block copy, each
 * split-tile slot and arrival-counter access and each output element it
 * writes by plain stores, and the KV4 attention each output and split
 * partial it writes, against the extent of its buffer; an access outside it
 * is skipped and sets bit 8 of the status word (qoq_workspace_status and
 * qoq_noalloc_status then return QOQ_ERR_DEVICE).  Results are otherwise
 * those of the release build.  A debugging aid with no counterpart in the
 * paper.
 */
int qoq_bounds_checked(void);

/*
 * qoq_quantize_weights -- progressive group quantization of fp16 weights on
 * the device ([QS-summary] "渐进式组量化" eq. 4/5 and "保护性量化范围";
 * [QS-review] 3.1).  One-time, load-time operation.
 *   group == 128: step 1, per output row n: s_w[n] = fp16(max_k|W[n,k]| / 119)
 *     (1.0 for an all-zero row), q8 = clamp(rne(W / s_w), -119, 119);
 *     step 2, per group of 128 k: lo = min(0, min q8), hi = max(0, max q8),
 *     s_g = max(1, ceil((hi - lo) / 15)), z = clamp(rne(-lo / s_g), 0, 15),
 *     q4 = clamp(rne(q8 / s_g) + z, 0, 15).  rne = round half to even;
 *     divisions of floats are IEEE fp32.
 *   group == 0 (per-channel W4, [QS-summary] "逐通道W4A8 GEMM中的快速反量化"):
 *     lo/hi = min/max(0, W[n,:]), s_w[n] = fp16((hi - lo) / 15) (1.0 if 0),
 *     z[n] = clamp(rne(-lo / s_w), 0, 15), q4 = clamp(rne(W / s_w) + z, 0, 15).
 * W   : fp16 [N][K].              q4 : uint8 [N][K], one code (0..15) per byte.
 * s_g : uint8 [N][K/128] (group==128; ignored and may be NULL for group==0).
 * z   : uint8 [N][K/128] (group==128) or [N] (group==0).
 * s_w : fp16 [N].
 * Requirements: N, K > 0; K % 128 == 0 for group 128.
 */
int qoq_quantize_weights(const uint16_t *W, int N, int K, int group, uint8_t *q4, uint8_t *s_g,
                         uint8_t *z, uint16_t *s_w, qoq_stream_t stream);

/* Bytes of the packed weight buffer for an N x K matrix (0 if unsupported). */
size_t qoq_packed_weight_bytes(int N, int K, int group);

/*
 * qoq_pack_weights -- device-side reorder of integer codes into the GEMM's
 * compute order ([QS-summary] "计算感知权重重排序"; [QS-review] 3.2: weights are
 * static, so they are stored once in the order the main loop reads them).
 * Layout of `packed` (qoq_packed_weight_bytes bytes, 16-byte aligned):
 *   256-byte header (magic "QOQW", version, N, K, group, block size, count of
 *   illegal codes), then (N/128) x (K/128) blocks, row-tile major: 8192 bytes
 *   of 4-bit codes for 128 rows x 128 k, followed (group mode) by 512 bytes
 *   of metadata, 4 per row: s_g, z, and the sum of the row's 128 codes as a
 *   little-endian uint16.  Within a block, 16-byte chunk
 *   (p*128 + r), p = 0..3, holds row r, k = 32p..32p+31 as four 32-bit words;
 *   word j covers k = 32p+8j+(0..7) and its byte b holds the code of
 *   k = 8j+b (low nibble) and k = 8j+b+4 (high nibble).  Per-channel mode
 *   appends z [N] (padded to 16 bytes).
 * Codes that break the GEMM's byte-lane bounds (q4 > 15, z > 15, s_g > 17,
 * or (q4 - z) * s_g outside [-128, 127]) are counted in the header; the GEMM
 * refuses such a buffer with QOQ_ERR_DEVICE (reported via the status word).
 * q4 [N][K] (16-byte aligned), s_g/z as in qoq_quantize_weights.
 * Requirements: N % 128 == 0, K % 128 == 0, group in {0, 128}.
 */
int qoq_pack_weights(const uint8_t *q4, const uint8_t *s_g, const uint8_t *z, int N, int K,
                     int group, void *packed, qoq_stream_t stream);

/* Inverse of qoq_pack_weights (tests and checkpoint inspection). */
int qoq_unpack_weights(const void *packed, int N, int K, int group, uint8_t *q4, uint8_t *s_g,
                       uint8_t *z, qoq_stream_t stream);

/*
 * qoq_quant_act -- per-token symmetric INT8 activation quantization
 * ([QS-review] 3.2 runtime precision map: every GEMM consumes INT8
 * activations, quantized by the kernel before it).  Per row m:
 *   s_x[m] = fp16(max_k |X[m,k]| / 127) (IEEE fp32 division, then round to
 *   fp16); Qx = clamp(rne(X / s_x), -127, 127); an all-zero scale gives an
 *   all-zero row; t_x[m] = sum_k Qx[m,k] (the t_X = X·1_k row sum of
 *   [QS-summary] eq. 13, needed by the per-channel GEMM).  Inputs must be
 *   finite.
 * X fp16 [M][K], Qx int8 [M][K] (both 16-byte aligned), s_x fp16 [M],
 * t_x int32 [M] or NULL.  Requirements: M, K > 0, K % 8 == 0.
 */
int qoq_quant_act(const uint16_t *X, int M, int K, int8_t *Qx, uint16_t *s_x, int32_t *t_x,
                  qoq_stream_t stream);

/*
 * Launch flag (qoq_quant_act_ex flags, qoq_gemm_options.flags):
 * QOQ_LAUNCH_OVERLAP launches the kernel as a programmatic dependent of the
 * kernel that precedes it in the stream (CUDA programmatic dependent
 * launch), so its launch and setup overlap that kernel's end.  The kernel
 * waits for the preceding kernel to complete before it reads its
 * activations, scales, workspace or output, and before it writes anything.
 * The GEMM also reads its packed weights and weight scales before that wait,
 * so with this flag they must not be written by a kernel that may still be
 * running (weights are static in serving).  Also valid inside CUDA graph
 * capture.
 */
#define QOQ_LAUNCH_OVERLAP 1u

/*
 * GEMM option flag (qoq_gemm_options.flags): QOQ_PLAN_RULES plans the launch
 * by the planner's rules alone.  Without it an automatic plan (no kernel,
 * tokens_per_tile or num_ctas forced) first looks the shape up in the
 * library's measured dispatch table: launch choices timed per (N, K, group,
 * M) on a GPU with the same SM count (the offline per-shape policy table of
 * the ADAngel review, "离线 Oracle Policy Map 与在线查表"), an entry covering
 * the token counts above the next smaller tuned M of its shape up to its own.
 */
#define QOQ_PLAN_RULES 2u

/*
 * Bytes of an activation operand (0 for an invalid shape or kind; requires
 * K % 128 == 0).  An activation operand is the INT8 activation of
 * qoq_quant_act in the order and encoding one GEMM path's tensor cores
 * consume (the activation-side counterpart of the compute-aware weight
 * reordering of [QS-summary] "计算感知权重重排序"); the GEMM lands it in shared
 * memory with TMA, without conversion work.  Two kinds, numbered like the
 * path that reads them (qoq_gemm_path):
 *   kind 1, fp16-operand path: Qx as fp16, [M][K] (int8 values are exact in
 *     fp16), 2*M*K bytes.
 *   kind 2, fp8-operand path:
 *     [u_hi plane: M x K bytes][u_lo plane: M x K bytes][t_g: (K/128) x Mp int32]
 *     with u = Qx + 128 = 16*u_hi + u_lo (u_hi, u_lo in [0, 15]),
 *     t_g[g][m] = sum of Qx[m, k] over the 128 k of group g, and Mp = M
 *     rounded up to a multiple of 4.
 */
size_t qoq_act_operand_bytes(int M, int K, int kind);

/*
 * qoq_quant_act_ex -- qoq_quant_act, and, when act_operand is not NULL, also
 * the activation operand of the given kind (qoq_act_operand_bytes(M, K,
 * kind) bytes, 16-byte aligned, written completely; requires K % 128 == 0).
 * Pass it to the GEMM with qoq_gemm_options.act_operand, for a GEMM whose
 * qoq_gemm_path equals `kind`; without it, the GEMM builds the operand itself
 * in its workspace with one extra kernel launch.  Same results in both cases.
 * kind is ignored when act_operand is NULL; otherwise it must be 1 or 2
 * (QOQ_ERR_INVALID_ARG).  flags: 0 or QOQ_LAUNCH_OVERLAP (other bits:
 * QOQ_ERR_UNSUPPORTED).
 */
int qoq_quant_act_ex(const uint16_t *X, int M, int K, int8_t *Qx, uint16_t *s_x, int32_t *t_x,
                     int kind, void *act_operand, uint32_t flags, qoq_stream_t stream);

/*
 * qoq_rmsnorm_quant_act -- RMS normalization fused with the per-token INT8
 * quantization of qoq_quant_act_ex: the norm in front of the QKV projection
 * and the FFN's first layer, into which the QServe runtime fuses the
 * activation quantization so that every GEMM receives INT8 activations
 * ([QS-summary] "QServe系统运行时"; [QS-review] 4, step 2).  The pages call
 * the norm LayerNorm; the Llama-family blocks use its RMS form, which this
 * computes.  Per row m, in fp32:
 *   r = 1 / sqrt(sum_k X[m,k]^2 / K + eps)   (0 when the root is 0)
 *   y[m,k] = fp16_rn((X[m,k] * r) * gamma[k])
 * and then exactly qoq_quant_act_ex on the fp16 row y: Qx, s_x, t_x and the
 * activation operand of `kind` (act_operand may be NULL).  Y, if not NULL,
 * receives y [M][K] (fp16): the rows the quantizer saw.
 * X fp16 [M][K], gamma fp16 [K], Qx int8 [M][K], Y fp16 [M][K] (each 16-byte
 * aligned), s_x fp16 [M], t_x int32 [M] or NULL.  eps >= 0 and finite
 * (QOQ_ERR_INVALID_ARG otherwise).  Requirements: M, K > 0, K % 8 == 0
 * (K % 128 == 0 with an activation operand).  flags: 0 or
 * QOQ_LAUNCH_OVERLAP.
 */
int qoq_rmsnorm_quant_act(const uint16_t *X, const uint16_t *gamma, float eps, int M, int K, int8_t *Qx,
                          uint16_t *s_x, int32_t *t_x, int kind, void *act_operand, uint16_t *Y, uint32_t flags,
                          qoq_stream_t stream);

/*
 * qoq_silu_mul_quant_act -- the SwiGLU activation in front of the FFN's
 * second layer (down = SiLU(gate) * up, "01 inference papers and
 * experiments" book chapter, FFN/MLP module), fused with the per-token INT8
 * quantization ([QS-summary] "QServe系统运行时": quantization fused into the
 * activation kernel).  H [M][2F] fp16 is the gate_up projection's output,
 * gate in columns 0..F-1, up in F..2F-1.  Per element, in fp32:
 *   y[m,f] = fp16_rn((g / (1 + exp(-g))) * u),  g = H[m,f], u = H[m,F+f]
 * (the CUDA fast intrinsics __expf and __fdividef, then a product: y within
 * 1.4e-5 relative of the exact value before its fp16 rounding), then exactly
 * qoq_quant_act_ex on the fp16 row y [F].  Y (optional) receives y [M][F].
 * Inputs must be finite with |y| < 65504.  H, Qx, Y 16-byte aligned.
 * Requirements: M, F > 0, F % 8 == 0 (F % 128 == 0 with an activation
 * operand).  flags: 0 or QOQ_LAUNCH_OVERLAP.
 */
int qoq_silu_mul_quant_act(const uint16_t *H, int M, int F, int8_t *Qx, uint16_t *s_x, int32_t *t_x, int kind,
                           void *act_operand, uint16_t *Y, uint32_t flags, qoq_stream_t stream);

/*
 * Workspace bytes qoq_w4a8_gemm needs for this shape on the current device:
 * a 256-byte status word area, one arrival counter per persistent CTA and
 * one int32 partial-tile slot (tokens-per-tile x 128) per persistent CTA,
 * used when a CTA's share of the work ends inside an output tile; then
 * scratch for the activation operand of the GEMM's path
 * (qoq_act_operand_bytes), used when the caller passes none.  The workspace
 * must be zero-filled once
 * before first use (qoq_workspace_init); every successful call leaves the
 * status word, counters and slots zero-filled again (after a
 * QOQ_ERR_TIMEOUT, re-initialise it); the activation scratch needs no
 * initialisation.
 */
size_t qoq_gemm_workspace_bytes(int M, int N, int K, int group);

/* Zero-fill a workspace (enqueued on `stream`). */
int qoq_workspace_init(void *workspace, size_t bytes, qoq_stream_t stream);

/*
 * qoq_w4a8_gemm -- the W4A8 GEMM with fused fp16 epilogue.
 *   group == 128 ([QS-summary] "逐组W4A8 GEMM中的快速反量化"; [QS-review] 3.2):
 *     acc[m,n] = sum_k Qx[m,k] * (q4[n,k] - z[n,k/128]) * s_g[n,k/128]  (exact int32)
 *   group == 0 ([QS-summary] eq. 13, zero folded into the epilogue):
 *     acc[m,n] = sum_k Qx[m,k] * q4[n,k] - z[n] * t_x[m]                 (exact int32)
 *   O[m,n] = fp16_rn(fp32(acc) * s_x[m] * s_w[n])   (fp32 products, left to right)
 * Qx int8 [M][K] (16-byte aligned); s_x fp16 [M]; t_x int32 [M] (group 0
 * only, may be NULL for group 128); packed from qoq_pack_weights for the same
 * N, K, group (16-byte aligned); s_w fp16 [N]; O fp16 [M][N] (16-byte aligned: the
 * output tiles are written by tensor bulk copies); workspace of
 * ws_bytes >= qoq_gemm_workspace_bytes(M, N, K, group), 16-byte aligned.
 * Requirements: M > 0, N % 128 == 0, K % 128 == 0, group in {0, 128}.
 * Device-side failures (a bounded wait expiring, mismatched or illegal packed
 * weights) do not fault: they set bits in the workspace status word, read by
 * qoq_workspace_status.
 */
int qoq_w4a8_gemm(const int8_t *Qx, const uint16_t *s_x, const int32_t *t_x, const void *packed,
                  const uint16_t *s_w, int M, int N, int K, int group, uint16_t *O,
                  void *workspace, size_t ws_bytes, qoq_stream_t stream);

/*
 * qoq_w4a8_gemm_i32 -- same GEMM, but writes the exact int32 accumulators
 * acc [M][N] (after the per-channel zero fold, before scaling) instead of O.
 * Test / debugging entry point; s_x and s_w may be NULL.
 */
int qoq_w4a8_gemm_i32(const int8_t *Qx, const int32_t *t_x, const void *packed, int M, int N,
                      int K, int group, int32_t *acc, void *workspace, size_t ws_bytes,
                      qoq_stream_t stream);

/*
 * Options for qoq_w4a8_gemm_ex (tests and tuning).  Zero-initialised fields
 * mean "automatic".
 *   tokens_per_tile : 16, 32, 64 or 128 (MMA N per CTA), 0 = automatic.
 *   num_ctas        : persistent CTAs that share the work (stream-K: the
 *                     tiles x K/128 k-stages are cut into num_ctas equal
 *                     contiguous ranges), 0 = one per SM; clamped to the
 *                     number of k-stages.
 *   timeout_ns      : bound of every device-side wait, 0 = 2 s.
 *   debug_flags     : bit 0 = the copy warp withholds the second stage, so
 *                     the bounded waits expire (timeout path test); bit 1 =
 *                     a split tile's last contributor never finishes it
 *                     directly, every contributor publishes its partial
 *                     (tests the fix-up by the last arriver).
 *   acc_out         : if non-NULL, int32 accumulators are written here
 *                     instead of O.
 *   kernel          : 0 = automatic, 1 = fp16-operand tensor-core path
 *                     (dequantized weights), 2 = fp8-operand path (4-bit
 *                     codes and split activations as exact e4m3, group 128
 *                     only, tokens_per_tile 16 or 32), 3 = CUDA-core dp4a
 *                     path (M <= 8; num_ctas = the K split, a thread-block
 *                     cluster of 1, 2, 4 or 8 CTAs per 128-row tile, raised
 *                     to the next of those sizes while one CTA's slice of
 *                     the activations would not fit in shared memory; no
 *                     activation operand).  Automatic: the measured dispatch
 *                     table for the shape, else dp4a up to 4 tokens, fp8 up
 *                     to 32 (g128), fp16 above.
 *   act_operand     : the activation operand written by qoq_quant_act_ex for
 *                     the same Qx (16-byte aligned), of the kind equal to
 *                     this GEMM's qoq_gemm_path; the GEMM reads it instead
 *                     of building it.  NULL = build it in the workspace.
 *   flags           : 0, QOQ_LAUNCH_OVERLAP and / or QOQ_PLAN_RULES (see
 *                     above; other bits: QOQ_ERR_UNSUPPORTED).
 *   schedule        : order of the tensor-core paths' work, 0 = automatic;
 *                     1 = stream-K only (each CTA one contiguous range of
 *                     the tiles x K/128 k-stages, tiles token-tile fastest);
 *                     2 = with two or more waves of tiles, all but the last
 *                     one to two waves go whole to the CTAs round-robin
 *                     (CTA c: tiles c, c + P, ...), token-tile fastest, the
 *                     rest stream-K; 3 = as 2 with the tiles in bands of
 *                     about sqrt(P * tokens_per_tile / 32) weight tiles,
 *                     weight-tile fastest within a band; 4 = as 2 with the
 *                     tiles weight-tile fastest (every weight tile of one
 *                     token tile, then the next token tile).
 */
typedef struct {
    int tokens_per_tile;
    int num_ctas;
    uint64_t timeout_ns;
    uint32_t debug_flags;
    int32_t *acc_out;
    int kernel;
    const void *act_operand;
    uint32_t flags;
    int schedule;
} qoq_gemm_options;

/* Workspace bytes for a GEMM run with the given options. */
size_t qoq_gemm_workspace_bytes_ex(int M, int N, int K, int group, const qoq_gemm_options *opt);

/*
 * The path a GEMM of this shape and options takes on the current device:
 * 1 = fp16-operand path, 2 = fp8-operand path, 3 = CUDA-core dp4a path, or
 * minus a qoq_status for invalid arguments.  For 1 and 2 it is also the kind
 * of activation operand the GEMM reads (qoq_quant_act_ex); path 3 reads Qx
 * itself.
 */
int qoq_gemm_path(int M, int N, int K, int group, const qoq_gemm_options *opt);

/*
 * The launch plan a GEMM of this shape and options gets on a GPU with
 * num_sms streaming multiprocessors, computed on the host by the library's
 * planner without a GPU (the GEMM entry points plan for the current device):
 *   path            : 1 = fp16-operand path, 2 = fp8-operand path (as
 *                     qoq_gemm_path);
 *   tokens_per_tile : tokens of one output tile (the MMA's N);
 *   num_ctas        : persistent CTAs (stream-K ranges);
 *   tiles           : output tiles (token tiles x N/128 weight tiles);
 *   k_stages        : tiles x K/128, the k-stages of work the CTAs share;
 *   workspace_bytes : as qoq_gemm_workspace_bytes_ex on such a GPU.
 * Returns QOQ_OK; QOQ_ERR_INVALID_ARG for a NULL out, num_sms <= 0 or
 * non-positive sizes; QOQ_ERR_UNSUPPORTED for an unsupported shape, group or
 * option value.  *out is written only on QOQ_OK.
 */
typedef struct {
    int path;
    int tokens_per_tile;
    int num_ctas;
    long long tiles;
    long long k_stages;
    size_t workspace_bytes;
} qoq_gemm_plan_info;

int qoq_gemm_plan(int M, int N, int K, int group, int num_sms, const qoq_gemm_options *opt,
                  qoq_gemm_plan_info *out);

int qoq_w4a8_gemm_ex(const int8_t *Qx, const uint16_t *s_x, const int32_t *t_x,
                     const void *packed, const uint16_t *s_w, int M, int N, int K, int group,
                     uint16_t *O, void *workspace, size_t ws_bytes, const qoq_gemm_options *opt,
                     qoq_stream_t stream);

/*
 * qoq_w4a8_gemm_noalloc -- the same GEMM (same arguments and results as
 * qoq_w4a8_gemm) for callers that cannot allocate device memory: for
 * example a plugin inside another framework's engine that is handed only its
 * input and output buffers, or a latency-critical path that must not call
 * cudaMalloc because it can synchronize the device.  The paper has no
 * counterpart of this entry point.
 * Its scratch (status word, arrival counters, partial-tile slots) is a fixed
 * 8 MiB array inside the library, which every GPU that loads the library
 * keeps until the process exits.  It never calls cudaMalloc, cudaFree or any
 * allocating routine.
 *  - Limit: a call needs qoq_gemm_workspace_bytes(M, N, K, group) <= 8 MiB;
 *    larger shapes are rejected with QOQ_ERR_WORKSPACE before any launch.
 *    The need depends on the whole shape, not on M alone: on a 152-SM GB300
 *    every Llama-3-8B linear layer fits up to M = 64 (qkv and o also at M = 128,
 *    whose planner picks half-width tiles), while Qwen1.5-72B down
 *    (N = 8192, K = 29568) at M = 64 needs about 8.8 MB and is rejected.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    outside any stream capture.
 *  - Every call re-zeroes the part of the array it uses (cudaMemsetAsync on
 *    `stream`), then launches the GEMM.  All calls share the one array, so
 *    calls that overlap on the GPU (different streams, no ordering between
 *    them) race and give wrong results; order them on one stream.
 *  - Device-side status bits (bounded-wait expiry, packed-weight mismatch)
 *    go to the array's status word; QOQ_OK means the launch was enqueued.
 *    Read the word with qoq_noalloc_status after a call and before the
 *    next one (the next call clears it).
 * Device ordinals of 64 and above: QOQ_ERR_UNSUPPORTED.
 */
int qoq_w4a8_gemm_noalloc(const int8_t *Qx, const uint16_t *s_x, const int32_t *t_x,
                          const void *packed, const uint16_t *s_w, int M, int N, int K, int group,
                          uint16_t *O, qoq_stream_t stream);

/*
 * qoq_noalloc_status -- the device status word of the allocation-free GEMM's
 * internal array on the current device, for callers of
 * qoq_w4a8_gemm_noalloc (which cannot pass a workspace to
 * qoq_workspace_status).  Synchronizes `stream`, copies the word to
 * *host_status, clears it, and returns QOQ_OK, QOQ_ERR_TIMEOUT or
 * QOQ_ERR_DEVICE by the bits found (1 = a bounded wait expired, 2 =
 * packed-weight header mismatch or illegal codes, 8 = bounds-check build
 * only: an access outside its buffer was skipped; 8 takes precedence over 1).
 * Allocates nothing.  The
 * paper has no counterpart of it.
 */
int qoq_noalloc_status(uint32_t *host_status, qoq_stream_t stream);

/*
 * ---------------------------------------------------------------- KV4 ----
 * The paged KV cache with per-head dynamic INT4 keys and values, and the
 * decode attention that reads it ([QS-summary] "QServe系统运行时": paged KV
 * cache, the per-head FP16 scale and zero point stored right after the
 * quantized KV features inside each page and updated online; "QServe中的KV4
 * 注意力"; [QS-review] 3.2 "KV 缓存管理" and 4, step 4).
 *
 * Quantization of one key or value vector (one token, one KV head, 128
 * values; eq. 1 of [QS-summary] "整数量化" with FP16 scale and zero):
 *   lo = min x, hi = max x; s = fp16((hi - lo) / 15) (1.0 when 0);
 *   z = fp16(rne(-lo / s)) (an integer); q = clamp(rne(x / s) + z, 0, 15);
 *   x ~ (q - z) * s.  Divisions IEEE fp32, rne = half to even.
 *
 * Page format: a page holds QOQ_KV4_PAGE_TOKENS = 64 token slots of one
 * sequence for all KV heads, head dim QOQ_KV4_HEAD_DIM = 128, and takes
 * qoq_kv4_page_bytes(H_kv) = H_kv * 8704 bytes: per KV head h, at offset
 * 8704 h, one chunk
 *   [K codes: 64 slots x 64 B][K meta: 64 slots x 4 B]
 *   [V codes: 64 slots x 64 B][V meta: 64 slots x 4 B]
 * A meta word holds s (fp16 bits, low half) and z (fp16 bits, high half).
 * The 64 code bytes of a slot are sixteen little-endian 32-bit words, word i
 * at byte 4 i; nibble j of a word (bits 4j .. 4j+3) holds one code:
 *   K: word i = 4 r + jj; with a = j & 3, b = j >> 2 the nibble holds
 *      dimension 32 jj + 16 (a & 1) + 8 (a >> 1) + 2 r + b;
 *   V: word i = 2 g + w; the nibble holds dimension g + 8 (8 w + j).
 * (The order in which the attention kernel's tensor-core fragments read the
 * codes.)  A pool of pages is one buffer of num_pages pages; a sequence's
 * page_table row lists its pages in token order: token position p of
 * sequence b lives in page page_table[b][p / 64], slot p % 64.
 */
#define QOQ_KV4_PAGE_TOKENS 64
#define QOQ_KV4_HEAD_DIM 128

/* Bytes of one KV4 page for num_kv_heads heads (0 if num_kv_heads is not in 1..1024). */
size_t qoq_kv4_page_bytes(int num_kv_heads);

/*
 * qoq_kv4_append -- quantize new key / value vectors into their cache slots
 * (the online update of the pages).  K, V fp16 [num_tokens][num_kv_heads][128]
 * (16-byte aligned); token t goes to sequence token_seq[t], position
 * token_pos[t] (int32 [num_tokens]); page_table int32 [num_seqs][max_pages];
 * pages: num_pages pages (16-byte aligned).  A token whose sequence,
 * position or page index is out of range is skipped and bit 4 is ORed into
 * *status (device uint32, may be NULL).  Two tokens of the same slot in one
 * call race.  Requirements: all counts > 0, num_kv_heads <= 1024.
 */
int qoq_kv4_append(const uint16_t *K, const uint16_t *V, int num_tokens, int num_kv_heads, const int32_t *token_seq,
                   const int32_t *token_pos, const int32_t *page_table, int num_seqs, int max_pages, void *pages,
                   int num_pages, uint32_t *status, qoq_stream_t stream);

/* Workspace bytes of qoq_kv4_decode_attention on the current device (0 for invalid arguments). */
size_t qoq_kv4_attention_workspace_bytes(int B, int num_q_heads, int num_kv_heads, int max_pages);

/*
 * qoq_kv4_decode_attention -- one decode step of attention over the KV4
 * cache, for B sequences with one query token each:
 *   Khat_t = (q_t - z_t) s_t (per token and KV head), Vhat_t likewise;
 *   O[b,h,:] = sum_t softmax_t(softmax_scale * Q[b,h,:] . Khat_t) Vhat_t
 * over the seq_lens[b] cached tokens of sequence b, query head h reading KV
 * head h / (num_q_heads / num_kv_heads) (grouped-query attention).
 * Q, O fp16 [B][num_q_heads][128] (16-byte aligned); pages as written by
 * qoq_kv4_append (num_pages in the pool); page_table int32 [B][max_pages];
 * seq_lens int32 [B] in [0, 64 max_pages] (a sequence of length 0 gives a
 * zero output); workspace >= qoq_kv4_attention_workspace_bytes, 16-byte
 * aligned, zero-filled once before first use (its first word is the
 * status word read by qoq_workspace_status: bit 4 = a length or page index
 * out of range, whose tokens are then skipped or read as stale slots).
 * Computed in fp32 with fp16 tensor-core operands (exact 4-bit codes and an
 * fp16 hi + lo pair for each softmax weight times scale); the fp16 output is
 * within 2e-3 * max_d |O[b,h,:]| + 1 fp16 ulp of the exact result.
 * Requirements: num_q_heads a multiple of num_kv_heads with a ratio of 1, 2,
 * 4 or 8; softmax_scale > 0 and finite; B, num_kv_heads <= 65535.
 */
int qoq_kv4_decode_attention(const uint16_t *Q, const void *pages, int num_pages, const int32_t *page_table,
                             const int32_t *seq_lens, int B, int num_q_heads, int num_kv_heads, int max_pages,
                             float softmax_scale, uint16_t *O, void *workspace, size_t ws_bytes,
                             qoq_stream_t stream);

/*
 * qoq_workspace_status -- synchronizes `stream`, copies the workspace status
 * word to *host_status, clears it on the device, and returns QOQ_OK,
 * QOQ_ERR_TIMEOUT or QOQ_ERR_DEVICE according to the bits found
 * (1 = a bounded wait expired, 2 = packed-weight header mismatch/illegal,
 * 4 = a KV4 sequence length or page index out of range, 8 = bounds-check
 * build only: an access outside its buffer was skipped; 8 takes precedence
 * over 1, whose expired wait it causes).
 */
int qoq_workspace_status(void *workspace, uint32_t *host_status, qoq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QOQ_H_ */

// Library-internal declarations shared by the CUDA translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

namespace qoq {

// Device ordinals the library serves (per-device state is kept in arrays of
// this size); the entry points return QOQ_ERR_UNSUPPORTED on a higher ordinal.
constexpr int kMaxDevices = 64;

// ------------------------------------------------------------------------
// Packed weight format (written by the packer, read by the GEMM).
// [header: 256 B]
// [blocks: (N/128) x (K/128) blocks, n-tile major, k-group minor]
//   each block = 8192 B of 4-bit codes for 128 rows x 128 k, then, in group
//   mode only, 512 B of metadata: per row r, byte 4r = s_g, byte 4r+1 = z,
//   bytes 4r+2..4r+3 = sum of the row's 128 codes (little-endian uint16).
//   Code layout inside a block: 512 chunks of 16 B; chunk (p * 128 + r),
//   p = 0..3, holds the 32 codes of row r at k = 32p .. 32p + 31 as four
//   32-bit words; word j covers k = 32p + 8j + (0..7); byte b of a word holds
//   the code of k = 8j + b in its low nibble and of k = 8j + b + 4 in its high
//   nibble.
// [per-channel mode only: z [N] bytes, padded to 16 B]
// ------------------------------------------------------------------------
constexpr uint32_t kPackedMagic = 0x57514F51u;  // "QOQW"
constexpr uint32_t kPackedVersion = 2u;
constexpr size_t kHeaderBytes = 256;
constexpr uint32_t kCodeBytes = 8192;           // 128 x 128 x 4 bit
constexpr uint32_t kMetaBytes = 512;            // 128 rows x (s_g, z, code sum)
constexpr int kTileN = 128;                     // weight rows per tile
constexpr int kTileK = 128;                     // k per stage = one group

struct PackedHeader {
    uint32_t magic;
    uint32_t version;
    int32_t N;
    int32_t K;
    int32_t group;
    uint32_t block_bytes;
    uint32_t illegal;     // codes that break the byte-lane bounds (0 when legal)
    uint32_t reserved[57];
};
static_assert(sizeof(PackedHeader) == kHeaderBytes, "header size");

__host__ __device__ inline uint32_t block_bytes(int group) { return group ? kCodeBytes + kMetaBytes : kCodeBytes; }

__host__ __device__ inline size_t packed_bytes(int N, int K, int group) {
    size_t blocks = static_cast<size_t>(N / kTileN) * static_cast<size_t>(K / kTileK);
    size_t b = kHeaderBytes + blocks * block_bytes(group);
    if (group == 0) b += (static_cast<size_t>(N) + 15) / 16 * 16;
    return b;
}

__host__ __device__ inline size_t packed_z_offset(int N, int K) {
    return kHeaderBytes + static_cast<size_t>(N / kTileN) * static_cast<size_t>(K / kTileK) * kCodeBytes;
}

// Workspace layout: [status word + pad: 256 B][ctas arrival counters][ctas x BT x 128
// int32 partial-tile slots][activation operand scratch].
constexpr size_t kWsStatusBytes = 256;

// Activation operands: the INT8 activation in the order and encoding a GEMM
// path's tensor cores consume, written by quant_act_ex (or by a preparation
// kernel the GEMM launches itself) and landed in shared memory by TMA.
//  kind 1 (fp16-operand path): Qx as fp16, [M][K] (every int8 value is an
//    exact fp16 number).
//  kind 2 (fp8-operand path):
//    [u_hi plane: M x K bytes][u_lo plane: M x K bytes][t_g: (K/128) x Mp int32]
//    u = Qx + 128 = 16 * u_hi + u_lo; each plane byte is its own e4m3 encoding
//    of value * 2^-9.  t_g[g][m] = sum of Qx[m, k] over the 128 k of group g.
//    Mp = M rounded up to 4 keeps every t_g row 16-byte aligned for TMA.
// The kind equals the GemmPath value of the path that reads it.
__host__ __device__ inline int act_tg_pitch(int M) { return (M + 3) & ~3; }
__host__ __device__ inline size_t act_planes_bytes(int M, int K) { return 2 * static_cast<size_t>(M) * K; }
__host__ __device__ inline size_t act_operand_bytes(int M, int K, int kind) {
    if (kind == 1) return 2 * static_cast<size_t>(M) * K;
    if (kind == 3) return 0;  // the CUDA-core path reads Qx itself
    return act_planes_bytes(M, K) + static_cast<size_t>(K / kTileK) * act_tg_pitch(M) * 4;
}

enum GemmPath : int {
    kPathF16 = 1,          // weights dequantized to exact fp16, kind::f16 MMA
    kPathF8 = 2,           // raw 4-bit codes and split activations as exact e4m3, kind::f8f6f4 MMA
    kPathGemv = 3,         // decode batches (M <= 4; up to 8 when forced): CUDA-core dp4a, K split over a cluster
};

struct GemmPlan {
    int path;              // GemmPath
    int BT;                // tokens per tile: 16, 32, 64 or 128 (GEMV path: tokens per launch, 1, 2, 4 or 8)
    int tok_tiles;         // ceil(M / BT)
    int n_tiles;           // N / 128
    int G;                 // K / 128 k-stages per tile
    long long tiles;       // tok_tiles * n_tiles
    long long total;       // tiles * G stages of work
    int ctas;              // persistent CTAs (stream-K ranges)
    size_t ws_bytes;       // workspace needed
    size_t counters_offset;
    size_t slots_offset;
    size_t act_offset;     // activation operand scratch (used when the caller passes none)
    size_t zero_bytes;     // leading workspace bytes that must be zero before a launch
    int gv_csize;          // GEMV path: CTAs per cluster (K split), 1, 2, 4 or 8
    int dp_tiles;          // tensor-core paths: tiles handed out whole, round-robin, before stream-K
    int band;              // weight tiles per band of the tile order (0: token-tile fastest)
    int sched;             // the schedule chosen: 1 to 4 (as force_sched); 0 on the GEMV path
};

// Kernel path, tile shape and persistent-CTA count for one GEMM.
// force_path / force_bt / force_ctas (0 = automatic) pin the choice for tests.
// use_table: consult the measured dispatch table before the rules.
// force_sched: 0 automatic, 1 stream-K only, 2 data-parallel waves then
// stream-K (tiles token-tile fastest), 3 as 2 with banded tile order, 4 as 2
// with the tiles weight-tile fastest.
GemmPlan plan_gemm(int M, int N, int K, int group, int num_sms, int force_path = 0, int force_bt = 0,
                   int force_ctas = 0, bool use_table = true, int force_sched = 0);

// Launchers (return cudaError_t of the launch).
cudaError_t launch_quant_act(const uint16_t *X, int M, int K, int8_t *Qx, uint16_t *s_x,
                             int32_t *t_x, int act_kind, void *act_operand, bool pdl, cudaStream_t stream);
// The same quantization of rows produced by the fp16 kernel in front of the
// GEMM, fused into it: RMS norm of X [M][K] (gamma [K], eps), or SiLU(G) * U
// of H = [G | U] [M][2F].  Y (optional) receives the fp16 rows quantized.
cudaError_t launch_rmsnorm_quant(const uint16_t *X, const uint16_t *gamma, float eps, uint16_t *Y, int M, int K,
                                 int8_t *Qx, uint16_t *s_x, int32_t *t_x, int act_kind, void *act_operand,
                                 bool pdl, cudaStream_t stream);
cudaError_t launch_silu_mul_quant(const uint16_t *H, uint16_t *Y, int M, int F, int8_t *Qx, uint16_t *s_x,
                                  int32_t *t_x, int act_kind, void *act_operand, bool pdl, cudaStream_t stream);
// Activation operand of the given kind from already quantized activations.
cudaError_t launch_act_operand(const int8_t *Qx, int M, int K, int act_kind, void *act_operand,
                               cudaStream_t stream);
cudaError_t launch_quantize_weights(const uint16_t *W, int N, int K, int group, uint8_t *q4,
                                    uint8_t *s_g, uint8_t *z, uint16_t *s_w, cudaStream_t stream);
cudaError_t launch_pack(const uint8_t *q4, const uint8_t *s_g, const uint8_t *z, int N, int K,
                        int group, void *packed, cudaStream_t stream);
cudaError_t launch_unpack(const void *packed, int N, int K, int group, uint8_t *q4, uint8_t *s_g,
                          uint8_t *z, cudaStream_t stream);

// KV4 paged cache: 64 tokens per page, head dim 128; per KV head one chunk
// of [K codes 64 x 64 B][K (s, z) 64 x 4 B][V codes 64 x 64 B][V (s, z) 64 x 4 B].
constexpr int kKv4PageTokens = 64;
constexpr uint32_t kKv4HeadChunkBytes = 2 * (kKv4PageTokens * 64 + kKv4PageTokens * 4);  // 8704

struct Kv4Plan {
    int splits;            // CTAs per (sequence, KV head), each over pages_per_split pages
    int pages_per_split;
    size_t partial_offset; // workspace offset of the split partials
    size_t ws_bytes;
};
Kv4Plan plan_kv4_attention(int B, int hq, int hkv, int max_pages, int num_sms);
cudaError_t launch_kv4_append(const uint16_t *K, const uint16_t *V, int n_tok, int hkv, const int32_t *tok_seq,
                              const int32_t *tok_pos, const int32_t *page_table, int num_seqs, int max_pages,
                              int num_pages, void *pages, uint32_t *status, cudaStream_t stream);
cudaError_t launch_kv4_attention(const uint16_t *Q, const void *pages, const int32_t *page_table,
                                 const int32_t *seq_lens, int B, int hq, int hkv, int max_pages, int num_pages,
                                 float scale, uint16_t *O, void *ws, const Kv4Plan &plan, uint64_t timeout_ns,
                                 cudaStream_t stream);

struct GemmArgs {
    const int8_t *Qx;
    const uint16_t *s_x;
    const int32_t *t_x;
    const void *packed;
    const uint16_t *s_w;
    int M, N, K, group;
    const void *act;      // activation operand of the plan's kind, or null (built in the workspace)
    uint16_t *O;          // fp16 output, or null when acc_out is set
    int32_t *acc_out;     // int32 pre-scale accumulators (test/debug mode)
    void *ws;
    uint32_t debug_flags;
    uint64_t timeout_ns;
    bool pdl;             // launch as a programmatic dependent of the preceding kernel
};

cudaError_t launch_gemm(const GemmArgs &a, const GemmPlan &plan, cudaStream_t stream);
cudaError_t launch_gemm_f8(const GemmArgs &a, const GemmPlan &plan, cudaStream_t stream);
cudaError_t launch_gemv(const GemmArgs &a, const GemmPlan &plan, cudaStream_t stream);

// Debug flag: the TMA producer withholds the second stage's load, so the
// consumers' bounded waits expire (exercises the timeout path).
constexpr uint32_t kDebugWithholdStage = 1u;
// Debug flag: a split tile's last contributor never finishes it directly;
// every contributor publishes its partial (exercises the fix-up by the last
// arriver).
constexpr uint32_t kDebugAlwaysPublish = 2u;

// Launch, optionally as a programmatic dependent of the preceding kernel in
// the stream (the kernel itself calls griddepcontrol.wait before it touches
// memory that kernel may still be writing).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          bool pdl, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1u : 0u;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace qoq

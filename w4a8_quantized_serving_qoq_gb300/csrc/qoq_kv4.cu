// KV4 cache and decode attention for sm_103a.
//
// Sources: "QServe: W4A8KV4 Quantization and System Co-design for Efficient
// LLM Serving" (papercache summary), sections "QServe系统运行时" (paged KV
// cache; per-head FP16 scale and zero stored right after the quantized KV
// features of each page, updated online) and "QServe中的KV4注意力"; "QServe：
// 把 W4A8KV4 的理论收益做成实测吞吐的量化—系统协同设计" (zenmind review),
// sections 3.2 ("KV 缓存管理") and 4 (step 4: decode attention reads INT4
// K/V, FP16 QK^T and SV products, scales and zeros fetched up front).
//
// Page format (64 tokens, head dim 128; include/qoq.h states it in full):
// per KV head one 8704-byte chunk [K codes 64 x 64 B][K (s, z) 64 x 4 B]
// [V codes 64 x 64 B][V (s, z) 64 x 4 B].  The nibble order of a token's
// 64 code bytes is the order the attention kernel's tensor-core fragments
// read (the KV-side counterpart of the pages' compute-aware weight reorder),
// so a lane's operand comes from one 16-byte (K) or four 8-byte (V) shared
// memory loads.
//
// GB300 design of the attention (one CTA per sequence, KV head and split of
// the sequence's pages):
//  * a producer warp streams each page's 8704-byte head chunk into a 4-stage
//    shared-memory ring with one bulk TMA copy;
//  * four consumer warps take one 16-token tile of every page each;
//  * the raw 4-bit codes are the tensor-core operands, as exact fp16
//    subnormals (one mask per two codes); the scales and zeros are applied
//    per token around the products:
//      q . Khat_t = s_t * (q . c_t - z_t * sum(q)),
//      sum_t p_t Vhat_t = sum_t (p_t s_t) c_t - sum_t p_t s_t z_t,
//    so no multiply per cached element;
//  * QK^T and PV are warp-level mma.sync m16n8k16 (fp16 in, fp32 out).  The
//    scores are computed as S^T with 16 tokens as rows (the K codes are the
//    A operand) and the G query heads that share a KV head (grouped-query
//    attention) as the 8 columns, each head twice for G <= 4; one movmatrix
//    transpose per 8 x 8 half turns the weight tile into PV's B fragment.
//    The weights p_t s_t enter PV as an fp16 pair hi + lo (hi = fp16(x), lo
//    = fp16(x - hi)), hi through the first copy of the columns and lo
//    through the second (G = 8: two PV n-tiles), so the fp16 operand loses
//    no accuracy against fp32;
//  * online softmax in fp32 per warp, rescaling the accumulators only when
//    the running maximum grows by more than 2^8; the warps' states are
//    merged in shared memory; with several splits per sequence the partial
//    states go to the workspace and a second kernel merges them.
#include <cuda.h>
#include <cuda_fp16.h>

#include <mutex>

#include "qoq_device.cuh"
#include "qoq_internal.h"

namespace qoq {
namespace {

constexpr int kHD = 128;                  // head dim
constexpr int kPageTok = kKv4PageTokens;  // tokens per page
constexpr uint32_t kCodesBytes = kPageTok * 64;       // 4096
constexpr uint32_t kMetaBytesKv = kPageTok * 4;       // 256
constexpr uint32_t kChunkBytes = kKv4HeadChunkBytes;  // 8704
constexpr uint32_t kVOff = kCodesBytes + kMetaBytesKv;
constexpr int kStages = 4;
constexpr int kConsumerWarps = 4;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr uint32_t kStatusBadIndex = 4u;  // a sequence length or page index out of range
constexpr int kRankMaxB = 256;            // batches up to this size run longest sequence first

__device__ __forceinline__ float h2f(uint16_t b) { return __half2float(__ushort_as_half(b)); }
__device__ __forceinline__ uint16_t f2h_rn(float f) { return __half_as_ushort(__float2half_rn(f)); }
__device__ __forceinline__ void named_bar_sync_kv(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

// ---------------------------------------------------------------- append --
// Dimension held by nibble s of word jj of the 16-byte K chunk r of a token:
// a = s & 3, b = s >> 2, dim = 32 jj + 16 (a & 1) + 8 (a >> 1) + 2 r + b.
// (Nibbles 0/4 and 2/6 fall in the k-chunk 32 jj .. +15, nibbles 1/5 and 3/7
// in 32 jj + 16 .. +31, so one mask per k-chunk gives uniform factors.)
__device__ __forceinline__ int k_nibble_dim(int r, int jj, int s) {
    const int a = s & 3, b = s >> 2;
    return 32 * jj + 16 * (a & 1) + 8 * (a >> 1) + 2 * r + b;
}
// Dimension held by nibble s of word w of the 8-byte V group g of a token:
// dim = g + 8 (8 w + s).
__device__ __forceinline__ int v_nibble_dim(int g, int w, int s) { return g + 8 * (8 * w + s); }

// One warp quantizes one 128-value vector (eq. 1 with FP16 scale and zero)
// and writes its 64 code bytes (in the K or V order) and its (s, z) word.
template <bool kIsK>
__device__ __forceinline__ void quantize_vec(const uint16_t *__restrict__ x, uint8_t *codes_dst, uint32_t *meta_dst,
                                             uint8_t *stage) {
    const int lane = threadIdx.x & 31;
    const uint2 raw = *reinterpret_cast<const uint2 *>(x + 4 * lane);
    float v[4] = {h2f(static_cast<uint16_t>(raw.x & 0xffffu)), h2f(static_cast<uint16_t>(raw.x >> 16)),
                  h2f(static_cast<uint16_t>(raw.y & 0xffffu)), h2f(static_cast<uint16_t>(raw.y >> 16))};
    float lo = fminf(fminf(v[0], v[1]), fminf(v[2], v[3]));
    float hi = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    uint16_t sb = f2h_rn(__fdiv_rn(__fsub_rn(hi, lo), 15.0f));
    if ((sb & 0x7fffu) == 0) sb = 0x3c00u;  // 1.0
    const float sf = h2f(sb);
    const uint16_t zb = f2h_rn(static_cast<float>(__float2int_rn(__fdiv_rn(-lo, sf))));
    const int zi = static_cast<int>(h2f(zb));  // an integer held exactly by the fp16 value
#pragma unroll
    for (int i = 0; i < 4; ++i) stage[4 * lane + i] = static_cast<uint8_t>(clampi(__float2int_rn(__fdiv_rn(v[i], sf)) + zi, 0, 15));
    __syncwarp();
    if (lane < 16) {
        uint32_t w = 0;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const int d = kIsK ? k_nibble_dim(lane >> 2, lane & 3, s) : v_nibble_dim(lane >> 1, lane & 1, s);
            w |= static_cast<uint32_t>(stage[d]) << (4 * s);
        }
        reinterpret_cast<uint32_t *>(codes_dst)[lane] = w;
    }
    if (lane == 0) *meta_dst = static_cast<uint32_t>(sb) | (static_cast<uint32_t>(zb) << 16);
    __syncwarp();
}

// One warp per (token, KV head): quantize its key and value vectors into
// the token's slot of its page.  Out-of-range sequence positions or page
// indices skip the token and set kStatusBadIndex.
__global__ void __launch_bounds__(256) kv4_append_kernel(const uint16_t *__restrict__ K, const uint16_t *__restrict__ V,
                                                         int n_tok, int hkv, const int32_t *__restrict__ tok_seq,
                                                         const int32_t *__restrict__ tok_pos,
                                                         const int32_t *__restrict__ page_table, int num_seqs,
                                                         int max_pages, int num_pages, uint8_t *__restrict__ pages,
                                                         uint32_t *status) {
    __shared__ uint8_t stage[8][kHD];
    const int warp = threadIdx.x >> 5;
    const long long item = static_cast<long long>(blockIdx.x) * 8 + warp;
    if (item >= static_cast<long long>(n_tok) * hkv) return;
    const int t = static_cast<int>(item / hkv), h = static_cast<int>(item % hkv);
    const int seq = tok_seq[t], pos = tok_pos[t];
    int page = -1;
    if (seq >= 0 && seq < num_seqs && pos >= 0 && pos / kPageTok < max_pages)
        page = page_table[static_cast<size_t>(seq) * max_pages + pos / kPageTok];
    if (page < 0 || page >= num_pages) {
        if ((threadIdx.x & 31) == 0 && status) atomicOr(status, kStatusBadIndex);
        return;
    }
    const int slot = pos % kPageTok;
    uint8_t *chunk = pages + (static_cast<size_t>(page) * hkv + h) * kChunkBytes;
    const size_t src = (static_cast<size_t>(t) * hkv + h) * kHD;
    quantize_vec<true>(K + src, chunk + slot * 64, reinterpret_cast<uint32_t *>(chunk + kCodesBytes) + slot,
                       stage[warp]);
    quantize_vec<false>(V + src, chunk + kVOff + slot * 64,
                        reinterpret_cast<uint32_t *>(chunk + kVOff + kCodesBytes) + slot, stage[warp]);
}

// ------------------------------------------------------------- attention --
struct AttnParams {
    const uint16_t *Q;        // [B][Hq][128]
    const uint8_t *pages;
    const int32_t *page_table;  // [B][max_pages]
    const int32_t *seq_lens;    // [B]
    uint16_t *O;              // [B][Hq][128]
    float *partial;           // [B][Hkv][splits][G][2 + 128] when splits > 1
    uint32_t *status;
    int B, hq, hkv, G, max_pages, num_pages, splits, pages_per_split;
    float scale_log2;         // softmax scale * log2(e)
    uint64_t timeout_ns;
};

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose of an 8 x 8 matrix of 16-bit elements held as the warp's m8n8
// fragments (lane l holds row l / 4, columns 2 (l % 4) and + 1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

// 2^x for x <= 0 (the hardware approximation; relative error about 2^-22,
// results below 2^-126 flush to zero, which a softmax weight can afford).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Four-bit codes enter the tensor core as fp16 subnormals: a nibble c in
// bits 0..3 of a half is exactly c * 2^-24, in bits 4..7 exactly 16 c *
// 2^-24 (at most 240 * 2^-24, still subnormal).  So a mask of a 32-bit word
// yields two codes (one per half) with no conversion arithmetic; the factor
// 2^-24 (or 2^-20) is taken out of the fp32 result.
constexpr uint32_t kLo = 0x000F000Fu, kHi = 0x00F000F0u;
constexpr float kF1 = 16777216.0f;   // 2^24
constexpr float kF16 = 1048576.0f;   // 2^20

template <int NSV>  // PV n-tiles: 1 for G <= 4, 2 for G = 8
__global__ void __launch_bounds__(kThreads, NSV == 1 ? 4 : 3) kv4_attention_kernel(const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + kStages * kChunkBytes);
    uint64_t *empty = full + kStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + kStages);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, h = blockIdx.y;
    int b = blockIdx.z;
    if (p.splits == 1 && p.B <= kRankMaxB) {
        // Launch order longest sequence first: the CTAs are handed to the SMs
        // in launch order, so each SM's share mixes long and short sequences
        // (and the SMs that get one CTA more get short ones).  Block z takes
        // the sequence of rank z in (length descending, index ascending).
        __shared__ int s_len[kRankMaxB];
        __shared__ int s_b;
        for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
            const int Li = p.seq_lens[i];
            s_len[i] = Li < 0 ? 0 : (Li > p.max_pages * kPageTok ? p.max_pages * kPageTok : Li);
        }
        if (threadIdx.x == 0) s_b = b;
        __syncthreads();
        for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
            const int Li = s_len[i];
            int rank = 0;
            for (int o = 0; o < p.B; ++o) rank += (s_len[o] > Li || (s_len[o] == Li && o < i)) ? 1 : 0;
            if (rank == static_cast<int>(blockIdx.z)) s_b = i;
        }
        __syncthreads();
        b = s_b;
    }
    const int G = p.G;
    int L = p.seq_lens[b];
    if (L < 0 || L > p.max_pages * kPageTok) {
        if (threadIdx.x == 0) atomicOr(p.status, kStatusBadIndex);
        L = L < 0 ? 0 : p.max_pages * kPageTok;
    }
    const int npages = (L + kPageTok - 1) / kPageTok;
    const int pg0 = split * p.pages_per_split;
    const int pg1 = min(npages, pg0 + p.pages_per_split);
    const int n_my = pg1 > pg0 ? pg1 - pg0 : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------ page producer --
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < n_my; ++i) {
                const int s = i % kStages, use = i / kStages;
                if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, abort_flag, p.status, p.timeout_ns)) break;
                int page = p.page_table[static_cast<size_t>(b) * p.max_pages + pg0 + i];
                if (page < 0 || page >= p.num_pages) {
                    atomicOr(p.status, kStatusBadIndex);
                    page = -1;
                }
                mbar_arrive_expect_tx(&full[s], page >= 0 ? kChunkBytes : 0u);
                if (page >= 0)
                    tma_load_1d(ring + s * kChunkBytes, p.pages + (static_cast<size_t>(page) * p.hkv + h) * kChunkBytes,
                                kChunkBytes, &full[s]);
                issued = i + 1;
            }
            // every copy issued must land before the CTA exits
            for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
                mbar_wait(&full[i % kStages], (i / kStages) & 1, nullptr, p.status, p.timeout_ns);
        }
        return;
    }

    // ---------------------------------------------------- consumer warps --
    // Fragment coordinates of m16n8k16: quad row g4 = lane / 4, column pair r.
    const int g4 = lane >> 2, r = lane & 3;
    // Columns of the score tile S^T [16 tokens][8]: for G <= 4, column c <
    // 2G holds query head c mod G (the copy at c >= G feeds the lo half of
    // the PV weights), the others are zero; for G = 8 column c is head c.
    // B operand of QK^T (Q^T, k = dims, n = columns): this lane's column is
    // g4; its two registers per 16-dim k-chunk j are dims 16 j + 2r (+1) and
    // 16 j + 2r + 8 (+9).
    const int ncols = NSV == 2 ? 8 : 2 * G;
    uint32_t qb[8][2];
    float qsum = 0.f;
    {
        const bool ok = g4 < ncols;
        const uint16_t *qr = p.Q + (static_cast<size_t>(b) * p.hq + h * G + (ok ? g4 % G : 0)) * kHD;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t x0 = ok ? *reinterpret_cast<const uint32_t *>(qr + 16 * j + 2 * r) : 0u;
            const uint32_t x1 = ok ? *reinterpret_cast<const uint32_t *>(qr + 16 * j + 2 * r + 8) : 0u;
            qb[j][0] = x0;
            qb[j][1] = x1;
            qsum += h2f(static_cast<uint16_t>(x0 & 0xffffu)) + h2f(static_cast<uint16_t>(x0 >> 16)) +
                    h2f(static_cast<uint16_t>(x1 & 0xffffu)) + h2f(static_cast<uint16_t>(x1 >> 16));
        }
    }
    qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
    qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);  // sum(q) of column g4's head
    // This lane's score / PV columns: c = 2r + e, e = 0, 1.
    bool col_ok[2], col_hi[2];
    float qs[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int c = 2 * r + e;
        col_ok[e] = c < ncols;
        col_hi[e] = NSV == 2 || c < G;  // G = 8: both halves of every column (n-tiles 0 and 1)
        qs[e] = __shfl_sync(0xffffffffu, qsum, 4 * c);
    }

    // Softmax state of this lane's two columns, over its own tokens; the
    // reference maximum m_ref is uniform over the eight lanes of a column.
    // The exponentials use m_ref, which is raised only when a tile's maximum
    // exceeds it by more than 2^8 (m_plus = m_ref + 8, or -inf before the
    // column's first score; weights up to 256 are harmless in fp32 / fp16),
    // so the PV accumulators are rescaled rarely.
    constexpr float kSlack = 8.0f;
    float m_ref[2] = {0.f, 0.f}, m_plus[2] = {-INFINITY, -INFINITY}, l_part[2] = {0.f, 0.f}, c_part[2] = {0.f, 0.f};
    // Bytes of the packed PV weight pair (G <= 4): for each of the lane's
    // columns the hi half (from the first operand) or the lo half.
    const uint32_t half_sel = (col_hi[0] ? 0x0010u : 0x0054u) | (col_hi[1] ? 0x3200u : 0x7600u);
    float acc[NSV][8][4];
#pragma unroll
    for (int n = 0; n < NSV; ++n)
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[n][mt][i] = 0.f;

    const int tile0 = warp * 16;  // this warp's 16 tokens of every page
    for (int i = 0; i < n_my; ++i) {
        const int s = i % kStages, use = i / kStages;
        if (!mbar_wait_warp(&full[s], use & 1, abort_flag, p.status, p.timeout_ns)) break;
        const uint8_t *ck = ring + s * kChunkBytes;
        const int tok0 = (pg0 + i) * kPageTok + tile0;
        // ---- S^T: rows = tokens tile0 + g4 (+8), columns as above.  A
        // fragment of k-word jj: the 16-byte K chunk r of the two tokens;
        // even k-chunks hold codes at factor 2^-24 (mask kLo), odd ones at
        // 2^-20 (mask kHi).
        float se[4] = {0.f, 0.f, 0.f, 0.f}, so[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const uint4 k0 = *reinterpret_cast<const uint4 *>(ck + (tile0 + g4) * 64 + 16 * r);
            const uint4 k8 = *reinterpret_cast<const uint4 *>(ck + (tile0 + 8 + g4) * 64 + 16 * r);
            const uint32_t w0[4] = {k0.x, k0.y, k0.z, k0.w}, w8[4] = {k8.x, k8.y, k8.z, k8.w};
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const uint32_t s0 = w0[jj] >> 8, s8 = w8[jj] >> 8;
                const uint32_t alo[4] = {w0[jj] & kLo, w8[jj] & kLo, s0 & kLo, s8 & kLo};
                const uint32_t ahi[4] = {w0[jj] & kHi, w8[jj] & kHi, s0 & kHi, s8 & kHi};
                mma16816(se, alo, qb[2 * jj][0], qb[2 * jj][1]);
                mma16816(so, ahi, qb[2 * jj + 1][0], qb[2 * jj + 1][1]);
            }
        }
        // Per token (g4 and g4 + 8 of the tile): in range?  Score factors
        // a = 2^24 ks scale and b = kz ks scale (so x = (se + so / 16) a -
        // b sum(q)), and the V scale / zero, zeroed out of range (unwritten
        // slots may hold any bits: select, never multiply, their values).
        // Score value v is token g4 + 8 (v >> 1), column 2r + (v & 1).
        float ka[2], kb[2], vsc[2], vzc[2];
        bool tin[2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const uint32_t km = *reinterpret_cast<const uint32_t *>(ck + kCodesBytes + 4 * (tile0 + 8 * t + g4));
            const uint32_t vm = *reinterpret_cast<const uint32_t *>(ck + kVOff + kCodesBytes + 4 * (tile0 + 8 * t + g4));
            tin[t] = tok0 + g4 + 8 * t < L;
            const float kss = __fmul_rn(h2f(static_cast<uint16_t>(km & 0xffffu)), p.scale_log2);
            ka[t] = __fmul_rn(kss, kF1);
            kb[t] = __fmul_rn(h2f(static_cast<uint16_t>(km >> 16)), kss);
            vsc[t] = tin[t] ? h2f(static_cast<uint16_t>(vm & 0xffffu)) : 0.f;
            vzc[t] = tin[t] ? h2f(static_cast<uint16_t>(vm >> 16)) : 0.f;
        }
        float x[4];
        bool raise = false;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int t = v >> 1, e = v & 1;
            const float xs = __fmaf_rn(__fmaf_rn(so[v], 0.0625f, se[v]), ka[t], -__fmul_rn(kb[t], qs[e]));
            x[v] = tin[t] && col_ok[e] ? xs : -INFINITY;
            raise |= x[v] > m_plus[e];  // m_plus = -inf until the column has a score
        }
        if (__any_sync(0xffffffffu, raise)) {
            // column maxima of the tile over the eight lanes of each column
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float tmax = fmaxf(x[e], x[2 + e]);
                tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
                tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
                tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
                if (tmax > m_plus[e]) {
                    const float alpha = m_plus[e] == -INFINITY ? 0.f : ex2(m_ref[e] - tmax);
                    m_ref[e] = tmax;
                    m_plus[e] = tmax + kSlack;
                    l_part[e] *= alpha;
                    c_part[e] *= alpha;
                    // PV column 2r + e is this lane's column e in every n-tile
#pragma unroll
                    for (int n = 0; n < NSV; ++n)
#pragma unroll
                        for (int mt = 0; mt < 8; ++mt) {
                            acc[n][mt][e] *= alpha;
                            acc[n][mt][2 + e] *= alpha;
                        }
                }
            }
        }
        // weights w = p_t * s_t of the V scale and the zero correction, as
        // an fp16 pair hi + lo; the PV weight of column c is hi (c < G) or
        // lo (a copy column) for G <= 4, both (n-tiles 0 and 1) for G = 8.
        // p = 2^(x - m_ref) is 0 for masked scores (x = -inf, m_ref finite).
        uint32_t pw[NSV][2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            float w[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float pt = ex2(__fsub_rn(x[2 * t + e], m_ref[e]));
                w[e] = __fmul_rn(pt, vsc[t]);
                l_part[e] += pt;
                c_part[e] = __fmaf_rn(w[e], vzc[t], c_part[e]);
            }
            const __half2 hi = __floats2half2_rn(w[0], w[1]);
            const float2 hf = __half22float2(hi);
            const __half2 lo = __floats2half2_rn(__fsub_rn(w[0], hf.x), __fsub_rn(w[1], hf.y));
            const uint32_t hw = *reinterpret_cast<const uint32_t *>(&hi), lw = *reinterpret_cast<const uint32_t *>(&lo);
            if (NSV == 2) {
                pw[0][t] = hw;
                pw[NSV - 1][t] = lw;
            } else {
                pw[0][t] = __byte_perm(hw, lw, half_sel);
            }
        }
        // PV B fragment (k = tokens, n = columns) by transposing the two
        // 8 x 8 halves of the weight tile
        uint32_t pb[NSV][2];
#pragma unroll
        for (int n = 0; n < NSV; ++n) {
            pb[n][0] = movmatrix_trans(pw[n][0]);
            pb[n][1] = movmatrix_trans(pw[n][1]);
        }
        // ---- O^T += Vc^T W: rows = dims g4 + 8 nt' of the V group g4, k = tokens
        const uint8_t *cv = ck + kVOff + 8 * g4;
        const uint2 va = *reinterpret_cast<const uint2 *>(cv + (tile0 + 2 * r) * 64);
        const uint2 vb = *reinterpret_cast<const uint2 *>(cv + (tile0 + 2 * r + 1) * 64);
        const uint2 vc = *reinterpret_cast<const uint2 *>(cv + (tile0 + 2 * r + 8) * 64);
        const uint2 vd = *reinterpret_cast<const uint2 *>(cv + (tile0 + 2 * r + 9) * 64);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with the page slot
        // pairs (token 2r | token 2r+1) and (2r+8 | 2r+9) of the nibbles nt = 8 w + s
        uint32_t ya[4], yc[4];
        ya[0] = __byte_perm(va.x, vb.x, 0x5410);
        ya[1] = __byte_perm(va.x, vb.x, 0x7632);
        ya[2] = __byte_perm(va.y, vb.y, 0x5410);
        ya[3] = __byte_perm(va.y, vb.y, 0x7632);
        yc[0] = __byte_perm(vc.x, vd.x, 0x5410);
        yc[1] = __byte_perm(vc.x, vd.x, 0x7632);
        yc[2] = __byte_perm(vc.y, vd.y, 0x5410);
        yc[3] = __byte_perm(vc.y, vd.y, 0x7632);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            // y = ya[q] holds nibbles nt = 4q .. 4q+3: even nt at factor 2^-24
            // (mask kLo), odd nt at 2^-20 (mask kHi) -> m-tiles 2q and 2q+1
            const uint32_t a8 = ya[q] >> 8, c8 = yc[q] >> 8;
            const uint32_t af0[4] = {ya[q] & kLo, ya[q] & kHi, yc[q] & kLo, yc[q] & kHi};
            const uint32_t af1[4] = {a8 & kLo, a8 & kHi, c8 & kLo, c8 & kHi};
#pragma unroll
            for (int n = 0; n < NSV; ++n) {
                mma16816(acc[n][2 * q], af0, pb[n][0], pb[n][1]);
                mma16816(acc[n][2 * q + 1], af1, pb[n][0], pb[n][1]);
            }
        }
    }

    // ---- the lane's partial sums over its tokens, summed over its column's lanes
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            l_part[e] += __shfl_xor_sync(0xffffffffu, l_part[e], o);
            c_part[e] += __shfl_xor_sync(0xffffffffu, c_part[e], o);
        }

    // ---- merge the four warps' states in shared memory (the ring is free
    // once every consumer passed its last page; the producer waits only for
    // copies it issued, which have all landed by then)
    named_bar_sync_kv(1, 32 * kConsumerWarps);
    float *mrg = reinterpret_cast<float *>(ring);  // [warp][G][2 + 128 + 1]: m, l, O..., c
    const int stride = 2 + kHD + 1;
    // accumulator rows: m-tile mt covers nibbles nt = 2 mt (dims g4 + 16 mt,
    // factor 2^-24) and nt = 2 mt + 1 (dims g4 + 8 + 16 mt, factor 2^-20);
    // columns 2r + e
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
#pragma unroll
        for (int n = 0; n < NSV; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int col = 2 * r + e;
                const bool hi_col = NSV == 2 ? n == 0 : col < G;
                const bool lo_col = NSV == 2 ? n == 1 : (col >= G && col < 2 * G);
                if (pass == 0 ? !hi_col : !lo_col) continue;
                const int hd = NSV == 2 ? col : (hi_col ? col : col - G);
                if (hd >= G) continue;
                float *dst = mrg + (warp * G + hd) * stride + 2;
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    const float v0 = __fmul_rn(acc[n][mt][e], kF1), v1 = __fmul_rn(acc[n][mt][2 + e], kF16);
                    if (pass == 0) {
                        dst[g4 + 16 * mt] = v0;
                        dst[g4 + 8 + 16 * mt] = v1;
                    } else {
                        dst[g4 + 16 * mt] += v0;
                        dst[g4 + 8 + 16 * mt] += v1;
                    }
                }
            }
        named_bar_sync_kv(1, 32 * kConsumerWarps);
    }
    if (g4 == 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int col = 2 * r + e;
            if (col < G) {
                float *dst = mrg + (warp * G + col) * stride;
                dst[0] = m_plus[e] == -INFINITY ? -INFINITY : m_ref[e];  // -inf: no score in this warp
                dst[1] = l_part[e];
                dst[2 + kHD] = c_part[e];
            }
        }
    }
    named_bar_sync_kv(1, 32 * kConsumerWarps);
    // one consumer thread per (head, dim) pair of the output
    for (int idx = threadIdx.x; idx < G * kHD; idx += 32 * kConsumerWarps) {
        const int hd = idx / kHD, d = idx % kHD;
        float M = -INFINITY;
        for (int w2 = 0; w2 < kConsumerWarps; ++w2) M = fmaxf(M, mrg[(w2 * G + hd) * stride]);
        float Ls = 0.f, Os = 0.f;
        for (int w2 = 0; w2 < kConsumerWarps; ++w2) {
            const float *src = mrg + (w2 * G + hd) * stride;
            const float f = src[0] == -INFINITY ? 0.f : ex2(src[0] - M);
            Ls = __fmaf_rn(f, src[1], Ls);
            Os = __fmaf_rn(f, __fsub_rn(src[2 + d], src[2 + kHD]), Os);
        }
        const size_t hq_idx = static_cast<size_t>(b) * p.hq + h * G + hd;
        if (p.splits == 1) {
            if (!in_bounds(hq_idx * kHD + d, 1, static_cast<unsigned long long>(p.B) * p.hq * kHD, p.status)) continue;
            p.O[hq_idx * kHD + d] = f2h_rn(Ls > 0.f ? __fdiv_rn(Os, Ls) : 0.f);
        } else {
            const size_t part_off =
                ((static_cast<size_t>(b) * p.hkv + h) * p.splits + split) * G * (2 + kHD) + hd * (2 + kHD);
            if (!in_bounds(part_off, 2 + kHD,
                           static_cast<unsigned long long>(p.B) * p.hkv * p.splits * G * (2 + kHD), p.status))
                continue;
            float *part = p.partial + part_off;
            if (d == 0) {
                part[0] = M;
                part[1] = Ls;
            }
            part[2 + d] = Os;
        }
    }
}

// Merge of the splits of one (sequence, query head): one thread per dim.
__global__ void kv4_combine_kernel(const float *__restrict__ partial, int hq, int hkv, int G, int splits,
                                   uint16_t *__restrict__ O) {
    const int b = blockIdx.y, qh = blockIdx.x, d = threadIdx.x;
    const int h = qh / G, hd = qh % G;
    const float *base = partial + (static_cast<size_t>(b) * hkv + h) * splits * G * (2 + kHD) + hd * (2 + kHD);
    const size_t sstride = static_cast<size_t>(G) * (2 + kHD);
    float M = -INFINITY;
    for (int s = 0; s < splits; ++s) M = fmaxf(M, base[s * sstride]);
    float Ls = 0.f, Os = 0.f;
    for (int s = 0; s < splits; ++s) {
        const float *src = base + s * sstride;
        const float f = src[0] == -INFINITY ? 0.f : exp2f(src[0] - M);
        Ls = __fmaf_rn(f, src[1], Ls);
        Os = __fmaf_rn(f, src[2 + d], Os);
    }
    O[(static_cast<size_t>(b) * hq + qh) * kHD + d] = f2h_rn(Ls > 0.f ? __fdiv_rn(Os, Ls) : 0.f);
}

constexpr size_t kAttnSmem = 128 + kStages * kChunkBytes + 2 * kStages * 8 + 16;

template <int NSV>
cudaError_t launch_attn(const AttnParams &p, cudaStream_t stream) {
    static std::mutex mu;
    static bool configured[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!configured[dev]) {
            e = cudaFuncSetAttribute(kv4_attention_kernel<NSV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kAttnSmem));
            if (e != cudaSuccess) return e;
            // the whole unified L1 / shared memory as shared memory, so that
            // four CTAs (4 x 35 KB) fit beside each other
            e = cudaFuncSetAttribute(kv4_attention_kernel<NSV>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     static_cast<int>(cudaSharedmemCarveoutMaxShared));
            if (e != cudaSuccess) return e;
            configured[dev] = true;
        }
    }
    const dim3 grid(p.splits, p.hkv, p.B);
    kv4_attention_kernel<NSV><<<grid, kThreads, kAttnSmem, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess || p.splits == 1) return e;
    kv4_combine_kernel<<<dim3(p.hq, p.B), kHD, 0, stream>>>(p.partial, p.hq, p.hkv, p.G, p.splits, p.O);
    return cudaGetLastError();
}

}  // namespace

Kv4Plan plan_kv4_attention(int B, int hq, int hkv, int max_pages, int num_sms) {
    Kv4Plan pl{};
    const long long base = static_cast<long long>(B) * hkv;
    // As many splits as keep the whole grid resident at once (one wave: 4
    // CTAs per SM, 3 for G = 8), at least two pages per split.  A second,
    // partial wave costs more than the shorter splits save (measured: batch
    // 64 x ~1K tokens 25.8 us in one wave against 31.2 us in 1.7 waves).
    const int G0 = hkv > 0 ? hq / hkv : 0;
    const long long cap = static_cast<long long>(G0 > 4 ? 3 : 4) * num_sms;
    long long splits = cap / base;
    const long long max_splits = (max_pages + 1) / 2;
    if (splits > max_splits) splits = max_splits;
    if (splits < 1) splits = 1;
    pl.pages_per_split = static_cast<int>((max_pages + splits - 1) / splits);
    pl.splits = (max_pages + pl.pages_per_split - 1) / pl.pages_per_split;
    const int G = G0;
    pl.partial_offset = kWsStatusBytes;
    pl.ws_bytes = kWsStatusBytes + (pl.splits > 1 ? static_cast<size_t>(base) * pl.splits * G * (2 + kHD) * 4 : 0);
    return pl;
}

cudaError_t launch_kv4_append(const uint16_t *K, const uint16_t *V, int n_tok, int hkv, const int32_t *tok_seq,
                              const int32_t *tok_pos, const int32_t *page_table, int num_seqs, int max_pages,
                              int num_pages, void *pages, uint32_t *status, cudaStream_t stream) {
    const long long items = static_cast<long long>(n_tok) * hkv;
    const unsigned blocks = static_cast<unsigned>((items + 7) / 8);
    kv4_append_kernel<<<blocks, 256, 0, stream>>>(K, V, n_tok, hkv, tok_seq, tok_pos, page_table, num_seqs, max_pages,
                                                  num_pages, static_cast<uint8_t *>(pages), status);
    return cudaGetLastError();
}

cudaError_t launch_kv4_attention(const uint16_t *Q, const void *pages, const int32_t *page_table,
                                 const int32_t *seq_lens, int B, int hq, int hkv, int max_pages, int num_pages,
                                 float scale, uint16_t *O, void *ws, const Kv4Plan &plan, uint64_t timeout_ns,
                                 cudaStream_t stream) {
    AttnParams p;
    p.Q = Q;
    p.pages = static_cast<const uint8_t *>(pages);
    p.page_table = page_table;
    p.seq_lens = seq_lens;
    p.O = O;
    p.partial = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + plan.partial_offset);
    p.status = static_cast<uint32_t *>(ws);
    p.B = B;
    p.hq = hq;
    p.hkv = hkv;
    p.G = hq / hkv;
    p.max_pages = max_pages;
    p.num_pages = num_pages;
    p.splits = plan.splits;
    p.pages_per_split = plan.pages_per_split;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.timeout_ns = timeout_ns;
    return p.G <= 4 ? launch_attn<1>(p, stream) : launch_attn<2>(p, stream);
}

}  // namespace qoq

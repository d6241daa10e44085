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
//    scores are computed transposed, the G query heads that share a KV head
//    (grouped-query attention) as rows, twice, so that the score fragment of
//    a lane is already its B fragment for PV: the weights p_t s_t enter PV
//    as an fp16 pair hi + lo (hi = fp16(x), lo = fp16(x - hi)), hi through
//    the first copy of the rows and lo through the second, so the fp16
//    operand loses no accuracy against fp32;
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

// 2^x for x <= 0 (the hardware approximation; relative error about 2^-22,
// results below 2^-126 flush to zero, which a softmax weight can afford).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// An fp16 pair (hi, lo) with hi + lo = x to about 2^-22 relative.
__device__ __forceinline__ void split_f16(float x, uint16_t &hi, uint16_t &lo) {
    const __half h = __float2half_rn(x);
    hi = __half_as_ushort(h);
    lo = f2h_rn(__fsub_rn(x, __half2float(h)));
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
__global__ void __launch_bounds__(kThreads) kv4_attention_kernel(const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + kStages * kChunkBytes);
    uint64_t *empty = full + kStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + kStages);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
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
    // S^T = Q Khat^T with the query heads as rows: row rho < 2G holds head
    // rho mod G (the second copy feeds the lo half of the PV weights), the
    // other rows are zero.  This lane's score rows: g4 (and g4 + 8).
    const bool row_ok = g4 < 2 * G;
    const int my_head = row_ok ? g4 % G : 0;
    uint32_t qa[8][4];
    float qsum = 0.f;
    {
        const uint16_t *qr0 = p.Q + (static_cast<size_t>(b) * p.hq + h * G + my_head) * kHD;
        const bool ok8 = g4 + 8 < 2 * G;
        const uint16_t *qr8 = p.Q + (static_cast<size_t>(b) * p.hq + h * G + (ok8 ? (g4 + 8) % G : 0)) * kHD;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t x0 = row_ok ? *reinterpret_cast<const uint32_t *>(qr0 + 16 * j + 2 * r) : 0u;
            const uint32_t x1 = row_ok ? *reinterpret_cast<const uint32_t *>(qr0 + 16 * j + 2 * r + 8) : 0u;
            qa[j][0] = x0;
            qa[j][1] = ok8 ? *reinterpret_cast<const uint32_t *>(qr8 + 16 * j + 2 * r) : 0u;
            qa[j][2] = x1;
            qa[j][3] = ok8 ? *reinterpret_cast<const uint32_t *>(qr8 + 16 * j + 2 * r + 8) : 0u;
            qsum += h2f(static_cast<uint16_t>(x0 & 0xffffu)) + h2f(static_cast<uint16_t>(x0 >> 16)) +
                    h2f(static_cast<uint16_t>(x1 & 0xffffu)) + h2f(static_cast<uint16_t>(x1 >> 16));
        }
    }
    qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
    qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);  // sum(q) of this lane's head

    // Softmax state of this lane's head, over its own tokens; the maximum
    // m_used is uniform over the quad.  The exponentials use m_used, which is
    // raised only when a tile's maximum exceeds it by more than 2^8 (weights
    // up to 256 are harmless in fp32 / fp16), so the PV accumulators are
    // rescaled rarely.
    constexpr float kSlack = 8.0f;
    float m_used = -INFINITY, l_part = 0.f, c_part = 0.f;
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
        // ---- S^T: rows = heads, columns = tokens tile0 + 8 nt + {2r, 2r+1}
        // (n-tile nt); even k-chunks hold codes at factor 2^-24, odd ones at 2^-20
        float se[2][4], so[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) se[nt][e] = so[nt][e] = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const uint4 kv = *reinterpret_cast<const uint4 *>(ck + (tile0 + 8 * nt + g4) * 64 + 16 * r);
            const uint32_t kw[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const uint32_t w8 = kw[jj] >> 8;
                mma16816(se[nt], qa[2 * jj], kw[jj] & kLo, w8 & kLo);
                mma16816(so[nt], qa[2 * jj + 1], kw[jj] & kHi, w8 & kHi);
            }
        }
        // K scale and zero of the lane's four tokens 8 nt + 2r + e
        const uint2 km0 = *reinterpret_cast<const uint2 *>(ck + kCodesBytes + 4 * (tile0 + 2 * r));
        const uint2 km1 = *reinterpret_cast<const uint2 *>(ck + kCodesBytes + 4 * (tile0 + 8 + 2 * r));
        const uint32_t kmw[4] = {km0.x, km0.y, km1.x, km1.y};
        float x[4];
        float tmax = -INFINITY;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int nt = t >> 1, e = t & 1;
            const float dot = __fmaf_rn(se[nt][e], kF1, __fmul_rn(so[nt][e], kF16));  // q . c_t
            const float ks = h2f(static_cast<uint16_t>(kmw[t] & 0xffffu)), kz = h2f(static_cast<uint16_t>(kmw[t] >> 16));
            const bool in = row_ok && tok0 + 8 * nt + 2 * r + e < L;
            x[t] = in ? __fmul_rn(__fmul_rn(__fsub_rn(dot, __fmul_rn(kz, qsum)), ks), p.scale_log2) : -INFINITY;
            tmax = fmaxf(tmax, x[t]);
        }
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
        const bool raise = tmax > m_used + kSlack || (m_used == -INFINITY && tmax != -INFINITY);
        if (__any_sync(0xffffffffu, raise)) {
            const float m_new = raise ? tmax : m_used;
            const float alpha = (m_used == -INFINITY || !raise) ? (m_used == -INFINITY ? 0.f : 1.f) : ex2(m_used - m_new);
            m_used = m_new;
            l_part *= alpha;
            c_part *= alpha;
            // PV column c (of either n-tile) belongs to the head of score row c
            const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * r);
            const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * r + 4);
#pragma unroll
            for (int n = 0; n < NSV; ++n)
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    acc[n][mt][0] *= a0;
                    acc[n][mt][1] *= a1;
                    acc[n][mt][2] *= a0;
                    acc[n][mt][3] *= a1;
                }
        }
        // weights w_t = p_t * s_t of the V scale and the zero correction
        const uint2 vm0 = *reinterpret_cast<const uint2 *>(ck + kVOff + kCodesBytes + 4 * (tile0 + 2 * r));
        const uint2 vm1 = *reinterpret_cast<const uint2 *>(ck + kVOff + kCodesBytes + 4 * (tile0 + 8 + 2 * r));
        const uint32_t vmw[4] = {vm0.x, vm0.y, vm1.x, vm1.y};
        uint16_t whi[4], wlo[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            // masked tokens may sit in never-written slots: select, never multiply, their scales
            const float pt = x[t] == -INFINITY ? 0.f : ex2(__fsub_rn(x[t], m_used));
            const float vs = h2f(static_cast<uint16_t>(vmw[t] & 0xffffu)), vz = h2f(static_cast<uint16_t>(vmw[t] >> 16));
            const float w = pt != 0.f ? __fmul_rn(pt, vs) : 0.f;
            l_part += pt;
            c_part = w != 0.f ? __fmaf_rn(w, vz, c_part) : c_part;
            split_f16(w, whi[t], wlo[t]);
        }
        // PV B fragment, column g4 (n-tile n): hi part of head g4 for g4 < G,
        // lo part for G <= g4 < 2G (G <= 4); for G = 8 n-tile 0 is hi, 1 is lo
        uint32_t pb[NSV][2];
#pragma unroll
        for (int n = 0; n < NSV; ++n) {
            const bool hi_part = NSV == 2 ? n == 0 : g4 < G;
            const uint16_t *src = hi_part ? whi : wlo;
            pb[n][0] = row_ok ? (static_cast<uint32_t>(src[0]) | (static_cast<uint32_t>(src[1]) << 16)) : 0u;
            pb[n][1] = row_ok ? (static_cast<uint32_t>(src[2]) | (static_cast<uint32_t>(src[3]) << 16)) : 0u;
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

    // ---- the lane's partial sums over its tokens, summed over the quad
    l_part += __shfl_xor_sync(0xffffffffu, l_part, 1);
    l_part += __shfl_xor_sync(0xffffffffu, l_part, 2);
    c_part += __shfl_xor_sync(0xffffffffu, c_part, 1);
    c_part += __shfl_xor_sync(0xffffffffu, c_part, 2);

    // ---- merge the four warps' states in shared memory (the ring is free
    // once every consumer passed its last page; the producer waits only for
    // copies it issued, which have all landed by then)
    named_bar_sync_kv(1, 32 * kConsumerWarps);
    float *mrg = reinterpret_cast<float *>(ring);  // [warp][G][2 + 128 + 1]: m, l, O..., c
    const int stride = 2 + kHD + 1;
    // accumulator rows: m-tile mt covers nibbles nt = 2 mt (dims g4 + 16 mt,
    // factor 2^-24) and nt = 2 mt + 1 (dims g4 + 8 + 16 mt, factor 2^-20);
    // columns 8 n + 2r + e
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
#pragma unroll
        for (int n = 0; n < NSV; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int col = (NSV == 2 ? 0 : 0) + 2 * r + e;
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
    if (r == 0 && g4 < G) {
        float *dst = mrg + (warp * G + g4) * stride;
        dst[0] = m_used;
        dst[1] = l_part;
        dst[2 + kHD] = c_part;
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
            p.O[hq_idx * kHD + d] = f2h_rn(Ls > 0.f ? __fdiv_rn(Os, Ls) : 0.f);
        } else {
            float *part = p.partial + ((static_cast<size_t>(b) * p.hkv + h) * p.splits + split) * G * (2 + kHD) +
                          hd * (2 + kHD);
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
    // about four CTAs per SM over the whole grid, at least two pages per split
    long long splits = (4LL * num_sms + base - 1) / base;
    const long long max_splits = (max_pages + 1) / 2;
    if (splits > max_splits) splits = max_splits;
    if (splits < 1) splits = 1;
    pl.pages_per_split = static_cast<int>((max_pages + splits - 1) / splits);
    pl.splits = (max_pages + pl.pages_per_split - 1) / pl.pages_per_split;
    const int G = hkv > 0 ? hq / hkv : 0;
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

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
//    integers (one bit-or and one fp16x2 subtract per two codes); the scales
//    and zeros are applied per token around the products:
//      q . Khat_t = s_t * (q . c_t - z_t * sum(q)),
//      sum_t p_t Vhat_t = sum_t (p_t s_t) c_t - sum_t p_t s_t z_t,
//    so no multiply per cached element;
//  * QK^T and PV are warp-level mma.sync m16n8k16 (fp16 in, fp32 out): the
//    G query heads that share a KV head (grouped-query attention) are the
//    N = 8 columns of QK^T; for PV the weights p_t s_t enter as an fp16
//    pair hi + lo (hi = fp16(x), lo = fp16(x - hi)) in spare columns, so the
//    fp16 operand loses no accuracy against fp32;
//  * online softmax in fp32 with exp2f per warp; the warps' states are
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
// a = s & 3, b = s >> 2, dim = 32 jj + 16 (a >> 1) + 8 (a & 1) + 2 r + b.
__device__ __forceinline__ int k_nibble_dim(int r, int jj, int s) {
    const int a = s & 3, b = s >> 2;
    return 32 * jj + 16 * (a >> 1) + 8 * (a & 1) + 2 * r + b;
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

// Two 4-bit codes (nibbles s and s + 4 of w, shifted down by 4s) as an
// fp16x2 of their exact integer values: 0x6400 | c is the fp16 1024 + c.
__device__ __forceinline__ uint32_t codes_f16x2(uint32_t w_shifted) {
    uint32_t h = (w_shifted & 0x000F000Fu) | 0x64006400u;
    const __half2 r = __hsub2(*reinterpret_cast<const __half2 *>(&h), __halves2half2(__ushort_as_half(0x6400u),
                                                                                    __ushort_as_half(0x6400u)));
    return *reinterpret_cast<const uint32_t *>(&r);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    return static_cast<uint32_t>(f2h_rn(lo)) | (static_cast<uint32_t>(f2h_rn(hi)) << 16);
}

template <int NSV>  // PV n-tiles: ceil(2G / 8)
__global__ void __launch_bounds__(kThreads) kv4_attention_kernel(const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    float *pstage = reinterpret_cast<float *>(ring + kStages * kChunkBytes);    // [4 warps][16 tokens][8 heads]
    uint64_t *full = reinterpret_cast<uint64_t *>(pstage + kConsumerWarps * 128);
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
    } else {
        // ------------------------------------------------ consumer warps --
        const int g4 = lane >> 2, r = lane & 3;
        // Q^T fragments (k = dims, n = the G query heads of this KV head)
        // and sum(q) per head, loaded once.
        uint32_t qb[8][2];
        float qsum_part = 0.f;
        {
            const bool valid = g4 < G;
            const uint16_t *qrow = p.Q + (static_cast<size_t>(b) * p.hq + h * G + (valid ? g4 : 0)) * kHD;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t lo = valid ? *reinterpret_cast<const uint32_t *>(qrow + 16 * j + 2 * r) : 0u;
                const uint32_t hi = valid ? *reinterpret_cast<const uint32_t *>(qrow + 16 * j + 2 * r + 8) : 0u;
                qb[j][0] = lo;
                qb[j][1] = hi;
                qsum_part += h2f(static_cast<uint16_t>(lo & 0xffffu)) + h2f(static_cast<uint16_t>(lo >> 16)) +
                             h2f(static_cast<uint16_t>(hi & 0xffffu)) + h2f(static_cast<uint16_t>(hi >> 16));
            }
        }
        qsum_part += __shfl_xor_sync(0xffffffffu, qsum_part, 1);
        qsum_part += __shfl_xor_sync(0xffffffffu, qsum_part, 2);  // sum(q) of head g4, in every lane of its quad
        // this lane's QK^T columns are heads 2r and 2r + 1
        const float qs0 = __shfl_sync(0xffffffffu, qsum_part, 8 * r);
        const float qs1 = __shfl_sync(0xffffffffu, qsum_part, 8 * r + 4);
        const bool hv0 = 2 * r < G, hv1 = 2 * r + 1 < G;

        float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f}, c_run[2] = {0.f, 0.f};
        float acc[NSV][8][4];
#pragma unroll
        for (int n = 0; n < NSV; ++n)
#pragma unroll
            for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[n][mt][i] = 0.f;
        // PV columns of this lane: n-tile n, column 8n + 2r + e -> head of
        // that column and whether the hi or the lo part enters it
        float *pst = pstage + warp * 128;

        for (int i = 0; i < n_my; ++i) {
            const int s = i % kStages, use = i / kStages;
            if (!mbar_wait_warp(&full[s], use & 1, abort_flag, p.status, p.timeout_ns)) break;
            const uint8_t *ck = ring + s * kChunkBytes;
            const int tile0 = warp * 16;                       // this warp's tile of the page
            const int tok0 = (pg0 + i) * kPageTok + tile0;     // position of its first token
            // ---- S = Q K^T for 16 tokens x 8 columns
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
            const uint4 k0 = *reinterpret_cast<const uint4 *>(ck + (tile0 + g4) * 64 + 16 * r);
            const uint4 k1 = *reinterpret_cast<const uint4 *>(ck + (tile0 + g4 + 8) * 64 + 16 * r);
            const uint32_t kw0[4] = {k0.x, k0.y, k0.z, k0.w}, kw1[4] = {k1.x, k1.y, k1.z, k1.w};
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int a = 2 * half;
                    const uint32_t af[4] = {codes_f16x2(kw0[jj] >> (4 * a)), codes_f16x2(kw1[jj] >> (4 * a)),
                                            codes_f16x2(kw0[jj] >> (4 * (a + 1))), codes_f16x2(kw1[jj] >> (4 * (a + 1)))};
                    mma16816(sc, af, qb[2 * jj + half][0], qb[2 * jj + half][1]);
                }
            }
            const uint32_t km0 = *reinterpret_cast<const uint32_t *>(ck + kCodesBytes + 4 * (tile0 + g4));
            const uint32_t km1 = *reinterpret_cast<const uint32_t *>(ck + kCodesBytes + 4 * (tile0 + g4 + 8));
            const float ks0 = h2f(static_cast<uint16_t>(km0 & 0xffffu)), kz0 = h2f(static_cast<uint16_t>(km0 >> 16));
            const float ks1 = h2f(static_cast<uint16_t>(km1 & 0xffffu)), kz1 = h2f(static_cast<uint16_t>(km1 >> 16));
            const bool in0 = tok0 + g4 < L, in1 = tok0 + g4 + 8 < L;
            // scores in log2 units: scale * log2(e) * s_t * (q.c - z_t sum q)
            float x[4];
            x[0] = in0 && hv0 ? __fmul_rn(__fmul_rn(__fsub_rn(sc[0], __fmul_rn(kz0, qs0)), ks0), p.scale_log2) : -INFINITY;
            x[1] = in0 && hv1 ? __fmul_rn(__fmul_rn(__fsub_rn(sc[1], __fmul_rn(kz0, qs1)), ks0), p.scale_log2) : -INFINITY;
            x[2] = in1 && hv0 ? __fmul_rn(__fmul_rn(__fsub_rn(sc[2], __fmul_rn(kz1, qs0)), ks1), p.scale_log2) : -INFINITY;
            x[3] = in1 && hv1 ? __fmul_rn(__fmul_rn(__fsub_rn(sc[3], __fmul_rn(kz1, qs1)), ks1), p.scale_log2) : -INFINITY;
            // ---- online softmax over the tile (heads 2r, 2r + 1)
            float tmax[2] = {fmaxf(x[0], x[2]), fmaxf(x[1], x[3])};
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                tmax[0] = fmaxf(tmax[0], __shfl_xor_sync(0xffffffffu, tmax[0], o));
                tmax[1] = fmaxf(tmax[1], __shfl_xor_sync(0xffffffffu, tmax[1], o));
            }
            float alpha[2], mnew[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                mnew[e] = fmaxf(m_run[e], tmax[e]);
                alpha[e] = mnew[e] == -INFINITY ? 1.f : exp2f(m_run[e] - mnew[e]);
                m_run[e] = mnew[e];
            }
            float pr[4];
            pr[0] = x[0] == -INFINITY ? 0.f : exp2f(x[0] - mnew[0]);
            pr[1] = x[1] == -INFINITY ? 0.f : exp2f(x[1] - mnew[1]);
            pr[2] = x[2] == -INFINITY ? 0.f : exp2f(x[2] - mnew[0]);
            pr[3] = x[3] == -INFINITY ? 0.f : exp2f(x[3] - mnew[1]);
            // V weights p_t * s_t and their zero-point correction p_t s_t z_t
            const uint32_t vm0 = *reinterpret_cast<const uint32_t *>(ck + kVOff + kCodesBytes + 4 * (tile0 + g4));
            const uint32_t vm1 = *reinterpret_cast<const uint32_t *>(ck + kVOff + kCodesBytes + 4 * (tile0 + g4 + 8));
            const float vs0 = h2f(static_cast<uint16_t>(vm0 & 0xffffu)), vz0 = h2f(static_cast<uint16_t>(vm0 >> 16));
            const float vs1 = h2f(static_cast<uint16_t>(vm1 & 0xffffu)), vz1 = h2f(static_cast<uint16_t>(vm1 >> 16));
            // (masked tokens may sit in never-written slots: select, never multiply, their scales)
            const float w[4] = {pr[0] != 0.f ? __fmul_rn(pr[0], vs0) : 0.f, pr[1] != 0.f ? __fmul_rn(pr[1], vs0) : 0.f,
                                pr[2] != 0.f ? __fmul_rn(pr[2], vs1) : 0.f, pr[3] != 0.f ? __fmul_rn(pr[3], vs1) : 0.f};
            const float cz[4] = {w[0] != 0.f ? __fmul_rn(w[0], vz0) : 0.f, w[1] != 0.f ? __fmul_rn(w[1], vz0) : 0.f,
                                 w[2] != 0.f ? __fmul_rn(w[2], vz1) : 0.f, w[3] != 0.f ? __fmul_rn(w[3], vz1) : 0.f};
            float lsum[2] = {pr[0] + pr[2], pr[1] + pr[3]};
            float csum[2] = {cz[0] + cz[2], cz[1] + cz[3]};
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    lsum[e] += __shfl_xor_sync(0xffffffffu, lsum[e], o);
                    csum[e] += __shfl_xor_sync(0xffffffffu, csum[e], o);
                }
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                l_run[e] = __fmaf_rn(l_run[e], alpha[e], lsum[e]);
                c_run[e] = __fmaf_rn(c_run[e], alpha[e], csum[e]);
            }
            // rescale the PV accumulators by their head's alpha: column
            // 8n + 2r + e holds head hd = col (< G, hi part) or col - G (lo
            // part); its softmax state is component hd & 1 of the lanes of quad
            // column hd >> 1
            float ascale[NSV][2];
#pragma unroll
            for (int n = 0; n < NSV; ++n) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int col = 8 * n + 2 * r + e;
                    const int hd = col < G ? col : (col < 2 * G ? col - G : 0);
                    const float a0 = __shfl_sync(0xffffffffu, alpha[0], (lane & ~3) | (hd >> 1));
                    const float a1 = __shfl_sync(0xffffffffu, alpha[1], (lane & ~3) | (hd >> 1));
                    ascale[n][e] = (hd & 1) ? a1 : a0;
                }
            }
#pragma unroll
            for (int n = 0; n < NSV; ++n)
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    acc[n][mt][0] *= ascale[n][0];
                    acc[n][mt][1] *= ascale[n][1];
                    acc[n][mt][2] *= ascale[n][0];
                    acc[n][mt][3] *= ascale[n][1];
                }
            // transpose the weights through shared memory into the B layout
            // (k = tokens, n = columns): [token][head]
            pst[g4 * 8 + 2 * r] = w[0];
            pst[g4 * 8 + 2 * r + 1] = w[1];
            pst[(g4 + 8) * 8 + 2 * r] = w[2];
            pst[(g4 + 8) * 8 + 2 * r + 1] = w[3];
            __syncwarp();
            uint32_t pb[NSV][2];
#pragma unroll
            for (int n = 0; n < NSV; ++n) {
                const int col = 8 * n + g4;
                const bool hi_part = col < G, lo_part = col >= G && col < 2 * G;
                const int hd = hi_part ? col : (lo_part ? col - G : 0);
                float v4[4] = {pst[(2 * r) * 8 + hd], pst[(2 * r + 1) * 8 + hd], pst[(2 * r + 8) * 8 + hd],
                               pst[(2 * r + 9) * 8 + hd]};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float hv = __half2float(__float2half_rn(v4[e]));
                    v4[e] = hi_part ? hv : (lo_part ? __fsub_rn(v4[e], hv) : 0.f);
                }
                pb[n][0] = pack_f16x2(v4[0], v4[1]);
                pb[n][1] = pack_f16x2(v4[2], v4[3]);
            }
            __syncwarp();
            // ---- O^T += Vc^T (dims x tokens) * W (tokens x columns)
            const uint8_t *cv = ck + kVOff;
            const uint2 va = *reinterpret_cast<const uint2 *>(cv + (tile0 + 2 * r) * 64 + 8 * g4);
            const uint2 vb = *reinterpret_cast<const uint2 *>(cv + (tile0 + 2 * r + 1) * 64 + 8 * g4);
            const uint2 vc = *reinterpret_cast<const uint2 *>(cv + (tile0 + 2 * r + 8) * 64 + 8 * g4);
            const uint2 vd = *reinterpret_cast<const uint2 *>(cv + (tile0 + 2 * r + 9) * 64 + 8 * g4);
            // fp16x2 of (token 2r, token 2r+1) and (token 2r+8, token 2r+9) for
            // the 16 dims g4 + 8 nt, nt = 8 w + s
            uint32_t pa[16], pc[16];
#pragma unroll
            for (int ww = 0; ww < 2; ++ww) {
                const uint32_t xa = ww ? va.y : va.x, xb = ww ? vb.y : vb.x;
                const uint32_t xc = ww ? vc.y : vc.x, xd = ww ? vd.y : vd.x;
                const uint32_t lo_ab = __byte_perm(xa, xb, 0x5410), hi_ab = __byte_perm(xa, xb, 0x7632);
                const uint32_t lo_cd = __byte_perm(xc, xd, 0x5410), hi_cd = __byte_perm(xc, xd, 0x7632);
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4) {
                    pa[8 * ww + s4] = codes_f16x2(lo_ab >> (4 * s4));
                    pa[8 * ww + 4 + s4] = codes_f16x2(hi_ab >> (4 * s4));
                    pc[8 * ww + s4] = codes_f16x2(lo_cd >> (4 * s4));
                    pc[8 * ww + 4 + s4] = codes_f16x2(hi_cd >> (4 * s4));
                }
            }
            // every warp is done with this page slot (the V codes are in registers)
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const uint32_t af[4] = {pa[2 * mt], pa[2 * mt + 1], pc[2 * mt], pc[2 * mt + 1]};
#pragma unroll
                for (int n = 0; n < NSV; ++n) mma16816(acc[n][mt], af, pb[n][0], pb[n][1]);
            }
        }

        // ---- merge the four warps' states in shared memory (the ring is free
        // once every consumer passed its last page; the producer only waits
        // for copies it issued, which have all landed by then)
        named_bar_sync_kv(1, 32 * kConsumerWarps);
        float *mrg = reinterpret_cast<float *>(ring);  // [warp][G][2 + 128 + 1]: m, l, O..., c
        const int stride = 2 + kHD + 1;
        // column values of this lane: n-tile n, col 8n + 2r + e, dims g4 + 16 mt (+ 8)
#pragma unroll
        for (int n = 0; n < NSV; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int col = 8 * n + 2 * r + e;
                if (col < 2 * G) {
                    const int hd = col < G ? col : col - G;
                    float *dst = mrg + (warp * G + hd) * stride + 2;
                    if (col < G) {
#pragma unroll
                        for (int mt = 0; mt < 8; ++mt) {
                            dst[g4 + 16 * mt] = acc[n][mt][e];
                            dst[g4 + 8 + 16 * mt] = acc[n][mt][2 + e];
                        }
                    }
                }
            }
        named_bar_sync_kv(1, 32 * kConsumerWarps);
#pragma unroll
        for (int n = 0; n < NSV; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int col = 8 * n + 2 * r + e;
                if (col >= G && col < 2 * G) {
                    float *dst = mrg + (warp * G + col - G) * stride + 2;
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        dst[g4 + 16 * mt] += acc[n][mt][e];
                        dst[g4 + 8 + 16 * mt] += acc[n][mt][2 + e];
                    }
                }
            }
        if (g4 == 0) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int hd = 2 * r + e;
                if (hd < G) {
                    float *dst = mrg + (warp * G + hd) * stride;
                    dst[0] = m_run[e];
                    dst[1] = l_run[e];
                    dst[2 + kHD] = c_run[e];
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
                const float f = src[0] == -INFINITY ? 0.f : exp2f(src[0] - M);
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

constexpr size_t kAttnSmem = 128 + kStages * kChunkBytes + kConsumerWarps * 128 * 4 + 2 * kStages * 8 + 16;

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

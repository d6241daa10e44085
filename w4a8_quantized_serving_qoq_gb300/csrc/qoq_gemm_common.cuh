// Pieces shared by the two W4A8 GEMM kernels (fp16-operand and fp8-operand
// tensor-core paths): kernel parameters, the persistent stream-K schedule,
// the output write, small shared-memory helpers and the tensor-map encoder.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include <mutex>

#include "qoq_device.cuh"
#include "qoq_internal.h"

namespace qoq {
namespace {

struct GemmParams {
    const uint8_t *packed;
    const uint16_t *s_x;
    const int32_t *t_x;
    const uint16_t *s_w;
    uint16_t *O;
    int32_t *acc_out;
    uint32_t *status;
    uint32_t *counters;     // [ctas] arrival counters of split tiles
    int32_t *slots;         // [ctas][BT][128] int32 partial tiles
    int M, N, K, group, G;
    int tok_tiles;
    long long total;        // tiles * G stages
    int ctas;
    int dp_tiles;           // work tiles [0, dp_tiles) go whole to CTAs round-robin; the rest is stream-K
    int band;               // weight tiles per band of the tile order (0: token-tile fastest)
    uint32_t debug_flags;
    uint64_t timeout_ns;
#ifdef QOQ_DEBUG_BOUNDS
    // Buffer extents (bounds-check build only: the release kernels keep the
    // smaller parameter block): bytes of the packed weights, int32 words of
    // the slot array, arrival counters.
    unsigned long long packed_bytes, slot_words, n_counters;
#endif
};

// The extents above from the workspace layout of a plan (slot array and
// counters as the plan laid them out, not as the kernel would compute them).
inline void set_extents(GemmParams &p, const GemmPlan &plan, int N, int K, int group) {
#ifdef QOQ_DEBUG_BOUNDS
    p.packed_bytes = packed_bytes(N, K, group);
    p.n_counters = (plan.slots_offset - plan.counters_offset) / 4;
    p.slot_words = plan.zero_bytes > plan.slots_offset ? (plan.zero_bytes - plan.slots_offset) / 4 : 0;
#else
    (void)p, (void)plan, (void)N, (void)K, (void)group;
#endif
}

// Bounds-check build: bytes [off, off + n) of the packed weights.
__device__ __forceinline__ bool weights_in_bounds(const GemmParams &p, unsigned long long off, unsigned long long n) {
#ifdef QOQ_DEBUG_BOUNDS
    return in_bounds(off, n, p.packed_bytes, p.status);
#else
    return true;
#endif
}

// Bounds-check build: one split tile's slot (all its rows) and its arrival
// counter.  A failure is recorded by in_bounds; the caller raises the abort.
template <int BT>
__device__ __forceinline__ bool slot_in_bounds(const GemmParams &p, int slot_idx) {
#ifdef QOQ_DEBUG_BOUNDS
    return in_bounds(static_cast<unsigned long long>(slot_idx) * (BT * kTileN), BT * kTileN, p.slot_words, p.status) &&
           in_bounds(static_cast<unsigned long long>(slot_idx), 1, p.n_counters, p.status);
#else
    return true;
#endif
}

__device__ __forceinline__ float h2f(uint16_t b) { return __half2float(__ushort_as_half(b)); }

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Persistent schedule, data-parallel then stream-K.  The first dp_tiles
// tiles (a multiple of the CTA count, used when there are at least two waves
// of tiles) go whole to the CTAs round-robin: CTA c takes tiles c, c + P,
// c + 2P, ..., so the CTAs running at one time work on consecutive tiles,
// which share weight and activation tiles in L2.  The remaining tiles x G
// k-stages are cut into P contiguous, equal ranges; CTA c owns
// [base + c R / P, base + (c + 1) R / P), base = dp_tiles G, R = the remaining
// stages.  A range crosses tile boundaries; each piece inside one tile is a
// segment.  Positions map to tiles through tile_at (the banded order).
struct Segment {
    int seq;   // position in the work order (stage indices are seq * G + k)
    int tile;  // the output tile: token tile tile % tok_tiles, weight tile tile / tok_tiles
    int k0, k1;
};

// The tile at position j of the work order.  With band = 0 the order is
// token-tile fastest (tile j).  Otherwise the weight tiles form bands of
// `band` tiles; a band's tiles come weight-tile fastest, so P consecutive
// positions (the tiles CTAs work on at one time) cover about band weight
// tiles x P / band token tiles, a working set of band * (weight tile) +
// (P / band) * (activation tile) that the planner keeps inside L2.
__device__ __forceinline__ int tile_at(uint32_t j, const GemmParams &p) {
    if (p.band <= 0) return static_cast<int>(j);
    const uint32_t tt = static_cast<uint32_t>(p.tok_tiles), nt = static_cast<uint32_t>(p.N / kTileN);
    const uint32_t bw = static_cast<uint32_t>(p.band), per_band = bw * tt;
    const uint32_t b = j / per_band, r = j - b * per_band;
    const uint32_t w = (b + 1) * bw <= nt ? bw : nt - b * bw;  // the last band may be narrower
    const uint32_t tok = r / w, n = b * bw + (r - tok * w);
    return static_cast<int>(n * tt + tok);
}

struct SegmentWalker {
    uint32_t dp_next, dp_end, dp_step;
    uint32_t w, w1, G;  // total stages < 2^31 (checked on the host)
    // ctas * total < 2^32 (checked on the host), so 32-bit arithmetic is exact.
    __device__ SegmentWalker(const GemmParams &p, int cta)
        : dp_next(static_cast<uint32_t>(cta)), dp_end(static_cast<uint32_t>(p.dp_tiles)),
          dp_step(static_cast<uint32_t>(p.ctas)), G(static_cast<uint32_t>(p.G)), pp(&p) {
        const uint32_t base = static_cast<uint32_t>(p.dp_tiles) * G;
        const uint32_t R = static_cast<uint32_t>(p.total) - base;
        w = base + static_cast<uint32_t>(cta) * R / static_cast<uint32_t>(p.ctas);
        w1 = base + static_cast<uint32_t>(cta + 1) * R / static_cast<uint32_t>(p.ctas);
    }
    __device__ bool next(Segment &s) {
        if (dp_next < dp_end) {
            s.seq = static_cast<int>(dp_next);
            s.tile = tile_at(dp_next, *pp);
            s.k0 = 0;
            s.k1 = static_cast<int>(G);
            dp_next += dp_step;
            return true;
        }
        if (w >= w1) return false;
        const uint32_t t = w / G;
        s.seq = static_cast<int>(t);
        s.tile = tile_at(t, *pp);
        s.k0 = static_cast<int>(w - t * G);
        const uint32_t end = w1 - t * G;
        s.k1 = static_cast<int>(end < G ? end : G);
        w = t * G + static_cast<uint32_t>(s.k1);
        return true;
    }
    const GemmParams *pp;
};

// CTA whose stream-K range holds global stage `s` (s in the stream-K part:
// only split tiles ask, and every split tile lies there).
__device__ __forceinline__ int cta_of_stage(uint32_t s, const GemmParams &p) {
    const uint32_t base = static_cast<uint32_t>(p.dp_tiles) * static_cast<uint32_t>(p.G);
    const uint32_t R = static_cast<uint32_t>(p.total) - base;
    return static_cast<int>(((s - base + 1) * static_cast<uint32_t>(p.ctas) - 1) / R);
}

// Split-tile completion, decided by one thread: true when every other
// contributor of the tile has published its partial (arrival counter ==
// number of other contributors), so this CTA can finish the tile with its own
// partial still on chip.  The contributor that owns the tile's first k-stage
// processes its part at the end of its range, about when contributors whose
// whole range lies in the tile finish theirs, so it waits for them, bounded
// (then it publishes instead).  No wait cycle exists: a CTA publishes the
// partial of its first segment (processed at the start of its range) before
// it can wait at the end, and only first-stage owners wait.
constexpr uint64_t kFinishWaitNs = 10000;

__device__ __forceinline__ bool finish_directly(const GemmParams &p, int cta, int slot_idx, uint32_t tfirst,
                                                volatile int *abort_flag) {
    const uint32_t others =
        static_cast<uint32_t>(cta_of_stage(tfirst + static_cast<uint32_t>(p.G) - 1u, p) - slot_idx);
    if (ld_acquire_gpu_u32(p.counters + slot_idx) == others) return true;
    if (cta != slot_idx) return false;
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < kFinishWaitNs) {
        __nanosleep(256);
        if (*abort_flag) return false;
        if (ld_acquire_gpu_u32(p.counters + slot_idx) == others) return true;
    }
    return false;
}

// Final output of one accumulator: per-channel zero fold, then either the
// int32 value (test mode) or fp16(acc * s_x[m] * s_w[n]).
__device__ __forceinline__ void write_out(const GemmParams &p, int m, int n, int acc, int zc, int tx,
                                          float sx, float sw) {
    const size_t idx = static_cast<size_t>(m) * p.N + n;
    if (!in_bounds(idx, 1, static_cast<unsigned long long>(p.M) * p.N, p.status)) return;
    acc -= zc * tx;
    if (p.acc_out)
        p.acc_out[idx] = acc;
    else
        p.O[idx] = __half_as_ushort(__float2half_rn(__fmul_rn(__fmul_rn(static_cast<float>(acc), sx), sw)));
}

// Staging stores: no memory clobber, so a run of them pipelines; the
// proxy fence and barrier that follow them are volatile asm too and stay after.
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v));
}

__device__ __forceinline__ void st_shared_b32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v));
}

// Sixteen consecutive 32-bit shared-memory words (16-byte aligned) into registers.
__device__ __forceinline__ void ld_shared_x16(uint32_t addr, uint32_t (&r)[16]) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(r[4 * q]), "=r"(r[4 * q + 1]), "=r"(r[4 * q + 2]), "=r"(r[4 * q + 3])
                     : "r"(addr + 16u * q));
}

// fp16 output of one accumulator (per-channel zero fold, then the two scales).
__device__ __forceinline__ uint16_t out_fp16(int acc, int zc, int tx, float sx, float sw) {
    return __half_as_ushort(__float2half_rn(__fmul_rn(__fmul_rn(static_cast<float>(acc - zc * tx), sx), sw)));
}

__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ int ld_shared_s32(uint32_t addr) {
    int v;
    asm volatile("ld.shared.s32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ int ld_cg_s32(const int32_t *p) {
    int v;
    asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

using CUtensorMapEncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                              const cuuint64_t *, const cuuint64_t *,
                                              const cuuint32_t *, const cuuint32_t *,
                                              CUtensorMapInterleave, CUtensorMapSwizzle,
                                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

CUtensorMapEncodeTiledFn get_encode_fn() {
    static CUtensorMapEncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult qres;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &qres) == cudaSuccess &&
            qres == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CUtensorMapEncodeTiledFn>(ptr);
    });
    return fn;
}

}  // namespace
}  // namespace qoq

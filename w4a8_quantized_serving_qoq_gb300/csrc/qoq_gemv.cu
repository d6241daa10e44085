// W4A8 GEMM for decode batches (M <= 8) on the CUDA cores: the GEMV regime,
// where a launch streams the 4-bit weights once and does a handful of
// multiply-adds per weight.
//
// Sources: "QServe: W4A8KV4 Quantization and System Co-design for Efficient
// LLM Serving" (papercache summary), sections "逐组W4A8 GEMM中的快速反量化"
// (dequantization in byte lanes, multiply then subtract, legal under the
// protective range) and "逐通道W4A8 GEMM中的快速反量化" (eq. 13: the zero
// folded out of the main loop through t_x); "QServe：把 W4A8KV4 的理论收益做
// 成实测吞吐的量化—系统协同设计" (zenmind review) 3.2: for small m, slice the
// reduction dimension and reduce the partial sums on chip.
//
// GB300 design:
//  * one lane per weight row: a 128-row tile of the packed weights is read
//    by four warps as 512-byte coalesced rows of 16-byte chunks (the packed
//    block order), non-allocating in L1;
//  * one 32-bit multiply-add per 4 weights gives (q4 - z) * s_g + 128 in each
//    byte (no carries: the protective range keeps (q4 - z) s_g in
//    [-127, 127]); dp4a.u32.s32 multiplies the four biased weights with four
//    INT8 activations and accumulates in exact int32; the bias comes out as
//    128 * (sum of the group's activations), computed once per CTA;
//    per-channel weights need no dequantization at all (raw q4, then
//    - z * t_x at the end);
//  * the K dimension is split over the CTAs of a thread-block cluster and over
//    two warp groups in each CTA; the int32 partial sums are reduced across
//    the cluster through distributed shared memory: each CTA adds its sums
//    into the CTA that finishes their rows (every CTA finishes an equal share
//    of the tile's rows), so no partial sum leaves the chip and no workspace
//    round trip or split-tile tail follows;
//  * under programmatic dependent launch the weights of the first blocks are
//    loaded before the wait for the preceding kernel (weights are static).
#include <cuda.h>
#include <cuda_fp16.h>

#include <mutex>

#include "qoq_device.cuh"
#include "qoq_internal.h"

namespace qoq {
namespace {

constexpr int kGvThreads = 256;  // 8 warps: rows 32 (w % 4) .. +31 of the tile, K half w / 4

struct GemvParams {
    const uint8_t *packed;
    const int8_t *Qx;
    const uint16_t *s_x;
    const int32_t *t_x;
    const uint16_t *s_w;
    uint16_t *O;
    int32_t *acc_out;
    uint32_t *status;
    int M, N, K, group, G;
    int csize;     // CTAs per cluster: the K split
    int nb_max;    // blocks (128 k) per CTA, at most
#ifdef QOQ_DEBUG_BOUNDS
    unsigned long long packed_bytes;  // extent of the packed weights (bounds-check build only)
#endif
};

__device__ __forceinline__ float h2f_gv(uint16_t b) { return __half2float(__ushort_as_half(b)); }

__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const void *p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The two halves of a cluster barrier, so that work can run between them.
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// *local (the same offset in CTA `rank` of the cluster) += v, in that CTA's
// shared memory.
__device__ __forceinline__ void red_dsmem_add_s32(int *local, uint32_t rank, int v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("red.shared::cluster.add.s32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}

// One packed 128 x 128 block as this lane (weight row r) sees it.
struct BlockRegs {
    uint4 c[4];     // k = 32 p .. 32 p + 31, p = 0..3
    uint32_t meta;  // s_g | z << 8 | code sum << 16 (group mode)
};

__device__ __forceinline__ void load_block(BlockRegs &br, const uint8_t *blk, int r, bool group) {
#pragma unroll
    for (int p4 = 0; p4 < 4; ++p4) br.c[p4] = ld_stream_v4(blk + 16 * (p4 * 128 + r));
    br.meta = group ? ld_stream_u32(blk + kCodeBytes + 4 * r) : 0u;
}

// kAhead: weight blocks in flight ahead of the one being multiplied (2; or
// 1 for a single token when each warp has at most two blocks: they are all
// requested before the dependency wait either way, and the fewer registers
// let four CTAs share an SM, so the CTAs of a launch fit beside the
// running one and start early).
template <int MT, int kAhead>
__global__ void __launch_bounds__(kGvThreads, (MT == 1 && kAhead == 1) ? 4 : (MT <= 4 ? 3 : 2))
    w4a8_gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(16) uint8_t gv_smem[];
    const int nbm = p.nb_max;
    uint32_t *xs = reinterpret_cast<uint32_t *>(gv_smem);                    // [MT][nbm * 32] words of Qx
    int *gsum = reinterpret_cast<int *>(gv_smem + MT * nbm * 128);           // [MT][nbm]
    int *part = gsum + MT * nbm;  // [2 K halves][MT][128] sums; with a cluster [MT][128 / csize] totals
    __shared__ int hdr_ok;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = 32 * (warp & 3) + lane;  // weight row in the tile
    const int half = warp >> 2;
    const int tile = blockIdx.y;
    const uint32_t crank = p.csize > 1 ? cluster_rank() : 0u;
    const bool group = p.group != 0;
    const uint32_t bb = block_bytes(p.group);
    // blocks of this CTA, then of this warp's K half
    const int kb0 = static_cast<int>(crank) * p.G / p.csize, kb1 = (static_cast<int>(crank) + 1) * p.G / p.csize;
    const int nb = kb1 - kb0;
    const int hmid = kb0 + nb / 2;
    const int wb0 = half ? hmid : kb0;
    int wb1 = half ? kb1 : hmid;
    const uint8_t *tile_base = p.packed + kHeaderBytes + static_cast<size_t>(tile) * p.G * bb;

    // The header is checked before any weight is read (a call whose N or K
    // disagrees with the buffer must not read past it).  The decision is the
    // same in every CTA of every cluster, so none reaches a cluster barrier.
    if (threadIdx.x == 0) {
        griddep_launch_dependents();
        const PackedHeader *h = reinterpret_cast<const PackedHeader *>(p.packed);
        hdr_ok = (h->magic == kPackedMagic && h->version == kPackedVersion && h->N == p.N && h->K == p.K &&
                  h->group == p.group && h->illegal == 0u) ? 1 : 0;
    }
    for (int idx = threadIdx.x; idx < MT * nbm; idx += kGvThreads) gsum[idx] = 0;
    __syncthreads();
    if (!hdr_ok) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) {
            griddep_wait();  // the status word may still be in use by the preceding kernel
            atomicOr(p.status, kStatusBadPacked);
        }
        return;
    }
    // Bounds-check build: a weight range outside the buffer is skipped (the
    // CTA still takes every cluster barrier, with zero sums).
#ifdef QOQ_DEBUG_BOUNDS
    if (!in_bounds(kHeaderBytes + (static_cast<unsigned long long>(tile) * p.G + wb0) * bb,
                   static_cast<unsigned long long>(wb1 - wb0) * bb, p.packed_bytes, p.status))
        wb1 = wb0;
#endif
    const int rows = 128 / p.csize, row0 = static_cast<int>(crank) * rows;  // the tile rows this CTA finishes
    if (p.csize > 1) {
        // Every CTA of the cluster adds its sums of this CTA's rows into this
        // CTA's totals: zero them, and let the peers know (the barrier's
        // wait comes only before the adds).
        for (int idx = threadIdx.x; idx < MT * rows; idx += kGvThreads) part[idx] = 0;
        cluster_arrive();
    }
    // Weights are static: the first two blocks stream in while the preceding
    // kernel finishes.  The loop keeps two blocks in flight ahead of the one
    // it multiplies (the weight stream is bound by bytes in flight x latency:
    // with one block ahead a 4096 x 16384 launch ran at 3.8 TB/s).
    BlockRegs cur{}, nx1{}, nx2{};
    if (wb0 < wb1) load_block(cur, tile_base + static_cast<size_t>(wb0) * bb, r, group);
    if (wb0 + 1 < wb1) load_block(nx1, tile_base + static_cast<size_t>(wb0 + 1) * bb, r, group);
    static_assert(kAhead == 1 || kAhead == 2, "blocks ahead");
    griddep_wait();
    // This CTA's activations [M][nb * 128] into shared memory (tokens >= M read as 0),
    // and per (token, block) the sum of its 128 activations (the bias of the
    // biased weight bytes), gathered with shared-memory atomics.
    const int words = nb * 32;
    for (int idx = threadIdx.x; idx < MT * words / 4; idx += kGvThreads) {
        const int m = idx / (words / 4), q = idx % (words / 4);
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (m < p.M) {
            v = __ldg(reinterpret_cast<const uint4 *>(p.Qx + static_cast<size_t>(m) * p.K + kb0 * 128) + q);
            if (group) {
                const int t = __dp4a(static_cast<int>(v.x), 0x01010101,
                                     __dp4a(static_cast<int>(v.y), 0x01010101,
                                            __dp4a(static_cast<int>(v.z), 0x01010101,
                                                   __dp4a(static_cast<int>(v.w), 0x01010101, 0))));
                atomicAdd(gsum + m * nbm + q / 8, t);
            }
        }
        reinterpret_cast<uint4 *>(xs + m * nbm * 32)[q] = v;
    }
    __syncthreads();

    int acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0;
    for (int b = wb0; b < wb1; ++b) {
        if constexpr (kAhead == 2)
            if (b + 2 < wb1) load_block(nx2, tile_base + static_cast<size_t>(b + 2) * bb, r, group);
        const int jb = b - kb0;  // block index inside the CTA's activation slice
        const uint32_t s = group ? (cur.meta & 0xffu) : 1u;
        const uint32_t z = group ? ((cur.meta >> 8) & 0xffu) : 0u;
        // group mode: bytes (q - z) s + 128; per-channel: the raw codes q
        const uint32_t cst = group ? static_cast<uint32_t>(128 - static_cast<int>(z * s)) * 0x01010101u : 0u;
#pragma unroll
        for (int p4 = 0; p4 < 4; ++p4) {
            const uint32_t w4[4] = {cur.c[p4].x, cur.c[p4].y, cur.c[p4].z, cur.c[p4].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t ulo = (w4[j] & 0x0F0F0F0Fu) * s + cst;         // k = 32 p + 8 j + 0..3
                const uint32_t uhi = ((w4[j] >> 4) & 0x0F0F0F0Fu) * s + cst;  // k = 32 p + 8 j + 4..7
                const int wi = jb * 32 + 8 * p4 + 2 * j;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (m < p.M) {
                        const uint2 x = *reinterpret_cast<const uint2 *>(xs + m * nbm * 32 + wi);
                        acc[m] = dp4a_us(ulo, x.x, acc[m]);
                        acc[m] = dp4a_us(uhi, x.y, acc[m]);
                    }
                }
            }
        }
        if (group) {
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[m] -= 128 * gsum[m * nbm + jb];
        }
        cur = nx1;
        if constexpr (kAhead == 2) {
            nx1 = nx2;
        } else {
            if (b + 2 < wb1) load_block(nx1, tile_base + static_cast<size_t>(b + 2) * bb, r, group);
        }
    }

    // ---- reduction of the K split.  With a cluster, each thread adds its
    // sums into the totals of the CTA that finishes its row (a shared-memory
    // reduction in that CTA, through distributed shared memory), so after one
    // barrier every CTA holds the complete sums of its share of the rows.
    // Without one, the two K halves meet in this CTA's shared memory.
    if (p.csize > 1) {
        cluster_wait();  // every CTA of the cluster has zeroed its totals
        const uint32_t owner = static_cast<uint32_t>(r / rows);
        const int rr = r % rows;
#pragma unroll
        for (int m = 0; m < MT; ++m)
            if (m < p.M) red_dsmem_add_s32(part + m * rows + rr, owner, acc[m]);
        cluster_arrive();
        cluster_wait();  // every addition into this CTA's totals has landed
    } else {
#pragma unroll
        for (int m = 0; m < MT; ++m) part[(half * MT + m) * 128 + r] = acc[m];
        __syncthreads();
    }
    for (int idx = threadIdx.x; idx < MT * rows; idx += kGvThreads) {
        const int m = idx / rows, rl = idx % rows, rr = row0 + rl;
        if (m >= p.M) continue;
        const int tot = p.csize > 1 ? part[m * rows + rl] : part[m * 128 + rr] + part[(MT + m) * 128 + rr];
        const int n = tile * 128 + rr;
        int res = tot;
        if (!group) res -= static_cast<int>(p.packed[packed_z_offset(p.N, p.K) + n]) * p.t_x[m];
        const size_t idx_o = static_cast<size_t>(m) * p.N + n;
        if (!in_bounds(idx_o, 1, static_cast<unsigned long long>(p.M) * p.N, p.status)) continue;
        if (p.acc_out)
            p.acc_out[idx_o] = res;
        else
            p.O[idx_o] = __half_as_ushort(__float2half_rn(
                __fmul_rn(__fmul_rn(static_cast<float>(res), h2f_gv(p.s_x[m])), h2f_gv(p.s_w[n]))));
    }
}

template <int MT, int kAhead>
cudaError_t launch_gemv_mt(const GemmArgs &a, const GemmPlan &plan, cudaStream_t stream) {
    const int nb_max = (plan.G + plan.gv_csize - 1) / plan.gv_csize;
    const size_t smem = static_cast<size_t>(MT) * nb_max * 128 + static_cast<size_t>(MT) * nb_max * 4 +
                        2 * static_cast<size_t>(MT) * 128 * 4;  // activations, group sums, two halves' sums
    static std::mutex mu;
    static size_t configured[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (configured[dev] < smem) {
            e = cudaFuncSetAttribute(w4a8_gemv_kernel<MT, kAhead>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem));
            if (e != cudaSuccess) return e;
            configured[dev] = smem;
        }
    }
    GemvParams p;
    p.packed = static_cast<const uint8_t *>(a.packed);
    p.Qx = a.Qx;
    p.s_x = a.s_x;
    p.t_x = a.t_x;
    p.s_w = a.s_w;
    p.O = a.O;
    p.acc_out = a.acc_out;
    p.status = static_cast<uint32_t *>(a.ws);
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.group = a.group;
    p.G = plan.G;
    p.csize = plan.gv_csize;
    p.nb_max = nb_max;
#ifdef QOQ_DEBUG_BOUNDS
    p.packed_bytes = packed_bytes(a.N, a.K, a.group);
#endif
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.gv_csize, plan.n_tiles);
    cfg.blockDim = dim3(kGvThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (plan.gv_csize > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = static_cast<unsigned>(plan.gv_csize);
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (a.pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = na ? attr : nullptr;
    cfg.numAttrs = static_cast<unsigned>(na);
    return cudaLaunchKernelEx(&cfg, w4a8_gemv_kernel<MT, kAhead>, p);
}

}  // namespace

cudaError_t launch_gemv(const GemmArgs &a, const GemmPlan &plan, cudaStream_t stream) {
    switch (plan.BT) {
        case 1: {
            // at most two blocks per warp (its K half of the CTA's blocks): one ahead suffices
            const int nb_max = (plan.G + plan.gv_csize - 1) / plan.gv_csize;
            return (nb_max + 1) / 2 <= 2 ? launch_gemv_mt<1, 1>(a, plan, stream) : launch_gemv_mt<1, 2>(a, plan, stream);
        }
        case 2: return launch_gemv_mt<2, 2>(a, plan, stream);
        case 4: return launch_gemv_mt<4, 2>(a, plan, stream);
        case 8: return launch_gemv_mt<8, 2>(a, plan, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qoq

// W4A8 GEMM for sm_103a: O[m,n] = s_x[m] * s_w[n] * sum_k Qx[m,k] * w8[n,k],
// w8 = (q4 - z) * s_g (progressive group quantization, g = 128), or
// w8 = q4 with the zero folded into the epilogue (per-channel variant).
//
// Sources: "QServe: W4A8KV4 Quantization and System Co-design for Efficient
// LLM Serving" (papercache summary), sections "逐通道W4A8 GEMM中的快速反量化"
// (eq. 13) and "逐组W4A8 GEMM中的快速反量化"; "QServe：把 W4A8KV4 的理论收益做成
// 实测吞吐的量化—系统协同设计" (zenmind review), sections 3.2 and 4 (step 3).
//
// GB300 design (sm_103a has no tcgen05 INT8 MMA, so the exact integer
// product runs on the fp16 tensor-core path):
//  * swap-AB: the MMA's M = 128 weight rows, its N = BT tokens (16..128);
//  * two warps stream the stages with TMA into two rings: warp 0 one bulk
//    copy of the packed 8 KB weight block (+ 512 B of group metadata) per
//    stage into a deep weight ring, without waiting for the preceding
//    kernel; warp 3, after that wait, two 2D tensor copies of the
//    activation operand (Qx as exact fp16, written by the activation
//    quantizer or by a preparation kernel) straight into the MMA's B layout
//    (128-byte swizzle, rows past M zero-filled) in a shorter ring;
//  * 8 converter warps turn weight codes into fp16 operands in registers
//    with byte-lane SIMD: one 32-bit multiply-add per 4 weights yields
//    (q4 - z) * s_g + 128 in each byte (legal because the protective range
//    keeps every product in [-128, 127]), then byte -> fp16 by exponent
//    splicing and one fp16x2 subtract, stored to TMEM as the A operand
//    (per-channel weights: the raw codes as fp16 subnormals, see kPC);
//  * two threads issue tcgen05.mma on alternate stages (kind::f16, fp32
//    accumulation in TMEM).  Operands are integers with |product| <= 127 *
//    128, so an fp32 sum over 1024 k (8 stages) stays below 2^24 and is exact
//    in any order; each 1024-k chunk is drained by the epilogue warps into
//    int32 sums held in their registers (one weight row per thread, all BT
//    tokens), which also hand the chunk buffer back zeroed at once (two chunk
//    buffers so the MMAs never wait on the drain);
//  * epilogue: int32 result (per-channel: minus z[n] * t_x[m]) scaled by
//    s_x[m] * s_w[n] in fp32 and rounded to fp16, staged in shared memory 16
//    tokens at a time and written by a tensor bulk store; with a K split, the
//    int32 partials of 16 tokens (8 KB, contiguous in the tile's workspace
//    slot) go out as one bulk reduce-add, and the last CTA of a tile applies
//    the epilogue and re-zeroes the slot with bulk copies of a zero block.
//  * every wait is bounded; on expiry the kernel records kStatusTimeout in the
//    workspace status word, drains its own copies/MMAs and frees TMEM.
#include <cuda.h>
#include <cuda_fp16.h>

#include <cmath>
#include <mutex>

#include "qoq_gemm_common.cuh"

namespace qoq {
namespace {

constexpr int kThreads = 512;          // 16 warps
constexpr int kConvThreads = 256;      // warps 8..15: two groups of 4 warps
constexpr int kConvWarps = kConvThreads / 32;
constexpr int kConvGroupWarps = kConvWarps / 2;  // one group converts one stage
constexpr int kEpiWarps = 4;           // warps 4..7
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kChunkStages = 8;        // 8 x 128 k = 1024 k per exact fp32 chunk
constexpr uint32_t kWRawBytes = 9216;  // 8704 B block slot rounded to 1 KB

template <int BT>
struct Cfg {
    // TMEM columns: two fp32 chunk accumulators of BT columns from kChunk0
    // (the int32 sums live in the epilogue threads' registers), then
    // kOpStages fp16 weight operand slots of 64 columns (128 lanes x 64
    // columns = 128 rows x 128 k each) from kA0.
    static constexpr int kOpStages = 4;
    // Two rings of TMA stages: packed weight blocks (kWStages slots of
    // kWRawBytes, released by the converters once read into registers) and
    // the B operand (kBStages slots, released by the MMAs' commit).  The
    // weight ring runs far ahead of the MMAs to cover HBM latency; the
    // activation operand comes from L2.
    static constexpr int kWStages = BT == 128 ? 10 : (BT == 64 ? 12 : 14);
    static constexpr int kBStages = BT == 16 ? 8 : (BT == 32 ? 6 : (BT == 64 ? 4 : 3));
    static constexpr uint32_t kChunk0 = 0;
    static constexpr uint32_t kA0 = ((kChunk0 + 2 * BT + 63) / 64) * 64;
    static constexpr uint32_t kTmemCols = 512;
    // Registers per thread by warpgroup for BT >= 64 (the epilogue holds BT
    // int32 sums per thread): warps 0-3 (TMA producers, MMA issuers) give up
    // registers to warps 4-7 (epilogue); the converters keep the launch
    // allocation.  128 x 80 + 128 x 176 + 256 x 128 = 512 x 128, the launch
    // allocation, which the host checks before the first launch.
    static constexpr bool kRegSplit = BT >= 64;
    static constexpr uint32_t kRegLow = 80, kRegEpi = 176, kRegLaunch = 128;
    static_assert(128 * kRegLow + 128 * kRegEpi + 256 * kRegLaunch == 512 * kRegLaunch, "register split");
    // B slot: two 128-byte-swizzled atoms of BT rows x 64 fp16 (k 0..63,
    // k 64..127), landed by TMA from the fp16 activation operand.
    static constexpr uint32_t kBAtom = static_cast<uint32_t>(BT) * 128u;
    static constexpr uint32_t kBBytes = 2 * kBAtom;
    static constexpr int kNumBars = 2 * kWStages + 2 * kBStages + 2 * kOpStages + 4 + 1 + 2;
    // Epilogue staging: two 8 KB buffers (16 tokens x 128 rows of int32
    // partials or fp16 outputs, written by the epilogue threads and sent out
    // by one bulk copy each; during a split-tile fix-up they receive slot rows
    // by bulk loads), an 8 KB block of zeros that re-zeroes partial slots,
    // and two 4 KB fp16 output buffers for the fix-up.
    static constexpr uint32_t kStgBytes = 8192;
    static constexpr uint32_t kStgRegion = 4 * kStgBytes;
    static constexpr uint32_t kMiscBytes = 2048;  // barriers + flags, then s_x / t_x of the current tile
    static constexpr uint32_t kSmemBytes =
        kBStages * kBBytes + kWStages * kWRawBytes + kStgRegion + kMiscBytes + 1024;
    static_assert(kA0 + 64 * kOpStages <= kTmemCols, "TMEM columns");
    // The converter groups and the MMA issuers alternate stages; with even
    // depths every weight slot and operand slot is waited on by one group (or
    // one issuer) in stage order, which keeps their parity waits exact.
    static_assert(kWStages % 2 == 0 && kOpStages % 2 == 0, "even weight-ring and operand-slot depths");
    static_assert(kWRawBytes % 1024 == 0 && kBAtom % 1024 == 0, "1 KB aligned swizzled atoms");
    static_assert(kNumBars * 8 + 64 <= 1024, "barrier area (the tile scales start at +1024)");
    static_assert(kSmemBytes <= 232448, "shared memory");
};

// int32 test output of one block of 16 tokens for this thread's weight row:
// the values were stored to this thread's own slots (token i at 4*(i*128+et))
// of the buffer at buf; one rolled loop keeps the epilogue's code small.
__device__ __forceinline__ void write_block_i32(const GemmParams &p, uint32_t buf, int m0j, int n, int zc,
                                             const float *sx16, const int *tx16, float sw, bool live) {
    const int et = static_cast<int>(threadIdx.x) - 128;
#pragma unroll 1
    for (int i = 0; i < 16; ++i) {
        const int m = m0j + i;
        if (live && m < p.M) write_out(p, m, n, ld_shared_s32(buf + 4u * (i * kTileN + et)), zc, tx16[i], sx16[i], sw);
    }
}

// D[tmem] += A[tmem] * B[smem desc]^T (kind::f16, accumulating), the B
// descriptor passed as its two 32-bit words.
__device__ __forceinline__ void mma_f16_tmem_a_acc(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                                   uint32_t idesc) {
    asm volatile(
        "{\n .reg .pred p;\n .reg .b64 bd;\n setp.ne.b32 p, 1, 0;\n mov.b64 bd, {%2, %3};\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, p;\n}\n"
        ::"r"(d_tmem), "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc)
        : "memory");
}

// Four INT8 / biased bytes -> two fp16x2 words holding the signed values.
// Input byte b is v + 128 (v in [-128, 127]); 0x64XX is the fp16 1024 + XX.
__device__ __forceinline__ void biased_bytes_to_f16x4(uint32_t u, uint32_t &lo, uint32_t &hi) {
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140u);
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342u);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u));  // 1152
    const __half2 ha = __hsub2(*reinterpret_cast<const __half2 *>(&a), bias);
    const __half2 hb = __hsub2(*reinterpret_cast<const __half2 *>(&b), bias);
    lo = *reinterpret_cast<const uint32_t *>(&ha);
    hi = *reinterpret_cast<const uint32_t *>(&hb);
}

// kAccOut: the int32 test output (GemmParams::acc_out) instead of fp16 O.  A
// separate instantiation, so that the fp16 kernel carries no code for it.
// kPC: per-channel weights (group == 0).  Their raw codes q in [0, 15] enter
// the MMA as fp16 subnormals (the byte q in the low bits of a half is exactly
// q * 2^-24, so a byte permute with zero bytes is the whole conversion); a
// chunk's sums, at most 1024 * 15 * 127 * 2^-24, stay exact in fp32, and the
// drain scales them back by 2^24.  (The g128 codes carry the bias 128 of the
// byte-lane dequantization, which would limit an exact chunk to 512 k.)
template <int BT, bool kAccOut, bool kPC>
__global__ void __launch_bounds__(kThreads, 1)
    w4a8_gemm_kernel(const __grid_constant__ CUtensorMap qx_map, const __grid_constant__ CUtensorMap o_map,
                     const GemmParams p) {
    using C = Cfg<BT>;
    constexpr int RW = C::kWStages;
    constexpr int RB = C::kBStages;
    constexpr int OPS = C::kOpStages;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *b_base = smem;                                      // B operand ring
    uint8_t *w_base = b_base + RB * C::kBBytes;                  // weight ring
    uint8_t *stg_base = w_base + RW * kWRawBytes;                // 2 staging buffers, then the zero block
    uint64_t *bars = reinterpret_cast<uint64_t *>(stg_base + C::kStgRegion);
    uint64_t *w_full = bars;
    uint64_t *w_empty = w_full + RW;
    uint64_t *b_full = w_empty + RW;
    uint64_t *b_empty = b_full + RB;
    uint64_t *op_full = b_empty + RB;
    uint64_t *op_empty = op_full + OPS;
    uint64_t *chunk_full = op_empty + OPS;
    uint64_t *chunk_empty = chunk_full + 2;
    uint64_t *mma_done = chunk_empty + 2;
    uint64_t *fix_bar = mma_done + 1;  // [2]: slot rows landed in staging buffer 0 / 1
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fix_bar + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *hdr_ok = abort_flag + 1;
    volatile int *is_last = abort_flag + 2;
    volatile int *fin_flag = abort_flag + 3;
    float *tile_sx = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(bars) + 1024);
    int *tile_tx = reinterpret_cast<int *>(tile_sx + 128);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const uint32_t bb = block_bytes(p.group);
    const uint64_t tmo = p.timeout_ns;

    if (threadIdx.x == 0) {
        griddep_launch_dependents();
        prefetch_tensormap(&qx_map);
        const PackedHeader *h = reinterpret_cast<const PackedHeader *>(p.packed);
        const bool ok = h->magic == kPackedMagic && h->version == kPackedVersion && h->N == p.N &&
                        h->K == p.K && h->group == p.group && h->illegal == 0u;
        *hdr_ok = ok ? 1 : 0;
        *abort_flag = 0;
        *is_last = 0;
        for (int i = 0; i < RW; ++i) {
            mbar_init(&w_full[i], 1);
            mbar_init(&w_empty[i], kConvGroupWarps);  // the converter group of the stage
        }
        for (int i = 0; i < RB; ++i) {
            mbar_init(&b_full[i], 1);
            mbar_init(&b_empty[i], 1);  // the MMA commit of the stage
        }
        for (int i = 0; i < OPS; ++i) {
            mbar_init(&op_full[i], kConvGroupWarps);
            mbar_init(&op_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&chunk_full[i], 2);           // one commit per issuing thread
            mbar_init(&chunk_empty[i], kEpiWarps);  // phase 0: zeroed at start
        }
        mbar_init(mma_done, 2);
        mbar_init(&fix_bar[0], 1);
        mbar_init(&fix_bar[1], 1);
        fence_barrier_init();
    }
    // The zero block is read by bulk copies (async proxy).
    for (int i = threadIdx.x; i < static_cast<int>(C::kStgBytes / 16); i += kThreads)
        st_shared_v4(smem_u32(stg_base + 2 * C::kStgBytes) + 16u * i, 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const bool run = (*hdr_ok != 0);
    if (!run && threadIdx.x == 0) {
        griddep_wait();  // the status word may still be in use by the preceding kernel
        atomicOr(p.status, kStatusBadPacked);
    }

    if (warp < 4) {
        // warpgroup 0: weight producer (warp 0), MMA issuers (1, 2), activation producer (3)
        if constexpr (C::kRegSplit) setmaxnreg_dec<C::kRegLow>();
        if (run && warp == 0) {
            // ------------------------------------------- weight TMA producer --
            // Weight blocks are never written by a preceding kernel, so this
            // producer does not wait for the launch dependency: under launch
            // overlap its first RW stages stream in while the preceding kernel
            // finishes.
            if (lane == 0) {
                const bool withhold = (p.debug_flags & kDebugWithholdStage) != 0;
                SegmentWalker walk(p, cta);
                Segment sg;
                int st = 0, issued = 0;
                bool stop = false;
                while (!stop && walk.next(sg)) {
                    const int n_tile = sg.tile / p.tok_tiles;
                    const uint8_t *wblk = p.packed + kHeaderBytes + (static_cast<size_t>(n_tile) * p.G) * bb;
                    for (int k = sg.k0; k < sg.k1; ++k, ++st) {
                        const int slot = st % RW, use = st / RW;
                        if (withhold && st == 1) {
                            stop = true;
                            break;
                        }
                        if (use > 0 && !mbar_wait(&w_empty[slot], (use - 1) & 1, abort_flag, p.status, tmo)) {
                            stop = true;
                            break;
                        }
                        if (!weights_in_bounds(p, kHeaderBytes + (static_cast<unsigned long long>(n_tile) * p.G + k) * bb,
                                               bb)) {
                            *abort_flag = 1;
                            stop = true;
                            break;
                        }
                        mbar_arrive_expect_tx(&w_full[slot], bb);
                        tma_load_1d(w_base + slot * kWRawBytes, wblk + static_cast<size_t>(k) * bb, bb, &w_full[slot]);
                        issued = st + 1;
                    }
                }
                // Drain: every issued copy must land before the CTA exits.
                for (int t = (issued > RW ? issued - RW : 0); t < issued; ++t)
                    mbar_wait(&w_full[t % RW], (t / RW) & 1, nullptr, p.status, tmo);
            }
        } else if (run && warp == 3) {
            // ------------------------------------- activation TMA producer --
            if (lane == 0) {
                griddep_wait();  // the activation operand may be written by the preceding kernel
                SegmentWalker walk(p, cta);
                Segment sg;
                int st = 0, issued = 0;
                bool stop = false;
                while (!stop && walk.next(sg)) {
                    const int tok_tile = sg.tile % p.tok_tiles;
                    for (int k = sg.k0; k < sg.k1; ++k, ++st) {
                        const int slot = st % RB, use = st / RB;
                        if (use > 0 && !mbar_wait(&b_empty[slot], (use - 1) & 1, abort_flag, p.status, tmo)) {
                            stop = true;
                            break;
                        }
                        uint8_t *dst = b_base + slot * C::kBBytes;
                        mbar_arrive_expect_tx(&b_full[slot], C::kBBytes);
                        tma_load_2d(dst, &qx_map, k * kTileK, tok_tile * BT, &b_full[slot]);
                        tma_load_2d(dst + C::kBAtom, &qx_map, k * kTileK + 64, tok_tile * BT, &b_full[slot]);
                        issued = st + 1;
                    }
                }
                for (int t = (issued > RB ? issued - RB : 0); t < issued; ++t)
                    mbar_wait(&b_full[t % RB], (t / RB) & 1, nullptr, p.status, tmo);
            }
        } else if (run && (warp == 1 || warp == 2)) {
            // ------------------------------------------------ MMA issuers --
            // Two threads take alternate stages (warp 1 even, warp 2 odd): a
            // barrier wait issued after a thread's own MMAs queues behind them,
            // so with one issuer every wait idled the tensor pipe.  Their MMAs
            // into a chunk buffer have no mutual order, so none of them clears
            // the accumulator: the epilogue hands out every chunk buffer zeroed,
            // and each issuer commits to chunk_full at every chunk end (the
            // barrier counts both).  The fp32 partial sums are exact integers,
            // so the order of the MMAs does not change the result.
            if (lane == 0) {
                constexpr uint32_t idesc = idesc_f16_f32(128, BT);
                const int par = warp - 1;
                SegmentWalker walk(p, cta);
                Segment sg;
                int st = 0, gc = 0;
                bool stop = false;
                while (!stop && walk.next(sg)) {
                    const int len = sg.k1 - sg.k0;
                    // chunk by chunk (chunks start at multiples of kChunkStages
                    // of the segment); this thread's stages of a chunk are those
                    // of its parity, two apart
                    for (int i0 = 0; i0 < len && !stop; i0 += kChunkStages) {
                        const int cur = gc++;
                        const int i1 = min(len, i0 + kChunkStages);
                        const int ib = i0 + (((st + i0) & 1) != par ? 1 : 0);
                        if (ib < i1 && !mbar_wait(&chunk_empty[cur & 1], (cur >> 1) & 1, abort_flag, p.status, tmo)) {
                            stop = true;
                            break;
                        }
                        const uint32_t d_tmem = tmem + C::kChunk0 + static_cast<uint32_t>((cur & 1) * BT);
                        for (int i = ib; i < i1; i += 2) {
                            const int s = st + i;
                            const int os = s % OPS, ouse = s / OPS, bs = s % RB;
                            if (!mbar_wait(&op_full[os], ouse & 1, abort_flag, p.status, tmo)) {
                                stop = true;
                                break;
                            }
                            tc_fence_after();
                            const uint32_t a_tmem = tmem + C::kA0 + static_cast<uint32_t>(os) * 64u;
                            // The slot's descriptor once; each k step adds its byte offset / 16
                            // to the address field (bits 0-13, no carry: shared-memory
                            // addresses stay below 2^18), a 32-bit add on the low word.
                            const uint64_t bd0 = desc_kmajor_sw128(smem_u32(b_base + bs * C::kBBytes));
                            const uint32_t bd_lo = static_cast<uint32_t>(bd0), bd_hi = static_cast<uint32_t>(bd0 >> 32);
    #pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                const uint32_t off = ((kk >> 2) * C::kBAtom + (kk & 3) * 32) >> 4;
                                mma_f16_tmem_a_acc(d_tmem, a_tmem + 8u * kk, bd_lo + off, bd_hi, idesc);
                            }
                            mma_commit(&op_empty[os]);
                            mma_commit(&b_empty[bs]);
                        }
                        if (!stop) mma_commit(&chunk_full[cur & 1]);
                    }
                    st += len;
                }
                // All of this thread's MMAs must finish before TMEM is released.
                mma_commit(mma_done);
                mbar_wait(mma_done, 0, nullptr, p.status, tmo);
            }
        }
    } else if (warp < 8) {
        // warpgroup 1: epilogue
        if constexpr (C::kRegSplit) setmaxnreg_inc<C::kRegEpi>();
        if (run) {
            // ------------------------------------------------ epilogue warps --
            // Each thread owns one weight row of the tile (its TMEM lane) and keeps
            // that row's int32 sums for all BT tokens of the segment in registers:
            // a drained chunk is added into them and its buffer goes back to the
            // MMAs at once (zeroed); the tile's output then leaves from registers.
            griddep_wait();  // scales, workspace and output may belong to the preceding kernel
            const int et = threadIdx.x - 128;           // TMEM lane == weight row in tile
            const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
            constexpr int NB = BT / 16;                 // blocks of 16 tokens
            SegmentWalker walk(p, cta);
            Segment sg;
            int gc = 0;
            int stg_use = 0;  // staging buffers used so far (buffer stg_use & 1 is next)
            uint32_t fix_n0 = 0, fix_n1 = 0;  // fix-up loads consumed per staging buffer (mbarrier phases)
            uint32_t zero16[16];
    #pragma unroll
            for (int i = 0; i < 16; ++i) zero16[i] = 0u;
            {
                // Both chunk buffers start zeroed (the MMAs only accumulate).
                for (int j = 0; j < 2 * NB; ++j) tmem_st16(tl + C::kChunk0 + static_cast<uint32_t>(16 * j), zero16);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&chunk_empty[0]);
                    mbar_arrive(&chunk_empty[1]);
                }
            }
            // All four epilogue warps take every named barrier below the same number
            // of times: they walk the same segments and leave the walk together,
            // on a decision read from the shared abort flag after a barrier (any
            // failed wait has raised it before that barrier).
            bool ok = true;
            while (walk.next(sg)) {
                const int tok_tile = sg.tile % p.tok_tiles, n_tile = sg.tile / p.tok_tiles;
                const int m0 = tok_tile * BT, n = n_tile * kTileN + et;
                const bool split = !(sg.k0 == 0 && sg.k1 == p.G);
                const float sw = p.s_w ? h2f(p.s_w[n]) : 0.f;
                const int zc = (p.group == 0) ? p.packed[packed_z_offset(p.N, p.K) + n] : 0;
                const uint32_t tfirst = static_cast<uint32_t>(sg.seq) * static_cast<uint32_t>(p.G);
                const int slot_idx = split ? cta_of_stage(tfirst, p) : 0;
                int32_t *slot = p.slots + static_cast<size_t>(slot_idx) * (BT * kTileN);
                const int nch = (sg.k1 - sg.k0 + kChunkStages - 1) / kChunkStages;
                // Stage this tile's per-token scale (and row sums) in shared memory.
                named_bar_sync(2, kEpiThreads);
                if (et < BT) {
                    const int m = m0 + et;
                    tile_sx[et] = (m < p.M && p.s_x) ? h2f(p.s_x[m]) : 0.f;
                    tile_tx[et] = (m < p.M && p.group == 0) ? p.t_x[m] : 0;
                }
                named_bar_sync(2, kEpiThreads);
                int acc[BT];
    #pragma unroll
                for (int i = 0; i < BT; ++i) acc[i] = 0;
                for (int c = 0; c < nch; ++c) {
                    const int cur = gc++;
                    const int cb = cur & 1;
                    // A failed wait does not leave the loop: every epilogue warp
                    // must take the same named barriers; the abort flag, read by
                    // the issuing thread after each barrier, stops all output.
                    ok = mbar_wait_warp(&chunk_full[cb], (cur >> 1) & 1, abort_flag, p.status, tmo);
                    tc_fence_after();
                    const uint32_t cbase = tl + C::kChunk0 + static_cast<uint32_t>(cb * BT);
    #pragma unroll
                    for (int j = 0; j < NB; j += 2) {
                        // two 16-column loads in flight, then the zeros back
                        uint32_t f0[16], f1[16];
                        tmem_ld16(cbase + static_cast<uint32_t>(16 * j), f0);
                        if (j + 1 < NB) tmem_ld16(cbase + static_cast<uint32_t>(16 * j + 16), f1);
                        tmem_wait_ld_regs(f0);
                        if (j + 1 < NB) tmem_wait_ld_regs(f1);
                        tmem_st16(cbase + static_cast<uint32_t>(16 * j), zero16);
                        if (j + 1 < NB) tmem_st16(cbase + static_cast<uint32_t>(16 * j + 16), zero16);
    #pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            if constexpr (kPC) {  // 2^24 undoes the subnormal codes
                                acc[16 * j + i] += __float2int_rn(__fmul_rn(__uint_as_float(f0[i]), 16777216.0f));
                                if (j + 1 < NB)
                                    acc[16 * j + 16 + i] += __float2int_rn(__fmul_rn(__uint_as_float(f1[i]), 16777216.0f));
                            } else {
                                acc[16 * j + i] += __float2int_rn(__uint_as_float(f0[i]));
                                if (j + 1 < NB) acc[16 * j + 16 + i] += __float2int_rn(__uint_as_float(f1[i]));
                            }
                        }
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&chunk_empty[cb]);
                }
                if (!split) {
                    if constexpr (kAccOut) {
                        // int32 test output: per block of 16 tokens, this thread's
                        // values go through its own slots of the fix-up output
                        // buffers (unused in this mode) into one rolled loop.
                        const uint32_t ibuf = smem_u32(stg_base) + 3 * C::kStgBytes;
    #pragma unroll
                        for (int j = 0; j < NB; ++j) {
    #pragma unroll
                            for (int i = 0; i < 16; ++i)
                                st_shared_b32(ibuf + 4u * (i * kTileN + et), static_cast<uint32_t>(acc[16 * j + i]));
                            write_block_i32(p, ibuf, m0 + 16 * j, n, zc, tile_sx + 16 * j, tile_tx + 16 * j, sw, ok);
                        }
                    } else {
                        // fp16 outputs: blocks of 16 tokens x 128 rows (4 KB each)
                        // staged four at a time across both staging buffers, then
                        // one tensor store per block (rows past M are clipped by
                        // the copy): two barriers per four blocks.
                        constexpr int kRound = 4;
    #pragma unroll
                        for (int j0 = 0; j0 < NB; j0 += kRound) {
                            if (et == 0) bulk_wait_read<0>();  // earlier copies have read the staging buffers
                            named_bar_sync(3, kEpiThreads);
    #pragma unroll
                            for (int jj = 0; jj < kRound; ++jj) {
                                const int j = j0 + jj;
                                if (j >= NB) break;
                                const uint32_t buf = smem_u32(stg_base) + static_cast<uint32_t>(jj) * (C::kStgBytes / 2);
                                uint32_t sxv[16], txv[16];
                                ld_shared_x16(smem_u32(tile_sx + 16 * j), sxv);
                                ld_shared_x16(smem_u32(tile_tx + 16 * j), txv);
                                uint16_t o[16];
    #pragma unroll
                                for (int i = 0; i < 16; ++i)
                                    o[i] = out_fp16(acc[16 * j + i], zc, static_cast<int>(txv[i]), __uint_as_float(sxv[i]), sw);
    #pragma unroll
                                for (int i = 0; i < 16; ++i) st_shared_u16(buf + 2u * (i * kTileN + et), o[i]);
                            }
                            fence_proxy_async_smem();
                            named_bar_sync(3, kEpiThreads);
                            if (et == 0 && *abort_flag == 0) {
    #pragma unroll
                                for (int jj = 0; jj < kRound; ++jj) {
                                    if (j0 + jj >= NB) break;
                                    tma_store_2d(&o_map, stg_base + jj * (C::kStgBytes / 2), n_tile * kTileN, m0 + 16 * (j0 + jj));
                                }
                                bulk_commit();
                            }
                        }
                        // The other users of the staging buffers take them in turn
                        // with one copy allowed in flight: leave none.
                        if (et == 0) bulk_wait_read<0>();
                    }
                } else {
                    // Split tile: if every other contributor has already published
                    // its partial, this CTA is the last one and finishes the tile
                    // with its own partial still in registers.
                    named_bar_sync(3, kEpiThreads);
                    if (et == 0) {
                        int f = 0;
                        if (!slot_in_bounds<BT>(p, slot_idx)) *abort_flag = 1;
                        if (*abort_flag == 0 && !(p.debug_flags & kDebugAlwaysPublish))
                            f = finish_directly(p, cta, slot_idx, tfirst, abort_flag) ? 1 : 0;
                        *fin_flag = f;
                    }
                    named_bar_sync(3, kEpiThreads);
                    const bool fin_seg = *fin_flag != 0;
                    bool do_fix = fin_seg;
                    if (!fin_seg) {
                        // Publish: each block of 16 tokens (8 KB, rows 16j.. of the
                        // slot are contiguous) goes out as one bulk reduce-add.
    #pragma unroll
                        for (int j = 0; j < NB; ++j) {
                            if (et == 0) bulk_wait_read<1>();
                            named_bar_sync(3, kEpiThreads);
                            const uint32_t buf = smem_u32(stg_base) + (stg_use & 1) * C::kStgBytes;
    #pragma unroll
                            for (int i = 0; i < 16; ++i)
                                st_shared_b32(buf + 4u * (i * kTileN + et), static_cast<uint32_t>(acc[16 * j + i]));
                            fence_proxy_async_smem();
                            named_bar_sync(3, kEpiThreads);
                            if (et == 0 && *abort_flag == 0) {
                                bulk_reduce_add_s32(slot + 16 * j * kTileN, stg_base + (stg_use & 1) * C::kStgBytes,
                                                    C::kStgBytes);
                                bulk_commit();
                            }
                            ++stg_use;
                        }
                        // Every epilogue thread reaches both named barriers once per
                        // publish.  A failed wait anywhere has raised abort_flag
                        // before the first barrier, so the decision below is uniform.
                        // One thread issued this tile's partial reductions; it waits
                        // for them to complete, publishes them with a fence and the
                        // arrival counter, and learns whether this CTA is the last.
                        named_bar_sync(1, kEpiThreads);
                        if (et == 0) {
                            int last_cta = 0;
                            if (*abort_flag == 0) {
                                bulk_wait<0>();
                                __threadfence();
                                const uint32_t tlast = tfirst + static_cast<uint32_t>(p.G) - 1u;
                                const unsigned expected =
                                    static_cast<unsigned>(cta_of_stage(tlast, p) - slot_idx + 1);
                                const unsigned prev = atomicAdd(p.counters + slot_idx, 1u);
                                last_cta = (prev + 1 == expected) ? 1 : 0;
                                if (last_cta) __threadfence();
                            }
                            *is_last = last_cta;
                        }
                        named_bar_sync(1, kEpiThreads);
                        do_fix = *is_last != 0;
                    }
                    if (do_fix) {
                        // Fix-up: out = (own partial, when finishing directly) + the
                        // slot's sums.  Slot rows of 16 tokens (8 KB) come in by bulk
                        // loads, two in flight through the staging buffers; each
                        // block's rows are then re-zeroed and its fp16 outputs leave
                        // through the two fix-up output buffers.
                        if (et == 0) {
                            bulk_wait_read<0>();        // staging buffers no longer read by earlier copies
                            fence_proxy_async_global();  // the counter acquire orders the loads below
                            for (int q = 0; q < (NB < 2 ? NB : 2); ++q) {
                                mbar_arrive_expect_tx(&fix_bar[q], C::kStgBytes);
                                tma_load_1d(stg_base + q * C::kStgBytes, slot + 16 * q * kTileN, C::kStgBytes, &fix_bar[q]);
                            }
                        }
    #pragma unroll
                        for (int j = 0; j < NB; ++j) {
                            const int q = j & 1;
                            // The loads always complete (they read the workspace), so
                            // this wait ignores the abort flag: none is left in flight.
                            mbar_wait_warp(&fix_bar[q], (q ? fix_n1 : fix_n0) & 1u, nullptr, p.status, tmo);
                            if (q) ++fix_n1; else ++fix_n0;
                            const uint32_t sbuf = smem_u32(stg_base) + q * C::kStgBytes;
                            int tot[16];
    #pragma unroll
                            for (int i = 0; i < 16; ++i)
                                tot[i] = ld_shared_s32(sbuf + 4u * (i * kTileN + et)) + (fin_seg ? acc[16 * j + i] : 0);
                            if (et == 0) bulk_wait_read<1>();  // output buffer q: its store from block j-2 has read it
                            named_bar_sync(3, kEpiThreads);     // ... and every thread has read staging buffer q
                            if (et == 0) {
                                if (*abort_flag == 0) {
                                    bulk_store(slot + 16 * j * kTileN, stg_base + 2 * C::kStgBytes, C::kStgBytes);
                                    bulk_commit();
                                }
                                if (j + 2 < NB) {
                                    mbar_arrive_expect_tx(&fix_bar[q], C::kStgBytes);
                                    tma_load_1d(stg_base + q * C::kStgBytes, slot + 16 * (j + 2) * kTileN, C::kStgBytes,
                                                &fix_bar[q]);
                                }
                            }
                            if constexpr (kAccOut) {
                                const uint32_t ibuf = smem_u32(stg_base) + 3 * C::kStgBytes;
    #pragma unroll
                                for (int i = 0; i < 16; ++i) st_shared_b32(ibuf + 4u * (i * kTileN + et), static_cast<uint32_t>(tot[i]));
                                write_block_i32(p, ibuf, m0 + 16 * j, n, zc, tile_sx + 16 * j, tile_tx + 16 * j, sw,
                                                *abort_flag == 0);
                                continue;
                            }
                            const uint32_t obuf = smem_u32(stg_base) + 3 * C::kStgBytes + q * (C::kStgBytes / 2);
                            uint32_t sxv[16], txv[16];
                            ld_shared_x16(smem_u32(tile_sx + 16 * j), sxv);
                            ld_shared_x16(smem_u32(tile_tx + 16 * j), txv);
                            uint16_t o[16];
    #pragma unroll
                            for (int i = 0; i < 16; ++i)
                                o[i] = out_fp16(tot[i], zc, static_cast<int>(txv[i]), __uint_as_float(sxv[i]), sw);
    #pragma unroll
                            for (int i = 0; i < 16; ++i) st_shared_u16(obuf + 2u * (i * kTileN + et), o[i]);
                            fence_proxy_async_smem();
                            named_bar_sync(3, kEpiThreads);
                            if (et == 0 && *abort_flag == 0) {
                                tma_store_2d(&o_map, stg_base + 3 * C::kStgBytes + q * (C::kStgBytes / 2), n_tile * kTileN,
                                             m0 + 16 * j);
                                bulk_commit();
                            }
                        }
                        if (et == 0 && *abort_flag == 0) p.counters[slot_idx] = 0u;
                    }
                }
                named_bar_sync(1, kEpiThreads);  // also: is_last is rewritten by the next split segment
                if (*abort_flag != 0) break;
            }
            // Bulk copies read shared memory until they have read it: wait for that
            // before exit (their global writes complete on their own, and are
            // visible to every later grid, a dependent one's dependency wait included).
            if (et == 0) bulk_wait_read<0>();
            (void)ok;
        }
    } else if (run) {
        // ---------------------------------------------- converter warps --
        // Two groups of four warps take alternate stages, so one group's
        // waits and fences overlap the other group's arithmetic.  In a group,
        // warp w converts weight rows 32*(w%4) .. +31 (its TMEM lane quarter)
        // over the whole 128-k stage.
        const int cg = (warp - 8) >> 2;
        const int wr = (warp & 3) * 32 + lane;   // weight row == TMEM lane
        const uint32_t a_lane = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        SegmentWalker walk(p, cta);
        Segment sg;
        int st = 0;
        bool stop = false;
        while (!stop && walk.next(sg)) {
            for (int k = sg.k0; k < sg.k1; ++k, ++st) {
                if ((st & 1) != cg) continue;
                const int ws = st % RW, wuse = st / RW, bs = st % RB, buse = st / RB;
                const int os = st % OPS, ouse = st / OPS;
                if (!mbar_wait_warp(&w_full[ws], wuse & 1, abort_flag, p.status, tmo)) {
                    stop = true;
                    break;
                }
                const uint32_t wraw = smem_u32(w_base + ws * kWRawBytes);

                // Weights: row wr, 4 raw chunks of 32 k -> 128 fp16 -> 64 TMEM
                // columns of this thread's lane (2 fp16 per column).  The whole
                // stage is converted into registers before the wait for its
                // operand slot, so only the TMEM store follows the MMAs that
                // free the slot.
                uint32_t s = 1, zz = 0;
                if (!kPC) {
                    uint16_t meta;
                    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(meta) : "r"(wraw + kCodeBytes + 4 * wr));
                    s = meta & 0xffu;
                    zz = meta >> 8;
                }
                const uint32_t cst = static_cast<uint32_t>(128 - static_cast<int>(zz * s)) * 0x01010101u;
                uint32_t a_frag[2][32];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const uint4 v = ld_shared_v4(wraw + (((h * 2 + i) * 128 + wr) << 4));
                        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t lo = w4[j] & 0x0F0F0F0Fu;
                            const uint32_t hi = (w4[j] >> 4) & 0x0F0F0F0Fu;
                            uint32_t *f = a_frag[h] + 16 * i + 4 * j;
                            if (kPC) {
                                // raw codes as fp16 subnormals q * 2^-24
                                f[0] = __byte_perm(lo, 0u, 0x4140u);
                                f[1] = __byte_perm(lo, 0u, 0x4342u);
                                f[2] = __byte_perm(hi, 0u, 0x4140u);
                                f[3] = __byte_perm(hi, 0u, 0x4342u);
                            } else {
                                const uint32_t ulo = lo * s + cst;  // bytes: (q - z) * s + 128
                                const uint32_t uhi = hi * s + cst;
                                biased_bytes_to_f16x4(ulo, f[0], f[1]);
                                biased_bytes_to_f16x4(uhi, f[2], f[3]);
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&w_empty[ws]);  // this warp is done reading the weight slot
                if (ouse > 0 && !mbar_wait_warp(&op_empty[os], (ouse - 1) & 1, abort_flag, p.status, tmo)) {
                    stop = true;
                    break;
                }
                tc_fence_after();
                const uint32_t a_dst = a_lane + C::kA0 + static_cast<uint32_t>(os) * 64u;
                tmem_st32(a_dst, a_frag[0]);
                tmem_st32(a_dst + 32u, a_frag[1]);
                tmem_wait_st();
                tc_fence_before();
                // The B operand of this stage, copied after the dependency
                // wait, must have landed before the MMAs (ordered after
                // op_full) read it; the weights were converted without it.
                // A parity wait is exact only once the slot's previous phase
                // has completed: with an odd ring depth the previous use of
                // this B slot belongs to the other converter group, which
                // this one may have overtaken, so first wait for that use's
                // MMA commit (it follows the previous b_full phase).  With an
                // even depth the same group waited for it and this returns
                // at once.
                if ((buse > 0 && !mbar_wait_warp(&b_empty[bs], (buse - 1) & 1, abort_flag, p.status, tmo)) ||
                    !mbar_wait_warp(&b_full[bs], buse & 1, abort_flag, p.status, tmo)) {
                    stop = true;
                    break;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&op_full[os]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int BT>
cudaError_t launch_bt(const GemmArgs &a, const GemmPlan &plan, cudaStream_t stream) {
    using C = Cfg<BT>;
    static std::mutex mu;
    static bool configured[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!configured[dev]) {
            for (auto kern : {w4a8_gemm_kernel<BT, false, false>, w4a8_gemm_kernel<BT, true, false>,
                              w4a8_gemm_kernel<BT, false, true>, w4a8_gemm_kernel<BT, true, true>}) {
                e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::kSmemBytes));
                if (e != cudaSuccess) return e;
                if (C::kRegSplit) {
                    // The warpgroup register split adds up to the launch
                    // allocation only at this per-thread count; any other would
                    // leave the epilogue's increase waiting, so refuse to launch.
                    cudaFuncAttributes fa;
                    e = cudaFuncGetAttributes(&fa, kern);
                    if (e != cudaSuccess) return e;
                    if (fa.numRegs != static_cast<int>(C::kRegLaunch)) return cudaErrorInvalidConfiguration;
                }
            }
            configured[dev] = true;
        }
    }
    CUtensorMapEncodeTiledFn enc = get_encode_fn();
    if (!enc) return cudaErrorNotSupported;
    uint8_t *ws0 = static_cast<uint8_t *>(a.ws);
    const void *act = a.act;
    if (!act) {
        // No precomputed operand: build the fp16 copy of Qx in the workspace first.
        void *scratch = ws0 + plan.act_offset;
        e = launch_act_operand(a.Qx, a.M, a.K, kPathF16, scratch, stream);
        if (e != cudaSuccess) return e;
        act = scratch;
    }
    // fp16 activation operand [M][K]: one box = 64 k (128 bytes) x BT tokens.
    CUtensorMap map;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.K), static_cast<cuuint64_t>(a.M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.K) * 2u};
    const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(BT)};
    const cuuint32_t estr[2] = {1u, 1u};
    CUresult cr = enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(act), dims, strides, box,
                      estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
    // fp16 output O [M][N]: one store box = 128 rows of a tile x 16 tokens.
    // (Unused in the int32 test mode.)
    CUtensorMap o_map{};
    if (a.O) {
        const cuuint64_t odims[2] = {static_cast<cuuint64_t>(a.N), static_cast<cuuint64_t>(a.M)};
        const cuuint64_t ostrides[1] = {static_cast<cuuint64_t>(a.N) * 2u};
        const cuuint32_t obox[2] = {static_cast<cuuint32_t>(kTileN), 16u};
        cr = enc(&o_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.O, odims, ostrides, obox, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }

    GemmParams p;
    uint8_t *ws = static_cast<uint8_t *>(a.ws);
    p.packed = static_cast<const uint8_t *>(a.packed);
    p.s_x = a.s_x;
    p.t_x = a.t_x;
    p.s_w = a.s_w;
    p.O = a.O;
    p.acc_out = a.acc_out;
    p.status = reinterpret_cast<uint32_t *>(ws);
    p.counters = reinterpret_cast<uint32_t *>(ws + plan.counters_offset);
    p.slots = reinterpret_cast<int32_t *>(ws + plan.slots_offset);
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.group = a.group;
    p.G = plan.G;
    p.tok_tiles = plan.tok_tiles;
    p.total = plan.total;
    p.ctas = plan.ctas;
    p.dp_tiles = plan.dp_tiles;
    p.band = plan.band;
    p.debug_flags = a.debug_flags;
    p.timeout_ns = a.timeout_ns;
    set_extents(p, plan, a.N, a.K, a.group);
    dim3 grid(plan.ctas);
    if (a.acc_out)
        return p.group ? launch_kernel(w4a8_gemm_kernel<BT, true, false>, grid, dim3(kThreads), C::kSmemBytes, stream,
                                       a.pdl, map, o_map, p)
                       : launch_kernel(w4a8_gemm_kernel<BT, true, true>, grid, dim3(kThreads), C::kSmemBytes, stream,
                                       a.pdl, map, o_map, p);
    return p.group ? launch_kernel(w4a8_gemm_kernel<BT, false, false>, grid, dim3(kThreads), C::kSmemBytes, stream,
                                   a.pdl, map, o_map, p)
                   : launch_kernel(w4a8_gemm_kernel<BT, false, true>, grid, dim3(kThreads), C::kSmemBytes, stream,
                                   a.pdl, map, o_map, p);
}

}  // namespace

namespace {
// Measured launch choices: for a shape (N, K, group) tuned on a GPU with
// num_sms SMs, the fastest (path, tokens per tile, CTA count or cluster
// size) found at token count M, timed on that GPU against the other
// candidates and the rules below (the ADAngel review's offline per-shape
// policy table, looked up at run time).  An entry covers the token counts
// above the next smaller tuned M of the same shape, up to its own M.
struct DispatchEntry {
    int N, K, group, M, num_sms, path, bt, ctas, sched;
};
const DispatchEntry kDispatchTable[] = {
#include "qoq_dispatch_table.inc"
    {0, 0, 0, 0, 0, 0, 0, 0, 0}  // end
};

const DispatchEntry *find_dispatch(int M, int N, int K, int group, int num_sms) {
    const DispatchEntry *best = nullptr;
    for (const DispatchEntry *e = kDispatchTable; e->N != 0; ++e) {
        if (e->N != N || e->K != K || e->group != group || e->num_sms != num_sms || e->M < M) continue;
        if (!best || e->M < best->M) best = e;
    }
    return best;
}

// Shared memory of a GEMV-path CTA: activations and their group sums for its
// blocks, and two int32 reduction buffers (the launcher sizes it the same way).
size_t gemv_smem_bytes(int MT, int G, int csize) {
    const size_t nb = static_cast<size_t>((G + csize - 1) / csize);
    return MT * nb * 128 + MT * nb * 4 + 2 * static_cast<size_t>(MT) * 128 * 4;
}
constexpr size_t kGemvSmemMax = 200u << 10;
}  // namespace

GemmPlan plan_gemm(int M, int N, int K, int group, int num_sms, int force_path, int force_bt,
                   int force_ctas, bool use_table, int force_sched) {
    if (use_table && force_path == 0 && force_bt == 0 && force_ctas == 0 && force_sched == 0) {
        if (const DispatchEntry *e = find_dispatch(M, N, K, group, num_sms)) {
            const GemmPlan t = plan_gemm(M, N, K, group, num_sms, e->path, e->bt, e->ctas, false, e->sched);
            if (t.path == e->path) return t;  // else the rules below
        }
    }
    GemmPlan pl{};
    const int G = K / kTileK, n_tiles = N / kTileN;
    // Decode batches of at most 4 tokens: the CUDA-core GEMV path, whose
    // launches carry no tensor-core setup, when its shared memory fits (the
    // path takes up to 8 tokens when forced; from 5 tokens its dp4a work per
    // weight outweighs the tensor cores' setup: gate_up at 8 tokens 54.8 us
    // against 19.7 on the fp8 path).
    int mt = M <= 1 ? 1 : (M <= 2 ? 2 : (M <= 4 ? 4 : 8));
    int csize = 1;
    if (M <= 8 && num_sms > 0) {
        // The largest cluster (K split) that keeps at most six 256-thread CTAs
        // per SM and at least one 128-k block per K half of a CTA.
        for (int c = 8; c >= 1; c >>= 1) {
            if (static_cast<long long>(n_tiles) * c <= 6LL * num_sms && G >= 2 * c) {
                csize = c;
                break;
            }
        }
        if (force_path == kPathGemv && force_ctas > 0) csize = force_ctas >= 8 ? 8 : (force_ctas >= 4 ? 4 : (force_ctas >= 2 ? 2 : 1));
        while (csize < 8 && gemv_smem_bytes(mt, G, csize) > kGemvSmemMax) csize *= 2;
    }
    const bool gemv_ok = M <= 8 && (group == 0 || group == 128) && gemv_smem_bytes(mt, G, csize) <= kGemvSmemMax;
    if (force_path == kPathGemv || (force_path == 0 && force_bt == 0 && gemv_ok && M <= 4)) {
        if (!gemv_ok) {
            // forced for a shape the path cannot take: report an empty plan
            pl.path = 0;
            return pl;
        }
        pl.path = kPathGemv;
        pl.BT = mt;
        pl.tok_tiles = 1;
        pl.n_tiles = n_tiles;
        pl.G = G;
        pl.tiles = n_tiles;
        pl.total = static_cast<long long>(n_tiles) * G;
        pl.gv_csize = csize;
        pl.sched = 0;
        pl.ctas = n_tiles * csize;
        pl.counters_offset = kWsStatusBytes;
        pl.slots_offset = kWsStatusBytes;
        pl.zero_bytes = kWsStatusBytes;
        pl.act_offset = kWsStatusBytes;
        pl.ws_bytes = kWsStatusBytes;
        return pl;
    }
    // The fp8 path (4 MMAs per 128-k group, per-group exact drain) wins for
    // decode batches; larger token tiles keep the fp16 path.
    int path = force_path;
    if (path == 0) path = (group == 128 && M <= 32) ? kPathF8 : kPathF16;
    if (group != 128) path = kPathF16;
    int bt = force_bt;
    if (force_path == 0 && force_bt == 0 && M > 32 && num_sms > 0) {
        // Few k-stages per CTA at the natural tile (64 tokens up to M = 64,
        // else 128): half-width token tiles double the work units, which
        // balances the stream-K ranges and halves each split tile's fix-up;
        // measured faster up to 13.5 stages per CTA (Llama-3-8B qkv and o at
        // M = 64 and 128, o at M = 256), slower from 20 (qkv at M = 256).
        const long long nat = M <= 64 ? 64 : 128;
        const long long stages = (M + nat - 1) / nat * (N / kTileN) * static_cast<long long>(K / kTileK);
        if (stages <= 16LL * num_sms) {
            if (M <= 64 && group == 128) {
                path = kPathF8;
                bt = 32;
            } else if (M > 64) {
                bt = 64;
            }
        }
    }
    if (path == kPathF8) {
        if (bt != 16 && bt != 32) bt = M <= 16 ? 16 : 32;
    } else if (bt == 0) {
        bt = M <= 16 ? 16 : (M <= 32 ? 32 : (M <= 64 ? 64 : 128));
    }
    pl.path = path;
    pl.BT = bt;
    pl.tok_tiles = (M + bt - 1) / bt;
    pl.n_tiles = N / kTileN;
    pl.G = K / kTileK;
    pl.tiles = static_cast<long long>(pl.tok_tiles) * pl.n_tiles;
    pl.total = pl.tiles * pl.G;
    long long ctas = force_ctas > 0 ? force_ctas : num_sms;
    if (force_ctas <= 0 && num_sms > 16) {
        if (pl.tiles <= num_sms && pl.tiles * 5 >= static_cast<long long>(num_sms) * 3) {
            // The tiles fill at least 60 % of one wave: one whole tile per CTA
            // (no split tiles, no fix-ups) beats stream-K over every SM.
            ctas = pl.tiles;
        } else if (M <= 32) {
            // Decode sizes: leave 8 SMs free so that the first CTAs of the
            // kernel launched behind this one (typically the next layer's
            // activation quantizer, one CTA per token) start at once
            // instead of waiting for this GEMM's CTAs to leave.
            ctas = num_sms - 8;
        }
    }
    if (ctas > pl.total) ctas = pl.total;
    pl.ctas = static_cast<int>(ctas);
    pl.gv_csize = 0;
    // At least two waves of tiles: all but the last one to two waves go whole
    // to the CTAs round-robin (concurrent CTAs share their weight and
    // activation tiles in L2), the rest is balanced by stream-K.
    // Schedule (measured per shape by the dispatch table; the rule: data-
    // parallel waves for K up to 8192, where the DRAM traffic of the
    // prefill shapes fell most, stream-K only for longer K).
    int sched = force_sched > 0 ? force_sched : (K <= 8192 ? 2 : 1);
    if (pl.tiles < 2 * ctas) sched = 1;  // fewer than two waves: stream-K only
    pl.sched = sched;
    pl.dp_tiles = sched >= 2 ? static_cast<int>((pl.tiles / ctas - 1) * ctas) : 0;
    // Banded order (schedule 3): bands of about sqrt(P * BT / 32) weight tiles (a weight
    // tile moves 64 bytes per k and an activation tile 2 BT, so this minimises
    // the working set band * 64 + (P / band) * 2 BT bytes per k of the tiles
    // the CTAs hold at one time), the bands made about equal.
    pl.band = 0;
    if (sched == 4) pl.band = pl.n_tiles;  // one band: weight-tile fastest
    if (sched == 3 && pl.tok_tiles > 1) {
        const int b = static_cast<int>(std::lround(std::sqrt(static_cast<double>(ctas) * bt / 32.0)));
        const int nb = (pl.n_tiles + (b < 1 ? 1 : b) - 1) / (b < 1 ? 1 : b);
        pl.band = (pl.n_tiles + nb - 1) / nb;
    }
    pl.counters_offset = kWsStatusBytes;
    pl.slots_offset = kWsStatusBytes + (static_cast<size_t>(pl.ctas) * 4 + 255) / 256 * 256;
    pl.zero_bytes = pl.slots_offset + static_cast<size_t>(pl.ctas) * bt * kTileN * 4;
    pl.act_offset = (pl.zero_bytes + 255) / 256 * 256;
    pl.ws_bytes = pl.act_offset + act_operand_bytes(M, K, path);
    return pl;
}

cudaError_t launch_gemm(const GemmArgs &a, const GemmPlan &plan, cudaStream_t stream) {
    if (plan.path == kPathGemv) return launch_gemv(a, plan, stream);
    if (plan.path == kPathF8) return launch_gemm_f8(a, plan, stream);
    switch (plan.BT) {
        case 16: return launch_bt<16>(a, plan, stream);
        case 32: return launch_bt<32>(a, plan, stream);
        case 64: return launch_bt<64>(a, plan, stream);
        case 128: return launch_bt<128>(a, plan, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qoq

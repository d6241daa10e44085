// W4A8 GEMM, fp8-operand tensor-core path (decode batches, group = 128).
//
// Same result as the fp16-operand path (qoq_gemm.cu):
//   acc[m,n] = sum_g s_g[n,g] * sum_{k in g} Qx[m,k] * (q4[n,k] - z[n,g]),
//   O = fp16(acc * s_x[m] * s_w[n]),
// computed with exact integer arithmetic on the kind::f8f6f4 tensor cores:
//  * a 4-bit code q placed in a byte is the e4m3 number q * 2^-9, exactly
//    (e4m3 subnormals continue linearly into the first normal binade), so the
//    packed codes become the A operand by a nibble -> byte split, without any
//    multiply;
//  * an activation is split as u = Qx + 128 = 16*uh + ul with uh, ul in
//    [0, 15], stored the same way; the two planes are stacked along the MMA's
//    N dimension (2*BT rows), which costs nothing for N <= 128.  The planes
//    and the per-group activation sums t_g come precomputed (the activation
//    operand written by the activation quantizer, or by a preparation kernel
//    launched before this one), so TMA lands the B operand directly in its
//    swizzled shared-memory layout;
//  * per 128-k group, D_h = 2^-18 sum q*uh and D_l = 2^-18 sum q*ul are exact in
//    the fp32 accumulator (|sum| <= 128*15*15 = 28800 units of 2^-18);
//  * the epilogue turns each group into an integer without a conversion
//    instruction: 48 + 16*D_h + D_l lies in [32, 64), where fp32 values are
//    spaced by 2^-18, so its bit pattern minus that of 48 is
//    P = sum_k q*u = sum_k q*Qx + 128*sum_k q.  Then
//      acc += s_g * (P - 128*sum_k q - z*t_g[m]),  t_g[m] = sum_{k in g} Qx[m,k].
//    sum_k q comes with the packed metadata.
// K-stages are 256 wide (two groups per TMA transaction), four MMAs (K = 32)
// per group.  Roles (20 warps): warp 0 TMA, warps 1 and 2 issue the MMAs of
// alternate stages (warp 1 also allocates TMEM), warps 4-7 and 16-19 two
// converter groups that take alternate stages (one
// TMEM lane quarter per warp: codes -> bytes -> TMEM), warps 8-15 drain (two
// per lane quarter, one half of the tokens each).  A drained stage also
// proves its MMAs complete, so the drain's release of a stage's metadata
// slot is what frees the matching TMEM operand slot too.  Persistent
// stream-K schedule, bounded waits, and tile outputs as in the fp16 path:
// fp16 tiles by tensor bulk stores; a split tile's partial published by one
// bulk reduce-add, finished by the last contributor (directly, when every
// other partial is already published) from one bulk load of the slot.
#include <cuda.h>
#include <cuda_fp16.h>

#include <mutex>

#include "qoq_gemm_common.cuh"

namespace qoq {
namespace {

constexpr int kF8Threads = 640;
constexpr int kF8ConvWarps = 4;      // per converter group: warps 4..7 and 16..19
constexpr int kF8EpiWarps = 8;       // warps 8..15
constexpr int kF8EpiThreads = 32 * kF8EpiWarps;
constexpr int kGroupsPerStage = 2;
constexpr uint32_t kBlockBytesG = kCodeBytes + kMetaBytes;  // 8704

template <int BT>
struct F8Cfg {
    static constexpr int kNmma = 2 * BT;                  // uh plane rows + ul plane rows
    static constexpr int kRawStages = BT == 16 ? 6 : 5;
    static constexpr int kOpStages = 4;                   // TMEM A slots == metadata slots
    static constexpr int kAuxStages = kOpStages;
    // Raw slot: [B planes, group 0 | group 1][t_g 2 x BT][weight blocks 2 x 8704].
    static constexpr uint32_t kPlaneGroupBytes = static_cast<uint32_t>(kNmma) * 128u;
    static constexpr uint32_t kTgOff = kGroupsPerStage * kPlaneGroupBytes;
    static constexpr uint32_t kTgBytes = kGroupsPerStage * static_cast<uint32_t>(BT) * 4u;
    static constexpr uint32_t kWOff = kTgOff + kTgBytes;
    static constexpr uint32_t kRawSlotBytes = (kWOff + kGroupsPerStage * kBlockBytesG + 1023u) / 1024u * 1024u;
    static constexpr uint32_t kAuxMetaBytes = kGroupsPerStage * 128u * 4u;
    static constexpr uint32_t kAuxStageBytes = kAuxMetaBytes + kTgBytes;
    // TMEM: D buffers [kDSets stage sets][2 groups] x kNmma columns, then A
    // slots of 64 columns (128 rows x 256 k bytes).  With as many D sets as
    // metadata slots (BT = 16), the converter's wait for the drain of stage
    // s - 4 already frees the D set of stage s, so the MMA issuers wait on
    // op_full alone; BT = 32 has room for two sets and waits on d_empty too.
    static constexpr int kDSets = BT == 16 ? 4 : 2;
    static constexpr uint32_t kA0 = static_cast<uint32_t>(kDSets) * 2u * kNmma;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr int kNumBars = 3 * kRawStages + kOpStages + 2 * kAuxStages + 2 * kDSets + 1 + 1 + 1;
    // Tile output staging: int32 [BT][128] (a split tile's partials, or the
    // slot read back for the fix-up), an 8 KB zero block that re-zeroes
    // slots, and fp16 [BT][128] outputs; all moved by bulk copies.
    static constexpr uint32_t kStgI32Bytes = static_cast<uint32_t>(BT) * kTileN * 4u;
    static constexpr uint32_t kZeroBytes = 8192;
    static constexpr uint32_t kOutBytes = static_cast<uint32_t>(BT) * kTileN * 2u;
    // ... and an int32 [BT][128] buffer into which the prefetch warp loads
    // the slot of the split tile this CTA finishes.
    static constexpr uint32_t kPreOff = kStgI32Bytes + kZeroBytes + kOutBytes;
    static constexpr uint32_t kEpiRegion = kPreOff + kStgI32Bytes;
    static constexpr uint32_t kMiscBytes = 2048;
    static constexpr uint32_t kSmemBytes =
        kRawStages * kRawSlotBytes + kAuxStages * kAuxStageBytes + kEpiRegion + kMiscBytes + 1024;
    static_assert(kA0 + 64u * kOpStages <= kTmemCols, "TMEM columns");
    static_assert(kDSets == 2 || kDSets == kAuxStages, "D sets: double buffered, or one per metadata slot");
    static_assert(kNumBars * 8 + 64 <= 1024, "barrier area");
    static_assert(kSmemBytes <= 232448, "shared memory");
    static_assert(kPlaneGroupBytes % 1024 == 0 && kRawSlotBytes % 1024 == 0, "1 KB aligned swizzled tiles");
    static_assert(kWOff % 16 == 0 && kTgOff % 16 == 0, "16-byte aligned bulk copies");
    static_assert((kAuxStages * kAuxStageBytes) % 8 == 0, "barrier alignment");
};

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f8f6f4, the B descriptor
// passed as its two 32-bit words: _first overwrites D, _acc accumulates.
__device__ __forceinline__ void mma_f8_tmem_a_first(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                                    uint32_t idesc) {
    asm volatile(
        "{\n .reg .pred p;\n .reg .b64 bd;\n setp.ne.b32 p, 0, 0;\n mov.b64 bd, {%2, %3};\n"
        " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], bd, %4, p;\n}\n"
        ::"r"(d_tmem), "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc)
        : "memory");
}

__device__ __forceinline__ void mma_f8_tmem_a_acc(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                                  uint32_t idesc) {
    asm volatile(
        "{\n .reg .pred p;\n .reg .b64 bd;\n setp.ne.b32 p, 1, 0;\n mov.b64 bd, {%2, %3};\n"
        " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], bd, %4, p;\n}\n"
        ::"r"(d_tmem), "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *map, int32_t x, int32_t y,
                                            int32_t z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z),
          "r"(smem_u32(bar))
        : "memory");
}

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[N]);

template <>
__device__ __forceinline__ void tmem_ld_cols<8>(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7])
                 : "r"(taddr));
}

template <>
__device__ __forceinline__ void tmem_ld_cols<16>(uint32_t taddr, uint32_t (&r)[16]) {
    tmem_ld16(taddr, r);
}

template <int N>
__device__ __forceinline__ void tmem_wait_ld_pin(uint32_t (&a)[N], uint32_t (&b)[N]) {
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+r"(a[i]), "+r"(b[i]));
}

// kAccOut: the int32 test output (GemmParams::acc_out) instead of fp16 O.  A
// separate instantiation, so that the fp16-output kernel carries no code for it.
template <int BT, bool kAccOut>
__global__ void __launch_bounds__(kF8Threads, 1)
    w4a8_gemm_f8_kernel(const __grid_constant__ CUtensorMap plane_map, const __grid_constant__ CUtensorMap tg_map,
                        const __grid_constant__ CUtensorMap o_map, const GemmParams p) {
    using C = F8Cfg<BT>;
    constexpr int R = C::kRawStages, OPS = C::kOpStages, AUX = C::kAuxStages, DS = C::kDSets;
    constexpr int HT = BT / 2;  // tokens per drain thread
    extern __shared__ uint8_t smem_dyn[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *raw_base = smem;                                    // [B planes | t_g | 2 weight blocks]
    uint8_t *aux_base = raw_base + R * C::kRawSlotBytes;         // [meta 2x128x4 | t_g 2xBT]
    uint8_t *epi_base = aux_base + AUX * C::kAuxStageBytes;      // [int32 BTx128 | zeros 8 KB | fp16 BTx128]
    uint64_t *bars = reinterpret_cast<uint64_t *>(epi_base + C::kEpiRegion);
    uint64_t *raw_full = bars;           // weight blocks of a raw slot landed
    uint64_t *raw_empty = raw_full + R;
    uint64_t *act_full = raw_empty + R;  // activation planes and t_g of a raw slot landed
    uint64_t *op_full = act_full + R;
    uint64_t *aux_full = op_full + OPS;
    uint64_t *aux_empty = aux_full + AUX;
    uint64_t *d_full = aux_empty + AUX;
    uint64_t *d_empty = d_full + DS;
    uint64_t *mma_done = d_empty + DS;
    uint64_t *fix_bar = mma_done + 1;  // slot rows landed in the int32 staging (fix-up)
    uint64_t *pre_bar = fix_bar + 1;   // slot rows landed in the prefetch buffer
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(pre_bar + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *hdr_ok = abort_flag + 1;
    volatile int *is_last = abort_flag + 2;
    volatile int *fin_flag = abort_flag + 3;
    // 0: open; 1: the prefetch warp has loaded (or is loading) the finished
    // tile's slot; 2: the drain has decided without it.  Changed by atomicCAS.
    int *pre_state = const_cast<int *>(abort_flag + 4);
    float *tile_sx = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(bars) + 1024);
    int *tile_tx = reinterpret_cast<int *>(tile_sx + 128);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const uint64_t tmo = p.timeout_ns;

    if (threadIdx.x == 0) {
        griddep_launch_dependents();
        prefetch_tensormap(&plane_map);
        prefetch_tensormap(&tg_map);
        const PackedHeader *h = reinterpret_cast<const PackedHeader *>(p.packed);
        const bool ok = h->magic == kPackedMagic && h->version == kPackedVersion && h->N == p.N &&
                        h->K == p.K && h->group == p.group && h->illegal == 0u && p.group == 128;
        *hdr_ok = ok ? 1 : 0;
        *abort_flag = 0;
        *is_last = 0;
        *pre_state = 0;
        for (int i = 0; i < R; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], kF8ConvWarps + 1);  // one converter group + the MMA commit
            mbar_init(&act_full[i], 1);
        }
        for (int i = 0; i < OPS; ++i) mbar_init(&op_full[i], kF8ConvWarps);
        for (int i = 0; i < AUX; ++i) {
            mbar_init(&aux_full[i], kF8ConvWarps);
            mbar_init(&aux_empty[i], kF8EpiWarps);
        }
        for (int i = 0; i < DS; ++i) {
            mbar_init(&d_full[i], 1);
            mbar_init(&d_empty[i], kF8EpiWarps);
        }
        mbar_init(mma_done, 2);  // one commit per issuing thread
        mbar_init(fix_bar, 1);
        mbar_init(pre_bar, 1);
        fence_barrier_init();
    }
    // The zero block is read by bulk copies (async proxy).
    for (int i = threadIdx.x; i < static_cast<int>(C::kZeroBytes / 16); i += kF8Threads)
        st_shared_v4(smem_u32(epi_base + C::kStgI32Bytes) + 16u * i, 0u, 0u, 0u, 0u);
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

    if (run && warp == 0) {
        // ------------------------------------------------ TMA producer --
        if (lane == 0) {
            // Before the dependency wait (programmatic dependent launch): the
            // weight blocks of the first R stages, which no preceding kernel
            // writes.  Each stage's barrier is armed for all its bytes; the
            // activation operand copies follow after the wait.
            const bool withhold = (p.debug_flags & kDebugWithholdStage) != 0;
            int pre_max = withhold ? 1 : R;
            int pre = 0;
            {
                SegmentWalker w0(p, cta);
                Segment s0;
                while (pre < pre_max && w0.next(s0)) {
                    const int n_tile = s0.tile / p.tok_tiles;
                    const uint8_t *wrow = p.packed + kHeaderBytes + static_cast<size_t>(n_tile) * p.G * kBlockBytesG;
                    for (int k = s0.k0; k < s0.k1 && pre < pre_max; k += kGroupsPerStage, ++pre) {
                        const int ng = min(kGroupsPerStage, s0.k1 - k);
                        if (!weights_in_bounds(p, kHeaderBytes + (static_cast<unsigned long long>(n_tile) * p.G + k) * kBlockBytesG,
                                               static_cast<unsigned long long>(ng) * kBlockBytesG)) {
                            *abort_flag = 1;
                            pre_max = pre;  // the main loop stops at this stage
                            break;
                        }
                        uint8_t *dst = raw_base + pre * C::kRawSlotBytes;
                        mbar_arrive_expect_tx(&raw_full[pre], ng * kBlockBytesG);
                        tma_load_1d(dst + C::kWOff, wrow + static_cast<size_t>(k) * kBlockBytesG, ng * kBlockBytesG,
                                    &raw_full[pre]);
                    }
                }
            }
            griddep_wait();
            SegmentWalker walk(p, cta);
            Segment sg;
            int st = 0, issued = 0;
            bool stop = false;
            while (!stop && walk.next(sg)) {
                const int tok_tile = sg.tile % p.tok_tiles, n_tile = sg.tile / p.tok_tiles;
                const int m0 = tok_tile * BT;
                const uint8_t *wrow = p.packed + kHeaderBytes + static_cast<size_t>(n_tile) * p.G * kBlockBytesG;
                for (int k = sg.k0; k < sg.k1; k += kGroupsPerStage, ++st) {
                    const int ng = min(kGroupsPerStage, sg.k1 - k);
                    const int slot = st % R, use = st / R;
                    if (use > 0 && !mbar_wait(&raw_empty[slot], (use - 1) & 1, abort_flag, p.status, tmo)) {
                        stop = true;
                        break;
                    }
                    if (withhold && st == 1) {
                        stop = true;
                        break;
                    }
                    if (st >= pre &&
                        !weights_in_bounds(p, kHeaderBytes + (static_cast<unsigned long long>(n_tile) * p.G + k) * kBlockBytesG,
                                           static_cast<unsigned long long>(ng) * kBlockBytesG)) {
                        *abort_flag = 1;
                        stop = true;
                        break;
                    }
                    uint8_t *dst = raw_base + slot * C::kRawSlotBytes;
                    if (st >= pre) {
                        mbar_arrive_expect_tx(&raw_full[slot], ng * kBlockBytesG);
                        tma_load_1d(dst + C::kWOff, wrow + static_cast<size_t>(k) * kBlockBytesG, ng * kBlockBytesG,
                                    &raw_full[slot]);
                    }
                    mbar_arrive_expect_tx(&act_full[slot], ng * C::kPlaneGroupBytes + C::kTgBytes);
                    for (int g = 0; g < ng; ++g)
                        tma_load_3d(dst + g * C::kPlaneGroupBytes, &plane_map, (k + g) * kTileK, m0, 0,
                                    &act_full[slot]);
                    tma_load_2d(dst + C::kTgOff, &tg_map, m0, k, &act_full[slot]);
                    issued = st + 1;
                }
            }
            for (int t = (issued > R ? issued - R : 0); t < issued; ++t) {
                mbar_wait(&raw_full[t % R], (t / R) & 1, nullptr, p.status, tmo);
                mbar_wait(&act_full[t % R], (t / R) & 1, nullptr, p.status, tmo);
            }
            // Weight blocks issued before the dependency wait for stages the
            // walk never reached (it stopped early) must land as well.
            for (int t = issued; t < pre; ++t) mbar_wait(&raw_full[t % R], (t / R) & 1, nullptr, p.status, tmo);
        }
    } else if (run && (warp == 1 || warp == 2)) {
        // ------------------------------------------------ MMA issuers --
        // Two issuing threads take alternate stages (warp 1 even, warp 2
        // odd).  A barrier wait issued after
        // a thread's own MMAs queues behind them, so with one issuer every
        // wait left the tensor pipe idle; with two, one thread waits while
        // the other's MMAs execute.  tcgen05.commit tracks the MMAs of the
        // committing thread, which are exactly those of its own stages.
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(128, C::kNmma);  // e4m3 x e4m3 -> f32 for kind::f8f6f4
            const int par = warp - 1;
            SegmentWalker walk(p, cta);
            Segment sg;
            int st = 0;
            bool stop = false;
            while (!stop && walk.next(sg)) {
                for (int k = sg.k0; k < sg.k1; k += kGroupsPerStage, ++st) {
                    if ((st & 1) != par) continue;
                    const int ng = min(kGroupsPerStage, sg.k1 - k);
                    const int rs = st % R, os = st % OPS, ouse = st / OPS;
                    const int ds = st % DS, duse = st / DS;
                    if ((DS < AUX && duse > 0 &&
                         !mbar_wait(&d_empty[ds], (duse - 1) & 1, abort_flag, p.status, tmo)) ||
                        !mbar_wait(&op_full[os], ouse & 1, abort_flag, p.status, tmo)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t b_base = smem_u32(raw_base + rs * C::kRawSlotBytes);
                    for (int g = 0; g < ng; ++g) {
                        const uint32_t d_tmem = tmem + static_cast<uint32_t>((2 * ds + g) * C::kNmma);
                        const uint32_t a_tmem = tmem + C::kA0 + static_cast<uint32_t>(os) * 64u + 32u * g;
                        // the group's descriptor once; each k step adds 32 bytes / 16 to the
                        // address field (low word, no carry below 2^18)
                        const uint64_t bd0 = desc_kmajor_sw128(b_base + g * C::kPlaneGroupBytes);
                        const uint32_t lo = static_cast<uint32_t>(bd0), hi = static_cast<uint32_t>(bd0 >> 32);
                        mma_f8_tmem_a_first(d_tmem, a_tmem, lo, hi, idesc);
#pragma unroll
                        for (int kk = 1; kk < 4; ++kk) mma_f8_tmem_a_acc(d_tmem, a_tmem + 8u * kk, lo + 2u * kk, hi, idesc);
                    }
                    mma_commit(&raw_empty[rs]);
                    mma_commit(&d_full[ds]);
                }
            }
            // All of this thread's MMAs must finish before TMEM is released.
            mma_commit(mma_done);
            mbar_wait(mma_done, 0, nullptr, p.status, tmo);
        }
    } else if (run && warp == 3) {
        // --------------------------------------------- slot prefetch warp --
        // The split tile this CTA finishes (its range's last segment, when the
        // tile's first k-stage lies in this range) needs the other
        // contributors' sums from the tile's slot.  They publish them at the
        // start of their own ranges, usually long before this CTA reaches the
        // tile's end, so this warp polls the arrival counter and, once it is
        // complete, loads the slot into the prefetch buffer: the drain then
        // finishes the tile with neither a counter read nor a load on its
        // path.  pre_state (compare-and-swap) makes either this load or the
        // drain's own decision happen, never both.
        if (lane == 0 && !(p.debug_flags & kDebugAlwaysPublish)) {
            SegmentWalker w(p, cta);
            Segment sg, last{0, 0, 0, 0};
            while (w.next(sg)) last = sg;
            const bool split = last.k1 > last.k0 && !(last.k0 == 0 && last.k1 == p.G);
            const uint32_t tfirst = static_cast<uint32_t>(last.seq) * static_cast<uint32_t>(p.G);
            if (split && cta_of_stage(tfirst, p) == cta && slot_in_bounds<BT>(p, cta)) {
                griddep_wait();  // the workspace belongs to the preceding kernel until it completes
                const uint32_t others = static_cast<uint32_t>(
                    cta_of_stage(tfirst + static_cast<uint32_t>(p.G) - 1u, p) - cta);
                const uint64_t t0 = globaltimer_ns();
                bool ready = false;
                while (*abort_flag == 0 && abort_flag[4] == 0 && globaltimer_ns() - t0 < tmo) {
                    if (ld_acquire_gpu_u32(p.counters + cta) == others) {
                        ready = true;
                        break;
                    }
                    __nanosleep(256);
                }
                if (ready && atomicCAS(pre_state, 0, 1) == 0) {
                    const int32_t *slot = p.slots + static_cast<size_t>(cta) * (BT * kTileN);
                    fence_proxy_async_global();  // the counter acquire orders the load below
                    mbar_arrive_expect_tx(pre_bar, C::kStgI32Bytes);
                    tma_load_1d(epi_base + C::kPreOff, slot, C::kStgI32Bytes, pre_bar);
                    // Never left in flight at exit (the load reads the workspace).
                    mbar_wait(pre_bar, 0u, nullptr, p.status, tmo);
                }
            }
        }
    } else if (run && ((warp >= 4 && warp < 8) || warp >= 16)) {
        // ---------------------------------------------- converter warps --
        // Group 0 (warps 4-7) takes even stages, group 1 (warps 16-19) odd
        // ones, so one group's waits overlap the other's conversion.
        const int cg = warp >= 16 ? 1 : 0;
        const int wr = (warp & 3) * 32 + lane;  // weight row == TMEM lane
        const uint32_t a_lane = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        SegmentWalker walk(p, cta);
        Segment sg;
        int st = 0;
        bool stop = false;
        while (!stop && walk.next(sg)) {
            for (int k = sg.k0; k < sg.k1; k += kGroupsPerStage, ++st) {
                if ((st & 1) != cg) continue;
                const int ng = min(kGroupsPerStage, sg.k1 - k);
                const int rs = st % R, ruse = st / R, os = st % OPS, as = st % AUX, ause = st / AUX;
                // aux_empty of this slot means the drain finished stage st - AUX,
                // whose MMAs therefore completed: TMEM A slot os is free as well.
                // A parity wait is exact only once the slot's previous phase has
                // completed; with an odd ring depth the previous use of this raw
                // slot belongs to the other converter group, so first wait for
                // its release (raw_empty, which follows both of its fill phases).
                if ((ruse > 0 && !mbar_wait_warp(&raw_empty[rs], (ruse - 1) & 1, abort_flag, p.status, tmo)) ||
                    !mbar_wait_warp(&raw_full[rs], ruse & 1, abort_flag, p.status, tmo) ||
                    (ause > 0 && !mbar_wait_warp(&aux_empty[as], (ause - 1) & 1, abort_flag, p.status, tmo))) {
                    stop = true;
                    break;
                }
                tc_fence_after();
                const uint8_t *raw = raw_base + rs * C::kRawSlotBytes;
                const uint32_t wraw = smem_u32(raw) + C::kWOff;
                uint8_t *aux = aux_base + as * C::kAuxStageBytes;
                uint32_t *aux_meta = reinterpret_cast<uint32_t *>(aux);

                // Weights: row wr, 128 k per group -> 128 code bytes (e4m3 q * 2^-9)
                // -> 32 TMEM columns of this lane per group.
                for (int g = 0; g < ng; ++g) {
                    const uint32_t blk = wraw + g * kBlockBytesG;
                    uint32_t a_frag[32];
#pragma unroll
                    for (int pp = 0; pp < 4; ++pp) {
                        const uint4 v = ld_shared_v4(blk + ((pp * 128 + wr) << 4));
                        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            a_frag[8 * pp + 2 * j] = w4[j] & 0x0F0F0F0Fu;             // k = 8j .. 8j+3
                            a_frag[8 * pp + 2 * j + 1] = (w4[j] >> 4) & 0x0F0F0F0Fu;  // k = 8j+4 .. 8j+7
                        }
                    }
                    tmem_st32(a_lane + C::kA0 + static_cast<uint32_t>(os) * 64u + 32u * g, a_frag);
                    uint32_t meta;
                    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(meta) : "r"(blk + kCodeBytes + 4 * wr));
                    aux_meta[g * 128 + wr] = meta;
                }
                // The activation planes and sums of this stage, copied after the
                // dependency wait, must have landed before the sums are copied
                // and the MMAs (ordered after op_full) read the planes; the
                // weights above were converted without waiting for them.
                if (!mbar_wait_warp(&act_full[rs], ruse & 1, abort_flag, p.status, tmo)) {
                    tmem_wait_st();
                    stop = true;
                    break;
                }
                // Per-group activation sums for the drain: [2 groups][BT] int32.
                if ((warp & 3) == 0) {
                    const int *src = reinterpret_cast<const int *>(raw + C::kTgOff);
                    int *dstg = reinterpret_cast<int *>(aux + C::kAuxMetaBytes);
                    for (int i = lane; i < kGroupsPerStage * BT; i += 32) dstg[i] = src[i];
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&raw_empty[rs]);
                    mbar_arrive(&op_full[os]);
                    mbar_arrive(&aux_full[as]);
                }
            }
        }
    } else if (run && warp >= 8 && warp < 16) {
        // ------------------------------------------------- drain warps --
        griddep_wait();  // scales, workspace and output may belong to the preceding kernel
        const int ew = warp - 8;
        const int et = threadIdx.x - 256;          // 0..255 among the drain threads
        const int row = (ew & 3) * 32 + lane;      // weight row == TMEM lane
        const int hs = ew >> 2;                    // token half
        const uint32_t tl = tmem + (static_cast<uint32_t>((ew & 3) * 32) << 16);
        const int bits48 = 0x42400000;             // fp32 48.0
        uint32_t fix_n = 0;                        // fix-up loads consumed (fix_bar phases)
        SegmentWalker walk(p, cta);
        Segment sg;
        int st = 0;
        while (walk.next(sg)) {
            const int tok_tile = sg.tile % p.tok_tiles, n_tile = sg.tile / p.tok_tiles;
            const int m0 = tok_tile * BT, n = n_tile * kTileN + row;
            const bool split = !(sg.k0 == 0 && sg.k1 == p.G);
            const float sw = p.s_w ? h2f(p.s_w[n]) : 0.f;
            const uint32_t tfirst = static_cast<uint32_t>(sg.seq) * static_cast<uint32_t>(p.G);
            const int slot_idx = split ? cta_of_stage(tfirst, p) : 0;
            int32_t *slot = p.slots + static_cast<size_t>(slot_idx) * (BT * kTileN);
            named_bar_sync(2, kF8EpiThreads);
            if (et < BT) {
                const int m = m0 + et;
                tile_sx[et] = (m < p.M && p.s_x) ? h2f(p.s_x[m]) : 0.f;
                tile_tx[et] = 0;
            }
            named_bar_sync(2, kF8EpiThreads);
            int acc[HT];
#pragma unroll
            for (int i = 0; i < HT; ++i) acc[i] = 0;
            bool ok = true;
            for (int k = sg.k0; k < sg.k1 && ok; k += kGroupsPerStage, ++st) {
                const int ng = min(kGroupsPerStage, sg.k1 - k);
                const int ds = st % DS, duse = st / DS, as = st % AUX, ause = st / AUX;
                ok = mbar_wait_warp(&aux_full[as], ause & 1, abort_flag, p.status, tmo) &&
                     mbar_wait_warp(&d_full[ds], duse & 1, abort_flag, p.status, tmo);
                if (!ok) break;
                tc_fence_after();
                const uint8_t *aux = aux_base + as * C::kAuxStageBytes;
                const uint32_t *aux_meta = reinterpret_cast<const uint32_t *>(aux);
                const int *aux_tg = reinterpret_cast<const int *>(aux + C::kAuxMetaBytes);
                auto group_sum = [&](int g, const uint32_t (&dh)[HT], const uint32_t (&dl)[HT]) {
                    const uint32_t meta = aux_meta[g * 128 + row];
                    const int s = static_cast<int>(meta & 0xffu), z = static_cast<int>((meta >> 8) & 0xffu);
                    const int base = bits48 + 128 * static_cast<int>(meta >> 16);
                    uint32_t tg[HT];
                    const uint32_t tga = smem_u32(aux_tg + g * BT + hs * HT);
#pragma unroll
                    for (int q = 0; q < HT / 4; ++q)
                        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(tg[4 * q]), "=r"(tg[4 * q + 1]), "=r"(tg[4 * q + 2]), "=r"(tg[4 * q + 3])
                                     : "r"(tga + 16u * q));
#pragma unroll
                    for (int i = 0; i < HT; ++i) {
                        const float y = __fmaf_rn(__uint_as_float(dh[i]), 16.0f,
                                                  __fadd_rn(__uint_as_float(dl[i]), 48.0f));
                        const int corr = z * static_cast<int>(tg[i]) + base;
                        acc[i] += s * (__float_as_int(y) - corr);
                    }
                };
                const uint32_t dcol = static_cast<uint32_t>(2 * ds * C::kNmma + hs * HT);
                if constexpr (HT <= 8) {
                    // Both groups' accumulators in one TMEM round trip.
                    uint32_t dh0[HT], dl0[HT], dh1[HT], dl1[HT];
                    tmem_ld_cols<HT>(tl + dcol, dh0);
                    tmem_ld_cols<HT>(tl + dcol + BT, dl0);
                    if (ng > 1) {
                        tmem_ld_cols<HT>(tl + dcol + C::kNmma, dh1);
                        tmem_ld_cols<HT>(tl + dcol + C::kNmma + BT, dl1);
                    }
                    tmem_wait_ld_pin<HT>(dh0, dl0);
                    tmem_wait_ld_pin<HT>(dh1, dl1);
                    group_sum(0, dh0, dl0);
                    if (ng > 1) group_sum(1, dh1, dl1);
                } else {
                    for (int g = 0; g < ng; ++g) {
                        uint32_t dh[HT], dl[HT];
                        tmem_ld_cols<HT>(tl + dcol + g * C::kNmma, dh);
                        tmem_ld_cols<HT>(tl + dcol + g * C::kNmma + BT, dl);
                        tmem_wait_ld_pin<HT>(dh, dl);
                        group_sum(g, dh, dl);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&d_empty[ds]);
                    mbar_arrive(&aux_empty[as]);
                }
            }
            // ---- tile output.  Every drain thread takes the same named
            // barriers below; the abort flag, read by the issuing thread,
            // stops all global writes after a failed wait.
            const uint32_t stg = smem_u32(epi_base);                                   // int32 [BT][128]
            const uint8_t *zero_blk = epi_base + C::kStgI32Bytes;
            const uint32_t outb = smem_u32(epi_base + C::kStgI32Bytes + C::kZeroBytes);  // fp16 [BT][128]
            auto store_outputs = [&](const int (&val)[HT]) {
                // fp16 tile through the staging buffer, 16 tokens per tensor store
                if (et == 0) bulk_wait_read<0>();
                named_bar_sync(3, kF8EpiThreads);
#pragma unroll
                for (int i = 0; i < HT; ++i) {
                    const int ml = hs * HT + i;
                    st_shared_u16(outb + 2u * (ml * kTileN + row), out_fp16(val[i], 0, 0, tile_sx[ml], sw));
                }
                fence_proxy_async_smem();
                named_bar_sync(3, kF8EpiThreads);
                if (et == 0 && *abort_flag == 0) {
                    for (int b = 0; b < BT / 16; ++b)
                        tma_store_2d(&o_map, epi_base + C::kStgI32Bytes + C::kZeroBytes + b * 16 * kTileN * 2,
                                     n_tile * kTileN, m0 + 16 * b);
                    bulk_commit();
                }
            };
            if (!split) {
                if constexpr (kAccOut) {
#pragma unroll
                    for (int i = 0; i < HT; ++i) {
                        const int ml = hs * HT + i, m = m0 + ml;
                        if (ok && m < p.M) write_out(p, m, n, acc[i], 0, 0, tile_sx[ml], sw);
                    }
                } else {
                    store_outputs(acc);
                }
            } else {
                // If every other contributor has published its partial, this
                // CTA is the last one and finishes the tile with its own
                // partial still in registers.
                named_bar_sync(3, kF8EpiThreads);
                if (et == 0) {
                    int f = 0;
                    if (!slot_in_bounds<BT>(p, slot_idx)) *abort_flag = 1;
                    if (*abort_flag == 0 && !(p.debug_flags & kDebugAlwaysPublish)) {
                        // The tile's first k-stage is in this range only for the
                        // range's last segment.  If the prefetch warp already
                        // found every other partial published, its buffer holds
                        // the slot (f = 2); otherwise the claim stops it.
                        if (slot_idx == cta && atomicCAS(pre_state, 0, 2) == 1)
                            f = 2;
                        else
                            f = finish_directly(p, cta, slot_idx, tfirst, abort_flag) ? 1 : 0;
                    }
                    *fin_flag = f;
                }
                named_bar_sync(3, kF8EpiThreads);
                const int fmode = *fin_flag;
                const bool fin = fmode != 0;
                bool do_fix = fin;
                if (!fin) {
                    // Publish: the [BT][128] int32 partial (contiguous in the
                    // slot) as one bulk reduce-add; when it has completed, a
                    // fence and the arrival counter; the last arriver fixes up.
                    if (et == 0) bulk_wait_read<0>();
                    named_bar_sync(3, kF8EpiThreads);
#pragma unroll
                    for (int i = 0; i < HT; ++i)
                        st_shared_b32(stg + 4u * ((hs * HT + i) * kTileN + row), static_cast<uint32_t>(acc[i]));
                    fence_proxy_async_smem();
                    named_bar_sync(1, kF8EpiThreads);
                    if (et == 0) {
                        int last_cta = 0;
                        if (*abort_flag == 0) {
                            bulk_reduce_add_s32(slot, epi_base, C::kStgI32Bytes);
                            bulk_commit();
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
                    named_bar_sync(1, kF8EpiThreads);
                    do_fix = *is_last != 0;
                }
                if (do_fix) {
                    // Fix-up: the slot's sums (one bulk load) plus, when finishing
                    // directly, this CTA's own partial; then fp16 outputs, the
                    // slot re-zeroed and the counter reset.
                    uint32_t src = stg;
                    if (fmode == 2) {
                        // Loaded by the prefetch warp (the load always completes).
                        mbar_wait_warp(pre_bar, 0u, nullptr, p.status, tmo);
                        src = smem_u32(epi_base + C::kPreOff);
                    } else {
                        if (et == 0) {
                            bulk_wait_read<0>();         // the staging buffers are no longer read
                            fence_proxy_async_global();  // the counter acquire orders the load below
                            mbar_arrive_expect_tx(fix_bar, C::kStgI32Bytes);
                            tma_load_1d(epi_base, slot, C::kStgI32Bytes, fix_bar);
                        }
                        // The load always completes (it reads the workspace), so this
                        // wait ignores the abort flag: it is never left in flight.
                        mbar_wait_warp(fix_bar, fix_n & 1u, nullptr, p.status, tmo);
                        ++fix_n;
                    }
                    int tot[HT];
#pragma unroll
                    for (int i = 0; i < HT; ++i)
                        tot[i] = ld_shared_s32(src + 4u * ((hs * HT + i) * kTileN + row)) + (fin ? acc[i] : 0);
                    if constexpr (kAccOut) {
#pragma unroll
                        for (int i = 0; i < HT; ++i) {
                            const int ml = hs * HT + i;
                            if (*abort_flag == 0 && m0 + ml < p.M) write_out(p, m0 + ml, n, tot[i], 0, 0, tile_sx[ml], sw);
                        }
                    } else {
                        store_outputs(tot);
                    }
                    if (et == 0 && *abort_flag == 0) {
                        for (uint32_t b = 0; b < C::kStgI32Bytes; b += C::kZeroBytes)
                            bulk_store(reinterpret_cast<uint8_t *>(slot) + b, zero_blk, C::kZeroBytes);
                        bulk_commit();
                        p.counters[slot_idx] = 0u;
                    }
                }
            }
            named_bar_sync(1, kF8EpiThreads);
            if (*abort_flag != 0) break;
        }
        // Bulk copies read shared memory until they have read it: wait for that
        // before exit (their global writes complete on their own, and are
        // visible to every later grid, a dependent one's dependency wait included).
        if (et == 0) bulk_wait_read<0>();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int BT>
cudaError_t launch_f8_bt(const GemmArgs &a, const GemmPlan &plan, cudaStream_t stream) {
    using C = F8Cfg<BT>;
    static std::mutex mu;
    static bool configured[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!configured[dev]) {
            for (auto kern : {w4a8_gemm_f8_kernel<BT, false>, w4a8_gemm_f8_kernel<BT, true>}) {
                e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::kSmemBytes));
                if (e != cudaSuccess) return e;
            }
            configured[dev] = true;
        }
    }
    CUtensorMapEncodeTiledFn enc = get_encode_fn();
    if (!enc) return cudaErrorNotSupported;
    uint8_t *ws = static_cast<uint8_t *>(a.ws);
    const uint8_t *act = static_cast<const uint8_t *>(a.act);
    if (!act) {
        // No precomputed operand: build it from Qx in the workspace first.
        uint8_t *scratch = ws + plan.act_offset;
        e = launch_act_operand(a.Qx, a.M, a.K, kPathF8, scratch, stream);
        if (e != cudaSuccess) return e;
        act = scratch;
    }
    // B planes [2][M][K] bytes: one box = one group = {128 k, BT tokens, 2 planes}.
    CUtensorMap plane_map, tg_map;
    {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.K), static_cast<cuuint64_t>(a.M), 2u};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.K),
                                       static_cast<cuuint64_t>(a.M) * static_cast<cuuint64_t>(a.K)};
        const cuuint32_t box[3] = {128u, static_cast<cuuint32_t>(BT), 2u};
        const cuuint32_t estr[3] = {1u, 1u, 1u};
        CUresult cr = enc(&plane_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(act), dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    // t_g [K/128][Mp] int32: one box = {BT tokens, 2 groups}; tokens past M read as 0.
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.M), static_cast<cuuint64_t>(plan.G)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(act_tg_pitch(a.M)) * 4u};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(BT), static_cast<cuuint32_t>(kGroupsPerStage)};
        const cuuint32_t estr[2] = {1u, 1u};
        CUresult cr = enc(&tg_map, CU_TENSOR_MAP_DATA_TYPE_INT32, 2,
                          const_cast<uint8_t *>(act + act_planes_bytes(a.M, a.K)), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    // fp16 output O [M][N]: one store box = 128 rows of a tile x 16 tokens (unused in the int32 test mode).
    CUtensorMap o_map{};
    if (a.O) {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.N), static_cast<cuuint64_t>(a.M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.N) * 2u};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(kTileN), 16u};
        const cuuint32_t estr[2] = {1u, 1u};
        CUresult cr = enc(&o_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.O, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    GemmParams p;
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
    if (a.acc_out)
        return launch_kernel(w4a8_gemm_f8_kernel<BT, true>, dim3(plan.ctas), dim3(kF8Threads), C::kSmemBytes, stream,
                             a.pdl, plane_map, tg_map, o_map, p);
    return launch_kernel(w4a8_gemm_f8_kernel<BT, false>, dim3(plan.ctas), dim3(kF8Threads), C::kSmemBytes, stream,
                         a.pdl, plane_map, tg_map, o_map, p);
}

}  // namespace

cudaError_t launch_gemm_f8(const GemmArgs &a, const GemmPlan &plan, cudaStream_t stream) {
    if (a.group != 128) return cudaErrorInvalidValue;
    switch (plan.BT) {
        case 16: return launch_f8_bt<16>(a, plan, stream);
        case 32: return launch_f8_bt<32>(a, plan, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qoq

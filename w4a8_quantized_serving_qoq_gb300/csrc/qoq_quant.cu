// Quantizers on the device:
//  * per-token symmetric INT8 activation quantization (the step the QServe
//    runtime fuses into the kernel before each GEMM; here a standalone,
//    memory-bound kernel), and
//  * the offline progressive group weight quantizer (per-channel INT8 in the
//    protective range [-119, 119], then per-group UINT4 with a UINT8 scale and
//    a UINT4 zero), plus the per-channel UINT4 variant.
// Sources: "QServe: W4A8KV4 Quantization and System Co-design for Efficient LLM
// Serving" (papercache summary), sections "整数量化" (eq. 1), "渐进式组量化"
// (eq. 4/5) and "保护性量化范围"; "QServe：把 W4A8KV4 的理论收益做成实测吞吐的
// 量化—系统协同设计" (zenmind review), sections 3.1 and 3.2.
// Every float that decides an integer code is an IEEE fp32 division rounded
// to nearest-even (__fdiv_rn), then rounded half-to-even to an integer.
#include <cuda_fp16.h>

#include <mutex>

#include "qoq_internal.h"
#include "qoq_device.cuh"

namespace qoq {
namespace {

__device__ __forceinline__ float h2f(uint16_t b) { return __half2float(__ushort_as_half(b)); }
__device__ __forceinline__ uint16_t f2h_rn(float f) { return __half_as_ushort(__float2half_rn(f)); }

__device__ __forceinline__ int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

// 16-byte asynchronous copy global -> shared (L2 only), tracked by the
// issuing thread's commit groups; cp_async_wait<N> returns once at most N of
// its groups are still in flight (a hardware wait on the thread's own copies).
__device__ __forceinline__ void cp_async16(uint32_t smem_dst, const void *gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_dst), "l"(gmem_src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Round-half-even of a / b for integers, b > 0.
__device__ __forceinline__ int rne_div(int a, int b) {
    int q = a / b, r = a - q * b;
    if (r < 0) { q -= 1; r += b; }
    if (2 * r > b || (2 * r == b && (q & 1))) q += 1;
    return q;
}

// Block-wide reduction (blockDim.x a multiple of 32, at most 1024): warp
// shuffles, one partial per warp in shared memory, then every warp reduces
// the partials with shuffles again (identity for the missing lanes).
template <typename T, typename Op>
__device__ __forceinline__ T block_reduce(T v, Op op, T *sh, T identity) {
    for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    __syncthreads();
    if (lane == 0) sh[warp] = v;
    __syncthreads();
    v = lane < nw ? sh[lane] : identity;
    for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

struct MaxOp { __device__ float operator()(float a, float b) const { return fmaxf(a, b); } };
struct MinOp { __device__ float operator()(float a, float b) const { return fminf(a, b); } };
struct SumOp { __device__ int operator()(int a, int b) const { return a + b; } };

// Round-to-nearest-even of t by one addition: for |t| < 2^22 the fp32 sum
// t + 1.5 * 2^23 has unit spacing, so the addition rounds t to an integer
// (ties to even), and the sum's bits are 0x4B400000 + rne(t): its low byte
// is the two's-complement INT8 code.
constexpr float kRneMagic = 12582912.0f;

// Quantize eight fp16 values (one 16-byte load) with scale sf; returns the
// eight INT8 codes as two words, adds them to sum and, for kF16, also returns
// them as fp16 (exact integers) in *f16.
// rne(x / s) with the quotient rounded to fp32 first, as the definition
// states, without a division per element: inv = RN(1/s) and t = RN(x * inv)
// differ from x/s by at most 127.1 * 2^-23 < 1.6e-5, and RN(x/s) by at most
// half an ulp of 127 (3.9e-6) more.  So t and RN(x/s) round to the same
// integer unless t lies within 3e-5 of a half-integer (|t - rne(t)| >
// 0.49997); there the IEEE division decides.  Codes are clamped to
// [-127, 127] (clamping t first gives the same codes: rne is monotone and
// maps +-127 to themselves); s = 0 gives inv = 0 and zero codes.  The clamp
// can only act when s is an fp16 subnormal (kClamp): a normal s is within
// 2^-11 relative of max|x| / 127, so |t| < 127.07 and rne(t) is in range.
// Paired fp32 arithmetic (sm_100 and later): one instruction rounds two
// independent fp32 operations exactly as two scalar ones would.
__device__ __forceinline__ uint64_t f32x2_pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f32x2_unpack(uint64_t v, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f32x2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f32x2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f32x2_sub(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

template <bool kF16, bool kClamp>
__device__ __forceinline__ uint2 quant8(const uint4 v, float sf, float inv, int &sum, uint4 *f16) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float t[8], r[8], qf[8];  // x / s, t + magic (the code in its low byte), rne(t)
    bool tie = false;
    if constexpr (!kClamp) {
        // the same roundings as the scalar form below, two values per instruction
        const uint64_t inv2 = f32x2_pack(inv, inv), mg2 = f32x2_pack(kRneMagic, kRneMagic);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint64_t T = f32x2_mul(f32x2_pack(h2f(static_cast<uint16_t>(w[j] & 0xffffu)),
                                                    h2f(static_cast<uint16_t>(w[j] >> 16))),
                                         inv2);
            const uint64_t R = f32x2_add(T, mg2);
            const uint64_t Q = f32x2_sub(R, mg2);
            float d0, d1;
            f32x2_unpack(f32x2_sub(T, Q), d0, d1);
            f32x2_unpack(T, t[2 * j], t[2 * j + 1]);
            f32x2_unpack(R, r[2 * j], r[2 * j + 1]);
            f32x2_unpack(Q, qf[2 * j], qf[2 * j + 1]);
            tie |= fabsf(d0) > 0.49997f || fabsf(d1) > 0.49997f;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint16_t hb = static_cast<uint16_t>((j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xffffu));
            t[j] = fminf(fmaxf(__fmul_rn(h2f(hb), inv), -127.0f), 127.0f);
            r[j] = __fadd_rn(t[j], kRneMagic);
            qf[j] = __fsub_rn(r[j], kRneMagic);
            tie |= fabsf(__fsub_rn(t[j], qf[j])) > 0.49997f;
        }
    }
    if (tie) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (fabsf(__fsub_rn(t[j], qf[j])) > 0.49997f) {
                const uint16_t hb = static_cast<uint16_t>((j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xffffu));
                const int q = clampi(__float2int_rn(__fdiv_rn(h2f(hb), sf)), -127, 127);
                qf[j] = static_cast<float>(q);
                r[j] = __fadd_rn(qf[j], kRneMagic);
            }
        }
    }
    uint32_t b[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) b[j] = __float_as_uint(r[j]);
    const uint32_t q0 = __byte_perm(__byte_perm(b[0], b[1], 0x0040u), __byte_perm(b[2], b[3], 0x0040u), 0x5410u);
    const uint32_t q1 = __byte_perm(__byte_perm(b[4], b[5], 0x0040u), __byte_perm(b[6], b[7], 0x0040u), 0x5410u);
    sum = __dp4a(static_cast<int>(q0), 0x01010101, sum);
    sum = __dp4a(static_cast<int>(q1), 0x01010101, sum);
    if constexpr (kF16) {
        uint32_t h[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __half2 p = __floats2half2_rn(qf[2 * j], qf[2 * j + 1]);
            h[j] = *reinterpret_cast<const uint32_t *>(&p);
        }
        *f16 = make_uint4(h[0], h[1], h[2], h[3]);
    }
    return make_uint2(q0, q1);
}

// Running max of |x| over eight fp16 values, taken on packed halves (the
// maximum of fp16 values is exact in fp16).
__device__ __forceinline__ float amax8(const uint4 v, float amax) {
    const uint32_t w[4] = {v.x & 0x7fff7fffu, v.y & 0x7fff7fffu, v.z & 0x7fff7fffu, v.w & 0x7fff7fffu};
    const __half2 m = __hmax2(__hmax2(*reinterpret_cast<const __half2 *>(&w[0]), *reinterpret_cast<const __half2 *>(&w[1])),
                              __hmax2(*reinterpret_cast<const __half2 *>(&w[2]), *reinterpret_cast<const __half2 *>(&w[3])));
    return fmaxf(amax, fmaxf(__low2float(m), __high2float(m)));
}

// fp8-path operand bytes of eight INT8 codes (two words): u = Qx + 128
// (flip of the sign bit), then its high and low nibble planes.
__device__ __forceinline__ void split_u(uint2 q, uint2 &hi, uint2 &lo) {
    const uint32_t u0 = q.x ^ 0x80808080u, u1 = q.y ^ 0x80808080u;
    hi = make_uint2((u0 >> 4) & 0x0F0F0F0Fu, (u1 >> 4) & 0x0F0F0F0Fu);
    lo = make_uint2(u0 & 0x0F0F0F0Fu, u1 & 0x0F0F0F0Fu);
}

// fp16-path operand of four INT8 codes (one word): the same integers as
// fp16 (exact), two fp16x2 words.
__device__ __forceinline__ uint2 int8x4_to_f16x4(uint32_t w) {
    uint32_t h[4];
#pragma unroll
    for (int b = 0; b < 4; ++b)
        h[b] = __half_as_ushort(__int2half_rn(static_cast<int>(static_cast<int8_t>((w >> (8 * b)) & 0xffu))));
    return make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
}

constexpr int kActCache = 4;  // 16-byte items per thread kept in registers between the passes

// Where the fp16 row the quantizer sees comes from: the activations
// themselves, or the output of the fp16 kernel in front of the GEMM, into
// which the QServe runtime fuses the quantization ("QServe: W4A8KV4
// Quantization and System Co-design for Efficient LLM Serving", section
// "QServe系统运行时"): the norm before the QKV projection and the FFN's first
// layer, the SwiGLU activation before the FFN's second layer.
enum : int {
    kSrcX = 0,        // X [M][K]
    kSrcRmsNorm = 1,  // fp16(X * r * gamma), r = 1 / sqrt(mean_k X^2 + eps), X [M][K]
    kSrcSiluMul = 2,  // fp16(SiLU(G) * U) of H = [G | U] [M][2K], SiLU(g) = g / (1 + e^-g)
};

struct RowSrc {
    const uint16_t *X;      // X, or H for kSrcSiluMul
    const uint16_t *gamma;  // [K] (kSrcRmsNorm)
    float eps;              // (kSrcRmsNorm)
    uint16_t *Y;            // optional [M][K]: the fp16 rows the quantizer saw
};

struct AddF { __device__ float operator()(float a, float b) const { return __fadd_rn(a, b); } };

__device__ __forceinline__ float sumsq8(const uint4 v, float ss) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float a = h2f(static_cast<uint16_t>(w[j] & 0xffffu)), b = h2f(static_cast<uint16_t>(w[j] >> 16));
        ss = __fmaf_rn(a, a, ss);
        ss = __fmaf_rn(b, b, ss);
    }
    return ss;
}

// Eight normalized values: fp16((x * r) * gamma), each product rounded in
// fp32 (paired fp32 multiplies, the same roundings as scalar ones).
__device__ __forceinline__ uint4 norm8(const uint4 x, const uint4 g, float r) {
    const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, gs[4] = {g.x, g.y, g.z, g.w};
    const uint64_t r2 = f32x2_pack(r, r);
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint64_t X = f32x2_pack(h2f(static_cast<uint16_t>(xs[j] & 0xffffu)), h2f(static_cast<uint16_t>(xs[j] >> 16)));
        const uint64_t G = f32x2_pack(h2f(static_cast<uint16_t>(gs[j] & 0xffffu)), h2f(static_cast<uint16_t>(gs[j] >> 16)));
        float lo, hi;
        f32x2_unpack(f32x2_mul(f32x2_mul(X, r2), G), lo, hi);
        const __half2 p = __floats2half2_rn(lo, hi);
        o[j] = *reinterpret_cast<const uint32_t *>(&p);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// fp16(SiLU(g) * u) in fp32 with the fast intrinsics: __expf (relative
// error below 1.3e-5 for |g| <= 90, i.e. wherever fp16 inputs give a
// non-zero result), __fdividef (2 ulp) and a product, so y is within 1.4e-5
// relative of the exact value before its fp16 rounding (2^-11 relative).
// Large negative g: e^-g overflows to inf (or 1 + e^-g exceeds 2^126) and
// SiLU(g) = -0, where the exact value rounds to zero in fp16 too.
__device__ __forceinline__ float silu_mul1(float g, float u) {
    return __fmul_rn(__fdividef(g, __fadd_rn(1.0f, __expf(-g))), u);
}

__device__ __forceinline__ uint4 silu8(const uint4 g, const uint4 u) {
    const uint32_t gs[4] = {g.x, g.y, g.z, g.w}, us[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t lo = f2h_rn(silu_mul1(h2f(static_cast<uint16_t>(gs[j] & 0xffffu)),
                                             h2f(static_cast<uint16_t>(us[j] & 0xffffu))));
        const uint32_t hi = f2h_rn(silu_mul1(h2f(static_cast<uint16_t>(gs[j] >> 16)), h2f(static_cast<uint16_t>(us[j] >> 16))));
        o[j] = lo | (hi << 16);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// The outputs of one token row m: the codes, the optional fp16 row the
// quantizer saw, and the activation operand of kind kAct (0 none, 1 the fp16
// copy of Qx, 2 the fp8-path planes of u = Qx + 128 and the per-group sums
// t_g, whose padding columns M .. Mp-1 the last row also zero-fills).
template <int kAct>
struct RowOut {
    uint2 *qrow;
    uint4 *yrow;
    uint4 *frow = nullptr;
    uint2 *hrow = nullptr, *lrow = nullptr;
    int32_t *tg = nullptr;
    int pitch;
    size_t m;
    int M;
    __device__ RowOut(int8_t *Qx, uint16_t *Y, uint8_t *act, size_t m_, int M_, int K)
        : qrow(reinterpret_cast<uint2 *>(Qx + m_ * K)),
          yrow(Y ? reinterpret_cast<uint4 *>(Y + m_ * K) : nullptr),
          pitch(act_tg_pitch(M_)),
          m(m_),
          M(M_) {
        if (kAct == 1) frow = reinterpret_cast<uint4 *>(act + 2 * m_ * K);
        if (kAct == 2) {
            hrow = reinterpret_cast<uint2 *>(act + m_ * K);
            lrow = reinterpret_cast<uint2 *>(act + static_cast<size_t>(M_) * K + m_ * K);
            tg = reinterpret_cast<int32_t *>(act + act_planes_bytes(M_, K));
        }
    }
};

// Quantizes and writes item i (8 values v) of the row, adding its codes to
// tsum.  Lanes with i >= nv write nothing; for kind 2 every lane of the warp
// must call it together (the 16 items of a 128-k group are summed by
// half-warp shuffles, so i runs over consecutive items in each half-warp).
// kNoClampPath: rows with a normal scale take the quantizer without the
// clamp (a second inlined copy).  Measured faster in the 256-thread
// row-streaming kernel (rows up to 16 KB: quant 16.7 -> 15.8 us at M = 4096,
// K = 4096) and slower in the 512-thread one (K = 14336: 48.8 -> 52.4 us);
// the one-CTA-per-row kernel, register-capped at 1,024-thread rows, keeps
// the single clamped copy too.
template <int kAct, bool kNoClampPath>
__device__ __forceinline__ void emit8(const RowOut<kAct> &o, int i, int nv, const uint4 v, float sf, float inv,
                                      int &tsum) {
    int part = 0;
    uint2 q = make_uint2(0u, 0u);
    if (i < nv) {
        uint4 f16;
        if (kNoClampPath && sf >= 6.103515625e-05f)  // 2^-14, the smallest normal fp16 (uniform across the row)
            q = quant8<kAct == 1, false>(v, sf, inv, part, &f16);
        else
            q = quant8<kAct == 1, true>(v, sf, inv, part, &f16);
        o.qrow[i] = q;
        if (o.yrow) o.yrow[i] = v;
        if (kAct == 1) o.frow[i] = f16;
    }
    tsum += part;
    if (kAct == 2) {
        if (i < nv) {
            uint2 hi, lo;
            split_u(q, hi, lo);
            o.hrow[i] = hi;
            o.lrow[i] = lo;
        }
#pragma unroll
        for (int s = 8; s > 0; s >>= 1) part += __shfl_xor_sync(0xffffffffu, part, s);
        if ((threadIdx.x & 15) == 0 && i < nv) {
            int32_t *tcol = o.tg + static_cast<size_t>(i >> 4) * o.pitch;
            tcol[o.m] = part;
            if (o.m + 1 == static_cast<size_t>(o.M))
                for (int mm = o.M; mm < o.pitch; ++mm) tcol[mm] = 0;
        }
    }
}

// One CTA per token row.  The row is the fp16 row of the source (kSrc);
// s_x = fp16(max|x| / 127); Qx = clamp(rne(x / s_x), -127, 127); an all-zero
// scale gives an all-zero row; t_x = row sum of Qx.  kAct selects an
// activation operand written alongside: 0 none, 1 the fp16 copy of Qx, 2 the
// fp8-path planes of u = Qx + 128 and the per-group sums t_g (the last row's
// CTA also zero-fills the padding columns M .. Mp-1 of t_g).
// The trip count of every loop is uniform across the CTA (blockDim.x is a
// multiple of 32), so the half-warp shuffles that sum one 128-k group (16
// items of 8) always run with every lane present.  A source item is
// recomputed from the same loads with the same rounded operations wherever
// it is needed again, so every pass sees identical fp16 values.
template <int kAct, int kSrc>
__global__ void __launch_bounds__(kSrc == kSrcX ? 1024 : 512) quant_act_kernel(const RowSrc src, int M, int K, int8_t *__restrict__ Qx,
                                 uint16_t *__restrict__ s_x, int32_t *__restrict__ t_x,
                                 uint8_t *__restrict__ act) {
    __shared__ float shf[32];
    __shared__ int shi[32];
    // Under programmatic dependent launch: let the next kernel start
    // launching, then wait for the previous one before reading the source
    // or writing.  The source row is prefetched into L2 first (16-byte
    // aligned, a multiple of 16 bytes: K % 8 == 0): the wait covers the
    // previous kernel's writes, and L2 holds the current data of every line.
    const size_t m = blockIdx.x;
    const uint4 *row = reinterpret_cast<const uint4 *>(src.X + m * (kSrc == kSrcSiluMul ? 2 * static_cast<size_t>(K) : K));
    const uint4 *urow = row + (K >> 3);  // up half of an [G | U] row
    const uint4 *grow = reinterpret_cast<const uint4 *>(src.gamma);
    if (threadIdx.x == 0) {
        griddep_launch_dependents();
        prefetch_l2_bulk(row, static_cast<uint32_t>(K) * 2u);
        if (kSrc == kSrcSiluMul) prefetch_l2_bulk(urow, static_cast<uint32_t>(K) * 2u);
    }
    griddep_wait();
    const int nv = K >> 3, bd = blockDim.x, tid = threadIdx.x;
    uint4 cache[kActCache];
    float r = 0.f;
    if constexpr (kSrc == kSrcRmsNorm) {
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < kActCache; ++j) {
            const int i = tid + j * bd;
            cache[j] = make_uint4(0u, 0u, 0u, 0u);
            if (i < nv) cache[j] = __ldg(row + i);
            ss = sumsq8(cache[j], ss);
        }
        for (int i = tid + kActCache * bd; i < nv; i += bd) ss = sumsq8(__ldg(row + i), ss);
        ss = block_reduce(ss, AddF(), shf, 0.f);
        const float v = __fadd_rn(__fdiv_rn(ss, static_cast<float>(K)), src.eps);
        r = v > 0.f ? __frsqrt_rn(v) : 0.f;  // an all-zero row with eps = 0 stays zero
    }
    // fp16 item i (8 values) of the row the quantizer sees.
    auto item = [&](int i) -> uint4 {
        if constexpr (kSrc == kSrcRmsNorm) return norm8(__ldg(row + i), __ldg(grow + i), r);
        else if constexpr (kSrc == kSrcSiluMul) return silu8(__ldg(row + i), __ldg(urow + i));
        else return __ldg(row + i);
    };
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < kActCache; ++j) {
        const int i = tid + j * bd;
        if constexpr (kSrc == kSrcRmsNorm) {
            cache[j] = i < nv ? norm8(cache[j], __ldg(grow + i), r) : make_uint4(0u, 0u, 0u, 0u);
        } else {
            cache[j] = i < nv ? item(i) : make_uint4(0u, 0u, 0u, 0u);
        }
        amax = amax8(cache[j], amax);
    }
    for (int i = tid + kActCache * bd; i < nv; i += bd) amax = amax8(item(i), amax);
    amax = block_reduce(amax, MaxOp(), shf, 0.f);
    const uint16_t sbits = f2h_rn(__fdiv_rn(amax, 127.0f));
    const float sf = h2f(sbits);
    const float inv = sf != 0.f ? __frcp_rn(sf) : 0.f;

    const RowOut<kAct> out(Qx, kSrc != kSrcX ? src.Y : nullptr, act, m, M, K);
    int tsum = 0;
#pragma unroll
    for (int j = 0; j < kActCache; ++j)
        if (j * bd < nv) emit8<kAct, false>(out, tid + j * bd, nv, cache[j], sf, inv, tsum);
    for (int base = kActCache * bd; base < nv; base += bd) {
        const int i = base + tid;
        emit8<kAct, false>(out, i, nv, i < nv ? item(i) : make_uint4(0u, 0u, 0u, 0u), sf, inv, tsum);
    }
    if (t_x) tsum = block_reduce(tsum, SumOp(), shi, 0);  // t_x is uniform across the CTA
    if (tid == 0) {
        s_x[m] = sbits;
        if (t_x) t_x[m] = tsum;
    }
}

// The same quantizer for many rows (bandwidth-bound sizes): persistent CTAs
// take rows blockIdx.x, blockIdx.x + gridDim.x, ... and stream them through
// a ring of kRing row buffers in shared memory with 16-byte asynchronous
// copies, kRing - 1 rows ahead of the one being quantized, so each SM keeps
// several rows in flight with few registers.  The row is then read from
// shared memory only: the norm / activation values overwrite the source in
// place after the pass that computes them (with the max), and the last pass
// quantizes them.  gamma (kSrcRmsNorm) is staged once per CTA.  Arithmetic,
// rounding and outputs are those of quant_act_kernel.  Every loop's trip
// count is uniform across the CTA, as the group-sum shuffles require.
template <int kAct, int kSrc, int kRing, int kT>
__global__ void __launch_bounds__(kT) quant_rows_kernel(const RowSrc src, int M, int K, int8_t *__restrict__ Qx,
                                                        uint16_t *__restrict__ s_x, int32_t *__restrict__ t_x,
                                                        uint8_t *__restrict__ act) {
    extern __shared__ uint4 rows_smem[];
    __shared__ float shf[32];
    __shared__ int shi[32];
    const int nv = K >> 3;                                  // 16-byte items (8 values) of a row
    const int items = kSrc == kSrcSiluMul ? 2 * nv : nv;    // source items per row ([G | U] for SiLU-mul)
    const int tid = threadIdx.x;
    // Rows of this CTA (the grid is at most M wide).
    const int rows = (M - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1;
    uint4 *gam = rows_smem;                                      // [nv] (kSrcRmsNorm)
    uint4 *ring = rows_smem + (kSrc == kSrcRmsNorm ? nv : 0);   // kRing x [items]
    const uint4 *srcv = reinterpret_cast<const uint4 *>(src.X);
    if (tid == 0) griddep_launch_dependents();
    griddep_wait();  // the source rows may be written by the preceding kernel
    auto issue = [&](int t) {
        if (t < rows) {
            const size_t m = blockIdx.x + static_cast<size_t>(t) * gridDim.x;
            const uint4 *row = srcv + m * items;
            const uint32_t dst = smem_u32(ring + static_cast<size_t>(t % kRing) * items);
            for (int i = tid; i < items; i += kT) cp_async16(dst + 16u * i, row + i);
        }
        cp_async_commit();  // possibly empty: every thread commits one group per row index
    };
    if constexpr (kSrc == kSrcRmsNorm) {
        const uint4 *g = reinterpret_cast<const uint4 *>(src.gamma);
        for (int i = tid; i < nv; i += kT) cp_async16(smem_u32(gam + i), g + i);  // joins row 0's group
    }
#pragma unroll
    for (int t = 0; t < kRing - 1; ++t) issue(t);
    for (int t = 0; t < rows; ++t) {
        issue(t + kRing - 1);
        cp_async_wait<kRing - 1>();  // this thread's copies of row t have landed
        __syncthreads();             // ... and every other thread's
        const size_t m = blockIdx.x + static_cast<size_t>(t) * gridDim.x;
        uint4 *buf = ring + static_cast<size_t>(t % kRing) * items;
        float r = 0.f;
        if constexpr (kSrc == kSrcRmsNorm) {
            float ss = 0.f;
            for (int i = tid; i < nv; i += kT) ss = sumsq8(buf[i], ss);
            ss = block_reduce(ss, AddF(), shf, 0.f);
            const float v = __fadd_rn(__fdiv_rn(ss, static_cast<float>(K)), src.eps);
            r = v > 0.f ? __frsqrt_rn(v) : 0.f;
        }
        float amax = 0.f;
        for (int i = tid; i < nv; i += kT) {
            uint4 y = buf[i];
            if constexpr (kSrc == kSrcRmsNorm) y = norm8(y, gam[i], r);
            if constexpr (kSrc == kSrcSiluMul) y = silu8(y, buf[nv + i]);
            if constexpr (kSrc != kSrcX) buf[i] = y;  // this thread's own item, read back below
            amax = amax8(y, amax);
        }
        amax = block_reduce(amax, MaxOp(), shf, 0.f);
        const uint16_t sbits = f2h_rn(__fdiv_rn(amax, 127.0f));
        const float sf = h2f(sbits);
        const float inv = sf != 0.f ? __frcp_rn(sf) : 0.f;
        const RowOut<kAct> out(Qx, kSrc != kSrcX ? src.Y : nullptr, act, m, M, K);
        int tsum = 0;
        for (int base = 0; base < nv; base += kT) {
            const int i = base + tid;
            emit8<kAct, kT == 256>(out, i, nv, i < nv ? buf[i] : make_uint4(0u, 0u, 0u, 0u), sf, inv, tsum);
        }
        if (t_x) tsum = block_reduce(tsum, SumOp(), shi, 0);
        if (tid == 0) {
            s_x[m] = sbits;
            if (t_x) t_x[m] = tsum;
        }
        __syncthreads();  // buffer t % kRing is refilled by the next iteration's copies
    }
    cp_async_wait<0>();
}

// fp16-path activation operand from INT8 activations: 8 codes per thread
// and step, grid-stride over the whole matrix.
__global__ void act_operand_f16_kernel(const int8_t *__restrict__ Qx, size_t n8, uint8_t *__restrict__ act) {
    const uint2 *src = reinterpret_cast<const uint2 *>(Qx);
    uint4 *dst = reinterpret_cast<uint4 *>(act);
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n8;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const uint2 q = __ldg(src + i);
        const uint2 a = int8x4_to_f16x4(q.x), b = int8x4_to_f16x4(q.y);
        dst[i] = make_uint4(a.x, a.y, b.x, b.y);
    }
}

// fp8-path activation operand from INT8 activations: one CTA per token row,
// one 16-byte item (16 codes) per thread and step; eight items form a group.
__global__ void act_operand_kernel(const int8_t *__restrict__ Qx, int M, int K, uint8_t *__restrict__ act) {
    const size_t m = blockIdx.x;
    const int nv = K >> 4, pitch = act_tg_pitch(M);
    const uint4 *row = reinterpret_cast<const uint4 *>(Qx + m * K);
    uint4 *hrow = reinterpret_cast<uint4 *>(act + m * K);
    uint4 *lrow = reinterpret_cast<uint4 *>(act + static_cast<size_t>(M) * K + m * K);
    int32_t *tg = reinterpret_cast<int32_t *>(act + act_planes_bytes(M, K));
    for (int base = 0; base < nv; base += blockDim.x) {
        const int i = base + threadIdx.x;
        int part = 0;
        if (i < nv) {
            const uint4 v = __ldg(row + i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                part = __dp4a(static_cast<int>(w[j]), 0x01010101, part);
                const uint32_t u = w[j] ^ 0x80808080u;
                hi[j] = (u >> 4) & 0x0F0F0F0Fu;
                lo[j] = u & 0x0F0F0F0Fu;
            }
            hrow[i] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            lrow[i] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if ((threadIdx.x & 7) == 0 && i < nv) {
            int32_t *tcol = tg + static_cast<size_t>(i >> 3) * pitch;
            tcol[m] = part;
            if (m + 1 == static_cast<size_t>(M))
                for (int mm = M; mm < pitch; ++mm) tcol[mm] = 0;  // padding columns
        }
    }
}

// Progressive group quantization of one weight row per CTA.
__global__ void quantize_group_kernel(const uint16_t *__restrict__ W, int K, int g,
                                      uint8_t *__restrict__ q4, uint8_t *__restrict__ s_g,
                                      uint8_t *__restrict__ zp, uint16_t *__restrict__ s_w) {
    __shared__ float shf[32];
    const size_t n = blockIdx.x;
    const uint16_t *row = W + n * K;
    float amax = 0.f;
    for (int k = threadIdx.x; k < K; k += blockDim.x) amax = fmaxf(amax, fabsf(h2f(row[k])));
    amax = block_reduce(amax, MaxOp(), shf, 0.f);
    uint16_t sbits = f2h_rn(__fdiv_rn(amax, 119.0f));
    if ((sbits & 0x7fffu) == 0) sbits = 0x3c00u;  // 1.0
    const float sf = h2f(sbits);
    if (threadIdx.x == 0) s_w[n] = sbits;
    const int G = K / g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int per_lane = g / 32;  // g is a multiple of 32, at most 512
    for (int gi = warp; gi < G; gi += nw) {
        int q8[16];
        int lo = 0, hi = 0;
        for (int i = 0; i < per_lane; ++i) {
            const int k = gi * g + i * 32 + lane;
            q8[i] = clampi(__float2int_rn(__fdiv_rn(h2f(row[k]), sf)), -119, 119);
            lo = min(lo, q8[i]);
            hi = max(hi, q8[i]);
        }
        for (int o = 16; o > 0; o >>= 1) {
            lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
            hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        }
        int s = (hi - lo + 14) / 15;
        if (s < 1) s = 1;
        const int z = clampi(rne_div(-lo, s), 0, 15);
        for (int i = 0; i < per_lane; ++i) {
            const int k = gi * g + i * 32 + lane;
            q4[n * K + k] = static_cast<uint8_t>(clampi(rne_div(q8[i], s) + z, 0, 15));
        }
        if (lane == 0) {
            s_g[n * G + gi] = static_cast<uint8_t>(s);
            zp[n * G + gi] = static_cast<uint8_t>(z);
        }
    }
}

// Per-channel asymmetric UINT4 of one weight row per CTA.
__global__ void quantize_channel_kernel(const uint16_t *__restrict__ W, int K,
                                        uint8_t *__restrict__ q4, uint8_t *__restrict__ zp,
                                        uint16_t *__restrict__ s_w) {
    __shared__ float shf[32];
    const size_t n = blockIdx.x;
    const uint16_t *row = W + n * K;
    float lo = 0.f, hi = 0.f;
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
        const float v = h2f(row[k]);
        lo = fminf(lo, v);
        hi = fmaxf(hi, v);
    }
    lo = block_reduce(lo, MinOp(), shf, 0.f);
    hi = block_reduce(hi, MaxOp(), shf, 0.f);
    uint16_t sbits = f2h_rn(__fdiv_rn(__fsub_rn(hi, lo), 15.0f));
    if ((sbits & 0x7fffu) == 0) sbits = 0x3c00u;
    const float sf = h2f(sbits);
    const int z = clampi(__float2int_rn(__fdiv_rn(-lo, sf)), 0, 15);
    if (threadIdx.x == 0) {
        s_w[n] = sbits;
        zp[n] = static_cast<uint8_t>(z);
    }
    for (int k = threadIdx.x; k < K; k += blockDim.x)
        q4[n * K + k] = static_cast<uint8_t>(clampi(__float2int_rn(__fdiv_rn(h2f(row[k]), sf)) + z, 0, 15));
}

}  // namespace

namespace {
// Launch of the row-streaming quantizer: 256 threads and kRing = 4 row
// buffers for rows of up to 16 KB, else 512 threads and 2 buffers (enough
// warps per SM for the arithmetic); as many CTAs as fit on the GPU (at most
// M).  Returns false (nothing launched) when not even one CTA fits in shared
// memory.
template <int kAct, int kSrc, int kRing, int kT>
bool launch_rows_ring(const RowSrc &src, int M, int K, int8_t *Qx, uint16_t *s_x, int32_t *t_x, uint8_t *act,
                      bool pdl, cudaStream_t stream, cudaError_t *err) {
    auto kern = quant_rows_kernel<kAct, kSrc, kRing, kT>;
    const size_t nv = static_cast<size_t>(K) / 8;
    const size_t items = kSrc == kSrcSiluMul ? 2 * nv : nv;
    const size_t smem = 16 * ((kSrc == kSrcRmsNorm ? nv : 0) + kRing * items);
    constexpr size_t kMaxDyn = 232448 - 1024;  // the per-block opt-in limit less room for the static arrays
    if (smem > kMaxDyn) return false;
    static std::mutex mu;
    static bool configured[kMaxDevices] = {};
    static int sms[kMaxDevices] = {};
    int dev = 0;
    if ((*err = cudaGetDevice(&dev)) != cudaSuccess) return true;
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return true;
    }
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!configured[dev]) {
            if ((*err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kMaxDyn))) != cudaSuccess ||
                (*err = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
                return true;
            configured[dev] = true;
        }
    }
    int per_sm = 0;
    if ((*err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kT, smem)) != cudaSuccess) return true;
    if (per_sm < 1) return false;
    const long long ctas = static_cast<long long>(sms[dev]) * per_sm;
    const dim3 grid(static_cast<unsigned>(ctas < M ? ctas : M)), block(kT);
    *err = launch_kernel(kern, grid, block, smem, stream, pdl, src, M, K, Qx, s_x, t_x, act);
    return true;
}

template <int kAct, int kSrc>
bool launch_rows(const RowSrc &src, int M, int K, int8_t *Qx, uint16_t *s_x, int32_t *t_x, uint8_t *act,
                 bool pdl, cudaStream_t stream, cudaError_t *err) {
    const size_t row_bytes = static_cast<size_t>(K) * (kSrc == kSrcSiluMul ? 4 : 2);
    if (row_bytes <= 16384)
        return launch_rows_ring<kAct, kSrc, 4, 256>(src, M, K, Qx, s_x, t_x, act, pdl, stream, err);
    return launch_rows_ring<kAct, kSrc, 2, 512>(src, M, K, Qx, s_x, t_x, act, pdl, stream, err);
}

// Rows at which the row-streaming kernel takes over (about two rows per SM).
constexpr int kRowsKernelMinM = 296;

template <int kSrc>
cudaError_t launch_quant_src(const RowSrc &src, int M, int K, int8_t *Qx, uint16_t *s_x, int32_t *t_x,
                             int act_kind, uint8_t *act, bool pdl, cudaStream_t stream) {
    if (!act) act_kind = 0;
    if (M >= kRowsKernelMinM) {
        cudaError_t e = cudaSuccess;
        bool done;
        if (act_kind == 1) done = launch_rows<1, kSrc>(src, M, K, Qx, s_x, t_x, act, pdl, stream, &e);
        else if (act_kind == 2) done = launch_rows<2, kSrc>(src, M, K, Qx, s_x, t_x, act, pdl, stream, &e);
        else done = launch_rows<0, kSrc>(src, M, K, Qx, s_x, t_x, nullptr, pdl, stream, &e);
        if (done) return e;
    }
    // One CTA per row; about two 16-byte items per thread keeps the per-row
    // latency short (few rows) without idle warps; many rows: 256 threads.
    const int nv = K / 8;
    int threads = (nv / 2 + 31) / 32 * 32;
    const int max_threads = kSrc == kSrcX ? 1024 : 512;  // the kernels' launch bounds
    threads = threads < 128 ? 128 : (threads > max_threads ? max_threads : threads);
    if (M >= 296) threads = 256;
    const dim3 grid(M), block(threads);
    if (act_kind == 1)
        return launch_kernel(quant_act_kernel<1, kSrc>, grid, block, 0, stream, pdl, src, M, K, Qx, s_x, t_x, act);
    if (act_kind == 2)
        return launch_kernel(quant_act_kernel<2, kSrc>, grid, block, 0, stream, pdl, src, M, K, Qx, s_x, t_x, act);
    return launch_kernel(quant_act_kernel<0, kSrc>, grid, block, 0, stream, pdl, src, M, K, Qx, s_x, t_x,
                         static_cast<uint8_t *>(nullptr));
}
}  // namespace

cudaError_t launch_quant_act(const uint16_t *X, int M, int K, int8_t *Qx, uint16_t *s_x,
                             int32_t *t_x, int act_kind, void *act_operand, bool pdl, cudaStream_t stream) {
    const RowSrc src{X, nullptr, 0.f, nullptr};
    return launch_quant_src<kSrcX>(src, M, K, Qx, s_x, t_x, act_kind, static_cast<uint8_t *>(act_operand), pdl,
                                   stream);
}

cudaError_t launch_rmsnorm_quant(const uint16_t *X, const uint16_t *gamma, float eps, uint16_t *Y, int M, int K,
                                 int8_t *Qx, uint16_t *s_x, int32_t *t_x, int act_kind, void *act_operand,
                                 bool pdl, cudaStream_t stream) {
    const RowSrc src{X, gamma, eps, Y};
    return launch_quant_src<kSrcRmsNorm>(src, M, K, Qx, s_x, t_x, act_kind, static_cast<uint8_t *>(act_operand),
                                         pdl, stream);
}

cudaError_t launch_silu_mul_quant(const uint16_t *H, uint16_t *Y, int M, int F, int8_t *Qx, uint16_t *s_x,
                                  int32_t *t_x, int act_kind, void *act_operand, bool pdl, cudaStream_t stream) {
    const RowSrc src{H, nullptr, 0.f, Y};
    return launch_quant_src<kSrcSiluMul>(src, M, F, Qx, s_x, t_x, act_kind, static_cast<uint8_t *>(act_operand),
                                         pdl, stream);
}

cudaError_t launch_act_operand(const int8_t *Qx, int M, int K, int act_kind, void *act_operand,
                               cudaStream_t stream) {
    uint8_t *act = static_cast<uint8_t *>(act_operand);
    if (act_kind == 1) {
        const size_t n8 = static_cast<size_t>(M) * K / 8;
        const size_t blocks = (n8 + 255) / 256;
        act_operand_f16_kernel<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(Qx, n8, act);
    } else {
        act_operand_kernel<<<M, 256, 0, stream>>>(Qx, M, K, act);
    }
    return cudaGetLastError();
}

cudaError_t launch_quantize_weights(const uint16_t *W, int N, int K, int group, uint8_t *q4,
                                    uint8_t *s_g, uint8_t *z, uint16_t *s_w, cudaStream_t stream) {
    if (group > 0)
        quantize_group_kernel<<<N, 256, 0, stream>>>(W, K, group, q4, s_g, z, s_w);
    else
        quantize_channel_kernel<<<N, 256, 0, stream>>>(W, K, q4, z, s_w);
    return cudaGetLastError();
}

}  // namespace qoq

/*
 * QoQ W4A8 oracle -- TEST INFRASTRUCTURE, NOT PRODUCT CODE.
 *
 * A plain, single-threaded, deliberately slow CPU restatement of what the
 * W4A8 path computes: the progressive group quantizer of the weights, the
 * per-channel W4 quantizer, the per-token INT8 activation quantizer, the
 * integer GEMM and the fp64 epilogue.  Only the test-suite, the smoke check
 * and the CPU-baseline leg of the benchmark may load or call it.  It shares no
 * code, header, table or helper with the CUDA library; the two are checked
 * against each other, never built from each other.
 *
 * Sources (web pages on QServe / QoQ):
 *   [QS-review]  "QServe：把 W4A8KV4 的理论收益做成实测吞吐的量化—系统协同设计"
 *                (zenmind.me architect's review), sections 3.1 and 3.2.
 *   [QS-summary] "QServe: W4A8KV4 Quantization and System Co-design for
 *                Efficient LLM Serving" (papercache.org summary), sections
 *                "整数量化" (eq. 1), "渐进式组量化" (eq. 4/5),
 *                "保护性量化范围", "逐通道W4A8 GEMM中的快速反量化" (eq. 13),
 *                "逐组W4A8 GEMM中的快速反量化".
 *   [Book-4.1]   "01 inference papers and experiments" book chapter,
 *                section 4.1 "均匀量化的数学基础" (symmetric INT8 range).
 *
 * Floating point: the fp16 <-> fp32 conversions are written here from the
 * IEEE 754 binary16 definition.  Where a float decides an integer code (a
 * scale division followed by rounding), the decision is taken in IEEE fp32
 * with round-to-nearest-even, the precision the CUDA path uses; the final
 * epilogue is fp64.  Build without -ffast-math and with -ffp-contract=off.
 *
 * Parity pins: every function here is pinned by tests that do not re-type its
 * formula (worked example printed on the pages, exhaustive sweeps, closed
 * forms, brute force, library routines).  None is "parity unpinned".
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------- */
/* IEEE 754 binary16 <-> binary32, from the format definition.               */
/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.        */
/* ------------------------------------------------------------------------- */

ORACLE_API float oracle_half_to_float(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0x1f) {
        if (f == 0) v = INFINITY;
        else v = NAN;
    } else if (e == 0) {
        v = ldexp((double)f, -24); /* subnormal: f * 2^-24 */
    } else {
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    }
    return (float)(sign ? -v : v); /* every binary16 value is exact in binary32 */
}

/* Round a binary32 value to the nearest binary16 value, ties to even. */
ORACLE_API uint16_t oracle_float_to_half_rn(float x) {
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return (uint16_t)(sign | 0x7e00);
    double a = fabs((double)x);
    if (isinf(x)) return (uint16_t)(sign | 0x7c00);
    if (a == 0.0) return sign;
    /* Find the binade: the spacing of binary16 values around a.
     * Normal range [2^-14, 65504]: spacing 2^(e-10) in binade [2^e, 2^(e+1)).
     * Subnormal range (0, 2^-14): spacing 2^-24. */
    int e;
    frexp(a, &e); /* a = m * 2^e with m in [0.5, 1) => a in [2^(e-1), 2^e) */
    int binade = e - 1;
    if (binade < -14) binade = -14;
    double ulp = ldexp(1.0, binade - 10);
    double n = a / ulp;            /* exact: division by a power of two */
    double fl = floor(n);
    double rem = n - fl;           /* exact */
    double r;
    if (rem > 0.5) r = fl + 1.0;
    else if (rem < 0.5) r = fl;
    else r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    double v = r * ulp;            /* rounded magnitude */
    if (v >= 65520.0) return (uint16_t)(sign | 0x7c00); /* overflow to inf */
    if (v >= 65504.0) v = 65504.0;
    /* Encode v, which is now exactly a binary16 value. */
    if (v < ldexp(1.0, -14)) {
        return (uint16_t)(sign | (uint16_t)(v / ldexp(1.0, -24)));
    }
    int ee;
    double m = frexp(v, &ee); /* v = m * 2^ee, m in [0.5,1) */
    int exp_field = ee - 1 + 15;
    int frac = (int)((m * 2.0 - 1.0) * 1024.0); /* exact */
    return (uint16_t)(sign | (exp_field << 10) | frac);
}

/* ------------------------------------------------------------------------- */
/* Rounding to integers, ties to even ("⌈·⌋" of eq. 1, read as              */
/* round-half-even everywhere).                                              */
/* ------------------------------------------------------------------------- */

/* Round-half-even of a binary32 value to an integer. */
ORACLE_API int64_t oracle_rne_f32(float x) {
    double d = (double)x;
    double fl = floor(d);
    double rem = d - fl; /* exact */
    double r;
    if (rem > 0.5) r = fl + 1.0;
    else if (rem < 0.5) r = fl;
    else r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    return (int64_t)r;
}

/* Round-half-even of the rational a / b, b > 0, in exact integer arithmetic. */
ORACLE_API int64_t oracle_rne_div(int64_t a, int64_t b) {
    int64_t q = a / b, r = a % b;
    if (r < 0) { q -= 1; r += b; } /* floor division: 0 <= r < b */
    if (2 * r > b) q += 1;
    else if (2 * r == b && (q & 1)) q += 1;
    return q;
}

static int64_t clamp64(int64_t v, int64_t lo, int64_t hi) {
    return v < lo ? lo : (v > hi ? hi : v);
}

/* ------------------------------------------------------------------------- */
/* Progressive group quantization, step 2 on one group ([QS-summary]         */
/* "渐进式组量化" eq. 5 as described in words, with eq. 1 for the            */
/* asymmetric quantizer and "保护性量化范围" for the reconstruction          */
/* ⌊q/s⌉·s).  Input: the INT8 intermediate codes of one group.  Output: the  */
/* UINT8 group scale s_g, the UINT4 zero z and the UINT4 codes q4.           */
/*   lo = min(0, min q8), hi = max(0, max q8)      (0 kept in range)         */
/*   s_g = max(1, ceil((hi - lo) / 15))            (UINT8, qmax - qmin = 15) */
/*   z   = clamp(rne(-lo / s_g), 0, 15)            (eq. 1 with qmin = 0)     */
/*   q4  = clamp(rne(q8 / s_g) + z, 0, 15)                                   */
/* Returns the number of codes whose reconstruction (q4 - z) * s_g leaves    */
/* the INT8 range [-128, 127].                                               */
/* ------------------------------------------------------------------------- */
ORACLE_API int oracle_group_step(const int32_t *q8, int len, uint8_t *q4,
                                 uint8_t *s_g, uint8_t *z) {
    int32_t lo = 0, hi = 0;
    for (int i = 0; i < len; i++) {
        if (q8[i] < lo) lo = q8[i];
        if (q8[i] > hi) hi = q8[i];
    }
    int64_t range = (int64_t)hi - lo;
    int64_t s = (range + 14) / 15; /* ceil(range / 15) */
    if (s < 1) s = 1;
    int64_t zz = clamp64(oracle_rne_div(-(int64_t)lo, s), 0, 15);
    int bad = 0;
    for (int i = 0; i < len; i++) {
        int64_t q = clamp64(oracle_rne_div(q8[i], s) + zz, 0, 15);
        q4[i] = (uint8_t)q;
        int64_t w8 = (q - zz) * s;
        if (w8 < -128 || w8 > 127) bad++;
    }
    *s_g = (uint8_t)s;
    *z = (uint8_t)zz;
    return bad;
}

/* ------------------------------------------------------------------------- */
/* Progressive group quantization of a weight matrix W [N][K] (fp16 bits,    */
/* row n = output channel).                                                  */
/* Step 1 ([QS-summary] eq. 4; [QS-review] 3.1): per-output-channel          */
/* symmetric INT8 with an fp16 channel scale, clipped to the protective      */
/* range [-119, 119]:                                                        */
/*   a = max_k |W[n,k]|,  s_w = fp16_rn(a / 119)  (1.0 if that is 0)         */
/*   q8 = clamp(rne(W / s_w), -119, 119)                                     */
/* Step 2: oracle_group_step on each group of g consecutive k.               */
/* Outputs: q4 [N][K] (one code per byte), s_g [N][K/g], z [N][K/g],         */
/* s_w [N] (fp16 bits), optionally q8 [N][K].  Returns the number of         */
/* reconstructions outside [-128, 127] (0 under the protective range).       */
/* ------------------------------------------------------------------------- */
ORACLE_API int64_t oracle_quantize_weights_group(
    const uint16_t *W, int N, int K, int g, uint8_t *q4, uint8_t *s_g,
    uint8_t *z, uint16_t *s_w, int8_t *q8_out) {
    int G = K / g;
    int64_t bad = 0;
    int32_t *q8 = (int32_t *)malloc(sizeof(int32_t) * (size_t)g);
    if (!q8) return -1;
    for (int n = 0; n < N; n++) {
        const uint16_t *row = W + (size_t)n * K;
        float a = 0.0f;
        for (int k = 0; k < K; k++) {
            float v = fabsf(oracle_half_to_float(row[k]));
            if (v > a) a = v;
        }
        uint16_t sh = oracle_float_to_half_rn(a / 119.0f);
        if ((sh & 0x7fff) == 0) sh = 0x3c00; /* 1.0 */
        s_w[n] = sh;
        float sf = oracle_half_to_float(sh);
        for (int gi = 0; gi < G; gi++) {
            for (int i = 0; i < g; i++) {
                float wv = oracle_half_to_float(row[gi * g + i]);
                q8[i] = (int32_t)clamp64(oracle_rne_f32(wv / sf), -119, 119);
                if (q8_out) q8_out[(size_t)n * K + gi * g + i] = (int8_t)q8[i];
            }
            bad += oracle_group_step(q8, g, q4 + (size_t)n * K + gi * g,
                                     s_g + (size_t)n * G + gi,
                                     z + (size_t)n * G + gi);
        }
    }
    free(q8);
    return bad;
}

/* ------------------------------------------------------------------------- */
/* Per-channel W4 (no group step), for the per-channel GEMM ([QS-summary]    */
/* "逐通道W4A8 GEMM中的快速反量化"; [QS-review] 3.2 per-channel case).       */
/* The pages say only "per-channel" with a UINT4 zero and fp16 scale; the    */
/* plainest reading is eq. 1 applied per output row to the fp16 weights:     */
/*   lo = min(0, min W[n,:]), hi = max(0, max W[n,:])   (in fp32)            */
/*   s_W = fp16_rn((hi - lo) / 15)   (1.0 if that is 0)                      */
/*   z   = clamp(rne(-lo / s_W), 0, 15)                                      */
/*   q4  = clamp(rne(W / s_W) + z, 0, 15)                                    */
/* ------------------------------------------------------------------------- */
ORACLE_API void oracle_quantize_weights_channel(const uint16_t *W, int N, int K,
                                                uint8_t *q4, uint8_t *z,
                                                uint16_t *s_W) {
    for (int n = 0; n < N; n++) {
        const uint16_t *row = W + (size_t)n * K;
        float lo = 0.0f, hi = 0.0f;
        for (int k = 0; k < K; k++) {
            float v = oracle_half_to_float(row[k]);
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
        float range = hi - lo;
        uint16_t sh = oracle_float_to_half_rn(range / 15.0f);
        if ((sh & 0x7fff) == 0) sh = 0x3c00;
        s_W[n] = sh;
        float sf = oracle_half_to_float(sh);
        int64_t zz = clamp64(oracle_rne_f32(-lo / sf), 0, 15);
        z[n] = (uint8_t)zz;
        for (int k = 0; k < K; k++) {
            float v = oracle_half_to_float(row[k]);
            q4[(size_t)n * K + k] = (uint8_t)clamp64(oracle_rne_f32(v / sf) + zz, 0, 15);
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Per-token symmetric INT8 activations ([QS-review] 3.2 runtime precision   */
/* map: every GEMM takes INT8 activations with per-token scales;             */
/* [Book-4.1]: symmetric INT8 range [-127, 127]).  Row m of X [M][K]:        */
/*   s_x = fp16_rn(max_k |X[m,k]| / 127)                                     */
/*   s_x == 0  ->  Qx[m,:] = 0                                               */
/*   else Qx = clamp(rne(X / s_x), -127, 127)   (IEEE fp32 division)         */
/*   t_x = sum_k Qx[m,k]  (the row sum "t_X = X·1_k" of [QS-summary] eq. 13, */
/*                         taken on the integer codes)                       */
/* ------------------------------------------------------------------------- */
ORACLE_API void oracle_quant_act(const uint16_t *X, int M, int K, int8_t *Qx,
                                 uint16_t *s_x, int32_t *t_x) {
    for (int m = 0; m < M; m++) {
        const uint16_t *row = X + (size_t)m * K;
        float a = 0.0f;
        for (int k = 0; k < K; k++) {
            float v = fabsf(oracle_half_to_float(row[k]));
            if (v > a) a = v;
        }
        uint16_t sh = oracle_float_to_half_rn(a / 127.0f);
        s_x[m] = sh;
        float sf = oracle_half_to_float(sh);
        int32_t t = 0;
        for (int k = 0; k < K; k++) {
            int64_t q = 0;
            if (sf != 0.0f)
                q = clamp64(oracle_rne_f32(oracle_half_to_float(row[k]) / sf), -127, 127);
            Qx[(size_t)m * K + k] = (int8_t)q;
            t += (int32_t)q;
        }
        if (t_x) t_x[m] = t;
    }
}

/* ------------------------------------------------------------------------- */
/* Integer GEMM, per-group weights ([QS-review] 3.2 / 4 step 3: the INT4     */
/* weight is dequantized to the INT8 intermediate, then an INT8 x INT8       */
/* product accumulates in INT32):                                            */
/*   acc[m,n] = sum_k Qx[m,k] * (q4[n,k] - z[n,k/g]) * s_g[n,k/g]            */
/* ------------------------------------------------------------------------- */
ORACLE_API void oracle_gemm_i32_group(const int8_t *Qx, const uint8_t *q4,
                                      const uint8_t *s_g, const uint8_t *z,
                                      int M, int N, int K, int g, int32_t *acc) {
    int G = K / g;
    for (int m = 0; m < M; m++) {
        for (int n = 0; n < N; n++) {
            int32_t s = 0;
            for (int k = 0; k < K; k++) {
                int32_t w8 = ((int32_t)q4[(size_t)n * K + k] - z[(size_t)n * G + k / g]) *
                             (int32_t)s_g[(size_t)n * G + k / g];
                s += (int32_t)Qx[(size_t)m * K + k] * w8;
            }
            acc[(size_t)m * N + n] = s;
        }
    }
}

/* The same sum, at a list of (m, n) output positions only. */
ORACLE_API void oracle_gemm_i32_group_at(const int8_t *Qx, const uint8_t *q4,
                                         const uint8_t *s_g, const uint8_t *z,
                                         int M, int N, int K, int g,
                                         const int32_t *ms, const int32_t *ns,
                                         int count, int32_t *out) {
    int G = K / g;
    (void)M; (void)N;
    for (int i = 0; i < count; i++) {
        int m = ms[i], n = ns[i];
        int32_t s = 0;
        for (int k = 0; k < K; k++) {
            int32_t w8 = ((int32_t)q4[(size_t)n * K + k] - z[(size_t)n * G + k / g]) *
                         (int32_t)s_g[(size_t)n * G + k / g];
            s += (int32_t)Qx[(size_t)m * K + k] * w8;
        }
        out[i] = s;
    }
}

/* ------------------------------------------------------------------------- */
/* Integer GEMM, per-channel weights, with the zero folded out of the sum    */
/* ([QS-summary] eq. 13, [QS-review] 3.2 per-channel case):                  */
/*   acc[m,n] = sum_k Qx[m,k] * q4[n,k]  -  z[n] * t_x[m]                    */
/* which equals sum_k Qx[m,k] * (q4[n,k] - z[n]) exactly.                    */
/* ------------------------------------------------------------------------- */
ORACLE_API void oracle_gemm_i32_channel(const int8_t *Qx, const int32_t *t_x,
                                        const uint8_t *q4, const uint8_t *z,
                                        int M, int N, int K, int32_t *acc) {
    for (int m = 0; m < M; m++) {
        for (int n = 0; n < N; n++) {
            int32_t s = 0;
            for (int k = 0; k < K; k++)
                s += (int32_t)Qx[(size_t)m * K + k] * (int32_t)q4[(size_t)n * K + k];
            acc[(size_t)m * N + n] = s - (int32_t)z[n] * t_x[m];
        }
    }
}

ORACLE_API void oracle_gemm_i32_channel_at(const int8_t *Qx, const int32_t *t_x,
                                           const uint8_t *q4, const uint8_t *z,
                                           int M, int N, int K,
                                           const int32_t *ms, const int32_t *ns,
                                           int count, int32_t *out) {
    (void)M; (void)N;
    for (int i = 0; i < count; i++) {
        int m = ms[i], n = ns[i];
        int32_t s = 0;
        for (int k = 0; k < K; k++)
            s += (int32_t)Qx[(size_t)m * K + k] * (int32_t)q4[(size_t)n * K + k];
        out[i] = s - (int32_t)z[n] * t_x[m];
    }
}

/* ------------------------------------------------------------------------- */
/* fp64 epilogue: O[m,n] = s_x[m] * s_w[n] * acc[m,n] ([QS-review] 3.2: the  */
/* GEMM output is fp16, scaled per token and per output channel).            */
/* ------------------------------------------------------------------------- */
ORACLE_API void oracle_epilogue_f64(const int32_t *acc, const uint16_t *s_x,
                                    const uint16_t *s_w, int M, int N, double *O) {
    for (int m = 0; m < M; m++) {
        double sx = (double)oracle_half_to_float(s_x[m]);
        for (int n = 0; n < N; n++) {
            double sw = (double)oracle_half_to_float(s_w[n]);
            O[(size_t)m * N + n] = sx * sw * (double)acc[(size_t)m * N + n];
        }
    }
}

/* ------------------------------------------------------------------------- */
/* The FP16 kernels in front of the GEMMs, into which the QServe runtime     */
/* fuses the per-token INT8 activation quantization ([QS-summary]           */
/* "QServe系统运行时"; [QS-review] §4 ②: the norm before the QKV projection  */
/* and the FFN's first layer, the activation kernel before the FFN's second  */
/* layer).  Both are written here in fp64 from their definitions.           */
/*                                                                           */
/* RMS normalization.  The pages call the norm LayerNorm; the Llama-family  */
/* blocks of the workloads use its RMS form (no mean subtraction, no bias):  */
/*   Y[m,k] = gamma[k] * X[m,k] / sqrt(mean_k X[m,k]^2 + eps)                */
/* X [M][K] and gamma [K] are fp16 bits; Y [M][K] fp64.                      */
/* ------------------------------------------------------------------------- */
ORACLE_API void oracle_rmsnorm_f64(const uint16_t *X, const uint16_t *gamma, double eps,
                                   int M, int K, double *Y) {
    for (int m = 0; m < M; m++) {
        const uint16_t *row = X + (size_t)m * K;
        double ss = 0.0;
        for (int k = 0; k < K; k++) {
            double v = (double)oracle_half_to_float(row[k]);
            ss += v * v;
        }
        double denom = sqrt(ss / (double)K + eps);
        for (int k = 0; k < K; k++) {
            double v = (double)oracle_half_to_float(row[k]);
            double gk = (double)oracle_half_to_float(gamma[k]);
            Y[(size_t)m * K + k] = denom > 0.0 ? gk * v / denom : 0.0;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* SwiGLU activation of the FFN ("01 inference papers and experiments" book  */
/* chapter, FFN/MLP module ⑤: down = SiLU(gate) ⊙ up · W_down):              */
/*   A[m,f] = SiLU(G[m,f]) * U[m,f],  SiLU(g) = g / (1 + exp(-g))            */
/* H [M][2F] is the gate_up projection's fp16 output with the gate in       */
/* columns 0..F-1 and the up projection in columns F..2F-1; A [M][F] fp64.  */
/* ------------------------------------------------------------------------- */
ORACLE_API void oracle_silu_mul_f64(const uint16_t *H, int M, int F, double *A) {
    for (int m = 0; m < M; m++) {
        const uint16_t *row = H + (size_t)m * 2 * F;
        for (int f = 0; f < F; f++) {
            double g = (double)oracle_half_to_float(row[f]);
            double u = (double)oracle_half_to_float(row[F + f]);
            A[(size_t)m * F + f] = g / (1.0 + exp(-g)) * u;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* KV4: per-head dynamic INT4 quantization of the KV cache ([QS-summary]    */
/* "QServe系统运行时", KV cache management: paged cache, and right after the */
/* quantized KV features of each page the per-head FP16 scale and zero,     */
/* updated online; [QS-review] §3.2 "KV 缓存管理").  Each key or value      */
/* vector of one token and one head (d values) gets eq. 1 of "整数量化"     */
/* with an FP16 scale and an FP16 zero point:                                */
/*   lo = min x, hi = max x                                                  */
/*   s = fp16_rn((hi - lo) / 15)   (1.0 when that is 0)                      */
/*   z = fp16_rn(rne(-lo / s))     (an integer, kept as FP16)                */
/*   q = clamp(rne(x / s) + z, 0, 15)                                        */
/* so that x is reconstructed as (q - z) * s.  Divisions are IEEE fp32,      */
/* rne = round half to even.  x [n][d] fp16 bits; q [n][d] one code per      */
/* byte; s, z [n] fp16 bits.                                                 */
/* ------------------------------------------------------------------------- */
ORACLE_API void oracle_kv4_quantize(const uint16_t *x, int n, int d, uint8_t *q,
                                    uint16_t *s, uint16_t *z) {
    for (int i = 0; i < n; i++) {
        const uint16_t *v = x + (size_t)i * d;
        float lo = oracle_half_to_float(v[0]), hi = lo;
        for (int k = 1; k < d; k++) {
            float f = oracle_half_to_float(v[k]);
            if (f < lo) lo = f;
            if (f > hi) hi = f;
        }
        uint16_t sh = oracle_float_to_half_rn((hi - lo) / 15.0f);
        if ((sh & 0x7fff) == 0) sh = 0x3c00;
        float sf = oracle_half_to_float(sh);
        int64_t zi = oracle_rne_f32(-lo / sf);
        uint16_t zh = oracle_float_to_half_rn((float)zi);
        float zf = oracle_half_to_float(zh); /* an integer: rne result, kept as fp16 */
        s[i] = sh;
        z[i] = zh;
        for (int k = 0; k < d; k++) {
            int64_t c = oracle_rne_f32(oracle_half_to_float(v[k]) / sf) + (int64_t)zf;
            q[(size_t)i * d + k] = (uint8_t)clamp64(c, 0, 15);
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Decode attention over a KV4 cache, in fp64 ([QS-summary] "QServe中的KV4  */
/* 注意力"; [QS-review] §4 step ④: the attention of the decode step reads   */
/* the INT4 K/V, dequantizes, and computes softmax(q K^T) V).  One query    */
/* token of one sequence; the G query heads of one KV head (grouped-query   */
/* attention share the KV head); L cached tokens:                           */
/*   Khat[t,k] = (Kq[t,k] - Kz[t]) * Ks[t],  Vhat likewise                  */
/*   S[h,t] = scale * sum_k Q[h,k] * Khat[t,k]                              */
/*   P[h,t] = exp(S[h,t] - max_t S[h,t]) / sum_t exp(...)                   */
/*   O[h,k] = sum_t P[h,t] * Vhat[t,k]                                      */
/* Q [G][d] fp16 bits; Kq, Vq [L][d] codes; Ks, Kz, Vs, Vz [L] fp16 bits;    */
/* O [G][d] fp64.  L >= 1.                                                   */
/* ------------------------------------------------------------------------- */
ORACLE_API void oracle_kv4_attention_f64(const uint16_t *Q, int G, int d, int L,
                                         const uint8_t *Kq, const uint16_t *Ks, const uint16_t *Kz,
                                         const uint8_t *Vq, const uint16_t *Vs, const uint16_t *Vz,
                                         double scale, double *O) {
    double *S = (double *)malloc(sizeof(double) * (size_t)L);
    if (!S) return;
    for (int h = 0; h < G; h++) {
        double mx = -INFINITY;
        for (int t = 0; t < L; t++) {
            double ks = (double)oracle_half_to_float(Ks[t]);
            double kz = (double)oracle_half_to_float(Kz[t]);
            double acc = 0.0;
            for (int k = 0; k < d; k++) {
                double kh = ((double)Kq[(size_t)t * d + k] - kz) * ks;
                acc += (double)oracle_half_to_float(Q[(size_t)h * d + k]) * kh;
            }
            S[t] = scale * acc;
            if (S[t] > mx) mx = S[t];
        }
        double den = 0.0;
        for (int t = 0; t < L; t++) {
            S[t] = exp(S[t] - mx);
            den += S[t];
        }
        for (int k = 0; k < d; k++) O[(size_t)h * d + k] = 0.0;
        for (int t = 0; t < L; t++) {
            double p = S[t] / den;
            double vs = (double)oracle_half_to_float(Vs[t]);
            double vz = (double)oracle_half_to_float(Vz[t]);
            for (int k = 0; k < d; k++)
                O[(size_t)h * d + k] += p * ((double)Vq[(size_t)t * d + k] - vz) * vs;
        }
    }
    free(S);
}

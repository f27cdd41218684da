/*
 * r9q oracle — plain, slow, single-threaded CPU reference for the block-scaled
 * fp8 (e4m3) GEMM path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * bench's CPU-baseline leg may load this library.  The CUDA library shares no
 * code, header, table or constant with this file, and the product path never
 * calls it.
 *
 * What is computed, and where it is stated:
 *  - fp8 e4m3 ("e4m3fn" of the OCP 8-bit floating point specification, v1.0,
 *    section 5.3): bias 7, no infinities, S.1111.111 is NaN, largest finite
 *    448, smallest normal 2^-6, subnormals in steps of 2^-9.
 *  - per-token-group-128 activation quantisation: r9700-stack v0.3.1 release
 *    notes, "What changed for someone running it" (fused activation quant in
 *    the dense fp8 block GEMM).  The statement of the operation fixes
 *    scale = amax/448 in fp32, round-to-nearest-even, saturation to +-448.
 *  - fp8 weights with one fp32 scale per 128x128 block, fp32 accumulation,
 *    bf16 output: the same statement; fp8 weight-only GEMMs with bf16
 *    activations: v0.3.1 notes (fp8 hyper-connection decode GEMMs, bf16 MMA
 *    against the unquantised activations); exact block-scaled variant:
 *    v0.3.0 notes, "What changed".
 *  - silu(gate)*up epilogue on the gate_up output and the fp8 row quant that
 *    feeds the down GEMM: releases page, v0.3.3 "What changed" (fused MoE
 *    decode path).
 *
 * Arithmetic conventions (the plainest reading where the pages are silent):
 *  - x/s is one IEEE fp32 division, then one RNE rounding to e4m3 (no
 *    reciprocal multiply).  An all-zero group has s = 0 and all codes 0x00.
 *  - GEMM: per 128-wide k-block an fp32 partial summed in increasing k, then
 *    acc = acc + partial * (as * ws), blocks in increasing order, all fp32 with
 *    no fused multiply-add (built with -ffp-contract=off), then RNE to bf16.
 *  - SwiGLU: g, u are the bf16-rounded gate_up outputs; h = bf16(silu(g) * u)
 *    evaluated in fp32 as a separate SwiGLU pass after a bf16 GEMM would:
 *    e = exp(-g), d = 1 + e, silu = g / d, h = silu * u, each step one IEEE
 *    fp32 rounding, then RNE to bf16.  exp is written out below (Cody and
 *    Waite's reduction, Taylor polynomial) so that its every rounding is
 *    fixed; the fused path must give the separate pass's bits.
 *
 * Parity pins: tests/test_oracle_pins.py (worked examples, brute force,
 * closed forms, library special cases).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define R9O_BLOCK 128

#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads of the GEMM loops.  The plain build is single-threaded; a build
 * with -fopenmp (the CPU-baseline timing only) splits the independent output
 * elements over threads.  Each element is computed by the same sequence of
 * operations either way, so the results are identical. */
void r9o_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int r9o_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------- bf16 ---- */

static float bf16_bits_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

float r9o_bf16_to_f32(uint16_t h) { return bf16_bits_to_f32(h); }

/* Round a double to the nearest bf16 (8-bit significand), ties to even.
 * Written from the definition: scale into [2^7, 2^8) (or the subnormal
 * quantum 2^-133), round the scaled value with rint (ties-to-even under the
 * default rounding mode), scale back.  Overflow goes to +-inf. */
uint16_t r9o_f64_to_bf16(double v) {
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    double r;
    if (a < 0x1p-126) {                       /* bf16 subnormal range */
        r = rint(a * 0x1p133) * 0x1p-133;
    } else {
        int e;
        (void)frexp(a, &e);                   /* a = f * 2^e, f in [0.5, 1) */
        double q = rint(ldexp(a, 8 - e));     /* integer in [128, 256] */
        r = ldexp(q, e - 8);
    }
    if (r >= 0x1p128) return sign | 0x7F80;   /* rounds past the largest finite */
    /* r is now exactly representable as bf16 and therefore as float. */
    float f = (float)r;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

uint16_t r9o_f32_to_bf16(float v) { return r9o_f64_to_bf16((double)v); }

void r9o_f32_to_bf16_array(const float* x, int64_t n, uint16_t* y) {
    for (int64_t i = 0; i < n; ++i) y[i] = r9o_f32_to_bf16(x[i]);
}

/* ---------------------------------------------------------------- e4m3 ---- */

/* Value of an e4m3 code (OCP FP8 E4M3): S.EEEE.MMM, bias 7. */
double r9o_e4m3_decode(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    double v = (e == 0) ? (double)m * 0x1p-9 : ldexp(8.0 + m, e - 10);
    return s ? -v : v;
}

/* fp32 -> e4m3, round to nearest with ties to even, saturating: anything whose
 * rounding would leave the finite range becomes +-448 (0x7E / 0xFE); the NaN
 * code is never produced for finite input.  Inputs in [448, 464] round to 448
 * (464 is the tie between 448 = 1.110b*2^8 and the non-existent 480 = 1.111b*2^8
 * and goes to the even significand), larger ones saturate to it. */
uint8_t r9o_e4m3_encode(float v) {
    if (isnan(v)) return 0x7F;               /* outside the contract */
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0) return sign | 0x7E;
    if (a < 0x1p-6) {
        /* subnormal range, quantum 2^-9; q == 8 is the smallest normal 0x08 */
        double q = rint(a * 0x1p9);
        return sign | (uint8_t)q;
    }
    int e;
    (void)frexp(a, &e);
    int E = e - 1;                           /* a in [2^E, 2^(E+1)), E in [-6, 8] */
    double q = rint(ldexp(a, 3 - E));        /* significand * 8, in [8, 16] */
    /* q == 16 carries into the next binade: ((E+7)<<3) + 8 == (E+8)<<3 */
    return sign | (uint8_t)(((E + 7) << 3) + ((int)q - 8));
}

void r9o_e4m3_encode_array(const float* x, int64_t n, uint8_t* q) {
    for (int64_t i = 0; i < n; ++i) q[i] = r9o_e4m3_encode(x[i]);
}

/* Encode the fp32 bit patterns [lo, lo + n). */
void r9o_e4m3_encode_bits(uint32_t lo, int64_t n, uint8_t* q) {
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u = lo + (uint32_t)i;
        float f;
        memcpy(&f, &u, sizeof f);
        q[i] = r9o_e4m3_encode(f);
    }
}

/* --------------------------------------------------------- quantisation ---- */

/* Per-token group quantisation of bf16 activations x[M][K] with groups of G
 * consecutive K (G = 128 on the path; G is a parameter so the "one scale per
 * row" reading can be evaluated too).  q[M][K] e4m3 codes, s[M][K/G] fp32. */
void r9o_quant_group(const uint16_t* x, int64_t M, int64_t K, int64_t G,
                     uint8_t* q, float* s) {
    int64_t ng = K / G;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t g = 0; g < ng; ++g) {
            const uint16_t* xg = x + m * K + g * G;
            uint8_t* qg = q + m * K + g * G;
            float amax = 0.0f;
            for (int64_t i = 0; i < G; ++i) {
                float a = fabsf(bf16_bits_to_f32(xg[i]));
                if (a > amax) amax = a;
            }
            float sc = amax / 448.0f;
            s[m * ng + g] = sc;
            for (int64_t i = 0; i < G; ++i) {
                if (amax == 0.0f) {
                    qg[i] = 0x00;
                } else {
                    float t = bf16_bits_to_f32(xg[i]) / sc;
                    qg[i] = r9o_e4m3_encode(t);
                }
            }
        }
    }
}

/* Weight quantisation, one fp32 scale per 128x128 block of w[N][K] (set-up,
 * not the hot path): s = amax/448 over the block, q = e4m3(w/s). */
void r9o_quant_block128(const float* w, int64_t N, int64_t K, uint8_t* q, float* s) {
    int64_t NB = N / R9O_BLOCK, KB = K / R9O_BLOCK;
    for (int64_t nb = 0; nb < NB; ++nb) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            float amax = 0.0f;
            for (int64_t r = 0; r < R9O_BLOCK; ++r)
                for (int64_t c = 0; c < R9O_BLOCK; ++c) {
                    float a = fabsf(w[(nb * R9O_BLOCK + r) * K + kb * R9O_BLOCK + c]);
                    if (a > amax) amax = a;
                }
            float sc = amax / 448.0f;
            s[nb * KB + kb] = sc;
            for (int64_t r = 0; r < R9O_BLOCK; ++r)
                for (int64_t c = 0; c < R9O_BLOCK; ++c) {
                    int64_t i = (nb * R9O_BLOCK + r) * K + kb * R9O_BLOCK + c;
                    q[i] = (amax == 0.0f) ? 0x00 : r9o_e4m3_encode(w[i] / sc);
                }
        }
    }
}

/* ------------------------------------------------------------------ GEMM ---- */

static float g_e4m3_table[256];
static int g_table_ready = 0;

static void ensure_table(void) {
    if (g_table_ready) return;
    for (int c = 0; c < 256; ++c) g_e4m3_table[c] = (float)r9o_e4m3_decode((uint8_t)c);
    g_table_ready = 1;
}

/* W8A8: y[m][n] = bf16( sum_kb (sum_{k in kb} aq[m][k]*w[n][k]) * (as[m][kb]*ws[n/128][kb]) ).
 * rows: optional list of nrows token indices to evaluate (NULL = all M, in
 * order); outputs acc/y are indexed by position in that list.  Products of two
 * e4m3 values are exact in fp32. */
void r9o_gemm_w8a8(const uint8_t* aq, const float* as, const uint8_t* w, const float* ws,
                   int64_t M, int64_t N, int64_t K, const int64_t* rows, int64_t nrows,
                   float* acc_out, uint16_t* y) {
    ensure_table();
    int64_t KB = K / R9O_BLOCK;
    int64_t cnt = rows ? nrows : M;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t i = 0; i < cnt; ++i) {
        for (int64_t n = 0; n < N; ++n) {
            int64_t m = rows ? rows[i] : i;
            float acc = 0.0f;
            for (int64_t kb = 0; kb < KB; ++kb) {
                float p = 0.0f;
                for (int64_t k = kb * R9O_BLOCK; k < (kb + 1) * R9O_BLOCK; ++k)
                    p = p + g_e4m3_table[aq[m * K + k]] * g_e4m3_table[w[n * K + k]];
                float sc = as[m * KB + kb] * ws[(n / R9O_BLOCK) * KB + kb];
                acc = acc + p * sc;
            }
            if (acc_out) acc_out[i * N + n] = acc;
            if (y) y[i * N + n] = r9o_f32_to_bf16(acc);
        }
    }
}

/* Weight-only: y[m][n] = bf16( sum_kb (sum_{k in kb} x[m][k]*w[n][k]) * ws[n/128][kb] )
 * with x the unquantised bf16 activations. */
void r9o_gemm_w8bf16(const uint16_t* x, const uint8_t* w, const float* ws,
                     int64_t M, int64_t N, int64_t K, const int64_t* rows, int64_t nrows,
                     float* acc_out, uint16_t* y) {
    ensure_table();
    int64_t KB = K / R9O_BLOCK;
    int64_t cnt = rows ? nrows : M;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t i = 0; i < cnt; ++i) {
        for (int64_t n = 0; n < N; ++n) {
            int64_t m = rows ? rows[i] : i;
            float acc = 0.0f;
            for (int64_t kb = 0; kb < KB; ++kb) {
                float p = 0.0f;
                for (int64_t k = kb * R9O_BLOCK; k < (kb + 1) * R9O_BLOCK; ++k)
                    p = p + bf16_bits_to_f32(x[m * K + k]) * g_e4m3_table[w[n * K + k]];
                acc = acc + p * ws[(n / R9O_BLOCK) * KB + kb];
            }
            if (acc_out) acc_out[i * N + n] = acc;
            if (y) y[i * N + n] = r9o_f32_to_bf16(acc);
        }
    }
}

/* ------------------------------------------------------------------ exp ---- */

/* e^x in fp32 by the method of W. J. Cody and W. Waite ("Software Manual for
 * the Elementary Functions", 1980, chapter on EXP): write x = k*ln2 + r with k
 * the integer nearest to x*log2(e), so |r| <= ln2/2; ln2 is carried as a head
 * (ln2 rounded to fp32) plus a tail (the fp32 rounding of what the head
 * misses), and r is formed with one fused multiply-add per part.  e^r is the
 * Taylor series of the exponential to degree 7, sum_{n<=7} r^n/n!, evaluated
 * by Horner's rule with fused multiply-adds (the first neglected term,
 * r^8/8!, is below 1e-8 relative for |r| <= ln2/2).  Finally e^x = e^r * 2^k
 * with a single rounding (ldexpf).  Arguments beyond the fp32 range are
 * settled first: above 88.8 the result overflows (+inf), below -104 it is
 * less than half the smallest subnormal (+0).  Each constant is the fp32
 * value nearest to the stated real number. */
static const float kLog2e = 0x1.715476p+0f;    /* 1/ln 2 */
static const float kLn2Hi = 0x1.62e430p-1f;    /* ln 2 */
static const float kLn2Lo = -0x1.05c610p-29f;  /* ln 2 - kLn2Hi */
static const float kInv3f = 0x1.555556p-3f;    /* 1/3! */
static const float kInv4f = 0x1.555556p-5f;    /* 1/4! */
static const float kInv5f = 0x1.111112p-7f;    /* 1/5! */
static const float kInv6f = 0x1.6c16c2p-10f;   /* 1/6! */
static const float kInv7f = 0x1.a01a02p-13f;   /* 1/7! */

float r9o_expf(float x) {
    if (x > 88.8f) return INFINITY;
    if (x < -104.0f) return 0.0f;
    float k = rintf(x * kLog2e);
    float r = fmaf(-k, kLn2Hi, x);
    r = fmaf(-k, kLn2Lo, r);
    float p = kInv7f;
    p = fmaf(p, r, kInv6f);
    p = fmaf(p, r, kInv5f);
    p = fmaf(p, r, kInv4f);
    p = fmaf(p, r, kInv3f);
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    return ldexpf(p, (int)k);
}

void r9o_expf_array(const float* x, int64_t n, float* y) {
    for (int64_t i = 0; i < n; ++i) y[i] = r9o_expf(x[i]);
}

/* --------------------------------------------------------------- SwiGLU ---- */

/* silu(g) * u in fp32: e = exp(-g), silu = g / (1 + e), times u; each
 * operation rounded once (g < -88.8 gives e = +inf and silu = -0). */
float r9o_silu_mul(float g, float u) {
    float e = r9o_expf(-g);
    float d = 1.0f + e;
    float silu = g / d;
    return silu * u;
}

/* h[m][128j + c] = bf16( silu(g) * u ), g = gu[m][256j + c], u = gu[m][256j + 128 + c]:
 * the gate_up output interleaves gate and up per 128 rows (gate first). */
void r9o_swiglu_interleaved(const uint16_t* gu, int64_t M, int64_t I, uint16_t* h) {
    for (int64_t m = 0; m < M; ++m)
        for (int64_t j = 0; j < I / R9O_BLOCK; ++j)
            for (int64_t c = 0; c < R9O_BLOCK; ++c) {
                float g = bf16_bits_to_f32(gu[m * 2 * I + 2 * R9O_BLOCK * j + c]);
                float u = bf16_bits_to_f32(gu[m * 2 * I + 2 * R9O_BLOCK * j + R9O_BLOCK + c]);
                h[m * I + R9O_BLOCK * j + c] = r9o_f32_to_bf16(r9o_silu_mul(g, u));
            }
}

/* Expert MLP at decode: gate_up GEMM -> silu(gate)*up -> group-128 row quant
 * of h -> down GEMM.  weight_only != 0 runs both GEMMs on unquantised bf16
 * activations instead (no quant of x or h).  Every output pointer except y
 * may be NULL.  Shapes: x[M][H], w_gu[2I][H], s_gu[2I/128][H/128],
 * w_dn[Hout][I], s_dn[Hout/128][I/128]. */
int r9o_gate_up_swiglu_down(const uint16_t* x, const uint8_t* w_gu, const float* s_gu,
                            const uint8_t* w_dn, const float* s_dn,
                            int64_t M, int64_t H, int64_t I, int64_t Hout, int weight_only,
                            uint16_t* gu_out, uint16_t* h_out, uint8_t* hq_out, float* hs_out,
                            uint16_t* y) {
    uint16_t* gu = (uint16_t*)malloc(sizeof(uint16_t) * M * 2 * I);
    uint16_t* h = (uint16_t*)malloc(sizeof(uint16_t) * M * I);
    uint8_t* hq = (uint8_t*)malloc((size_t)(M * I));
    float* hs = (float*)malloc(sizeof(float) * M * (I / R9O_BLOCK));
    uint8_t* xq = (uint8_t*)malloc((size_t)(M * H));
    float* xs = (float*)malloc(sizeof(float) * M * (H / R9O_BLOCK));
    if (!gu || !h || !hq || !hs || !xq || !xs) {
        free(gu); free(h); free(hq); free(hs); free(xq); free(xs);
        return -1;
    }
    if (weight_only) {
        r9o_gemm_w8bf16(x, w_gu, s_gu, M, 2 * I, H, NULL, 0, NULL, gu);
    } else {
        r9o_quant_group(x, M, H, R9O_BLOCK, xq, xs);
        r9o_gemm_w8a8(xq, xs, w_gu, s_gu, M, 2 * I, H, NULL, 0, NULL, gu);
    }
    r9o_swiglu_interleaved(gu, M, I, h);
    if (weight_only) {
        r9o_gemm_w8bf16(h, w_dn, s_dn, M, Hout, I, NULL, 0, NULL, y);
    } else {
        r9o_quant_group(h, M, I, R9O_BLOCK, hq, hs);
        r9o_gemm_w8a8(hq, hs, w_dn, s_dn, M, Hout, I, NULL, 0, NULL, y);
    }
    if (gu_out) memcpy(gu_out, gu, sizeof(uint16_t) * M * 2 * I);
    if (h_out) memcpy(h_out, h, sizeof(uint16_t) * M * I);
    if (hq_out && !weight_only) memcpy(hq_out, hq, (size_t)(M * I));
    if (hs_out && !weight_only) memcpy(hs_out, hs, sizeof(float) * M * (I / R9O_BLOCK));
    free(gu); free(h); free(hq); free(hs); free(xq); free(xs);
    return 0;
}

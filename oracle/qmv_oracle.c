/*
 * qmv_oracle.c -- plain, slow CPU oracle for the weight-only-quantized skinny
 * matmul path: the fp32 -> Q8_1 activation quantizer, the Q4_0 x Q8_1 mat-vec
 * (MMVQ), the NVFP4 W4A16 and the FP8 W8A16 skinny GEMM.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark may load this library. It shares no code, header, table or
 * helper with the CUDA path; it is compiled with
 *     gcc -O2 -ffp-contract=off -fPIC -shared
 * so that every fp32 operation below is a single IEEE operation in round to
 * nearest even, on x86_64 and aarch64 alike.
 *
 * Every result here is the plain definition written out: decode each stored
 * code to its exact real value, multiply, sum in fp64. No blocking, no fusion.
 *
 * Sources (the method):
 *  - "Machine Learning on NVIDIA CMP", sections "TL;DR" and "The DP2A patch":
 *    decode is the MMVQ quantized mat x vec, an int8 x int8 dot with int32
 *    accumulation per 4-byte word, over llama.cpp's Q4_0 blocks
 *    (section "llama.cpp results", Llama-2-7B-Q4_0).
 *  - "v100-skinny README", section "How QPN works": QPN2 = NVFP4 W4A16
 *    (e2m1 codes, FP8 scale per 16 weights, a global scale), QPN8 = FP8 e4m3
 *    W8A16 (one contiguous byte stream), fp16 activations.
 * Sources (the formats the pages only name):
 *  - IEEE 754 binary16 for fp16.
 *  - OCP Microscaling Formats (MX) v1.0 for the E2M1 and E4M3 element types
 *    (E4M3 is the "FN" variant: bias 7, no infinities, S.1111.111 = NaN).
 *  - The Q4_0 block is llama.cpp's: fp16 scale d then 16 bytes of nibbles,
 *    element j in the low nibble of byte j, element j+16 in its high nibble,
 *    value d * (q - 8).
 *  - The Q8_1 block: fp16 d8, fp16 s8, 32 int8 q; d8 = max|x| / 127,
 *    q = round(x / d8) (half away from zero), s8 = d8 * sum(q).
 *
 * Parity pins (what ties this file to something other than itself) live in
 * tests/test_oracle_*.py: hand-derived golden blocks, library decoders
 * (numpy float16, torch float8_e4m3fn), closed forms, special cases and fp64
 * brute force on tiny inputs.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Element decoders and encoders                                            */
/* ------------------------------------------------------------------------ */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_fp16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);                 /* f/1024 * 2^-14 */
    } else if (e == 31) {
        v = (f != 0) ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* Round a non-negative double holding an integer plus a fraction to the
 * nearest integer, ties to even. */
static double round_half_even(double q)
{
    double fl = floor(q);
    double frac = q - fl;
    if (frac > 0.5) return fl + 1.0;
    if (frac < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* fp32 -> binary16, round to nearest even, overflow to infinity. */
uint16_t oracle_float_to_fp16(float x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs((double)x);
    if (isnan(x)) return (uint16_t)(sign | 0x7e00u);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u); /* half-way above 65504 rounds to even = inf */
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: unit 2^-24; a rounded count of 1024 is the smallest normal */
        double q = round_half_even(a * ldexp(1.0, 24));
        return (uint16_t)(sign | (uint16_t)q);
    }
    int ex;
    frexp(a, &ex);          /* a = fr * 2^ex, fr in [0.5, 1) */
    int E = ex - 1;         /* a in [2^E, 2^(E+1)) */
    double q = round_half_even(a * ldexp(1.0, 10 - E)); /* in [1024, 2048] */
    if (q == 2048.0) { q = 1024.0; E += 1; }
    if (E > 15) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(q - 1024.0));
}

/* OCP E4M3 (FN): S EEEE MMM, bias 7; E = 0 is subnormal M * 2^-9;
 * S.1111.111 is NaN; no infinities; largest finite 448. */
double oracle_e4m3_to_double(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xf;
    int m = b & 0x7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp((double)(8 + m), e - 10);       /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* OCP E2M1: S EE M, bias 1. The eight magnitudes, in code order. */
static const double kE2M1Magnitude[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double oracle_e2m1_to_double(uint8_t code)
{
    double v = kE2M1Magnitude[code & 0x7];
    return (code & 0x8) ? -v : v;
}

/* Nearest E2M1 code to v (ties to the even code, i.e. the one whose mantissa
 * bit is 0), saturating at +-6. Used by the round-trip check of the table. */
uint8_t oracle_e2m1_encode(double v)
{
    uint8_t sign = (v < 0.0 || (v == 0.0 && signbit(v))) ? 0x8 : 0x0;
    double a = fabs(v);
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c < 8; ++c) {
        double err = fabs(kE2M1Magnitude[c] - a);
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(sign | best);
}

/* ------------------------------------------------------------------------ */
/* Q8_1 activation quantizer                                               */
/* ------------------------------------------------------------------------ */

/*
 * x: fp32 [M][K] row-major; xq: M * (K/32) blocks of 36 bytes, row-major:
 *   bytes 0..1  d8 (binary16, little-endian)
 *   bytes 2..3  s8 (binary16, little-endian)
 *   bytes 4..35 q[0..31] (int8)
 * Per block, in fp32: amax = max|x_i|; d = amax / 127; q_i = 0 if d == 0 else
 * clamp(roundf(x_i / d), -127, 127); d8 = fp16(d); s8 = fp16(d * (float)sum q).
 * K must be a multiple of 32.
 */
void oracle_quantize_q8_1(const float *x, uint8_t *xq, int64_t M, int64_t K)
{
    int64_t nb = K / 32;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *xb = x + m * K + b * 32;
            uint8_t *blk = xq + (m * nb + b) * 36;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                float a = fabsf(xb[i]);
                if (a > amax) amax = a;
            }
            float d = amax / 127.0f;
            int sum = 0;
            for (int i = 0; i < 32; ++i) {
                int q = 0;
                if (d != 0.0f) {
                    float r = roundf(xb[i] / d);
                    if (r > 127.0f) r = 127.0f;
                    if (r < -127.0f) r = -127.0f;
                    q = (int)r;
                }
                sum += q;
                blk[4 + i] = (uint8_t)(int8_t)q;
            }
            uint16_t d8 = oracle_float_to_fp16(d);
            uint16_t s8 = oracle_float_to_fp16(d * (float)sum);
            blk[0] = (uint8_t)(d8 & 0xff);
            blk[1] = (uint8_t)(d8 >> 8);
            blk[2] = (uint8_t)(s8 & 0xff);
            blk[3] = (uint8_t)(s8 >> 8);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Q4_0 x Q8_1                                                              */
/* ------------------------------------------------------------------------ */

static uint16_t read_u16le(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* Unsigned nibble j (0..31) of a Q4_0 block's 16 data bytes. */
static int q4_0_nibble(const uint8_t *qs, int j)
{
    return (j < 16) ? (qs[j] & 0x0f) : (qs[j - 16] >> 4);
}

/*
 * Integer block dot products of the MMVQ inner loop ("The DP2A patch": int8 x
 * int8 products summed in int32):
 *   S[m][n][b] = sum_j q4u_j * q8_j       (q4u the unsigned nibble, 0..15)
 *   T[m][b]    = sum_j q8_j
 * w: Q4_0 [N][K/32] blocks of 18 bytes; xq: Q8_1 [M][K/32] blocks of 36 bytes.
 */
void oracle_q4_0_block_dots(const uint8_t *w, const uint8_t *xq, int64_t M, int64_t N,
                            int64_t K, int32_t *S, int32_t *T)
{
    int64_t nb = K / 32;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t b = 0; b < nb; ++b) {
            const int8_t *q8 = (const int8_t *)(xq + (m * nb + b) * 36 + 4);
            int32_t t = 0;
            for (int j = 0; j < 32; ++j) t += q8[j];
            T[m * nb + b] = t;
            for (int64_t n = 0; n < N; ++n) {
                const uint8_t *qs = w + (n * nb + b) * 18 + 2;
                int32_t s = 0;
                for (int j = 0; j < 32; ++j) s += q4_0_nibble(qs, j) * q8[j];
                S[(m * N + n) * nb + b] = s;
            }
        }
    }
}

/*
 * y[m][n] = sum_k w[n][k] * xhat[m][k] in fp64, where
 *   w[n][k]    = d4 * (q4u - 8)           (d4 the block's fp16 scale)
 *   xhat[m][k] = d8 * q8                  (d8 the Q8_1 block's stored fp16 scale)
 * bound[m][n] = sum_k |w[n][k] * xhat[m][k]| (the scale of the tolerance).
 */
void oracle_q4_0_q8_1(const uint8_t *w, const uint8_t *xq, int64_t M, int64_t N, int64_t K,
                      double *y, double *bound)
{
    int64_t nb = K / 32;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t *wb = w + (n * nb + b) * 18;
                const uint8_t *xb = xq + (m * nb + b) * 36;
                double d4 = oracle_fp16_to_double(read_u16le(wb));
                double d8 = oracle_fp16_to_double(read_u16le(xb));
                const int8_t *q8 = (const int8_t *)(xb + 4);
                for (int j = 0; j < 32; ++j) {
                    double wv = d4 * (double)(q4_0_nibble(wb + 2, j) - 8);
                    double xv = d8 * (double)q8[j];
                    acc += wv * xv;
                    mag += fabs(wv * xv);
                }
            }
            y[m * N + n] = acc;
            bound[m * N + n] = mag;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* NVFP4 W4A16                                                              */
/* ------------------------------------------------------------------------ */

/*
 * codes:  [N][K/2] bytes; k even in the low nibble, k odd in the high nibble
 * scales: [N][K/16] E4M3 bytes, one per 16 consecutive k of the row
 * g:      per-tensor fp32 scale
 * x:      fp16 [M][K] (binary16 bit patterns)
 * y[m][n] = sum_k e2m1(code[n][k]) * e4m3(scale[n][k/16]) * g * x[m][k]  (fp64)
 */
void oracle_nvfp4_w4a16(const uint8_t *codes, const uint8_t *scales, float g,
                        const uint16_t *x, int64_t M, int64_t N, int64_t K,
                        double *y, double *bound)
{
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                uint8_t byte = codes[n * (K / 2) + k / 2];
                uint8_t code = (k % 2 == 0) ? (uint8_t)(byte & 0x0f) : (uint8_t)(byte >> 4);
                double wv = oracle_e2m1_to_double(code) *
                            oracle_e4m3_to_double(scales[n * (K / 16) + k / 16]) * (double)g;
                double xv = oracle_fp16_to_double(x[m * K + k]);
                acc += wv * xv;
                mag += fabs(wv * xv);
            }
            y[m * N + n] = acc;
            bound[m * N + n] = mag;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* FP8 W8A16                                                                */
/* ------------------------------------------------------------------------ */

/*
 * w:  [N][K] E4M3 bytes; rs: fp32 [N] per-row scale; x: fp16 [M][K]
 * y[m][n] = sum_k e4m3(w[n][k]) * rs[n] * x[m][k]  (fp64)
 */
void oracle_fp8_w8a16(const uint8_t *w, const float *rs, const uint16_t *x, int64_t M,
                      int64_t N, int64_t K, double *y, double *bound)
{
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double wv = oracle_e4m3_to_double(w[n * K + k]) * (double)rs[n];
                double xv = oracle_fp16_to_double(x[m * K + k]);
                acc += wv * xv;
                mag += fabs(wv * xv);
            }
            y[m * N + n] = acc;
            bound[m * N + n] = mag;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Q4_K x Q8_1                                                              */
/* ------------------------------------------------------------------------ */

/*
 * The Q4_K super-block ("Machine Learning on NVIDIA CMP", section "llama.cpp
 * results" names the Q4_K_M models; the pages do not print the layout, which is
 * llama.cpp's GGUF K-quant format): 256 weights in 144 bytes,
 *   bytes 0..1    d     (fp16) scale of the sub-block scales
 *   bytes 2..3    dmin  (fp16) scale of the sub-block minimums
 *   bytes 4..15   eight 6-bit sub-block scales sc[j] and minimums mn[j], packed:
 *                 j < 4:  sc = byte[j] & 63,  mn = byte[j+4] & 63
 *                 j >= 4: sc = (byte[j+4] & 15) | (byte[j-4] >> 6) << 4
 *                         mn = (byte[j+4] >> 4) | (byte[j]   >> 6) << 4
 *   bytes 16..143 128 bytes of unsigned nibbles: byte 32c + e holds element
 *                 64c + e in its low nibble and element 64c + 32 + e in its high
 *                 nibble (c = 0..3, e = 0..31), i.e. sub-block 2c in the low and
 *                 sub-block 2c + 1 in the high nibbles of the same 32 bytes.
 * Element i of sub-block j (32 weights) has the value
 *   w = d * sc[j] * q - dmin * mn[j].
 */

/* The 6-bit scale and minimum of sub-block j (0..7) from the 12 packed bytes. */
void oracle_q4_k_scale_min(const uint8_t *p, int j, int *sc, int *mn)
{
    if (j < 4) {
        *sc = p[j] & 63;
        *mn = p[j + 4] & 63;
    } else {
        *sc = (p[j + 4] & 15) | ((p[j - 4] >> 6) << 4);
        *mn = (p[j + 4] >> 4) | ((p[j] >> 6) << 4);
    }
}

/* Unsigned nibble of element i (0..255) of a super-block's 128 data bytes. */
static int q4_k_nibble(const uint8_t *qs, int i)
{
    int c = i / 64, r = i % 64;
    return (r < 32) ? (qs[32 * c + r] & 0x0f) : (qs[32 * c + r - 32] >> 4);
}

/* Dequantized value of element i (0..255) of one 144-byte super-block. */
double oracle_q4_k_weight(const uint8_t *blk, int i)
{
    int sc, mn;
    oracle_q4_k_scale_min(blk + 4, i / 32, &sc, &mn);
    double d = oracle_fp16_to_double(read_u16le(blk));
    double dmin = oracle_fp16_to_double(read_u16le(blk + 2));
    return d * (double)sc * (double)q4_k_nibble(blk + 16, i) - dmin * (double)mn;
}

/*
 * Integer dots of the MMVQ inner loop per 32-weight sub-block b (= Q8_1 block b):
 *   S[m][n][b] = sum_i q4u_i * q8_i   (q4u the unsigned nibble, 0..15)
 * w: Q4_K [N][K/256] super-blocks of 144 bytes; xq: Q8_1 [M][K/32] blocks.
 */
void oracle_q4_k_block_dots(const uint8_t *w, const uint8_t *xq, int64_t M, int64_t N,
                            int64_t K, int32_t *S)
{
    int64_t nsb = K / 256, nb = K / 32;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t *qs = w + (n * nsb + b / 8) * 144 + 16;
                const int8_t *q8 = (const int8_t *)(xq + (m * nb + b) * 36 + 4);
                int32_t s = 0;
                for (int i = 0; i < 32; ++i) s += q4_k_nibble(qs, (int)(b % 8) * 32 + i) * q8[i];
                S[(m * N + n) * nb + b] = s;
            }
        }
    }
}

/*
 * y[m][n] = sum_k w[n][k] * xhat[m][k] in fp64, w the dequantized Q4_K value above
 * and xhat = d8 * q8 the dequantized Q8_1 activation; bound = sum_k |w * xhat|.
 */
void oracle_q4_k_q8_1(const uint8_t *w, const uint8_t *xq, int64_t M, int64_t N, int64_t K,
                      double *y, double *bound)
{
    int64_t nsb = K / 256, nb = K / 32;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const uint8_t *xb = xq + (m * nb + k / 32) * 36;
                double wv = oracle_q4_k_weight(w + (n * nsb + k / 256) * 144, (int)(k % 256));
                double xv = oracle_fp16_to_double(read_u16le(xb)) * (double)((const int8_t *)(xb + 4))[k % 32];
                acc += wv * xv;
                mag += fabs(wv * xv);
            }
            y[m * N + n] = acc;
            bound[m * N + n] = mag;
        }
    }
}

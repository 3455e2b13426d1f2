/*
 * NVFP4 oracle: a plain, slow, obviously-correct CPU restatement of the NVFP4
 * quantizer that the Full-Stack FP4 pages build on.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may link,
 * load or call this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header or table with
 * the CUDA path.
 *
 * Sources for what is computed here:
 *   - "Full-Stack FP4: Stable LLM Pretraining with Quantized Projections,
 *     Optimizers, and Attention" (gist.science explainer, es/fr), section 1
 *     (Problem statement): the target is NVFP4 on Blackwell tensor cores;
 *     section 3 (Key contributions): "standard NVFP4" quantization of the
 *     linear projections; section 2.2 (Q-AdamW): stochastic rounding (SR).
 *   - The pages never define the NVFP4 encoding.  This file takes the
 *     plainest reading of the format: E2M1 element codes (grid
 *     +-{0,0.5,1,1.5,2,3,4,6}), one unsigned E4M3 scale per 16 contiguous
 *     elements, one FP32 tensor scale; round-to-nearest-even (RTN) for
 *     weights/activations, SR for gradients.  Every choice the pages leave
 *     open is marked READING below.
 *
 * Precision: every step is the single FP32 operation written in the source
 * (compile with -ffp-contract=off, no fast-math), so the results are fixed to
 * the bit.  Rounding to E4M3 and E2M1 is done by brute force: enumerate every
 * finite value of the format and take the nearest one, ties to the even code.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <float.h>

/* ------------------------------------------------------------------ */
/* BF16                                                                */
/* ------------------------------------------------------------------ */

/* BF16 is the upper half of an IEEE binary32; widening is exact. */
float oracle_bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round a double to the nearest BF16, ties to the even pattern, overflow to
 * +-inf.  Works on the value: find the two neighbouring BF16 numbers
 * lo <= |v| < hi (spacing 2^(e-7) in binade e, 2^-133 below 2^-126) and take
 * the nearer one.  Rounding the double to binary32 first would round twice. */
uint16_t oracle_f64_to_bf16_rn(double v) {
    if (v != v) return 0x7FC0;
    uint16_t sign = (v < 0 || (v == 0 && signbit(v))) ? 0x8000 : 0;
    double a = fabs(v);
    /* largest finite BF16 = (2 - 2^-7) * 2^127 ; halfway to 2^128 rounds up */
    double maxf = ldexp(2.0 - ldexp(1.0, -7), 127);
    double over = ldexp(2.0 - ldexp(1.0, -8), 127);
    if (a >= over) return sign | 0x7F80; /* +-inf */
    if (a >= maxf) return sign | 0x7F7F;
    if (a == 0) return sign;
    int e;
    frexp(a, &e);            /* a = m * 2^e, m in [0.5,1) */
    int exp_unbiased = e - 1; /* a in [2^(e-1), 2^e) */
    if (exp_unbiased < -126) exp_unbiased = -126; /* subnormal spacing */
    double ulp = ldexp(1.0, exp_unbiased - 7);     /* 8 significant bits */
    double q = floor(a / ulp);                      /* exact: power-of-two division */
    double lo = q * ulp, hi = (q + 1) * ulp;
    double pick;
    if (a - lo < hi - a) pick = lo;
    else if (a - lo > hi - a) pick = hi;
    else pick = (fmod(q, 2.0) == 0.0) ? lo : hi;
    float pf = (float)pick; /* exact: pick is a BF16 value */
    uint32_t u;
    memcpy(&u, &pf, 4);
    return sign | (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------ */
/* E4M3 (the block-scale format): 1 sign, 4 exponent bits (bias 7),    */
/* 3 mantissa bits, no infinities, 0x7F / 0xFF are NaN, max 448.       */
/* Scales are unsigned, so only bytes 0x00..0x7E are produced.         */
/* ------------------------------------------------------------------ */

double oracle_e4m3_value(uint8_t b) {
    int s = (b >> 7) & 1, e = (b >> 3) & 0xF, m = b & 7;
    if (e == 0xF && m == 7) return NAN;
    double mag = (e == 0) ? ldexp((double)m, -9)                 /* m/8 * 2^-6 */
                          : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* The 127 non-negative finite E4M3 values, filled from oracle_e4m3_value
 * when the library is loaded (so the search below does no ldexp). */
static double E4M3_POS[127];
__attribute__((constructor)) static void fill_e4m3_table(void) {
    for (int b = 0; b <= 0x7E; ++b) E4M3_POS[b] = oracle_e4m3_value((uint8_t)b);
}

/* Nearest non-negative finite E4M3 value to v (v >= 0), ties to the even
 * code, values beyond 448 saturate to 448 (they are nearest to it).
 * READING: round-to-nearest-even with saturation for the block scale. */
uint8_t oracle_e4m3_encode_rn_sat(float v) {
    double x = (double)v;
    if (x > 448.0) x = 448.0; /* saturate first: far values would tie in FP64 */
    uint8_t best = 0;
    double bestd = INFINITY;
    for (int b = 0; b <= 0x7E; ++b) {
        double d = fabs(E4M3_POS[b] - x);
        if (d < bestd || (d == bestd && (b & 1) == 0)) {
            best = (uint8_t)b;
            bestd = d;
        }
    }
    return best;
}

/* ------------------------------------------------------------------ */
/* E2M1 (the element format): code = sign<<3 | index, index 0..7 over  */
/* the magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}.                         */
/* ------------------------------------------------------------------ */

static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double oracle_e2m1_value(uint8_t code) {
    double m = E2M1_MAG[code & 7];
    return (code & 8) ? -m : m;
}

/* RTN: nearest magnitude, ties to the even index, saturating at 6.
 * READING: the sign bit is kept for values that round to zero (so a
 * negative input gives code 0x8, "negative zero"), as an IEEE conversion
 * does. */
uint8_t oracle_e2m1_rtn(float y) {
    uint8_t sign = signbit(y) ? 8 : 0;
    double a = fabs((double)y);
    if (a > 6.0) a = 6.0; /* saturate first: far values would tie in FP64 */
    int best = 0;
    double bestd = INFINITY;
    for (int i = 0; i < 8; ++i) {
        double d = fabs(E2M1_MAG[i] - a);
        if (d < bestd || (d == bestd && (i & 1) == 0)) {
            best = i;
            bestd = d;
        }
    }
    return sign | (uint8_t)best;
}

/* SR: with a = min(|y|, 6), lo = largest grid magnitude <= a and sp the gap
 * to the next grid magnitude, round up iff rnd16 < frac * 65536 where
 * frac = (a - lo) / sp.  Both the subtraction and the division by a power
 * of two are exact in FP32, so frac is exact.  READING: 16 random bits per
 * element, the comparison above, sign kept as for RTN. */
uint8_t oracle_e2m1_sr(float y, uint32_t rnd16) {
    uint8_t sign = signbit(y) ? 8 : 0;
    float a = fabsf(y);
    if (a > 6.0f) a = 6.0f;
    int lo = 0;
    for (int i = 0; i < 8; ++i)
        if (E2M1_MAG[i] <= (double)a) lo = i;
    if (lo == 7) return sign | 7;
    float lov = (float)E2M1_MAG[lo];
    float sp = (float)(E2M1_MAG[lo + 1] - E2M1_MAG[lo]);
    float frac = (a - lov) / sp;
    float thresh = frac * 65536.0f;
    int up = ((float)rnd16 < thresh) ? 1 : 0;
    return sign | (uint8_t)(lo + up);
}

/* ------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw: "Parallel random numbers: */
/* as easy as 1, 2, 3", SC'11).  A round multiplies counter words 0 and */
/* 2 by two fixed odd constants into 64-bit products; the new counter   */
/* is (hi(c2*M1)^c1^k0, lo(c2*M1), hi(c0*M0)^c3^k1, lo(c0*M0)); the key */
/* is bumped by the Weyl constants between rounds.                      */
/* ------------------------------------------------------------------ */

void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += W0;
            k1 += W1;
        }
        uint64_t p0 = (uint64_t)M0 * (uint64_t)c0;
        uint64_t p1 = (uint64_t)M1 * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The 16 random bits that drive SR of element e (its row-major index in
 * the SOURCE tensor) in stream `stream` under `seed`.
 * READING (the pages fix no generator): key = (seed lo32, seed hi32),
 * counter = (j lo32, j hi32, stream, 0) with j = e / 8; element e takes
 * output word (e % 8) / 2, its low half when e is even, high half when odd. */
uint32_t oracle_sr_bits(uint64_t seed, uint32_t stream, uint64_t e) {
    uint64_t j = e / 8;
    uint32_t ctr[4] = {(uint32_t)j, (uint32_t)(j >> 32), stream, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    uint32_t w = out[(e % 8) / 2];
    return (e % 2 == 0) ? (w & 0xFFFFu) : (w >> 16);
}

/* ------------------------------------------------------------------ */
/* Tensor amax and the FP32 tensor scale                               */
/* ------------------------------------------------------------------ */

float oracle_amax_bf16(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld) {
    float m = 0.0f;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            float a = fabsf(oracle_bf16_to_f32(x[r * ld + c]));
            if (a > m) m = a;
        }
    return m;
}

/* READING: S_t is the decode scale amax / (6 * 448) = amax / 2688, one
 * correctly-rounded FP32 division; an all-zero tensor has S_t = 0. */
float oracle_tensor_scale(float amax) {
    if (amax == 0.0f) return 0.0f;
    return amax / 2688.0f;
}

/* ------------------------------------------------------------------ */
/* Quantize one block of 16 values (already widened to FP32).          */
/*   s_b = E4M3_rn_sat( amax_b / (6 * S_t) )                            */
/*   d   = s_b * S_t            inv = 1 / d (capped at FLT_MAX)         */
/*   y   = x * inv              code = E2M1(y)  (RTN or SR)             */
/* READING: a block whose scale rounds to 0 (or S_t = 0) gets inv = 0,   */
/* i.e. every code is a signed zero.  inv is capped at FLT_MAX so that   */
/* tiny tensors (amax < ~4e-33) never form 0 * inf.                       */
/* ------------------------------------------------------------------ */

static uint8_t block_scale(const float* v, int n, float S_t, float* inv_out) {
    float amax_b = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(v[i]);
        if (a > amax_b) amax_b = a;
    }
    uint8_t s_b = 0;
    if (S_t > 0.0f) {
        float denom = 6.0f * S_t;
        float ratio = amax_b / denom;
        s_b = oracle_e4m3_encode_rn_sat(ratio);
    }
    float inv = 0.0f;
    if (s_b != 0) {
        float d = (float)oracle_e4m3_value(s_b) * S_t;
        inv = 1.0f / d;
        if (inv > FLT_MAX) inv = FLT_MAX;
    }
    *inv_out = inv;
    return s_b;
}

/* Row orientation: blocks of 16 along cols.  x is rows x cols (leading
 * dimension ld, in elements); cols must be a multiple of 16.
 * codes: rows x cols/2 bytes, row-major, element 2i in the low nibble.
 * scales: rows x cols/16 bytes, row-major (the MMA layout is a separate
 * permutation, oracle_mma_scale_offset).
 * mode 0 = RTN, 1 = SR (seed, stream; element index e = r*cols + c). */
void oracle_quantize_rows(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                          int mode, uint64_t seed, uint32_t stream, float S_t,
                          uint8_t* codes, uint8_t* scales) {
    int64_t kb = cols / 16;
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < kb; ++b) {
            float v[16];
            for (int i = 0; i < 16; ++i) v[i] = oracle_bf16_to_f32(x[r * ld + b * 16 + i]);
            float inv;
            uint8_t s_b = block_scale(v, 16, S_t, &inv);
            scales[r * kb + b] = s_b;
            for (int i = 0; i < 16; ++i) {
                float y = v[i] * inv;
                uint8_t q;
                if (mode == 0) q = oracle_e2m1_rtn(y);
                else q = oracle_e2m1_sr(y, oracle_sr_bits(seed, stream, (uint64_t)(r * cols + b * 16 + i)));
                int64_t idx = r * cols + b * 16 + i; /* element index in the codes tensor */
                uint8_t* byte = &codes[idx / 2];
                if (idx % 2 == 0) *byte = (uint8_t)((*byte & 0xF0) | q);
                else *byte = (uint8_t)((*byte & 0x0F) | (q << 4));
            }
        }
    }
}

/* Row orientation of an FP32 tensor (RTN only): the same block rule as
 * oracle_quantize_rows applied to FP32 inputs (used by the optimizer-state
 * codec, whose transformed values are FP32). */
void oracle_quantize_rows_f32(const float* x, int64_t rows, int64_t cols, float S_t,
                              uint8_t* codes, uint8_t* scales) {
    int64_t kb = cols / 16;
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < kb; ++b) {
            float v[16];
            for (int i = 0; i < 16; ++i) v[i] = x[r * cols + b * 16 + i];
            float inv;
            uint8_t s_b = block_scale(v, 16, S_t, &inv);
            scales[r * kb + b] = s_b;
            for (int i = 0; i < 16; ++i) {
                uint8_t q = oracle_e2m1_rtn(v[i] * inv);
                int64_t idx = r * cols + b * 16 + i;
                uint8_t* byte = &codes[idx / 2];
                if (idx % 2 == 0) *byte = (uint8_t)((*byte & 0xF0) | q);
                else *byte = (uint8_t)((*byte & 0x0F) | (q << 4));
            }
        }
    }
}

/* Column orientation: blocks of 16 along rows, emitted as the transposed
 * (cols x rows) tensor, i.e. output row c holds source column c.  rows must
 * be a multiple of 16.  codes: cols x rows/2 bytes; scales: cols x rows/16.
 * The SR element index e is the SOURCE row-major index r*cols + c. */
void oracle_quantize_cols(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                          int mode, uint64_t seed, uint32_t stream, float S_t,
                          uint8_t* codes, uint8_t* scales) {
    int64_t kb = rows / 16;
    #pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < cols; ++c) {
        for (int64_t b = 0; b < kb; ++b) {
            float v[16];
            for (int i = 0; i < 16; ++i) v[i] = oracle_bf16_to_f32(x[(b * 16 + i) * ld + c]);
            float inv;
            uint8_t s_b = block_scale(v, 16, S_t, &inv);
            scales[c * kb + b] = s_b;
            for (int i = 0; i < 16; ++i) {
                int64_t r = b * 16 + i;
                float y = v[i] * inv;
                uint8_t q;
                if (mode == 0) q = oracle_e2m1_rtn(y);
                else q = oracle_e2m1_sr(y, oracle_sr_bits(seed, stream, (uint64_t)(r * cols + c)));
                int64_t idx = c * rows + r; /* element index in the transposed codes tensor */
                uint8_t* byte = &codes[idx / 2];
                if (idx % 2 == 0) *byte = (uint8_t)((*byte & 0xF0) | q);
                else *byte = (uint8_t)((*byte & 0x0F) | (q << 4));
            }
        }
    }
}

/* Dequantize: out[r][c] = e2m1(code) * e4m3(s_b) * S_t, exact in FP64
 * (a 4-bit value times an 8-bit value times an FP32 is exact in 53 bits). */
void oracle_dequantize(const uint8_t* codes, const uint8_t* scales, float S_t,
                       int64_t rows, int64_t cols, double* out) {
    int64_t kb = cols / 16;
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            int64_t idx = r * cols + c;
            uint8_t byte = codes[idx / 2];
            uint8_t q = (idx % 2 == 0) ? (byte & 0xF) : (byte >> 4);
            out[idx] = oracle_e2m1_value(q) * oracle_e4m3_value(scales[r * kb + c / 16]) * (double)S_t;
        }
}

/* ------------------------------------------------------------------ */
/* Scale layout read by the block-scaled tensor-core MMA.               */
/* The row-major scale matrix [rows][kb] is cut into atoms of 128 rows  */
/* x 4 scale columns (512 bytes).  Atoms are stored row-block-major      */
/* (all atoms of rows 0..127 first, in k order).  Inside an atom, scale  */
/* (r, k) sits at byte (r % 32) * 16 + (r / 32) * 4 + k.  rows and kb are */
/* padded up to multiples of 128 and 4.                                  */
/* READING: this is the hardware's published block-scale layout; it is a */
/* pure index permutation and changes no value.                          */
/* ------------------------------------------------------------------ */

int64_t oracle_mma_scale_offset(int64_t r, int64_t k, int64_t kb) {
    int64_t atoms_k = (kb + 3) / 4;
    int64_t atom = (r / 128) * atoms_k + (k / 4);
    int64_t rr = r % 128;
    return atom * 512 + (rr % 32) * 16 + (rr / 32) * 4 + (k % 4);
}

int64_t oracle_mma_scale_bytes(int64_t rows, int64_t kb) {
    return ((rows + 127) / 128) * 128 * ((kb + 3) / 4) * 4;
}

/* Permute row-major scales into the MMA layout (padding bytes left 0). */
void oracle_scales_to_mma(const uint8_t* rowmajor, int64_t rows, int64_t kb, uint8_t* mma) {
    memset(mma, 0, (size_t)oracle_mma_scale_bytes(rows, kb));
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < kb; ++k)
            mma[oracle_mma_scale_offset(r, k, kb)] = rowmajor[r * kb + k];
}

/* ------------------------------------------------------------------ */
/* Array helpers (elementwise loops over the scalar definitions above)  */
/* ------------------------------------------------------------------ */

void oracle_f64_to_bf16_rn_array(const double* v, int64_t n, uint16_t* out) {
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f64_to_bf16_rn(v[i]);
}

void oracle_e4m3_encode_array(const float* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode_rn_sat(v[i]);
}

void oracle_e2m1_rtn_array(const float* y, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_rtn(y[i]);
}

void oracle_e2m1_sr_array(const float* y, const uint32_t* rnd16, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_sr(y[i], rnd16[i]);
}

void oracle_sr_bits_array(uint64_t seed, uint32_t stream, uint64_t e0, int64_t n, uint32_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_sr_bits(seed, stream, e0 + (uint64_t)i);
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    extern void omp_set_num_threads(int);
    omp_set_num_threads(n);
#else
    (void)n;
#endif
}

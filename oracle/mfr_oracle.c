/*
 * CPU oracle for the MoE finalize + residual + RMSNorm path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this file: only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * It is deliberately plain and slow: one token at a time, one column at a
 * time, no blocking, no vectors, no threads.  Build with
 *     gcc -O2 -std=c11 -fno-fast-math -ffp-contract=off -fPIC -shared -lm
 * so that a fused multiply-add happens only where fmaf() is written.
 *
 * What it computes, and where each step is stated:
 *
 *  [A] "FlashInfer MoE 성능 최적화: CuTe DSL을 활용한 Deterministic Finalize
 *      개선기" (flashinfer PR 5319 analysis), section 1, the new CuTe-DSL
 *      finalize kernel: the k expert outputs of a token are accumulated with
 *      FP32 fused multiply-adds (round to nearest) and converted to BF16 only
 *      at the very end; the unfused finalize is the deterministic one.
 *  [B] "Blackwell 아키텍처를 위한 MoE All-Reduce Fusion 최적화: FlashInfer의
 *      'Cake' 백엔드 분석" (flashinfer PR 4730 analysis), section 2, the fusion
 *      strategy: sum the expert outputs, add the residual, then RMSNorm, all
 *      in one pass.
 *  [C] "FlashInfer, Muse-Spark-Open을 위한 융합 정규화 및 TP/EP MoE 최적화로
 *      성능 극대화" (flashinfer PR 6544 analysis), section 1.1 (the residual
 *      stream is kept in FP32) and section 2.1 (the finalize reads the rows
 *      straight from the GEMM2 result, i.e. in expert-grouped order through
 *      an index map).
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes): the accumulator starts at +0 and the residual is added once after
 * the k slots; slots run j = 0..k-1 in the order stored; weights are used as
 * given; FMA without flush-to-zero; RMS over the FP32 updated residual with
 * eps inside the square root; y = x / rms * gamma (not 1 + gamma); an index
 * outside [0, R) makes its slot contribute nothing and is counted.
 *
 * A second reading of [C] section 2.1 (an RMSNorm per expert row before the
 * weighted sum, no residual) is kept apart at the end of the file.
 *
 * Precision: steps [A] and the residual add are FP32, exactly as the pages fix
 * them.  The normalisation is not fixed by the pages, so the oracle computes
 * it in double and rounds once, from double, to BF16 (nearest, ties to even).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

/* ---- BF16 <-> binary64 ---------------------------------------------------- */

/* A BF16 value is the upper half of the FP32 encoding; widening is exact. */
double mfr_oracle_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * Nearest BF16 to a double, ties to even, with a single rounding.
 * BF16 has 8 significant bits, exponents -126..127 for normal numbers and a
 * fixed spacing of 2^-133 below 2^-126.  The value is divided by its BF16
 * spacing (a power of two, so exactly), rounded to an integer with the
 * default nearest-even mode, and multiplied back.  Results at or above 2^128
 * overflow to infinity.  NaN maps to the quiet NaN 0x7FC0 with its sign.
 */
uint16_t mfr_oracle_bf16_from_f64(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x))
        return (uint16_t)(sign | 0x7FC0u);
    double a = fabs(x);
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0)
        return sign;
    int e;
    (void)frexp(a, &e);          /* a in [2^(e-1), 2^e) */
    int lead = e - 1;            /* exponent of the leading bit */
    if (lead < -126)
        lead = -126;             /* subnormal range: fixed spacing */
    double spacing = ldexp(1.0, lead - 7);
    double q = nearbyint(a / spacing);
    double r = q * spacing;
    if (r >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80u);
    float f = (float)r;          /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFFu));
}

void mfr_oracle_bf16_from_f64_array(const double* x, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = mfr_oracle_bf16_from_f64(x[i]);
}

/* ---- steps a3-a5: gather, FP32 weighted sum, residual --------------------- */

static int slot_valid(int32_t r, int64_t R)
{
    return r >= 0 && (int64_t)r < R;
}

/* Number of slots of token t whose index lies outside [0, R). */
static int64_t count_bad_slots(int64_t t, int64_t k, int64_t R, const int32_t* idx)
{
    int64_t bad = 0;
    for (int64_t j = 0; j < k; ++j)
        if (!slot_valid(idx[t * k + j], R))
            ++bad;
    return bad;
}

/*
 * acc = +0; for j = 0..k-1: acc = fmaf(w[t,j], E[idx[t,j], h], acc)   [A]
 * x   = residual_in[t, h] + acc   (one FP32 add)                       [B][C]
 * Rows i of x correspond to tokens[i] (or to i when tokens is NULL).
 * Returns the number of (token, slot) pairs whose index was out of range.
 */
int64_t mfr_oracle_weighted_residual(int64_t T, int64_t H, int64_t k, int64_t R,
                                     const uint16_t* expert_out, const int32_t* idx,
                                     const float* w, const float* residual_in,
                                     float* x, const int64_t* tokens, int64_t ntokens)
{
    int64_t bad = 0;
    int64_t n = tokens ? ntokens : T;
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = tokens ? tokens[i] : i;
        bad += count_bad_slots(t, k, R, idx);
        for (int64_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int64_t j = 0; j < k; ++j) {
                int32_t r = idx[t * k + j];
                if (!slot_valid(r, R))
                    continue;
                float e = bf16_to_f32(expert_out[(int64_t)r * H + h]);
                acc = fmaf(w[t * k + j], e, acc);
            }
            x[i * H + h] = residual_in[t * H + h] + acc;
        }
    }
    return bad;
}

/* ---- steps a6-a7: RMSNorm in double --------------------------------------- */

/*
 * y[h] = x[h] / sqrt(mean_h(x^2) + eps) * gamma[h], in double, for n rows of
 * width H.  This is the plain definition of RMSNorm applied to the updated
 * FP32 residual [B].
 */
void mfr_oracle_rmsnorm_f64(int64_t n, int64_t H, const float* x,
                            const uint16_t* gamma, float eps, double* y)
{
    for (int64_t i = 0; i < n; ++i) {
        const float* xr = x + i * H;
        double ss = 0.0;
        for (int64_t h = 0; h < H; ++h)
            ss += (double)xr[h] * (double)xr[h];
        double inv = 1.0 / sqrt(ss / (double)H + (double)eps);
        for (int64_t h = 0; h < H; ++h)
            y[i * H + h] = (double)xr[h] * inv * mfr_oracle_bf16_to_f64(gamma[h]);
    }
}

/* ---- the whole path ------------------------------------------------------- */

/*
 * residual_out[i, :] = x of token tokens[i] (FP32);
 * out[i, :]          = BF16(RMSNorm(x) * gamma), one rounding from double.
 * Works one token at a time so a sampled subset of a large workload needs
 * only H doubles of scratch, which the caller passes in ``y_scratch``.
 */
int64_t mfr_oracle_finalize_residual_rmsnorm(
    int64_t T, int64_t H, int64_t k, int64_t R,
    const uint16_t* expert_out, const int32_t* idx, const float* w,
    const float* residual_in, const uint16_t* gamma, float eps,
    float* residual_out, uint16_t* out,
    const int64_t* tokens, int64_t ntokens, double* y_scratch)
{
    int64_t bad = 0;
    int64_t n = tokens ? ntokens : T;
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = tokens ? tokens[i] : i;
        float* xr = residual_out + i * H;
        bad += mfr_oracle_weighted_residual(T, H, k, R, expert_out, idx, w,
                                            residual_in, xr, &t, 1);
        mfr_oracle_rmsnorm_f64(1, H, xr, gamma, eps, y_scratch);
        for (int64_t h = 0; h < H; ++h)
            out[i * H + h] = mfr_oracle_bf16_from_f64(y_scratch[h]);
    }
    return bad;
}

/*
 * Finalize only (no residual, no norm): out = BF16(acc) with acc the FP32
 * weighted sum of [A].  This is the plain "MoE finalize" of the PR 5319 page.
 */
int64_t mfr_oracle_finalize_only(int64_t T, int64_t H, int64_t k, int64_t R,
                                 const uint16_t* expert_out, const int32_t* idx,
                                 const float* w, uint16_t* out,
                                 const int64_t* tokens, int64_t ntokens)
{
    int64_t bad = 0;
    int64_t n = tokens ? ntokens : T;
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = tokens ? tokens[i] : i;
        bad += count_bad_slots(t, k, R, idx);
        for (int64_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int64_t j = 0; j < k; ++j) {
                int32_t r = idx[t * k + j];
                if (!slot_valid(r, R))
                    continue;
                acc = fmaf(w[t * k + j], bf16_to_f32(expert_out[(int64_t)r * H + h]), acc);
            }
            out[i * H + h] = mfr_oracle_bf16_from_f64((double)acc);
        }
    }
    return bad;
}

/* ---- per-expert RMSNorm before the weighted sum (a reading) ----------------
 *
 * [C] section 2.1 names a TP finalize that fuses the TP reduction, an RMSNorm
 * per expert and the weighted accumulation, straight from the GEMM2 result,
 * and gives no formula.  On one GPU the TP reduction is the identity; the
 * plainest reading is taken: each gathered expert row is RMS-normalised over
 * its own H columns with the shared gamma, and the normalised rows are summed
 * with the router weights.  No residual.
 *     n_j[h]    = E[r_j, h] / sqrt(mean_h(E[r_j, :]^2) + eps) * gamma[h]
 *     y[t, h]   = sum_j w[t, j] * n_j[h]            (slots j = 0..k-1 as stored)
 *     out[t, h] = BF16(y[t, h])
 * Everything in double, one rounding to BF16; a slot whose index lies outside
 * [0, R) contributes nothing and is counted.
 */

/* y (double [n, H]) of the tokens asked for; returns the bad-slot count. */
int64_t mfr_oracle_expert_rmsnorm_f64(int64_t T, int64_t H, int64_t k, int64_t R,
                                      const uint16_t* expert_out, const int32_t* idx,
                                      const float* w, const uint16_t* gamma, float eps,
                                      double* y, const int64_t* tokens, int64_t ntokens)
{
    int64_t bad = 0;
    int64_t n = tokens ? ntokens : T;
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = tokens ? tokens[i] : i;
        double* yr = y + i * H;
        bad += count_bad_slots(t, k, R, idx);
        for (int64_t h = 0; h < H; ++h)
            yr[h] = 0.0;
        for (int64_t j = 0; j < k; ++j) {
            int32_t r = idx[t * k + j];
            if (!slot_valid(r, R))
                continue;
            const uint16_t* row = expert_out + (int64_t)r * H;
            double ss = 0.0;
            for (int64_t h = 0; h < H; ++h) {
                double e = mfr_oracle_bf16_to_f64(row[h]);
                ss += e * e;
            }
            double inv = 1.0 / sqrt(ss / (double)H + (double)eps);
            double wj = (double)w[t * k + j];
            for (int64_t h = 0; h < H; ++h)
                yr[h] += wj * (mfr_oracle_bf16_to_f64(row[h]) * inv * mfr_oracle_bf16_to_f64(gamma[h]));
        }
    }
    return bad;
}

/* out = BF16(y) for the tokens asked for, one token at a time through an
 * H-double scratch row. */
int64_t mfr_oracle_finalize_expert_rmsnorm(int64_t T, int64_t H, int64_t k, int64_t R,
                                           const uint16_t* expert_out, const int32_t* idx,
                                           const float* w, const uint16_t* gamma, float eps,
                                           uint16_t* out, const int64_t* tokens, int64_t ntokens,
                                           double* y_scratch)
{
    int64_t bad = 0;
    int64_t n = tokens ? ntokens : T;
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = tokens ? tokens[i] : i;
        bad += mfr_oracle_expert_rmsnorm_f64(T, H, k, R, expert_out, idx, w, gamma, eps,
                                             y_scratch, &t, 1);
        for (int64_t h = 0; h < H; ++h)
            out[i * H + h] = mfr_oracle_bf16_from_f64(y_scratch[h]);
    }
    return bad;
}

/* ---- NVFP4 quantisation of the normalised output ---------------------------
 *
 * The PR 6544 analysis (section 2.3) names an RMSNorm + NVFP4 quantisation
 * fusion but not the format.  The format used here is the public NVFP4
 * description: 4-bit E2M1 elements (sign, 2 exponent bits with bias 1, 1
 * mantissa bit: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), one E4M3 scale per
 * block of 16 consecutive elements of a row, and one FP32 tensor scale s_enc
 * chosen by the caller.  For a block with elements y_i (FP32):
 *     amax = max |y_i|
 *     sf   = E4M3( (amax / 6) * s_enc )        nearest-even, saturating at 448
 *     dec  = value(sf) / s_enc                 (the block's decode scale)
 *     enc  = sf == 0 ? 0 : 1 / dec
 *     q_i  = E2M1( y_i * enc )                 nearest-even, saturating at 6
 * and y_i is recovered as value(q_i) * value(sf) / s_enc.  The divisions and
 * products are single FP32 operations, as the kernel performs them, so that
 * both sides take the integer decisions in the same precision.  Codes are
 * packed two per byte, element 2j in the low nibble of byte j.
 */

/* E4M3: bias 7, 3 mantissa bits, normal exponents -6..8, subnormal spacing
 * 2^-9, largest finite 448, no infinities.  Nearest-even; magnitudes above
 * 448 saturate to 448; NaN gives 0x7F. */
uint8_t mfr_oracle_e4m3_from_f64(double x)
{
    uint8_t sign = signbit(x) ? 0x80u : 0u;
    if (isnan(x))
        return 0x7Fu;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    if (isinf(a))                                    /* saturates like any large value */
        return (uint8_t)(sign | 0x7Eu);
    int e;
    (void)frexp(a, &e);
    int lead = e - 1;
    if (lead < -6)
        lead = -6;
    double spacing = ldexp(1.0, lead - 3);
    double r = nearbyint(a / spacing) * spacing;
    if (r > 448.0)
        r = 448.0;
    if (r == 0.0)
        return sign;
    (void)frexp(r, &e);
    lead = e - 1;
    if (lead < -6)                                   /* subnormal: units of 2^-9 */
        return (uint8_t)(sign | (uint8_t)(r / ldexp(1.0, -9)));
    int mant = (int)(r / ldexp(1.0, lead - 3)) - 8;  /* 0..7 */
    return (uint8_t)(sign | (uint8_t)(((lead + 7) << 3) | mant));
}

double mfr_oracle_e4m3_to_f64(uint8_t b)
{
    double s = (b & 0x80u) ? -1.0 : 1.0;
    int ef = (b >> 3) & 0xF, m = b & 7;
    if (ef == 0xF && m == 7)
        return NAN;
    if (ef == 0)
        return s * m * ldexp(1.0, -9);
    return s * (8 + m) * ldexp(1.0, ef - 7 - 3);
}

static const double k_e2m1_mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* E2M1: the nearest of the eight magnitudes; on a tie the code whose mantissa
 * bit is 0 (codes 0, 2, 4, 6); anything beyond 6 gives 6.  Sign in bit 3. */
uint8_t mfr_oracle_e2m1_from_f64(double x)
{
    uint8_t sign = signbit(x) ? 0x8u : 0u;
    if (isnan(x))
        return 0x7u;
    double a = fabs(x);
    int best = 0;
    for (int i = 1; i < 8; ++i) {
        double d = fabs(a - k_e2m1_mag[i]), db = fabs(a - k_e2m1_mag[best]);
        if (d < db || (d == db && (i & 1) == 0 && (best & 1) == 1))
            best = i;
    }
    return (uint8_t)(sign | best);
}

double mfr_oracle_e2m1_to_f64(uint8_t c)
{
    return ((c & 0x8u) ? -1.0 : 1.0) * k_e2m1_mag[c & 7];
}

/* The last three steps for one block of 16 elements whose scale is already
 * chosen, sv being the value of its E4M3 byte: dec = sv / s_enc, enc = 1 / dec
 * (0 for a zero scale), q_i = E2M1(y_i * enc), packed into 8 bytes. */
static void nvfp4_encode_block(const float* yb, float sv, float s_enc, uint8_t* qb)
{
    float dec = sv / s_enc;
    float enc = (sv == 0.0f) ? 0.0f : 1.0f / dec;
    for (int j = 0; j < 16; j += 2) {
        float p0 = yb[j] * enc, p1 = yb[j + 1] * enc;
        uint8_t c0 = mfr_oracle_e2m1_from_f64((double)p0);
        uint8_t c1 = mfr_oracle_e2m1_from_f64((double)p1);
        qb[j / 2] = (uint8_t)(c0 | (c1 << 4));
    }
}

/* Quantises n rows of width H (H a multiple of 16) as described above.
 * q_packed: n x H/2 bytes; sf: n x H/16 bytes. */
void mfr_oracle_nvfp4_quantize(int64_t n, int64_t H, const float* y, float s_enc,
                               uint8_t* q_packed, uint8_t* sf)
{
    for (int64_t i = 0; i < n; ++i) {
        for (int64_t b = 0; b < H / 16; ++b) {
            const float* yb = y + i * H + b * 16;
            float amax = 0.0f;
            for (int j = 0; j < 16; ++j)
                if (fabsf(yb[j]) > amax)
                    amax = fabsf(yb[j]);
            float v = (amax / 6.0f) * s_enc;
            uint8_t s8 = mfr_oracle_e4m3_from_f64((double)v);
            float sv = (float)mfr_oracle_e4m3_to_f64(s8);
            sf[i * (H / 16) + b] = s8;
            nvfp4_encode_block(yb, sv, s_enc, q_packed + i * (H / 2) + b * 8);
        }
    }
}

/* The codes of n rows of width H for block scales that the caller chooses
 * (sf: n x H/16 E4M3 bytes), by the same steps as mfr_oracle_nvfp4_quantize
 * after its scale choice.  Used to check an implementation whose scale
 * differs from the quantiser's only where the scale's own rounding decision
 * is ambiguous: its codes must then be those of its scale. */
void mfr_oracle_nvfp4_encode(int64_t n, int64_t H, const float* y, float s_enc,
                             const uint8_t* sf, uint8_t* q_packed)
{
    for (int64_t i = 0; i < n; ++i)
        for (int64_t b = 0; b < H / 16; ++b)
            nvfp4_encode_block(y + i * H + b * 16, (float)mfr_oracle_e4m3_to_f64(sf[i * (H / 16) + b]),
                               s_enc, q_packed + i * (H / 2) + b * 8);
}

/* The block scales of n rows (S scale bytes per row, one per 16 columns) in
 * the tiled layout that block-scaled FP4 GEMMs read, from the public
 * description of the 1-D block-scaling-factor layout: the scale matrix,
 * padded to a multiple of 128 rows and of 4 columns, is cut into tiles of
 * 128 rows x 4 columns, each stored as 512 consecutive bytes, tiles in
 * row-major order of (row / 128, column / 4); inside a tile, scale (r, c)
 * sits at byte (r mod 32) * 16 + ((r / 32) mod 4) * 4 + (c mod 4).  Bytes of
 * the padding are not written. */
void mfr_oracle_nvfp4_swizzle_scales(int64_t n, int64_t S, const uint8_t* sf, uint8_t* out)
{
    int64_t col_tiles = (S + 3) / 4;
    for (int64_t r = 0; r < n; ++r)
        for (int64_t c = 0; c < S; ++c) {
            int64_t tile = (r / 128) * col_tiles + c / 4;
            int64_t within = (r % 32) * 16 + ((r / 32) % 4) * 4 + (c % 4);
            out[tile * 512 + within] = sf[r * S + c];
        }
}

/* The whole path with the NVFP4 epilogue: the residual as above, RMSNorm in
 * double, the normalised value rounded once to FP32 (the precision the
 * quantiser works in), then quantised. */
int64_t mfr_oracle_finalize_residual_rmsnorm_nvfp4(
    int64_t T, int64_t H, int64_t k, int64_t R,
    const uint16_t* expert_out, const int32_t* idx, const float* w,
    const float* residual_in, const uint16_t* gamma, float eps, float s_enc,
    float* residual_out, uint8_t* q_packed, uint8_t* sf,
    const int64_t* tokens, int64_t ntokens, double* y_scratch, float* y32_scratch)
{
    int64_t bad = 0;
    int64_t n = tokens ? ntokens : T;
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = tokens ? tokens[i] : i;
        float* xr = residual_out + i * H;
        bad += mfr_oracle_weighted_residual(T, H, k, R, expert_out, idx, w, residual_in, xr, &t, 1);
        mfr_oracle_rmsnorm_f64(1, H, xr, gamma, eps, y_scratch);
        for (int64_t h = 0; h < H; ++h)
            y32_scratch[h] = (float)y_scratch[h];
        mfr_oracle_nvfp4_quantize(1, H, y32_scratch, s_enc, q_packed + i * (H / 2), sf + i * (H / 16));
    }
    return bad;
}

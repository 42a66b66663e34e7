/*
 * CPU oracle for hybrid-granularity FP8 quantization and the scaled GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file; only the test suite, the package's smoke check and the bench's
 * CPU-baseline / reference arm do.  It shares no code, header, table or
 * constant generator with the CUDA library.
 *
 * Everything is plain C99 in double precision (except the FP32-scale variant,
 * whose steps are single-precision operations by definition), written to be
 * checked by eye against the definitions it follows:
 *
 *  - "FP8 Formats for Deep Learning", abstract and core claim: the two FP8
 *    encodings E4M3 (4 exponent bits, 3 mantissa bits, no infinities, a single
 *    NaN mantissa pattern S.1111.111) and E5M2 (5 exponent bits, 2 mantissa
 *    bits, IEEE-754 special values); ordinary IEEE rounding (round to nearest,
 *    ties to even) applies ("Axiom & free-parameter ledger").
 *  - "A Comprehensive FP8 Training Recipe for Reasoning-Enhanced Language
 *    Models", "Core claim" and "What carries the argument": weights scaled per
 *    block, activations per token, each scale an exponent-only UE8M0 power of
 *    two rounded UP so that the scaled tensor never leaves the FP8 range.
 *  - "Characterization and Mitigation of Training Instabilities in
 *    Microscaling Formats", "What carries the argument": MX blocks share one
 *    power-of-two scale; a scaled magnitude beyond the element format's
 *    largest value is clamped to the largest code.
 *
 * Readings taken where the pages are silent:
 *  - block sizes: 128x128 weight blocks, 1x128 activation groups in the tiled
 *    variant, 32-element MX blocks (the recipe page says the block size is not
 *    reported);
 *  - UE8M0 (round-up) exponent: the smallest integer e with amax <= FMAX*2^e,
 *    clamped to [-127, 127]; amax = 0 gives -127;
 *  - MX exponent: floor(log2 amax) - emax, emax the exponent of the element
 *    format's largest normal (8 for E4M3, 15 for E5M2), clamped the same way;
 *  - a group holding a NaN or an infinity gets scale byte 0xFF (E8M0 NaN) and
 *    every code in it is 0x7F (a NaN in both encodings);
 *  - signed zero is kept: a negative value that rounds to zero encodes 0x80.
 *
 * All functions return 0 on success and a negative value on a bad argument.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#define ORC_E4M3 0
#define ORC_E5M2 1

#define ORC_GRAN_ROW 0
#define ORC_GRAN_1x128 1
#define ORC_GRAN_128x128 2
#define ORC_GRAN_MX32 3

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* Exact value of a BF16 bit pattern (1 sign, 8 exponent bits with bias 127,
 * 7 mantissa bits, IEEE-754 special values). */
double orc_bf16_to_double(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int ef = (bits >> 7) & 0xFF;
    int mf = bits & 0x7F;
    double v;
    if (ef == 0xFF) {
        v = (mf == 0) ? INFINITY : NAN;
    } else if (ef == 0) {
        v = ldexp((double)mf / 128.0, -126);          /* subnormal */
    } else {
        v = ldexp(1.0 + (double)mf / 128.0, ef - 127); /* normal */
    }
    return sign ? -v : v;
}

/* Exact value of an FP8 code, read field by field from the format
 * definitions.  E4M3: bias 7, exponent field 15 with mantissa 7 is the only
 * NaN, no infinities.  E5M2: bias 15, exponent field 31 is infinity (mantissa
 * 0) or NaN (mantissa != 0), as in IEEE-754. */
double orc_fp8_decode(uint8_t code, int fmt)
{
    int sign = (code >> 7) & 1;
    int ebits = (fmt == ORC_E4M3) ? 4 : 5;
    int mbits = 7 - ebits;
    int bias = (fmt == ORC_E4M3) ? 7 : 15;
    int emask = (1 << ebits) - 1;
    int mmask = (1 << mbits) - 1;
    int ef = (code >> mbits) & emask;
    int mf = code & mmask;
    double v;
    if (fmt == ORC_E4M3 && ef == emask && mf == mmask) {
        v = NAN;
    } else if (fmt == ORC_E5M2 && ef == emask) {
        v = (mf == 0) ? INFINITY : NAN;
    } else if (ef == 0) {
        v = ldexp((double)mf / (double)(1 << mbits), 1 - bias);
    } else {
        v = ldexp(1.0 + (double)mf / (double)(1 << mbits), ef - bias);
    }
    return sign ? -v : v;
}

/* The largest finite code of each format with the sign bit clear:
 * E4M3 0x7E (S.1111.110), E5M2 0x7B (S.11110.11). */
static int orc_max_code(int fmt) { return (fmt == ORC_E4M3) ? 0x7E : 0x7B; }

double orc_fp8_max(int fmt) { return orc_fp8_decode((uint8_t)orc_max_code(fmt), fmt); }

/* Round-to-nearest-even encode of an exact double.
 *
 * Written as the plain definition: among the finite non-negative codes
 * 0x00..max (whose values increase strictly with the code), pick the one
 * nearest to |y|; on an exact tie pick the code whose last mantissa bit is 0.
 * The sign bit is copied from y, so -0 and negative values that round to zero
 * give 0x80.
 *
 * Overflow (|y| beyond the largest finite value): with saturate != 0 the
 * result is the largest finite code (the MX clamp).  Without it, values that
 * round past the largest finite value give infinity (E5M2) or NaN (E4M3, which
 * has no infinity); values below that midpoint round down to the maximum as
 * usual.  A NaN input gives 0x7F. */
uint8_t orc_fp8_encode(double y, int fmt, int saturate)
{
    if (isnan(y)) return 0x7F;
    int neg = signbit(y) ? 1 : 0;
    double a = fabs(y);
    int maxc = orc_max_code(fmt);
    double vmax = orc_fp8_decode((uint8_t)maxc, fmt);
    uint8_t mag;
    if (a > vmax) {
        /* spacing of the top binade = vmax - value of the code just below */
        double ulp = vmax - orc_fp8_decode((uint8_t)(maxc - 1), fmt);
        double mid = vmax + ulp / 2.0;
        if (saturate || a < mid) {
            mag = (uint8_t)maxc;
        } else {
            mag = (fmt == ORC_E5M2) ? 0x7C : 0x7F; /* infinity / NaN */
        }
    } else {
        /* binary search: largest code lo with value(lo) <= a */
        int lo = 0, hi = maxc;
        while (lo < hi) {
            int mid = (lo + hi + 1) / 2;
            if (orc_fp8_decode((uint8_t)mid, fmt) <= a) lo = mid; else hi = mid - 1;
        }
        if (lo == maxc) {
            mag = (uint8_t)lo;
        } else {
            double vlo = orc_fp8_decode((uint8_t)lo, fmt);
            double vhi = orc_fp8_decode((uint8_t)(lo + 1), fmt);
            double dlo = a - vlo, dhi = vhi - a;
            if (dlo < dhi) mag = (uint8_t)lo;
            else if (dhi < dlo) mag = (uint8_t)(lo + 1);
            else mag = (lo % 2 == 0) ? (uint8_t)lo : (uint8_t)(lo + 1); /* tie: even */
        }
    }
    if (mag == 0x7F && fmt == ORC_E4M3) return 0x7F; /* NaN keeps one pattern */
    return (uint8_t)(mag | (neg << 7));
}

/* ------------------------------------------------------------------------ */
/* Scale exponents                                                           */
/* ------------------------------------------------------------------------ */

/* UE8M0 round-up rule: the smallest e in [-127, 127] with amax <= FMAX*2^e
 * (the scaled group then fits the FP8 range).  Returns 128 (byte 0xFF) for a
 * non-finite amax. */
int orc_ue8m0_exp(double amax, int fmt)
{
    if (!isfinite(amax)) return 128;
    double fmax = orc_fp8_max(fmt);
    int e = -127;
    while (e < 127 && amax > ldexp(fmax, e)) e++;
    return e;
}

/* MX rule: e = floor(log2 amax) - emax, clamped to [-127, 127]; emax is the
 * exponent of the element format's largest normal value.  frexp is exact:
 * amax = f*2^p with f in [0.5, 1), so floor(log2 amax) = p - 1. */
int orc_mx_exp(double amax, int fmt)
{
    if (!isfinite(amax)) return 128;
    int emax = (fmt == ORC_E4M3) ? 8 : 15;
    if (amax == 0.0) return -127;
    int p;
    (void)frexp(amax, &p);
    int e = (p - 1) - emax;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* ------------------------------------------------------------------------ */
/* Group quantization                                                        */
/* ------------------------------------------------------------------------ */

/* Quantize one group of n BF16 values whose elements sit at x[i*stride].
 * mx == 0: UE8M0 round-up scale, plain RNE cast (cannot overflow).
 * mx != 0: MX floor scale, saturating RNE cast.
 * Codes go to q[i*qstride]; the scale byte (e + 127, or 0xFF) is returned.
 * *nsat (if non-null) is increased by the number of elements whose scaled
 * magnitude exceeded the format's largest value (MX clamp events). */
static uint8_t orc_quant_group(const uint16_t *x, ptrdiff_t stride, int n, int fmt, int mx,
                               uint8_t *q, ptrdiff_t qstride, uint64_t *nsat)
{
    double amax = 0.0;
    int nonfinite = 0;
    for (int i = 0; i < n; i++) {
        double v = orc_bf16_to_double(x[i * stride]);
        if (!isfinite(v)) nonfinite = 1;
        else if (fabs(v) > amax) amax = fabs(v);
    }
    if (nonfinite) {
        for (int i = 0; i < n; i++) q[i * qstride] = 0x7F;
        return 0xFF;
    }
    int e = mx ? orc_mx_exp(amax, fmt) : orc_ue8m0_exp(amax, fmt);
    double fmax = orc_fp8_max(fmt);
    for (int i = 0; i < n; i++) {
        double y = ldexp(orc_bf16_to_double(x[i * stride]), -e); /* exact */
        if (nsat && fabs(y) > fmax) (*nsat)++;
        q[i * qstride] = orc_fp8_encode(y, fmt, mx);
    }
    return (uint8_t)(e + 127);
}

/* Activation quantizer, one scale per token or per 1x128 group.
 *   x     [rows, cols] BF16 bits, row stride ld_x (elements)
 *   group 0 = one scale per row (token); 128 = one per 128 consecutive columns
 *   transpose = 0: q [rows, cols] (ld_q), scale [rows, ngroups] (ld_s)
 *   transpose = 1: groups run along the rows (128 consecutive rows of one
 *                  column share a scale); output is written transposed:
 *                  q [cols, rows] (ld_q), scale [cols, rows/128] (ld_s). */
int orc_quant_token(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int group,
                    int transpose, int fmt, uint8_t *q, int64_t ld_q, uint8_t *scale, int64_t ld_s)
{
    if (rows < 0 || cols < 0 || (group != 0 && group != 128)) return -1;
    if (transpose && group != 128) return -1;
    if (!transpose) {
        int64_t g = group ? group : cols;
        if (g == 0 || cols % g) return -1;
        for (int64_t r = 0; r < rows; r++)
            for (int64_t c0 = 0; c0 < cols; c0 += g)
                scale[r * ld_s + c0 / g] = orc_quant_group(x + r * ld_x + c0, 1, (int)g, fmt, 0,
                                                           q + r * ld_q + c0, 1, NULL);
    } else {
        if (rows % 128) return -1;
        for (int64_t c = 0; c < cols; c++)
            for (int64_t r0 = 0; r0 < rows; r0 += 128)
                scale[c * ld_s + r0 / 128] = orc_quant_group(x + r0 * ld_x + c, ld_x, 128, fmt, 0,
                                                             q + c * ld_q + r0, 1, NULL);
    }
    return 0;
}

/* Weight quantizer, one scale per 128x128 block (block scale = the UE8M0
 * round-up of the block's amax).  scale [rows/128, cols/128] (ld_s).
 * If q_t is non-null the same codes are also written transposed,
 * q_t [cols, rows] (ld_qt), and the scale grid transposed into
 * scale_t [cols/128, rows/128] (ld_st). */
int orc_quant_block128(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                       uint8_t *q, int64_t ld_q, uint8_t *scale, int64_t ld_s,
                       uint8_t *q_t, int64_t ld_qt, uint8_t *scale_t, int64_t ld_st)
{
    if (rows % 128 || cols % 128) return -1;
    for (int64_t rb = 0; rb < rows / 128; rb++) {
        for (int64_t cb = 0; cb < cols / 128; cb++) {
            /* amax over the whole block before any cast */
            double amax = 0.0;
            int nonfinite = 0;
            for (int64_t r = 0; r < 128; r++)
                for (int64_t c = 0; c < 128; c++) {
                    double v = orc_bf16_to_double(x[(rb * 128 + r) * ld_x + cb * 128 + c]);
                    if (!isfinite(v)) nonfinite = 1;
                    else if (fabs(v) > amax) amax = fabs(v);
                }
            int e = nonfinite ? 128 : orc_ue8m0_exp(amax, fmt);
            for (int64_t r = 0; r < 128; r++)
                for (int64_t c = 0; c < 128; c++) {
                    int64_t gr = rb * 128 + r, gc = cb * 128 + c;
                    uint8_t code;
                    if (nonfinite) code = 0x7F;
                    else code = orc_fp8_encode(ldexp(orc_bf16_to_double(x[gr * ld_x + gc]), -e), fmt, 0);
                    q[gr * ld_q + gc] = code;
                    if (q_t) q_t[gc * ld_qt + gr] = code;
                }
            scale[rb * ld_s + cb] = (uint8_t)(e + 127);
            if (scale_t) scale_t[cb * ld_st + rb] = (uint8_t)(e + 127);
        }
    }
    return 0;
}

/* MXFP8 quantizer: one shared E8M0 scale per 32 consecutive elements of a row,
 * saturating cast.  scale [rows, cols/32] (ld_s).  *clamp_count (if non-null)
 * receives the number of elements clamped to the largest code because their
 * scaled magnitude exceeded it. */
int orc_quant_mx32(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                   uint8_t *q, int64_t ld_q, uint8_t *scale, int64_t ld_s, uint64_t *clamp_count)
{
    if (cols % 32) return -1;
    uint64_t nsat = 0;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c0 = 0; c0 < cols; c0 += 32)
            scale[r * ld_s + c0 / 32] = orc_quant_group(x + r * ld_x + c0, 1, 32, fmt, 1,
                                                        q + r * ld_q + c0, 1, &nsat);
    if (clamp_count) *clamp_count = nsat;
    return 0;
}

/* MX clamp monitor.  "Characterization and Mitigation of Training
 * Instabilities in Microscaling Formats" proposes watching how many values
 * are clamped into the last quantization bin, and how many blocks are, as an
 * early warning of divergence ("What would settle it", "If this is right"),
 * and names the collapse of a tightly clustered block onto one bin as the
 * mechanism ("What carries the argument").  This quantizes exactly as
 * orc_quant_mx32 (same q and scale) and counts, over the whole tensor:
 *   stats[0]  elements whose scaled magnitude exceeded the format's largest
 *             value (saturated: written as the largest code)
 *   stats[1]  elements whose code has the largest finite magnitude (the last
 *             bin), saturated or rounded there
 *   stats[2]  blocks holding at least one saturated element
 *   stats[3]  blocks whose 32 codes are all the same byte (same-bin collapse);
 *             blocks of zeros and blocks holding a non-finite value excluded
 * row_sat[r] (if non-null) = saturated elements in row r. */
int orc_mx32_monitor(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                     uint8_t *q, int64_t ld_q, uint8_t *scale, int64_t ld_s, uint64_t *stats,
                     uint64_t *row_sat)
{
    if (cols % 32 || !stats) return -1;
    const uint8_t top = orc_fp8_encode(orc_fp8_max(fmt), fmt, 1);
    for (int i = 0; i < 4; i++) stats[i] = 0;
    for (int64_t r = 0; r < rows; r++) {
        uint64_t rs = 0;
        for (int64_t c0 = 0; c0 < cols; c0 += 32) {
            const uint16_t *xb = x + r * ld_x + c0;
            uint8_t *qb = q + r * ld_q + c0;
            uint64_t nsat = 0;
            uint8_t sb = orc_quant_group(xb, 1, 32, fmt, 1, qb, 1, &nsat);
            scale[r * ld_s + c0 / 32] = sb;
            int allzero = 1, same = 1;
            for (int i = 0; i < 32; i++) {
                if (orc_bf16_to_double(xb[i]) != 0.0) allzero = 0;
                if (qb[i] != qb[0]) same = 0;
                if ((qb[i] & 0x7F) == top) stats[1]++;
            }
            stats[0] += nsat;
            rs += nsat;
            if (nsat) stats[2]++;
            if (same && !allzero && sb != 0xFF) stats[3]++;
        }
        if (row_sat) row_sat[r] = rs;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* FP32-scale variant                                                        */
/* ------------------------------------------------------------------------ */

/* "A Comprehensive FP8 Training Recipe ..." compares its UE8M0 recipe with
 * an "FP8 w. FP32 scale" arm that its setup does not define (referee
 * comments).  The reading taken here is the ordinary FP32 scaling of FP8
 * recipes, at the same granularities: per group,
 *   d = fl32(amax / FMAX)      the stored FP32 scale (x ~ decode(q) * d)
 *   m = fl32(FMAX / amax)      the multiplier applied before the cast
 *   q = RNE_sat(fl32(x * m))   saturating nearest-even FP8 encoding
 * with amax = 0 giving d = m = 1, and a NaN or infinity in the group giving
 * d = NaN and codes 0x7F.  Every step is one IEEE single-precision operation
 * (the oracle is built with contraction off), so the CUDA path reaches the
 * same bits. */
static float orc_quant_group_f32(const uint16_t *x, ptrdiff_t stride, int n, int fmt,
                                 uint8_t *q, ptrdiff_t qstride)
{
    double amax = 0.0;
    int nonfinite = 0;
    for (int i = 0; i < n; i++) {
        double v = orc_bf16_to_double(x[i * stride]);
        if (!isfinite(v)) nonfinite = 1;
        else if (fabs(v) > amax) amax = fabs(v);
    }
    if (nonfinite) {
        for (int i = 0; i < n; i++) q[i * qstride] = 0x7F;
        return NAN;
    }
    const float fmax = (float)orc_fp8_max(fmt);
    const float a = (float)amax;                 /* exact: BF16 values are FP32 values */
    const float d = (a == 0.0f) ? 1.0f : a / fmax;
    const float m = (a == 0.0f) ? 1.0f : fmax / a;
    for (int i = 0; i < n; i++) {
        const float xf = (float)orc_bf16_to_double(x[i * stride]);
        const float y = xf * m;
        q[i * qstride] = orc_fp8_encode((double)y, fmt, 1);
    }
    return d;
}

/* Per-token (group 0) or 1x128 (group 128) quantization with FP32 scales:
 * q [rows, cols] (ld_q), scale [rows, ngroups] floats (ld_s floats). */
int orc_quant_token_f32s(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int group,
                         int fmt, uint8_t *q, int64_t ld_q, float *scale, int64_t ld_s)
{
    if (rows < 0 || cols < 0 || (group != 0 && group != 128)) return -1;
    int64_t g = group ? group : cols;
    if (g == 0 || cols % g) return -1;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c0 = 0; c0 < cols; c0 += g)
            scale[r * ld_s + c0 / g] = orc_quant_group_f32(x + r * ld_x + c0, 1, (int)g, fmt,
                                                           q + r * ld_q + c0, 1);
    return 0;
}

/* 128x128-block quantization with FP32 scales (block amax over the whole
 * block); optional transposed copy of the codes and the scale grid. */
int orc_quant_block128_f32s(const uint16_t *x, int64_t rows, int64_t cols, int64_t ld_x, int fmt,
                            uint8_t *q, int64_t ld_q, float *scale, int64_t ld_s,
                            uint8_t *q_t, int64_t ld_qt, float *scale_t, int64_t ld_st)
{
    if (rows % 128 || cols % 128) return -1;
    uint8_t blk[128 * 128];
    uint16_t tmp[128 * 128];
    for (int64_t rb = 0; rb < rows / 128; rb++) {
        for (int64_t cb = 0; cb < cols / 128; cb++) {
            /* the block as one group of 16384 elements, row-major */
            for (int r = 0; r < 128; r++)
                for (int c = 0; c < 128; c++)
                    tmp[r * 128 + c] = x[(rb * 128 + r) * ld_x + cb * 128 + c];
            float d = orc_quant_group_f32(tmp, 1, 128 * 128, fmt, blk, 1);
            scale[rb * ld_s + cb] = d;
            for (int r = 0; r < 128; r++)
                for (int c = 0; c < 128; c++) {
                    q[(rb * 128 + r) * ld_q + cb * 128 + c] = blk[r * 128 + c];
                    if (q_t) q_t[(cb * 128 + c) * ld_qt + rb * 128 + r] = blk[r * 128 + c];
                }
            if (scale_t) scale_t[cb * ld_st + rb] = d;
        }
    }
    return 0;
}

/* x_hat = decode(q) * d for an operand with FP32 scales (ROW, 1x128 or
 * 128x128 layout as in orc_dequant); out [rows, k] dense. */
int orc_dequant_f32s(const uint8_t *q, int64_t ld_q, const float *scale, int64_t ld_s, int gran,
                     int fmt, int64_t rows, int64_t k, double *out)
{
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < k; c++) {
            float d;
            switch (gran) {
            case ORC_GRAN_ROW: d = scale[r * ld_s]; break;
            case ORC_GRAN_1x128: d = scale[r * ld_s + c / 128]; break;
            case ORC_GRAN_128x128: d = scale[(r / 128) * ld_s + c / 128]; break;
            default: return -1;
            }
            out[r * k + c] = orc_fp8_decode(q[r * ld_q + c], fmt) * (double)d;
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Dequantization and the reference GEMM                                     */
/* ------------------------------------------------------------------------ */

/* Scale byte that applies to element (r, k) of a K-contiguous operand. */
static uint8_t orc_scale_at(const uint8_t *scale, int64_t ld_s, int gran, int64_t r, int64_t k)
{
    switch (gran) {
    case ORC_GRAN_ROW: return scale[r * ld_s];
    case ORC_GRAN_1x128: return scale[r * ld_s + k / 128];
    case ORC_GRAN_128x128: return scale[(r / 128) * ld_s + k / 128];
    default: return scale[r * ld_s + k / 32];
    }
}

/* x_hat = decode(q) * 2^(byte - 127); byte 0xFF (E8M0 NaN) gives NaN. */
static double orc_dequant_at(const uint8_t *q, int64_t ld_q, const uint8_t *scale, int64_t ld_s,
                             int gran, int fmt, int64_t r, int64_t k)
{
    uint8_t sb = orc_scale_at(scale, ld_s, gran, r, k);
    if (sb == 0xFF) return NAN;
    return ldexp(orc_fp8_decode(q[r * ld_q + k], fmt), (int)sb - 127);
}

/* Dequantize a whole K-contiguous operand to doubles, out [rows, k] dense. */
int orc_dequant(const uint8_t *q, int64_t ld_q, const uint8_t *scale, int64_t ld_s, int gran,
                int fmt, int64_t rows, int64_t k, double *out)
{
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < k; c++)
            out[r * k + c] = orc_dequant_at(q, ld_q, scale, ld_s, gran, fmt, r, c);
    return 0;
}

/* Re-quantization of stored FP8 activations for the weight-gradient GEMM.
 * The recipe keeps activations in FP8 and quantizes every GEMM operand with
 * fine-grained power-of-two scales ("A Comprehensive FP8 Training Recipe
 * ...", "What carries the argument"); the weight gradient contracts over
 * tokens, so its operands need groups that run along the tokens.  Here the
 * source is the stored operand itself: q [rows = tokens, cols] K-contiguous
 * with per-token (ROW) or 1x128-along-K scales.  Every element is
 * dequantized exactly, x_hat = decode(q) * 2^(byte - 127), and x_hat is
 * quantized again with 1x128 groups along the tokens (UE8M0 round-up, RNE,
 * format fmt_out), written transposed:
 *   q_t [cols, rows] (ld_qt), scale_t [cols, rows/128] (ld_st).
 * A token whose scale byte is 0xFF, or a NaN / infinite code, makes its
 * output group non-finite (scale 0xFF, codes 0x7F). */
int orc_requant_t(const uint8_t *q, int64_t rows, int64_t cols, int64_t ld_q,
                  const uint8_t *scale, int64_t ld_s, int gran, int fmt_in, int fmt_out,
                  uint8_t *q_t, int64_t ld_qt, uint8_t *scale_t, int64_t ld_st)
{
    if (rows % 128 || (gran != ORC_GRAN_ROW && gran != ORC_GRAN_1x128)) return -1;
    if (gran == ORC_GRAN_1x128 && cols % 128) return -1;
    double v[128];
    for (int64_t c = 0; c < cols; c++) {
        for (int64_t r0 = 0; r0 < rows; r0 += 128) {
            double amax = 0.0;
            int nonfinite = 0;
            for (int i = 0; i < 128; i++) {
                v[i] = orc_dequant_at(q, ld_q, scale, ld_s, gran, fmt_in, r0 + i, c);
                if (!isfinite(v[i])) nonfinite = 1;
                else if (fabs(v[i]) > amax) amax = fabs(v[i]);
            }
            uint8_t *out = q_t + c * ld_qt + r0;
            if (nonfinite) {
                for (int i = 0; i < 128; i++) out[i] = 0x7F;
                scale_t[c * ld_st + r0 / 128] = 0xFF;
                continue;
            }
            int e = orc_ue8m0_exp(amax, fmt_out);
            for (int i = 0; i < 128; i++) out[i] = orc_fp8_encode(ldexp(v[i], -e), fmt_out, 0);
            scale_t[c * ld_st + r0 / 128] = (uint8_t)(e + 127);
        }
    }
    return 0;
}

/* Reference scaled GEMM at chosen output positions:
 *   C_ref[i,j] = sum_k a_hat[i,k] * b_hat[j,k]        (fp64)
 *   S[i,j]     = sum_k |a_hat[i,k] * b_hat[j,k]|      (the tolerance scale)
 * for the n pairs (ii[t], jj[t]).  A is [M, K] and B is [N, K], both
 * K-contiguous FP8 codes with their scale grids, dequantized on the fly.  The
 * operation C = A * B^T with both operands K-contiguous is the common form of
 * fprop, dgrad and wgrad once the operands are quantized. */
int orc_gemm_ref_pairs(const uint8_t *qa, int64_t ld_a, const uint8_t *sa, int64_t ld_sa, int gran_a,
                       int fmt_a, const uint8_t *qb, int64_t ld_b, const uint8_t *sb, int64_t ld_sb,
                       int gran_b, int fmt_b, int64_t K, const int64_t *ii, const int64_t *jj,
                       int64_t n, double *c_ref, double *s_abs)
{
    for (int64_t t = 0; t < n; t++) {
        double acc = 0.0, sabs = 0.0;
        for (int64_t k = 0; k < K; k++) {
            double p = orc_dequant_at(qa, ld_a, sa, ld_sa, gran_a, fmt_a, ii[t], k) *
                       orc_dequant_at(qb, ld_b, sb, ld_sb, gran_b, fmt_b, jj[t], k);
            acc += p;
            sabs += fabs(p);
        }
        c_ref[t] = acc;
        s_abs[t] = sabs;
    }
    return 0;
}

/* Full reference product of dense double operands: a [M, K], b [N, K];
 * c [M, N] and s [M, N] as above. */
int orc_gemm_ref_dense(const double *a, const double *b, int64_t M, int64_t N, int64_t K,
                       double *c, double *s)
{
    for (int64_t i = 0; i < M; i++)
        for (int64_t j = 0; j < N; j++) {
            double acc = 0.0, sabs = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double p = a[i * K + k] * b[j * K + k];
                acc += p;
                sabs += fabs(p);
            }
            c[i * N + j] = acc;
            s[i * N + j] = sabs;
        }
    return 0;
}

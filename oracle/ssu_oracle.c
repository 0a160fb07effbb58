/*
 * ssu_oracle.c -- plain, slow, double-precision CPU definition of the Mamba-2
 * selective state update (SSU).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker the CUDA path is compared
 * against.  Only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark load it; the library under test never does, and the two share no
 * code, header, table or helper.
 *
 * What it follows (page "Mamba / SSU" of the MATE documentation, unless noted):
 *   - Intro paragraph: Mamba-2 keeps ONE decay per head, A[h].
 *   - "SSU at a glance", rows State, A / D / dt_bias, B / C, Output,
 *     dt_softplus: shapes, per-head fp32 parameters, heads divisible by groups.
 *   - "SSU toolchain requirements": the recurrence runs in (at least) fp32 and
 *     the state is stored back in the state dtype.  Here it runs in double and
 *     is rounded to nearest-even only when stored.
 *   - "SSU at a glance", rows Slot semantics and Variable-length and MTP
 *     decode: slot tables addressed by strides, pad slots read as a zero state
 *     and are never written, disable_state_update leaves the pool unchanged,
 *     the read slot is seeded at max(num_accepted - 1, 0), every token
 *     publishes its state to its own destination entry (or its own read-table
 *     entry when no destination table is given), empty sequences are skipped.
 *   - Article "ReplaySSM: Cache SSM Inputs, Not State" (lpnh.cn), section
 *     三个瓶颈: S_t = alpha_t * S_{t-1} + Delta_t * v_t k_t^T, y_t = S_t q_t,
 *     i.e. y is read from the UPDATED state; v = x, k = B, q = C,
 *     alpha = exp(A * dt').
 *   - The task's formula order: dt' = softplus(dt + dt_bias) (optional),
 *     dA = exp(A[h] dt'), state = state*dA + dt'*x*B, y = state.C + D*x,
 *     optional y *= silu(z).
 *
 * Readings taken where the pages are silent:
 *   - head -> group map: contiguous blocks, g = h / (heads / groups).  PARITY
 *     UNPINNED by the pages (they only require divisibility).
 *   - no table at all: sequence b uses slot b for reading and writing.
 *   - SLOTS_PER_ROW mode: entry = cu_seqlens[b] + t ("one entry per packed
 *     row").  SLOTS_STRIDED mode: entry = b*s0 + t*s1 (page-literal).
 *   - inputs in which one sequence writes a slot that another sequence reads
 *     or writes have no deterministic answer; the oracle refuses them
 *     (return code 2) instead of defining them.
 *   - softplus is log(1 + e^v), evaluated as max(v,0) + log1p(exp(-|v|)).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "ssu_oracle.h"

/* ------------------------------------------------------------------------ */
/* Exact decoding of the stored formats into double.                        */
/* ------------------------------------------------------------------------ */

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double half_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);              /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 1024), e - 25);  /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void *base, int64_t i, int dtype)
{
    switch (dtype) {
    case ORC_F32: return (double)((const float *)base)[i];
    case ORC_F16: return half_bits_to_double(((const uint16_t *)base)[i]);
    case ORC_BF16: return bf16_bits_to_double(((const uint16_t *)base)[i]);
    case ORC_F64: return ((const double *)base)[i];
    }
    return NAN;
}

/* ------------------------------------------------------------------------ */
/* Round-to-nearest-even from double into a narrower binary format.        */
/* frac_bits: stored fraction bits; emin: exponent of the smallest normal;  */
/* emax: exponent of the largest finite value.                              */
/* ------------------------------------------------------------------------ */
static double round_to_format(double v, int frac_bits, int emin, int emax)
{
    if (v == 0.0 || isnan(v) || isinf(v))
        return v;
    int e2;
    frexp(v, &e2);                 /* |v| = m * 2^e2, 0.5 <= m < 1 */
    int lead = e2 - 1;             /* exponent of the leading bit   */
    if (lead < emin)
        lead = emin;               /* subnormal range: fixed quantum */
    double quantum = ldexp(1.0, lead - frac_bits);
    /* v / quantum is exact (division by a power of two); nearbyint rounds to
     * nearest, ties to even, in the default rounding mode. */
    double r = nearbyint(v / quantum) * quantum;
    double maxfinite = ldexp(2.0 - ldexp(1.0, -frac_bits), emax);
    if (fabs(r) > maxfinite)
        return v > 0 ? INFINITY : -INFINITY;
    return r;
}

static uint16_t double_to_half_bits(double v)
{
    double r = round_to_format(v, 10, -14, 15);
    uint16_t sign = signbit(r) ? 0x8000 : 0;
    double a = fabs(r);
    if (isnan(r)) return 0x7e00;
    if (isinf(r)) return sign | 0x7c00;
    if (a == 0.0) return sign;
    if (a < ldexp(1.0, -14))                       /* subnormal */
        return sign | (uint16_t)(a / ldexp(1.0, -24));
    int e2;
    double m = frexp(a, &e2);                      /* a = m 2^e2, m in [0.5,1) */
    int biased = (e2 - 1) + 15;
    uint16_t frac = (uint16_t)((m * 2.0 - 1.0) * 1024.0);
    return sign | (uint16_t)(biased << 10) | frac;
}

static uint16_t double_to_bf16_bits(double v)
{
    if (isnan(v)) return 0x7fc0;
    double r = round_to_format(v, 7, -126, 127);
    float f = (float)r;                            /* exact: r fits in 8 bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

static void store_elem(void *base, int64_t i, int dtype, double v)
{
    switch (dtype) {
    case ORC_F32: ((float *)base)[i] = (float)round_to_format(v, 23, -126, 127); break;
    case ORC_F16: ((uint16_t *)base)[i] = double_to_half_bits(v); break;
    case ORC_BF16: ((uint16_t *)base)[i] = double_to_bf16_bits(v); break;
    case ORC_F64: ((double *)base)[i] = v; break;
    }
}

/* Exposed so the tests can check the conversions against known encodings. */
double orc_decode(uint32_t bits, int dtype)
{
    if (dtype == ORC_F32) {
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    if (dtype != ORC_F16 && dtype != ORC_BF16)
        return 0.0; /* 64-bit values do not fit the 32 bits */
    const uint16_t h = (uint16_t)bits;
    return load_elem(&h, 0, dtype);
}

uint32_t orc_encode(double v, int dtype)
{
    if (dtype == ORC_F32) {
        float f = (float)round_to_format(v, 23, -126, 127);
        uint32_t u;
        memcpy(&u, &f, sizeof u);
        return u;
    }
    if (dtype == ORC_F16) return double_to_half_bits(v);
    return double_to_bf16_bits(v);
}

/* ------------------------------------------------------------------------ */
/* The low-precision read copy (ReplaySSM, 低精度读写分离).                 */
/* ------------------------------------------------------------------------ */

/* OCP FP8 E4M3: 1 sign, 4 exponent bits (bias 7), 3 fraction bits; exponent
 * field 0 holds subnormals f * 2^-9; S.1111.111 is NaN, so the largest finite
 * value is 1.75 * 2^8 = 448 and there are no infinities. */
double orc_e4m3_decode(uint8_t code)
{
    int sign = code >> 7;
    int e = (code >> 3) & 0xf;
    int f = code & 7;
    double v;
    if (e == 15 && f == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)f, -9);
    else
        v = ldexp((double)(f + 8), e - 10);  /* (1 + f/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* Round to nearest even onto the E4M3 grid, values past the largest finite
 * one clamped to +-448 ("saturate to finite").  NaN maps to the NaN code. */
uint8_t orc_e4m3_encode(double v)
{
    if (isnan(v))
        return 0x7f;
    uint8_t sign = signbit(v) ? 0x80 : 0;
    double r = fabs(round_to_format(v, 3, -6, 8));
    if (isinf(r) || r > 448.0)
        r = 448.0;
    if (r == 0.0)
        return sign;
    if (r < ldexp(1.0, -6))                     /* subnormal: r = f * 2^-9 */
        return sign | (uint8_t)(r / ldexp(1.0, -9));
    int e2;
    double m = frexp(r, &e2);                   /* r = m 2^e2, m in [0.5, 1) */
    int biased = (e2 - 1) + 7;
    uint8_t frac = (uint8_t)((m * 2.0 - 1.0) * 8.0);
    return sign | (uint8_t)(biased << 3) | frac;
}

/* FP4 E2M1: 1 sign, 2 exponent bits (bias 1), 1 fraction bit; exponent
 * field 0 holds the subnormal 0.5; no infinities and no NaN, so the
 * magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4 and 6 (codes 0-7, bit 3 the sign). */
double orc_e2m1_decode(uint8_t code)
{
    const int e = (code >> 1) & 3, f = code & 1;
    const double v = e == 0 ? 0.5 * f : ldexp(1.0 + 0.5 * f, e - 1);
    return (code & 8) ? -v : v;
}

/* Round to nearest even onto the E2M1 grid, magnitudes past 6 clamped to 6
 * ("saturate to finite"); NaN, which the format cannot hold, maps to +6. */
uint8_t orc_e2m1_encode(double v)
{
    if (isnan(v))
        return 7;
    const uint8_t sign = signbit(v) ? 8 : 0;
    double r = fabs(round_to_format(v, 1, 0, 2));
    if (isinf(r) || r > 6.0)
        r = 6.0;
    for (uint8_t code = 0; code < 8; ++code)
        if (orc_e2m1_decode(code) == r)
            return sign | code;
    return sign; /* not reached: every rounded magnitude is on the grid */
}

/* Floats of one row's NVFP4 scale record: the fp32 row scale, then the
 * dstate / 16 E4M3 block scale codes, padded to a multiple of 16 bytes. */
int64_t orc_nvfp4_scale_words(int64_t dstate) { return (4 + dstate / 16 + 15) / 16 * 4; }

/* One state row into its read copy (format per orc_shadow_refresh).  The
 * E4M3 form maps the row's largest magnitude amax onto the largest finite
 * E4M3 value, 448: each value v is stored as the code of v * 448 / amax
 * (the quotient in double, then rounded to nearest even onto the E4M3
 * grid), and the row keeps the scale amax / 448 in fp32 (the type it is
 * stored in), so that code * scale gives v back.  An all-zero row keeps
 * zero codes and the scale 1. */
static void shadow_row(const double *v, int64_t n, int32_t format, void *codes, float *scale)
{
    if (format == ORC_SHADOW_F16) {
        for (int64_t i = 0; i < n; ++i)
            ((uint16_t *)codes)[i] = double_to_half_bits(v[i]);
        return;
    }
    if (format == ORC_SHADOW_NVFP4) {
        /* Two scale levels, as NVFP4 defines them: the row's largest magnitude
         * amax maps onto 6 * 448, the product of the largest E2M1 and E4M3
         * values, through the fp32 row scale s = amax / (6 * 448); each block
         * of 16 elements keeps the E4M3 code of (its largest magnitude) /
         * (6 s), which maps the block's largest onto 6; an element is the E2M1
         * code of v / (block scale * s), quotients in double, both roundings
         * to nearest even.  An all-zero row keeps s = 1 and zero codes; a block
         * whose scale rounds to zero keeps zero codes. */
        double amax = 0.0;
        for (int64_t i = 0; i < n; ++i)
            if (fabs(v[i]) > amax)
                amax = fabs(v[i]);
        const float s = amax > 0.0 ? (float)round_to_format(amax / (6.0 * 448.0), 23, -126, 127) : 1.0f;
        scale[0] = s;
        uint8_t *bcodes = (uint8_t *)(scale + 1);
        uint8_t *out = (uint8_t *)codes;
        for (int64_t k = 0; k < n / 16; ++k) {
            double bmax = 0.0;
            for (int64_t i = 16 * k; i < 16 * k + 16; ++i)
                if (fabs(v[i]) > bmax)
                    bmax = fabs(v[i]);
            bcodes[k] = orc_e4m3_encode(bmax / (6.0 * (double)s));
            const double bs = orc_e4m3_decode(bcodes[k]);
            for (int64_t i = 16 * k; i < 16 * k + 16; ++i) {
                const uint8_t c = bs > 0.0 ? orc_e2m1_encode(v[i] / (bs * (double)s)) : 0;
                if (i % 2 == 0)
                    out[i / 2] = c;
                else
                    out[i / 2] |= (uint8_t)(c << 4);
            }
        }
        return;
    }
    double amax = 0.0;
    for (int64_t i = 0; i < n; ++i)
        if (fabs(v[i]) > amax)
            amax = fabs(v[i]);
    *scale = amax > 0.0 ? (float)round_to_format(amax / 448.0, 23, -126, 127) : 1.0f;
    for (int64_t i = 0; i < n; ++i)
        ((uint8_t *)codes)[i] = orc_e4m3_encode(amax > 0.0 ? v[i] * 448.0 / amax : v[i]);
}

static double shadow_value(const void *codes, const float *scale, int64_t row, int64_t n, int64_t i, int32_t format)
{
    if (format == ORC_SHADOW_F16)
        return half_bits_to_double(((const uint16_t *)codes)[row * n + i]);
    if (format == ORC_SHADOW_NVFP4) {
        const float *rec = scale + row * orc_nvfp4_scale_words(n);
        const uint8_t byte = ((const uint8_t *)codes)[(row * n + i) / 2];
        const uint8_t c = i % 2 == 0 ? (byte & 15) : (byte >> 4);
        return orc_e2m1_decode(c) * orc_e4m3_decode(((const uint8_t *)(rec + 1))[i / 16]) * (double)rec[0];
    }
    return orc_e4m3_decode(((const uint8_t *)codes)[row * n + i]) * (double)scale[row];
}

/* Byte offset of row `row`'s codes and float offset of its scales. */
static size_t shadow_code_offset(int64_t row, int64_t n, int32_t format)
{
    return format == ORC_SHADOW_F16 ? (size_t)(row * n) * 2 : format == ORC_SHADOW_NVFP4 ? (size_t)(row * n) / 2 : (size_t)(row * n);
}
static int64_t shadow_scale_offset(int64_t row, int64_t n, int32_t format)
{
    return format == ORC_SHADOW_NVFP4 ? row * orc_nvfp4_scale_words(n) : row;
}

int orc_shadow_refresh(const void *state, int32_t state_dtype, int64_t rows, int64_t dstate, int32_t format,
                       void *shadow, float *scale)
{
    if (format != ORC_SHADOW_F16 && format != ORC_SHADOW_E4M3 && format != ORC_SHADOW_NVFP4)
        return ORC_INVALID;
    if (format != ORC_SHADOW_F16 && scale == NULL)
        return ORC_INVALID;
    if (format == ORC_SHADOW_NVFP4 && dstate % 16 != 0)
        return ORC_INVALID;
    double *v = malloc(sizeof(double) * (size_t)dstate);
    if (!v)
        return ORC_INVALID;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t i = 0; i < dstate; ++i)
            v[i] = load_elem(state, r * dstate + i, state_dtype);
        shadow_row(v, dstate, format, (char *)shadow + shadow_code_offset(r, dstate, format),
                   scale ? scale + shadow_scale_offset(r, dstate, format) : NULL);
    }
    free(v);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Scalar functions of the method.                                          */
/* ------------------------------------------------------------------------ */

/* softplus(v) = log(1 + e^v), in a form that neither overflows nor cancels. */
double orc_softplus(double v)
{
    return fmax(v, 0.0) + log1p(exp(-fabs(v)));
}

/* silu(z) = z * sigmoid(z) = z / (1 + e^-z). */
double orc_silu(double z)
{
    return z / (1.0 + exp(-z));
}

/* ------------------------------------------------------------------------ */
/* Slot resolution ("Slot semantics" row).                                  */
/* ------------------------------------------------------------------------ */

static int64_t table_entry(const orc_table *t, int64_t b, int64_t step, int64_t row_start)
{
    if (t->mode == ORC_SLOTS_PER_ROW)
        return row_start + step;
    return b * t->s0 + step * t->s1;
}

/* Slot read or written by (sequence b, step) through table t.  Writes the
 * slot to *slot, returns 0, or returns -1 when the entry is outside the
 * table.  A NULL table means "no table": slot b. */
static int resolve(const orc_table *t, int64_t b, int64_t step, int64_t row_start, int64_t *slot)
{
    if (t == NULL || t->entries == NULL) {
        *slot = b;
        return 0;
    }
    int64_t e = table_entry(t, b, step, row_start);
    if (e < 0 || e >= t->extent)
        return -1;
    *slot = t->entries[e];
    return 0;
}

static void set_err(char *err, int errlen, const char *msg, int64_t a, int64_t b)
{
    if (err && errlen > 0)
        snprintf(err, (size_t)errlen, msg, (long long)a, (long long)b);
}

/* ------------------------------------------------------------------------ */
/* The update.                                                              */
/* ------------------------------------------------------------------------ */

int orc_ssu_run(const orc_problem *pr, char *err, int errlen)
{
    const int64_t H = pr->heads, P = pr->dim, N = pr->dstate, G = pr->groups;
    if (H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G != 0) {
        set_err(err, errlen, "bad shape: heads=%lld groups=%lld", H, G);
        return ORC_INVALID;
    }
    const int64_t heads_per_group = H / G;
    const int64_t nseq = pr->nseq;
    const orc_table *rtab = (pr->read.entries != NULL) ? &pr->read : NULL;
    const orc_table *wtab = (pr->dst.entries != NULL) ? &pr->dst : rtab;

    /* Sequence extents.  With no cu_seqlens, sequence b is row b, length 1. */
    int64_t *start = malloc(sizeof(int64_t) * (size_t)(nseq + 1));
    if (!start) return ORC_INVALID;
    for (int64_t b = 0; b <= nseq; ++b)
        start[b] = pr->cu_seqlens ? pr->cu_seqlens[b] : b;
    if (start[0] != 0 || start[nseq] != pr->rows) {
        set_err(err, errlen, "cu_seqlens must start at 0 and end at rows (%lld, got %lld)",
                pr->rows, start[nseq]);
        free(start);
        return ORC_INVALID;
    }
    for (int64_t b = 0; b < nseq; ++b) {
        if (start[b + 1] < start[b]) {
            set_err(err, errlen, "cu_seqlens decreases at sequence %lld%lld", b, 0);
            free(start);
            return ORC_INVALID;
        }
    }

    /* Resolve every slot first and check it. */
    int64_t *seed = malloc(sizeof(int64_t) * (size_t)(nseq > 0 ? nseq : 1));
    int64_t *wslot = malloc(sizeof(int64_t) * (size_t)(pr->rows > 0 ? pr->rows : 1));
    int64_t *writer = malloc(sizeof(int64_t) * (size_t)pr->slots);
    if (!seed || !wslot || !writer) {
        free(start); free(seed); free(wslot); free(writer);
        return ORC_INVALID;
    }
    int rc = ORC_OK;
    for (int64_t s = 0; s < pr->slots; ++s)
        writer[s] = -1;
    for (int64_t b = 0; b < nseq && rc == ORC_OK; ++b) {
        int64_t len = start[b + 1] - start[b];
        if (len == 0) {
            seed[b] = pr->pad_slot_id;
            continue;
        }
        /* Seed step: max(num_accepted - 1, 0); none given => step 0. */
        int64_t t_seed = 0;
        if (pr->num_accepted != NULL) {
            t_seed = pr->num_accepted[b] - 1;
            if (t_seed < 0) t_seed = 0;
        }
        /* A per-row table holds one entry per packed row ("SSU at a glance",
         * Slot semantics): the seed step must be one of the sequence's own
         * rows, or the entry would belong to another sequence. */
        if (rtab != NULL && rtab->entries != NULL && rtab->mode == ORC_SLOTS_PER_ROW && t_seed >= len) {
            set_err(err, errlen, "seed step past the rows of sequence %lld (step %lld)", b, t_seed);
            rc = ORC_INVALID;
            break;
        }
        if (resolve(rtab, b, t_seed, start[b], &seed[b]) != 0) {
            set_err(err, errlen, "read-table entry out of range (sequence %lld, step %lld)", b, t_seed);
            rc = ORC_INVALID;
            break;
        }
        if (seed[b] != pr->pad_slot_id && (seed[b] < 0 || seed[b] >= pr->slots)) {
            set_err(err, errlen, "seed slot %lld of sequence %lld out of range", seed[b], b);
            rc = ORC_INVALID;
            break;
        }
        for (int64_t t = 0; t < len; ++t) {
            int64_t r = start[b] + t, w;
            if (resolve(wtab, b, t, start[b], &w) != 0) {
                set_err(err, errlen, "destination entry out of range (sequence %lld, step %lld)", b, t);
                rc = ORC_INVALID;
                break;
            }
            if (w != pr->pad_slot_id && (w < 0 || w >= pr->slots)) {
                set_err(err, errlen, "destination slot %lld of row %lld out of range", w, r);
                rc = ORC_INVALID;
                break;
            }
            wslot[r] = w;
            if (w != pr->pad_slot_id && !pr->disable_state_update) {
                if (writer[w] != -1 && writer[w] != b) {
                    set_err(err, errlen, "slot %lld is written by two sequences (second: %lld)", w, b);
                    rc = ORC_ALIASING;
                    break;
                }
                writer[w] = b;
            }
        }
    }
    /* A seed that another sequence overwrites has no defined value. */
    for (int64_t b = 0; b < nseq && rc == ORC_OK; ++b) {
        if (start[b + 1] == start[b] || seed[b] == pr->pad_slot_id)
            continue;
        if (writer[seed[b]] != -1 && writer[seed[b]] != b) {
            set_err(err, errlen, "seed slot %lld of sequence %lld is written by another sequence",
                    seed[b], b);
            rc = ORC_ALIASING;
        }
    }
    if (rc != ORC_OK) {
        free(start); free(seed); free(wslot); free(writer);
        return rc;
    }

    if (pr->slot_touched != NULL) {
        for (int64_t b = 0; b < nseq; ++b) {
            if (start[b + 1] == start[b]) continue;
            if (seed[b] != pr->pad_slot_id) pr->slot_touched[seed[b]] |= ORC_TOUCH_READ;
            if (pr->disable_state_update) continue;
            for (int64_t r = start[b]; r < start[b + 1]; ++r)
                if (wslot[r] != pr->pad_slot_id) pr->slot_touched[wslot[r]] |= ORC_TOUCH_WRITTEN;
        }
    }

    double *S = malloc(sizeof(double) * (size_t)N);
    if (!S) {
        free(start); free(seed); free(wslot); free(writer);
        return ORC_INVALID;
    }
    for (int64_t b = 0; b < nseq; ++b) {
        for (int64_t h = 0; h < H; ++h) {
            const int64_t g = h / heads_per_group;
            const double A = (double)pr->A[h];
            const double Dh = pr->D ? (double)pr->D[h] : 0.0;
            const double bias = pr->dt_bias ? (double)pr->dt_bias[h] : 0.0;
            for (int64_t p = 0; p < P; ++p) {
                if (start[b + 1] == start[b])
                    continue;                       /* empty sequence: skipped */
                /* Seed: a pad slot reads as a zero state.  Seeds come from the
                 * input pool, which no write of this call touches. */
                for (int64_t n = 0; n < N; ++n)
                    S[n] = (seed[b] == pr->pad_slot_id)
                               ? 0.0
                               : load_elem(pr->state_in, ((seed[b] * H + h) * P + p) * N + n,
                                           pr->state_dtype);
                for (int64_t r = start[b]; r < start[b + 1]; ++r) {
                    const int64_t xi = (r * H + h) * P + p;
                    const int64_t dti = pr->dt_per_head ? (r * H + h) : xi;
                    double d = load_elem(pr->dt, dti, pr->dt_dtype) + bias;
                    if (pr->dt_softplus)
                        d = orc_softplus(d);
                    const double dA = exp(A * d);
                    const double xv = load_elem(pr->x, xi, pr->io_dtype);
                    const int64_t bc = (r * G + g) * N;
                    double y = 0.0;
                    for (int64_t n = 0; n < N; ++n) {
                        S[n] = S[n] * dA + d * xv * load_elem(pr->B, bc + n, pr->io_dtype);
                        y += S[n] * load_elem(pr->C, bc + n, pr->io_dtype);
                    }
                    y += Dh * xv;
                    if (pr->z != NULL)
                        y *= orc_silu(load_elem(pr->z, xi, pr->io_dtype));
                    if (pr->y_exact != NULL)
                        pr->y_exact[xi] = y;
                    store_elem(pr->y, xi, pr->io_dtype, y);
                    /* Publish this token's state (never re-read: S stays in
                     * double for the next token). */
                    if (!pr->disable_state_update && wslot[r] != pr->pad_slot_id)
                        for (int64_t n = 0; n < N; ++n)
                            store_elem(pr->state_out, ((wslot[r] * H + h) * P + p) * N + n,
                                       pr->state_dtype, S[n]);
                }
            }
        }
    }
    free(S);
    free(start); free(seed); free(wslot); free(writer);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* ReplaySSM decode step (article "ReplaySSM: Cache SSM Inputs, Not State", */
/* section 核心做法): the state of a slot is a checkpoint S_ckpt plus the     */
/* inputs (v, Delta, k) = (x, dt', B) of the c steps since the last fold.    */
/* Each call appends the current token's inputs as entry c.  While the      */
/* buffer is not full (c + 1 < L) y is read out of checkpoint and buffer     */
/* without forming the state (the unrolled recurrence):                      */
/*   y = gamma_{0:c} (S_ckpt . q) + sum_j gamma_{j+1:c} Delta_j v_j (k_j . q) */
/* with gamma_{i:c} = prod_{m=i..c} exp(A Delta_m), q = C, plus D x and the  */
/* silu gate, and nothing but the new entry is written.  When it is full     */
/* (c + 1 = L) the buffer is folded into the checkpoint step by step, the    */
/* state is written back once, y is read out of it, and the buffer empties. */
/* Readings: on a fold step y comes from the folded state (so that L = 1 is  */
/* the plain update, as the article states); a pad slot has no history:     */
/* zero state, the current token only, nothing written, count 0.            */
/* ------------------------------------------------------------------------ */
int orc_replay_run(const orc_replay_problem *pr, char *err, int errlen)
{
    const int64_t H = pr->heads, P = pr->dim, N = pr->dstate, G = pr->groups, Lb = pr->len;
    if (H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G != 0 || Lb < 1) {
        set_err(err, errlen, "bad shape: heads=%lld len=%lld", H, Lb);
        return ORC_INVALID;
    }
    if (pr->shadow_format != ORC_SHADOW_NONE &&
        ((pr->shadow_format != ORC_SHADOW_F16 && pr->shadow_format != ORC_SHADOW_E4M3 &&
          pr->shadow_format != ORC_SHADOW_NVFP4) ||
         pr->shadow == NULL || (pr->shadow_format != ORC_SHADOW_F16 && pr->shadow_scale == NULL) ||
         (pr->shadow_format == ORC_SHADOW_NVFP4 && pr->dstate % 16 != 0))) {
        set_err(err, errlen, "bad read copy (format %lld, or its arrays missing)", pr->shadow_format, 0);
        return ORC_INVALID;
    }
    const int64_t heads_per_group = H / G;
    int64_t *owner = malloc(sizeof(int64_t) * (size_t)pr->slots);
    double *S = malloc(sizeof(double) * (size_t)N);
    if (!owner || !S) {
        free(owner); free(S);
        return ORC_INVALID;
    }
    for (int64_t s = 0; s < pr->slots; ++s)
        owner[s] = -1;
    int rc = ORC_OK;
    for (int64_t b = 0; b < pr->batch && rc == ORC_OK; ++b) {
        const int64_t slot = pr->slot_of ? pr->slot_of[b] : b;
        if (slot == pr->pad_slot_id)
            continue;
        if (slot < 0 || slot >= pr->slots) {
            set_err(err, errlen, "slot %lld of sequence %lld out of range", slot, b);
            rc = ORC_INVALID;
        } else if (owner[slot] != -1) {
            set_err(err, errlen, "slot %lld is used by two sequences (second: %lld)", slot, b);
            rc = ORC_ALIASING;
        } else if (pr->count_in[b] < 0 || pr->count_in[b] >= Lb) {
            set_err(err, errlen, "buffered count %lld of sequence %lld not in [0, L)", pr->count_in[b], b);
            rc = ORC_INVALID;
        } else {
            owner[slot] = b;
        }
    }
    if (rc != ORC_OK) {
        free(owner); free(S);
        return rc;
    }
    for (int64_t b = 0; b < pr->batch; ++b) {
        const int64_t slot = pr->slot_of ? pr->slot_of[b] : b;
        const int pad = slot == pr->pad_slot_id;
        const int64_t c = pad ? 0 : pr->count_in[b];
        const int fold = pad || c + 1 == Lb;
        pr->count_out[b] = (pad || fold) ? 0 : c + 1;
        for (int64_t h = 0; h < H; ++h) {
            const int64_t g = h / heads_per_group;
            const double A = (double)pr->A[h];
            const double Dh = pr->D ? (double)pr->D[h] : 0.0;
            const double bias = pr->dt_bias ? (double)pr->dt_bias[h] : 0.0;
            const int64_t bc_now = (b * G + g) * N;
            for (int64_t p = 0; p < P; ++p) {
                const int64_t xi = (b * H + h) * P + p;
                const int64_t dti = pr->dt_per_head ? (b * H + h) : xi;
                double d = load_elem(pr->dt, dti, pr->dt_dtype) + bias;
                if (pr->dt_softplus)
                    d = orc_softplus(d);
                const double xv = load_elem(pr->x, xi, pr->io_dtype);
                double y;
                if (fold) {
                    /* S_ckpt, then each buffered step, then the current one. */
                    for (int64_t n = 0; n < N; ++n)
                        S[n] = pad ? 0.0
                                   : load_elem(pr->ckpt_in, ((slot * H + h) * P + p) * N + n, pr->state_dtype);
                    for (int64_t j = 0; j < c; ++j) {
                        const int64_t e = ((slot * Lb + j) * H + h) * P + p;
                        const double dj = (double)pr->dtbuf[e];
                        const double xj = load_elem(pr->xbuf, e, pr->io_dtype);
                        const double aj = exp(A * dj);
                        const int64_t be = ((slot * Lb + j) * G + g) * N;
                        for (int64_t n = 0; n < N; ++n)
                            S[n] = S[n] * aj + dj * xj * load_elem(pr->Bbuf, be + n, pr->io_dtype);
                    }
                    const double a = exp(A * d);
                    y = 0.0;
                    for (int64_t n = 0; n < N; ++n) {
                        S[n] = S[n] * a + d * xv * load_elem(pr->B, bc_now + n, pr->io_dtype);
                        y += S[n] * load_elem(pr->C, bc_now + n, pr->io_dtype);
                    }
                    if (!pad) {
                        const int64_t row = (slot * H + h) * P + p;
                        for (int64_t n = 0; n < N; ++n)
                            store_elem(pr->ckpt_out, row * N + n, pr->state_dtype, S[n]);
                        if (pr->shadow_format != ORC_SHADOW_NONE) {
                            /* the read copy of the checkpoint as stored */
                            for (int64_t n = 0; n < N; ++n)
                                S[n] = load_elem(pr->ckpt_out, row * N + n, pr->state_dtype);
                            shadow_row(S, N, pr->shadow_format,
                                       (char *)pr->shadow + shadow_code_offset(row, N, pr->shadow_format),
                                       pr->shadow_scale ? pr->shadow_scale + shadow_scale_offset(row, N, pr->shadow_format)
                                                        : NULL);
                        }
                    }
                } else {
                    /* Output from checkpoint and buffer: walk the entries from
                     * the newest (the current token, entry c) to the oldest,
                     * w = gamma_{j+1:c}; after the walk w = gamma_{0:c}. */
                    double w = 1.0, hist = 0.0, kq;
                    kq = 0.0;
                    for (int64_t n = 0; n < N; ++n)
                        kq += load_elem(pr->B, bc_now + n, pr->io_dtype) * load_elem(pr->C, bc_now + n, pr->io_dtype);
                    hist += w * d * xv * kq;
                    w *= exp(A * d);
                    for (int64_t j = c - 1; j >= 0; --j) {
                        const int64_t e = ((slot * Lb + j) * H + h) * P + p;
                        const double dj = (double)pr->dtbuf[e];
                        const double xj = load_elem(pr->xbuf, e, pr->io_dtype);
                        const int64_t be = ((slot * Lb + j) * G + g) * N;
                        kq = 0.0;
                        for (int64_t n = 0; n < N; ++n)
                            kq += load_elem(pr->Bbuf, be + n, pr->io_dtype) * load_elem(pr->C, bc_now + n, pr->io_dtype);
                        hist += w * dj * xj * kq;
                        w *= exp(A * dj);
                    }
                    /* S_ckpt . C, from the read copy when there is one */
                    double sq = 0.0;
                    const int64_t row = (slot * H + h) * P + p;
                    for (int64_t n = 0; n < N; ++n)
                        sq += (pr->shadow_format != ORC_SHADOW_NONE
                                   ? shadow_value(pr->shadow, pr->shadow_scale, row, N, n, pr->shadow_format)
                                   : load_elem(pr->ckpt_in, row * N + n, pr->state_dtype)) *
                              load_elem(pr->C, bc_now + n, pr->io_dtype);
                    y = w * sq + hist;
                    /* Append the current token as entry c (v and k keep their
                     * bits; the processed step is stored in fp32). */
                    const int64_t e = ((slot * Lb + c) * H + h) * P + p;
                    memcpy((char *)pr->xbuf + e * (pr->io_dtype == ORC_F32 ? 4 : 2),
                           (const char *)pr->x + xi * (pr->io_dtype == ORC_F32 ? 4 : 2),
                           pr->io_dtype == ORC_F32 ? 4 : 2);
                    pr->dtbuf[e] = (float)d;
                    if (h % heads_per_group == 0 && p == 0) {
                        const int64_t be = ((slot * Lb + c) * G + g) * N;
                        const size_t es = pr->io_dtype == ORC_F32 ? 4 : 2;
                        memcpy((char *)pr->Bbuf + be * es, (const char *)pr->B + bc_now * es, es * (size_t)N);
                    }
                }
                y += Dh * xv;
                if (pr->z != NULL)
                    y *= orc_silu(load_elem(pr->z, xi, pr->io_dtype));
                if (pr->y_exact != NULL)
                    pr->y_exact[xi] = y;
                store_elem(pr->y, xi, pr->io_dtype, y);
            }
        }
    }
    free(owner);
    free(S);
    return ORC_OK;
}


/* ------------------------------------------------------------------------ */
/* Speculative decoding on the checkpoint + buffer form (article            */
/* "ReplaySSM", section 投机解码回滚): the drafts go into the buffer after    */
/* the committed entries and each draft's output is read from the state     */
/* through it (causal mask); commit is the caller moving the count.  The    */
/* outputs are computed by running the recurrence in double from the        */
/* checkpoint through the entries, which the unrolled form only reorders.   */
/* Readings: the flush fires when c + 2T >= L (the article's rule, one      */
/* window early) and happens before the drafts are appended; the drafts     */
/* read the checkpoint as stored after it; every step, the drafts' own      */
/* included, uses its processed dt' as stored in fp32 (what a later fold    */
/* will see); a pad slot is a zero state with no history.                   */
/* ------------------------------------------------------------------------ */
int orc_replay_verify_run(const orc_verify_problem *pr, char *err, int errlen)
{
    const int64_t H = pr->heads, P = pr->dim, N = pr->dstate, G = pr->groups, Lb = pr->len, T = pr->ntok;
    if (H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G != 0 || Lb < 1 || T < 1 || T > Lb) {
        set_err(err, errlen, "bad shape: len=%lld drafts=%lld", Lb, T);
        return ORC_INVALID;
    }
    const int64_t heads_per_group = H / G;
    int64_t *owner = malloc(sizeof(int64_t) * (size_t)pr->slots);
    double *S = malloc(sizeof(double) * (size_t)N);
    if (!owner || !S) {
        free(owner); free(S);
        return ORC_INVALID;
    }
    for (int64_t s = 0; s < pr->slots; ++s)
        owner[s] = -1;
    int rc = ORC_OK;
    for (int64_t b = 0; b < pr->batch && rc == ORC_OK; ++b) {
        const int64_t slot = pr->slot_of ? pr->slot_of[b] : b;
        if (slot == pr->pad_slot_id)
            continue;
        if (slot < 0 || slot >= pr->slots) {
            set_err(err, errlen, "slot %lld of sequence %lld out of range", slot, b);
            rc = ORC_INVALID;
        } else if (owner[slot] != -1) {
            set_err(err, errlen, "slot %lld is used by two sequences (second: %lld)", slot, b);
            rc = ORC_ALIASING;
        } else if (pr->count_in[b] < 0 || pr->count_in[b] >= Lb) {
            set_err(err, errlen, "committed count %lld of sequence %lld not in [0, L)", pr->count_in[b], b);
            rc = ORC_INVALID;
        } else {
            owner[slot] = b;
        }
    }
    if (rc != ORC_OK) {
        free(owner); free(S);
        return rc;
    }
    const size_t es = pr->io_dtype == ORC_F32 ? 4 : 2;
    for (int64_t b = 0; b < pr->batch; ++b) {
        const int64_t slot = pr->slot_of ? pr->slot_of[b] : b;
        const int pad = slot == pr->pad_slot_id;
        const int64_t c_in = pad ? 0 : pr->count_in[b];
        const int fold = !pad && c_in + 2 * T >= Lb;
        const int64_t c = fold ? 0 : c_in;
        pr->count_out[b] = c;
        /* First every head's fold (the drafts' B, shared by a group, will
         * overwrite the entries the other heads of the group fold). */
        for (int64_t h = 0; fold && h < H; ++h) {
            const int64_t g = h / heads_per_group;
            const double A = (double)pr->A[h];
            for (int64_t p = 0; p < P; ++p) {
                const int64_t row = (slot * H + h) * P + p;
                for (int64_t n = 0; n < N; ++n)
                    S[n] = load_elem(pr->ckpt_in, row * N + n, pr->state_dtype);
                for (int64_t j = 0; j < c_in; ++j) {
                    const int64_t e = ((slot * Lb + j) * H + h) * P + p;
                    const double dj = (double)pr->dtbuf[e];
                    const double xj = load_elem(pr->xbuf, e, pr->io_dtype);
                    const double aj = exp(A * dj);
                    const int64_t be = ((slot * Lb + j) * G + g) * N;
                    for (int64_t n = 0; n < N; ++n)
                        S[n] = S[n] * aj + dj * xj * load_elem(pr->Bbuf, be + n, pr->io_dtype);
                }
                for (int64_t n = 0; n < N; ++n)
                    store_elem(pr->ckpt_out, row * N + n, pr->state_dtype, S[n]);
            }
        }
        /* Then the drafts: from the checkpoint as stored and the committed
         * entries (none after a fold), each read out after its own step and
         * appended as entry c + k. */
        for (int64_t h = 0; h < H; ++h) {
            const int64_t g = h / heads_per_group;
            const double A = (double)pr->A[h];
            const double Dh = pr->D ? (double)pr->D[h] : 0.0;
            const double bias = pr->dt_bias ? (double)pr->dt_bias[h] : 0.0;
            for (int64_t p = 0; p < P; ++p) {
                const int64_t row = (slot * H + h) * P + p;
                for (int64_t n = 0; n < N; ++n)
                    S[n] = pad ? 0.0 : load_elem(fold ? pr->ckpt_out : pr->ckpt_in, row * N + n, pr->state_dtype);
                for (int64_t j = 0; j < c; ++j) {
                    const int64_t e = ((slot * Lb + j) * H + h) * P + p;
                    const double dj = (double)pr->dtbuf[e];
                    const double xj = load_elem(pr->xbuf, e, pr->io_dtype);
                    const double aj = exp(A * dj);
                    const int64_t be = ((slot * Lb + j) * G + g) * N;
                    for (int64_t n = 0; n < N; ++n)
                        S[n] = S[n] * aj + dj * xj * load_elem(pr->Bbuf, be + n, pr->io_dtype);
                }
                for (int64_t k = 0; k < T; ++k) {
                    const int64_t r = b * T + k;
                    const int64_t xi = (r * H + h) * P + p;
                    const int64_t dti = pr->dt_per_head ? (r * H + h) : xi;
                    double d = load_elem(pr->dt, dti, pr->dt_dtype) + bias;
                    if (pr->dt_softplus)
                        d = orc_softplus(d);
                    d = (double)(float)d;  /* the step as stored */
                    const double xv = load_elem(pr->x, xi, pr->io_dtype);
                    const int64_t bc = (r * G + g) * N;
                    const double a = exp(A * d);
                    double y = 0.0;
                    for (int64_t n = 0; n < N; ++n) {
                        S[n] = S[n] * a + d * xv * load_elem(pr->B, bc + n, pr->io_dtype);
                        y += S[n] * load_elem(pr->C, bc + n, pr->io_dtype);
                    }
                    y += Dh * xv;
                    if (pr->z != NULL)
                        y *= orc_silu(load_elem(pr->z, xi, pr->io_dtype));
                    if (pr->y_exact != NULL)
                        pr->y_exact[xi] = y;
                    store_elem(pr->y, xi, pr->io_dtype, y);
                    if (!pad) {  /* draft k becomes entry c + k */
                        const int64_t e = ((slot * Lb + c + k) * H + h) * P + p;
                        memcpy((char *)pr->xbuf + (size_t)e * es, (const char *)pr->x + (size_t)xi * es, es);
                        pr->dtbuf[e] = (float)d;
                        if (h % heads_per_group == 0 && p == 0) {
                            const int64_t be = ((slot * Lb + c + k) * G + g) * N;
                            memcpy((char *)pr->Bbuf + (size_t)be * es, (const char *)pr->B + (size_t)bc * es,
                                   es * (size_t)N);
                        }
                    }
                }
            }
        }
    }
    free(owner);
    free(S);
    return ORC_OK;
}


/* ------------------------------------------------------------------------ */
/* Packed variable-length SSD prefill (MATE "Mamba / SSU", SSD packed        */
/* prefill; API reference of ssd_combined_fwd_varlen): the recurrence over   */
/* each sequence's tokens, chunk by chunk in order, the entering state of a  */
/* chunk decided by seq_idx (the page: seq_idx, not last_chunk_indices, is   */
/* the authority), dt clamped to dt_limit after softplus.                    */
/* ------------------------------------------------------------------------ */
int orc_ssd_run(const orc_ssd_problem *pr, char *err, int errlen)
{
    const int64_t H = pr->heads, P = pr->dim, N = pr->dstate, G = pr->groups, T = pr->tokens;
    if (H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G != 0 || pr->nchunks < 0 || T < 0 || pr->nseq < 0) {
        set_err(err, errlen, "bad shape: heads=%lld groups=%lld", H, G);
        return ORC_INVALID;
    }
    if (pr->cu_chunk[0] != 0 || pr->cu_chunk[pr->nchunks] != T) {
        set_err(err, errlen, "cu_chunk_seqlens must start at 0 and end at tokens (%lld)", T, 0);
        return ORC_INVALID;
    }
    for (int64_t c = 0; c < pr->nchunks; ++c) {
        if (pr->cu_chunk[c + 1] < pr->cu_chunk[c]) {
            set_err(err, errlen, "cu_chunk_seqlens decreases at chunk %lld", c, 0);
            return ORC_INVALID;
        }
        if (pr->seq_idx[c] < 0 || pr->seq_idx[c] >= pr->nseq) {
            set_err(err, errlen, "seq_idx[%lld] = %lld out of range", c, pr->seq_idx[c]);
            return ORC_INVALID;
        }
    }
    const int64_t hpg = H / G;
    double *S = malloc(sizeof(double) * (size_t)N);
    if (!S)
        return ORC_INVALID;
    for (int64_t h = 0; h < H; ++h) {
        const int64_t g = h / hpg;
        const double A = (double)pr->A[h];
        const double Dh = pr->D ? (double)pr->D[h] : 0.0;
        const double bias = pr->dt_bias ? (double)pr->dt_bias[h] : 0.0;
        for (int64_t p = 0; p < P; ++p) {
            for (int64_t c = 0; c < pr->nchunks; ++c) {
                const int64_t b = pr->seq_idx[c];
                if (c == 0 || pr->seq_idx[c] != pr->seq_idx[c - 1]) {
                    /* the chunk opens sequence b */
                    for (int64_t n = 0; n < N; ++n)
                        S[n] = pr->initial_states
                                   ? load_elem(pr->initial_states, ((b * H + h) * P + p) * N + n, pr->state_dtype)
                                   : 0.0;
                }
                for (int64_t t = pr->cu_chunk[c]; t < pr->cu_chunk[c + 1]; ++t) {
                    double d = load_elem(pr->dt, t * H + h, pr->dt_dtype) + bias;
                    if (pr->dt_softplus)
                        d = orc_softplus(d);
                    d = fmin(fmax(d, pr->dt_lo), pr->dt_hi);
                    const double a = exp(A * d);
                    const double xv = load_elem(pr->x, (t * H + h) * P + p, pr->io_dtype);
                    double y = 0.0;
                    for (int64_t n = 0; n < N; ++n) {
                        S[n] = S[n] * a + d * xv * load_elem(pr->B, (t * G + g) * N + n, pr->io_dtype);
                        y += S[n] * load_elem(pr->C, (t * G + g) * N + n, pr->io_dtype);
                    }
                    y += Dh * xv;
                    if (pr->z != NULL)
                        y *= orc_silu(load_elem(pr->z, (t * H + h) * P + p, pr->io_dtype));
                    if (pr->y_exact != NULL)
                        pr->y_exact[(t * H + h) * P + p] = y;
                    store_elem(pr->y, (t * H + h) * P + p, pr->io_dtype, y);
                }
                for (int64_t n = 0; n < N; ++n)
                    store_elem(pr->states, ((c * H + h) * P + p) * N + n, pr->state_dtype, S[n]);
            }
        }
    }
    free(S);
    return ORC_OK;
}

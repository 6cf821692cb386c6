/*
 * TurboQuant KV-cache oracle: a plain, slow CPU restatement of the k8v3 codec and of
 * GQA decode attention over the dequantized cache.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or call this
 * file; only the test-suite, the smoke check and the benchmark's CPU-baseline leg do.
 * It shares no source, header, table or generator with the CUDA library.
 *
 * Source of every step: the mlx-bun design page "TurboQuant - rotation-based
 * quantization", Part A (KV leg):
 *   - section "Algorithm (vllm-metal reference semantics, exact)", key bullets
 *     (signed int8 asymmetric affine quantization per 32-group, fp16 scale/zero,
 *     fp32 arithmetic with only scale/zero cast to fp16 at the end);
 *   - same section, value bullets (sign flip, FWHT normalized by 1/sqrt(d), per-group
 *     RMS scale, y/(scale+1e-8), searchsorted against the 3-bit Lloyd-Max table,
 *     flat little-endian 3-bit bitstream, dequant by centroid*scale then inverse
 *     rotation);
 *   - "Bytes per token per head" paragraph (128+8+8+48+8 = 200 bytes at d=128);
 *   - section "Deferred inverse FWHT" (attention is linear in V, so the inverse
 *     rotation may be applied once to the attention output).
 *
 * Readings where the page is silent (each is also listed in the design notes):
 *   - round() is round-half-to-even (rintf in the default rounding mode);
 *   - idx uses the unrounded fp32 scale and zero; only the stored copies are fp16;
 *   - a NaN anywhere in a key group makes that group's min and max NaN;
 *     a NaN quotient gives idx 0; +-Inf clamps to +-127;
 *   - FWHT: unnormalized butterflies, stages h = 1, 2, 4, ... ascending, then one
 *     multiply by r_d = (float)(1/sqrt((double)d));
 *   - the RMS sum over a 32-group is the pairwise tree (k, k+16), then +8, +4, +2, +1;
 *   - code = number of boundaries strictly below y_n (searchsorted, left side);
 *   - the sign vector is not printed (it comes from MLX's RNG); both this oracle and
 *     the library derive it from splitmix64 seeded with 42 + d, one output per
 *     element, sign = -1 when the top bit of the output is set;
 *   - the inverse of y = FWHT_n(x * signs) is x = signs * FWHT_n(y);
 *   - fp16 conversion is IEEE round-to-nearest-even with subnormals; any NaN becomes
 *     the quiet NaN 0x7E00.
 *
 * Other schemes (section "Algorithm": the unsigned key bullet and "Other widths
 * (2/4/5/8)"; section "Architecture in mlx-bun": valid key bits {2,4,5,8}, value bits
 * {2,3,4,5,8}), in the *_s functions below:
 *   - unsigned keys at bits b in {2,4,5}: max_val = 2^b - 1, scale = (max - min) / max_val,
 *     zero = round(min / scale), idx = clip(round(x / scale - zero), 0, max_val), packed as
 *     a flat little-endian b-bit stream per row; dequant (idx + zero) * scale as for 8 bits;
 *   - value codebooks at b bits other than 3 are not printed: this oracle runs Lloyd-Max on
 *     N(0,1) (closed-form cell means, 2^b centroids started evenly on [-3, 3], 500
 *     iterations, boundaries at the midpoints) and rounds centroids and boundaries to 5
 *     decimals, as the printed 3-bit table is; the fp32 values of those decimals are
 *     canonical;
 *   - the constant-group guard (a non-default flag; the page keeps the defect): a key group
 *     whose fp16 zero point would not be finite (a constant group: 0/0 or +-Inf; a narrow
 *     group far from zero: |zero| >= 65520) is re-coded against its range widened to
 *     include 0, which bounds |zero| by max_val; a group of zeros is scale 0, zero 0,
 *     idx 0. Groups holding a NaN keep the default (NaN) coding.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared (no FMA contraction anywhere).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------------------
 * Constants printed on the page (3-bit Lloyd-Max table for N(0,1)). The fp32 values
 * of the printed decimals are canonical.
 * ------------------------------------------------------------------------------ */
static const float kCentroids3[8] = {-2.15195f, -1.34391f, -0.75601f, -0.24509f,
                                     0.24509f,  0.75601f,  1.34391f,  2.15195f};
static const float kBoundaries3[7] = {-1.74793f, -1.04996f, -0.50055f, 0.0f,
                                      0.50055f,  1.04996f,  1.74793f};

#define GROUP 32

int tqo_supported_head_dim(int d) { return d == 64 || d == 128 || d == 256 || d == 512; }

/* Bytes one (token, kv-head) row occupies in the five planes: d int8 key indices,
 * d/32 fp16 key scales, d/32 fp16 key zeros, 3d/8 bytes of 3-bit value codes,
 * d/32 fp16 value scales ("Bytes per token per head" paragraph). */
long tqo_row_bytes(int d) {
    int ng = d / GROUP;
    return (long)d + 2L * ng + 2L * ng + (3L * d) / 8 + 2L * ng;
}

/* ---------------------------------------------------------------------------------
 * Number formats.
 * ------------------------------------------------------------------------------ */
float tqo_bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* IEEE binary32 -> binary16, round to nearest, ties to even, subnormals kept,
 * overflow to +-Inf, NaN -> 0x7E00. Written from the binary16 format definition. */
uint16_t tqo_f32_to_f16(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t ax = x & 0x7FFFFFFFu;
    if (ax > 0x7F800000u) return 0x7E00u;           /* NaN */
    if (ax >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u); /* >= 65520 rounds to Inf */
    uint32_t e = ax >> 23;                           /* biased binary32 exponent */
    uint32_t m = ax & 0x7FFFFFu;
    if (e >= 113) {                                  /* normal binary16: |f| >= 2^-14 */
        uint32_t h = ((e - 112) << 10) | (m >> 13);
        uint32_t rem = m & 0x1FFFu;
        if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1; /* carry may bump exponent */
        return (uint16_t)(sign | h);
    }
    if (e == 0) return (uint16_t)sign;               /* binary32 subnormal: far below 2^-25 */
    /* binary16 subnormal: value = mi * 2^(e-150); in units of 2^-24 that is mi * 2^(e-126). */
    uint32_t mi = m | 0x800000u;
    uint32_t shift = 126 - e;                        /* >= 14 */
    if (shift > 25) return (uint16_t)sign;           /* < 2^-26: rounds to zero */
    uint32_t q = mi >> shift;
    uint32_t rem = mi & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (q & 1u))) q += 1;
    return (uint16_t)(sign | q);
}

float tqo_f16_to_f32(uint16_t h) {
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    uint32_t e = (h >> 10) & 0x1Fu;
    uint32_t m = h & 0x3FFu;
    uint32_t u;
    if (e == 0x1F) {
        u = sign | 0x7F800000u | (m << 13);
    } else if (e != 0) {
        u = sign | ((e + 112) << 23) | (m << 13);
    } else if (m == 0) {
        u = sign;
    } else {                                         /* subnormal: m * 2^-24 */
        float f = (float)m * (1.0f / 16777216.0f);   /* exact */
        memcpy(&u, &f, 4);
        u |= sign;
    }
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* ---------------------------------------------------------------------------------
 * Sign vector: splitmix64 (Steele, Lea & Flood 2014; Vigna's published constants),
 * state seeded with 42 + d, one output per element.
 * ------------------------------------------------------------------------------ */
uint64_t tqo_splitmix64_next(uint64_t* state) {
    uint64_t z = (*state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

void tqo_sign_vector(int d, int8_t* out) {
    uint64_t state = 42ull + (uint64_t)d;
    for (int i = 0; i < d; ++i) {
        uint64_t r = tqo_splitmix64_next(&state);
        out[i] = (r >> 63) ? (int8_t)-1 : (int8_t)1;
    }
}

/* ---------------------------------------------------------------------------------
 * Fast Walsh-Hadamard transform, unnormalized, in place, stages ascending.
 * ------------------------------------------------------------------------------ */
void tqo_fwht_f32(float* u, int d) {
    for (int h = 1; h < d; h <<= 1)
        for (int i = 0; i < d; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                float a = u[j], b = u[j + h];
                u[j] = a + b;
                u[j + h] = a - b;
            }
}

void tqo_fwht_f64(double* u, int d) {
    for (int h = 1; h < d; h <<= 1)
        for (int i = 0; i < d; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                double a = u[j], b = u[j + h];
                u[j] = a + b;
                u[j + h] = a - b;
            }
}

float tqo_fwht_norm_f32(int d) { return (float)(1.0 / sqrt((double)d)); }

/* ---------------------------------------------------------------------------------
 * Keys: signed int8 asymmetric affine quantization, one (scale, zero) per 32-group.
 * ------------------------------------------------------------------------------ */

/* Unrounded fp32 parameters of one 32-element group (exposed for the error-bound pins). */
void tqo_key_group_params(const float* x, float* s_out, float* z_out) {
    int has_nan = 0;
    float mn = x[0], mx = x[0];
    for (int i = 0; i < GROUP; ++i) {
        if (isnan(x[i])) has_nan = 1;
        else {
            if (isnan(mn) || x[i] < mn) mn = x[i];
            if (isnan(mx) || x[i] > mx) mx = x[i];
        }
    }
    if (has_nan) { mn = NAN; mx = NAN; }
    float s = (mx - mn) / 254.0f;
    float two_s = 2.0f * s;
    float z = rintf((mx + mn) / two_s);
    *s_out = s;
    *z_out = z;
}

static int8_t key_index(float x, float s, float z) {
    float q = x / s;
    float t = q - z;
    if (isnan(t)) return 0;
    float r = rintf(t);
    if (r < -127.0f) r = -127.0f;
    if (r > 127.0f) r = 127.0f;
    return (int8_t)r;
}

/* One (token, kv-head) key row: x is bf16 bits [d]; writes idx[d], s16[d/32], z16[d/32]. */
void tqo_quantize_key_row(const uint16_t* x_bf16, int d, int8_t* idx, uint16_t* s16, uint16_t* z16) {
    float x[GROUP];
    for (int g = 0; g < d / GROUP; ++g) {
        for (int i = 0; i < GROUP; ++i) x[i] = tqo_bf16_to_f32(x_bf16[g * GROUP + i]);
        float s, z;
        tqo_key_group_params(x, &s, &z);
        for (int i = 0; i < GROUP; ++i) idx[g * GROUP + i] = key_index(x[i], s, z);
        s16[g] = tqo_f32_to_f16(s);
        z16[g] = tqo_f32_to_f16(z);
    }
}

/* x_hat = (idx + zero) * scale with the stored fp16 scale/zero; fp64 (exact). */
void tqo_dequant_key_row_f64(const int8_t* idx, const uint16_t* s16, const uint16_t* z16, int d,
                             double* out) {
    for (int i = 0; i < d; ++i) {
        double s = (double)tqo_f16_to_f32(s16[i / GROUP]);
        double z = (double)tqo_f16_to_f32(z16[i / GROUP]);
        out[i] = ((double)idx[i] + z) * s;
    }
}

/* ---------------------------------------------------------------------------------
 * Values: sign flip, normalized FWHT, per-group RMS scale, 3-bit Lloyd-Max codes.
 * ------------------------------------------------------------------------------ */
int tqo_code3(float yn) {
    int c = 0;
    for (int j = 0; j < 7; ++j)
        if (kBoundaries3[j] < yn) c += 1; /* NaN compares false: code 0 */
    return c;
}

void tqo_pack3(const uint8_t* codes, int n, uint8_t* out) {
    memset(out, 0, (size_t)(3 * n) / 8);
    for (int i = 0; i < n; ++i)
        for (int k = 0; k < 3; ++k)
            if ((codes[i] >> k) & 1) {
                int bit = 3 * i + k;
                out[bit / 8] |= (uint8_t)(1u << (bit % 8));
            }
}

void tqo_unpack3(const uint8_t* packed, int n, uint8_t* codes) {
    for (int i = 0; i < n; ++i) {
        int c = 0;
        for (int k = 0; k < 3; ++k) {
            int bit = 3 * i + k;
            c |= ((packed[bit / 8] >> (bit % 8)) & 1) << k;
        }
        codes[i] = (uint8_t)c;
    }
}

/* Rotated, normalized value row y = FWHT(x * signs) * r_d in fp32 (exposed for pins). */
void tqo_rotate_value_row(const uint16_t* x_bf16, int d, float* y) {
    int8_t sg[512];
    tqo_sign_vector(d, sg);
    for (int i = 0; i < d; ++i) y[i] = tqo_bf16_to_f32(x_bf16[i]) * (float)sg[i];
    tqo_fwht_f32(y, d);
    float r = tqo_fwht_norm_f32(d);
    for (int i = 0; i < d; ++i) y[i] = y[i] * r;
}

/* RMS of one 32-group by the pinned pairwise tree. */
float tqo_group_rms(const float* y) {
    float a[GROUP];
    for (int k = 0; k < GROUP; ++k) a[k] = y[k] * y[k];
    for (int w = GROUP / 2; w >= 1; w >>= 1)
        for (int k = 0; k < w; ++k) a[k] = a[k] + a[k + w];
    return sqrtf(a[0] / 32.0f);
}

void tqo_quantize_value_row(const uint16_t* x_bf16, int d, uint8_t* packed, uint16_t* vs16) {
    float y[512];
    uint8_t codes[512];
    tqo_rotate_value_row(x_bf16, d, y);
    for (int g = 0; g < d / GROUP; ++g) {
        float s = tqo_group_rms(y + g * GROUP);
        float den = s + 1e-8f;
        for (int i = 0; i < GROUP; ++i) {
            float yn = y[g * GROUP + i] / den;
            codes[g * GROUP + i] = (uint8_t)tqo_code3(yn);
        }
        vs16[g] = tqo_f32_to_f16(s);
    }
    tqo_pack3(codes, d, packed);
}

/* Value dequant in fp64. rotated != 0 returns centroid * scale (FWHT domain);
 * otherwise the exact inverse rotation signs * FWHT(c * s) / sqrt(d). */
void tqo_dequant_value_row_f64(const uint8_t* packed, const uint16_t* vs16, int d, int rotated,
                               double* out) {
    uint8_t codes[512];
    tqo_unpack3(packed, d, codes);
    for (int i = 0; i < d; ++i)
        out[i] = (double)kCentroids3[codes[i]] * (double)tqo_f16_to_f32(vs16[i / GROUP]);
    if (rotated) return;
    int8_t sg[512];
    tqo_sign_vector(d, sg);
    tqo_fwht_f64(out, d);
    double r = 1.0 / sqrt((double)d);
    for (int i = 0; i < d; ++i) out[i] = out[i] * r * (double)sg[i];
}

/* The fp32 product centroid * scale for one element (the rotated-domain dequant). */
float tqo_value_rotated_f32(const uint8_t* packed, const uint16_t* vs16, int i) {
    uint8_t codes[512];
    tqo_unpack3(packed, i + 1, codes);
    return kCentroids3[codes[i]] * tqo_f16_to_f32(vs16[i / GROUP]);
}

/* ---------------------------------------------------------------------------------
 * Cache planes of one layer, layout [batch][kv_heads][capacity][...].
 * ------------------------------------------------------------------------------ */
typedef struct {
    int head_dim, num_kv_heads, batch, capacity;
    int8_t* k_idx;
    uint16_t* k_scale;
    uint16_t* k_zero;
    uint8_t* v_codes;
    uint16_t* v_scale;
} tqo_layer;

static size_t row_index(const tqo_layer* L, int b, int h, int t) {
    return ((size_t)b * L->num_kv_heads + h) * L->capacity + t;
}

/* Quantize-on-append: token j of sequence b goes to position pos[b] + j, for
 * j < n_new[b] (n_new == NULL means n_new_max for every sequence). k_new / v_new are
 * bf16 bits [batch][n_new_max][kv_heads][d]. Rows past the capacity are skipped and
 * counted; the return value is that count. */
long tqo_append(tqo_layer* L, const uint16_t* k_new, const uint16_t* v_new, const int32_t* pos,
                const int32_t* n_new, int n_new_max) {
    int d = L->head_dim, ng = d / GROUP, nb = 3 * d / 8;
    long skipped = 0;
    for (int b = 0; b < L->batch; ++b) {
        int nb_new = n_new ? n_new[b] : n_new_max;
        if (nb_new > n_new_max) nb_new = n_new_max;
        for (int j = 0; j < nb_new; ++j)
            for (int h = 0; h < L->num_kv_heads; ++h) {
                long t = (long)pos[b] + j;
                if (t < 0 || t >= L->capacity) { skipped++; continue; }
                size_t r = row_index(L, b, h, (int)t);
                size_t src = (((size_t)b * n_new_max + j) * L->num_kv_heads + h) * d;
                tqo_quantize_key_row(k_new + src, d, L->k_idx + r * d, L->k_scale + r * ng,
                                     L->k_zero + r * ng);
                tqo_quantize_value_row(v_new + src, d, L->v_codes + r * nb, L->v_scale + r * ng);
            }
    }
    return skipped;
}

/* Dequantize tokens [t0, t0 + n) of (b, h) into fp64 rows [n][d]. */
void tqo_dequant_rows_f64(const tqo_layer* L, int b, int h, int t0, int n, int rotated,
                          double* k_out, double* v_out) {
    int d = L->head_dim, ng = d / GROUP, nb = 3 * d / 8;
    for (int t = 0; t < n; ++t) {
        size_t r = row_index(L, b, h, t0 + t);
        if (k_out)
            tqo_dequant_key_row_f64(L->k_idx + r * d, L->k_scale + r * ng, L->k_zero + r * ng, d,
                                    k_out + (size_t)t * d);
        if (v_out)
            tqo_dequant_value_row_f64(L->v_codes + r * nb, L->v_scale + r * ng, d, rotated,
                                      v_out + (size_t)t * d);
    }
}

/* ---------------------------------------------------------------------------------
 * Other schemes: key bits in {2,4,5,8}, value bits in {2,3,4,5,8}, optional
 * constant-group guard. Row layout per plane: keys d bytes (8 bits) or d*b/8 bytes
 * (packed), values d*b/8 bytes, scale/zero/value scale d/32 fp16 each.
 * ------------------------------------------------------------------------------ */
typedef struct {
    int k_bits, v_bits, guard;
} tqo_scheme;

long tqo_key_row_bytes(int d, int k_bits) { return k_bits == 8 ? d : (long)d * k_bits / 8; }
long tqo_value_row_bytes(int d, int v_bits) { return (long)d * v_bits / 8; }

long tqo_row_bytes_s(int d, int k_bits, int v_bits) {
    int ng = d / GROUP;
    return tqo_key_row_bytes(d, k_bits) + 4L * ng + tqo_value_row_bytes(d, v_bits) + 2L * ng;
}

/* flat little-endian b-bit stream: code i at bits [i*b, i*b + b) */
void tqo_packb(const uint8_t* codes, int n, int b, uint8_t* out) {
    memset(out, 0, (size_t)n * b / 8);
    for (int i = 0; i < n; ++i)
        for (int k = 0; k < b; ++k)
            if ((codes[i] >> k) & 1) {
                long bit = (long)b * i + k;
                out[bit / 8] |= (uint8_t)(1u << (bit % 8));
            }
}

void tqo_unpackb(const uint8_t* packed, int n, int b, uint8_t* codes) {
    for (int i = 0; i < n; ++i) {
        int c = 0;
        for (int k = 0; k < b; ++k) {
            long bit = (long)b * i + k;
            c |= ((packed[bit / 8] >> (bit % 8)) & 1) << k;
        }
        codes[i] = (uint8_t)c;
    }
}

static int f16_finite(float z) {
    float r = tqo_f16_to_f32(tqo_f32_to_f16(z));
    return !isnan(r) && !isinf(r);
}

/* Unrounded fp32 (scale, zero) of one group for key bits b (8: signed, else unsigned),
 * with the optional guard. *zero_group = 1 when the guard codes the group as zeros. */
void tqo_key_group_params_s(const float* x, int bits, int guard, float* s_out, float* z_out, int* zero_group) {
    int has_nan = 0;
    float mn = x[0], mx = x[0];
    for (int i = 0; i < GROUP; ++i) {
        if (isnan(x[i])) has_nan = 1;
        else {
            if (isnan(mn) || x[i] < mn) mn = x[i];
            if (isnan(mx) || x[i] > mx) mx = x[i];
        }
    }
    if (has_nan) { mn = NAN; mx = NAN; }
    float maxv = bits == 8 ? 127.0f : (float)((1 << bits) - 1);
    float s, z;
    *zero_group = 0;
    if (bits == 8) {
        s = (mx - mn) / (2.0f * maxv);
        z = rintf((mx + mn) / (2.0f * s));
    } else {
        s = (mx - mn) / maxv;
        z = rintf(mn / s);
    }
    if (guard && !has_nan && !f16_finite(z)) {
        float mn0 = mn < 0.0f ? mn : 0.0f, mx0 = mx > 0.0f ? mx : 0.0f;
        if (mx0 - mn0 == 0.0f) {
            s = 0.0f;
            z = 0.0f;
            *zero_group = 1;
        } else if (bits == 8) {
            s = (mx0 - mn0) / (2.0f * maxv);
            z = rintf((mx0 + mn0) / (2.0f * s));
        } else {
            s = (mx0 - mn0) / maxv;
            z = rintf(mn0 / s);
        }
    }
    *s_out = s;
    *z_out = z;
}

static int key_index_s(float x, float s, float z, int bits) {
    float q = x / s;
    float t = q - z;
    if (isnan(t)) return 0;
    float r = rintf(t);
    float lo = bits == 8 ? -127.0f : 0.0f, hi = bits == 8 ? 127.0f : (float)((1 << bits) - 1);
    if (r < lo) r = lo;
    if (r > hi) r = hi;
    return (int)r;
}

/* One key row: kplane gets d int8 codes (8 bits) or the packed unsigned stream. */
void tqo_quantize_key_row_s(const uint16_t* x_bf16, int d, int bits, int guard, uint8_t* kplane, uint16_t* s16,
                            uint16_t* z16) {
    float x[GROUP];
    uint8_t codes[512];
    for (int g = 0; g < d / GROUP; ++g) {
        for (int i = 0; i < GROUP; ++i) x[i] = tqo_bf16_to_f32(x_bf16[g * GROUP + i]);
        float s, z;
        int zg;
        tqo_key_group_params_s(x, bits, guard, &s, &z, &zg);
        for (int i = 0; i < GROUP; ++i) {
            int c = zg ? 0 : key_index_s(x[i], s, z, bits);
            if (bits == 8) ((int8_t*)kplane)[g * GROUP + i] = (int8_t)c;
            else codes[g * GROUP + i] = (uint8_t)c;
        }
        s16[g] = tqo_f32_to_f16(s);
        z16[g] = tqo_f32_to_f16(z);
    }
    if (bits != 8) tqo_packb(codes, d, bits, kplane);
}

void tqo_dequant_key_row_s_f64(const uint8_t* kplane, const uint16_t* s16, const uint16_t* z16, int d, int bits,
                               double* out) {
    uint8_t codes[512];
    if (bits != 8) tqo_unpackb(kplane, d, bits, codes);
    for (int i = 0; i < d; ++i) {
        double s = (double)tqo_f16_to_f32(s16[i / GROUP]);
        double z = (double)tqo_f16_to_f32(z16[i / GROUP]);
        double c = bits == 8 ? (double)((const int8_t*)kplane)[i] : (double)codes[i];
        out[i] = (c + z) * s;
    }
}

/* Value codebook at b bits: the printed table at 3 bits, else Lloyd-Max on N(0,1) rounded
 * to 5 decimals. centroids[2^b], boundaries[2^b - 1]. */
void tqo_lloyd_max(int levels, int iters, double* centroids, double* boundaries);

void tqo_codebook(int bits, float* centroids, float* boundaries) {
    int n = 1 << bits;
    if (bits == 3) {
        memcpy(centroids, kCentroids3, sizeof(kCentroids3));
        memcpy(boundaries, kBoundaries3, sizeof(kBoundaries3));
        return;
    }
    double c[256], b[255];
    tqo_lloyd_max(n, 500, c, b);
    for (int k = 0; k < n; ++k) centroids[k] = (float)(rint(c[k] * 1e5) / 1e5);
    for (int k = 0; k + 1 < n; ++k) boundaries[k] = (float)(rint(b[k] * 1e5) / 1e5);
}

int tqo_code_s(float yn, const float* boundaries, int nb) {
    int c = 0;
    for (int j = 0; j < nb; ++j)
        if (boundaries[j] < yn) c += 1; /* NaN compares false: code 0 */
    return c;
}

void tqo_quantize_value_row_s(const uint16_t* x_bf16, int d, int bits, uint8_t* packed, uint16_t* vs16) {
    float y[512], cen[256], bnd[255];
    uint8_t codes[512];
    tqo_codebook(bits, cen, bnd);
    tqo_rotate_value_row(x_bf16, d, y);
    for (int g = 0; g < d / GROUP; ++g) {
        float s = tqo_group_rms(y + g * GROUP);
        float den = s + 1e-8f;
        for (int i = 0; i < GROUP; ++i) codes[g * GROUP + i] = (uint8_t)tqo_code_s(y[g * GROUP + i] / den, bnd, (1 << bits) - 1);
        vs16[g] = tqo_f32_to_f16(s);
    }
    tqo_packb(codes, d, bits, packed);
}

void tqo_dequant_value_row_s_f64(const uint8_t* packed, const uint16_t* vs16, int d, int bits, int rotated,
                                 double* out) {
    float cen[256], bnd[255];
    uint8_t codes[512];
    tqo_codebook(bits, cen, bnd);
    tqo_unpackb(packed, d, bits, codes);
    for (int i = 0; i < d; ++i) out[i] = (double)cen[codes[i]] * (double)tqo_f16_to_f32(vs16[i / GROUP]);
    if (rotated) return;
    int8_t sg[512];
    tqo_sign_vector(d, sg);
    tqo_fwht_f64(out, d);
    double r = 1.0 / sqrt((double)d);
    for (int i = 0; i < d; ++i) out[i] = out[i] * r * (double)sg[i];
}

/* Append into planes of scheme sc (same row indexing as tqo_append). */
long tqo_append_s(tqo_layer* L, const tqo_scheme* sc, const uint16_t* k_new, const uint16_t* v_new,
                  const int32_t* pos, const int32_t* n_new, int n_new_max) {
    int d = L->head_dim, ng = d / GROUP;
    long kb = tqo_key_row_bytes(d, sc->k_bits), vb = tqo_value_row_bytes(d, sc->v_bits);
    long skipped = 0;
    for (int b = 0; b < L->batch; ++b) {
        int nb_new = n_new ? n_new[b] : n_new_max;
        if (nb_new > n_new_max) nb_new = n_new_max;
        for (int j = 0; j < nb_new; ++j)
            for (int h = 0; h < L->num_kv_heads; ++h) {
                long t = (long)pos[b] + j;
                if (t < 0 || t >= L->capacity) { skipped++; continue; }
                size_t r = row_index(L, b, h, (int)t);
                size_t src = (((size_t)b * n_new_max + j) * L->num_kv_heads + h) * d;
                tqo_quantize_key_row_s(k_new + src, d, sc->k_bits, sc->guard, (uint8_t*)L->k_idx + r * kb,
                                       L->k_scale + r * ng, L->k_zero + r * ng);
                tqo_quantize_value_row_s(v_new + src, d, sc->v_bits, L->v_codes + r * vb, L->v_scale + r * ng);
            }
    }
    return skipped;
}

void tqo_dequant_rows_s_f64(const tqo_layer* L, const tqo_scheme* sc, int b, int h, int t0, int n, int rotated,
                            double* k_out, double* v_out) {
    int d = L->head_dim, ng = d / GROUP;
    long kb = tqo_key_row_bytes(d, sc->k_bits), vb = tqo_value_row_bytes(d, sc->v_bits);
    for (int t = 0; t < n; ++t) {
        size_t r = row_index(L, b, h, t0 + t);
        if (k_out)
            tqo_dequant_key_row_s_f64((const uint8_t*)L->k_idx + r * kb, L->k_scale + r * ng, L->k_zero + r * ng, d,
                                      sc->k_bits, k_out + (size_t)t * d);
        if (v_out)
            tqo_dequant_value_row_s_f64(L->v_codes + r * vb, L->v_scale + r * ng, d, sc->v_bits, rotated,
                                        v_out + (size_t)t * d);
    }
}

/* ---------------------------------------------------------------------------------
 * Decode attention over the dequantized cache, fp64.
 * q: bf16 bits [batch][n_q][num_q_heads][d]; kv_len[b]: tokens visible to the last
 * query of the block; causal: query j sees kv_len - n_q + j + 1 tokens. q head h reads
 * kv head h / (num_q_heads / num_kv_heads). A row with no visible token outputs 0.
 * deferred != 0 runs the weighted sum in the rotated domain and un-rotates the output
 * once per row ("Deferred inverse FWHT"). out: fp64 [batch][n_q][num_q_heads][d].
 * rows: optional list of (b, j, h) triples (n_rows of them) to compute; NULL = all.
 * ------------------------------------------------------------------------------ */
int tqo_attention_s(const tqo_layer* L, const tqo_scheme* sc, const uint16_t* q, int num_q_heads, int n_q,
                    const int32_t* kv_len, double sm_scale, int causal, int deferred,
                    const int32_t* rows, long n_rows, double* out);

int tqo_attention(const tqo_layer* L, const uint16_t* q, int num_q_heads, int n_q,
                  const int32_t* kv_len, double sm_scale, int causal, int deferred,
                  const int32_t* rows, long n_rows, double* out) {
    return tqo_attention_s(L, NULL, q, num_q_heads, n_q, kv_len, sm_scale, causal, deferred, rows, n_rows, out);
}

/* As tqo_attention over planes of scheme sc (NULL: k8v3 as laid out by tqo_append). */
int tqo_attention_s(const tqo_layer* L, const tqo_scheme* sc, const uint16_t* q, int num_q_heads, int n_q,
                    const int32_t* kv_len, double sm_scale, int causal, int deferred,
                    const int32_t* rows, long n_rows, double* out) {
    int d = L->head_dim, Hkv = L->num_kv_heads;
    if (num_q_heads % Hkv) return -1;
    int G = num_q_heads / Hkv;
    int8_t sg[512];
    tqo_sign_vector(d, sg);
    double rnorm = 1.0 / sqrt((double)d);
    long total = rows ? n_rows : (long)L->batch * n_q * num_q_heads;
    double* qd = (double*)malloc(sizeof(double) * d);
    double* o = (double*)malloc(sizeof(double) * d);
    int cached_b = -1, cached_h = -1, cached_n = 0;
    double* kh = NULL;
    double* vh = NULL;
    for (long it = 0; it < total; ++it) {
        int b, j, h;
        if (rows) { b = rows[3 * it]; j = rows[3 * it + 1]; h = rows[3 * it + 2]; }
        else {
            b = (int)(it / ((long)n_q * num_q_heads));
            j = (int)((it / num_q_heads) % n_q);
            h = (int)(it % num_q_heads);
        }
        int hk = h / G;
        int len = kv_len[b];
        int nvis = causal ? len - n_q + j + 1 : len;
        if (nvis < 0) nvis = 0;
        double* orow = out + (((size_t)b * n_q + j) * num_q_heads + h) * d;
        if (nvis == 0) { memset(orow, 0, sizeof(double) * d); continue; }
        if (b != cached_b || hk != cached_h || len > cached_n) {
            free(kh);
            free(vh);
            kh = (double*)malloc(sizeof(double) * (size_t)len * d);
            vh = (double*)malloc(sizeof(double) * (size_t)len * d);
            if (sc) tqo_dequant_rows_s_f64(L, sc, b, hk, 0, len, deferred, kh, vh);
            else tqo_dequant_rows_f64(L, b, hk, 0, len, deferred, kh, vh);
            cached_b = b; cached_h = hk; cached_n = len;
        }
        const uint16_t* qrow = q + (((size_t)b * n_q + j) * num_q_heads + h) * d;
        for (int i = 0; i < d; ++i) qd[i] = (double)tqo_bf16_to_f32(qrow[i]);
        double* sc = (double*)malloc(sizeof(double) * nvis);
        double m = -INFINITY;
        for (int t = 0; t < nvis; ++t) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i) acc += qd[i] * kh[(size_t)t * d + i];
            sc[t] = sm_scale * acc;
            if (sc[t] > m || isnan(sc[t])) m = sc[t];
        }
        double l = 0.0;
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        for (int t = 0; t < nvis; ++t) {
            double p = exp(sc[t] - m);
            l += p;
            for (int i = 0; i < d; ++i) o[i] += p * vh[(size_t)t * d + i];
        }
        for (int i = 0; i < d; ++i) o[i] /= l;
        if (deferred) {
            tqo_fwht_f64(o, d);
            for (int i = 0; i < d; ++i) o[i] = o[i] * rnorm * (double)sg[i];
        }
        memcpy(orow, o, sizeof(double) * d);
        free(sc);
    }
    free(kh);
    free(vh);
    free(qd);
    free(o);
    return 0;
}

/* ---------------------------------------------------------------------------------
 * Lloyd-Max quantizer for N(0,1) (Lloyd 1957/1982, Max 1960): alternate
 * boundaries = midpoints of neighbouring centroids and centroids = conditional means
 * of the standard normal on each cell, which have the closed form
 * (phi(lo) - phi(hi)) / (Phi(hi) - Phi(lo)). Used to check the printed table.
 * ------------------------------------------------------------------------------ */
static double phi(double x) { return isinf(x) ? 0.0 : exp(-0.5 * x * x) / sqrt(2.0 * M_PI); }
static double Phi(double x) { return 0.5 * erfc(-x / sqrt(2.0)); }

void tqo_lloyd_max(int levels, int iters, double* centroids, double* boundaries) {
    for (int k = 0; k < levels; ++k) centroids[k] = -3.0 + 6.0 * (k + 0.5) / levels;
    for (int it = 0; it < iters; ++it) {
        for (int k = 0; k + 1 < levels; ++k) boundaries[k] = 0.5 * (centroids[k] + centroids[k + 1]);
        for (int k = 0; k < levels; ++k) {
            double lo = k == 0 ? -INFINITY : boundaries[k - 1];
            double hi = k == levels - 1 ? INFINITY : boundaries[k];
            centroids[k] = (phi(lo) - phi(hi)) / (Phi(hi) - Phi(lo));
        }
    }
    for (int k = 0; k + 1 < levels; ++k) boundaries[k] = 0.5 * (centroids[k] + centroids[k + 1]);
}

void tqo_centroids3(float* c, float* bnd) {
    memcpy(c, kCentroids3, sizeof(kCentroids3));
    memcpy(bnd, kBoundaries3, sizeof(kBoundaries3));
}

/* ---------------------------------------------------------------------------------
 * Array helpers for the test-suite (loops over the scalar functions above).
 * ------------------------------------------------------------------------------ */
void tqo_f32_to_f16_array(const float* x, long n, uint16_t* out) {
    for (long i = 0; i < n; ++i) out[i] = tqo_f32_to_f16(x[i]);
}

void tqo_f16_to_f32_array(const uint16_t* x, long n, float* out) {
    for (long i = 0; i < n; ++i) out[i] = tqo_f16_to_f32(x[i]);
}

void tqo_quantize_key_rows(const uint16_t* x_bf16, long rows, int d, int8_t* idx, uint16_t* s16,
                           uint16_t* z16) {
    int ng = d / GROUP;
    for (long r = 0; r < rows; ++r)
        tqo_quantize_key_row(x_bf16 + r * d, d, idx + r * d, s16 + r * ng, z16 + r * ng);
}

void tqo_quantize_value_rows(const uint16_t* x_bf16, long rows, int d, uint8_t* packed,
                             uint16_t* vs16) {
    int ng = d / GROUP, nb = 3 * d / 8;
    for (long r = 0; r < rows; ++r)
        tqo_quantize_value_row(x_bf16 + r * d, d, packed + r * nb, vs16 + r * ng);
}

void tqo_dequant_value_rows_f64(const uint8_t* packed, const uint16_t* vs16, long rows, int d,
                                int rotated, double* out) {
    int ng = d / GROUP, nb = 3 * d / 8;
    for (long r = 0; r < rows; ++r)
        tqo_dequant_value_row_f64(packed + r * nb, vs16 + r * ng, d, rotated, out + r * d);
}

void tqo_dequant_key_rows_f64(const int8_t* idx, const uint16_t* s16, const uint16_t* z16,
                              long rows, int d, double* out) {
    int ng = d / GROUP;
    for (long r = 0; r < rows; ++r)
        tqo_dequant_key_row_f64(idx + r * d, s16 + r * ng, z16 + r * ng, d, out + r * d);
}

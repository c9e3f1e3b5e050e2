/*
 * nvfp4_oracle.c -- plain, slow CPU oracle for the per-token NVFP4 W4A4 forward path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load this library.  It shares
 * no code, header, table or helper with the CUDA library; it reads bf16 bit
 * patterns and fp32 arrays handed to it by the caller and writes plain arrays.
 *
 * Every floating-point step is an IEEE binary32 operation with round to
 * nearest even (compiled with -O2 -ffp-contract=off, no fast-math), unless
 * it says fp64.  Each function names the passage of the source pages it
 * restates:
 *   [miniTE]   "miniTE Technical Report: Stable and Efficient Reinforcement
 *              Learning with Native NVFP4" (infix.io/research/miniTE)
 *   [4bitter]  "The 4-bitter Lesson" (humans& blog post)
 *   [TRIAGE]   the TRIAGE paper, section 2.3 "Low-Precision Rollout with NVFP4"
 *
 * Readings where the pages are silent (op order, ties, zero rows, sign of
 * zero, nibble order, scale-factor layout, router renormalisation) are the
 * ones written next to each function.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Formats                                                                   */
/* ------------------------------------------------------------------------ */

/* E2M1 magnitudes for the three low bits of a 4-bit code; bit 3 is the sign.
 * [miniTE] 2.2 (E2M1 value, decode x^ = q s_b s_g); [4bitter] "Four-Over-Six"
 * (grid 0, 0.5, 1, 1.5, 2, 3, 4, 6). */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_decode(uint8_t code) {
    double m = E2M1_MAG[code & 7];
    return (code & 8) ? -m : m;
}

/* E4M3 (OCP FP8): bias 7, 3 mantissa bits, subnormals m*2^-9, 0x7F/0xFF NaN,
 * no infinity, max finite 448.  [miniTE] 2.2 / 5.1 ("E4M3 scale for each
 * block of 16 elements"). */
double orc_e4m3_decode(uint8_t b) {
    int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);          /* 0.mmm * 2^-6 */
    else        v = ldexp((double)(8 + m), e - 10); /* 1.mmm * 2^(e-7) */
    return s ? -v : v;
}

/* Sorted table of the 127 finite non-negative E4M3 values, index == code. */
static double E4M3_POS[127];
static int e4m3_table_ready = 0;
static void e4m3_table_init(void) {
    if (e4m3_table_ready) return;
    for (int c = 0; c < 127; ++c) E4M3_POS[c] = orc_e4m3_decode((uint8_t)c);
    e4m3_table_ready = 1;
}

/* Non-negative fp32 -> E4M3 code: nearest finite value, ties to the even
 * code (even mantissa LSB), values above 448 saturate to 448 (0x7E),
 * subnormals kept.  Reading of "E4M3 block scale" with the rounding rule
 * round-to-nearest-even, saturating. */
uint8_t orc_e4m3_encode(float u) {
    double x = (double)u;
    int lo, hi;
    e4m3_table_init();
    if (!(x > 0.0)) return 0;             /* 0 (u is never negative here) */
    if (x >= 448.0) return 0x7E;
    /* binary search for the bracketing pair E4M3_POS[lo] <= x < E4M3_POS[hi] */
    lo = 0; hi = 126;
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (E4M3_POS[mid] <= x) lo = mid; else hi = mid;
    }
    {
        double dlo = x - E4M3_POS[lo], dhi = E4M3_POS[hi] - x;
        if (dlo < dhi) return (uint8_t)lo;
        if (dhi < dlo) return (uint8_t)hi;
        return (uint8_t)((lo & 1) == 0 ? lo : hi); /* tie: even code */
    }
}

/* fp32 -> E2M1 code: nearest grid value, ties to the even code, |v| > 6
 * saturates to 6, the sign bit always copies the sign of v (so -0 and small
 * negatives that round to zero give 0x8). */
uint8_t orc_e2m1_encode(float v) {
    uint8_t sign = signbit(v) ? 8 : 0;
    double a = fabs((double)v);
    int best = 0;
    double bestd = a;
    for (int i = 1; i < 8; ++i) {
        double d = fabs(a - E2M1_MAG[i]);
        if (d < bestd || (d == bestd && (i & 1) == 0)) { best = i; bestd = d; }
    }
    if (a > 6.0) best = 7;
    return (uint8_t)(sign | best);
}

/* bf16 bit pattern -> fp32 (exact). */
static float bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* fp64 -> bf16 bit pattern, round to nearest even, from the definition:
 * 8 significant bits for |x| >= 2^-126, quantum 2^-133 below it, overflow to
 * infinity past the largest finite bf16. */
uint16_t orc_bf16_from_f64(double x) {
    double a = fabs(x), q, r;
    int e;
    float f;
    uint32_t u;
    if (isnan(x)) return 0x7FC0;
    if (a == 0.0) return signbit(x) ? 0x8000 : 0x0000;
    if (a >= ldexp(1.0, -126)) {
        frexp(a, &e);               /* a = m * 2^e, 0.5 <= m < 1 */
        q = ldexp(a, 8 - e);        /* in [128, 256): exact scaling */
        q = nearbyint(q);           /* round to nearest even (default mode) */
        r = ldexp(q, e - 8);
    } else {
        q = nearbyint(ldexp(a, 133));
        r = ldexp(q, -133);
    }
    if (r > ldexp(255.0, 120)) r = INFINITY; /* largest finite bf16: 1.9921875 * 2^127 */
    f = (float)r;                   /* exact: r is representable in bf16 */
    memcpy(&u, &f, 4);
    u >>= 16;
    if (signbit(x)) u |= 0x8000u;
    return (uint16_t)u;
}

void orc_bf16_from_f64_array(const double* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_from_f64(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Quantization                                                              */
/* ------------------------------------------------------------------------ */

/* Per-token (per_tensor == 0) or per-tensor (per_tensor == 1) NVFP4
 * quantization of a bf16 matrix x [rows x cols] with row stride ld.
 *
 * [miniTE] 2.2: x^ = q * s_b * s_g, s_b an E4M3 scale per 16 elements, s_g an
 * fp32 outer scale per tensor, per expert or per row.  [miniTE] 2.3 and the
 * [4bitter] baseline recipe: per-token activation scale reduced over the
 * hidden dimension of one row; weights keep one fp32 scale per tensor.
 * [miniTE] 5.6: gs = gamax / 2688 (2688 = 6 * 448), all-zero rows give zero.
 * [miniTE] 5.3: the quantizer may reuse an amax computed by the producer
 * (amax_in, nullable; one value per row, or one value in per-tensor mode).
 *
 * Steps (reading of the missing display equation of [miniTE] 5.1, in this order):
 *   amax = max_j |x_j|                       (row, or whole tensor)
 *   s_g  = amax / 2688                        if s_g == 0: row is all zero
 *   t    = 6 * s_g
 *   per 16-block: bmax = max |x_j|; u = bmax / t; s_b = E4M3(u)
 *     s_b == 0: the 16 codes are 0x0 (block underflow)
 *     else d = s_b * s_g;  v_j = x_j * (1 / d)   when d is a normal fp32
 *                          v_j = x_j / d          when d is subnormal
 *     q_j = E2M1(v_j)
 * Outputs: codes [rows x cols/2] (element 2i in the low nibble of byte i),
 * sf_lin [rows x cols/16] one E4M3 byte per block (row-major, unswizzled),
 * scale [rows] (per-token) or [1] (per-tensor) holding s_g.
 * Requires cols % 16 == 0. */
void orc_quantize(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                  int per_tensor, const float* amax_in,
                  uint8_t* codes, uint8_t* sf_lin, float* scale) {
    const int64_t nblk = cols / 16;
    float tensor_amax = 0.0f;
    if (per_tensor) {
        if (amax_in) {
            tensor_amax = amax_in[0];
        } else {
            for (int64_t r = 0; r < rows; ++r)
                for (int64_t j = 0; j < cols; ++j) {
                    float a = fabsf(bf16_to_f32(x[r * ld + j]));
                    if (a > tensor_amax) tensor_amax = a;
                }
        }
    }
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* xr = x + r * ld;
        uint8_t* cr = codes + r * (cols / 2);
        uint8_t* sr = sf_lin + r * nblk;
        float amax, s_g, t;
        if (per_tensor) {
            amax = tensor_amax;
        } else if (amax_in) {
            amax = amax_in[r];
        } else {
            amax = 0.0f;
            for (int64_t j = 0; j < cols; ++j) {
                float a = fabsf(bf16_to_f32(xr[j]));
                if (a > amax) amax = a;
            }
        }
        s_g = amax / 2688.0f;
        if (per_tensor) { if (r == 0) scale[0] = s_g; } else scale[r] = s_g;
        if (s_g == 0.0f) {
            memset(cr, 0, (size_t)(cols / 2));
            memset(sr, 0, (size_t)nblk);
            continue;
        }
        t = 6.0f * s_g;
        for (int64_t b = 0; b < nblk; ++b) {
            float bmax = 0.0f, u, sbf, d, rcp = 0.0f;
            uint8_t sb, q[16];
            int use_div;
            for (int j = 0; j < 16; ++j) {
                float a = fabsf(bf16_to_f32(xr[b * 16 + j]));
                if (a > bmax) bmax = a;
            }
            u = bmax / t;
            sb = orc_e4m3_encode(u);
            sr[b] = sb;
            if (sb == 0) {
                memset(q, 0, sizeof q);
            } else {
                sbf = (float)orc_e4m3_decode(sb);
                d = sbf * s_g;
                use_div = !(d >= FLT_MIN);
                if (!use_div) rcp = 1.0f / d;
                for (int j = 0; j < 16; ++j) {
                    float xv = bf16_to_f32(xr[b * 16 + j]);
                    float v = use_div ? xv / d : xv * rcp;
                    q[j] = orc_e2m1_encode(v);
                }
            }
            for (int j = 0; j < 8; ++j)
                cr[b * 8 + j] = (uint8_t)(q[2 * j] | (q[2 * j + 1] << 4));
        }
    }
}

/* Four-over-six: per 16-block, the block max maps to 6 (the plain rule) or
 * to 4, whichever encodes the block with the smaller error; 4 only when its
 * error is strictly smaller.  [4bitter] "Four-Over-Six for RL Weights and
 * Activations": a value near 5/6 of the range can be off by 1/6 of the range
 * with max -> 6, by 1/8 with max -> 4; a candidate decodes as
 * fp4_value * fp8_scale * amax / (E2M1_MAXVAL * E4M3_4OVER6_MAXVAL); the
 * error of each candidate is summed per block (MSE or MAE) in fp32 against
 * the target scaled down by the inverse of that factor, in FP32 accumulation.
 *
 * Readings (the pages name but do not print them):
 *   E2M1_MAXVAL = 6, E4M3_4OVER6_MAXVAL = 256: the largest power of two whose
 *     3/2 multiple (the block scale of a max -> 4 candidate) stays within
 *     E4M3's 448.  So s_g = amax / 1536.
 *   inv = 1536 / amax (fp32 division), target t_j = x_j * inv (fp32).
 *   candidate c in {6, 4}: u = bmax / (c * s_g); s_b = E4M3(u); codes as in
 *     orc_quantize with d = s_b * s_g; dq_j = e2m1(q_j) * s_b (exact);
 *     diff_j = dq_j - t_j; err = sum over j = 0..15 in order of diff_j^2
 *     (err_kind 1, MSE) or |diff_j| (err_kind 2, MAE), each step one fp32
 *     operation (no fused multiply-add).
 *   The row amax, zero rows and per-tensor mode as in orc_quantize.
 * Outputs as orc_quantize, plus choice[rows x cols/16] = 4 or 6 (nullable). */
static void encode_block(const uint16_t* xb, float s_g, float t, uint8_t* sb_out, uint8_t q[16]) {
    float bmax = 0.0f, u, d, rcp = 0.0f;
    int use_div;
    uint8_t sb;
    for (int j = 0; j < 16; ++j) {
        float a = fabsf(bf16_to_f32(xb[j]));
        if (a > bmax) bmax = a;
    }
    u = bmax / t;
    sb = orc_e4m3_encode(u);
    *sb_out = sb;
    if (sb == 0) {
        memset(q, 0, 16);
        return;
    }
    d = (float)orc_e4m3_decode(sb) * s_g;
    use_div = !(d >= FLT_MIN);
    if (!use_div) rcp = 1.0f / d;
    for (int j = 0; j < 16; ++j) {
        float xv = bf16_to_f32(xb[j]);
        q[j] = orc_e2m1_encode(use_div ? xv / d : xv * rcp);
    }
}

static float block_error(const uint16_t* xb, uint8_t sb, const uint8_t q[16], float inv, int err_kind) {
    float sbf = (float)orc_e4m3_decode(sb), err = 0.0f;
    for (int j = 0; j < 16; ++j) {
        float dq = (float)orc_e2m1_decode(q[j]) * sbf;
        float tj = bf16_to_f32(xb[j]) * inv;
        float diff = dq - tj;
        err = err + (err_kind == 1 ? diff * diff : fabsf(diff));
    }
    return err;
}

void orc_quantize_46(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                     int per_tensor, const float* amax_in, int err_kind,
                     uint8_t* codes, uint8_t* sf_lin, float* scale, uint8_t* choice) {
    const int64_t nblk = cols / 16;
    float tensor_amax = 0.0f;
    if (per_tensor) {
        if (amax_in) {
            tensor_amax = amax_in[0];
        } else {
            for (int64_t r = 0; r < rows; ++r)
                for (int64_t j = 0; j < cols; ++j) {
                    float a = fabsf(bf16_to_f32(x[r * ld + j]));
                    if (a > tensor_amax) tensor_amax = a;
                }
        }
    }
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t* xr = x + r * ld;
        uint8_t* cr = codes + r * (cols / 2);
        uint8_t* sr = sf_lin + r * nblk;
        float amax, s_g, inv;
        if (per_tensor) {
            amax = tensor_amax;
        } else if (amax_in) {
            amax = amax_in[r];
        } else {
            amax = 0.0f;
            for (int64_t j = 0; j < cols; ++j) {
                float a = fabsf(bf16_to_f32(xr[j]));
                if (a > amax) amax = a;
            }
        }
        s_g = amax / 1536.0f;
        if (per_tensor) { if (r == 0) scale[0] = s_g; } else scale[r] = s_g;
        if (s_g == 0.0f) {
            memset(cr, 0, (size_t)(cols / 2));
            memset(sr, 0, (size_t)nblk);
            if (choice) memset(choice + r * nblk, 6, (size_t)nblk);
            continue;
        }
        inv = 1536.0f / amax;
        for (int64_t b = 0; b < nblk; ++b) {
            const uint16_t* xb = xr + b * 16;
            uint8_t sb6, sb4, q6[16], q4[16], *q;
            float e6, e4;
            int four;
            encode_block(xb, s_g, 6.0f * s_g, &sb6, q6);
            encode_block(xb, s_g, 4.0f * s_g, &sb4, q4);
            e6 = block_error(xb, sb6, q6, inv, err_kind);
            e4 = block_error(xb, sb4, q4, inv, err_kind);
            four = e4 < e6;
            q = four ? q4 : q6;
            sr[b] = four ? sb4 : sb6;
            if (choice) choice[r * nblk + b] = (uint8_t)(four ? 4 : 6);
            for (int j = 0; j < 8; ++j)
                cr[b * 8 + j] = (uint8_t)(q[2 * j] | (q[2 * j + 1] << 4));
        }
    }
}

/* Dequantize to fp64: out[r][j] = q * s_b * s_g (each product exact in fp64).
 * [miniTE] 2.2 decode rule. */
void orc_dequantize(const uint8_t* codes, const uint8_t* sf_lin, const float* scale,
                    int64_t rows, int64_t cols, int per_tensor, double* out) {
    const int64_t nblk = cols / 16;
    e4m3_table_init();
    for (int64_t r = 0; r < rows; ++r) {
        double sg = per_tensor ? (double)scale[0] : (double)scale[r];
        for (int64_t b = 0; b < nblk; ++b) {
            uint8_t s = sf_lin[r * nblk + b];
            double sb = s < 127 ? E4M3_POS[s] : orc_e4m3_decode(s);
            for (int64_t j = b * 16; j < b * 16 + 16; ++j) {
                uint8_t byte = codes[r * (cols / 2) + j / 2];
                uint8_t c = (j & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
                out[r * cols + j] = orc_e2m1_decode(c) * sb * sg;
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Scale-factor layout                                                       */
/* ------------------------------------------------------------------------ */

/* Byte offset of block scale (r, c) in the swizzled layout consumed by
 * block-scaled tensor-core MMA.  The pages only say scales are moved into the
 * MMA layout ([miniTE] 5.4 "scale-layout transfer"); the layout itself is the
 * publicly documented block-scale layout for 16-element blocks: the
 * [rows x cols/16] matrix is zero-padded to a multiple of 128 rows and 4
 * columns, cut into 128x4 tiles of 512 bytes stored tile-row-major (the tiles
 * of one 128-row band are consecutive), and inside a tile
 * offset = (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4). */
int64_t orc_sf_offset(int64_t r, int64_t c, int64_t sf_cols) {
    int64_t sp = (sf_cols + 3) / 4 * 4;
    return ((r / 128) * (sp / 4) + c / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4);
}

int64_t orc_sf_bytes(int64_t rows, int64_t sf_cols) {
    return (rows + 127) / 128 * 128 * ((sf_cols + 3) / 4 * 4);
}

/* sf_lin [rows x sf_cols] -> swizzled buffer (orc_sf_bytes bytes), padding 0.
 * row_map (nullable) gives the destination row of each source row. */
void orc_sf_swizzle(const uint8_t* sf_lin, int64_t rows, int64_t sf_cols,
                    const int64_t* row_map, int64_t dst_rows, uint8_t* out) {
    memset(out, 0, (size_t)orc_sf_bytes(dst_rows, sf_cols));
    for (int64_t r = 0; r < rows; ++r) {
        int64_t dr = row_map ? row_map[r] : r;
        for (int64_t c = 0; c < sf_cols; ++c)
            out[orc_sf_offset(dr, c, sf_cols)] = sf_lin[r * sf_cols + c];
    }
}

/* Inverse: read the rows listed in row_map (or 0..rows-1) back to linear. */
void orc_sf_unswizzle(const uint8_t* sw, int64_t rows, int64_t sf_cols,
                      const int64_t* row_map, uint8_t* sf_lin) {
    for (int64_t r = 0; r < rows; ++r) {
        int64_t sr = row_map ? row_map[r] : r;
        for (int64_t c = 0; c < sf_cols; ++c)
            sf_lin[r * sf_cols + c] = sw[orc_sf_offset(sr, c, sf_cols)];
    }
}

/* ------------------------------------------------------------------------ */
/* Routing                                                                   */
/* ------------------------------------------------------------------------ */

/* Top-k routing over E experts for T tokens.  z_e = logit_e + bias_e (fp32);
 * the k largest z in descending order, ties to the lower expert index;
 * weights are the softmax over the k selected z, in fp64 (softmax over all E,
 * top-k, then renormalising to sum 1 gives the same numbers because the full
 * denominator cancels).  Router: top-8 of 128 experts ([miniTE] 6.4, D15
 * profiles: "top-k=8", 128 experts). */
void orc_route(const float* logits, const float* bias, int64_t T, int E, int k,
               int32_t* ids, double* w, float* z_out) {
    float* z = (float*)malloc(sizeof(float) * (size_t)E);
    char* taken = (char*)malloc((size_t)E);
    for (int64_t t = 0; t < T; ++t) {
        double denom = 0.0, zmax;
        for (int e = 0; e < E; ++e) { z[e] = logits[t * E + e] + bias[e]; taken[e] = 0; }
        if (z_out) for (int e = 0; e < E; ++e) z_out[t * E + e] = z[e];
        for (int s = 0; s < k; ++s) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || z[e] > z[best]) best = e; /* strict >: lower index wins ties */
            }
            taken[best] = 1;
            ids[t * k + s] = best;
        }
        zmax = (double)z[ids[t * k]];
        for (int s = 0; s < k; ++s) denom += exp((double)z[ids[t * k + s]] - zmax);
        for (int s = 0; s < k; ++s) w[t * k + s] = exp((double)z[ids[t * k + s]] - zmax) / denom;
    }
    free(z);
    free(taken);
}

/* Routing metadata ([miniTE] 5.2: contiguous buffers, device-side expert
 * offsets, padding handled in the grouped path).
 *   cnt[e]      rows routed to expert e
 *   off[e]      exclusive prefix of cnt (E+1 entries)
 *   poff[e]     exclusive prefix of ceil(cnt/128)*128 (E+1 entries): first
 *               scale-factor row of expert e in the 128-row-padded layout
 *   perm[r]     = t*k + slot of the r-th row, rows ordered by expert and,
 *               within an expert, by ascending token index (stable)
 *   inv[t*k+s]  = r such that perm[r] == t*k + s */
void orc_route_metadata(const int32_t* ids, int64_t T, int E, int k,
                        int32_t* cnt, int32_t* off, int32_t* poff,
                        int32_t* perm, int32_t* inv) {
    int64_t r = 0;
    for (int e = 0; e < E; ++e) cnt[e] = 0;
    for (int64_t i = 0; i < T * k; ++i) cnt[ids[i]]++;
    off[0] = 0; poff[0] = 0;
    for (int e = 0; e < E; ++e) {
        off[e + 1] = off[e] + cnt[e];
        poff[e + 1] = poff[e] + (cnt[e] + 127) / 128 * 128;
    }
    for (int e = 0; e < E; ++e)
        for (int64_t t = 0; t < T; ++t)
            for (int s = 0; s < k; ++s)
                if (ids[t * k + s] == e) { perm[r] = (int32_t)(t * k + s); inv[t * k + s] = (int32_t)r; ++r; }
}

/* ------------------------------------------------------------------------ */
/* MoE pieces                                                                */
/* ------------------------------------------------------------------------ */

/* SwiGLU on the FC1 output c [rows x 2F] = gate | up ([miniTE] 5.4: "C = gate
 * | up", "D = act(gate, up)"): D = gate * sigmoid(gate) * up in fp64, rounded
 * to bf16; amax[r] = max |D_bf16| over the row, the exact tensor that is then
 * quantized ([miniTE] 5.3, weighted SwiGLU + row amax).  prob (nullable)
 * multiplies row r by prob[r] before rounding (router weight applied at FC1). */
void orc_swiglu(const double* c, int64_t rows, int64_t F, const double* prob,
                uint16_t* d_bf16, float* amax) {
    for (int64_t r = 0; r < rows; ++r) {
        float m = 0.0f;
        for (int64_t j = 0; j < F; ++j) {
            double g = c[r * 2 * F + j], u = c[r * 2 * F + F + j];
            double v = g / (1.0 + exp(-g)) * u;
            uint16_t h;
            float a;
            if (prob) v *= prob[r];
            h = orc_bf16_from_f64(v);
            d_bf16[r * F + j] = h;
            a = fabsf(bf16_to_f32(h));
            if (a > m) m = a;
        }
        amax[r] = m;
    }
}

/* Router-weighted combine: out[t] = bf16( sum_s w[t,s] * y[inv[t,s]] ) in
 * fp64 (the weighted unpermute that ends the expert layer). */
void orc_combine(const double* y, int64_t H, const int32_t* inv, const double* w,
                 int64_t T, int k, uint16_t* out) {
    for (int64_t t = 0; t < T; ++t)
        for (int64_t h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int s = 0; s < k; ++s) acc += w[t * k + s] * y[(int64_t)inv[t * k + s] * H + h];
            out[t * H + h] = orc_bf16_from_f64(acc);
        }
}

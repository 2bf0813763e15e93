/*
 * kvq_oracle.c -- plain, slow CPU oracle for the block-quantised KV decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code, header, table or constant with the CUDA library.
 *
 * What it computes, and where the definition comes from:
 *
 *   - q8_0 and q4_0 block quantisers (32 values per block, one f16 scale) and the
 *     f16 control arm.  The pages fix only the storage cost of these formats:
 *     "HAL #582 -- per-layer KV compression study", section 1 (size model table:
 *     q8_0/q8_0 = 102 KiB/token = 8.5 bits per value, q4_0/q4_0 = 54 KiB/token =
 *     4.5 bits per value, f16 = 192 KiB/token).  The rounding rules are the plain
 *     reading of GGML-style q8_0 and q4_0 blocks, 32 values sharing one f16 scale:
 *       q8_0:  d = amax/127, codes round-half-away(x * (1/d)) in [-127, 127];
 *       q4_0:  m = the value of largest magnitude (first one on ties), d = m/-8,
 *              codes min(15, trunc(x * (1/d) + 8.5)) in [0, 15], two per byte
 *              (element i in the low nibble, element i+16 in the high nibble);
 *       f16:   round-to-nearest-even.
 *     All quantiser arithmetic is fp32 with one rounding per operation; the file
 *     must be compiled with -ffp-contract=off so that no multiply-add is fused.
 *
 *   - Exact softmax attention in fp64 over the dequantised cache (grouped-query:
 *     query head hq reads KV head hq / (Hq/Hkv)).  The pages require the fast
 *     reader to reproduce it: "logit-identical" / real_frac = 0 in HAL #582
 *     section 3b (finding 2) and section 5 (P0 note).
 *
 *   - The split-softmax merge (HAL #582 section 5, P2 read path: partials of key ranges
 *     combined without loss) in fp64.
 *
 *   - q4_1, q5_0, q5_1 (the further scalar types of the same study, section 5 P0 note
 *     and the P1 ladder, which prices q5_1 at 24 bytes per 32 values).  The pages name
 *     these GGML-style formats without defining them; the plain reading is:
 *       q4_1:  lo = min x, hi = max x, d = (hi - lo)/15, codes min(15, trunc((x - lo) *
 *              (1/d) + 0.5)) in [0, 15], stored d and lo as f16; x_hat = d*c + lo;
 *       q5_0:  as q4_0 with 5-bit codes: d = m/-16, codes min(31, trunc(x * (1/d) +
 *              16.5)) in [0, 31]; x_hat = d*(c - 16);
 *       q5_1:  as q4_1 with 5-bit codes: d = (hi - lo)/31, codes min(31, ...);
 *     every step one fp32 rounding (no fused multiply-add), (1/d) = 0 when d = 0.
 *
 * Natural (row-major) layouts are used throughout:
 *   q8_0 codes  int8   [rows][D]          scales f16 bits [rows][D/32]
 *   q4_0 bytes  uint8  [rows][D/2]        (block b = bytes 16b..16b+15)
 *   q5_0 codes  uint8  [rows][D]          (one code per value), scales [rows][D/32]
 *   q4_1, q5_1 codes uint8 [rows][D]      scales [rows][D/32][2] = (d, lo) f16 bits
 *   f16         uint16 [rows][D]
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define KVQO_F16 0
#define KVQO_Q8_0 1
#define KVQO_Q4_0 2
#define KVQO_Q4_1 3
#define KVQO_Q5_0 4
#define KVQO_Q5_1 5
#define QK 32

/* ---- f16 helpers: IEEE binary16, round-to-nearest-even via the compiler's _Float16 ---- */
static uint16_t f32_to_f16_bits(float x) {
    _Float16 h = (_Float16)x;
    uint16_t u;
    memcpy(&u, &h, 2);
    return u;
}

static double f16_bits_to_f64(uint16_t u) {
    _Float16 h;
    memcpy(&h, &u, 2);
    return (double)h;
}

int kvqo_abi_version(void) { return 1; }

/* ---- q8_0: one block of 32 fp32 values -> 32 int8 codes + f16 scale ---- */
static void quantize_block_q8_0(const float *x, int8_t *codes, uint16_t *scale) {
    float amax = 0.0f;
    for (int j = 0; j < QK; ++j) {
        float a = fabsf(x[j]);
        if (a > amax) amax = a;
    }
    float d = amax / 127.0f;
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    for (int j = 0; j < QK; ++j) {
        float y = x[j] * id;
        codes[j] = (int8_t)roundf(y); /* half away from zero */
    }
    *scale = f32_to_f16_bits(d);
}

/* ---- q4_0: one block -> 16 packed bytes + f16 scale ---- */
static void quantize_block_q4_0(const float *x, uint8_t *packed, uint16_t *scale) {
    float amax = 0.0f, m = 0.0f;
    for (int j = 0; j < QK; ++j) {
        float a = fabsf(x[j]);
        if (a > amax) { /* strict: the first index wins a tie */
            amax = a;
            m = x[j];
        }
    }
    float d = m / -8.0f;
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    int c[QK];
    for (int j = 0; j < QK; ++j) {
        float y = x[j] * id;   /* rounding 1 */
        float t = y + 8.5f;    /* rounding 2 (no fused multiply-add) */
        int v = (int)t;        /* t is in [0.5, 16.5]: truncation == floor */
        c[j] = v < 15 ? v : 15;
    }
    for (int i = 0; i < QK / 2; ++i)
        packed[i] = (uint8_t)(c[i] | (c[i + QK / 2] << 4));
    *scale = f32_to_f16_bits(d);
}

/* ---- q5_0: one block -> 32 codes in [0, 31] + f16 scale (q4_0 with 16 levels each side) ---- */
static void quantize_block_q5_0(const float *x, uint8_t *codes, uint16_t *scale) {
    float amax = 0.0f, m = 0.0f;
    for (int j = 0; j < QK; ++j) {
        float a = fabsf(x[j]);
        if (a > amax) {
            amax = a;
            m = x[j];
        }
    }
    float d = m / -16.0f;
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    for (int j = 0; j < QK; ++j) {
        float y = x[j] * id;
        float t = y + 16.5f;
        int v = (int)t;
        codes[j] = (uint8_t)(v < 31 ? v : 31);
    }
    *scale = f32_to_f16_bits(d);
}

/* ---- q4_1 / q5_1: one block -> codes in [0, levels] + f16 (d, lo): x_hat = d*c + lo ---- */
static void quantize_block_min(const float *x, int levels, uint8_t *codes, uint16_t *dm) {
    float lo = x[0], hi = x[0];
    for (int j = 1; j < QK; ++j) {
        if (x[j] < lo) lo = x[j];
        if (x[j] > hi) hi = x[j];
    }
    float d = (hi - lo) / (float)levels;
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    for (int j = 0; j < QK; ++j) {
        float t = x[j] - lo;   /* >= 0 */
        float y = t * id;
        float z = y + 0.5f;
        int v = (int)z;
        codes[j] = (uint8_t)(v < levels ? v : levels);
    }
    dm[0] = f32_to_f16_bits(d);
    dm[1] = f32_to_f16_bits(lo);
}

/* f16 scale values stored per 32-value block (2 for the types with a minimum). */
static int scales_per_block(int type) { return (type == KVQO_Q4_1 || type == KVQO_Q5_1) ? 2 : 1; }

/* Quantise n_rows rows of D fp32 values (D a multiple of 32). */
void kvqo_quantize_rows(int type, const float *x, int64_t n_rows, int D,
                        void *codes, uint16_t *scales, int n_threads) {
    const int nb = D / QK;
    int64_t r;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(static) if (n_threads != 1)
#endif
    for (r = 0; r < n_rows; ++r) {
        const float *xr = x + r * D;
        if (type == KVQO_F16) {
            uint16_t *o = (uint16_t *)codes + r * D;
            for (int j = 0; j < D; ++j) o[j] = f32_to_f16_bits(xr[j]);
        } else if (type == KVQO_Q8_0) {
            int8_t *o = (int8_t *)codes + r * D;
            for (int b = 0; b < nb; ++b)
                quantize_block_q8_0(xr + b * QK, o + b * QK, scales + r * nb + b);
        } else if (type == KVQO_Q4_0) {
            uint8_t *o = (uint8_t *)codes + r * (D / 2);
            for (int b = 0; b < nb; ++b)
                quantize_block_q4_0(xr + b * QK, o + b * (QK / 2), scales + r * nb + b);
        } else if (type == KVQO_Q5_0) {
            uint8_t *o = (uint8_t *)codes + r * D;
            for (int b = 0; b < nb; ++b)
                quantize_block_q5_0(xr + b * QK, o + b * QK, scales + r * nb + b);
        } else {
            uint8_t *o = (uint8_t *)codes + r * D;
            const int levels = type == KVQO_Q4_1 ? 15 : 31;
            for (int b = 0; b < nb; ++b)
                quantize_block_min(xr + b * QK, levels, o + b * QK, scales + (r * nb + b) * 2);
        }
    }
}

/* Dequantise one row into fp64: x_hat = f16(scale) * code (q8_0), f16(scale) * (code - 8) (q4_0). */
static void dequant_row(int type, const void *codes, const uint16_t *scales, int64_t row, int D,
                        double *out) {
    const int nb = D / QK;
    if (type == KVQO_F16) {
        const uint16_t *h = (const uint16_t *)codes + row * D;
        for (int j = 0; j < D; ++j) out[j] = f16_bits_to_f64(h[j]);
    } else if (type == KVQO_Q8_0) {
        const int8_t *q = (const int8_t *)codes + row * D;
        const uint16_t *s = scales + row * nb;
        for (int b = 0; b < nb; ++b) {
            double d = f16_bits_to_f64(s[b]);
            for (int j = 0; j < QK; ++j) out[b * QK + j] = d * (double)q[b * QK + j];
        }
    } else if (type == KVQO_Q4_0) {
        const uint8_t *p = (const uint8_t *)codes + row * (D / 2);
        const uint16_t *s = scales + row * nb;
        for (int b = 0; b < nb; ++b) {
            double d = f16_bits_to_f64(s[b]);
            for (int i = 0; i < QK / 2; ++i) {
                uint8_t byte = p[b * (QK / 2) + i];
                out[b * QK + i] = d * (double)((int)(byte & 0x0F) - 8);
                out[b * QK + i + QK / 2] = d * (double)((int)(byte >> 4) - 8);
            }
        }
    } else if (type == KVQO_Q5_0) {
        const uint8_t *c = (const uint8_t *)codes + row * D;
        const uint16_t *s = scales + row * nb;
        for (int b = 0; b < nb; ++b) {
            double d = f16_bits_to_f64(s[b]);
            for (int j = 0; j < QK; ++j) out[b * QK + j] = d * (double)((int)c[b * QK + j] - 16);
        }
    } else {
        const uint8_t *c = (const uint8_t *)codes + row * D;
        const uint16_t *s = scales + row * nb * 2;
        for (int b = 0; b < nb; ++b) {
            double d = f16_bits_to_f64(s[2 * b]), lo = f16_bits_to_f64(s[2 * b + 1]);
            for (int j = 0; j < QK; ++j) out[b * QK + j] = d * (double)c[b * QK + j] + lo;
        }
    }
}

void kvqo_dequantize_rows(int type, const void *codes, const uint16_t *scales, int64_t n_rows,
                          int D, double *out) {
    for (int64_t r = 0; r < n_rows; ++r) dequant_row(type, codes, scales, r, D, out + r * D);
}

/* Bytes per stored row of one cache plane (codes), and of its scales. */
static int64_t code_row_bytes(int type, int D) {
    return type == KVQO_F16 ? 2 * (int64_t)D : (type == KVQO_Q4_0 ? D / 2 : D);
}

/*
 * Softmax attention of one query head over keys [t0, t1) of one KV head, fp64.
 * Returns the unnormalised split triple: m = max_t s_t, l = sum_t exp(s_t - m),
 * o = sum_t exp(s_t - m) * v_hat_t, where s_t = scale * <q, k_hat_t>.
 * For an empty range: m = -inf, l = 0, o = 0.
 */
static void attend_range(int type_k, const void *k_codes, const uint16_t *k_scales,
                         int type_v, const void *v_codes, const uint16_t *v_scales,
                         int64_t row0, int64_t t0, int64_t t1, int D, const float *q,
                         double scale, double *o, double *m_out, double *l_out) {
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (t1 <= t0) {
        *m_out = -INFINITY;
        *l_out = 0.0;
        return;
    }
    double *s = (double *)malloc(sizeof(double) * (size_t)(t1 - t0));
    double *row = (double *)malloc(sizeof(double) * (size_t)D);
    double m = -INFINITY;
    for (int64_t t = t0; t < t1; ++t) {
        dequant_row(type_k, k_codes, k_scales, row0 + t, D, row);
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += (double)q[d] * row[d];
        s[t - t0] = scale * dot;
        if (s[t - t0] > m) m = s[t - t0];
    }
    double l = 0.0;
    for (int64_t t = t0; t < t1; ++t) {
        double p = exp(s[t - t0] - m);
        l += p;
        dequant_row(type_v, v_codes, v_scales, row0 + t, D, row);
        for (int d = 0; d < D; ++d) o[d] += p * row[d];
    }
    free(row);
    free(s);
    *m_out = m;
    *l_out = l;
}

/*
 * Decode attention for one sequence.
 *   q        fp32 [Hq][D]
 *   k_codes  [Hkv][cap][row bytes], k_scales [Hkv][cap][D/32 x scales per block]  (same for v)
 *   n        number of valid rows (n <= cap)
 *   out      fp64 [Hq][D] normalised output, lse fp64 [Hq] (natural log).
 * n == 0 gives out = 0 and lse = -inf.
 */
void kvqo_attention(int type_k, const void *k_codes, const uint16_t *k_scales, int type_v,
                    const void *v_codes, const uint16_t *v_scales, int n_kv_heads, int64_t cap,
                    int64_t n, int D, const float *q, int n_q_heads, float scale, double *out,
                    double *lse, int n_threads) {
    const int G = n_q_heads / n_kv_heads;
    int hq;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) if (n_threads != 1)
#endif
    for (hq = 0; hq < n_q_heads; ++hq) {
        const int h = hq / G;
        double m, l;
        double *o = out + (int64_t)hq * D;
        attend_range(type_k, k_codes, k_scales, type_v, v_codes, v_scales, (int64_t)h * cap, 0, n,
                     D, q + (int64_t)hq * D, (double)scale, o, &m, &l);
        if (n == 0) {
            lse[hq] = -INFINITY;
        } else {
            for (int d = 0; d < D; ++d) o[d] /= l;
            lse[hq] = m + log(l);
        }
    }
}

/* Split triples of one sequence over the key ranges given by bounds[0..S] (S ranges). */
void kvqo_attention_partials(int type_k, const void *k_codes, const uint16_t *k_scales,
                             int type_v, const void *v_codes, const uint16_t *v_scales,
                             int n_kv_heads, int64_t cap, int D, const float *q, int n_q_heads,
                             float scale, const int64_t *bounds, int S, double *part_o,
                             double *part_m, double *part_l) {
    const int G = n_q_heads / n_kv_heads;
    for (int hq = 0; hq < n_q_heads; ++hq) {
        const int h = hq / G;
        for (int s = 0; s < S; ++s) {
            int64_t idx = (int64_t)hq * S + s;
            attend_range(type_k, k_codes, k_scales, type_v, v_codes, v_scales, (int64_t)h * cap,
                         bounds[s], bounds[s + 1], D, q + (int64_t)hq * D, (double)scale,
                         part_o + idx * D, part_m + idx, part_l + idx);
        }
    }
}

/*
 * Merge of S split triples per row:
 *   M = max_s m_s,  w_s = exp(m_s - M),  out = sum_s w_s o_s / sum_s w_s l_s,
 *   lse = M + log(sum_s w_s l_s).   All splits empty -> out = 0, lse = -inf.
 */
void kvqo_combine(const double *part_o, const double *part_m, const double *part_l, int64_t rows,
                  int S, int D, double *out, double *lse) {
    for (int64_t r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (int s = 0; s < S; ++s)
            if (part_m[r * S + s] > M) M = part_m[r * S + s];
        double *o = out + r * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (M == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double L = 0.0;
        for (int s = 0; s < S; ++s) {
            double ms = part_m[r * S + s];
            if (ms == -INFINITY) continue;
            double w = exp(ms - M);
            L += w * part_l[r * S + s];
            for (int d = 0; d < D; ++d) o[d] += w * part_o[(r * S + s) * D + d];
        }
        for (int d = 0; d < D; ++d) o[d] /= L;
        lse[r] = M + log(L);
    }
}

int64_t kvqo_code_row_bytes(int type, int D) { return code_row_bytes(type, D); }
int kvqo_scales_per_block(int type) { return scales_per_block(type); }

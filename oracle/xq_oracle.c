/*
 * xq_oracle.c -- plain, slow, obviously-correct CPU oracle for the 4-bit
 * decode mat-vec on the integer route.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * CPU-baseline leg of bench.py may load this file's library.  The product
 * path (quantized_decode_mat_gb300) never calls it and shares no code, header,
 * constant or table with it: every layout number below is written out here
 * on purpose, independently of the CUDA sources.
 *
 * Sources (page title, section):
 *   [G]  "25 - Writing XPU Kernels" (The Cajeta Guide), section 25.2
 *        "Decode: one row, one wave, the bus is the ceiling" and example
 *        25.2.1 "an integer decode wave": the q8_K activation block (256 int8
 *        values, eight int32 sub-block sums at +256, one f32 scale at +288,
 *        320 bytes), the codebook block (f16 scale + 16 payload bytes, low
 *        nibbles are elements 0..15, high nibbles 16..31, nibble -> int8 via a
 *        16-entry table), the signed x signed integer dot, "reduce first,
 *        then scale once".
 *   [S]  "cajeta.xpu - one kernel, any device", section 2.3 "Coordinates,
 *        waves and collectives": the super-block stride 144 and the nibble
 *        group offset 16 + 32*g inside a super-block.
 *   [R]  "The kernel reference interpreter", section "Arithmetic": float32
 *        work is one rounding per operation with nothing contracted into an
 *        FMA; float16 rounds to nearest even; integers are exact.
 *
 * Readings where the pages are silent:
 *   - q8 scale rule: amax = max|x|, iscale = 127/amax (f32), q = clamp(
 *     rint(x*iscale), -127, 127) with round-half-even, d = amax/127 (f32);
 *     an all-zero block has d = 0 and q = 0; a NaN product gives q = 0.
 *   - q8 bytes 292..319 are written as zero.
 *   - Q4_K field layout (f16 d @0, f16 dmin @2, 12 bytes of 6-bit scales and
 *     mins @4, 128 nibble bytes @16) and the k-quant packing of the twelve
 *     scale bytes; nibble group g holds sub-block 2g in its low nibbles and
 *     sub-block 2g+1 in its high nibbles; w = d*sc*q - dmin*m.
 *   - The mat-vec result y is evaluated exactly in integers per block and then
 *     in binary64; that value is what the f32 GPU output is judged against.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared (no fast-math).
 * Planted-fault builds (-DORACLE_FAULT=k) exist only so that the tests can
 * prove that the pins catch each kind of mistake; see oracle_fault().
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#ifndef ORACLE_FAULT
#define ORACLE_FAULT 0
#endif

/* ---- layout, written out from [G] 25.2 / 25.2.1 and [S] 2.3 -------------- */
#define OQ8_VALUES 256      /* int8 values per activation block            */
#define OQ8_SUM_AT 256      /* eight int32 sub-block sums start here        */
#define OQ8_SCALE_AT 288    /* one f32 scale                                */
#define OQ8_BYTES 320       /* whole activation block                       */
#define OQ4K_BYTES 144      /* one super-block: 256 weights                 */
#define OQ4K_NIBBLES_AT 16  /* nibble payload starts after d, dmin, scales  */
#define OCB4_BYTES 18       /* codebook block: f16 scale + 16 payload bytes */
#define OCB4_WEIGHTS 32

int oracle_fault(void) { return ORACLE_FAULT; }

/* ---- little-endian field readers (byte order fixed by the format) -------- */
static uint16_t rd_u16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

static uint32_t rd_u32(const uint8_t *p) {
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) |
           ((uint32_t)p[3] << 24);
}

static void wr_u32(uint8_t *p, uint32_t v) {
    p[0] = (uint8_t)v;
    p[1] = (uint8_t)(v >> 8);
    p[2] = (uint8_t)(v >> 16);
    p[3] = (uint8_t)(v >> 24);
}

static int32_t rd_i32(const uint8_t *p) {
    uint32_t u = rd_u32(p);
    int32_t v;
    memcpy(&v, &u, 4);
    return v;
}

static float rd_f32(const uint8_t *p) {
    uint32_t u = rd_u32(p);
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* IEEE 754 binary16 -> binary64, from the format's definition: sign bit 15,
 * exponent bits 10..14 (bias 15), fraction bits 0..9; exponent 0 is the
 * subnormal range 2^-14 * f/1024; exponent 31 is inf/NaN.  Exact. */
double oracle_f16_to_f64(uint16_t h) {
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return s ? -v : v;
}

/* ---- q8 activation quantiser ([G] 25.2: 256 int8 values, eight sub-block
 * sums, one f32 scale, 320 bytes).  Rule: reading listed in the header. ---- */
static int8_t q8_round(float t) {
    if (t != t) return 0;                 /* NaN product (0 * inf)          */
    if (t >= 127.0f) return 127;
    if (t <= -127.0f) return -127;
#if ORACLE_FAULT == 5
    return (int8_t)roundf(t);             /* planted: ties away from zero   */
#else
    return (int8_t)rintf(t);              /* round half to even             */
#endif
}

void oracle_quantize_q8(const float *x, uint8_t *xq, int64_t cols, int64_t batch) {
    int64_t nb = cols / OQ8_VALUES;
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t blk = 0; blk < nb; ++blk) {
            const float *v = x + b * cols + blk * OQ8_VALUES;
            uint8_t *out = xq + (b * nb + blk) * OQ8_BYTES;
            float amax = 0.0f;
            for (int j = 0; j < OQ8_VALUES; ++j) {
                float a = fabsf(v[j]);
                if (a > amax) amax = a;
            }
            int8_t q[OQ8_VALUES];
            float d;
            if (amax == 0.0f) {
                for (int j = 0; j < OQ8_VALUES; ++j) q[j] = 0;
                d = 0.0f;
            } else {
                float iscale = 127.0f / amax;
                for (int j = 0; j < OQ8_VALUES; ++j) {
                    float t = v[j] * iscale;
                    q[j] = q8_round(t);
                }
#if ORACLE_FAULT == 8
                d = amax / 128.0f;        /* planted: wrong scale step      */
#else
                d = amax / 127.0f;
#endif
            }
            memset(out, 0, OQ8_BYTES);
            for (int j = 0; j < OQ8_VALUES; ++j) out[j] = (uint8_t)q[j];
            for (int s = 0; s < 8; ++s) {
                int32_t sum = 0;
                for (int i = 0; i < 32; ++i) sum += q[32 * s + i];
#if ORACLE_FAULT == 6
                int slot = (s + 1) & 7;   /* planted: sums in the wrong slot */
#else
                int slot = s;
#endif
                wr_u32(out + OQ8_SUM_AT + 4 * slot, (uint32_t)sum);
            }
            uint32_t du;
            memcpy(&du, &d, 4);
            wr_u32(out + OQ8_SCALE_AT, du);
        }
    }
}

/* Dequantised activation x_hat_j = d * q_j in binary64 (exact). */
void oracle_dequant_q8(const uint8_t *xq, double *out, int64_t cols, int64_t batch) {
    int64_t nb = cols / OQ8_VALUES;
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t blk = 0; blk < nb; ++blk) {
            const uint8_t *p = xq + (b * nb + blk) * OQ8_BYTES;
            double d = (double)rd_f32(p + OQ8_SCALE_AT);
            for (int j = 0; j < OQ8_VALUES; ++j)
                out[b * cols + blk * OQ8_VALUES + j] = d * (double)(int8_t)p[j];
        }
}

/* ---- Q4_K super-block unpack (144 bytes, 256 weights) --------------------
 * d = f16 @0, dmin = f16 @2, twelve packed scale bytes @4, nibbles @16.
 * Scales and mins, k-quant packing:
 *   j < 4 : sc_j = s[j] & 63,                        m_j = s[j+4] & 63
 *   j >= 4: sc_j = (s[j+4] & 15) | ((s[j-4] >> 6) << 4),
 *           m_j  = (s[j+4] >> 4) | ((s[j]   >> 6) << 4)
 * Nibbles: group g (0..3) is bytes 16+32g .. 16+32g+31 ([S] 2.3); its low
 * nibbles are weights 64g+i (sub-block 2g), its high nibbles 64g+32+i
 * (sub-block 2g+1). */
void oracle_q4k_unpack(const uint8_t *blk, double *d, double *dmin, uint8_t sc[8],
                       uint8_t m[8], uint8_t q[256]) {
    *d = oracle_f16_to_f64(rd_u16(blk));
    *dmin = oracle_f16_to_f64(rd_u16(blk + 2));
    const uint8_t *s = blk + 4;
    for (int j = 0; j < 4; ++j) {
        sc[j] = s[j] & 63;
        m[j] = s[j + 4] & 63;
    }
    for (int j = 4; j < 8; ++j) {
#if ORACLE_FAULT == 3
        m[j] = (uint8_t)((s[j + 4] & 15) | ((s[j - 4] >> 6) << 4));   /* planted */
        sc[j] = (uint8_t)((s[j + 4] >> 4) | ((s[j] >> 6) << 4));
#else
        sc[j] = (uint8_t)((s[j + 4] & 15) | ((s[j - 4] >> 6) << 4));
        m[j] = (uint8_t)((s[j + 4] >> 4) | ((s[j] >> 6) << 4));
#endif
    }
    const uint8_t *qs = blk + OQ4K_NIBBLES_AT;
    for (int g = 0; g < 4; ++g)
        for (int i = 0; i < 32; ++i) {
            uint8_t byte = qs[32 * g + i];
#if ORACLE_FAULT == 2
            q[64 * g + i] = byte >> 4;            /* planted: halves swapped */
            q[64 * g + 32 + i] = byte & 15;
#else
            q[64 * g + i] = byte & 15;
            q[64 * g + 32 + i] = byte >> 4;
#endif
        }
}

/* Dequantised weights w_j = d*sc_s*q_j - dmin*m_s in binary64, row-major. */
void oracle_dequant_q4k(const uint8_t *W, double *out, int64_t rows, int64_t cols) {
    int64_t nb = cols / 256;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t blk = 0; blk < nb; ++blk) {
            double d, dmin;
            uint8_t sc[8], m[8], q[256];
            oracle_q4k_unpack(W + (r * nb + blk) * OQ4K_BYTES, &d, &dmin, sc, m, q);
            for (int j = 0; j < 256; ++j) {
                int s = j / 32;
                out[r * cols + blk * 256 + j] = d * sc[s] * q[j] - dmin * m[s];
            }
        }
}

/* Per-sub-block integer dots dot[b][r][blk*8+s] = sum_i q_{32s+i} * xq_{32s+i}
 * (unsigned nibble x signed int8, exact in int32). */
void oracle_subdots_q4k(const uint8_t *W, const uint8_t *xq, int32_t *dots, int64_t rows,
                        int64_t cols, int64_t batch) {
    int64_t nb = cols / 256;
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t blk = 0; blk < nb; ++blk) {
                double d, dmin;
                uint8_t sc[8], m[8], q[256];
                oracle_q4k_unpack(W + (r * nb + blk) * OQ4K_BYTES, &d, &dmin, sc, m, q);
                const uint8_t *a = xq + (b * nb + blk) * OQ8_BYTES;
                for (int s = 0; s < 8; ++s) {
                    int32_t dot = 0;
                    for (int i = 0; i < 32; ++i)
                        dot += (int32_t)q[32 * s + i] * (int32_t)(int8_t)a[32 * s + i];
                    dots[(b * rows + r) * nb * 8 + blk * 8 + s] = dot;
                }
            }
}

/* Q4_K x q8 on the integer route ([G] 25.2: integer dot, then scale):
 *   y = sum_blk xs * ( d * S1 - dmin * S2 ),
 *   S1 = sum_s sc_s * dot_s,  S2 = sum_s m_s * bsum_s   (exact int64)
 * then binary64.  y_abs = sum_blk |xs*d*S1| + |xs*dmin*S2| (conditioning). */
void oracle_matvec_q4k(const uint8_t *W, const uint8_t *xq, double *y, double *y_abs,
                       int64_t rows, int64_t cols, int64_t batch) {
    int64_t nb = cols / 256;
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t r = 0; r < rows; ++r) {
            double acc = 0.0, aab = 0.0;
            for (int64_t blk = 0; blk < nb; ++blk) {
                double d, dmin;
                uint8_t sc[8], m[8], q[256];
                oracle_q4k_unpack(W + (r * nb + blk) * OQ4K_BYTES, &d, &dmin, sc, m, q);
                const uint8_t *a = xq + (b * nb + blk) * OQ8_BYTES;
                double xs = (double)rd_f32(a + OQ8_SCALE_AT);
                int64_t S1 = 0, S2 = 0;
                for (int s = 0; s < 8; ++s) {
                    int64_t dot = 0;
                    for (int i = 0; i < 32; ++i)
                        dot += (int64_t)q[32 * s + i] * (int64_t)(int8_t)a[32 * s + i];
                    S1 += (int64_t)sc[s] * dot;
                    S2 += (int64_t)m[s] * (int64_t)rd_i32(a + OQ8_SUM_AT + 4 * s);
                }
#if ORACLE_FAULT == 1
                S2 = 0;                                   /* planted: no min */
#endif
                double t1 = xs * (d * (double)S1);
#if ORACLE_FAULT == 7
                double t2 = xs * (dmin * (double)S2);     /* planted: sign   */
#else
                double t2 = -(xs * (dmin * (double)S2));
#endif
                acc += t1 + t2;
                aab += fabs(t1) + fabs(t2);
            }
            y[b * rows + r] = acc;
            if (y_abs) y_abs[b * rows + r] = aab;
        }
}

/* ---- nonlinear 4-bit codebook block (18 bytes, 32 weights) --------------
 * [G] 25.2.1: f16 scale then 16 payload bytes; element j < 16 is
 * kv[qs[j] & 15], element j >= 16 is kv[qs[j-16] >> 4]; kv is int8. */
void oracle_cb4_unpack(const uint8_t *blk, const int8_t kv[16], double *d, int8_t c[32]) {
    *d = oracle_f16_to_f64(rd_u16(blk));
    const uint8_t *qs = blk + 2;
    for (int j = 0; j < 16; ++j) {
#if ORACLE_FAULT == 4
        c[j] = kv[qs[j] >> 4];                    /* planted: halves swapped */
        c[j + 16] = kv[qs[j] & 15];
#else
        c[j] = kv[qs[j] & 15];
        c[j + 16] = kv[qs[j] >> 4];
#endif
    }
}

void oracle_dequant_cb4(const uint8_t *W, const int8_t kv[16], double *out, int64_t rows,
                        int64_t cols) {
    int64_t bpr = cols / OCB4_WEIGHTS;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < bpr; ++k) {
            double d;
            int8_t c[32];
            oracle_cb4_unpack(W + (r * bpr + k) * OCB4_BYTES, kv, &d, c);
            for (int j = 0; j < 32; ++j) out[r * cols + k * 32 + j] = d * c[j];
        }
}

/* dot[b][r][k] = sum_j c_j * xq_{32k+j}, signed x signed, exact. */
void oracle_subdots_cb4(const uint8_t *W, const int8_t kv[16], const uint8_t *xq,
                        int32_t *dots, int64_t rows, int64_t cols, int64_t batch) {
    int64_t bpr = cols / OCB4_WEIGHTS, nb = cols / 256;
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t k = 0; k < bpr; ++k) {
                double d;
                int8_t c[32];
                oracle_cb4_unpack(W + (r * bpr + k) * OCB4_BYTES, kv, &d, c);
                /* block k sits in q8 block k/8, at sub-block k%8 */
                const uint8_t *a = xq + (b * nb + k / 8) * OQ8_BYTES + (k % 8) * 32;
                int32_t dot = 0;
                for (int j = 0; j < 32; ++j) dot += (int32_t)c[j] * (int32_t)(int8_t)a[j];
                dots[(b * rows + r) * bpr + k] = dot;
            }
}

/* y = sum_k d_k * xs_{k/8} * dot_k, binary64; y_abs = sum_k |d_k*xs*dot_k|. */
void oracle_matvec_cb4(const uint8_t *W, const int8_t kv[16], const uint8_t *xq, double *y,
                       double *y_abs, int64_t rows, int64_t cols, int64_t batch) {
    int64_t bpr = cols / OCB4_WEIGHTS, nb = cols / 256;
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t r = 0; r < rows; ++r) {
            double acc = 0.0, aab = 0.0;
            for (int64_t k = 0; k < bpr; ++k) {
                double d;
                int8_t c[32];
                oracle_cb4_unpack(W + (r * bpr + k) * OCB4_BYTES, kv, &d, c);
                const uint8_t *a0 = xq + (b * nb + k / 8) * OQ8_BYTES;
                const uint8_t *a = a0 + (k % 8) * 32;
                double xs = (double)rd_f32(a0 + OQ8_SCALE_AT);
                int64_t dot = 0;
                for (int j = 0; j < 32; ++j) dot += (int64_t)c[j] * (int64_t)(int8_t)a[j];
                double t = d * xs * (double)dot;
                acc += t;
                aab += fabs(t);
            }
            y[b * rows + r] = acc;
            if (y_abs) y_abs[b * rows + r] = aab;
        }
}

/* ---- RMSNorm + q8 pack ([G] 25.2.3 "a sum across the whole workgroup", and
 * [G] 25.5: a fused tail ends with the next layer's norm and pack) ---------
 * One workgroup of 256 work-items (eight waves of 32) per vector of n values:
 *   item t   : ss_t = x_t^2 + x_{t+256}^2 + ..., added in that order from 0
 *              (the strided loop of the guide's RmsNorm kernel)
 *   wave w   : its 32 partials are combined by a butterfly over lane offsets
 *              16, 8, 4, 2, 1 (lane l adds the value of lane l^off; all lanes
 *              end with the same value, since f32 addition commutes)
 *   workgroup: from 0, the eight wave partials are added, wave 0 first
 *   scale    : 1 / sqrt(total / n + 1e-5), then y_i = x_i * scale
 * Every f32 operation rounds once; nothing is contracted.  The guide fixes
 * the strided per-item loop and the wave-0-upward order across waves; inside
 * a wave it calls the reduction the hardware's, and the butterfly above is
 * this library's reading.  The workgroup size 256 is also a reading. */
#define ORMS_ITEMS 256
#define ORMS_WAVE 32

float oracle_rmsnorm_sumsq(const float *x, int64_t n) {
    float ss[ORMS_ITEMS];
    for (int t = 0; t < ORMS_ITEMS; ++t) {
        float s = 0.0f;
#if ORACLE_FAULT == 11
        int64_t last = t;                         /* planted: reversed loop  */
        while (last + ORMS_ITEMS < n) last += ORMS_ITEMS;
        for (int64_t i = last; i >= t && i < n; i -= ORMS_ITEMS) {
#else
        for (int64_t i = t; i < n; i += ORMS_ITEMS) {
#endif
            float sq = x[i] * x[i];
            s = s + sq;
        }
        ss[t] = s;
    }
    float total = 0.0f;
    for (int w = 0; w < ORMS_ITEMS / ORMS_WAVE; ++w) {
        float v[ORMS_WAVE], nv[ORMS_WAVE];
        for (int l = 0; l < ORMS_WAVE; ++l) v[l] = ss[w * ORMS_WAVE + l];
#if ORACLE_FAULT == 10
        float seq = 0.0f;                         /* planted: lanes in order */
        for (int l = 0; l < ORMS_WAVE; ++l) seq = seq + v[l];
        v[0] = seq;
#else
        for (int off = ORMS_WAVE / 2; off > 0; off >>= 1) {
            for (int l = 0; l < ORMS_WAVE; ++l) nv[l] = v[l] + v[l ^ off];
            for (int l = 0; l < ORMS_WAVE; ++l) v[l] = nv[l];
        }
#endif
        total = total + v[0];
    }
    return total;
}

float oracle_rmsnorm_scale(const float *x, int64_t n) {
    float total = oracle_rmsnorm_sumsq(x, n);
    float mean = total / (float)n;
#if ORACLE_FAULT == 9
    float den = sqrtf(mean);                      /* planted: eps dropped    */
#else
    float den = sqrtf(mean + 0.00001f);
#endif
    return 1.0f / den;
}

/* x [batch][cols] -> y = x*scale per vector (f32) and xq = q8 blocks of y. */
void oracle_rmsnorm_q8(const float *x, uint8_t *xq, float *y, int64_t cols, int64_t batch) {
    for (int64_t b = 0; b < batch; ++b) {
        const float *v = x + b * cols;
        float *yb = y + b * cols;
        float scale = oracle_rmsnorm_scale(v, cols);
        for (int64_t i = 0; i < cols; ++i) yb[i] = v[i] * scale;
        oracle_quantize_q8(yb, xq + b * (cols / OQ8_VALUES) * OQ8_BYTES, cols, 1);
    }
}

/* ---- resident row layout of the codebook format ([G] 25.4 "one layout, and
 * the copy that reads the lines"; [G] 25.2.1 walks it) -----------------------
 * A resident row holds the f16 scales of its bpr blocks (block j's at byte
 * 2j), padded to a whole dword, then the blocks' 16-byte payloads (block j's
 * at prefix + 16j):
 *   prefix = ((2*bpr + 3) / 4) * 4,   row_bytes = prefix + 16*bpr.
 * The repack is chunked as on the page: a call moves blocks block_base ..
 * block_base + n_blocks - 1 of the row-major raw matrix (src holds exactly
 * those blocks, 18 bytes each) into the resident matrix dst.  Pad bytes
 * (bpr odd) are left as they are. */
int64_t oracle_cb4r_prefix(int64_t bpr) { return ((bpr * 2 + 3) / 4) * 4; }

int64_t oracle_cb4r_row_bytes(int64_t bpr) { return oracle_cb4r_prefix(bpr) + 16 * bpr; }

void oracle_repack_cb4(const uint8_t *src, uint8_t *dst, int64_t block_base, int64_t n_blocks,
                       int64_t cols) {
    int64_t bpr = cols / OCB4_WEIGHTS;
    int64_t prefix = oracle_cb4r_prefix(bpr), row_bytes = oracle_cb4r_row_bytes(bpr);
    for (int64_t b = 0; b < n_blocks; ++b) {
        int64_t gb = block_base + b;
        int64_t row = gb / bpr, j = gb % bpr;
        const uint8_t *blk = src + b * OCB4_BYTES;
        uint8_t *rp = dst + row * row_bytes;
#if ORACLE_FAULT == 13
        rp[2 * j] = blk[1];                       /* planted: scale bytes swapped */
        rp[2 * j + 1] = blk[0];
#else
        rp[2 * j] = blk[0];
        rp[2 * j + 1] = blk[1];
#endif
#if ORACLE_FAULT == 12
        memcpy(rp + 16 * j, blk + 2, 16);         /* planted: prefix not skipped  */
#else
        memcpy(rp + prefix + 16 * j, blk + 2, 16);
#endif
    }
}

/* Dequantised resident matrix, read the way [G] 25.2.1's kernel walks it. */
void oracle_dequant_cb4r(const uint8_t *Wr, const int8_t kv[16], double *out, int64_t rows,
                         int64_t cols) {
    int64_t bpr = cols / OCB4_WEIGHTS;
    int64_t prefix = oracle_cb4r_prefix(bpr), row_bytes = oracle_cb4r_row_bytes(bpr);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < bpr; ++j) {
            const uint8_t *rp = Wr + r * row_bytes;
            double d = oracle_f16_to_f64(rd_u16(rp + 2 * j));
            const uint8_t *qs = rp + prefix + 16 * j;
            for (int m = 0; m < 16; ++m) {
                out[r * cols + 32 * j + m] = d * kv[qs[m] & 15];
                out[r * cols + 32 * j + 16 + m] = d * kv[qs[m] >> 4];
            }
        }
}

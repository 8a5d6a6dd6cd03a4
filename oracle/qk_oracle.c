/*
 * qk_oracle.c -- CPU oracle for the quantised-weight GEMV / GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * constant generator with the CUDA library.
 *
 * What it computes (plain definitions, no blocking, no fusion):
 *
 *   1. Every weight is decoded on its own to double (f64):
 *        Q8_0 : w = d * q                     (d fp16, q int8)
 *        Q4_K : w = d * sc * q - dmin * m     (d, dmin fp16; sc, m 6-bit; q 4-bit)
 *      The device keeps the weights quantised and decodes each block inside
 *      the matmul, checked against a host dequantisation (nurllama 0.18.1 API
 *      reference, model.nu; nurllama README, "How it is checked").
 *   2. y[b][r] = sum_{c<K} W[r][c] * x[b][c] in f64, c in natural order,
 *      W row-major with the column index fastest (nurllama 0.18.1 API
 *      reference, kernels.nu layout contract).
 *   3. S[b][r] = sum_{c<K} |W[r][c] * x[b][c]|, used for the error bound.
 *   4. For the bf16 prefill GEMM a second reference rounds each weight to
 *      fp32 then to bf16 and each activation to bf16 (round to nearest even)
 *      before the same f64 sum.
 *
 * Readings of the block layouts (the pages name the formats but never print
 * their bytes; these are the GGUF conventions raw block bytes must follow):
 *   Q8_0 (34 B): bytes 0-1 fp16 d (little endian), bytes 2..33 q[0..31] int8.
 *   Q4_K (144 B): bytes 0-1 fp16 d, 2-3 fp16 dmin, 4-15 scales[12],
 *     16-143 qs[128].  Sub-block j (0..7) covers weights 32j..32j+31.
 *     j < 4 : sc = scales[j] & 63, m = scales[j+4] & 63
 *     j >= 4: sc = (scales[j+4] & 15) | ((scales[j-4] >> 6) << 4)
 *             m  = (scales[j+4] >> 4) | ((scales[j]   >> 6) << 4)
 *     qs is 4 chunks of 32 bytes; weight i of sub-block 2c is the low
 *     nibble of qs[32c+i], weight i of sub-block 2c+1 its high nibble.
 *   Q6_K (210 B): ql[128] | qh[64] | scales[16] int8 | fp16 d; weight i of
 *     a super-block takes 4 low bits from ql and 2 high bits from qh (see
 *     qko_decode_q6_k_row), w = d * scales[i/16] * (q - 32).
 *   A row is ceil(K/QK) whole blocks; columns >= K are ignored.
 *   Parity unpinned: these layouts against real GGUF files (none is at hand).
 *   They are pinned only by single-field probes written by hand from the
 *   layouts above (the probe files under tests/golden).
 *
 * The fp16 and bf16 conversions are written from the IEEE 754 encodings.
 * Compile with -O2 and without -ffast-math.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QKO_Q8_0 0
#define QKO_Q4_K 1
#define QKO_Q6_K 2

/* ---------------------------------------------------------------- fp16 / bf16 */

/* IEEE 754 binary16 bit pattern -> double (exact for every pattern). */
double qko_fp16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

/* double -> binary16, round to nearest, ties to even (one rounding). */
uint16_t qko_f64_to_fp16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v)) return 0x7E00;
    if (isinf(a)) return sign | 0x7C00;
    if (a == 0.0) return sign;
    int e2;
    frexp(a, &e2);            /* a = f * 2^e2, f in [0.5, 1) -> exponent e = e2 - 1 */
    int e = e2 - 1;
    if (e < -14) {
        /* subnormal range: value = n * 2^-24, n <= 1024 (1024 rolls into the
           smallest normal, whose bit pattern is exactly 1024). */
        double n = nearbyint(ldexp(a, 24));
        return sign | (uint16_t)n;
    }
    double m = nearbyint(ldexp(a, 10 - e));      /* in [1024, 2048] */
    if (m == 2048.0) { m = 1024.0; e += 1; }
    if (e > 15) return sign | 0x7C00;
    return sign | (uint16_t)((e + 15) << 10) | (uint16_t)((int)m - 1024);
}

/* fp32 -> bfloat16 bit pattern, round to nearest, ties to even. */
uint16_t qko_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))
        return (uint16_t)((u >> 16) | 0x0040);     /* quiet NaN */
    uint32_t keep = u >> 16;                       /* truncated bf16 */
    uint32_t rest = u & 0xFFFFu;                   /* dropped 16 bits */
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u)))
        keep += 1;                                 /* may carry into the exponent: correct */
    return (uint16_t)keep;
}

double qko_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* ---------------------------------------------------------------- decoders */

static uint16_t le16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* One Q8_0 row (ceil(K/32) blocks of 34 bytes) -> w[0..K). */
void qko_decode_q8_0_row(const uint8_t *row, int64_t K, double *w)
{
    for (int64_t c = 0; c < K; ++c) {
        const uint8_t *blk = row + (c / 32) * 34;
        double d = qko_fp16_to_f64(le16(blk));
        int8_t q = (int8_t)blk[2 + (c % 32)];
        w[c] = d * (double)q;
    }
}

/* 6-bit scale and min of sub-block j of a Q4_K super-block. */
static void q4_k_scale_min(const uint8_t *scales, int j, int *sc, int *m)
{
    if (j < 4) {
        *sc = scales[j] & 63;
        *m = scales[j + 4] & 63;
    } else {
        *sc = (scales[j + 4] & 15) | ((scales[j - 4] >> 6) << 4);
        *m = (scales[j + 4] >> 4) | ((scales[j] >> 6) << 4);
    }
}

/* One Q4_K row (ceil(K/256) super-blocks of 144 bytes) -> w[0..K). */
void qko_decode_q4_k_row(const uint8_t *row, int64_t K, double *w)
{
    for (int64_t c = 0; c < K; ++c) {
        const uint8_t *blk = row + (c / 256) * 144;
        int t = (int)(c % 256);           /* index inside the super-block */
        int j = t / 32;                   /* sub-block */
        int i = t % 32;                   /* index inside the sub-block */
        double d = qko_fp16_to_f64(le16(blk));
        double dmin = qko_fp16_to_f64(le16(blk + 2));
        int sc, m;
        q4_k_scale_min(blk + 4, j, &sc, &m);
        uint8_t byte = blk[16 + 32 * (j / 2) + i];
        int q = (j % 2 == 0) ? (byte & 15) : (byte >> 4);
        w[c] = d * (double)sc * (double)q - dmin * (double)m;
    }
}

/*
 * Q6_K (210 B per 256 weights): ql[128] | qh[64] | scales[16] int8 | fp16 d.
 * Weight i: n = i/128, cc = i%128, t = cc/32, l = cc%32; the low 4 bits are
 * the low (t < 2) or high (t >= 2) nibble of ql[64n + l + 32*(t%2)], the
 * high 2 bits are (qh[32n + l] >> 2t) & 3; w = d * scales[i/16] * (q - 32).
 */
void qko_decode_q6_k_row(const uint8_t *row, int64_t K, double *w)
{
    for (int64_t c = 0; c < K; ++c) {
        const uint8_t *blk = row + (c / 256) * 210;
        const int i = (int)(c % 256);
        const int n = i / 128, cc = i % 128, t = cc / 32, l = cc % 32;
        const uint8_t lbyte = blk[64 * n + l + 32 * (t % 2)];
        const int lo = t < 2 ? (lbyte & 15) : (lbyte >> 4);
        const int hi = (blk[128 + 32 * n + l] >> (2 * t)) & 3;
        const int q = lo | (hi << 4);
        const int sc = (int)(int8_t)blk[192 + i / 16];
        const double d = qko_fp16_to_f64(le16(blk + 208));
        w[c] = d * (double)sc * (double)(q - 32);
    }
}

static int64_t row_stride(int fmt, int64_t K)
{
    if (fmt == QKO_Q8_0) return ((K + 31) / 32) * 34;
    if (fmt == QKO_Q6_K) return ((K + 255) / 256) * 210;
    return ((K + 255) / 256) * 144;
}

static void decode_row(int fmt, const uint8_t *row, int64_t K, double *w)
{
    if (fmt == QKO_Q8_0) qko_decode_q8_0_row(row, K, w);
    else if (fmt == QKO_Q6_K) qko_decode_q6_k_row(row, K, w);
    else qko_decode_q4_k_row(row, K, w);
}

/* Decode whole rows: out[i*K + c] = W[rows[i]][c]. */
int qko_decode_rows(int fmt, const uint8_t *wq, int64_t K, const int64_t *rows,
                    int64_t n_rows, double *out)
{
    if (fmt != QKO_Q8_0 && fmt != QKO_Q4_K && fmt != QKO_Q6_K) return 1;
    int64_t stride = row_stride(fmt, K);
    for (int64_t i = 0; i < n_rows; ++i)
        decode_row(fmt, wq + rows[i] * stride, K, out + i * K);
    return 0;
}

/* ---------------------------------------------------------------- GEMV */

/*
 * y[b*n_rows + i] = sum_c W[rows[i]][c] * x[b*K + c]   (f64, natural order)
 * s[b*n_rows + i] = sum_c |W[rows[i]][c] * x[b*K + c]|
 * The batched form is the "several positions per launch, each weight read
 * once per chunk" matvec (nurllama 0.18.1 API reference, model.nu chunked
 * prefill); here it is just the same dot repeated for every position.
 */
int qko_gemv(int fmt, const uint8_t *wq, int64_t K, const int64_t *rows, int64_t n_rows,
             const float *x, int64_t batch, double *y, double *s)
{
    if (fmt != QKO_Q8_0 && fmt != QKO_Q4_K && fmt != QKO_Q6_K) return 1;
    int64_t stride = row_stride(fmt, K);
    double *w = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    if (!w) return 2;
    for (int64_t i = 0; i < n_rows; ++i) {
        decode_row(fmt, wq + rows[i] * stride, K, w);
        for (int64_t b = 0; b < batch; ++b) {
            double acc = 0.0, mag = 0.0;
            for (int64_t c = 0; c < K; ++c) {
                double p = w[c] * (double)x[b * K + c];
                acc += p;
                mag += fabs(p);
            }
            y[b * n_rows + i] = acc;
            if (s) s[b * n_rows + i] = mag;
        }
    }
    free(w);
    return 0;
}

/*
 * Batched expert matvec: "one batched matvec over all n_assign expert
 * assignments.  Output row a uses expert expid_dev[a] and input row a/xk of
 * x" (nurllama 0.18.1 API reference, kernels.nu `lk_matvec_experts`), the
 * experts of a projection living in one 3-D tensor [n_experts][rows][K]
 * evaluated as row ranges (nurllama README, "What it runs", llada2).  For
 * a < n_assign and r < rows:
 *   y[a][r] = sum_c W[expid[a]*rows + r][c] * x[a / xk][c]     (f64)
 * s[a][r] the magnitude sum.  Returns 3 if an expert id is out of range.
 */
int qko_experts(int fmt, const uint8_t *wq, int64_t n_experts, int64_t rows, int64_t K, const float *x,
                int64_t xk, const int32_t *expid, int64_t n_assign, double *y, double *s)
{
    if (xk < 1) return 4;
    int64_t *idx = (int64_t *)malloc(sizeof(int64_t) * (size_t)(rows > 0 ? rows : 1));
    if (!idx) return 2;
    for (int64_t a = 0; a < n_assign; ++a) {
        const int64_t e = expid[a];
        if (e < 0 || e >= n_experts) {
            free(idx);
            return 3;
        }
        for (int64_t r = 0; r < rows; ++r) idx[r] = e * rows + r;
        const int rc = qko_gemv(fmt, wq, K, idx, rows, x + (a / xk) * K, 1, y + a * rows, s ? s + a * rows : NULL);
        if (rc) {
            free(idx);
            return rc;
        }
    }
    free(idx);
    return 0;
}

/* silu(z) = z * sigma(z) = z / (1 + e^-z) */
static double silu(double z) { return z / (1.0 + exp(-z)); }

/*
 * Fused gate/up matvec with the SwiGLU product -- the decode FFN of the llama
 * shape is a SwiGLU FFN (nurllama README, "What it runs"); silumul computes
 * g <- silu(g) * u (nurllama 0.18.1 API reference, kernels.nu `lk_silumul`,
 * beside `lk_gelumul`), and loom's decode matvecs fold it into the gate/up
 * matvec (loom-port-llm SKILL.md, "Kernel inventory"); gate and up may be row ranges of one tensor (the
 * phi3 ffn_up).  For p < n:
 *   g[b][p] = sum_c W[gate_rows[p]][c] x[b][c]
 *   u[b][p] = sum_c W[up_rows[p]][c]   x[b][c]
 *   h[b][p] = silu(g) * u,   silu(z) = z / (1 + e^-z)   (all f64)
 * g, u and their magnitude sums sg, su (layout [batch][n]) are returned for
 * the error bound.
 */
int qko_swiglu(int fmt, const uint8_t *wq, int64_t K, const int64_t *gate_rows, const int64_t *up_rows,
               int64_t n, const float *x, int64_t batch, double *h, double *g, double *u, double *sg, double *su)
{
    int rc = qko_gemv(fmt, wq, K, gate_rows, n, x, batch, g, sg);
    if (rc) return rc;
    rc = qko_gemv(fmt, wq, K, up_rows, n, x, batch, u, su);
    if (rc) return rc;
    for (int64_t i = 0; i < batch * n; ++i) h[i] = silu(g[i]) * u[i];
    return 0;
}

/*
 * bf16 reference of the prefill GEMM: each weight is rounded to fp32 and then
 * to bf16, each activation to bf16 (both round-to-nearest-even), and the
 * products are summed in f64 in natural order.  Layout as qko_gemv with
 * M token rows in place of the batch.
 */
int qko_gemm_bf16(int fmt, const uint8_t *wq, int64_t K, const int64_t *rows, int64_t n_rows,
                  const float *x, int64_t M, double *y, double *s)
{
    if (fmt != QKO_Q8_0 && fmt != QKO_Q4_K && fmt != QKO_Q6_K) return 1;
    int64_t stride = row_stride(fmt, K);
    double *w = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    double *xb = (double *)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    if (!w || !xb) { free(w); free(xb); return 2; }
    for (int64_t e = 0; e < M * K; ++e) xb[e] = qko_bf16_to_f64(qko_f32_to_bf16(x[e]));
    for (int64_t i = 0; i < n_rows; ++i) {
        decode_row(fmt, wq + rows[i] * stride, K, w);
        for (int64_t c = 0; c < K; ++c)
            w[c] = qko_bf16_to_f64(qko_f32_to_bf16((float)w[c]));
        for (int64_t b = 0; b < M; ++b) {
            double acc = 0.0, mag = 0.0;
            for (int64_t c = 0; c < K; ++c) {
                double p = w[c] * xb[b * K + c];
                acc += p;
                mag += fabs(p);
            }
            y[b * n_rows + i] = acc;
            if (s) s[b * n_rows + i] = mag;
        }
    }
    free(w);
    free(xb);
    return 0;
}

/*
 * The SwiGLU form of the bf16 prefill GEMM (the swiglu mode beside store and
 * acc in loom's gen_gemm.py, loom-port-llm SKILL.md, "What the starter
 * generates"): g and u are the bf16 references of qko_gemm_bf16 for the gate
 * and up rows, h = silu(g) * u in f64 (layout [M][n]).
 */
int qko_swiglu_gemm_bf16(int fmt, const uint8_t *wq, int64_t K, const int64_t *gate_rows, const int64_t *up_rows,
                         int64_t n, const float *x, int64_t M, double *h, double *g, double *u, double *sg,
                         double *su)
{
    int rc = qko_gemm_bf16(fmt, wq, K, gate_rows, n, x, M, g, sg);
    if (rc) return rc;
    rc = qko_gemm_bf16(fmt, wq, K, up_rows, n, x, M, u, su);
    if (rc) return rc;
    for (int64_t i = 0; i < M * n; ++i) h[i] = silu(g[i]) * u[i];
    return 0;
}

/* ---------------------------------------------------------------- quantisers */

/*
 * Q8_0 encoder for round-trip checks (the nurllama README checks Q8_0
 * against its error bounds, "How it is checked").  Per 32-weight block: d = fp16(amax / 127),
 * q = clamp(round_half_even(w / d), -127, 127); an all-zero block gets
 * d = 0 and q = 0.  Columns >= K are encoded as zero.
 */
void qko_quantise_q8_0_row(const double *w, int64_t K, uint8_t *out)
{
    int64_t nb = (K + 31) / 32;
    for (int64_t bi = 0; bi < nb; ++bi) {
        double v[32];
        double amax = 0.0;
        for (int i = 0; i < 32; ++i) {
            int64_t c = bi * 32 + i;
            v[i] = c < K ? w[c] : 0.0;
            if (fabs(v[i]) > amax) amax = fabs(v[i]);
        }
        uint16_t dh = qko_f64_to_fp16(amax / 127.0);
        double d = qko_fp16_to_f64(dh);
        uint8_t *blk = out + bi * 34;
        blk[0] = (uint8_t)(dh & 0xFF);
        blk[1] = (uint8_t)(dh >> 8);
        for (int i = 0; i < 32; ++i) {
            double q = d > 0.0 ? nearbyint(v[i] / d) : 0.0;
            if (q > 127.0) q = 127.0;
            if (q < -127.0) q = -127.0;
            blk[2 + i] = (uint8_t)(int8_t)q;
        }
    }
}

/*
 * Q4_K encoder for round-trip checks (a plain min/max reading; the pages
 * give no quantiser).  Per 32-weight sub-block j: lo = min(0, min w),
 * hi = max w, scale_j = (hi - lo)/15, min_j = -lo.  Then
 * d = fp16(max scale_j / 63), dmin = fp16(max min_j / 63),
 * sc_j = clamp(round(scale_j / d), 0, 63), m_j = clamp(round(min_j / dmin), 0, 63),
 * and each q is the nearest of the 16 values d*sc_j*q - dmin*m_j (ties to
 * the lower q).  Columns >= K are encoded from zeros.
 */
void qko_quantise_q4_k_row(const double *w, int64_t K, uint8_t *out)
{
    int64_t nb = (K + 255) / 256;
    for (int64_t bi = 0; bi < nb; ++bi) {
        double v[256];
        for (int t = 0; t < 256; ++t) {
            int64_t c = bi * 256 + t;
            v[t] = c < K ? w[c] : 0.0;
        }
        double scale[8], mn[8], smax = 0.0, mmax = 0.0;
        for (int j = 0; j < 8; ++j) {
            double lo = 0.0, hi = v[32 * j];
            for (int i = 0; i < 32; ++i) {
                double a = v[32 * j + i];
                if (a < lo) lo = a;
                if (a > hi) hi = a;
            }
            scale[j] = (hi - lo) / 15.0;
            mn[j] = -lo;
            if (scale[j] > smax) smax = scale[j];
            if (mn[j] > mmax) mmax = mn[j];
        }
        uint16_t dh = qko_f64_to_fp16(smax / 63.0);
        uint16_t mh = qko_f64_to_fp16(mmax / 63.0);
        double d = qko_fp16_to_f64(dh), dmin = qko_fp16_to_f64(mh);
        int sc[8], m[8];
        for (int j = 0; j < 8; ++j) {
            double a = d > 0.0 ? nearbyint(scale[j] / d) : 0.0;
            double b = dmin > 0.0 ? nearbyint(mn[j] / dmin) : 0.0;
            sc[j] = a < 0.0 ? 0 : (a > 63.0 ? 63 : (int)a);
            m[j] = b < 0.0 ? 0 : (b > 63.0 ? 63 : (int)b);
        }
        uint8_t *blk = out + bi * 144;
        blk[0] = (uint8_t)(dh & 0xFF);
        blk[1] = (uint8_t)(dh >> 8);
        blk[2] = (uint8_t)(mh & 0xFF);
        blk[3] = (uint8_t)(mh >> 8);
        uint8_t *scales = blk + 4;
        for (int j = 0; j < 4; ++j) {
            scales[j] = (uint8_t)((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
            scales[j + 4] = (uint8_t)((m[j] & 63) | ((m[j + 4] >> 4) << 6));
            scales[j + 8] = (uint8_t)((sc[j + 4] & 15) | ((m[j + 4] & 15) << 4));
        }
        uint8_t *qs = blk + 16;
        memset(qs, 0, 128);
        for (int t = 0; t < 256; ++t) {
            int j = t / 32, i = t % 32;
            int best = 0;
            double best_err = INFINITY;
            for (int q = 0; q < 16; ++q) {
                double cand = d * (double)sc[j] * (double)q - dmin * (double)m[j];
                double err = fabs(cand - v[t]);
                if (err < best_err) { best_err = err; best = q; }
            }
            if (j % 2 == 0) qs[32 * (j / 2) + i] |= (uint8_t)best;
            else qs[32 * (j / 2) + i] |= (uint8_t)(best << 4);
        }
    }
}

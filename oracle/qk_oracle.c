/*
 * qk_oracle.c -- plain, slow CPU reference for the quantize-once activation path.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library calls, links or
 * includes this file. Only tests/, the smoke check and the CPU-baseline leg of
 * the benchmark load it. It shares no code, header, table or constant with the
 * CUDA path.
 *
 * Sources (page titles and sections):
 *   [P1] llama.cpp PR #117 "activation image emission": Overview, Coverage,
 *        "GLU producer evidence" (Q8_1 image of RMS and GLU producers, read by
 *        ordinary MUL_MAT and routed MUL_MAT_ID MMVQ; CPU NMSE bound 5e-4).
 *   [P2] minfer doc 52 "r49 A-quantize prepass shared-A dedup": section 1
 *        (Q8_0 prepass: per-32-block amax, rintf scaling, zero pad) and
 *        section 2 (quantize is a pure function of (x, nt, id)).
 *   [P3] TensorFold PR #1047 "padding rows no longer go through routed
 *        experts": "The fix" and "Receipt" (router, top-k and plan over the
 *        first live rows only; stable grouped plan).
 *
 * Floating point: compiled with -ffp-contract=off and no fast-math, so every
 * float operation below is one IEEE binary32 operation in the default
 * round-to-nearest-even mode. Where a float decides an integer (a code), the
 * decision is taken in binary32 exactly as written; everything else is
 * accumulated in double (binary64).
 *
 * Parity pins for every function live in tests/test_oracle_pins.py; the only
 * unpinned values are the softmax route weights, the RMSNorm and GLU F32
 * outputs beyond their stated tolerances (no page prints a worked number).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QB 32            /* elements per quant block (all formats here) */
#define Q8_1_BYTES 36    /* half d, half s, 32 int8 codes */
#define Q4_0_BYTES 18    /* half d, 16 bytes of nibbles */
#define Q8_0_BYTES 34    /* half d, 32 int8 codes */

/* ------------------------------------------------------------------------ */
/* IEEE binary32 -> binary16, round to nearest, ties to even (IEEE 754-2008  */
/* section 4.3.1), written from the format definitions: binary16 has a       */
/* 5-bit exponent with bias 15 and 10 stored significand bits; values below  */
/* 2^-14 are subnormal with quantum 2^-24; magnitudes that round to 2^16 or  */
/* more overflow to infinity. NaN maps to the quiet NaN of the same sign.    */
/* ------------------------------------------------------------------------ */
uint16_t or_f32_to_f16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t sign = (u >> 16) & 0x8000u;
    uint32_t bexp = (u >> 23) & 0xFFu;
    uint32_t frac = u & 0x7FFFFFu;

    if (bexp == 0xFFu)                       /* inf or NaN */
        return (uint16_t)(sign | (frac ? 0x7E00u : 0x7C00u));
    if (bexp == 0)                           /* zero or float subnormal (< 2^-126): rounds to zero */
        return (uint16_t)sign;

    int e = (int)bexp - 127;                 /* value = sig * 2^(e-23), sig in [2^23, 2^24) */
    uint32_t sig = frac | 0x800000u;
    if (e > 15)
        return (uint16_t)(sign | 0x7C00u);

    if (e >= -14) {                          /* binary16 normal range */
        uint32_t keep = sig >> 13;           /* 11 bits, leading one included */
        uint32_t rest = sig & 0x1FFFu;       /* 13 dropped bits */
        if (rest > 0x1000u || (rest == 0x1000u && (keep & 1u)))
            keep++;
        uint32_t hexp = (uint32_t)(e + 15);
        if (keep == 0x800u) {                /* rounding carried into the exponent */
            keep = 0x400u;
            hexp++;
        }
        if (hexp >= 31u)
            return (uint16_t)(sign | 0x7C00u);
        return (uint16_t)(sign | (hexp << 10) | (keep & 0x3FFu));
    }

    /* binary16 subnormal: value = m * 2^-24 with m = sig * 2^(e+1) */
    int shift = -e - 1;                      /* >= 14 */
    if (shift > 24)                          /* below 2^-25: rounds to zero */
        return (uint16_t)sign;
    uint32_t m = sig >> shift;
    uint32_t rest = sig & ((1u << shift) - 1u);
    uint32_t halfway = 1u << (shift - 1);
    if (rest > halfway || (rest == halfway && (m & 1u)))
        m++;                                 /* m == 0x400 is the smallest normal: still correct bits */
    return (uint16_t)(sign | m);
}

/* binary16 -> binary32 (exact: every binary16 value is a binary32 value). */
float or_f16_to_f32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    uint32_t hexp = (h >> 10) & 0x1Fu;
    uint32_t frac = h & 0x3FFu;
    uint32_t u;
    if (hexp == 0x1Fu) {
        u = sign | 0x7F800000u | (frac << 13);
    } else if (hexp == 0) {
        if (frac == 0) {
            u = sign;
        } else {                             /* subnormal: frac * 2^-24 */
            float v = (float)frac * 5.9604644775390625e-8f; /* exact: 2^-24 times an integer < 2^10 */
            memcpy(&u, &v, 4);
            u |= sign;
        }
    } else {
        u = sign | ((hexp - 15u + 127u) << 23) | (frac << 13);
    }
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Element-wise or_f32_to_f16 over an array (used by the exhaustive pin). */
void or_f32_to_f16_array(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = or_f32_to_f16(x[i]);
}

static void put_le16(uint8_t *p, uint16_t v)
{
    p[0] = (uint8_t)(v & 0xFFu);
    p[1] = (uint8_t)(v >> 8);
}

static uint16_t get_le16(const uint8_t *p)
{
    return (uint16_t)(p[0] | (p[1] << 8));
}

static int64_t live_count(const int32_t *live, int64_t T)
{
    if (!live)
        return T;
    int64_t n = *live;
    if (n < 0)
        n = 0;
    if (n > T)
        n = T;
    return n;
}

/* ------------------------------------------------------------------------ */
/* One 32-element block quantised as Q8 ([P1] Coverage: "standard Q8_1       */
/* activation image"; [P2] section 1: per-32-block amax, rintf scaling, zero  */
/* pad). Steps, all in binary32:                                             */
/*   amax = max |x_i|;  d = amax / 127;  q_i = rint(x_i / d) (ties to even);  */
/*   all-zero block -> d = 0 and q = 0.                                      */
/* Returns d and writes the 32 codes; *sum_q receives sum of the codes.      */
/* ------------------------------------------------------------------------ */
static float q8_block(const float v[QB], int8_t q[QB], int32_t *sum_q)
{
    float amax = 0.0f;
    for (int i = 0; i < QB; i++) {
        float a = fabsf(v[i]);
        if (a > amax)
            amax = a;
    }
    float d = amax / 127.0f;
    int32_t s = 0;
    if (amax == 0.0f) {
        memset(q, 0, QB);
        *sum_q = 0;
        return 0.0f;
    }
    for (int i = 0; i < QB; i++) {
        float r = rintf(v[i] / d);
        if (r > 127.0f)                      /* unreachable for finite input: |x_i| <= amax */
            r = 127.0f;
        if (r < -127.0f)
            r = -127.0f;
        q[i] = (int8_t)r;
        s += q[i];
    }
    *sum_q = s;
    return d;
}

/* Gathers block b of a row of length K, zero past K ([P1]: widths are padded
 * to whole blocks with zeros). */
static void load_block(const float *row, int64_t K, int64_t b, float v[QB])
{
    for (int i = 0; i < QB; i++) {
        int64_t idx = b * QB + i;
        v[i] = idx < K ? row[idx] : 0.0f;
    }
}

/*
 * Q8_1 image of rows [0, live): per block [d half LE][s half LE][32 codes],
 * s = half(d * sum(q)) with the product in binary32. Blocks from ceil(K/32)
 * to row_blocks are zero bytes. Rows >= live are not touched.
 */
void or_quantize_q8_1(const float *x, int64_t T, int64_t K, int64_t x_stride,
                      uint8_t *img, int64_t row_blocks, const int32_t *live)
{
    int64_t nlive = live_count(live, T);
    int64_t kb = (K + QB - 1) / QB;
    for (int64_t t = 0; t < nlive; t++) {
        const float *row = x + t * x_stride;
        uint8_t *out = img + t * row_blocks * Q8_1_BYTES;
        for (int64_t b = 0; b < row_blocks; b++) {
            uint8_t *blk = out + b * Q8_1_BYTES;
            if (b >= kb) {
                memset(blk, 0, Q8_1_BYTES);
                continue;
            }
            float v[QB];
            int8_t q[QB];
            int32_t sq;
            load_block(row, K, b, v);
            float d = q8_block(v, q, &sq);
            float sd = d * (float)sq;
            put_le16(blk + 0, or_f32_to_f16(d));
            put_le16(blk + 2, or_f32_to_f16(sd));
            memcpy(blk + 4, q, QB);
        }
    }
}

/*
 * Q8_0 image of rows [0, live) ([P2] section 1, the prefill prepass), stored
 * as two planes: codes qs[t][row_blocks*32] int8 and scales d[t][row_blocks]
 * half. Blocks from ceil(K/32) to row_blocks are zero. Rows >= live untouched.
 */
void or_quantize_q8_0(const float *x, int64_t T, int64_t K, int64_t x_stride,
                      int8_t *qs, uint16_t *dh, int64_t row_blocks, const int32_t *live)
{
    int64_t nlive = live_count(live, T);
    int64_t kb = (K + QB - 1) / QB;
    for (int64_t t = 0; t < nlive; t++) {
        const float *row = x + t * x_stride;
        for (int64_t b = 0; b < row_blocks; b++) {
            int8_t *qo = qs + (t * row_blocks + b) * QB;
            uint16_t *dout = dh + t * row_blocks + b;
            if (b >= kb) {
                memset(qo, 0, QB);
                *dout = 0;
                continue;
            }
            float v[QB];
            int32_t sq;
            load_block(row, K, b, v);
            float d = q8_block(v, qo, &sq);
            *dout = or_f32_to_f16(d);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* RMS producers ([P1] Coverage: RMS-alone, RMS+MUL, RMS+MUL+ADD, RMS+SCALE). */
/* y = x / sqrt(mean(x^2) + eps), then times w, times w plus b, or times a   */
/* scalar. Computed in binary64. kind: 0 plain, 1 mul, 2 mul+add, 3 scale.   */
/* ------------------------------------------------------------------------ */
void or_rmsnorm(const float *x, int64_t T, int64_t K, int64_t x_stride, int kind,
                const float *w, const float *b, double scale, double eps,
                double *y, const int32_t *live)
{
    int64_t nlive = live_count(live, T);
    for (int64_t t = 0; t < nlive; t++) {
        const float *row = x + t * x_stride;
        double ss = 0.0;
        for (int64_t i = 0; i < K; i++)
            ss += (double)row[i] * (double)row[i];
        double r = 1.0 / sqrt(ss / (double)K + eps);
        for (int64_t i = 0; i < K; i++) {
            double v = (double)row[i] * r;
            if (kind == 1)
                v = v * (double)w[i];
            else if (kind == 2)
                v = v * (double)w[i] + (double)b[i];
            else if (kind == 3)
                v = v * scale;
            y[t * K + i] = v;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* GLU producers ([P1] Coverage: F32 ReGLU, GeGLU, SwiGLU, GeGLU-erf,       */
/* GeGLU-quick, SwiGLU-OAI with alpha/limit; separate, packed and            */
/* packed-swapped inputs with independent row strides). The page names the  */
/* kinds only; the formulas are the published ones:                          */
/*   SwiGLU:      out = g * sigmoid(g) * u                                   */
/*   GeGLU-tanh:  out = 0.5 g (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))) * u  */
/*   ReGLU:       out = max(g, 0) * u                                        */
/*   GeGLU-erf:   out = 0.5 g (1 + erf(g / sqrt 2)) * u  (GELU, Hendrycks &  */
/*                Gimpel 2016, exact form)                                   */
/*   GeGLU-quick: out = g * sigmoid(1.702 g) * u  (the same paper's sigmoid  */
/*                approximation)                                             */
/*   SwiGLU-OAI:  x = min(g, limit), v = clamp(u, -limit, limit),            */
/*                out = x * sigmoid(alpha x) * (v + 1)  (gpt-oss MLP)        */
/*   SwiGLU-clamp: the same clamps on SwiGLU, out = x * sigmoid(x) * v (a    */
/*                reading: no formula is published with the name)           */
/* kind: 0 swiglu, 1 geglu-tanh, 2 reglu, 3 geglu-erf, 4 geglu-quick,         */
/* 5 swiglu-oai, 6 swiglu-clamp. layout: 0 separate (g at a, u at b),        */
/* 1 packed row [g | u] at a, 2 packed-swapped row [u | g] at a.             */
/* ------------------------------------------------------------------------ */
static double glu_value(int kind, double g, double u, double alpha, double limit)
{
    switch (kind) {
    case 0:
        return g / (1.0 + exp(-g)) * u;
    case 1: {
        const double c = 0.7978845608028654; /* sqrt(2/pi) */
        return 0.5 * g * (1.0 + tanh(c * (g + 0.044715 * g * g * g))) * u;
    }
    case 3:
        return 0.5 * g * (1.0 + erf(g / sqrt(2.0))) * u;
    case 4:
        return g / (1.0 + exp(-1.702 * g)) * u;
    case 5: {
        double x = g < limit ? g : limit;
        double v = u < -limit ? -limit : (u > limit ? limit : u);
        return x / (1.0 + exp(-alpha * x)) * (v + 1.0);
    }
    case 6: {
        double x = g < limit ? g : limit;
        double v = u < -limit ? -limit : (u > limit ? limit : u);
        return x / (1.0 + exp(-x)) * v;
    }
    default:
        return (g > 0.0 ? g : 0.0) * u;
    }
}

void or_glu(int kind, int layout, const float *a, int64_t a_stride,
            const float *bsrc, int64_t b_stride, int64_t T, int64_t N,
            double alpha, double limit, double *out, const int32_t *live)
{
    int64_t nlive = live_count(live, T);
    for (int64_t t = 0; t < nlive; t++) {
        const float *g, *u;
        if (layout == 0) {
            g = a + t * a_stride;
            u = bsrc + t * b_stride;
        } else if (layout == 1) {
            g = a + t * a_stride;
            u = g + N;
        } else {
            u = a + t * a_stride;
            g = u + N;
        }
        for (int64_t i = 0; i < N; i++)
            out[t * N + i] = glu_value(kind, (double)g[i], (double)u[i], alpha, limit);
    }
}

/* ------------------------------------------------------------------------ */
/* Weights. Canonical blocks (the common ggml byte layout):                  */
/*   Q4_0: [d half LE][16 bytes]; element j < 16 is the low nibble of byte j, */
/*         element j+16 the high nibble of byte j; value = (nibble - 8) * d.  */
/*   Q8_0: [d half LE][32 int8]; value = q * d.                              */
/* wtype: 0 = Q4_0, 1 = Q8_0. Dequantised to binary64 W[N][K].               */
/* ------------------------------------------------------------------------ */
static int w_code(int wtype, const uint8_t *blk, int j)
{
    if (wtype == 0) {
        uint8_t byte = blk[2 + (j & 15)];
        int nib = j < 16 ? (byte & 0x0F) : (byte >> 4);
        return nib;                          /* unsigned nibble 0..15 */
    }
    return (int)(int8_t)blk[2 + j];
}

static int w_block_bytes(int wtype)
{
    return wtype == 0 ? Q4_0_BYTES : Q8_0_BYTES;
}

void or_dequant(int wtype, const uint8_t *W, int64_t N, int64_t K, double *out)
{
    int64_t kb = K / QB;
    int bb = w_block_bytes(wtype);
    for (int64_t n = 0; n < N; n++)
        for (int64_t b = 0; b < kb; b++) {
            const uint8_t *blk = W + (n * kb + b) * bb;
            double d = (double)or_f16_to_f32(get_le16(blk));
            for (int j = 0; j < QB; j++) {
                int c = w_code(wtype, blk, j);
                double v = wtype == 0 ? (double)(c - 8) * d : (double)c * d;
                out[n * K + b * QB + j] = v;
            }
        }
}

/*
 * Quantised-path dot product of weight row n with Q8_1 image row ([P1]: MMVQ
 * reads the Q8_1 image). Block by block, from the stored halves:
 *   Q4_0: d_w * (d_a * D - 8 * s_a),  D = sum nibble_i * q_i   (integer)
 *   Q8_0: d_w * d_a * sum qw_i * q_i
 * summed in binary64.
 */
static double dot_q8_1(int wtype, const uint8_t *wrow, int64_t kb, const uint8_t *arow)
{
    int bb = w_block_bytes(wtype);
    double acc = 0.0;
    for (int64_t b = 0; b < kb; b++) {
        const uint8_t *wb = wrow + b * bb;
        const uint8_t *ab = arow + b * Q8_1_BYTES;
        double dw = (double)or_f16_to_f32(get_le16(wb));
        double da = (double)or_f16_to_f32(get_le16(ab));
        double sa = (double)or_f16_to_f32(get_le16(ab + 2));
        int64_t D = 0;
        for (int j = 0; j < QB; j++)
            D += (int64_t)w_code(wtype, wb, j) * (int64_t)(int8_t)ab[4 + j];
        if (wtype == 0)
            acc += dw * (da * (double)D - 8.0 * sa);
        else
            acc += dw * da * (double)D;
    }
    return acc;
}

/* y[t][n] (row stride N) for t < T (all image rows), all n < N. */
void or_proj_q8_1(int wtype, const uint8_t *W, int64_t N, int64_t K,
                  const uint8_t *img, int64_t row_blocks, int64_t T, double *y)
{
    int64_t kb = K / QB;
    int64_t wrow_bytes = kb * w_block_bytes(wtype);
    for (int64_t t = 0; t < T; t++)
        for (int64_t n = 0; n < N; n++)
            y[t * N + n] = dot_q8_1(wtype, W + n * wrow_bytes, kb,
                                    img + t * row_blocks * Q8_1_BYTES);
}

/*
 * Quantised-path dot with a Q8_0 activation image (split planes): per block
 *   d_w * d_a * sum (w_i) * q_i,  w_i = nibble - 8 (Q4_0) or the int8 code (Q8_0).
 * Computes y at the (rows[i], cols[j]) grid, out[i*ncols + j].
 */
void or_proj_q8_0_sampled(int wtype, const uint8_t *W, int64_t N, int64_t K,
                          const int8_t *qs, const uint16_t *dh, int64_t row_blocks,
                          const int64_t *rows, int64_t nrows,
                          const int64_t *cols, int64_t ncols, double *out)
{
    (void)N;
    int64_t kb = K / QB;
    int bb = w_block_bytes(wtype);
    int64_t wrow_bytes = kb * bb;
    for (int64_t i = 0; i < nrows; i++) {
        int64_t t = rows[i];
        for (int64_t jc = 0; jc < ncols; jc++) {
            int64_t n = cols[jc];
            const uint8_t *wrow = W + n * wrow_bytes;
            double acc = 0.0;
            for (int64_t b = 0; b < kb; b++) {
                const uint8_t *wb = wrow + b * bb;
                double dw = (double)or_f16_to_f32(get_le16(wb));
                double da = (double)or_f16_to_f32(dh[t * row_blocks + b]);
                const int8_t *qa = qs + (t * row_blocks + b) * QB;
                int64_t D = 0;
                for (int j = 0; j < QB; j++) {
                    int c = w_code(wtype, wb, j);
                    int wv = wtype == 0 ? c - 8 : c;
                    D += (int64_t)wv * (int64_t)qa[j];
                }
                acc += dw * da * (double)D;
            }
            out[i * ncols + jc] = acc;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Router top-k over the first live rows ([P3] "The fix": router and top-k   */
/* skip rows from the live count up). Probabilities: softmax over E logits  */
/* in binary64. Experts ranked by logit, larger first, equal logits to the   */
/* lower index (softmax is monotone, so this is the probability order too).  */
/* ids[r][0..k) in rank order; wts = the chosen probabilities.               */
/* ------------------------------------------------------------------------ */
void or_topk_route(const float *logits, int64_t rows, int E, int k,
                   int32_t *ids, double *wts, const int32_t *live)
{
    int64_t nlive = live_count(live, rows);
    char *taken = (char *)malloc((size_t)E);
    for (int64_t r = 0; r < nlive; r++) {
        const float *l = logits + r * E;
        double mx = -INFINITY;
        for (int e = 0; e < E; e++)
            if ((double)l[e] > mx)
                mx = (double)l[e];
        double z = 0.0;
        for (int e = 0; e < E; e++)
            z += exp((double)l[e] - mx);
        memset(taken, 0, (size_t)E);
        for (int s = 0; s < k; s++) {
            int best = -1;
            for (int e = 0; e < E; e++) {
                if (taken[e])
                    continue;
                if (best < 0 || l[e] > l[best])
                    best = e;
            }
            taken[best] = 1;
            ids[r * k + s] = best;
            wts[r * k + s] = exp((double)l[best] - mx) / z;
        }
    }
    free(taken);
}

/* ------------------------------------------------------------------------ */
/* Stable grouped plan of the live pairs ([P3] "The fix": counts and ranks,  */
/* exclusive-scan offsets, scatter; only the first live*k pairs). Pair p =   */
/* row*k + slot names expert ids[p]. counts[e] = pairs for e; offsets is the */
/* exclusive scan; items lists the pairs of expert 0, then 1, ..., each      */
/* group in ascending p. A pair whose id lies outside [0, E) names no expert */
/* and is left out (reading of the pages: such a pair has no expert work),   */
/* so offsets[E] = the number of live pairs with a valid id.                 */
/* ------------------------------------------------------------------------ */
void or_moe_plan(const int32_t *ids, int64_t rows, int k, int E,
                 int32_t *counts, int32_t *offsets, int32_t *items, const int32_t *live)
{
    int64_t npairs = live_count(live, rows) * k;
    for (int e = 0; e < E; e++)
        counts[e] = 0;
    for (int64_t p = 0; p < npairs; p++)
        if (ids[p] >= 0 && ids[p] < E)
            counts[ids[p]]++;
    offsets[0] = 0;
    for (int e = 0; e < E; e++)
        offsets[e + 1] = offsets[e] + counts[e];
    int32_t *fill = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    for (int e = 0; e < E; e++)
        fill[e] = offsets[e];
    for (int64_t p = 0; p < npairs; p++)
        if (ids[p] >= 0 && ids[p] < E)
            items[fill[ids[p]]++] = (int32_t)p;
    free(fill);
}

/*
 * Routed projection ([P1] MUL_MAT_ID; [P3] no expert work for padding): for
 * every planned item p, y[p][n] = dot(W_e row n, image row p / k) with
 * e = ids[p]. W holds E experts back to back, each [N][K] canonical blocks.
 * Pairs that are not planned are not written.
 */
void or_proj_id_q8_1(int wtype, const uint8_t *W, int E, int64_t N, int64_t K,
                     const uint8_t *img, int64_t row_blocks, const int32_t *ids, int k,
                     const int32_t *items, int64_t nitems, double *y)
{
    (void)E;
    int64_t kb = K / QB;
    int64_t wrow_bytes = kb * w_block_bytes(wtype);
    for (int64_t i = 0; i < nitems; i++) {
        int64_t p = items[i];
        int64_t row = p / k;
        const uint8_t *We = W + (int64_t)ids[p] * N * wrow_bytes;
        for (int64_t n = 0; n < N; n++)
            y[p * N + n] = dot_q8_1(wtype, We + n * wrow_bytes, kb,
                                    img + row * row_blocks * Q8_1_BYTES);
    }
}

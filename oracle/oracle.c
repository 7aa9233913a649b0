/*
 * oracle.c -- plain, slow CPU restatement of the a8w4 fused MoE layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code with the CUDA library.
 *
 * What it computes, stage by stage (the pages name the stages of the fused
 * operator -- activation quantisation, dispatch, the two expert GEMMs and the
 * combine, in one kernel -- in "sglang PR #47065", Title/switches; the fused EPLB remap and per-expert load recording
 * in "sglang PR #35619", Summary; a8w4 with MXFP4 routed experts in
 * "InferenceX PR #3430", draft-precision notes):
 *
 *   route    s = sigmoid(logit) (fp32, exp_spec below), key = s + bias,
 *            top-k by key (descending, ties -> lower expert), w = s / sum s
 *   eplb     phys = replicas[idx][(t + j) mod replica_count[idx]]
 *   record   counts[idx] += 1 per (token, slot) pair
 *   quant    MXFP8: per 32 values, X = clamp(floor(log2 amax) - 8, -127, 127),
 *            scale byte X + 127, codes e4m3(v / 2^X), round-to-nearest-even,
 *            saturating at +-448
 *   permute  pairs grouped by physical expert, ascending pair id inside
 *   GEMM1    G = A . W1^T with fp64 accumulation; gate = G[:, :I],
 *            up = G[:, I:]; h = silu(gate) * up; h -> MXFP8 along I
 *   GEMM2    y = deq(hq) . W2^T, fp64 accumulation
 *   combine  out[t] = bf16(sum_j w[t,j] * y[t,j]) in fp64, rounded to fp32
 *            then to bf16 (nearest-even)
 *
 * The a16w4 variant (bf16 activations with the same MXFP4 experts, the other
 * serving arms of "InferenceX PR #3430", draft-precision notes) skips the
 * activation quantisation: GEMM1 reads the bf16 hidden rows, h is rounded to
 * bf16 (the activation type of that arm) and GEMM2 reads it; routing,
 * dispatch and combine are the same.
 *
 * Where the pages are silent the plainest reading is taken; every such
 * reading is spelled out beside the function that makes it.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (no fast-math: the
 * routing score must be evaluated as the exact sequence of IEEE binary32
 * operations written below).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#if defined(__FAST_MATH__)
#error "the oracle must be built without fast-math"
#endif

static float f32_from_bits(uint32_t b) { float f; memcpy(&f, &b, 4); return f; }
static uint32_t bits_from_f32(float f) { uint32_t b; memcpy(&b, &f, 4); return b; }

/* ------------------------------------------------------------------------ *
 * Routing score.  Reading: the pages fix "sigmoid top-k routing" but no
 * evaluation; for the selected experts to be reproducible bit for bit, the
 * score is defined as this exact binary32 operation sequence (Cody-Waite
 * range reduction y = n ln2 + r with a two-part ln2, degree-7 Taylor
 * polynomial of e^r in Horner form, scaling by 2^n through the exponent
 * field).  Every operation is a single correctly rounded binary32 add, mul or
 * div; no fused multiply-add.
 * ------------------------------------------------------------------------ */
#define EXP_LO (-87.0f)
#define EXP_HI (88.0f)

float orc_exp_spec(float y)
{
    const float log2e = f32_from_bits(0x3FB8AA3Bu);   /* binary32(1/ln 2) */
    const float ln2_hi = f32_from_bits(0x3F317200u);  /* binary32(ln 2), low 8 bits cleared */
    const float ln2_lo = f32_from_bits(0x35BFBE8Eu);  /* binary32(ln 2 - ln2_hi) */
    const float c2 = 1.0f / 2.0f, c3 = 1.0f / 6.0f, c4 = 1.0f / 24.0f;
    const float c5 = 1.0f / 120.0f, c6 = 1.0f / 720.0f, c7 = 1.0f / 5040.0f;
    if (y < EXP_LO) y = EXP_LO;
    if (y > EXP_HI) y = EXP_HI;
    float n = rintf(y * log2e);                        /* nearest, ties to even */
    float r = y - n * ln2_hi;                          /* n * ln2_hi is exact */
    r = r - n * ln2_lo;
    float p = c7;
    p = p * r + c6;
    p = p * r + c5;
    p = p * r + c4;
    p = p * r + c3;
    p = p * r + c2;
    p = p * r + 1.0f;
    p = p * r + 1.0f;
    int ni = (int)n;                                   /* in [-126, 127] */
    return p * f32_from_bits((uint32_t)(ni + 127) << 23);
}

float orc_sigmoid_spec(float x)
{
    return 1.0f / (1.0f + orc_exp_spec(-x));
}

void orc_exp_spec_vec(int64_t n, const float *x, float *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = orc_exp_spec(x[i]);
}

void orc_sigmoid_spec_vec(int64_t n, const float *x, float *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = orc_sigmoid_spec(x[i]);
}

/* max |exp_spec(y) - exp(y)| in units of the binary32 ulp of exp(y), over
 * every stride-th binary32 value in [lo, hi] (same sign); used by the tests. */
double orc_exp_spec_max_ulp(float lo, float hi, int stride, int sigmoid)
{
    uint32_t a = bits_from_f32(lo), b = bits_from_f32(hi);
    uint32_t first = a < b ? a : b, last = a < b ? b : a;
    double worst = 0.0;
#pragma omp parallel for reduction(max : worst) schedule(static)
    for (int64_t u = first; u <= (int64_t)last; u += stride) {
        float y = f32_from_bits((uint32_t)u);
        double ref = sigmoid ? 1.0 / (1.0 + exp(-(double)y)) : exp((double)y);
        double got = sigmoid ? (double)orc_sigmoid_spec(y) : (double)orc_exp_spec(y);
        int e;
        frexp(ref, &e);                                 /* ref in [2^(e-1), 2^e) */
        int ue = e - 1 - 23;
        if (ue < -149) ue = -149;
        double err = fabs(got - ref) / ldexp(1.0, ue);
        if (err > worst) worst = err;
    }
    return worst;
}

/* ------------------------------------------------------------------------ *
 * route: top-k over key = s + bias.  Reading: the weights normalise s (not the
 * biased key) over the selected experts, summed in fp32 in selection order;
 * no group-limited routing and no extra routed scaling factor.
 * ------------------------------------------------------------------------ */
void orc_route(int64_t T, int E, int k, const float *logits, const float *bias,
               int32_t *idx, float *w)
{
#pragma omp parallel
    {
        float *s = (float *)malloc(sizeof(float) * E);
        float *key = (float *)malloc(sizeof(float) * E);
        char *used = (char *)malloc(E);
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            for (int e = 0; e < E; ++e) {
                s[e] = orc_sigmoid_spec(logits[t * E + e]);
                key[e] = s[e] + (bias ? bias[e] : 0.0f);
                used[e] = 0;
            }
            float S = 0.0f;
            for (int j = 0; j < k; ++j) {
                int best = -1;
                for (int e = 0; e < E; ++e)
                    if (!used[e] && (best < 0 || key[e] > key[best])) best = e;
                used[best] = 1;
                idx[t * k + j] = best;
                S = (j == 0) ? s[best] : S + s[best];
            }
            for (int j = 0; j < k; ++j) w[t * k + j] = s[idx[t * k + j]] / S;
        }
        free(s); free(key); free(used);
    }
}

/* eplb remap: token_ids[t] is the token's index within its forward call. */
void orc_eplb(int64_t T, int k, const int64_t *token_ids, const int32_t *idx,
              const int32_t *phys_of_logical, const int32_t *replica_counts, int R,
              int32_t *phys)
{
    for (int64_t t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int e = idx[t * k + j];
            int64_t tok = token_ids ? token_ids[t] : t;
            int slot = (int)((tok + j) % replica_counts[e]);
            phys[t * k + j] = phys_of_logical[(int64_t)e * R + slot];
        }
}

void orc_record(int64_t npairs, const int32_t *idx, int64_t *counts)
{
    for (int64_t i = 0; i < npairs; ++i) counts[idx[i]] += 1;
}

/* ------------------------------------------------------------------------ *
 * Element formats (OCP Microscaling v1.0 reading).
 *   e4m3: bias 7, no infinities, S.1111.111 is NaN, max 448, subnormals m*2^-9
 *   e2m1: bias 1, values +-{0, .5, 1, 1.5, 2, 3, 4, 6}
 *   e8m0: 2^(s - 127), s = 255 is NaN
 * ------------------------------------------------------------------------ */
double orc_e4m3_value(uint8_t c)
{
    int sgn = c >> 7, ex = (c >> 3) & 15, m = c & 7;
    double v;
    if (ex == 15 && m == 7) return NAN;
    if (ex == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, ex - 7);
    return sgn ? -v : v;
}

double orc_e2m1_value(uint8_t nib)
{
    int sgn = (nib >> 3) & 1, ex = (nib >> 1) & 3, m = nib & 1;
    double v = (ex == 0) ? 0.5 * m : ldexp(1.0 + m / 2.0, ex - 1);
    return sgn ? -v : v;
}

double orc_e8m0_value(uint8_t s)
{
    return s == 255 ? NAN : ldexp(1.0, (int)s - 127);
}

/* nearest e4m3 code to a (exact double), ties to even, saturating at 448 */
uint8_t orc_e4m3_encode(double a)
{
    uint8_t sgn = signbit(a) ? 0x80 : 0x00;
    a = fabs(a);
    if (a == 0.0) return sgn;
    int e;
    frexp(a, &e);
    e -= 1;                                  /* a in [2^e, 2^(e+1)) */
    if (e < -6) e = -6;                      /* subnormal range: quantum 2^-9 */
    double q = ldexp(1.0, e - 3);            /* spacing of representable values */
    double n = nearbyint(a / q);             /* exact quotient, ties to even */
    double v = n * q;
    if (v > 448.0) v = 448.0;
    if (v < ldexp(1.0, -6)) return sgn | (uint8_t)(v / ldexp(1.0, -9));
    frexp(v, &e);
    e -= 1;
    int mant = (int)(v / ldexp(1.0, e) * 8.0) - 8;
    return sgn | (uint8_t)((e + 7) << 3) | (uint8_t)mant;
}

/* MXFP8 quantisation of rows of exact values (row length K, K % 32 == 0).
 * Reading: a block whose amax is 0 gets scale byte 0 and all codes +0. */
void orc_mxfp8_quant(int64_t rows, int K, const float *v, uint8_t *q, uint8_t *s)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int b = 0; b < K / 32; ++b) {
            const float *blk = v + r * K + b * 32;
            double amax = 0.0;
            for (int i = 0; i < 32; ++i)
                if (fabs((double)blk[i]) > amax) amax = fabs((double)blk[i]);
            uint8_t *qb = q + r * K + b * 32;
            if (amax == 0.0) {
                s[r * (K / 32) + b] = 0;
                memset(qb, 0, 32);
                continue;
            }
            int e;
            frexp(amax, &e);
            int X = (e - 1) - 8;             /* emax(e4m3) = 8 */
            if (X < -127) X = -127;
            if (X > 127) X = 127;
            s[r * (K / 32) + b] = (uint8_t)(X + 127);
            for (int i = 0; i < 32; ++i) qb[i] = orc_e4m3_encode(ldexp((double)blk[i], -X));
        }
}

void orc_mxfp8_quant_bf16(int64_t rows, int K, const uint16_t *x, uint8_t *q, uint8_t *s)
{
    float *v = (float *)malloc(sizeof(float) * rows * K);
    for (int64_t i = 0; i < rows * K; ++i) v[i] = f32_from_bits((uint32_t)x[i] << 16);
    orc_mxfp8_quant(rows, K, v, q, s);
    free(v);
}

/* permute: order[] lists pair ids grouped by physical expert (ascending pair
 * id within a group), offsets[P+1] the unpadded group starts, pos[i] the
 * position of pair i in order[]. */
void orc_permute(int64_t npairs, int P, const int32_t *phys, int64_t *offsets,
                 int64_t *order, int64_t *pos)
{
    int64_t *fill = (int64_t *)calloc(P, sizeof(int64_t));
    for (int p = 0; p <= P; ++p) offsets[p] = 0;
    for (int64_t i = 0; i < npairs; ++i) offsets[phys[i] + 1] += 1;
    for (int p = 0; p < P; ++p) offsets[p + 1] += offsets[p];
    for (int64_t i = 0; i < npairs; ++i) {
        int p = phys[i];
        int64_t at = offsets[p] + fill[p]++;
        order[at] = i;
        pos[i] = at;
    }
    free(fill);
}

static uint16_t bf16_rne(float f)
{
    uint32_t b = bits_from_f32(f);
    if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x7FFFFFu)) return (uint16_t)((b >> 16) | 0x40);
    b += 0x7FFFu + ((b >> 16) & 1u);
    return (uint16_t)(b >> 16);
}

static double bf16_value(uint16_t h) { return (double)f32_from_bits((uint32_t)h << 16); }

/* one row of an MXFP4 matrix (K values) as exact doubles */
static void mxfp4_row(int K, const uint8_t *packed, const uint8_t *scale, double *out)
{
    for (int h = 0; h < K; ++h) {
        uint8_t byte = packed[h / 2];
        uint8_t nib = (h & 1) ? (byte >> 4) : (byte & 15);   /* element 2i = low nibble */
        out[h] = orc_e2m1_value(nib) * orc_e8m0_value(scale[h / 32]);
    }
}

static void mxfp8_rows(int64_t rows, int K, const uint8_t *q, const uint8_t *s, double *out)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int h = 0; h < K; ++h)
            out[r * K + h] = orc_e4m3_value(q[r * K + h]) * orc_e8m0_value(s[r * (K / 32) + h / 32]);
}

/* GEMM2 for rows of one expert: y[r][m] = sum_i deq(hq)[r][i] * W2[m][i] */
void orc_expert_down(int64_t rows, int H, int I, const uint8_t *hq, const uint8_t *hs,
                     const uint8_t *w2, const uint8_t *w2s, float *y)
{
    double *a = (double *)malloc(sizeof(double) * rows * I);
    mxfp8_rows(rows, I, hq, hs, a);
#pragma omp parallel
    {
        double *wrow = (double *)malloc(sizeof(double) * I);
#pragma omp for schedule(static)
        for (int m = 0; m < H; ++m) {
            mxfp4_row(I, w2 + (int64_t)m * (I / 2), w2s + (int64_t)m * (I / 32), wrow);
            for (int64_t r = 0; r < rows; ++r) {
                double acc = 0.0;
                for (int i = 0; i < I; ++i) acc += a[r * I + i] * wrow[i];
                y[r * H + m] = (float)acc;
            }
        }
        free(wrow);
    }
    free(a);
}

/* GEMM1 + SwiGLU + MXFP8 requant + GEMM2 for rows of one expert.
 * Readings: W1 rows 0..I-1 are the gate projection and rows I..2I-1 the up
 * projection (concatenated); silu(g) = g / (1 + e^-g); no clamp on gate/up.
 * g_out [rows,2I] and h_out [rows,I] (pre-quantisation) are optional. */
void orc_expert_ffn(int64_t rows, int H, int I, const uint8_t *xq, const uint8_t *xs,
                    const uint8_t *w1, const uint8_t *w1s, const uint8_t *w2,
                    const uint8_t *w2s, uint8_t *hq, uint8_t *hs, float *g_out,
                    float *h_out, float *y)
{
    double *a = (double *)malloc(sizeof(double) * rows * H);
    float *G = (float *)malloc(sizeof(float) * rows * 2 * I);
    float *h = (float *)malloc(sizeof(float) * rows * I);
    mxfp8_rows(rows, H, xq, xs, a);
#pragma omp parallel
    {
        double *wrow = (double *)malloc(sizeof(double) * H);
#pragma omp for schedule(static)
        for (int n = 0; n < 2 * I; ++n) {
            mxfp4_row(H, w1 + (int64_t)n * (H / 2), w1s + (int64_t)n * (H / 32), wrow);
            for (int64_t r = 0; r < rows; ++r) {
                double acc = 0.0;
                for (int k = 0; k < H; ++k) acc += a[r * H + k] * wrow[k];
                G[r * 2 * I + n] = (float)acc;
            }
        }
        free(wrow);
    }
    for (int64_t r = 0; r < rows; ++r)
        for (int i = 0; i < I; ++i) {
            double g = G[r * 2 * I + i], u = G[r * 2 * I + I + i];
            h[r * I + i] = (float)(g / (1.0 + exp(-g)) * u);
        }
    orc_mxfp8_quant(rows, I, h, hq, hs);
    if (g_out) memcpy(g_out, G, sizeof(float) * rows * 2 * I);
    if (h_out) memcpy(h_out, h, sizeof(float) * rows * I);
    free(a); free(G); free(h);
    orc_expert_down(rows, H, I, hq, hs, w2, w2s, y);
}


/* combine: ypair[(t*k + j)*H + m] is y of pair (t, j).  Reading: the top-k
 * weight is applied here, not inside GEMM2. */
void orc_combine(int64_t T, int k, int H, const float *w, const float *ypair, uint16_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int m = 0; m < H; ++m) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j)
                acc += (double)w[t * k + j] * (double)ypair[(t * k + j) * H + m];
            out[t * H + m] = bf16_rne((float)acc);
        }
}

/* ---- a16w4: bf16 activations x MXFP4 experts ---------------------------- */

/* GEMM2 for rows of one expert, bf16 input: y[r][m] = sum_i hb[r][i] * W2[m][i]
 * (fp64 accumulation of exact products, rounded to fp32). */
void orc_expert_down_a16(int64_t rows, int H, int I, const uint16_t *hb, const uint8_t *w2,
                         const uint8_t *w2s, float *y)
{
    double *a = (double *)malloc(sizeof(double) * rows * I);
    for (int64_t j = 0; j < rows * I; ++j) a[j] = bf16_value(hb[j]);
#pragma omp parallel
    {
        double *wrow = (double *)malloc(sizeof(double) * I);
#pragma omp for schedule(static)
        for (int m = 0; m < H; ++m) {
            mxfp4_row(I, w2 + (int64_t)m * (I / 2), w2s + (int64_t)m * (I / 32), wrow);
            for (int64_t r = 0; r < rows; ++r) {
                double acc = 0.0;
                for (int i = 0; i < I; ++i) acc += a[r * I + i] * wrow[i];
                y[r * H + m] = (float)acc;
            }
        }
        free(wrow);
    }
    free(a);
}

/* GEMM1 + SwiGLU + GEMM2 for rows of one expert with bf16 activations x.
 * G = x . W1^T (fp64, rounded to fp32); gate = G[:, :I], up = G[:, I:];
 * h = silu(gate) * up formed from the fp32 G, rounded to fp32 and then to
 * bf16 (nearest-even): hb is GEMM2's input.  g_out [rows,2I] and h_out
 * [rows,I] (h before the bf16 rounding) are optional. */
void orc_expert_ffn_a16(int64_t rows, int H, int I, const uint16_t *x, const uint8_t *w1,
                        const uint8_t *w1s, const uint8_t *w2, const uint8_t *w2s, uint16_t *hb,
                        float *g_out, float *h_out, float *y)
{
    double *a = (double *)malloc(sizeof(double) * rows * H);
    float *G = (float *)malloc(sizeof(float) * rows * 2 * I);
    for (int64_t j = 0; j < rows * H; ++j) a[j] = bf16_value(x[j]);
#pragma omp parallel
    {
        double *wrow = (double *)malloc(sizeof(double) * H);
#pragma omp for schedule(static)
        for (int n = 0; n < 2 * I; ++n) {
            mxfp4_row(H, w1 + (int64_t)n * (H / 2), w1s + (int64_t)n * (H / 32), wrow);
            for (int64_t r = 0; r < rows; ++r) {
                double acc = 0.0;
                for (int k = 0; k < H; ++k) acc += a[r * H + k] * wrow[k];
                G[r * 2 * I + n] = (float)acc;
            }
        }
        free(wrow);
    }
    for (int64_t r = 0; r < rows; ++r)
        for (int i = 0; i < I; ++i) {
            double g = G[r * 2 * I + i], u = G[r * 2 * I + I + i];
            float h = (float)(g / (1.0 + exp(-g)) * u);
            if (h_out) h_out[r * I + i] = h;
            hb[r * I + i] = bf16_rne(h);
        }
    if (g_out) memcpy(g_out, G, sizeof(float) * rows * 2 * I);
    free(a); free(G);
    orc_expert_down_a16(rows, H, I, hb, w2, w2s, y);
}

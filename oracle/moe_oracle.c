/*
 * CPU oracle for the fused Mixture-of-Experts layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, call or
 * load this file: only the tests, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code, header, table or helper with the CUDA
 * library; the two meet only through the seeded inputs.
 *
 * What it computes is the plain definition of the layer described on the
 * fused-MoE pages ("AITER" walk-through, section 3 "Fused MoE": gating ->
 * token reorder -> expert GEMMs -> weighted combine; the talk on group-GEMM
 * MoE kernels for Mixtral with a SwiGLU activation):
 *
 *   per token t:  l_e  = x_t . W_router[e] (+ bias_e)           (router)
 *                 ids  = the k largest l_e (ties -> lower e)     (top-k)
 *                 w_j  = softmax over the k selected logits      (renormalised)
 *                 for j: g = W_gate[e_j] x_t, u = W_up[e_j] x_t
 *                        a = silu(g) * u,  y_j = W_down[e_j] a   (SwiGLU expert)
 *                 out_t = sum_j w_j y_j   (j ascending)          (combine)
 *
 * plus the integer reorder ("moe_sorting" in section 3.1: tokens grouped by
 * expert, each expert padded to whole blocks, buffer of T*k + E*B - k
 * entries) and the two FP8 quantisation types the page names: per-128
 * block scaling ("per_1x128") and one scale per row ("per_Token": a scale
 * per token of the activations, per output channel of the weights), plus
 * the microscaling 4-bit format ("per_1x32", MXFP4: OCP Microscaling
 * Formats -- E2M1 elements sharing one power-of-two E8M0 scale per 32).
 *
 * Precision: inputs are bf16 (or e4m3 codes with fp32 scales) taken exactly;
 * every dot product of the expert GEMMs accumulates in fp64.  The router
 * logits are the one place where floating point decides an integer (the
 * expert ids), so they are taken in fp32 in one fixed summation order, the
 * same order the GPU router uses (see oracle_router_logit).
 *
 * Every routine is a straight loop over the definition; the only parallelism
 * is independent tokens split across POSIX threads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- bf16 */

static float bf16_to_float(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ---------------------------------------------------------------- e4m3 */
/*
 * OCP 8-bit floating point, E4M3 ("fn" variant): 1 sign bit, 4 exponent bits
 * with bias 7, 3 mantissa bits; exponent field 0 holds subnormals m/8 * 2^-6;
 * the pattern S.1111.111 is NaN and there is no infinity, so the largest
 * finite magnitude is 1.75 * 2^8 = 448.
 */
double oracle_e4m3_decode(uint8_t c)
{
    int s = (c >> 7) & 1;
    int E = (c >> 3) & 15;
    int m = c & 7;
    double v;
    if (E == 15 && m == 7)
        return NAN;
    if (E == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, E - 7);
    return s ? -v : v;
}

/* Round to nearest, ties to even, saturating to +-448 (no overflow to NaN). */
uint8_t oracle_e4m3_encode(float v)
{
    if (isnan(v))
        return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0)
        return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: multiples of 2^-9; 8 * 2^-9 is the smallest normal */
        double q = nearbyint(a * 512.0); /* default mode: nearest, ties to even */
        return sign | (uint8_t)q;
    }
    int e2;
    double m = frexp(a, &e2); /* a = m * 2^e2, m in [0.5, 1) */
    int E = e2 - 1;           /* a = (2m) * 2^E, 2m in [1, 2) */
    double frac = nearbyint((2.0 * m - 1.0) * 8.0);
    if (frac == 8.0) {
        frac = 0.0;
        E += 1;
    }
    if (E > 8)
        return sign | 0x7E;
    return sign | (uint8_t)(((E + 7) << 3) | (int)frac);
}

/* scale = amax / 448 in fp32 (1 when the group is all zero). */
static float group_scale(float amax)
{
    if (!(amax > 0.0f))
        return 1.0f;
    return amax / 448.0f;
}

/*
 * "per_1x128" activation quantisation: each row of X [R, C] is cut into
 * groups of 128 columns; each group gets scale = amax/448 and codes
 * e4m3(x / scale).  q [R, C] codes, s [R, C/128] fp32.
 */
void oracle_quant_1x128(const uint16_t *X, int R, int C, uint8_t *q, float *s)
{
    int G = C / 128;
    for (int r = 0; r < R; ++r) {
        for (int g = 0; g < G; ++g) {
            float amax = 0.0f;
            for (int c = g * 128; c < g * 128 + 128; ++c) {
                float v = fabsf(bf16_to_float(X[(size_t)r * C + c]));
                if (v > amax)
                    amax = v;
            }
            float sc = group_scale(amax);
            s[(size_t)r * G + g] = sc;
            for (int c = g * 128; c < g * 128 + 128; ++c)
                q[(size_t)r * C + c] = oracle_e4m3_encode(bf16_to_float(X[(size_t)r * C + c]) / sc);
        }
    }
}

/*
 * Weight quantisation with one fp32 scale per 128x128 block of W [R, C]
 * (rows = output features, columns = the reduction dim).  s [R/128, C/128].
 */
void oracle_quant_128x128(const uint16_t *W, long R, int C, uint8_t *q, float *s)
{
    int GC = C / 128;
    long GR = R / 128;
    for (long br = 0; br < GR; ++br) {
        for (int bc = 0; bc < GC; ++bc) {
            float amax = 0.0f;
            for (long r = br * 128; r < br * 128 + 128; ++r)
                for (int c = bc * 128; c < bc * 128 + 128; ++c) {
                    float v = fabsf(bf16_to_float(W[r * C + c]));
                    if (v > amax)
                        amax = v;
                }
            float sc = group_scale(amax);
            s[br * GC + bc] = sc;
            for (long r = br * 128; r < br * 128 + 128; ++r)
                for (int c = bc * 128; c < bc * 128 + 128; ++c)
                    q[r * C + c] = oracle_e4m3_encode(bf16_to_float(W[r * C + c]) / sc);
        }
    }
}

/*
 * "per_Token" quantisation: one scale per row of X [R, C] (a token of the
 * activations, an output channel of a weight matrix), scale = amax/448 over
 * the whole row, codes e4m3(x / scale).  q [R, C], s [R].
 */
void oracle_quant_rows(const uint16_t *X, long R, int C, uint8_t *q, float *s)
{
    for (long r = 0; r < R; ++r) {
        float amax = 0.0f;
        for (int c = 0; c < C; ++c) {
            float v = fabsf(bf16_to_float(X[r * C + c]));
            if (v > amax)
                amax = v;
        }
        float sc = group_scale(amax);
        s[r] = sc;
        for (int c = 0; c < C; ++c)
            q[r * C + c] = oracle_e4m3_encode(bf16_to_float(X[r * C + c]) / sc);
    }
}

/* ------------------------------------------------------- MXFP4 (1x32) */
/*
 * OCP Microscaling (MX) FP4: each element is E2M1 (1 sign, 2 exponent bits
 * with bias 1, 1 mantissa bit; no infinity or NaN): magnitudes 0, 0.5, 1,
 * 1.5, 2, 3, 4, 6.  Each block of 32 consecutive elements of a row shares
 * one scale X = 2^e stored as E8M0 (the biased exponent e + 127).  The MX
 * conversion rule: e = floor(log2(amax)) - 2, where 2 is the exponent of the
 * largest E2M1 power of two (4); elements are V / X rounded to nearest
 * (ties to even mantissa) and clamped to +-6.  An all-zero block takes
 * e = 0.  The codes here are one per byte (sign << 3 | magnitude index).
 */
static const double kE2M1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double oracle_e2m1_decode(uint8_t c)
{
    double v = kE2M1[c & 7];
    return (c & 8) ? -v : v;
}

uint8_t oracle_e2m1_encode(float v)
{
    uint8_t sign = signbit(v) ? 8 : 0;
    double a = fabs((double)v);
    if (isnan(v) || a >= 6.0)
        return sign | 7;
    int best = 0;
    for (int i = 1; i < 8; ++i) {
        double d = fabs(a - kE2M1[i]), db = fabs(a - kE2M1[best]);
        if (d < db || (d == db && (i & 1) == 0))  /* ties: the even mantissa (even index) */
            best = i;
    }
    return sign | (uint8_t)best;
}

/* Shared exponent of a block with the given amax (unbiased). */
int oracle_mx_exponent(float amax)
{
    if (!(amax > 0.0f))
        return 0;
    int e2;
    frexp((double)amax, &e2); /* amax = m * 2^e2, m in [0.5, 1): floor(log2 amax) = e2 - 1 */
    int e = (e2 - 1) - 2;
    if (e < -127)
        e = -127;
    if (e > 127)
        e = 127;
    return e;
}

typedef struct {
    const uint16_t *X;
    long r0, r1;
    int C;
    uint8_t *q, *s;
} mx4_job;

static void *mx4_worker(void *arg)
{
    mx4_job *J = (mx4_job *)arg;
    int C = J->C, G = C / 32;
    for (long r = J->r0; r < J->r1; ++r) {
        for (int g = 0; g < G; ++g) {
            float amax = 0.0f;
            for (int c = g * 32; c < g * 32 + 32; ++c) {
                float v = fabsf(bf16_to_float(J->X[r * C + c]));
                if (v > amax)
                    amax = v;
            }
            int e = oracle_mx_exponent(amax);
            double inv = ldexp(1.0, -e); /* exact power of two */
            J->s[r * G + g] = (uint8_t)(e + 127);
            for (int c = g * 32; c < g * 32 + 32; ++c)
                J->q[r * C + c] = oracle_e2m1_encode((float)((double)bf16_to_float(J->X[r * C + c]) * inv));
        }
    }
    return NULL;
}

static int clamp_threads(int nthreads, int work);

/*
 * Rows of X [R, C] (C % 32 == 0): codes q [R, C] (one per byte), E8M0 scales
 * s [R, C/32].  Rows are independent; they are split across nthreads.
 */
void oracle_quant_mx4_mt(const uint16_t *X, long R, int C, uint8_t *q, uint8_t *s, int nthreads)
{
    if (R <= 0)
        return;
    nthreads = clamp_threads(nthreads, R > 1 << 30 ? 1 << 30 : (int)R);
    pthread_t th[256];
    mx4_job jobs[256];
    for (int i = 0; i < nthreads; ++i) {
        jobs[i].X = X;
        jobs[i].C = C;
        jobs[i].q = q;
        jobs[i].s = s;
        jobs[i].r0 = R * i / nthreads;
        jobs[i].r1 = R * (i + 1) / nthreads;
        pthread_create(&th[i], NULL, mx4_worker, &jobs[i]);
    }
    for (int i = 0; i < nthreads; ++i)
        pthread_join(th[i], NULL);
}

void oracle_quant_mx4(const uint16_t *X, long R, int C, uint8_t *q, uint8_t *s)
{
    mx4_job J = {X, 0, R, C, q, s};
    mx4_worker(&J);
}

static double mx4_value(const uint8_t *q, const uint8_t *s, long idx, int C)
{
    return ldexp(oracle_e2m1_decode(q[idx]), (int)s[(idx / C) * (C / 32) + (idx % C) / 32] - 127);
}

/* -------------------------------------------------------------- router */
/*
 * Router logit in fp32, in one fixed order: the H products are dealt to 32
 * partial sums in chunks of 8 consecutive elements (element h goes to
 * partial (h / 8) mod 32), each partial adds its elements in ascending h,
 * then the 32 partials are combined pairwise by a butterfly with strides
 * 16, 8, 4, 2, 1 (partial i takes partial i + partial (i xor stride)).  A
 * bf16 x bf16 product is exact in fp32, so only this order matters.  The
 * bias (if any) is added last.
 */
float oracle_router_logit(const uint16_t *x, const uint16_t *w, int H, const float *bias, int e)
{
    float part[32];
    for (int i = 0; i < 32; ++i)
        part[i] = 0.0f;
    for (int h = 0; h < H; ++h) {
        float p = bf16_to_float(x[h]) * bf16_to_float(w[h]);
        part[(h / 8) % 32] = part[(h / 8) % 32] + p;
    }
    for (int stride = 16; stride >= 1; stride /= 2) {
        float nxt[32];
        for (int i = 0; i < 32; ++i)
            nxt[i] = part[i] + part[i ^ stride];
        for (int i = 0; i < 32; ++i)
            part[i] = nxt[i];
    }
    float l = part[0];
    if (bias)
        l = l + bias[e];
    return l;
}

/*
 * Top-k on the logits (largest first; an equal logit goes to the lower
 * expert index), then softmax over the k selected logits, which is the same
 * as softmax over all E followed by top-k and renormalisation (renorm = 1);
 * with renorm = 0 the weights are the softmax over all E experts evaluated
 * at the selected ones (they need not sum to 1).
 */
static void route_token_r(const float *logit, int E, int k, int renorm, int32_t *ids, double *w)
{
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            int taken = 0;
            for (int i = 0; i < j; ++i)
                if (ids[i] == e)
                    taken = 1;
            if (taken)
                continue;
            if (best < 0 || logit[e] > logit[best])
                best = e;
        }
        ids[j] = best;
    }
    double lmax = logit[ids[0]];
    double sum = 0.0;
    for (int j = 0; j < k; ++j) {
        w[j] = exp((double)logit[ids[j]] - lmax);
        sum += w[j];
    }
    if (!renorm) {
        sum = 0.0;
        for (int e = 0; e < E; ++e)
            sum += exp((double)logit[e] - lmax);
    }
    for (int j = 0; j < k; ++j)
        w[j] /= sum;
}

/* The layer's routing: renormalised over the k selected. */
static void route_token(const float *logit, int E, int k, int32_t *ids, double *w)
{
    route_token_r(logit, E, k, 1, ids, w);
}

typedef struct {
    const uint16_t *x, *Wr;
    const float *bias;
    int T, H, E, k, renorm;
    int32_t *ids;
    double *w;
    float *logits;
    int t0, t1;
} route_job;

static void *route_worker(void *arg)
{
    route_job *J = (route_job *)arg;
    float *l = (float *)malloc(sizeof(float) * J->E);
    for (int t = J->t0; t < J->t1; ++t) {
        for (int e = 0; e < J->E; ++e)
            l[e] = oracle_router_logit(J->x + (size_t)t * J->H, J->Wr + (size_t)e * J->H, J->H, J->bias, e);
        if (J->logits)
            memcpy(J->logits + (size_t)t * J->E, l, sizeof(float) * J->E);
        route_token_r(l, J->E, J->k, J->renorm, J->ids + (size_t)t * J->k, J->w + (size_t)t * J->k);
    }
    free(l);
    return NULL;
}

static int clamp_threads(int nthreads, int work)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > work)
        nthreads = work;
    if (nthreads > 256)
        nthreads = 256;
    return nthreads < 1 ? 1 : nthreads;
}

/* ids [T,k] int32, w [T,k] fp64, logits [T,E] fp32 (nullable); renorm as in route_token_r. */
int oracle_route(const uint16_t *x, const uint16_t *Wr, const float *bias, int T, int H, int E, int k, int renorm,
                 int32_t *ids, double *w, float *logits, int nthreads)
{
    if (T <= 0)
        return 0;
    nthreads = clamp_threads(nthreads, T);
    pthread_t th[256];
    route_job jobs[256];
    for (int i = 0; i < nthreads; ++i) {
        route_job J = {x, Wr, bias, T, H, E, k, renorm, ids, w, logits,
                       (int)((long)T * i / nthreads), (int)((long)T * (i + 1) / nthreads)};
        jobs[i] = J;
        pthread_create(&th[i], NULL, route_worker, &jobs[i]);
    }
    for (int i = 0; i < nthreads; ++i)
        pthread_join(th[i], NULL);
    return 0;
}

/* ---------------------------------------------------------- align-sort */
/*
 * Reorder the T*k slots (slot s = t*k + j) by expert.  Expert e's segment
 * holds its slots in ascending s, padded with the sentinel S = T*k up to a
 * whole number of blocks of B rows; segments follow in ascending e; experts
 * without slots get no block.  Buffers are sized as on the page:
 * P_max = T*k + E*B - k entries and ceil(P_max / B) blocks.  Unused entries
 * of sorted_ids hold S and unused block entries hold -1.
 */
int oracle_align_sort(const int32_t *ids, int T, int k, int E, int B, int32_t *sorted_ids,
                      int32_t *sorted_expert_ids, int32_t *num_post_padded, int32_t *counts)
{
    long S = (long)T * k;
    long P_max = S + (long)E * B - k;
    long NB_max = (P_max + B - 1) / B;
    for (long i = 0; i < P_max; ++i)
        sorted_ids[i] = (int32_t)S;
    for (long b = 0; b < NB_max; ++b)
        sorted_expert_ids[b] = -1;
    long pos = 0;
    for (int e = 0; e < E; ++e) {
        long cnt = 0;
        for (long s = 0; s < S; ++s)
            if (ids[s] == e)
                sorted_ids[pos + cnt++] = (int32_t)s;
        counts[e] = (int32_t)cnt;
        long padded = (cnt + B - 1) / B * B;
        for (long b = pos / B; b < (pos + padded) / B; ++b)
            sorted_expert_ids[b] = e;
        pos += padded;
    }
    *num_post_padded = (int32_t)pos;
    return 0;
}

/* ------------------------------------------------------------ forward */

static double silu(double g) { return g / (1.0 + exp(-g)); }

/*
 * Quantisation of the SwiGLU output a[0..I) between the two stages, as the
 * two-stage path does it (the intermediate is quantised before the down
 * projection): mode 1 per 1x128 group (e4m3, scale amax/448), mode 2 one
 * scale for the whole row (per token), mode 3 MXFP4 per 1x32 group; mode 0
 * keeps the value.  a is replaced by the dequantised value.
 */
static void requant_inter(int mode, double *a, int I)
{
    if (mode == 1) {
        for (int gi = 0; gi < I / 128; ++gi) {
            float amax = 0.0f;
            for (int i = gi * 128; i < gi * 128 + 128; ++i) {
                float v = fabsf((float)a[i]);
                if (v > amax)
                    amax = v;
            }
            float sc = group_scale(amax);
            for (int i = gi * 128; i < gi * 128 + 128; ++i)
                a[i] = oracle_e4m3_decode(oracle_e4m3_encode((float)a[i] / sc)) * (double)sc;
        }
    } else if (mode == 3) {
        for (int gi = 0; gi < I / 32; ++gi) {
            float amax = 0.0f;
            for (int i = gi * 32; i < gi * 32 + 32; ++i) {
                float v = fabsf((float)a[i]);
                if (v > amax)
                    amax = v;
            }
            int ex = oracle_mx_exponent(amax);
            for (int i = gi * 32; i < gi * 32 + 32; ++i)
                a[i] = ldexp(oracle_e2m1_decode(oracle_e2m1_encode((float)ldexp((double)(float)a[i], -ex))), ex);
        }
    } else if (mode == 2) {
        float amax = 0.0f;
        for (int i = 0; i < I; ++i) {
            float v = fabsf((float)a[i]);
            if (v > amax)
                amax = v;
        }
        float sc = group_scale(amax);
        for (int i = 0; i < I; ++i)
            a[i] = oracle_e4m3_decode(oracle_e4m3_encode((float)a[i] / sc)) * (double)sc;
    }
}

typedef struct {
    int mode; /* 0 bf16, 1 fp8 per 128x128 / 1x128 blocks, 2 fp8 per row, 3 mxfp4 per 1x32 */
    const uint16_t *x, *Wr;
    const float *bias;
    const uint16_t *Wgu, *Wd;                /* bf16 weights */
    const uint8_t *Wgu_q, *Wd_q;             /* e4m3 codes */
    const float *w1s, *w2s;                  /* block scales (mode 1) or row scales (mode 2) */
    const uint8_t *w1x, *w2x;                /* E8M0 scales per 1x32 (mode 3) */
    int T, H, I, E, k;
    const int64_t *tokens;
    int n0, n1;
    double *out; /* [n, H] */
} fwd_job;

static void token_input(int mode, const uint16_t *xrow, int H, double *xt, uint8_t *xq, float *xs, uint8_t *xsx);

static void *fwd_worker(void *arg)
{
    fwd_job *J = (fwd_job *)arg;
    int H = J->H, I = J->I, E = J->E, k = J->k;
    float *l = (float *)malloc(sizeof(float) * E);
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * k);
    double *w = (double *)malloc(sizeof(double) * k);
    double *xt = (double *)malloc(sizeof(double) * H);
    double *a = (double *)malloc(sizeof(double) * I);
    uint8_t *xq = (uint8_t *)malloc(H);
    float *xs = (float *)malloc(sizeof(float) * (H / 128 + 1));
    uint8_t *xsx = (uint8_t *)malloc(H / 32 + 1);
    for (int n = J->n0; n < J->n1; ++n) {
        long t = (long)J->tokens[n];
        const uint16_t *xrow = J->x + t * H;
        for (int e = 0; e < E; ++e)
            l[e] = oracle_router_logit(xrow, J->Wr + (size_t)e * H, H, J->bias, e);
        route_token(l, E, k, ids, w);
        token_input(J->mode, xrow, H, xt, xq, xs, xsx);
        double *o = J->out + (size_t)n * H;
        for (int h = 0; h < H; ++h)
            o[h] = 0.0;
        for (int j = 0; j < k; ++j) {
            int e = ids[j];
            for (int i = 0; i < I; ++i) {
                double g = 0.0, u = 0.0;
                size_t rg = ((size_t)e * 2 * I + i) * H;
                size_t ru = ((size_t)e * 2 * I + I + i) * H;
                if (J->mode == 0) {
                    for (int h = 0; h < H; ++h) {
                        g += (double)bf16_to_float(J->Wgu[rg + h]) * xt[h];
                        u += (double)bf16_to_float(J->Wgu[ru + h]) * xt[h];
                    }
                } else if (J->mode == 3) {
                    for (int h = 0; h < H; ++h) {
                        g += mx4_value(J->Wgu_q, J->w1x, (long)rg + h, H) * xt[h];
                        u += mx4_value(J->Wgu_q, J->w1x, (long)ru + h, H) * xt[h];
                    }
                } else if (J->mode == 2) {
                    /* one scale per output channel (row of the [E*2I, H] matrix) */
                    const double sg = J->w1s[(size_t)e * 2 * I + i];
                    const double su = J->w1s[(size_t)e * 2 * I + I + i];
                    for (int h = 0; h < H; ++h) {
                        g += oracle_e4m3_decode(J->Wgu_q[rg + h]) * sg * xt[h];
                        u += oracle_e4m3_decode(J->Wgu_q[ru + h]) * su * xt[h];
                    }
                } else {
                    /* block (row/128, col/128) of the [E*2I, H] matrix */
                    const float *sg = J->w1s + ((size_t)e * 2 * I + i) / 128 * (H / 128);
                    const float *su = J->w1s + ((size_t)e * 2 * I + I + i) / 128 * (H / 128);
                    for (int h = 0; h < H; ++h) {
                        g += oracle_e4m3_decode(J->Wgu_q[rg + h]) * (double)sg[h / 128] * xt[h];
                        u += oracle_e4m3_decode(J->Wgu_q[ru + h]) * (double)su[h / 128] * xt[h];
                    }
                }
                a[i] = silu(g) * u;
            }
            requant_inter(J->mode, a, I);
            for (int h = 0; h < H; ++h) {
                double y = 0.0;
                size_t rd = ((size_t)e * H + h) * I;
                if (J->mode == 0) {
                    for (int i = 0; i < I; ++i)
                        y += (double)bf16_to_float(J->Wd[rd + i]) * a[i];
                } else if (J->mode == 3) {
                    for (int i = 0; i < I; ++i)
                        y += mx4_value(J->Wd_q, J->w2x, (long)rd + i, I) * a[i];
                } else if (J->mode == 2) {
                    const double sd = J->w2s[(size_t)e * H + h];
                    for (int i = 0; i < I; ++i)
                        y += oracle_e4m3_decode(J->Wd_q[rd + i]) * sd * a[i];
                } else {
                    const float *sd = J->w2s + ((size_t)e * H + h) / 128 * (I / 128);
                    for (int i = 0; i < I; ++i)
                        y += oracle_e4m3_decode(J->Wd_q[rd + i]) * (double)sd[i / 128] * a[i];
                }
                o[h] += w[j] * y;
            }
        }
    }
    free(l);
    free(ids);
    free(w);
    free(xt);
    free(a);
    free(xq);
    free(xs);
    free(xsx);
    return NULL;
}

static int run_forward(fwd_job proto, int n_tokens, int nthreads)
{
    if (n_tokens <= 0)
        return 0;
    nthreads = clamp_threads(nthreads, n_tokens);
    pthread_t th[256];
    fwd_job jobs[256];
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = proto;
        jobs[i].n0 = (int)((long)n_tokens * i / nthreads);
        jobs[i].n1 = (int)((long)n_tokens * (i + 1) / nthreads);
        pthread_create(&th[i], NULL, fwd_worker, &jobs[i]);
    }
    for (int i = 0; i < nthreads; ++i)
        pthread_join(th[i], NULL);
    return 0;
}

/*
 * bf16 layer: x [T,H], W_router [E,H], bias [E] (nullable),
 * W_gate_up [E,2I,H] (gate rows first), W_down [E,H,I], all bf16 bits.
 * Computes out[n,:] (fp64) for the tokens listed in tokens[0..n_tokens).
 */
int oracle_moe_forward_bf16(const uint16_t *x, const uint16_t *Wr, const float *bias, const uint16_t *Wgu,
                            const uint16_t *Wd, int T, int H, int I, int E, int k, const int64_t *tokens,
                            int n_tokens, double *out, int nthreads)
{
    fwd_job J;
    memset(&J, 0, sizeof J);
    J.mode = 0;
    J.x = x;
    J.Wr = Wr;
    J.bias = bias;
    J.Wgu = Wgu;
    J.Wd = Wd;
    J.T = T;
    J.H = H;
    J.I = I;
    J.E = E;
    J.k = k;
    J.tokens = tokens;
    J.out = out;
    return run_forward(J, n_tokens, nthreads);
}

/*
 * Block-scaled FP8 layer: the router runs on the bf16 activations; the
 * expert GEMMs see x quantised per 1x128 group, weights as e4m3 codes with
 * one fp32 scale per 128x128 block (w1s [E*2I/128, H/128], w2s [E*H/128,
 * I/128]) and the SwiGLU output re-quantised per 1x128 group.  Products are
 * of the dequantised values (code * scale), accumulated in fp64.
 */
int oracle_moe_forward_fp8(const uint16_t *x, const uint16_t *Wr, const float *bias, const uint8_t *Wgu_q,
                           const float *w1s, const uint8_t *Wd_q, const float *w2s, int T, int H, int I, int E,
                           int k, const int64_t *tokens, int n_tokens, double *out, int nthreads)
{
    fwd_job J;
    memset(&J, 0, sizeof J);
    J.mode = 1;
    J.x = x;
    J.Wr = Wr;
    J.bias = bias;
    J.Wgu_q = Wgu_q;
    J.w1s = w1s;
    J.Wd_q = Wd_q;
    J.w2s = w2s;
    J.T = T;
    J.H = H;
    J.I = I;
    J.E = E;
    J.k = k;
    J.tokens = tokens;
    J.out = out;
    return run_forward(J, n_tokens, nthreads);
}

/*
 * Per-token FP8 layer ("per_Token" with e4m3 weights): the router runs on
 * the bf16 activations; the expert GEMMs see x quantised with one scale per
 * token, weights as e4m3 codes with one fp32 scale per output channel
 * (w1s [E*2I], w2s [E*H]) and the SwiGLU output re-quantised with one scale
 * per token over its whole intermediate row.  Products are of the
 * dequantised values, accumulated in fp64.
 */
int oracle_moe_forward_fp8_token(const uint16_t *x, const uint16_t *Wr, const float *bias, const uint8_t *Wgu_q,
                                 const float *w1s, const uint8_t *Wd_q, const float *w2s, int T, int H, int I,
                                 int E, int k, const int64_t *tokens, int n_tokens, double *out, int nthreads)
{
    fwd_job J;
    memset(&J, 0, sizeof J);
    J.mode = 2;
    J.x = x;
    J.Wr = Wr;
    J.bias = bias;
    J.Wgu_q = Wgu_q;
    J.w1s = w1s;
    J.Wd_q = Wd_q;
    J.w2s = w2s;
    J.T = T;
    J.H = H;
    J.I = I;
    J.E = E;
    J.k = k;
    J.tokens = tokens;
    J.out = out;
    return run_forward(J, n_tokens, nthreads);
}

/*
 * MXFP4 layer ("per_1x32", microscaling FP4): the router runs on the bf16
 * activations; the expert GEMMs see x quantised per 1x32 group, weights as
 * E2M1 codes (one per byte here) with an E8M0 scale per 1x32 group along K
 * (w1x [E*2I, H/32], w2x [E*H, I/32]) and the SwiGLU output re-quantised
 * per 1x32 group.  Products are of the dequantised values, accumulated in
 * fp64.
 */
int oracle_moe_forward_mxfp4(const uint16_t *x, const uint16_t *Wr, const float *bias, const uint8_t *Wgu_q,
                             const uint8_t *w1x, const uint8_t *Wd_q, const uint8_t *w2x, int T, int H, int I,
                             int E, int k, const int64_t *tokens, int n_tokens, double *out, int nthreads)
{
    fwd_job J;
    memset(&J, 0, sizeof J);
    J.mode = 3;
    J.x = x;
    J.Wr = Wr;
    J.bias = bias;
    J.Wgu_q = Wgu_q;
    J.w1x = w1x;
    J.Wd_q = Wd_q;
    J.w2x = w2x;
    J.T = T;
    J.H = H;
    J.I = I;
    J.E = E;
    J.k = k;
    J.tokens = tokens;
    J.out = out;
    return run_forward(J, n_tokens, nthreads);
}

/* ------------------------------------------- forward, expert by expert */
/*
 * The same layer as the per-token loop above, evaluated expert by expert so
 * that each weight row, once dequantised, serves up to EM_SLOTS slots of the
 * expert (the route-then-group view of the fused-MoE pages: tokens reordered
 * by expert, each expert's rows multiplied by its weights).  Every output
 * value is the same sum in the same order as in the per-token loop:
 *   g, u  = sum over h ascending of (dequantised weight * x), from 0.0
 *   y     = sum over i ascending of (dequantised down weight * a), from 0.0
 *   out_t = sum over j ascending of w_j * y_j, from 0.0
 * so the results are bit-identical to it; only the loop nest is reordered
 * (the slot index innermost), which is what makes full-size comparisons of
 * thousands of tokens affordable.  Tokens are taken in waves that bound the
 * per-slot buffer of y.
 */
#define EM_SLOTS 16

static double g_e4m3_tab[256];
static double g_e2m1_tab[16];
static double g_pow2_tab[256]; /* 2^(b - 127): the value of E8M0 byte b */
static pthread_once_t g_tab_once = PTHREAD_ONCE_INIT;

static void init_tables(void)
{
    for (int c = 0; c < 256; ++c)
        g_e4m3_tab[c] = oracle_e4m3_decode((uint8_t)c);
    for (int c = 0; c < 16; ++c)
        g_e2m1_tab[c] = oracle_e2m1_decode((uint8_t)c);
    for (int b = 0; b < 256; ++b)
        g_pow2_tab[b] = ldexp(1.0, b - 127); /* exact: 2^-127 .. 2^128 are normal doubles */
}

/*
 * Row `row` of a weight stack viewed as [rows][len] (len = the reduction
 * length), dequantised to fp64 exactly as the per-token loop does it: bf16
 * value; e4m3 code * scale of its 128x128 block; e4m3 code * scale of the
 * row; E2M1 code * 2^(E8M0 - 127) of its 1x32 group (the power of two is
 * exact, so this equals ldexp).
 */
static void dequant_row(int mode, const uint16_t *Wb, const uint8_t *Wq, const float *ws, const uint8_t *wx,
                        size_t row, int len, double *out)
{
    if (mode == 0) {
        const uint16_t *r = Wb + row * (size_t)len;
        for (int h = 0; h < len; ++h)
            out[h] = (double)bf16_to_float(r[h]);
    } else if (mode == 1) {
        const uint8_t *r = Wq + row * (size_t)len;
        const float *sb = ws + row / 128 * (size_t)(len / 128);
        for (int h = 0; h < len; ++h)
            out[h] = g_e4m3_tab[r[h]] * (double)sb[h / 128];
    } else if (mode == 2) {
        const uint8_t *r = Wq + row * (size_t)len;
        const double sr = ws[row];
        for (int h = 0; h < len; ++h)
            out[h] = g_e4m3_tab[r[h]] * sr;
    } else {
        const uint8_t *r = Wq + row * (size_t)len;
        const uint8_t *sx = wx + row * (size_t)(len / 32);
        for (int h = 0; h < len; ++h)
            out[h] = g_e2m1_tab[r[h] & 15] * g_pow2_tab[sx[h / 32]];
    }
}

/* The token row x_t as the expert GEMMs see it (bf16, or dequantised codes). */
static void token_input(int mode, const uint16_t *xrow, int H, double *xt, uint8_t *xq, float *xs, uint8_t *xsx)
{
    if (mode == 0) {
        for (int h = 0; h < H; ++h)
            xt[h] = bf16_to_float(xrow[h]);
    } else if (mode == 1) {
        oracle_quant_1x128(xrow, 1, H, xq, xs);
        for (int h = 0; h < H; ++h)
            xt[h] = oracle_e4m3_decode(xq[h]) * (double)xs[h / 128];
    } else if (mode == 2) {
        oracle_quant_rows(xrow, 1, H, xq, xs);
        for (int h = 0; h < H; ++h)
            xt[h] = oracle_e4m3_decode(xq[h]) * (double)xs[0];
    } else {
        oracle_quant_mx4(xrow, 1, H, xq, xsx);
        for (int h = 0; h < H; ++h)
            xt[h] = mx4_value(xq, xsx, h, H);
    }
}

typedef struct {
    fwd_job f;          /* weights, shape, mode */
    const int64_t *tok; /* tokens of this wave */
    int nw;
    double *xt;         /* [nw][H] */
    int32_t *ids;       /* [nw][k] */
    double *w;          /* [nw][k] */
    double *Y;          /* [nw][k][H] */
    double *out;        /* [nw][H] */
    int32_t *slots;     /* wave slots n*k + j grouped by expert, ascending within an expert */
    int32_t *item_e, *item_first, *item_len;
    int n_items;
    int next;           /* next unclaimed unit of the current phase */
    int phase;          /* 0 route + inputs, 1 expert items, 2 combine */
    pthread_mutex_t mu;
} em_state;

static int em_claim(em_state *S, int limit)
{
    pthread_mutex_lock(&S->mu);
    int i = S->next < limit ? S->next++ : -1;
    pthread_mutex_unlock(&S->mu);
    return i;
}

/* acc[s] = sum over h ascending of w[h] * X[h][s], from 0.0, for the EM_SLOTS columns of X [n][EM_SLOTS]. */
__attribute__((noinline)) static void em_dot(const double *w, const double *X, int n, double *acc)
{
    double a[EM_SLOTS];
    for (int s = 0; s < EM_SLOTS; ++s)
        a[s] = 0.0;
    for (int h = 0; h < n; ++h) {
        const double wh = w[h];
        const double *xr = X + (size_t)h * EM_SLOTS;
        for (int s = 0; s < EM_SLOTS; ++s)
            a[s] += wh * xr[s];
    }
    for (int s = 0; s < EM_SLOTS; ++s)
        acc[s] = a[s];
}

static void em_item(em_state *S, int it, double *Xt, double *wg, double *wu, double *At, double *acol)
{
    const fwd_job *J = &S->f;
    const int H = J->H, I = J->I, k = J->k, mode = J->mode;
    const int e = S->item_e[it], nb = S->item_len[it];
    const int32_t *sl = S->slots + S->item_first[it];
    for (int h = 0; h < H; ++h)
        for (int s = 0; s < EM_SLOTS; ++s)
            Xt[(size_t)h * EM_SLOTS + s] = s < nb ? S->xt[(size_t)(sl[s] / k) * H + h] : 0.0;
    for (int i = 0; i < I; ++i) {
        dequant_row(mode, J->Wgu, J->Wgu_q, J->w1s, J->w1x, (size_t)e * 2 * I + i, H, wg);
        dequant_row(mode, J->Wgu, J->Wgu_q, J->w1s, J->w1x, (size_t)e * 2 * I + I + i, H, wu);
        double g[EM_SLOTS], u[EM_SLOTS];
        em_dot(wg, Xt, H, g);
        em_dot(wu, Xt, H, u);
        for (int s = 0; s < EM_SLOTS; ++s)
            At[(size_t)i * EM_SLOTS + s] = silu(g[s]) * u[s];
    }
    if (mode != 0) {
        for (int s = 0; s < nb; ++s) {
            for (int i = 0; i < I; ++i)
                acol[i] = At[(size_t)i * EM_SLOTS + s];
            requant_inter(mode, acol, I);
            for (int i = 0; i < I; ++i)
                At[(size_t)i * EM_SLOTS + s] = acol[i];
        }
    }
    for (int h = 0; h < H; ++h) {
        dequant_row(mode, J->Wd, J->Wd_q, J->w2s, J->w2x, (size_t)e * H + h, I, wg);
        double y[EM_SLOTS];
        em_dot(wg, At, I, y);
        for (int s = 0; s < nb; ++s)
            S->Y[(size_t)sl[s] * H + h] = y[s];
    }
}

static void *em_worker(void *arg)
{
    em_state *S = (em_state *)arg;
    const fwd_job *J = &S->f;
    const int H = J->H, I = J->I, E = J->E, k = J->k;
    if (S->phase == 0) {
        float *l = (float *)malloc(sizeof(float) * E);
        uint8_t *xq = (uint8_t *)malloc(H);
        float *xs = (float *)malloc(sizeof(float) * (H / 128 + 1));
        uint8_t *xsx = (uint8_t *)malloc(H / 32 + 1);
        for (int n; (n = em_claim(S, S->nw)) >= 0;) {
            const uint16_t *xrow = J->x + (size_t)S->tok[n] * H;
            for (int e = 0; e < E; ++e)
                l[e] = oracle_router_logit(xrow, J->Wr + (size_t)e * H, H, J->bias, e);
            route_token(l, E, k, S->ids + (size_t)n * k, S->w + (size_t)n * k);
            token_input(J->mode, xrow, H, S->xt + (size_t)n * H, xq, xs, xsx);
        }
        free(l);
        free(xq);
        free(xs);
        free(xsx);
    } else if (S->phase == 1) {
        const int L = H > I ? H : I;
        double *Xt = (double *)malloc(sizeof(double) * (size_t)H * EM_SLOTS);
        double *At = (double *)malloc(sizeof(double) * (size_t)I * EM_SLOTS);
        double *wg = (double *)malloc(sizeof(double) * L);
        double *wu = (double *)malloc(sizeof(double) * L);
        double *acol = (double *)malloc(sizeof(double) * I);
        for (int it; (it = em_claim(S, S->n_items)) >= 0;)
            em_item(S, it, Xt, wg, wu, At, acol);
        free(Xt);
        free(At);
        free(wg);
        free(wu);
        free(acol);
    } else {
        for (int n; (n = em_claim(S, S->nw)) >= 0;) {
            double *o = S->out + (size_t)n * H;
            for (int h = 0; h < H; ++h)
                o[h] = 0.0;
            for (int j = 0; j < k; ++j) {
                const double wj = S->w[(size_t)n * k + j];
                const double *y = S->Y + ((size_t)n * k + j) * H;
                for (int h = 0; h < H; ++h)
                    o[h] += wj * y[h];
            }
        }
    }
    return NULL;
}

static void em_run_phase(em_state *S, int phase, int nthreads, int work)
{
    S->phase = phase;
    S->next = 0;
    int nt = clamp_threads(nthreads, work > 0 ? work : 1);
    pthread_t th[256];
    for (int i = 0; i < nt; ++i)
        pthread_create(&th[i], NULL, em_worker, S);
    for (int i = 0; i < nt; ++i)
        pthread_join(th[i], NULL);
}

/*
 * mode as in the per-token entries (0 bf16, 1 block FP8, 2 per-token FP8,
 * 3 MXFP4) with the same weight and scale arguments (unused ones NULL).
 * Returns 0, or -1 if scratch cannot be allocated.
 */
int oracle_moe_forward_expert_major(int mode, const uint16_t *x, const uint16_t *Wr, const float *bias,
                                    const void *Wgu, const void *w1scale, const void *Wd, const void *w2scale,
                                    int T, int H, int I, int E, int k, const int64_t *tokens, int n_tokens,
                                    double *out, int nthreads)
{
    pthread_once(&g_tab_once, init_tables);
    em_state S;
    memset(&S, 0, sizeof S);
    fwd_job *J = &S.f;
    J->mode = mode;
    J->x = x;
    J->Wr = Wr;
    J->bias = bias;
    if (mode == 0) {
        J->Wgu = (const uint16_t *)Wgu;
        J->Wd = (const uint16_t *)Wd;
    } else {
        J->Wgu_q = (const uint8_t *)Wgu;
        J->Wd_q = (const uint8_t *)Wd;
    }
    if (mode == 1 || mode == 2) {
        J->w1s = (const float *)w1scale;
        J->w2s = (const float *)w2scale;
    } else if (mode == 3) {
        J->w1x = (const uint8_t *)w1scale;
        J->w2x = (const uint8_t *)w2scale;
    }
    J->T = T;
    J->H = H;
    J->I = I;
    J->E = E;
    J->k = k;
    if (n_tokens <= 0)
        return 0;
    /* a wave keeps y of all its slots: at most ~512 MB */
    long wave = (512L << 20) / ((long)k * H * (long)sizeof(double));
    if (wave < 1)
        wave = 1;
    if (wave > n_tokens)
        wave = n_tokens;
    S.xt = (double *)malloc(sizeof(double) * (size_t)wave * H);
    S.ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)wave * k);
    S.w = (double *)malloc(sizeof(double) * (size_t)wave * k);
    S.Y = (double *)malloc(sizeof(double) * (size_t)wave * k * H);
    S.slots = (int32_t *)malloc(sizeof(int32_t) * (size_t)wave * k);
    long max_items = (long)wave * k / EM_SLOTS + E + 1;
    S.item_e = (int32_t *)malloc(sizeof(int32_t) * max_items);
    S.item_first = (int32_t *)malloc(sizeof(int32_t) * max_items);
    S.item_len = (int32_t *)malloc(sizeof(int32_t) * max_items);
    int32_t *cnt = (int32_t *)calloc((size_t)E + 1, sizeof(int32_t));
    int rc = 0;
    if (!S.xt || !S.ids || !S.w || !S.Y || !S.slots || !S.item_e || !S.item_first || !S.item_len || !cnt)
        rc = -1;
    pthread_mutex_init(&S.mu, NULL);
    for (long n0 = 0; rc == 0 && n0 < n_tokens; n0 += wave) {
        S.tok = tokens + n0;
        S.nw = (int)((n_tokens - n0) < wave ? (n_tokens - n0) : wave);
        S.out = out + (size_t)n0 * H;
        em_run_phase(&S, 0, nthreads, S.nw);
        /* group the wave's slots by expert (ascending slot within an expert) */
        for (int e = 0; e <= E; ++e)
            cnt[e] = 0;
        for (long s = 0; s < (long)S.nw * k; ++s)
            cnt[S.ids[s] + 1]++;
        for (int e = 0; e < E; ++e)
            cnt[e + 1] += cnt[e];
        S.n_items = 0;
        for (int e = 0; e < E; ++e) {
            int pos = cnt[e];
            for (long s = 0; s < (long)S.nw * k; ++s)
                if (S.ids[s] == e)
                    S.slots[pos++] = (int32_t)s;
            for (int f = cnt[e]; f < cnt[e + 1]; f += EM_SLOTS) {
                S.item_e[S.n_items] = e;
                S.item_first[S.n_items] = f;
                S.item_len[S.n_items] = cnt[e + 1] - f < EM_SLOTS ? cnt[e + 1] - f : EM_SLOTS;
                S.n_items++;
            }
        }
        em_run_phase(&S, 1, nthreads, S.n_items);
        em_run_phase(&S, 2, nthreads, S.nw);
    }
    pthread_mutex_destroy(&S.mu);
    free(S.xt);
    free(S.ids);
    free(S.w);
    free(S.Y);
    free(S.slots);
    free(S.item_e);
    free(S.item_first);
    free(S.item_len);
    free(cnt);
    return rc;
}

/* ------------------------------------------------------------ backward */
/*
 * Gradients of the bf16 layer (the training direction of the group GEMMs:
 * "dgrad" of both stages and "wgrad" of both weight stacks, plus the
 * router), for loss = sum_t dout_t . out_t.  The top-k choice is a
 * selection (no gradient); the weights of the chosen experts carry the
 * gradient to their logits through the softmax over the k:
 *
 *   dy_j = w_j dout                      dh_j = W_down[e_j]^T dy_j
 *   dg = dh * u * silu'(g)               du = dh * silu(g),
 *        silu'(g) = s (1 + g (1 - s)),   s = 1 / (1 + exp(-g))
 *   dx  = sum_j (W_gate[e_j]^T dg_j + W_up[e_j]^T du_j) + sum_j dl_j W_router[e_j]
 *   dw_j = dout . y_j                    dl_j = w_j (dw_j - sum_m w_m dw_m)
 *   dW_down[e] = sum over e's slots of dy h^T,  dW_gate[e] = sum dg x^T,
 *   dW_up[e] = sum du x^T,  dW_router[e] = sum_t dl_{t,e} x_t,  dbias_e = sum_t dl_{t,e}
 *
 * All in fp64 (the logits and the routing as in the forward).  Phase 1 runs
 * per token; phase 2 sums the weight gradients over tokens per expert row.
 */
typedef struct {
    const uint16_t *x, *Wr, *Wgu, *Wd, *dout;
    const float *bias;
    int T, H, I, E, k;
    int32_t *ids;    /* [T, k] */
    double *w;       /* [T, k] */
    double *dl;      /* [T, E] */
    double *hbuf;    /* [T*k, I]: h */
    double *dgbuf;   /* [T*k, I]: dg */
    double *dubuf;   /* [T*k, I]: du */
    double *dx;      /* [T, H] */
    int t0, t1;
} bwd_job;

static void *bwd_token_worker(void *arg)
{
    bwd_job *J = (bwd_job *)arg;
    int H = J->H, I = J->I, E = J->E, k = J->k;
    float *l = (float *)malloc(sizeof(float) * E);
    double *xt = (double *)malloc(sizeof(double) * H);
    double *dout = (double *)malloc(sizeof(double) * H);
    double *g = (double *)malloc(sizeof(double) * I);
    double *u = (double *)malloc(sizeof(double) * I);
    double *y = (double *)malloc(sizeof(double) * H);
    double *dw = (double *)malloc(sizeof(double) * k);
    for (int t = J->t0; t < J->t1; ++t) {
        const uint16_t *xrow = J->x + (size_t)t * H;
        for (int e = 0; e < E; ++e)
            l[e] = oracle_router_logit(xrow, J->Wr + (size_t)e * H, H, J->bias, e);
        int32_t *ids = J->ids + (size_t)t * k;
        double *w = J->w + (size_t)t * k;
        route_token(l, E, k, ids, w);
        for (int h = 0; h < H; ++h) {
            xt[h] = bf16_to_float(xrow[h]);
            dout[h] = bf16_to_float(J->dout[(size_t)t * H + h]);
        }
        double *dx = J->dx + (size_t)t * H;
        for (int h = 0; h < H; ++h)
            dx[h] = 0.0;
        for (int j = 0; j < k; ++j) {
            int e = ids[j];
            double *hh = J->hbuf + ((size_t)t * k + j) * I;
            double *dg = J->dgbuf + ((size_t)t * k + j) * I;
            double *du = J->dubuf + ((size_t)t * k + j) * I;
            for (int i = 0; i < I; ++i) {
                const uint16_t *rg = J->Wgu + ((size_t)e * 2 * I + i) * H;
                const uint16_t *ru = J->Wgu + ((size_t)e * 2 * I + I + i) * H;
                double gs = 0.0, us = 0.0;
                for (int h = 0; h < H; ++h) {
                    gs += (double)bf16_to_float(rg[h]) * xt[h];
                    us += (double)bf16_to_float(ru[h]) * xt[h];
                }
                g[i] = gs;
                u[i] = us;
                hh[i] = silu(gs) * us;
            }
            /* y_j and dh_j = W_down^T (w_j dout) */
            for (int i = 0; i < I; ++i)
                dg[i] = 0.0; /* dh accumulates here first */
            double dwj = 0.0;
            for (int h = 0; h < H; ++h) {
                const uint16_t *rd = J->Wd + ((size_t)e * H + h) * I;
                double yh = 0.0;
                for (int i = 0; i < I; ++i)
                    yh += (double)bf16_to_float(rd[i]) * hh[i];
                y[h] = yh;
                dwj += dout[h] * yh;
                double dyh = w[j] * dout[h];
                for (int i = 0; i < I; ++i)
                    dg[i] += (double)bf16_to_float(rd[i]) * dyh;
            }
            dw[j] = dwj;
            for (int i = 0; i < I; ++i) {
                double dh = dg[i];
                double sg = 1.0 / (1.0 + exp(-g[i]));
                dg[i] = dh * u[i] * sg * (1.0 + g[i] * (1.0 - sg));
                du[i] = dh * g[i] * sg;
            }
            for (int i = 0; i < I; ++i) {
                const uint16_t *rg = J->Wgu + ((size_t)e * 2 * I + i) * H;
                const uint16_t *ru = J->Wgu + ((size_t)e * 2 * I + I + i) * H;
                for (int h = 0; h < H; ++h)
                    dx[h] += dg[i] * (double)bf16_to_float(rg[h]) + du[i] * (double)bf16_to_float(ru[h]);
            }
        }
        /* softmax over the k chosen logits */
        double sw = 0.0;
        for (int j = 0; j < k; ++j)
            sw += w[j] * dw[j];
        double *dl = J->dl + (size_t)t * E;
        for (int e = 0; e < E; ++e)
            dl[e] = 0.0;
        for (int j = 0; j < k; ++j)
            dl[ids[j]] = w[j] * (dw[j] - sw);
        for (int j = 0; j < k; ++j) {
            const uint16_t *rr = J->Wr + (size_t)ids[j] * H;
            for (int h = 0; h < H; ++h)
                dx[h] += dl[ids[j]] * (double)bf16_to_float(rr[h]);
        }
    }
    free(l);
    free(xt);
    free(dout);
    free(g);
    free(u);
    free(y);
    free(dw);
    return NULL;
}

typedef struct {
    const bwd_job *P;
    double *dWgu, *dWd, *dWr, *dbias;
    int e0, e1; /* experts of this worker */
} wgrad_job;

static void *bwd_weight_worker(void *arg)
{
    wgrad_job *W = (wgrad_job *)arg;
    const bwd_job *J = W->P;
    int T = J->T, H = J->H, I = J->I, E = J->E, k = J->k;
    for (int e = W->e0; e < W->e1; ++e) {
        double *dWg = W->dWgu + (size_t)e * 2 * I * H;
        double *dWu = dWg + (size_t)I * H;
        double *dWd = W->dWd + (size_t)e * H * I;
        double *dWr = W->dWr + (size_t)e * H;
        memset(dWg, 0, sizeof(double) * 2 * I * H);
        memset(dWd, 0, sizeof(double) * H * I);
        memset(dWr, 0, sizeof(double) * H);
        double db = 0.0;
        for (int t = 0; t < T; ++t) {
            const uint16_t *xrow = J->x + (size_t)t * H;
            double dle = J->dl[(size_t)t * E + e];
            db += dle;
            for (int h = 0; h < H; ++h)
                dWr[h] += dle * (double)bf16_to_float(xrow[h]);
            for (int j = 0; j < k; ++j) {
                if (J->ids[(size_t)t * k + j] != e)
                    continue;
                const double *hh = J->hbuf + ((size_t)t * k + j) * I;
                const double *dg = J->dgbuf + ((size_t)t * k + j) * I;
                const double *du = J->dubuf + ((size_t)t * k + j) * I;
                double wj = J->w[(size_t)t * k + j];
                for (int h = 0; h < H; ++h) {
                    double dyh = wj * (double)bf16_to_float(J->dout[(size_t)t * H + h]);
                    for (int i = 0; i < I; ++i)
                        dWd[(size_t)h * I + i] += dyh * hh[i];
                }
                for (int i = 0; i < I; ++i)
                    for (int h = 0; h < H; ++h) {
                        double xv = (double)bf16_to_float(xrow[h]);
                        dWg[(size_t)i * H + h] += dg[i] * xv;
                        dWu[(size_t)i * H + h] += du[i] * xv;
                    }
            }
        }
        W->dbias[e] = db;
    }
    return NULL;
}

/*
 * Backward of the bf16 layer.  x, W_router, W_gate_up, W_down as in the
 * forward, dout [T, H] bf16 bits.  Outputs (fp64): dx [T, H],
 * dW_gate_up [E, 2I, H], dW_down [E, H, I], dW_router [E, H], dbias [E]
 * (always written; 0 where an expert takes no token).  Returns 0, or -1 if
 * the per-slot scratch cannot be allocated.
 */
int oracle_moe_backward_bf16(const uint16_t *x, const uint16_t *Wr, const float *bias, const uint16_t *Wgu,
                             const uint16_t *Wd, const uint16_t *dout, int T, int H, int I, int E, int k, double *dx,
                             double *dWgu, double *dWd, double *dWr, double *dbias, int nthreads)
{
    bwd_job P;
    memset(&P, 0, sizeof P);
    P.x = x;
    P.Wr = Wr;
    P.bias = bias;
    P.Wgu = Wgu;
    P.Wd = Wd;
    P.dout = dout;
    P.T = T;
    P.H = H;
    P.I = I;
    P.E = E;
    P.k = k;
    P.ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)T * k);
    P.w = (double *)malloc(sizeof(double) * (size_t)T * k);
    P.dl = (double *)malloc(sizeof(double) * (size_t)T * E);
    P.hbuf = (double *)malloc(sizeof(double) * (size_t)T * k * I);
    P.dgbuf = (double *)malloc(sizeof(double) * (size_t)T * k * I);
    P.dubuf = (double *)malloc(sizeof(double) * (size_t)T * k * I);
    P.dx = dx;
    int rc = 0;
    if (!P.ids || !P.w || !P.dl || !P.hbuf || !P.dgbuf || !P.dubuf) {
        rc = -1;
    } else if (T > 0) {
        int nt = clamp_threads(nthreads, T);
        pthread_t th[256];
        bwd_job jobs[256];
        for (int i = 0; i < nt; ++i) {
            jobs[i] = P;
            jobs[i].t0 = (int)((long)T * i / nt);
            jobs[i].t1 = (int)((long)T * (i + 1) / nt);
            pthread_create(&th[i], NULL, bwd_token_worker, &jobs[i]);
        }
        for (int i = 0; i < nt; ++i)
            pthread_join(th[i], NULL);
        int ne = clamp_threads(nthreads, E);
        wgrad_job wj[256];
        for (int i = 0; i < ne; ++i) {
            wj[i].P = &P;
            wj[i].dWgu = dWgu;
            wj[i].dWd = dWd;
            wj[i].dWr = dWr;
            wj[i].dbias = dbias;
            wj[i].e0 = (int)((long)E * i / ne);
            wj[i].e1 = (int)((long)E * (i + 1) / ne);
            pthread_create(&th[i], NULL, bwd_weight_worker, &wj[i]);
        }
        for (int i = 0; i < ne; ++i)
            pthread_join(th[i], NULL);
    }
    free(P.ids);
    free(P.w);
    free(P.dl);
    free(P.hbuf);
    free(P.dgbuf);
    free(P.dubuf);
    return rc;
}

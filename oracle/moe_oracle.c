/*
 * CPU ORACLE for the routed 4-bit MoE layer -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously correct C. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it. It shares no code, header,
 * table or helper with the CUDA library; neither includes the other.
 *
 * Source: the DiffusionGemma language-model page ("diffusion-gemma/model.ts"),
 * classes DiffRouter (router forward), DiffExperts (experts forward),
 * DiffusionGemmaDecoderLayer (the MoE and dense branches' norms) and
 * SelfConditioning (the dense 4-bit GeGLU MLP), logitsFromHidden (the tied
 * 4-bit head and its softcap), and
 * the vision page ("diffusion-gemma/vision.ts", manualRms) for the fp32
 * semantics of the no-scale RMS norm.
 *
 * Precision rules used here:
 *  - Every tensor the pages hold in the model dtype is rounded to bf16
 *    (round to nearest even) exactly where the pages produce it.
 *  - Where the pages fix the arithmetic precision it is followed: the RMS
 *    norm is fp32 (manualRms: x_f32 * rsqrt(mean(x^2) + eps), cast back;
 *    the fp32 mean is the exact mean rounded once) and the routing softmax
 *    is fp32 ("precise" softmax).
 *  - Where the pages are silent (matmul accumulation, GeGLU internals, the
 *    k-way sum of the combine) the oracle computes in double and rounds once
 *    to the bf16 of the exact value.
 *  - A 4-bit weight dequantises to the model dtype: w = bf16(S*q + B), as the
 *    pages' `dequantize` of a quantized table yields a bf16 matmul operand
 *    (DiffusionGemmaModel.dequantEmbedWeight, used by softEmbeddings).
 *
 * Every function is pinned by the CPU tests in tests/test_oracle_pins.py.
 *
 * Build: gcc -O2 -std=c11 -fopenmp -ffp-contract=off -shared -fPIC
 * (no contraction: each fp32 operation rounds exactly once).
 *
 * ORACLE_MUTANT (compile-time, tests only): plants one known mistake so the
 * tests can show that the pins catch it. 0 (default) is the oracle proper.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

typedef struct {
    int32_t T, H, E, k, inter, group, bits;
    float eps;
} oracle_dims;

/* One 4-bit QuantizedLinear [N, K]: packed codes [N, K/8] (low nibble
 * first), group scales and biases [N, K/g] as bf16 bits. */
typedef struct {
    const uint32_t* w;
    const uint16_t* s;
    const uint16_t* b;
} oracle_qlinear;

/* ---------------------------------------------------------------- bf16 --- */

/* bf16 bits -> float: exact widening (bf16 is the top half of an fp32). */
static float bf(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* float -> bf16 bits, round to nearest, ties to even. */
static uint16_t bf16_from_float(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))
        return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN */
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* double -> bf16 bits with ONE rounding (nearest, ties to even).
 * bf16 keeps 8 significant bits; normal exponents down to 2^-126 and
 * subnormals on the fixed grid 2^-133. */
static uint16_t bf16_from_double(double d) {
    if (isnan(d)) return 0x7FC0u;
    uint16_t sign = signbit(d) ? 0x8000u : 0u;
    double a = fabs(d);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                 /* a = m * 2^e, m in [0.5, 1) */
    int q = e - 8;                /* weight of the last kept bit */
    if (q < -133) q = -133;
    double r = nearbyint(ldexp(a, -q)); /* default mode: nearest-even */
    double v = ldexp(r, q);
    if (v >= 0x1p128) return (uint16_t)(sign | 0x7F80u); /* overflow -> inf */
    float f = (float)v;           /* exact: v has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(sign | (u >> 16));
}

/* Exported so the tests can pin the rounding helpers themselves. */
uint16_t oracle_bf16_from_float(float f) { return bf16_from_float(f); }
uint16_t oracle_bf16_from_double(double d) { return bf16_from_double(d); }

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------- router --- */

/*
 * DiffRouter.forward: x [T,H] -> indices [T,k], weights [T,k].
 *   normed = rms_norm(x, no weight, eps)        (fp32 inside, bf16 out)
 *   normed = normed * scale                      (bf16 op)
 *   normed = normed * hidden^-0.5                (bf16 op; scalar in bf16)
 *   scores = proj(normed)                        (bf16 out)
 *   indices = top-k of scores (argpartition, unordered on the page;
 *             emitted here as value descending, ties to the lower expert id)
 *   weights = softmax_precise(scores[indices]) * per_expert_scale[indices]
 *
 * Optional taps (NULL to skip): normed [T,H] bf16 after both scale ops,
 * logits_exact [T,E] double (before rounding), scores [T,E] bf16.
 * Returns 0, or -1 on bad sizes.
 */
int oracle_route(const oracle_dims* d, const uint16_t* x, const uint16_t* router_w,
                 const uint16_t* router_scale, const uint16_t* per_expert_scale,
                 int32_t* idx_out, uint16_t* w_out, uint16_t* normed_tap,
                 double* logits_exact_tap, uint16_t* scores_tap, int nthreads) {
    const int T = d->T, H = d->H, E = d->E, k = d->k;
    if (T < 0 || H <= 0 || E <= 0 || k <= 0 || k > E || k > 64) return -1;
    set_threads(nthreads);
    /* hidden^-0.5 enters as a scalar in the array dtype (bf16). */
#if ORACLE_MUTANT == 16
    const float root = (float)pow((double)H, -0.5); /* planted: the scalar kept in fp32 */
#else
    const float root = bf(bf16_from_double(pow((double)H, -0.5)));
#endif

#pragma omp parallel
    {
        uint16_t* n3 = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)H);
        double* lex = (double*)malloc(sizeof(double) * (size_t)E);
        uint16_t* s = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)E);
        int* taken = (int*)malloc(sizeof(int) * (size_t)E);
#pragma omp for schedule(static)
        for (int t = 0; t < T; ++t) {
            const uint16_t* xt = x + (size_t)t * H;
            /* RMSNormNoScale in fp32: mean of squares, + eps, rsqrt. The fp32
             * mean is the exact mean rounded once to fp32 (the squares of bf16
             * values and their sum are exact in double for these sizes). */
            double ss = 0.0;
            for (int h = 0; h < H; ++h) {
                double v = bf(xt[h]);
                ss += v * v;
            }
#if ORACLE_MUTANT == 1
            float mean = (float)(ss / (double)(H - 1)); /* planted: wrong divisor */
#else
            float mean = (float)(ss / (double)H);
#endif
            float denom = mean + d->eps;
            float r = (float)(1.0 / sqrt((double)denom)); /* rsqrt, rounded to fp32 */
            for (int h = 0; h < H; ++h) {
#if ORACLE_MUTANT == 17
                float nv = bf(xt[h]) * r;                                   /* planted: not cast to bf16 */
#else
                float nv = bf(bf16_from_float(bf(xt[h]) * r));             /* cast to bf16 */
#endif
                float n2 = bf(bf16_from_float(nv * bf(router_scale[h])));  /* * scale */
                n3[h] = bf16_from_float(n2 * root);                         /* * H^-0.5 */
            }
            if (normed_tap) memcpy(normed_tap + (size_t)t * H, n3, sizeof(uint16_t) * H);
            /* Projection to E logits (dense bf16 weight [E,H], out = n W^T). */
            for (int e = 0; e < E; ++e) {
                const uint16_t* we = router_w + (size_t)e * H;
                double acc = 0.0;
                for (int h = 0; h < H; ++h) acc += (double)bf(n3[h]) * (double)bf(we[h]);
                lex[e] = acc;
                s[e] = bf16_from_double(acc);
            }
            if (logits_exact_tap) memcpy(logits_exact_tap + (size_t)t * E, lex, sizeof(double) * E);
            if (scores_tap) memcpy(scores_tap + (size_t)t * E, s, sizeof(uint16_t) * E);
            /* Top-k: k passes of "largest remaining score, lowest id on ties". */
            for (int e = 0; e < E; ++e) taken[e] = 0;
            int32_t* it = idx_out + (size_t)t * k;
            for (int j = 0; j < k; ++j) {
                int best = -1;
                for (int e = 0; e < E; ++e) {
                    if (taken[e]) continue;
#if ORACLE_MUTANT == 2
                    if (best < 0 || bf(s[e]) >= bf(s[best])) best = e; /* planted: ties to higher id */
#else
                    if (best < 0 || bf(s[e]) > bf(s[best])) best = e;
#endif
                }
                taken[best] = 1;
                it[j] = best;
            }
            /* Precise softmax over the k gathered scores, fp32. */
            float mx = bf(s[it[0]]);
            for (int j = 1; j < k; ++j)
                if (bf(s[it[j]]) > mx) mx = bf(s[it[j]]);
            float ex[64];
            float sum = 0.0f;
            for (int j = 0; j < k; ++j) {
                ex[j] = (float)exp((double)(bf(s[it[j]]) - mx)); /* exp rounded to fp32 */
                sum += ex[j];
            }
            uint16_t* wt = w_out + (size_t)t * k;
            for (int j = 0; j < k; ++j) {
                float p = bf(bf16_from_float(ex[j] / sum)); /* softmax output, bf16 */
#if ORACLE_MUTANT == 3
                wt[j] = bf16_from_float(p * bf(per_expert_scale[j])); /* planted: wrong gather */
#else
                wt[j] = bf16_from_float(p * bf(per_expert_scale[it[j]])); /* * pes[idx] */
#endif
            }
        }
        free(n3);
        free(lex);
        free(s);
        free(taken);
    }
    return 0;
}

/* ----------------------------------------------------------- dispatch --- */

/*
 * The sorted path of DiffExperts.forward: order = argsort(idx.flat),
 * invOrder = argsort(order), rowIdx = order // k. Read as a stable sort of
 * the flat slots f = t*k + j by expert id (counting sort), so the result is
 * unique: perm[p] = f (p-th slot in expert order), inv[f] = p, and
 * offsets[e]..offsets[e+1] is expert e's slot range.
 * Returns 0, or -1 on an expert id out of range.
 */
int oracle_dispatch(int32_t T, int32_t k, int32_t E, const int32_t* idx, int32_t* perm,
                    int32_t* offsets, int32_t* inv) {
    const int64_t S = (int64_t)T * k;
    for (int e = 0; e <= E; ++e) offsets[e] = 0;
    for (int64_t f = 0; f < S; ++f) {
        if (idx[f] < 0 || idx[f] >= E) return -1;
        offsets[idx[f] + 1] += 1;
    }
    for (int e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
    int32_t* next = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    for (int e = 0; e < E; ++e) next[e] = offsets[e];
#if ORACLE_MUTANT == 4
    for (int64_t f = S - 1; f >= 0; --f) { /* planted: unstable (reverse) order */
#else
    for (int64_t f = 0; f < S; ++f) {
#endif
        int32_t p = next[idx[f]]++;
        perm[p] = (int32_t)f;
        inv[f] = p;
    }
    free(next);
    return 0;
}

/* ------------------------------------------------------------ experts --- */

/* Dequantise one expert's N x K block of a 4-bit affine weight:
 * q = nibble (K mod 8) of word [n, K/8] (low nibble first),
 * w = bf16(S[n, K/g] * q + B[n, K/g]) with one rounding. */
static void dequant_expert(const uint32_t* w, const uint16_t* sc, const uint16_t* bi, int N, int K,
                           int g, float* out) {
    for (int n = 0; n < N; ++n) {
        for (int kk = 0; kk < K; ++kk) {
            uint32_t word = w[(size_t)n * (K / 8) + kk / 8];
#if ORACLE_MUTANT == 5
            int q = (int)((word >> (4 * (7 - kk % 8))) & 0xFu); /* planted: high nibble first */
#else
            int q = (int)((word >> (4 * (kk % 8))) & 0xFu);
#endif
            double S = bf(sc[(size_t)n * (K / g) + kk / g]);
            double B = bf(bi[(size_t)n * (K / g) + kk / g]);
            out[(size_t)n * K + kk] = bf(bf16_from_double(S * q + B));
        }
    }
}

/* The router with the pages' 4-bit group-64 projection (DiffRouter.proj is a
 * QuantizedLinear): the weight [E, H] dequantises like the experts' weights,
 * w = bf16(S * q + B), and the router is then the dense one on that weight. */
int oracle_route_q4(const oracle_dims* d, const uint16_t* x, const uint32_t* rq_w, const uint16_t* rq_s,
                    const uint16_t* rq_b, const uint16_t* router_scale, const uint16_t* per_expert_scale,
                    int32_t* idx_out, uint16_t* w_out, double* logits_exact_tap, uint16_t* scores_tap,
                    int nthreads) {
    const int E = d->E, H = d->H, g = d->group;
    if (E <= 0 || H <= 0 || g <= 0 || H % g || H % 8) return -1;
    float* wf = (float*)malloc(sizeof(float) * (size_t)E * H);
    uint16_t* wb = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)E * H);
#if ORACLE_MUTANT == 10
    uint16_t* zb = (uint16_t*)calloc((size_t)E * (H / g), sizeof(uint16_t)); /* planted: biases dropped */
    dequant_expert(rq_w, rq_s, zb, E, H, g, wf);
    free(zb);
#else
    dequant_expert(rq_w, rq_s, rq_b, E, H, g, wf);
#endif
    for (size_t i = 0; i < (size_t)E * H; ++i) wb[i] = bf16_from_float(wf[i]); /* exact: already bf16 */
    int rc = oracle_route(d, x, wb, router_scale, per_expert_scale, idx_out, w_out, NULL, logits_exact_tap,
                          scores_tap, nthreads);
    free(wf);
    free(wb);
    return rc;
}

/* bf16(gelu_approx(g) * up), one rounding, where
 *   gelu_approx(g) = 0.5 g (1 + tanh(s)),  s = sqrt(2/pi) (g + 0.044715 g^3)
 * (the tanh approximation of GELU). 0.5 (1 + tanh(s)) equals the logistic
 * function of 2s; evaluated that way it keeps its relative accuracy where
 * 1 + tanh(s) cancels (s << 0). For s >= 0 the exact product lies strictly
 * between 0 and g*up (the logistic is < 1); where double cannot tell the
 * logistic from 1 (s > ~18.7) the product is moved one double ulp toward
 * zero, which rounds an exact bf16 tie of g*up the way the exact value does
 * and changes no other result. */
static uint16_t geglu_bf16(double g, double up) {
    const double c = sqrt(2.0 / 3.14159265358979323846);
    const double s = c * (g + 0.044715 * g * g * g);
    const double p = g * up; /* exact: a product of two bf16 values */
    double v;
    if (s < 0.0) {
        const double e = exp(2.0 * s);
        v = p * (e / (1.0 + e));
    } else {
        v = p / (1.0 + exp(-2.0 * s));
        if (v == p && p != 0.0) v = nextafter(p, 0.0);
    }
    return bf16_from_double(v);
}

/*
 * DiffExperts.forward: x [T,H], indices [T,k], weights [T,k] -> [T,H].
 * For every slot f = t*k + j with expert e = idx[f]:
 *   z = bf16(x[t] . W_gu[e]^T)           gate_up SwitchLinear, [2I]
 *   gate = z[0:I], up = z[I:2I]          split at moe_intermediate
 *   m = bf16(gelu_approx(gate) * up)     compiled geglu: one rounding
 *   y = bf16(m . W_dn[e]^T)              down SwitchLinear, [H]
 * and out[t] = bf16( sum_j bf16(y_{t,j} * w[t,j]) )   (mul, then sum over k).
 * The sorted/unsorted choice on the page changes no value, so the oracle
 * has one path. Optional taps (NULL to skip), per flat slot f:
 * z_tap [T*k, 2I], m_tap [T*k, I], y_tap [T*k, H].
 * Returns 0, or -1 on bad sizes / ids.
 */
int oracle_experts(const oracle_dims* d, const uint16_t* x, const int32_t* idx, const uint16_t* w,
                   const uint32_t* gu_w, const uint16_t* gu_s, const uint16_t* gu_b,
                   const uint32_t* dn_w, const uint16_t* dn_s, const uint16_t* dn_b, uint16_t* out,
                   uint16_t* z_tap, uint16_t* m_tap, uint16_t* y_tap, int nthreads) {
    const int T = d->T, H = d->H, E = d->E, k = d->k, I = d->inter, g = d->group;
    if (T < 0 || H <= 0 || E <= 0 || k <= 0 || I <= 0 || g <= 0) return -1;
    if (H % 8 || I % 8 || H % g || I % g || d->bits != 4) return -1;
    const int64_t S = (int64_t)T * k;
    for (int64_t f = 0; f < S; ++f)
        if (idx[f] < 0 || idx[f] >= E) return -1;
    set_threads(nthreads);
    uint16_t* y_all = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(S > 0 ? S : 1) * H);
    const size_t gu_words = (size_t)2 * I * (H / 8), gu_groups = (size_t)2 * I * (H / g);
    const size_t dn_words = (size_t)H * (I / 8), dn_groups = (size_t)H * (I / g);

#pragma omp parallel
    {
        float* wgu = (float*)malloc(sizeof(float) * (size_t)2 * I * H);
        float* wdn = (float*)malloc(sizeof(float) * (size_t)H * I);
        uint16_t* z = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)2 * I);
        uint16_t* m = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)I);
#pragma omp for schedule(dynamic, 1)
        for (int e = 0; e < E; ++e) {
            int used = 0;
            for (int64_t f = 0; f < S && !used; ++f) used = (idx[f] == e);
            if (!used) continue; /* an expert with no slots reads no weights */
            dequant_expert(gu_w + e * gu_words, gu_s + e * gu_groups, gu_b + e * gu_groups, 2 * I, H,
                           g, wgu);
            dequant_expert(dn_w + e * dn_words, dn_s + e * dn_groups, dn_b + e * dn_groups, H, I, g,
                           wdn);
            for (int64_t f = 0; f < S; ++f) {
                if (idx[f] != e) continue;
                const uint16_t* xt = x + (size_t)(f / k) * H;
                for (int n = 0; n < 2 * I; ++n) {
                    const float* wr = wgu + (size_t)n * H;
                    double acc = 0.0;
                    for (int h = 0; h < H; ++h) acc += (double)bf(xt[h]) * (double)wr[h];
                    z[n] = bf16_from_double(acc);
                }
                for (int n = 0; n < I; ++n) {
#if ORACLE_MUTANT == 6
                    m[n] = geglu_bf16(bf(z[n + I]), bf(z[n])); /* planted: halves swapped */
#else
                    m[n] = geglu_bf16(bf(z[n]), bf(z[n + I]));
#endif
                }
                uint16_t* yf = y_all + (size_t)f * H;
                for (int h = 0; h < H; ++h) {
                    const float* wr = wdn + (size_t)h * I;
                    double acc = 0.0;
                    for (int n = 0; n < I; ++n) acc += (double)bf(m[n]) * (double)wr[n];
                    yf[h] = bf16_from_double(acc);
                }
                if (z_tap) memcpy(z_tap + (size_t)f * 2 * I, z, sizeof(uint16_t) * 2 * I);
                if (m_tap) memcpy(m_tap + (size_t)f * I, m, sizeof(uint16_t) * I);
                if (y_tap) memcpy(y_tap + (size_t)f * H, yf, sizeof(uint16_t) * H);
            }
        }
        free(wgu);
        free(wdn);
        free(z);
        free(m);
    }

    /* (y * weights[..., None]).sum(-2): product in bf16, sum over k. */
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        for (int h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) {
                int64_t f = (int64_t)t * k + j;
#if ORACLE_MUTANT == 7
                acc += bf(y_all[(size_t)f * H + h]) * bf(w[f]) ; /* planted: product not rounded */
#else
                acc += bf(bf16_from_float(bf(y_all[(size_t)f * H + h]) * bf(w[f])));
#endif
            }
            out[(size_t)t * H + h] = bf16_from_double(acc);
        }
    }
    free(y_all);
    return 0;
}

/* RMSNorm with a weight: the decoder layer's plain nn.RMSNorm (the weight is
 * used as it is, no 1 + weight offset; "diffusion-gemma/model.ts", header
 * notes and DiffusionGemmaDecoderLayer), in fp32 like the router's norm:
 * r = rsqrt(mean(x^2) + eps) with the fp32 mean the exact mean rounded once,
 * then bf16((x * r) * w), each fp32 product rounded, one bf16 rounding.
 * weight NULL: RMSNormNoScale (an RMSNorm built with a null weight, as
 * SelfConditioning's post norm), bf16(x * r). */
int oracle_rms_norm(int32_t T, int32_t H, float eps, const uint16_t* x, const uint16_t* weight,
                    uint16_t* out) {
    if (T < 0 || H <= 0) return -1;
    for (int t = 0; t < T; ++t) {
        const uint16_t* xt = x + (size_t)t * H;
        double ss = 0.0;
        for (int h = 0; h < H; ++h) {
            double v = bf(xt[h]);
            ss += v * v;
        }
        float mean = (float)(ss / (double)H);
        float r = (float)(1.0 / sqrt((double)(mean + eps)));
        for (int h = 0; h < H; ++h) {
#if ORACLE_MUTANT == 18
            float nv = bf(bf16_from_float(bf(xt[h]) * r)); /* planted: x*r rounded before the weight */
#else
            float nv = bf(xt[h]) * r;
#endif
#if ORACLE_MUTANT == 8
            out[(size_t)t * H + h] = bf16_from_float(nv); /* planted: weight dropped */
#else
            out[(size_t)t * H + h] = weight ? bf16_from_float(nv * bf(weight[h])) : bf16_from_float(nv);
#endif
        }
    }
    return 0;
}

/* The MoE branch of a decoder layer (DiffusionGemmaDecoderLayer.forwardWith):
 * the router reads the residual, the experts read preFfNorm2(residual), and
 * the experts' combined output goes through postFfNorm2. */
int oracle_moe_branch(const oracle_dims* d, const uint16_t* residual, const uint16_t* router_w,
                      const uint16_t* router_scale, const uint16_t* per_expert_scale,
                      const uint16_t* pre_norm_w, const uint16_t* post_norm_w, const uint32_t* gu_w,
                      const uint16_t* gu_s, const uint16_t* gu_b, const uint32_t* dn_w, const uint16_t* dn_s,
                      const uint16_t* dn_b, uint16_t* out, int32_t* idx_out, uint16_t* w_out,
                      uint16_t* expert_in_tap, int nthreads) {
    const size_t n = (size_t)d->T * d->H;
    uint16_t* xe = (uint16_t*)malloc(sizeof(uint16_t) * (n ? n : 1));
    uint16_t* ye = (uint16_t*)malloc(sizeof(uint16_t) * (n ? n : 1));
#if ORACLE_MUTANT == 9
    /* planted: the router reads the expert input instead of the residual */
    int rc = oracle_rms_norm(d->T, d->H, d->eps, residual, pre_norm_w, xe);
    if (!rc)
        rc = oracle_route(d, xe, router_w, router_scale, per_expert_scale, idx_out, w_out, NULL, NULL, NULL,
                          nthreads);
#else
    int rc = oracle_route(d, residual, router_w, router_scale, per_expert_scale, idx_out, w_out, NULL, NULL,
                          NULL, nthreads);
    if (!rc) rc = oracle_rms_norm(d->T, d->H, d->eps, residual, pre_norm_w, xe);
#endif
    if (!rc && expert_in_tap) memcpy(expert_in_tap, xe, sizeof(uint16_t) * n);
    if (!rc)
        rc = oracle_experts(d, xe, idx_out, w_out, gu_w, gu_s, gu_b, dn_w, dn_s, dn_b, ye, NULL, NULL, NULL,
                            nthreads);
    if (!rc) rc = oracle_rms_norm(d->T, d->H, d->eps, ye, post_norm_w, out);
    free(xe);
    free(ye);
    return rc;
}

/* ---------------------------------------------------------- dense MLP --- */

/*
 * The dense 4-bit GeGLU MLP: x [T,H] -> [T,H] through three QuantizedLinears
 * (gate_proj and up_proj [I,H], down_proj [H,I], each a 4-bit group-g affine
 * weight) and the compiled geglu between them. SelfConditioning.forward
 * ("diffusion-gemma/model.ts") prints these steps; the decoder layer's
 * GegluMLP is imported from a file the pages do not print and is read as
 * the same three linears and geglu. Per token t:
 *   gate = bf16(x[t] . W_gate^T), up = bf16(x[t] . W_up^T)     [I] each
 *   m    = bf16(gelu_approx(gate) * up)                         one rounding
 *   out  = bf16(m . W_down^T)                                   [H]
 * Optional taps (NULL to skip): gate, up, m [T,I].
 * Returns 0, or -1 on bad sizes.
 */
int oracle_dense_mlp(int32_t T, int32_t H, int32_t I, int32_t g, const uint16_t* x, const oracle_qlinear* gate,
                     const oracle_qlinear* up, const oracle_qlinear* down, uint16_t* out, uint16_t* gate_tap,
                     uint16_t* up_tap, uint16_t* m_tap, int nthreads) {
    if (T < 0 || H <= 0 || I <= 0 || g <= 0 || H % 8 || I % 8 || H % g || I % g) return -1;
    set_threads(nthreads);
    float* wg = (float*)malloc(sizeof(float) * (size_t)I * H);
    float* wu = (float*)malloc(sizeof(float) * (size_t)I * H);
    float* wd = (float*)malloc(sizeof(float) * (size_t)H * I);
    dequant_expert(gate->w, gate->s, gate->b, I, H, g, wg);
    dequant_expert(up->w, up->s, up->b, I, H, g, wu);
    dequant_expert(down->w, down->s, down->b, H, I, g, wd);
#pragma omp parallel
    {
        uint16_t* gv = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)I);
        uint16_t* uv = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)I);
        uint16_t* m = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)I);
#pragma omp for schedule(dynamic, 1)
        for (int t = 0; t < T; ++t) {
            const uint16_t* xt = x + (size_t)t * H;
            for (int n = 0; n < I; ++n) {
                double ag = 0.0, au = 0.0;
                for (int h = 0; h < H; ++h) {
                    ag += (double)bf(xt[h]) * (double)wg[(size_t)n * H + h];
                    au += (double)bf(xt[h]) * (double)wu[(size_t)n * H + h];
                }
                gv[n] = bf16_from_double(ag);
                uv[n] = bf16_from_double(au);
            }
            for (int n = 0; n < I; ++n) {
#if ORACLE_MUTANT == 11
                m[n] = geglu_bf16(bf(uv[n]), bf(gv[n])); /* planted: gate and up linears swapped */
#else
                m[n] = geglu_bf16(bf(gv[n]), bf(uv[n]));
#endif
            }
            for (int h = 0; h < H; ++h) {
                double acc = 0.0;
                for (int n = 0; n < I; ++n) acc += (double)bf(m[n]) * (double)wd[(size_t)h * I + n];
                out[(size_t)t * H + h] = bf16_from_double(acc);
            }
            if (gate_tap) memcpy(gate_tap + (size_t)t * I, gv, sizeof(uint16_t) * I);
            if (up_tap) memcpy(up_tap + (size_t)t * I, uv, sizeof(uint16_t) * I);
            if (m_tap) memcpy(m_tap + (size_t)t * I, m, sizeof(uint16_t) * I);
        }
        free(gv);
        free(uv);
        free(m);
    }
    free(wg);
    free(wu);
    free(wd);
    return 0;
}

/* The decoder layer's dense branch (DiffusionGemmaDecoderLayer.forwardWith):
 * postFfNorm1(mlp(preFfNorm(h))), the two norms plain RMSNorms with their
 * weights (pre_feedforward_layernorm, post_feedforward_layernorm_1). */
int oracle_dense_branch(int32_t T, int32_t H, int32_t I, int32_t g, float eps, const uint16_t* h,
                        const uint16_t* pre_norm_w, const uint16_t* post_norm_w, const oracle_qlinear* gate,
                        const oracle_qlinear* up, const oracle_qlinear* down, uint16_t* out, int nthreads) {
    const size_t n = (size_t)T * (H > 0 ? H : 0);
    uint16_t* xn = (uint16_t*)malloc(sizeof(uint16_t) * (n ? n : 1));
    uint16_t* y = (uint16_t*)malloc(sizeof(uint16_t) * (n ? n : 1));
    int rc = oracle_rms_norm(T, H, eps, h, pre_norm_w, xn);
    if (!rc) rc = oracle_dense_mlp(T, H, I, g, xn, gate, up, down, y, NULL, NULL, NULL, nthreads);
#if ORACLE_MUTANT == 13
    if (!rc) rc = oracle_rms_norm(T, H, eps, y, pre_norm_w, out); /* planted: post norm takes the pre norm's weight */
#else
    if (!rc) rc = oracle_rms_norm(T, H, eps, y, post_norm_w, out);
#endif
    free(xn);
    free(y);
    return rc;
}

/* SelfConditioning.forward ("diffusion-gemma/model.ts"):
 *   s   = mlp(preNorm(signal))          preNorm: RMSNorm with its weight
 *   out = postNorm(bf16(embeds + s))    postNorm: RMSNormNoScale
 * The add is a bf16 op: the exact sum of two bf16 values rounded once. */
int oracle_self_conditioning(int32_t T, int32_t H, int32_t I, int32_t g, float eps, const uint16_t* embeds,
                             const uint16_t* signal, const uint16_t* pre_norm_w, const oracle_qlinear* gate,
                             const oracle_qlinear* up, const oracle_qlinear* down, uint16_t* out, int nthreads) {
    const size_t n = (size_t)T * (H > 0 ? H : 0);
    uint16_t* sn = (uint16_t*)malloc(sizeof(uint16_t) * (n ? n : 1));
    uint16_t* sv = (uint16_t*)malloc(sizeof(uint16_t) * (n ? n : 1));
    int rc = oracle_rms_norm(T, H, eps, signal, pre_norm_w, sn);
    if (!rc) rc = oracle_dense_mlp(T, H, I, g, sn, gate, up, down, sv, NULL, NULL, NULL, nthreads);
#if ORACLE_MUTANT == 12
    /* planted: the embeddings are added after the post norm */
    if (!rc) rc = oracle_rms_norm(T, H, eps, sv, NULL, sn);
    for (size_t i = 0; !rc && i < n; ++i) out[i] = bf16_from_double((double)bf(embeds[i]) + (double)bf(sn[i]));
#else
    for (size_t i = 0; !rc && i < n; ++i) sn[i] = bf16_from_double((double)bf(embeds[i]) + (double)bf(sv[i]));
    if (!rc) rc = oracle_rms_norm(T, H, eps, sn, NULL, out);
#endif
    free(sn);
    free(sv);
    return rc;
}

/* ------------------------------------------------------------ LM head --- */

/*
 * The tied 4-bit head with the final-logit softcap
 * (DiffusionGemmaModel.logitsFromHidden, "diffusion-gemma/model.ts"):
 *   logits = embed.asLinear(h)                bf16 [T, V]: h . W^T with the
 *                                             embedding table [V, H] as a
 *                                             4-bit group-g QuantizedLinear
 *   out    = softcap(float32(logits))         fp32 [T, V]
 * The softcap's formula is in a file the pages do not print; it is read as
 * the usual final-logit softcapping cap * tanh(x / cap), in fp32 steps (x /
 * cap rounded, tanh rounded once, the product rounded). cap <= 0: no cap.
 * The table is dequantised one vocabulary row at a time. Optional tap:
 * logits [T, V] bf16. Returns 0, or -1 on bad sizes.
 */
int oracle_lm_head(int32_t T, int32_t H, int32_t V, int32_t g, float cap, const uint16_t* h,
                   const oracle_qlinear* embed, float* out, uint16_t* logits_tap, int nthreads) {
    if (T < 0 || H <= 0 || V <= 0 || g <= 0 || H % 8 || H % g) return -1;
    set_threads(nthreads);
#pragma omp parallel
    {
        float* wr = (float*)malloc(sizeof(float) * (size_t)H);
#pragma omp for schedule(dynamic, 64)
        for (int v = 0; v < V; ++v) {
            dequant_expert(embed->w + (size_t)v * (H / 8), embed->s + (size_t)v * (H / g),
                           embed->b + (size_t)v * (H / g), 1, H, g, wr);
            for (int t = 0; t < T; ++t) {
                const uint16_t* ht = h + (size_t)t * H;
                double acc = 0.0;
                for (int k = 0; k < H; ++k) acc += (double)bf(ht[k]) * (double)wr[k];
                const uint16_t lb = bf16_from_double(acc);
                if (logits_tap) logits_tap[(size_t)t * V + v] = lb;
#if ORACLE_MUTANT == 15
                const float x = (float)acc; /* planted: the logit is not rounded to bf16 */
#else
                const float x = bf(lb);
#endif
                float o = x;
                if (cap > 0.0f) {
#if ORACLE_MUTANT == 14
                    o = (float)tanh((double)x) * cap; /* planted: tanh(x) * cap */
#else
                    const float q = x / cap;
                    o = (float)tanh((double)q) * cap;
#endif
                }
                out[(size_t)t * V + v] = o;
            }
        }
        free(wr);
    }
    return 0;
}

/* Router then experts on the same x: the layer as one call. */
int oracle_forward(const oracle_dims* d, const uint16_t* x, const uint16_t* router_w,
                   const uint16_t* router_scale, const uint16_t* per_expert_scale,
                   const uint32_t* gu_w, const uint16_t* gu_s, const uint16_t* gu_b,
                   const uint32_t* dn_w, const uint16_t* dn_s, const uint16_t* dn_b, uint16_t* out,
                   int32_t* idx_out, uint16_t* w_out, int nthreads) {
    int rc = oracle_route(d, x, router_w, router_scale, per_expert_scale, idx_out, w_out, NULL, NULL,
                          NULL, nthreads);
    if (rc) return rc;
    return oracle_experts(d, x, idx_out, w_out, gu_w, gu_s, gu_b, dn_w, dn_s, dn_b, out, NULL, NULL,
                          NULL, nthreads);
}

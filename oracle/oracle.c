/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, scalar FP64 evaluation of one decode step of a sigmoid-top-k
 * Mixture-of-Experts layer whose experts are stored as NVFP4 weights and run
 * weight-only (W4A16: BF16 activations, 4-bit weights).  Only tests, the smoke
 * check and the CPU-baseline leg of the benchmark may load this library; the
 * product path never does.  It shares no code, header, table or constant with
 * the CUDA kernels: every decoder below is written from the number formats'
 * definitions.
 *
 * Sources (pages are cited by title and section):
 *  [FLINT]  "vLLM Day-0 support for Recursive's Flint" --
 *           section "Flint model overview" (NVFP4 checkpoint run weight-only,
 *           W4A16, BF16 activations), section "Flint model architecture"
 *           (MoE bullet: 256 experts, sigmoid top-6 selection plus one shared
 *           expert), section "Optimisation strategy" (small-batch MoE kernels
 *           read only the selected experts' weights; the low-latency path folds
 *           routing and the expert combine into the neighbouring GEMVs).
 *  [INK2]   "Inkling 2 Small on vLLM: Day-0 Support" -- paragraph "Mixed-
 *           precision MoE and Four-Over-Six NVFP4" (16-element blocks, block
 *           maximum mapped to 6 or 4), section "vLLM integration and
 *           optimisation" (SwiGLU between gate/up and down), section "Accuracy
 *           evaluation" (the router runs in FP32; only reduction order may
 *           differ from the reference numerics).
 *  [ML4]    "Day 0 support for Mistral Large 4 on vLLM" -- "Highlights" and the
 *           "Model architecture" table (128 routed experts, top-4, one shared
 *           expert), section "Breakable CUDA graphs and fusions" (FP32 routing
 *           GEMM), section "Specialized decode" (its fused decode layer runs a
 *           softmax top-4 router).
 *
 * Readings where the pages are silent (the full list is kept in the design
 * notes of the repository):
 *  - NVFP4 = E2M1 codes, one E4M3 (fn variant) scale per 16 consecutive
 *    elements along K, one FP32 tensor scale per (expert, matrix).
 *  - Packing: K-major rows, element 2j in the low nibble of byte j, 2j+1 in the
 *    high nibble.  Gate/up are one [2I, H] matrix: rows < I gate, rows >= I up.
 *  - Dequantised weight = e2m1 * e4m3 * gs.  The first product is exact and the
 *    whole product needs at most 30 significant bits, so it is exact in FP64;
 *    the forward pass uses this exact value.  orc_dequant() returns it rounded
 *    once to FP32 (round to nearest even).
 *  - Router: logits in FP64 (the exact value of the FP32 router), score =
 *    sigmoid(logit).  Sigmoid is strictly increasing, so the top-k by score is
 *    the top-k by logit; the DECISION is taken on the FP32-rounded logit (the
 *    router's precision), descending, lowest expert index first on ties
 *    (equal FP32 logits).  The weights use the FP64 scores, normalised to sum
 *    to 1 when asked, then multiplied by the routed scale.
 *  - Softmax routing (score_func = 1, [ML4] specialized decode): score =
 *    exp(z_e - z_max) / sum over all experts of exp(z - z_max), in FP64.  It
 *    increases with the logit too, so the top-k decision is the same as with
 *    sigmoid; the weights are the chosen experts' softmax scores, normalised
 *    over the chosen ones when asked (then exp(z_j - z_max) / sum over the
 *    chosen of exp(z_i - z_max)), times the routed scale.
 *  - Router bias, when present, is added to the logit (plain linear layer).
 *  - Shared experts: ungated, weight 1, by default in the same NVFP4 format.
 *  - Other expert formats (the routed experts and the shared ones each have
 *    one; element k of a row is the k-th along K, as above):
 *      MXFP4  ([ML4] "MXFP4 experts at load, one layer at a time": E2M1 values
 *             with one E8M0 scale per 32 values): W = e2m1 * 2^(s - 127), no
 *             tensor scale; E8M0 code 255 is NaN.
 *      FP8 block-scaled ([ML4] "Highlights": the NVFP4 checkpoint keeps its
 *             shared experts in FP8 with block-scaled weights; the block is
 *             not given, and the reading here is 128 x 128): E4M3 (fn) codes,
 *             one byte per element, and one FP32 scale per 128 x 128 block of
 *             the stored [rows, cols] matrix, row-major over the blocks
 *             ([ceil(rows/128), ceil(cols/128)]): W = e4m3 * scale.
 *      MXFP8  ([INK2] "Mixed-precision MoE and Four-Over-Six NVFP4": the last
 *             8 layers' experts are MXFP8): E4M3 (fn) codes with one E8M0
 *             scale per 32 values along K: W = e4m3 * 2^(s - 127).
 *    Every product is exact in FP64 (at most 4 + 24 significant bits).
 *  - W4A4 (activations quantised to NVFP4 with "Four Over Six" block scales,
 *    [INK2] "Mixed-precision MoE and Four-Over-Six NVFP4": a per-token global
 *    scale plus, for each 16-element block, the block maximum scaled to 6 and
 *    to 4, keeping whichever reconstructs the block with the lower mean
 *    absolute error; [INK2] "MoE with fused activation quantisation": the
 *    tokens are quantised before gate/up and the SwiGLU output before down).
 *    Reading of the steps the page leaves open, all in FP32 (the precision
 *    the quantiser's decisions are taken in):
 *      a  = max |v| over the row (v: the BF16 row, exact in FP32);
 *      gs = a / 1792 (1792 = 4 * 448, so that the "4" candidate's largest
 *           block scale is E4M3's largest value); gs = 1 for an all-zero row;
 *      for each block b (16 consecutive elements) and c in {6, 4}:
 *        s_c = e4m3(m_b / (c * gs))      m_b = max |v| in the block; E4M3
 *                                        round to nearest even, saturating
 *        q_k = e2m1(v_k / (s_c * gs))    E2M1 round to nearest even (on a tie
 *                                        the code with mantissa bit 0),
 *                                        saturating at 6; all zero if s_c = 0
 *        r_k = e2m1(q_k) * s_c * gs      err_c = sum over k = 0..15 of
 *                                        |v_k - r_k|, summed in that order
 *      the block keeps c = 4 if err_4 < err_6, else c = 6 (ties go to 6, the
 *      plain NVFP4 choice).  The dequantised activation is e2m1 * e4m3 * gs,
 *      exact in FP64.  The router still reads the unquantised x; h is the
 *      BF16 SwiGLU output as in W4A16, quantised per (token, expert) row.
 *  - SwiGLU: h = silu(gate) * up, silu(z) = z / (1 + exp(-z)); h is rounded to
 *    BF16 (round to nearest even) before the down projection.
 *  - Output: sum of routing-weighted routed outputs plus the shared outputs,
 *    accumulated in FP64, rounded once to BF16.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared -fopenmp oracle.c -o liboracle.so -lm
 * (no fused multiply-adds: the quantiser's FP32 steps are each rounded)
 */
#include <math.h>
#include <stdint.h>

/* Test hook: a nonzero ORC_PLANT compiles exactly one deliberate mistake into
 * a separate library, so that a test can show that the pins catch it:
 *   1 softmax scores replaced by sigmoid, 2 normalisation ignored,
 *   3 gate and up rows swapped, 4 shared experts dropped from the combine,
 *   5 E2M1 subnormal (code 1) decoded as 1.0 instead of 0.5,
 *   6 MX scales taken per 16 elements instead of per 32,
 *   7 FP8 block scales indexed with rows and columns swapped,
 *   8 Four-Over-Six keeping the candidate with the larger error,
 *   9 Four-Over-Six ties going to 4.
 * The regular build plants nothing. */
#ifndef ORC_PLANT
#define ORC_PLANT 0
#endif
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* Number formats, written from their definitions.                           */
/* ------------------------------------------------------------------------- */

/* E2M1 (FP4): bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
 * Exponent 0 is subnormal: value = m * 0.5.  Otherwise (1 + m/2) * 2^(e-1).
 * The magnitudes are {0, 0.5, 1, 1.5, 2, 3, 4, 6}; 6 is the largest, matching
 * the "scale the block maximum to 6" rule of [INK2] and 4 is representable. */
double orc_e2m1(int code)
{
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = (e == 0) ? (ORC_PLANT == 5 ? 1.0 : 0.5) * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* E4M3, "fn" variant (finite, no infinities): bit 7 sign, bits 6..3 exponent
 * (bias 7), bits 2..0 mantissa.  Exponent 0 is subnormal: (m/8) * 2^-6.
 * Exponent 15 with mantissa 7 is NaN (0x7F, 0xFF); everything else is finite,
 * the largest magnitude being 1.75 * 2^8 = 448. */
double orc_e4m3(int code)
{
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) mag = ldexp(m / 8.0, -6);
    else mag = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* BF16 bits -> value (exact: a BF16 is the top half of an IEEE binary32). */
double orc_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Round a double to the nearest BF16 value (8 significant bits, exponent range
 * of binary32, gradual underflow), ties to even, overflow to infinity.  Direct
 * single rounding from FP64. */
double orc_bf16_round(double v)
{
    if (isnan(v) || isinf(v) || v == 0.0) return v;
    double a = fabs(v);
    int e;
    frexp(a, &e);             /* a in [2^(e-1), 2^e) */
    int lead = e - 1;
    if (lead < -126) lead = -126;           /* subnormal range: fixed quantum */
    double quantum = ldexp(1.0, lead - 7);  /* 8 significant bits */
    double n = a / quantum;                 /* exact: power-of-two scaling */
    double r = nearbyint(n);                /* default mode: ties to even */
    double res = r * quantum;
    if (res >= 0x1p128) res = INFINITY;     /* beyond the largest BF16 */
    return copysign(res, v);
}

uint16_t orc_double_to_bf16(double v)
{
    double r = orc_bf16_round(v);
    float f = (float)r;       /* exact: r is a BF16 value (or inf/nan) */
    uint32_t u;
    memcpy(&u, &f, 4);
    if (isnan(v)) return (uint16_t)0x7FC0u;
    return (uint16_t)(u >> 16);
}

/* E8M0 (the MX block scale): an unsigned biased exponent, value 2^(c - 127);
 * code 255 is NaN.  No sign, no mantissa. */
double orc_e8m0(int code)
{
    if ((code & 255) == 255) return NAN;
    return ldexp(1.0, (code & 255) - 127);
}

/* Expert weight formats. */
enum { ORC_NVFP4 = 0, ORC_MXFP4 = 1, ORC_FP8_BLOCK = 2, ORC_MXFP8 = 3 };

/* Bytes of the codes and of the scales of one [rows, cols] matrix. */
size_t orc_codes_bytes(int fmt, int rows, int cols)
{
    return (fmt == ORC_NVFP4 || fmt == ORC_MXFP4) ? (size_t)rows * (cols / 2) : (size_t)rows * cols;
}
size_t orc_scale_bytes(int fmt, int rows, int cols)
{
    switch (fmt) {
    case ORC_NVFP4: return (size_t)rows * (cols / 16);
    case ORC_FP8_BLOCK: return (size_t)((rows + 127) / 128) * ((cols + 127) / 128) * sizeof(float);
    default: return (size_t)rows * (cols / 32);
    }
}

/* Code nibble of element k in a K-major packed row (element 2j low nibble). */
static inline int nib(const uint8_t *row, int k)
{
    uint8_t b = row[k >> 1];
    return (k & 1) ? (b >> 4) : (b & 15);
}

/* Value tables filled from the closed forms above (speed only: the forward
 * pass decodes ~10^9 elements for the largest layer). */
static double tab_e2m1[16], tab_e4m3[256];
static void fill_tables(void)
{
    static int done = 0;
    if (done) return;
    for (int c = 0; c < 16; ++c) tab_e2m1[c] = orc_e2m1(c);
    for (int c = 0; c < 256; ++c) tab_e4m3[c] = orc_e4m3(c);
    done = 1;
}

/* Exact dequantised weight W[r][k] = e2m1 * e4m3 * gs (FP64, exact). */
static inline double wexact(const uint8_t *codes, const uint8_t *sf, double gs,
                            int cols, int r, int k)
{
    const uint8_t *row = codes + (size_t)r * (cols / 2);
    int sc = sf[(size_t)r * (cols / 16) + k / 16];
    return tab_e2m1[nib(row, k)] * tab_e4m3[sc] * gs;
}

/* The same in any expert format (gs is used by NVFP4 only). */
static inline double wexact_fmt(int fmt, const uint8_t *codes, const uint8_t *sf, double gs,
                                int cols, int r, int k)
{
    const int mxb = ORC_PLANT == 6 ? 16 : 32;   /* elements per MX scale */
    switch (fmt) {
    case ORC_MXFP4:
        return tab_e2m1[nib(codes + (size_t)r * (cols / 2), k)] *
               orc_e8m0(sf[(size_t)r * (cols / 32) + k / mxb]);
    case ORC_FP8_BLOCK: {
        const float *bs = (const float *)sf;
        const int nbc = (cols + 127) / 128;
        const size_t bi = ORC_PLANT == 7 ? (size_t)(k / 128) * nbc + r / 128 : (size_t)(r / 128) * nbc + k / 128;
        return tab_e4m3[codes[(size_t)r * cols + k]] * (double)bs[bi];
    }
    case ORC_MXFP8:
        return tab_e4m3[codes[(size_t)r * cols + k]] * orc_e8m0(sf[(size_t)r * (cols / 32) + k / mxb]);
    default:
        return wexact(codes, sf, gs, cols, r, k);
    }
}

/* Dequantise a [rows, cols] NVFP4 matrix to FP32: one rounding of the exact
 * product e2m1 * e4m3 * gs. */
void orc_dequant(const uint8_t *codes, const uint8_t *sf, float gs,
                 int rows, int cols, float *out)
{
    fill_tables();
    for (int r = 0; r < rows; ++r)
        for (int k = 0; k < cols; ++k)
            out[(size_t)r * cols + k] = (float)wexact(codes, sf, (double)gs, cols, r, k);
}

/* ------------------------------------------------------------------------- */
/* Four-Over-Six NVFP4 activation quantisation (FP32 decisions).             */
/* ------------------------------------------------------------------------- */

/* Round a non-negative FP32 value to the nearest E4M3 (fn) value, ties to
 * even (mantissa bit 0), saturating at 448; returns the code. */
int orc_e4m3_from_f32(float v)
{
    if (!(v > 0.0f)) return 0;                    /* zero (and NaN, not used) */
    if (v >= 448.0f) return 0x7E;
    int best = 0;
    double bd = 1e300;
    for (int c = 0; c <= 0x7E; ++c) {             /* every finite non-negative code */
        double d = fabs(orc_e4m3(c) - (double)v);
        /* nearest; on an exact tie the even code (codes ascend with the value,
         * so the two candidates are adjacent and differ in mantissa bit 0) */
        if (d < bd || (d == bd && (c & 1) == 0)) { bd = d; best = c; }
    }
    return best;
}

/* Round a FP32 value to the nearest E2M1 value, ties to even (mantissa bit
 * 0), saturating at +-6; returns the 4-bit code. */
int orc_e2m1_from_f32(float v)
{
    double a = fabs((double)v);
    int best = 0;
    double bd = 1e300;
    for (int c = 0; c < 8; ++c) {
        double d = fabs(orc_e2m1(c) - a);
        if (d < bd || (d == bd && (c & 1) == 0)) { bd = d; best = c; }
    }
    if (a > 6.0) best = 7;
    return (v < 0.0f && best != 0) ? (best | 8) : best;
}

/* Quantise one row of n BF16 values (n % 16 == 0): codes (one nibble per
 * byte, value = code), block scale codes [n/16] and choices [n/16] (4 or 6),
 * the global scale returned; deq[n] (optional) the dequantised values. */
float orc_quant_fos(const uint16_t *row, int n, uint8_t *codes, uint8_t *sf, uint8_t *choice, double *deq)
{
    float a = 0.0f;
    for (int k = 0; k < n; ++k) {
        float v = (float)orc_bf16_to_double(row[k]);
        a = fabsf(v) > a ? fabsf(v) : a;
    }
    const float gs = a > 0.0f ? a / 1792.0f : 1.0f;
    for (int b = 0; b < n / 16; ++b) {
        float v[16], m = 0.0f;
        for (int k = 0; k < 16; ++k) {
            v[k] = (float)orc_bf16_to_double(row[16 * b + k]);
            m = fabsf(v[k]) > m ? fabsf(v[k]) : m;
        }
        int sc_c[2], q_c[2][16];
        float err[2];
        const float cand[2] = {6.0f, 4.0f};
        for (int i = 0; i < 2; ++i) {
            const float cg = cand[i] * gs;
            sc_c[i] = orc_e4m3_from_f32(m / cg);
            const float s = (float)orc_e4m3(sc_c[i]);
            const float d = s * gs;
            float e = 0.0f;
            for (int k = 0; k < 16; ++k) {
                q_c[i][k] = s > 0.0f ? orc_e2m1_from_f32(v[k] / d) : 0;
                const float r = (float)orc_e2m1(q_c[i][k]) * s * gs;
                e += fabsf(v[k] - r);
            }
            err[i] = e;
        }
        int pick = (err[1] < err[0]) ? 1 : 0;                 /* ties: 6 */
        if (ORC_PLANT == 8) pick = (err[1] > err[0]) ? 1 : 0;
        if (ORC_PLANT == 9) pick = (err[1] <= err[0]) ? 1 : 0;
        sf[b] = (uint8_t)sc_c[pick];
        if (choice) choice[b] = (uint8_t)(pick ? 4 : 6);
        for (int k = 0; k < 16; ++k) {
            codes[16 * b + k] = (uint8_t)q_c[pick][k];
            if (deq) deq[16 * b + k] = orc_e2m1(q_c[pick][k]) * orc_e4m3(sc_c[pick]) * (double)gs;
        }
    }
    return gs;
}

/* Dequantise a [rows, cols] matrix of any expert format to FP32: one
 * rounding of the exact value (gs: NVFP4 only). */
void orc_dequant_fmt(int fmt, const uint8_t *codes, const uint8_t *sf, float gs,
                     int rows, int cols, float *out)
{
    fill_tables();
    for (int r = 0; r < rows; ++r)
        for (int k = 0; k < cols; ++k)
            out[(size_t)r * cols + k] = (float)wexact_fmt(fmt, codes, sf, (double)gs, cols, r, k);
}

/* ------------------------------------------------------------------------- */
/* The layer.                                                                 */
/* ------------------------------------------------------------------------- */

typedef struct {
    int H, E, k, I, S, Is;      /* hidden, routed experts, top-k, expert inter, shared count, shared inter */
    int normalize;              /* 1: routing weights normalised to sum to 1 */
    double routed_scale;        /* multiplies the routed weights (1.0) */
    const float *router_w;      /* [E, H] */
    const float *router_b;      /* [E] or NULL */
    const uint8_t *w13;         /* [E, 2I, H/2]  rows < I gate, rows >= I up */
    const uint8_t *w13_sf;      /* [E, 2I, H/16] */
    const float *w13_gs;        /* [E, 2] (gate, up) */
    const uint8_t *w2;          /* [E, H, I/2] */
    const uint8_t *w2_sf;       /* [E, H, I/16] */
    const float *w2_gs;         /* [E] */
    const uint8_t *sw13;        /* [S, 2Is, H/2] */
    const uint8_t *sw13_sf;     /* [S, 2Is, H/16] */
    const float *sw13_gs;       /* [S, 2] */
    const uint8_t *sw2;         /* [S, H, Is/2] */
    const uint8_t *sw2_sf;      /* [S, H, Is/16] */
    const float *sw2_gs;        /* [S] */
    int score_func;             /* 0: sigmoid per expert; 1: softmax over all experts */
    int efmt, sfmt;             /* weight format of the routed / shared experts (ORC_*) */
    int w4a4;                   /* 1: activations quantised with Four-Over-Six NVFP4 */
} orc_layer;

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* Router logits and scores for one token ([FLINT] architecture: sigmoid
 * scoring; [ML4] specialized decode: softmax scoring; [INK2] accuracy section
 * and [ML4] fusions: FP32 router, whose exact value this is). */
static void token_scores(const orc_layer *L, const uint16_t *xt, double *z, double *s)
{
    for (int e = 0; e < L->E; ++e) {
        double acc = 0.0;
        const float *wr = L->router_w + (size_t)e * L->H;
        for (int h = 0; h < L->H; ++h) acc += orc_bf16_to_double(xt[h]) * (double)wr[h];
        if (L->router_b) acc += (double)L->router_b[e];
        z[e] = acc;
        s[e] = sigmoid(acc);
    }
    if (L->score_func == 1 && ORC_PLANT != 1) {
        double zmax = z[0], den = 0.0;
        for (int e = 1; e < L->E; ++e) zmax = z[e] > zmax ? z[e] : zmax;
        for (int e = 0; e < L->E; ++e) den += exp(z[e] - zmax);
        for (int e = 0; e < L->E; ++e) s[e] = exp(z[e] - zmax) / den;
    }
}

/* Top-k: descending FP32-rounded logit (the order of the scores), lowest
 * index first on ties.  ids[j] in selection order; w[j] from the FP64 scores. */
static void token_topk(const orc_layer *L, const double *z, const double *s, int *ids, double *w)
{
    int E = L->E, K = L->k;
    char *taken = (char *)calloc((size_t)E, 1);
    for (int j = 0; j < K; ++j) {
        int best = -1;
        float bz = 0.0f;
        for (int e = 0; e < E; ++e) {
            if (taken[e]) continue;
            float ze = (float)z[e];
            if (best < 0 || ze > bz) { best = e; bz = ze; }   /* strict: ties keep lower e */
        }
        taken[best] = 1;
        ids[j] = best;
    }
    double sum = 0.0;
    for (int j = 0; j < K; ++j) sum += s[ids[j]];
    for (int j = 0; j < K; ++j) {
        double wj = (L->normalize && ORC_PLANT != 2) ? s[ids[j]] / sum : s[ids[j]];
        w[j] = wj * L->routed_scale;
    }
    free(taken);
}

/* Routing for T tokens: ids [T,k], w [T,k], optionally scores [T,E] (FP64
 * sigmoid) and logits [T,E]. */
int orc_route(const orc_layer *L, const uint16_t *x, int T, int *ids, double *w,
              double *scores, double *logits)
{
    double *z = (double *)malloc(sizeof(double) * L->E);
    double *s = (double *)malloc(sizeof(double) * L->E);
    if (!z || !s) { free(z); free(s); return -1; }
    for (int t = 0; t < T; ++t) {
        token_scores(L, x + (size_t)t * L->H, z, s);
        token_topk(L, z, s, ids + (size_t)t * L->k, w + (size_t)t * L->k);
        if (scores) memcpy(scores + (size_t)t * L->E, s, sizeof(double) * L->E);
        if (logits) memcpy(logits + (size_t)t * L->E, z, sizeof(double) * L->E);
    }
    free(z);
    free(s);
    return 0;
}

/* One expert MLP on one token ([INK2] integration section: SwiGLU between the
 * gate/up and the down projection):
 *   g_n = sum_k x_k Wg[n,k],  u_n = sum_k x_k Wu[n,k]
 *   h_n = bf16(silu(g_n) * u_n)
 *   y_m = sum_n h_n Wd[m,n]
 * All weights are the exact dequantised values. */
/* The W4A4 activation: the Four-Over-Six dequantised values of a row of
 * doubles that are BF16 values (x rows, h rows). */
static void quant_row(const double *v, int n, double *out)
{
    uint16_t *b = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)n);
    uint8_t *codes = (uint8_t *)malloc((size_t)n), *sf = (uint8_t *)malloc((size_t)n / 16 + 1);
    for (int k = 0; k < n; ++k) b[k] = orc_double_to_bf16(v[k]);
    orc_quant_fos(b, n, codes, sf, NULL, out);
    free(b); free(codes); free(sf);
}

static void expert_mlp(int fmt, int H, int I,
                       const uint8_t *w13, const uint8_t *w13_sf, const float *w13_gs,
                       const uint8_t *w2, const uint8_t *w2_sf, const float *w2_gs,
                       const double *x, double *h, double *y, int w4a4)
{
    double *xq = NULL;
    if (w4a4) {
        xq = (double *)malloc(sizeof(double) * (size_t)H);
        quant_row(x, H, xq);
        x = xq;
    }
    /* tensor scales: NVFP4 only */
    const int nv = fmt == ORC_NVFP4;
    double gsg = nv ? (double)w13_gs[0] : 1.0, gsu = nv ? (double)w13_gs[1] : 1.0;
    double gsd = nv ? (double)w2_gs[0] : 1.0;
    for (int n = 0; n < I; ++n) {
        double g = 0.0, u = 0.0;
        const int rg = ORC_PLANT == 3 ? I + n : n, ru = ORC_PLANT == 3 ? n : I + n;
        if (nv) {   /* the same values; the NVFP4 loop without the format switch runs faster */
            for (int k = 0; k < H; ++k) {
                g += x[k] * wexact(w13, w13_sf, gsg, H, rg, k);
                u += x[k] * wexact(w13, w13_sf, gsu, H, ru, k);
            }
        } else {
            for (int k = 0; k < H; ++k) {
                g += x[k] * wexact_fmt(fmt, w13, w13_sf, gsg, H, rg, k);
                u += x[k] * wexact_fmt(fmt, w13, w13_sf, gsu, H, ru, k);
            }
        }
        double silu = g * sigmoid(g);
        h[n] = orc_bf16_round(silu * u);
    }
    if (w4a4) {
        quant_row(h, I, h);
        free(xq);
    }
    for (int m = 0; m < H; ++m) {
        double acc = 0.0;
        if (nv)
            for (int n = 0; n < I; ++n) acc += h[n] * wexact(w2, w2_sf, gsd, I, m, n);
        else
            for (int n = 0; n < I; ++n) acc += h[n] * wexact_fmt(fmt, w2, w2_sf, gsd, I, m, n);
        y[m] = acc;
    }
}

/* Full decode step for T tokens.
 *  out      [T,H] BF16 bits (required)
 *  out_pre  [T,H] FP64 value before the final BF16 rounding (or NULL)
 *  ids, w   [T,k] routing result (or NULL)
 *  nthreads OpenMP threads for the per-(token, expert) work; the reduction is
 *           in a fixed order, so the result does not depend on it.
 * Per token: logits, sigmoid, top-k, normalise ([FLINT] architecture), the
 * selected experts only ([FLINT] optimisation strategy) plus the shared
 * experts, then the routing-weighted combine. */
int orc_forward(const orc_layer *L, const uint16_t *x, int T, uint16_t *out,
                double *out_pre, int *ids_out, double *w_out, int nthreads)
{
    int H = L->H, K = L->k, S = L->S, P = K + S;
    fill_tables();
    int Imax = L->I > L->Is ? L->I : L->Is;
    int *ids = (int *)malloc(sizeof(int) * (size_t)T * K);
    double *w = (double *)malloc(sizeof(double) * (size_t)T * K);
    double *y = (double *)malloc(sizeof(double) * (size_t)T * P * H);
    double *xd = (double *)malloc(sizeof(double) * (size_t)T * H);
    if (!ids || !w || !y || !xd) { free(ids); free(w); free(y); free(xd); return -1; }
    if (orc_route(L, x, T, ids, w, NULL, NULL) != 0) { free(ids); free(w); free(y); free(xd); return -1; }
    for (size_t i = 0; i < (size_t)T * H; ++i) xd[i] = orc_bf16_to_double(x[i]);

    int npairs = T * P;
    int nt = nthreads > 0 ? nthreads : 1;
    (void)nt;
#ifdef _OPENMP
    #pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
#endif
    for (int pi = 0; pi < npairs; ++pi) {
        int t = pi / P, j = pi % P;
        double *h = (double *)malloc(sizeof(double) * (size_t)Imax);
        double *yp = y + (size_t)pi * H;
        const double *xt = xd + (size_t)t * H;
        if (j < K) {
            int e = ids[(size_t)t * K + j];
            int I = L->I, f = L->efmt;
            int nv = f == ORC_NVFP4;
            expert_mlp(f, H, I,
                       L->w13 + (size_t)e * orc_codes_bytes(f, 2 * I, H),
                       L->w13_sf + (size_t)e * orc_scale_bytes(f, 2 * I, H),
                       nv ? L->w13_gs + 2 * (size_t)e : NULL,
                       L->w2 + (size_t)e * orc_codes_bytes(f, H, I),
                       L->w2_sf + (size_t)e * orc_scale_bytes(f, H, I),
                       nv ? L->w2_gs + e : NULL, xt, h, yp, L->w4a4);
        } else {
            int sidx = j - K, I = L->Is, f = L->sfmt;
            int nv = f == ORC_NVFP4;
            expert_mlp(f, H, I,
                       L->sw13 + (size_t)sidx * orc_codes_bytes(f, 2 * I, H),
                       L->sw13_sf + (size_t)sidx * orc_scale_bytes(f, 2 * I, H),
                       nv ? L->sw13_gs + 2 * (size_t)sidx : NULL,
                       L->sw2 + (size_t)sidx * orc_codes_bytes(f, H, I),
                       L->sw2_sf + (size_t)sidx * orc_scale_bytes(f, H, I),
                       nv ? L->sw2_gs + sidx : NULL, xt, h, yp, L->w4a4);
        }
        free(h);
    }

    /* Combine, fixed order: routed experts in selection order, then shared. */
    for (int t = 0; t < T; ++t) {
        for (int m = 0; m < H; ++m) {
            double acc = 0.0;
            for (int j = 0; j < K; ++j)
                acc += w[(size_t)t * K + j] * y[((size_t)t * P + j) * H + m];
            for (int sidx = 0; sidx < (ORC_PLANT == 4 ? 0 : S); ++sidx)
                acc += y[((size_t)t * P + K + sidx) * H + m];
            if (out_pre) out_pre[(size_t)t * H + m] = acc;
            out[(size_t)t * H + m] = orc_double_to_bf16(acc);
        }
    }
    if (ids_out) memcpy(ids_out, ids, sizeof(int) * (size_t)T * K);
    if (w_out) memcpy(w_out, w, sizeof(double) * (size_t)T * K);
    free(ids); free(w); free(y); free(xd);
    return 0;
}

/* Threads the OpenMP runtime would use (1 without OpenMP). */
int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * CPU oracle for the routed MoE expert layer (routing tables, forward,
 * backward).  TEST INFRASTRUCTURE ONLY: it is compiled and called by the
 * tests, by the package's smoke check and by the benchmark's CPU-baseline
 * leg, never by the product path.  It shares no code, header or constant
 * with the CUDA library; the two are written independently from the same
 * definitions.
 *
 * Sources of each definition:
 *  - routing tables: Primus-Turbo "Mega MoE" README, "Implementation Map"
 *    (a dispatch prologue builds routing tables from topk_idx) and the
 *    DeepGEMM Mega-MoE article, "Block-M Alignment for Irregular Token
 *    Counts" (per-expert token counts are padded to the GEMM block M).
 *  - forward / backward: the Mega MoE README, "Pipeline" (dispatch, L1
 *    grouped GEMM, SwiGLU, L2 grouped GEMM, top-k weighted combine, and the
 *    conjugate backward).
 *
 * Two instantiations of the numerical body:
 *   *_b16 : x, W1, W2, dY given as bfloat16 bit patterns (widened exactly),
 *           routing weights FP32, all arithmetic FP32.  This is the oracle
 *           the GPU results are compared with.
 *   *_f64 : every input and all arithmetic in FP64 (used for finite
 *           differences and the oracle's own pins).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------- FP8 activations */

/*
 * Per-token FP8 quantization of the layer input with power-of-two block
 * scales (DeepGEMM Mega-MoE article, usage example: the activations are cast
 * per token to FP8 with UE8M0 scale factors at a granularity of 32 elements
 * along the hidden dimension before dispatch).  For token t and group g
 * (elements 32g .. 32g+31 of the row):
 *   amax = max |x|;  e = the smallest integer with 448 * 2^e >= amax
 *   (e = 0 when amax = 0; e clamped to [-127, 127]);  sf[t, g] = e + 127
 *   (UE8M0: the byte is the biased exponent of the scale 2^e);
 *   q[t, i] = E4M3(x[t, i] / 2^e), round to nearest, ties to even, finite
 *   values saturating at +-448.
 * E4M3 (OCP FP8): sign bit, 4 exponent bits (bias 7), 3 mantissa bits; field
 * f > 0: (1 + m/8) 2^(f-7); f = 0: (m/8) 2^-6; f = 15, m = 7 is NaN, so the
 * largest finite value is 1.75 * 2^8 = 448.  The dequantized value is
 * decode(q) * 2^(sf - 127).  Plain loops; x is given as bfloat16 bits.
 */
double oracle_e4m3_decode(uint8_t c) {
    const int s = c >> 7, f = (c >> 3) & 15, m = c & 7;
    double v;
    if (f == 15 && m == 7) return NAN;
    if (f == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, f - 7);
    return s ? -v : v;
}

uint8_t oracle_e4m3_encode(double v) {
    if (isnan(v)) return 0x7F;
    const uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (a >= 448.0) return sign | 0x7E; /* 448 = f 15, m 6 */
    /* spacing of the representable values around a */
    double step;
    if (a < ldexp(1.0, -6)) {
        step = ldexp(1.0, -9);
    } else {
        int ex;
        frexp(a, &ex); /* a = r 2^ex, r in [0.5, 1): floor(log2 a) = ex - 1 */
        step = ldexp(1.0, ex - 1 - 3);
    }
    const double n = a / step;           /* exact: a has few bits, step a power of two */
    double r = floor(n);
    const double frac = n - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0; /* nearest, ties to even */
    const double q = r * step;
    if (q == 0.0) return sign;
    if (q < ldexp(1.0, -6)) return sign | (uint8_t)(q / ldexp(1.0, -9)); /* subnormal, f = 0 */
    int ex;
    const double fr = frexp(q, &ex); /* q = fr 2^ex: exponent field ex - 1 + 7 */
    const int f = ex - 1 + 7;
    const int m = (int)(fr * 16.0) - 8; /* (1 + m/8) = 2 fr */
    return sign | (uint8_t)(f << 3) | (uint8_t)m;
}

static int fp8_group_exponent(double amax) {
    if (amax == 0.0) return 0;
    /* smallest e with 448 * 2^e >= amax, where 448 * 2^e = 0.875 * 2^(e + 9) */
    int p;
    const double r = frexp(amax, &p); /* amax = r 2^p, r in [0.5, 1) */
    int e = r <= 0.875 ? p - 9 : p - 8;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

void oracle_quantize_fp8(int T, int H, int gran, const uint16_t* x, uint8_t* q, uint8_t* sf) {
    const int G = H / gran;
    for (int t = 0; t < T; ++t) {
        for (int g = 0; g < G; ++g) {
            double amax = 0.0;
            for (int i = 0; i < gran; ++i) {
                uint32_t b = (uint32_t)x[(size_t)t * H + (size_t)g * gran + i] << 16;
                float v;
                memcpy(&v, &b, 4);
                if (fabs((double)v) > amax) amax = fabs((double)v);
            }
            const int e = fp8_group_exponent(amax);
            sf[(size_t)t * G + g] = (uint8_t)(e + 127);
            for (int i = 0; i < gran; ++i) {
                uint32_t b = (uint32_t)x[(size_t)t * H + (size_t)g * gran + i] << 16;
                float v;
                memcpy(&v, &b, 4);
                q[(size_t)t * H + (size_t)g * gran + i] = oracle_e4m3_encode(ldexp((double)v, -e));
            }
        }
    }
}

/*
 * The same quantization of float64 values instead of bfloat16 bit patterns:
 * used for the activations between the two GEMMs of the FP8 forward (below),
 * which are computed, not stored as bf16.  One group of `gran` values.
 */
static void fp8_quantize_group_f64(const double* v, int gran, uint8_t* q, uint8_t* sf) {
    double amax = 0.0;
    for (int i = 0; i < gran; ++i)
        if (fabs(v[i]) > amax) amax = fabs(v[i]);
    const int e = fp8_group_exponent(amax);
    *sf = (uint8_t)(e + 127);
    for (int i = 0; i < gran; ++i) q[i] = oracle_e4m3_encode(ldexp(v[i], -e));
}

void oracle_quantize_fp8_f64(int T, int H, int gran, const double* x, uint8_t* q, uint8_t* sf) {
    const int G = H / gran;
    for (int t = 0; t < T; ++t)
        for (int g = 0; g < G; ++g)
            fp8_quantize_group_f64(x + (size_t)t * H + (size_t)g * gran, gran, q + (size_t)t * H + (size_t)g * gran,
                                   sf + (size_t)t * G + g);
}

/*
 * FP8 forward (DeepGEMM Mega-MoE article, "Code Example: Fused Overlap
 * Path": the layer runs on FP8 activations and transformed low-precision
 * weights).  The operands x, W1, W2 are given as the float64 values they
 * stand for (the dequantized E4M3 inputs and weights).  For each token t and
 * slot j with expert e, in float64:
 *   hg, hu, a = silu(hg) * hu                    as in the forward below;
 *   a is quantized like a token of the input: groups of 32 consecutive i,
 *     scale 2^e with the smallest e such that 448 * 2^e >= max|group|,
 *     aq[i] = E4M3(a[i] / 2^e), asf[g] = e + 127;
 *   o[c] = sum_i decode(aq[i]) 2^(asf[i / 32] - 127) W2[e, i, c];
 *   y[t, c] += w[t, j] o[c].
 * aq_out [n_tok][k][I] and asf_out [n_tok][k][I / 32] receive each slot's
 * quantized activations (zeros for a slot without a valid expert).  No
 * activation clamp.
 */
void oracle_forward_fp8(int T, int H, int I, int E, int k, const double* x, const double* W1, const double* W2,
                        const int32_t* topk_idx, const float* topk_w, int n_tok, const int32_t* tok_list,
                        double* y_out, uint8_t* aq_out, uint8_t* asf_out) {
    (void)T;
    const int G = I / 32;
#ifdef _OPENMP
#pragma omp parallel
#endif
    {
        double* hg = (double*)malloc(sizeof(double) * (size_t)I);
        double* hu = (double*)malloc(sizeof(double) * (size_t)I);
        double* a = (double*)malloc(sizeof(double) * (size_t)I);
        double* o = (double*)malloc(sizeof(double) * (size_t)H);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int n = 0; n < n_tok; ++n) {
            const int t = tok_list[n];
            double* y = y_out + (size_t)n * H;
            for (int c = 0; c < H; ++c) y[c] = 0.0;
            for (int j = 0; j < k; ++j) {
                uint8_t* aq = aq_out + ((size_t)n * k + j) * I;
                uint8_t* asf = asf_out + ((size_t)n * k + j) * G;
                memset(aq, 0, (size_t)I);
                memset(asf, 0, (size_t)G);
                const int e = topk_idx[(size_t)t * k + j];
                if (e < 0 || e >= E) continue;
                for (int i = 0; i < I; ++i) { hg[i] = 0.0; hu[i] = 0.0; }
                for (int h = 0; h < H; ++h) {
                    const double xv = x[(size_t)t * H + h];
                    const double* row = W1 + ((size_t)e * H + h) * (size_t)(2 * I);
                    for (int i = 0; i < I; ++i) {
                        hg[i] += xv * row[i];
                        hu[i] += xv * row[I + i];
                    }
                }
                for (int i = 0; i < I; ++i) a[i] = hg[i] / (1.0 + exp(-hg[i])) * hu[i];
                for (int g = 0; g < G; ++g) fp8_quantize_group_f64(a + 32 * g, 32, aq + 32 * g, asf + g);
                for (int c = 0; c < H; ++c) o[c] = 0.0;
                for (int i = 0; i < I; ++i) {
                    const double ai = oracle_e4m3_decode(aq[i]) * ldexp(1.0, (int)asf[i / 32] - 127);
                    const double* row = W2 + ((size_t)e * I + i) * (size_t)H;
                    for (int c = 0; c < H; ++c) o[c] += ai * row[c];
                }
                const double wv = (double)topk_w[(size_t)t * k + j];
                for (int c = 0; c < H; ++c) y[c] += wv * o[c];
            }
        }
        free(hg);
        free(hu);
        free(a);
        free(o);
    }
}

/* ----------------------------------------------------------------- router */

/*
 * Top-k gating from router logits (the step in front of the layer: the
 * Primus-Turbo "Mega MoE" README takes topk_idx / topk_weights from the
 * router, "Key points"; the ROCm Primus MoE guide's router produces them
 * from logits).  For each token t, over its E logits:
 *   key(v) = v, except that a NaN counts as -infinity;
 *   topk_idx[t, 0..k-1] = the k experts with the largest keys, in
 *     decreasing key order, equal keys in increasing expert id;
 *   topk_w[t, j] = exp(key_j - m) / sum_i exp(key_i - m) over the k selected
 *     keys, m = the largest selected key, computed in FP64 and rounded to
 *     FP32 (softmax over the selected logits).  When m is infinite the
 *     weights are the limit: 1/n on the n selected keys equal to m, 0 on the
 *     others.
 * Selection is done by k passes over the row, each taking the best key not
 * yet taken (plain loops, no sort).
 */
static double router_key(float v) { return isnan(v) ? -INFINITY : (double)v; }

void oracle_router_topk(int T, int E, int k, const float* logits, int32_t* topk_idx, float* topk_w) {
    char* taken = (char*)malloc((size_t)(E > 0 ? E : 1));
    double* key = (double*)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
    for (int t = 0; t < T; ++t) {
        const float* row = logits + (size_t)t * E;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || router_key(row[e]) > router_key(row[best])) best = e;
            }
            taken[best] = 1;
            topk_idx[(size_t)t * k + j] = best;
            key[j] = router_key(row[best]);
        }
        double m = key[0];
        if (isinf(m)) {
            int n = 0;
            for (int j = 0; j < k; ++j) n += key[j] == m;
            for (int j = 0; j < k; ++j) topk_w[(size_t)t * k + j] = key[j] == m ? (float)(1.0 / n) : 0.0f;
        } else {
            double sum = 0;
            for (int j = 0; j < k; ++j) sum += exp(key[j] - m);
            for (int j = 0; j < k; ++j) topk_w[(size_t)t * k + j] = (float)(exp(key[j] - m) / sum);
        }
    }
    free(taken);
    free(key);
}

/* ---------------------------------------------------------------- routing */

/* Row capacity of the block-M padded layout: the padded row count
 *   Mpad = sum_e ceil(c_e / bm) * bm
 * never exceeds T*k + min(E, T*k) * (bm - 1), and is a multiple of bm, so it
 * never exceeds that bound rounded down to a multiple of bm. */
int64_t oracle_rows_cap(int T, int E, int k, int bm) {
    int64_t tk = (int64_t)T * k;
    int64_t ne = tk < E ? tk : E;
    int64_t bound = tk + ne * (bm - 1);
    return (bound / bm) * bm;
}

/*
 * Routing tables for slots s = t*k + j (topk_idx is [T, k], row-major):
 *   counts[e]  number of slots with topk_idx[s] == e
 *   offs[e]    exclusive prefix sum of ceil(counts[e]/bm)*bm ; offs[E] = Mpad
 *   perm[r]    slot held by padded row r, -1 for padding rows and for every
 *              row r >= Mpad (array length = oracle_rows_cap)
 *              rows of expert e hold its slots in increasing s
 *   inv[s]     padded row of slot s, -1 when the slot is dropped
 *   tiles[m]   expert owning rows [m*bm, (m+1)*bm), -1 for m >= Mpad/bm
 *              (array length = oracle_rows_cap / bm)
 *   scal[0] = Mpad, scal[1] = Mpad / bm, scal[2] = number of slots whose id
 *   is neither -1 nor in [0, E) (they are dropped like -1).
 */
void oracle_route(int T, int E, int k, int bm, const int32_t* topk_idx,
                  int32_t* counts, int32_t* offs, int32_t* perm, int32_t* inv,
                  int32_t* tiles, int32_t* scal) {
    int64_t tk = (int64_t)T * k;
    int64_t cap = oracle_rows_cap(T, E, k, bm);
    int32_t n_invalid = 0;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t s = 0; s < tk; ++s) {
        int32_t e = topk_idx[s];
        if (e >= 0 && e < E) counts[e] += 1;
        else if (e != -1) n_invalid += 1;
    }
    offs[0] = 0;
    for (int e = 0; e < E; ++e) {
        int32_t padded = ((counts[e] + bm - 1) / bm) * bm;
        offs[e + 1] = offs[e] + padded;
    }
    int32_t mpad = offs[E];
    for (int64_t r = 0; r < cap; ++r) perm[r] = -1;
    for (int64_t s = 0; s < tk; ++s) inv[s] = -1;
    /* next free row of each expert; visiting slots in increasing s gives
     * the stable order within an expert */
    int32_t* next = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    for (int e = 0; e < E; ++e) next[e] = offs[e];
    for (int64_t s = 0; s < tk; ++s) {
        int32_t e = topk_idx[s];
        if (e < 0 || e >= E) continue;
        int32_t r = next[e]++;
        perm[r] = (int32_t)s;
        inv[s] = r;
    }
    free(next);
    int64_t ntiles_cap = cap / bm;
    for (int64_t m = 0; m < ntiles_cap; ++m) tiles[m] = -1;
    for (int e = 0; e < E; ++e)
        for (int32_t m = offs[e] / bm; m < offs[e + 1] / bm; ++m) tiles[m] = e;
    scal[0] = mpad;
    scal[1] = mpad / bm;
    scal[2] = n_invalid;
}

/* ---------------------------------------------- numerical instantiations */

static inline float bf16_widen(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

#define SUF b16
#define IN_T uint16_t
#define W_T float
#define REAL float
#define LD(p, i) bf16_widen((p)[(i)])
#include "moe_oracle_body.h"
#undef SUF
#undef IN_T
#undef W_T
#undef REAL
#undef LD

#define SUF f64
#define IN_T double
#define W_T double
#define REAL double
#define LD(p, i) ((p)[(i)])
#include "moe_oracle_body.h"
#undef SUF
#undef IN_T
#undef W_T
#undef REAL
#undef LD

/* Threads the OpenMP runtime will use (reported next to CPU timings). */
#ifdef _OPENMP
#include <omp.h>
int oracle_num_threads(void) { return omp_get_max_threads(); }
#else
int oracle_num_threads(void) { return 1; }
#endif

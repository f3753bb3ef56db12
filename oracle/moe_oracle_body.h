/*
 * Body of the CPU oracle for the routed MoE expert layer.  TEST INFRASTRUCTURE
 * ONLY: nothing on the product path includes, links or calls this file.
 *
 * This header is included twice by moe_oracle.c with different macro settings:
 *   SUF   function-name suffix
 *   IN_T  element type of x, W1, W2, dY as handed in
 *   LD(p, i)  widens element i of an IN_T array to REAL
 *   W_T   element type of the routing weights
 *   REAL  arithmetic type of every sum and product
 *
 * What is computed (Primus-Turbo "Mega MoE" README, section "Pipeline"; the
 * layer takes external routing, section "Key points"):
 *   for each token t and each of its k routing slots j with expert e:
 *     hg[i] = sum_h x[t,h] W1[e,h,i]          (gate half, columns [0, I))
 *     hu[i] = sum_h x[t,h] W1[e,h,I+i]        (up half,   columns [I, 2I))
 *     a[i]  = silu(hg[i]) * hu[i],  silu(z) = z / (1 + exp(-z))     (SwiGLU)
 *     o[c]  = sum_i a[i] W2[e,i,c]
 *     y[t,c] += w[t,j] * o[c]                 (top-k weighted sum, the combine)
 * and the plain chain rule of that for the backward pass (same page, the
 * backward paragraph under "Pipeline").  A slot whose expert id is outside
 * [0, E) (including -1) contributes nothing.
 *
 * Loops are per token and per slot, in plain order, with no blocking or
 * reordering beyond the sums as written above.
 */

#define CAT2(a, b) a##b
#define CAT(a, b) CAT2(a, b)
#define FN(name) CAT(name, SUF)

static REAL FN(sigmoid_)(REAL z) { return (REAL)1 / ((REAL)1 + (REAL)exp(-(double)z)); }

/* Activation clamp (reading of the DeepGEMM Mega-MoE article's
 * `activation_clamp` argument, given there without a formula): with c > 0
 * both SwiGLU inputs are clamped to [-c, c] before a = silu(gate) * up, and
 * the gradient passes where -c <= z <= c and is 0 outside; c <= 0 is no
 * clamp. */
static REAL FN(clamp_)(REAL z, double c) {
    if (c <= 0) return z;
    return z < (REAL)-c ? (REAL)-c : (z > (REAL)c ? (REAL)c : z);
}
static REAL FN(clamp_pass_)(REAL z, double c) { return (c <= 0 || (z >= (REAL)-c && z <= (REAL)c)) ? (REAL)1 : (REAL)0; }

/* Forward of one slot: fills hg, hu, a (length I) and o (length H) for token
 * row xt routed to the expert whose weights start at W1e / W2e. */
static void FN(slot_forward_)(int H, int I, const IN_T* x, size_t xoff,
                              const IN_T* W1, size_t w1off, const IN_T* W2, size_t w2off, double clamp,
                              REAL* hg, REAL* hu, REAL* a, REAL* o) {
    for (int i = 0; i < I; ++i) { hg[i] = 0; hu[i] = 0; }
    for (int h = 0; h < H; ++h) {
        REAL xv = LD(x, xoff + (size_t)h);
        size_t row = w1off + (size_t)h * (size_t)(2 * I);
        for (int i = 0; i < I; ++i) {
            hg[i] += xv * LD(W1, row + (size_t)i);
            hu[i] += xv * LD(W1, row + (size_t)I + (size_t)i);
        }
    }
    for (int i = 0; i < I; ++i) {
        REAL g = FN(clamp_)(hg[i], clamp), u = FN(clamp_)(hu[i], clamp);
        a[i] = g * FN(sigmoid_)(g) * u;
    }
    for (int c = 0; c < H; ++c) o[c] = 0;
    for (int i = 0; i < I; ++i) {
        REAL av = a[i];
        size_t row = w2off + (size_t)i * (size_t)H;
        for (int c = 0; c < H; ++c) o[c] += av * LD(W2, row + (size_t)c);
    }
}

/* Backward of one slot given the upstream gradient of the layer output for
 * this token (dYt) and the slot weight wv.  Fills da, dhg, dhu (length I).
 * Chain rule of the slot forward above:
 *   go[c]  = wv * dY[t,c]
 *   da[i]  = sum_c go[c] W2[e,i,c]
 *   dhg[i] = da[i] * hu[i] * s(hg[i]) * (1 + hg[i] (1 - s(hg[i])))   (d silu)
 *   dhu[i] = da[i] * silu(hg[i])                                                */
static void FN(slot_backward_)(int H, int I, const IN_T* dY, size_t dyoff, REAL wv,
                               const IN_T* W2, size_t w2off, double clamp,
                               const REAL* hg, const REAL* hu,
                               REAL* da, REAL* dhg, REAL* dhu) {
    for (int i = 0; i < I; ++i) {
        size_t row = w2off + (size_t)i * (size_t)H;
        REAL s = 0;
        for (int c = 0; c < H; ++c) s += wv * LD(dY, dyoff + (size_t)c) * LD(W2, row + (size_t)c);
        da[i] = s;
    }
    for (int i = 0; i < I; ++i) {
        REAL g = FN(clamp_)(hg[i], clamp), u = FN(clamp_)(hu[i], clamp);
        REAL sg = FN(sigmoid_)(g);
        dhg[i] = da[i] * u * sg * ((REAL)1 + g * ((REAL)1 - sg)) * FN(clamp_pass_)(hg[i], clamp);
        dhu[i] = da[i] * g * sg * FN(clamp_pass_)(hu[i], clamp);
    }
}

/* y rows for the listed tokens: y_out[n, :] is token tok_list[n]. */
void FN(oracle_forward_)(int T, int H, int I, int E, int k, double clamp,
                         const IN_T* x, const IN_T* W1, const IN_T* W2,
                         const int32_t* topk_idx, const W_T* topk_w,
                         int n_tok, const int32_t* tok_list, REAL* y_out) {
    (void)T;
#pragma omp parallel
    {
        REAL* hg = (REAL*)malloc(sizeof(REAL) * (size_t)I);
        REAL* hu = (REAL*)malloc(sizeof(REAL) * (size_t)I);
        REAL* a = (REAL*)malloc(sizeof(REAL) * (size_t)I);
        REAL* o = (REAL*)malloc(sizeof(REAL) * (size_t)H);
#pragma omp for schedule(dynamic, 1)
        for (int n = 0; n < n_tok; ++n) {
            int t = tok_list[n];
            REAL* y = y_out + (size_t)n * (size_t)H;
            for (int c = 0; c < H; ++c) y[c] = 0;
            for (int j = 0; j < k; ++j) {
                int e = topk_idx[(size_t)t * k + j];
                if (e < 0 || e >= E) continue;
                FN(slot_forward_)(H, I, x, (size_t)t * H, W1, (size_t)e * H * 2 * I,
                                  W2, (size_t)e * I * H, clamp, hg, hu, a, o);
                REAL wv = (REAL)topk_w[(size_t)t * k + j];
                for (int c = 0; c < H; ++c) y[c] += wv * o[c];
            }
        }
        free(hg); free(hu); free(a); free(o);
    }
}

/* dx rows and d(topk_w) rows for the listed tokens.
 *   dx[t,h]      = sum_j sum_i dhg[i] W1[e,h,i] + dhu[i] W1[e,h,I+i]
 *   dtopk_w[t,j] = sum_c dY[t,c] o[c]        (derivative of y w.r.t. w[t,j]) */
void FN(oracle_backward_tokens_)(int T, int H, int I, int E, int k, double clamp,
                                 const IN_T* x, const IN_T* W1, const IN_T* W2,
                                 const int32_t* topk_idx, const W_T* topk_w, const IN_T* dY,
                                 int n_tok, const int32_t* tok_list,
                                 REAL* dx_out, REAL* dtopk_w_out) {
    (void)T;
#pragma omp parallel
    {
        REAL* hg = (REAL*)malloc(sizeof(REAL) * (size_t)I);
        REAL* hu = (REAL*)malloc(sizeof(REAL) * (size_t)I);
        REAL* a = (REAL*)malloc(sizeof(REAL) * (size_t)I);
        REAL* o = (REAL*)malloc(sizeof(REAL) * (size_t)H);
        REAL* da = (REAL*)malloc(sizeof(REAL) * (size_t)I);
        REAL* dhg = (REAL*)malloc(sizeof(REAL) * (size_t)I);
        REAL* dhu = (REAL*)malloc(sizeof(REAL) * (size_t)I);
#pragma omp for schedule(dynamic, 1)
        for (int n = 0; n < n_tok; ++n) {
            int t = tok_list[n];
            REAL* dx = dx_out + (size_t)n * (size_t)H;
            for (int h = 0; h < H; ++h) dx[h] = 0;
            for (int j = 0; j < k; ++j) {
                int e = topk_idx[(size_t)t * k + j];
                REAL* dw = dtopk_w_out + (size_t)n * (size_t)k + (size_t)j;
                *dw = 0;
                if (e < 0 || e >= E) continue;
                size_t w1off = (size_t)e * H * 2 * I, w2off = (size_t)e * I * H;
                FN(slot_forward_)(H, I, x, (size_t)t * H, W1, w1off, W2, w2off, clamp, hg, hu, a, o);
                REAL s = 0;
                for (int c = 0; c < H; ++c) s += LD(dY, (size_t)t * H + (size_t)c) * o[c];
                *dw = s;
                REAL wv = (REAL)topk_w[(size_t)t * k + j];
                FN(slot_backward_)(H, I, dY, (size_t)t * H, wv, W2, w2off, clamp, hg, hu, da, dhg, dhu);
                for (int h = 0; h < H; ++h) {
                    size_t row = w1off + (size_t)h * (size_t)(2 * I);
                    REAL acc = 0;
                    for (int i = 0; i < I; ++i)
                        acc += dhg[i] * LD(W1, row + (size_t)i) + dhu[i] * LD(W1, row + (size_t)I + (size_t)i);
                    dx[h] += acc;
                }
            }
        }
        free(hg); free(hu); free(a); free(o); free(da); free(dhg); free(dhu);
    }
}

/* Full weight gradients of the listed experts (each sums over every slot
 * routed to it, in increasing slot order s = t*k + j):
 *   dW2[e,i,c]   = sum_slots a[i] * w * dY[t,c]
 *   dW1[e,h,i]   = sum_slots x[t,h] * dhg[i]
 *   dW1[e,h,I+i] = sum_slots x[t,h] * dhu[i]
 * An expert that receives no slot gets exactly zero.  The per-slot terms are
 * computed first; each output row is then summed over the slots in order
 * (rows are independent, so they are spread over threads). */
void FN(oracle_backward_experts_)(int T, int H, int I, int E, int k, double clamp,
                                  const IN_T* x, const IN_T* W1, const IN_T* W2,
                                  const int32_t* topk_idx, const W_T* topk_w, const IN_T* dY,
                                  int n_exp, const int32_t* exp_list,
                                  REAL* dW1_out, REAL* dW2_out) {
    int32_t* slots = (int32_t*)malloc(sizeof(int32_t) * (size_t)((int64_t)T * k + 1));
    for (int n = 0; n < n_exp; ++n) {
        int e = exp_list[n];
        REAL* dW1 = dW1_out + (size_t)n * H * 2 * I;
        REAL* dW2 = dW2_out + (size_t)n * I * H;
        int ns = 0;
        if (e >= 0 && e < E)
            for (int64_t s = 0; s < (int64_t)T * k; ++s)
                if (topk_idx[s] == e) slots[ns++] = (int32_t)s;
        size_t w1off = (size_t)(e < 0 ? 0 : e) * H * 2 * I, w2off = (size_t)(e < 0 ? 0 : e) * I * H;
        /* per-slot terms: a (times w), dhg, dhu */
        REAL* aw = (REAL*)malloc(sizeof(REAL) * ((size_t)ns * I + 1));
        REAL* dh = (REAL*)malloc(sizeof(REAL) * ((size_t)ns * 2 * I + 1));
#pragma omp parallel
        {
            REAL* hg = (REAL*)malloc(sizeof(REAL) * (size_t)I);
            REAL* hu = (REAL*)malloc(sizeof(REAL) * (size_t)I);
            REAL* a = (REAL*)malloc(sizeof(REAL) * (size_t)I);
            REAL* o = (REAL*)malloc(sizeof(REAL) * (size_t)H);
            REAL* da = (REAL*)malloc(sizeof(REAL) * (size_t)I);
#pragma omp for schedule(dynamic, 1)
            for (int q = 0; q < ns; ++q) {
                int64_t s = slots[q];
                int t = (int)(s / k);
                FN(slot_forward_)(H, I, x, (size_t)t * H, W1, w1off, W2, w2off, clamp, hg, hu, a, o);
                REAL wv = (REAL)topk_w[s];
                REAL* dhq = dh + (size_t)q * 2 * I;
                FN(slot_backward_)(H, I, dY, (size_t)t * H, wv, W2, w2off, clamp, hg, hu, da, dhq, dhq + I);
                for (int i = 0; i < I; ++i) aw[(size_t)q * I + i] = a[i] * wv;
            }
            free(hg); free(hu); free(a); free(o); free(da);
        }
#pragma omp parallel for schedule(static)
        for (int i = 0; i < I; ++i) {
            REAL* row = dW2 + (size_t)i * H;
            for (int c = 0; c < H; ++c) row[c] = 0;
            for (int q = 0; q < ns; ++q) {
                int t = (int)(slots[q] / k);
                REAL av = aw[(size_t)q * I + i];
                for (int c = 0; c < H; ++c) row[c] += av * LD(dY, (size_t)t * H + (size_t)c);
            }
        }
#pragma omp parallel for schedule(static)
        for (int h = 0; h < H; ++h) {
            REAL* row = dW1 + (size_t)h * 2 * I;
            for (int i = 0; i < 2 * I; ++i) row[i] = 0;
            for (int q = 0; q < ns; ++q) {
                int t = (int)(slots[q] / k);
                REAL xv = LD(x, (size_t)t * H + (size_t)h);
                const REAL* dhq = dh + (size_t)q * 2 * I;
                for (int i = 0; i < 2 * I; ++i) row[i] += xv * dhq[i];
            }
        }
        free(aw); free(dh);
    }
    free(slots);
}

#undef FN
#undef CAT
#undef CAT2

/*
 * moe_oracle.c -- plain FP64 CPU oracle for the local MoE forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA path.
 *
 * Every step is the plain definition of what the pages specify, written for a
 * reader to check by eye: no blocking, no fusion, no reordering.  All
 * arithmetic is double precision; inputs stored as F32/F16/BF16 are decoded
 * exactly to double here.  Loops parallelised with OpenMP only over
 * independent outputs (each output element is computed by one thread in a
 * fixed order), so results do not depend on the thread count.
 *
 * Sources (page title, section):
 *   [UG4]  ruDNN Benutzerhandbuch, section 4 "Routing-Vertrag": FP32 softmax
 *          over all experts before top-k, ties to the lower expert id,
 *          optional renormalisation then cast to the logits dtype, NaN weights
 *          for rows holding NaN, +inf or only -inf; indices U32 [T, top_k].
 *   [UG5]  same page, section 5 "Expertengewichte und Verteilung": input
 *          [T,H], gate/up [E,I,H], down [E,H,I]; dispatch drops no token;
 *          a stored map restores token order.
 *   [UG6]  same page, section 6 "MoE aufrufen": combine restores token order
 *          and sums expert outputs with the routing weights.
 *   [EXP]  ruDNN 0.1.25 source view, src/moe/experts.rs,
 *          SwiGluExperts::forward_dispatched_with_strategy: gate and up
 *          segmented grouped products (out = in . W[e]^T), silu(gate)*up,
 *          then the down product.  SwiGluExperts::new: bias-free weights.
 *   [SILU] MindSpeed-Ops PR 163 diffs, rms_norm_gated notes: silu(x) is
 *          x * sigmoid(x).
 *   [UG10] ruDNN Benutzerhandbuch, section 10: sigmoid group-limited routing.
 *   [UG12] same page, section 12 "MoE-Training erster Ordnung": the backward
 *          chain (combine, experts, dispatch, router).
 *   [EXPB] src/moe/experts.rs, ExpertTrainingCache::backward_with_strategy.
 *
 * Readings where the pages leave a step open (the same list is kept in the
 * design notes):
 *   R1 the selection key is the logit itself (softmax is strictly monotone,
 *      so this is top-k of the softmax); equal logits -> lower id; +0 == -0.
 *   R2 slot order of idx[t,:]: descending weight, ties -> lower id.
 *   R3 a poisoned row (any NaN, any +inf, or every entry -inf) is all-tied:
 *      idx = 0..k-1 and every weight NaN; it is still dispatched.
 *   R4 weights are always stored in the logits dtype (cast by round to
 *      nearest even), with or without renormalisation.
 *   R7 no intermediate rounding in the oracle.
 *   R8 the combine uses the cast weights.
 *
 * Parity status: every function below is pinned by the CPU test suite
 * (brute-force top-k enumeration, closed-form softmax cases, the NaN rule,
 * dispatch invariants and a library stable sort, a dense masked per-token
 * evaluation and the E=1/k=1 plain SwiGLU MLP).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* storage codes: 0 = F32, 1 = F16, 2 = BF16 */
enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2 };

/* ------------------------------------------------------------------------ */
/* exact decoding of stored elements to double                              */
/* ------------------------------------------------------------------------ */

static double decode_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    double v;
    if (expo == 0x1f) {
        v = mant ? NAN : INFINITY;
    } else if (expo == 0) {
        v = ldexp((double)mant, -24); /* subnormal: mant * 2^-24 */
    } else {
        v = ldexp((double)(mant | 0x400), expo - 25); /* 1.mant * 2^(e-15) */
    }
    return sign ? -v : v;
}

static double decode_bf16(uint16_t b) {
    uint32_t bits = (uint32_t)b << 16; /* bf16 is the top half of an f32 */
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double load_elem(const void* base, int dtype, int64_t i) {
    switch (dtype) {
    case OR_F32: return (double)((const float*)base)[i];
    case OR_F16: return decode_f16(((const uint16_t*)base)[i]);
    default:     return decode_bf16(((const uint16_t*)base)[i]);
    }
}

/* Round a double to the nearest value of the storage format (ties to even),
 * returned as a double.  Formats: precision p bits, minimum normal exponent
 * emin, maximum finite value fmax.  Overflow beyond the rounding threshold
 * gives infinity, as IEEE round-to-nearest does. */
double oracle_round_to_dtype(double v, int dtype) {
    if (isnan(v) || isinf(v) || v == 0.0) return v;
    int p, emin;
    double fmax;
    if (dtype == OR_F32) { p = 24; emin = -126; fmax = ldexp(2.0 - ldexp(1.0, -23), 127); }
    else if (dtype == OR_F16) { p = 11; emin = -14; fmax = 65504.0; }
    else { p = 8; emin = -126; fmax = ldexp(2.0 - ldexp(1.0, -7), 127); }
    int ex;
    frexp(fabs(v), &ex);          /* |v| = m * 2^ex, m in [0.5, 1) */
    int lead = ex - 1;            /* exponent of the leading bit */
    if (lead < emin) lead = emin; /* subnormal range: fixed quantum */
    double quantum = ldexp(1.0, lead - (p - 1));
    double r = rint(v / quantum) * quantum; /* rint: ties to even (default mode) */
    if (fabs(r) > fmax) return v > 0 ? INFINITY : -INFINITY;
    return r;
}

/* ------------------------------------------------------------------------ */
/* routing  [UG4]                                                           */
/* ------------------------------------------------------------------------ */

/* "a beats b" for selection: larger logit first, equal logits -> lower id. */
static int beats(double la, int64_t a, double lb, int64_t b) {
    if (la > lb) return 1;
    if (la < lb) return 0;
    return a < b; /* equal (including +0 vs -0) */
}

/* One row of the routing contract.
 *   l[0..E-1]      logits of the row, exact in double
 *   idx[0..k-1]    selected experts, descending weight (R2)
 *   w_pre[0..k-1]  weights before the cast (softmax value, optionally
 *                  renormalised over the selected set)
 *   w_cast[0..k-1] weights rounded to the logits dtype (R4)            */
static void route_row(const double* l, int64_t E, int k, int renorm, int wdtype,
                      uint32_t* idx, double* w_pre, double* w_cast) {
    int has_nan = 0, has_pinf = 0, all_ninf = 1;
    for (int64_t e = 0; e < E; ++e) {
        if (isnan(l[e])) has_nan = 1;
        if (l[e] == INFINITY) has_pinf = 1;
        if (l[e] != -INFINITY) all_ninf = 0;
    }
    if (has_nan || has_pinf || all_ninf) { /* R3: NaN weights, all-tied row */
        for (int j = 0; j < k; ++j) {
            idx[j] = (uint32_t)j;
            w_pre[j] = NAN;
            w_cast[j] = NAN;
        }
        return;
    }
    /* softmax over all experts: p_e = exp(l_e - m) / sum_i exp(l_i - m) */
    double m = -INFINITY;
    for (int64_t e = 0; e < E; ++e) if (l[e] > m) m = l[e];
    double s = 0.0;
    for (int64_t e = 0; e < E; ++e) s += exp(l[e] - m);

    /* top-k by (logit desc, id asc): k passes, each taking the best unused */
    char* used = (char*)calloc((size_t)E, 1);
    for (int j = 0; j < k; ++j) {
        int64_t best = -1;
        for (int64_t e = 0; e < E; ++e) {
            if (used[e]) continue;
            if (best < 0 || beats(l[e], e, l[best], best)) best = e;
        }
        used[best] = 1;
        idx[j] = (uint32_t)best;
        w_pre[j] = exp(l[best] - m) / s;
    }
    free(used);
    if (renorm) {
        double tot = 0.0;
        for (int j = 0; j < k; ++j) tot += w_pre[j];
        for (int j = 0; j < k; ++j) w_pre[j] = w_pre[j] / tot;
    }
    for (int j = 0; j < k; ++j) w_cast[j] = oracle_round_to_dtype(w_pre[j], wdtype);
}

/* logits: T*E stored elements of dtype ldt.  Outputs idx [T*k] u32,
 * w_pre [T*k], w_cast [T*k]. */
void oracle_route(const void* logits, int ldt, int64_t T, int64_t E, int k, int renorm,
                  uint32_t* idx, double* w_pre, double* w_cast) {
#pragma omp parallel
    {
        double* row = (double*)malloc((size_t)E * sizeof(double));
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            for (int64_t e = 0; e < E; ++e) row[e] = load_elem(logits, ldt, t * E + e);
            route_row(row, E, k, renorm, ldt, idx + t * k, w_pre + t * k, w_cast + t * k);
        }
        free(row);
    }
}

/* ------------------------------------------------------------------------ */
/* sigmoid group-limited routing  [UG10]                                    */
/* ------------------------------------------------------------------------ */
/* ruDNN Benutzerhandbuch, section 10 "Gruppenbeschraenktes Sigmoid-MoE-
 * Routing": scores are sigmoid(logit); an optional FP32 correction bias is
 * added for the selection only; experts form `groups` equal contiguous
 * groups; a group's score is the largest corrected score of its experts, or
 * the sum of its two largest when group_top_two is set; the
 * `selected_groups` best groups are kept and top_k experts are chosen among
 * their experts by corrected score; ties go to the lower id (group or
 * expert).  Weights are the original sigmoid values, optionally
 * renormalised over the selected experts, times `scale`.
 *
 * Readings (also in the design notes):
 *   S1 the selection runs in FP32 as the page states for the bias: the
 *      sigmoid is the correctly rounded FP32 value of 1/(1+exp(-x)) (computed
 *      in double, rounded once), the corrected score is its FP32 sum with the
 *      bias and the top-two group score is an FP32 sum;
 *   S2 slot order: descending corrected score, ties to the lower id;
 *   S3 a row holding a NaN logit or NaN corrected score is all-tied: idx =
 *      0..k-1 and NaN weights (the section 4 rule carried over);
 *   S4 weights are stored in the logits dtype (round to nearest even). */
static float sigmoid_f32(double x) { return (float)(1.0 / (1.0 + exp(-x))); }

/* "a beats b" on FP32 keys: larger first, equal -> lower id */
static int beats_f(float va, int64_t a, float vb, int64_t b) {
    if (va > vb) return 1;
    if (va < vb) return 0;
    return a < b;
}

void oracle_route_sigmoid_grouped(const void* logits, int ldt, int64_t T, int64_t E,
                                  const float* bias, int k, int groups, int selected_groups,
                                  int group_top_two, int renorm, double scale,
                                  uint32_t* idx, double* w_pre, double* w_cast) {
    const int64_t gs = E / groups;
#pragma omp parallel
    {
        float* c = (float*)malloc((size_t)E * sizeof(float));
        double* sig = (double*)malloc((size_t)E * sizeof(double));
        float* gscore = (float*)malloc((size_t)groups * sizeof(float));
        char* gsel = (char*)malloc((size_t)groups);
        char* used = (char*)malloc((size_t)E);
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            uint32_t* ix = idx + t * k;
            double* wp = w_pre + t * k;
            double* wc = w_cast + t * k;
            int poisoned = 0;
            for (int64_t e = 0; e < E; ++e) {
                const double l = load_elem(logits, ldt, t * E + e);
                sig[e] = 1.0 / (1.0 + exp(-l));          /* weight value, no rounding */
                c[e] = sigmoid_f32(l) + (bias ? bias[e] : 0.0f); /* FP32 selection key */
                if (isnan(l) || isnan(c[e])) poisoned = 1;
            }
            if (poisoned) {
                for (int j = 0; j < k; ++j) { ix[j] = (uint32_t)j; wp[j] = NAN; wc[j] = NAN; }
                continue;
            }
            /* group scores */
            for (int g = 0; g < groups; ++g) {
                float best = -INFINITY, second = -INFINITY;
                int64_t bi = -1;
                for (int64_t e = g * gs; e < (g + 1) * gs; ++e)
                    if (bi < 0 || beats_f(c[e], e, best, bi)) { best = c[e]; bi = e; }
                for (int64_t e = g * gs; e < (g + 1) * gs; ++e)
                    if (e != bi && c[e] > second) second = c[e];
                gscore[g] = group_top_two ? best + second : best;
                gsel[g] = 0;
            }
            /* keep the selected_groups best groups */
            for (int r = 0; r < selected_groups; ++r) {
                int bg = -1;
                for (int g = 0; g < groups; ++g)
                    if (!gsel[g] && (bg < 0 || beats_f(gscore[g], g, gscore[bg], bg))) bg = g;
                gsel[bg] = 1;
            }
            /* top_k experts of the kept groups by corrected score */
            for (int64_t e = 0; e < E; ++e) used[e] = !gsel[e / gs];
            double tot = 0.0;
            for (int j = 0; j < k; ++j) {
                int64_t be = -1;
                for (int64_t e = 0; e < E; ++e)
                    if (!used[e] && (be < 0 || beats_f(c[e], e, c[be], be))) be = e;
                used[be] = 1;
                ix[j] = (uint32_t)be;
                wp[j] = sig[be];
                tot += sig[be];
            }
            for (int j = 0; j < k; ++j) {
                if (renorm) wp[j] = wp[j] / tot;
                wp[j] = wp[j] * scale;
                wc[j] = oracle_round_to_dtype(wp[j], ldt);
            }
        }
        free(c); free(sig); free(gscore); free(gsel); free(used);
    }
}

/* ------------------------------------------------------------------------ */
/* dispatch  [UG5]                                                          */
/* ------------------------------------------------------------------------ */

/* Capacity-free dispatch into contiguous per-expert segments.
 *   c_e = number of slots (t,j) with idx[t,j] == e
 *   offsets[0] = 0, offsets[e+1] = offsets[e] + c_e
 *   segment e lists its slots in ascending flat slot index s = t*k + j
 *   (a stable counting sort of the slots by expert id)
 *   perm[r] = s, row_experts[r] = e for the r-th dispatched row.
 * Slots whose index is >= E are not dispatched; they are counted in
 * *invalid and the unused tail of perm/row_experts is set to 0xFFFFFFFF. */
void oracle_dispatch(const uint32_t* idx, int64_t T, int64_t E, int k,
                     uint32_t* offsets, uint32_t* row_experts, uint32_t* perm,
                     int64_t* invalid) {
    int64_t n = T * (int64_t)k;
    int64_t bad = 0;
    for (int64_t e = 0; e <= E; ++e) offsets[e] = 0;
    for (int64_t s = 0; s < n; ++s) {
        if (idx[s] < (uint64_t)E) offsets[idx[s] + 1] += 1;
        else ++bad;
    }
    for (int64_t e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
    uint64_t* fill = (uint64_t*)calloc((size_t)E, sizeof(uint64_t));
    for (int64_t s = 0; s < n; ++s) { /* ascending s: stable */
        uint32_t e = idx[s];
        if (e >= (uint64_t)E) continue;
        uint64_t r = offsets[e] + fill[e]++;
        perm[r] = (uint32_t)s;
        row_experts[r] = e;
    }
    free(fill);
    for (int64_t r = n - bad; r < n; ++r) { perm[r] = 0xFFFFFFFFu; row_experts[r] = 0xFFFFFFFFu; }
    *invalid = bad;
}

/* ------------------------------------------------------------------------ */
/* experts  [EXP], [SILU]                                                    */
/* ------------------------------------------------------------------------ */

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* One bias-free SwiGLU expert on one row:
 *   g_i = sum_h W_gate[e,i,h] x_h,  u_i = sum_h W_up[e,i,h] x_h
 *   a_i = silu(g_i) * u_i
 *   o_c = sum_i W_down[e,c,i] a_i                                        */
static void expert_row(const double* x, int64_t e, int64_t H, int64_t I,
                       const void* gate, const void* up, const void* down, int wdt,
                       double* a /* scratch [I] */, double* o /* [H] */) {
    for (int64_t i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        int64_t base = (e * I + i) * H;
        for (int64_t h = 0; h < H; ++h) {
            g += load_elem(gate, wdt, base + h) * x[h];
            u += load_elem(up, wdt, base + h) * x[h];
        }
        a[i] = silu(g) * u;
    }
    for (int64_t c = 0; c < H; ++c) {
        double acc = 0.0;
        int64_t base = (e * H + c) * I;
        for (int64_t i = 0; i < I; ++i) acc += load_elem(down, wdt, base + i) * a[i];
        o[c] = acc;
    }
}

/* Experts on dispatched rows: out[r,:] = expert_{row_experts[r]}(x_disp[r,:])
 * for r < offsets[E]; rows beyond are left untouched.  x_disp is given in
 * double (the caller decodes it), out is [N,H] double. */
void oracle_experts(const double* x_disp, const uint32_t* offsets, int64_t E,
                    const void* gate, const void* up, const void* down, int wdt,
                    int64_t H, int64_t I, double* out) {
    int64_t nrows = offsets[E];
#pragma omp parallel
    {
        double* a = (double*)malloc((size_t)I * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            int64_t e = 0;
            while (!(offsets[e] <= (uint64_t)r && (uint64_t)r < offsets[e + 1])) ++e;
            expert_row(x_disp + r * H, e, H, I, gate, up, down, wdt, a, out + r * H);
        }
        free(a);
    }
}

/* ------------------------------------------------------------------------ */
/* combine  [UG6]                                                           */
/* ------------------------------------------------------------------------ */

/* y[t,:] = sum_j w_cast[t,j] * expert_out[r(t,j),:], where r(t,j) is the
 * dispatched row holding slot s = t*k+j (the inverse of perm), summed in
 * ascending j.  A slot that was not dispatched makes its token's row NaN. */
void oracle_combine(const double* expert_out, const uint32_t* perm, const double* w_cast,
                    int64_t T, int k, int64_t H, double* y) {
    int64_t n = T * (int64_t)k;
    int64_t* row_of = (int64_t*)malloc((size_t)(n > 0 ? n : 1) * sizeof(int64_t));
    for (int64_t s = 0; s < n; ++s) row_of[s] = -1;
    for (int64_t r = 0; r < n; ++r)
        if (perm[r] != 0xFFFFFFFFu) row_of[perm[r]] = r;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t c = 0; c < H; ++c) y[t * H + c] = 0.0;
        for (int j = 0; j < k; ++j) {
            int64_t r = row_of[t * k + j];
            for (int64_t c = 0; c < H; ++c)
                y[t * H + c] += (r < 0) ? NAN : w_cast[t * k + j] * expert_out[r * H + c];
        }
    }
    free(row_of);
}

/* ------------------------------------------------------------------------ */
/* whole forward for a sample of tokens (route -> experts -> weighted sum)   */
/* ------------------------------------------------------------------------ */

/* For each listed token t: route its logits row, evaluate its k selected
 * experts on x[t,:] and sum them with the cast weights in slot order.
 * This is the per-token meaning of dispatch + experts + combine, used to
 * check large problems on a sample of tokens.  Outputs for sample i:
 * idx_out[i*k..], w_out[i*k..] (pre-cast), y_out[i*H..].
 * expert_slot (may be NULL): expert e's weights sit at position
 * expert_slot[e] of gate/up/down, so that a caller can pass only the
 * experts its sample touches; NULL means position e. */
void oracle_forward_tokens(const void* x, const void* logits, int ldt, int xdt,
                           int64_t T, int64_t E, int k, int renorm, int64_t H, int64_t I,
                           const void* gate, const void* up, const void* down,
                           const int64_t* expert_slot,
                           const int64_t* tokens, int64_t ntok,
                           uint32_t* idx_out, double* w_out, double* y_out) {
    (void)T;
#pragma omp parallel
    {
        double* row = (double*)malloc((size_t)E * sizeof(double));
        double* xt = (double*)malloc((size_t)H * sizeof(double));
        double* a = (double*)malloc((size_t)I * sizeof(double));
        double* o = (double*)malloc((size_t)H * sizeof(double));
        double* wc = (double*)malloc((size_t)k * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < ntok; ++i) {
            int64_t t = tokens[i];
            for (int64_t e = 0; e < E; ++e) row[e] = load_elem(logits, ldt, t * E + e);
            route_row(row, E, k, renorm, ldt, idx_out + i * k, w_out + i * k, wc);
            for (int64_t h = 0; h < H; ++h) xt[h] = load_elem(x, xdt, t * H + h);
            double* y = y_out + i * H;
            for (int64_t h = 0; h < H; ++h) y[h] = 0.0;
            for (int j = 0; j < k; ++j) {
                int64_t e = idx_out[i * k + j];
                if (expert_slot) e = expert_slot[e];
                if (e < 0) { /* caller did not pass this expert */
                    for (int64_t h = 0; h < H; ++h) o[h] = NAN;
                } else {
                    expert_row(xt, e, H, I, gate, up, down, xdt, a, o);
                }
                for (int64_t h = 0; h < H; ++h) y[h] += wc[j] * o[h];
            }
        }
        free(row); free(xt); free(a); free(o); free(wc);
    }
}

/* ------------------------------------------------------------------------ */
/* first-order training backward  [UG12], [EXPB]                            */
/* ------------------------------------------------------------------------ */
/* ruDNN Benutzerhandbuch, section 12 "MoE-Training erster Ordnung", and the
 * ExpertTrainingCache::backward of src/moe/experts.rs:
 *   1. combine backward: dexpert[r] = w[t,j] * dy[t] for the row r holding
 *      slot (t,j); dweights[t,j] = <expert_out[r], dy[t]> (FP32 on the pages);
 *   2. expert backward: for g = x W_gate^T, u = x W_up^T, a = silu(g) u,
 *      o = a W_down^T and upstream do:
 *        da = do W_down,  ddown = sum_r do_r^T a_r,
 *        dg = da u silu'(g),  du = da silu(g),
 *        dgate = sum_r dg_r^T x_r,  dup = sum_r du_r^T x_r,
 *        dinput = dg W_gate + du W_up     (weight gradients FP32 on the pages);
 *   3. dispatch backward: dx[t] = sum_j dinput[r(t,j)], no routing weights;
 *   4. router backward: gradient of the selected router weights (fixed
 *      selection) with respect to the logits; repeated indices gather;
 *      an index outside [0,E) makes the whole row NaN.
 * Pinned by central finite differences of the forward functions above. */

static double silu_grad(double z) {  /* d/dz z*sigmoid(z) */
    const double s = 1.0 / (1.0 + exp(-z));
    return s * (1.0 + z * (1.0 - s));
}

void oracle_combine_backward(const double* expert_out, const uint32_t* perm, const double* w,
                             const double* dy, int64_t T, int k, int64_t H,
                             double* dexpert, double* dweights) {
    int64_t n = T * (int64_t)k;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        const uint32_t s = perm[r];
        if (s == 0xFFFFFFFFu) continue;
        const int64_t t = s / (uint32_t)k;
        double dot = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            dexpert[r * H + h] = w[s] * dy[t * H + h];
            dot += expert_out[r * H + h] * dy[t * H + h];
        }
        dweights[s] = dot;
    }
}

void oracle_experts_backward(const double* x_disp, const uint32_t* offsets, int64_t E,
                             const void* gate, const void* up, const void* down, int wdt,
                             int64_t H, int64_t I, const double* dout,
                             double* dinput, double* dgate, double* dup, double* ddown) {
    const int64_t nrows = offsets[E];
    /* per-row quantities */
    double* g = (double*)malloc((size_t)(nrows > 0 ? nrows : 1) * I * sizeof(double));
    double* u = (double*)malloc((size_t)(nrows > 0 ? nrows : 1) * I * sizeof(double));
    double* da = (double*)malloc((size_t)(nrows > 0 ? nrows : 1) * I * sizeof(double));
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t e = 0;
        while (!(offsets[e] <= (uint64_t)r && (uint64_t)r < offsets[e + 1])) ++e;
        for (int64_t i = 0; i < I; ++i) {
            double gg = 0.0, uu = 0.0, dd = 0.0;
            for (int64_t h = 0; h < H; ++h) {
                gg += load_elem(gate, wdt, (e * I + i) * H + h) * x_disp[r * H + h];
                uu += load_elem(up, wdt, (e * I + i) * H + h) * x_disp[r * H + h];
                dd += dout[r * H + h] * load_elem(down, wdt, (e * H + h) * I + i);
            }
            g[r * I + i] = gg;
            u[r * I + i] = uu;
            da[r * I + i] = dd;
        }
        for (int64_t h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int64_t i = 0; i < I; ++i) {
                const double gg = g[r * I + i], uu = u[r * I + i], d = da[r * I + i];
                const double dg = d * uu * silu_grad(gg);
                const double du = d * silu(gg);
                acc += dg * load_elem(gate, wdt, (e * I + i) * H + h) +
                       du * load_elem(up, wdt, (e * I + i) * H + h);
            }
            dinput[r * H + h] = acc;
        }
    }
    /* weight gradients: sums over each expert's rows, taken in ascending row
     * order for every weight (rows outermost so that the row data is read
     * contiguously; the order of the additions is the same as a per-weight loop) */
    double* sl = (double*)malloc((size_t)(nrows > 0 ? nrows : 1) * I * sizeof(double));
#pragma omp parallel for
    for (int64_t j = 0; j < nrows * I; ++j) sl[j] = silu(g[j]);
    for (int64_t e = 0; e < E; ++e) {
        const int64_t r0 = offsets[e], r1 = offsets[e + 1];
#pragma omp parallel for schedule(dynamic, 4)
        for (int64_t i = 0; i < I; ++i) {
            double* sg = dgate + (e * I + i) * H;
            double* su = dup + (e * I + i) * H;
            for (int64_t h = 0; h < H; ++h) sg[h] = su[h] = 0.0;
            for (int64_t r = r0; r < r1; ++r) {
                const double gg = g[r * I + i], uu = u[r * I + i], d = da[r * I + i];
                const double cg = d * uu * silu_grad(gg), cu = d * silu(gg);
                for (int64_t h = 0; h < H; ++h) {
                    sg[h] += cg * x_disp[r * H + h];
                    su[h] += cu * x_disp[r * H + h];
                }
            }
        }
#pragma omp parallel for schedule(dynamic, 4)
        for (int64_t h = 0; h < H; ++h) {
            double* sd = ddown + (e * H + h) * I;
            for (int64_t i = 0; i < I; ++i) sd[i] = 0.0;
            for (int64_t r = r0; r < r1; ++r) {
                const double dd = dout[r * H + h];
                for (int64_t i = 0; i < I; ++i) sd[i] += dd * sl[r * I + i] * u[r * I + i];
            }
        }
    }
    free(sl);
    free(g); free(u); free(da);
}

void oracle_dispatch_backward(const double* dinput, const uint32_t* perm, int64_t T, int k,
                              int64_t H, double* dx) {
    int64_t n = T * (int64_t)k;
    for (int64_t i = 0; i < T * H; ++i) dx[i] = 0.0;
    for (int64_t r = 0; r < n; ++r) { /* ascending r per token: any fixed order, exact sums */
        if (perm[r] == 0xFFFFFFFFu) continue;
        const int64_t t = perm[r] / (uint32_t)k;
        for (int64_t h = 0; h < H; ++h) dx[t * H + h] += dinput[r * H + h];
    }
}

/* Selected router weights for a fixed selection idx (section 12
 * selected_router_weights): scoring 0 = softmax over all E, 1 = sigmoid;
 * optional renormalisation over the selected weights; times scale. */
void oracle_selected_router_weights(const double* logits, const int64_t* idx, int64_t T, int64_t E,
                                    int k, int scoring, int renorm, double scale, double* w) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const double* l = logits + t * E;
        int bad = 0;
        for (int j = 0; j < k; ++j) if (idx[t * k + j] < 0 || idx[t * k + j] >= E) bad = 1;
        if (bad) { for (int j = 0; j < k; ++j) w[t * k + j] = NAN; continue; }
        double m = -INFINITY, s = 0.0;
        if (scoring == 0) {
            for (int64_t e = 0; e < E; ++e) if (l[e] > m) m = l[e];
            for (int64_t e = 0; e < E; ++e) s += exp(l[e] - m);
        }
        double tot = 0.0;
        for (int j = 0; j < k; ++j) {
            const double x = l[idx[t * k + j]];
            w[t * k + j] = scoring == 0 ? exp(x - m) / s : 1.0 / (1.0 + exp(-x));
            tot += w[t * k + j];
        }
        for (int j = 0; j < k; ++j) w[t * k + j] = (renorm ? w[t * k + j] / tot : w[t * k + j]) * scale;
    }
}

/* Gradient of the selected router weights above with respect to the logits,
 * given dL/dw (dweights).  Chain rule through scale, renormalisation
 * (w_j = q_j / Q, Q = sum_m q_m) and the scoring:
 *   softmax: dq_m/dl_e = q_m (delta(e, idx_m) - p_e)
 *   sigmoid: dq_m/dl_e = q_m (1 - q_m) delta(e, idx_m)                    */
void oracle_router_backward(const double* logits, const int64_t* idx, const double* dw,
                            int64_t T, int64_t E, int k, int scoring, int renorm, double scale,
                            double* dlogits) {
#pragma omp parallel
    {
        double* p = (double*)malloc((size_t)E * sizeof(double));
        double* q = (double*)malloc((size_t)k * sizeof(double));
        double* c = (double*)malloc((size_t)k * sizeof(double));
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            const double* l = logits + t * E;
            double* d = dlogits + t * E;
            int bad = 0;
            for (int j = 0; j < k; ++j) if (idx[t * k + j] < 0 || idx[t * k + j] >= E) bad = 1;
            if (bad) { for (int64_t e = 0; e < E; ++e) d[e] = NAN; continue; }
            if (scoring == 0) {
                double m = -INFINITY, s = 0.0;
                for (int64_t e = 0; e < E; ++e) if (l[e] > m) m = l[e];
                for (int64_t e = 0; e < E; ++e) s += exp(l[e] - m);
                for (int64_t e = 0; e < E; ++e) p[e] = exp(l[e] - m) / s;
            }
            double Q = 0.0;
            for (int j = 0; j < k; ++j) {
                const double x = l[idx[t * k + j]];
                q[j] = scoring == 0 ? p[idx[t * k + j]] : 1.0 / (1.0 + exp(-x));
                Q += q[j];
            }
            /* c_m = dL/dq_m */
            double gq = 0.0;
            for (int j = 0; j < k; ++j) gq += dw[t * k + j] * q[j];
            for (int m = 0; m < k; ++m)
                c[m] = renorm ? scale * (dw[t * k + m] / Q - gq / (Q * Q)) : scale * dw[t * k + m];
            for (int64_t e = 0; e < E; ++e) d[e] = 0.0;
            double cq = 0.0;
            for (int m = 0; m < k; ++m) {
                const int64_t e = idx[t * k + m];
                if (scoring == 0) {
                    d[e] += c[m] * q[m];
                    cq += c[m] * q[m];
                } else {
                    d[e] += c[m] * q[m] * (1.0 - q[m]);
                }
            }
            if (scoring == 0)
                for (int64_t e = 0; e < E; ++e) d[e] -= p[e] * cq;
        }
        free(p); free(q); free(c);
    }
}

/* decoding helper for the Python side: n stored elements -> double */
void oracle_decode(const void* src, int dtype, int64_t n, double* dst) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) dst[i] = load_elem(src, dtype, i);
}

int oracle_num_threads(void);
#ifdef _OPENMP
#include <omp.h>
int oracle_num_threads(void) { return omp_get_max_threads(); }
void oracle_set_threads(int n) { omp_set_num_threads(n); }
#else
int oracle_num_threads(void) { return 1; }
void oracle_set_threads(int n) { (void)n; }
#endif

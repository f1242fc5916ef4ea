/*
 * CPU oracle for the split-residency routed MoE layer -- TEST INFRASTRUCTURE.
 * Only tests/, the smoke check and the benchmark's cpu_baseline leg use it.
 * See moe_oracle.h for the passages each function follows.
 *
 * Plain loops, no blocking or reordering beyond what the definitions state.
 * OpenMP only splits independent output rows across threads; it never
 * changes the order of any sum.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* OCP MX v1.0, FP4 E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit.
 * Exponent field 0 is subnormal: value = 2^(1-1) * (0 + m/2).
 * Otherwise value = 2^(E-1) * (1 + m/2).  No Inf/NaN encodings. */
double orc_e2m1_value(unsigned code) {
    unsigned sign = (code >> 3) & 1u;
    unsigned ex = (code >> 1) & 3u;
    unsigned man = code & 1u;
    double mag;
    if (ex == 0)
        mag = 0.5 * (double)man;
    else
        mag = ldexp(1.0 + 0.5 * (double)man, (int)ex - 1);
    return sign ? -mag : mag;
}

/* OCP MX v1.0, E8M0 scale: 2^(b - 127); 0xFF is NaN. */
double orc_e8m0_value(unsigned byte) {
    if ((byte & 0xFFu) == 0xFFu) return NAN;
    return ldexp(1.0, (int)(byte & 0xFFu) - 127);
}

void orc_dequant(const uint8_t *q, const uint8_t *s, int64_t rows, int64_t K, double *out) {
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < K; ++c) {
            uint8_t byte = q[r * (K / 2) + c / 2];
            unsigned code = (c % 2 == 0) ? (byte & 0x0Fu) : (byte >> 4);
            double scale = orc_e8m0_value(s[r * (K / 32) + c / 32]);
            out[r * K + c] = orc_e2m1_value(code) * scale;
        }
    }
}

float orc_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round to nearest, ties to even, on the bit pattern; NaN stays a quiet NaN. */
uint16_t orc_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------ router */

void orc_router_logits(const uint16_t *x, const uint16_t *w_router, const float *bias, int T, int E, int H,
                       float *logits) {
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            double sum = bias ? (double)bias[e] : 0.0;
            for (int h = 0; h < H; ++h)
                sum += (double)orc_bf16_to_f32(x[(int64_t)t * H + h]) *
                       (double)orc_bf16_to_f32(w_router[(int64_t)e * H + h]);
            logits[(int64_t)t * E + e] = (float)sum;
        }
    }
}

/* ---------------------------------------------------------------- routing */

/* a ranks before b: larger logit first, equal logits by lower expert id. */
static int ranks_before(float la, int a, float lb, int b) {
    if (la > lb) return 1;
    if (la < lb) return 0;
    return a < b;
}

/* A logit as routing reads it: NaN -> -infinity. */
static float routing_logit(float v) { return isnan(v) ? -INFINITY : v; }

void orc_route(const float *logits, int T, int E, int k, int32_t *ids, float *w) {
    float *l = (float *)malloc(sizeof(float) * (size_t)(E > 0 ? E : 1));
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) l[e] = routing_logit(logits[(int64_t)t * E + e]);
        int32_t *id = ids + (int64_t)t * k;
        /* selection: k passes, each taking the best expert not yet taken */
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                int taken = 0;
                for (int i = 0; i < j; ++i)
                    if (id[i] == e) taken = 1;
                if (taken) continue;
                if (best < 0 || ranks_before(l[e], e, l[best], best)) best = e;
            }
            id[j] = best;
        }
        /* softmax over the k picks, fp32, shifted by the largest (first) */
        float ex[64];
        float sum = 0.0f;
        for (int j = 0; j < k; ++j) {
            ex[j] = expf(l[id[j]] - l[id[0]]);
            sum = sum + ex[j];
        }
        for (int j = 0; j < k; ++j) w[(int64_t)t * k + j] = ex[j] / sum;
    }
    free(l);
}

/* ------------------------------------------------------------- residency */

void orc_initial_rowmap(const uint8_t *is_hot, int E, int32_t *row_map, int *n_hot, int *n_cold) {
    int h = 0, c = 0;
    for (int e = 0; e < E; ++e) {
        if (is_hot[e])
            row_map[e] = h++;
        else
            row_map[e] = -1 - (c++);
    }
    if (n_hot) *n_hot = h;
    if (n_cold) *n_cold = c;
}

void orc_split(const int32_t *row_map, int E, const int32_t *ids, int T, int k, orc_split_t *out) {
    (void)E;
    int P = T * k;
    for (int b = 0; b < 2; ++b) {
        /* local row of every slot in bank b, -1 if the slot is in the other */
        int32_t max_row = -1;
        for (int s = 0; s < P; ++s) {
            int32_t m = row_map[ids[s]];
            int in_b = (b == 0) ? (m >= 0) : (m < 0);
            int32_t r = (b == 0) ? m : (-1 - m);
            if (in_b && r > max_row) max_row = r;
        }
        int n_act = 0, n = 0;
        out->act_off[b][0] = 0;
        for (int32_t r = 0; r <= max_row; ++r) {
            int any = 0;
            for (int s = 0; s < P; ++s) {
                int32_t m = row_map[ids[s]];
                int in_b = (b == 0) ? (m >= 0) : (m < 0);
                int32_t rr = (b == 0) ? m : (-1 - m);
                if (in_b && rr == r) {
                    out->picks[b][n++] = s;
                    any = 1;
                }
            }
            if (any) {
                out->act_row[b][n_act] = r;
                out->act_off[b][n_act + 1] = n;
                ++n_act;
            }
        }
        out->n_picks[b] = n;
        out->n_act[b] = n_act;
    }
}

void orc_count(int32_t *counts, int E, const int32_t *ids, int T, int k, int count_on, int count_tmax) {
    (void)E;
    if (!count_on || T > count_tmax) return;
    for (int s = 0; s < T * k; ++s) counts[ids[s]] += 1;
}

/* -------------------------------------------------------------- expert FFN */

static void dequant_row(const uint8_t *q, const uint8_t *s, int64_t row, int K, double *out) {
    orc_dequant(q + row * (K / 2), s + row * (K / 32), 1, K, out);
}

static float silu_f32(float z) { return z / (1.0f + expf(-z)); }

/* ------------------------------------------------------ MXFP8 activations */

/* FP8 E4M3 (the OCP "E4M3" element type: exponent bias 7, 3 mantissa bits,
 * largest finite 448, no infinities): round to nearest, ties to even, and
 * saturate to +-448.  Normal binades [2^m, 2^(m+1)) for m >= -6 have spacing
 * 2^(m-3); below 2^-6 the subnormal spacing is 2^-9. */
double orc_e4m3_rne(double v) {
    if (isnan(v)) return v;
    double a = fabs(v);
    if (a == 0.0) return v;
    int ex;
    frexp(a, &ex);             /* a in [2^(ex-1), 2^ex) */
    int m = ex - 1;
    if (m < -6) m = -6;
    double step = ldexp(1.0, m - 3);
    double q = nearbyint(a / step) * step;   /* default rounding mode: ties to even */
    if (q > 448.0) q = 448.0;
    return copysign(q, v);
}

/* Shared exponent of one block: the smallest e with amax * 2^-e <= 448 (so no
 * element saturates), held to the e8m0 scale's range [-127, 127]; 0 for an
 * all-zero block. */
int orc_mx8_block_exponent(double amax) {
    if (!(amax > 0.0)) return 0;
    int e = (int)ceil(log2(amax / 448.0));
    while (ldexp(amax, -e) > 448.0) ++e;
    while (ldexp(amax, -(e - 1)) <= 448.0) --e;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* MXFP8 reading of a vector (n % 32 == 0): each block of 32 consecutive
 * elements shares 2^e (e from its largest |value|); out = e4m3(v 2^-e) 2^e. */
void orc_mx8_quantize(const double *v, int64_t n, double *out) {
    for (int64_t b = 0; b < n; b += 32) {
        double amax = 0.0;
        for (int i = 0; i < 32; ++i) amax = fmax(amax, fabs(v[b + i]));
        int e = orc_mx8_block_exponent(amax);
        for (int i = 0; i < 32; ++i) out[b + i] = ldexp(orc_e4m3_rne(ldexp(v[b + i], -e)), e);
    }
}

/* The expert FFN below, with the token rows (qx) and/or the gate/up output h
 * (qh) read as MXFP8 before the GEMM that consumes them. */
static void expert_ffn_impl(const uint8_t *w13_q, const uint8_t *w13_s, const uint8_t *w2_q,
                            const uint8_t *w2_s, int H, int I, const uint16_t *x, int n, uint16_t *y,
                            int qx, int qh);

void orc_expert_ffn(const uint8_t *w13_q, const uint8_t *w13_s, const uint8_t *w2_q,
                    const uint8_t *w2_s, int H, int I, const uint16_t *x, int n, uint16_t *y) {
    expert_ffn_impl(w13_q, w13_s, w2_q, w2_s, H, I, x, n, y, 0, 0);
}

void orc_expert_ffn_mx8(const uint8_t *w13_q, const uint8_t *w13_s, const uint8_t *w2_q,
                        const uint8_t *w2_s, int H, int I, const uint16_t *x, int n, uint16_t *y,
                        int qx, int qh) {
    expert_ffn_impl(w13_q, w13_s, w2_q, w2_s, H, I, x, n, y, qx, qh);
}

static void expert_ffn_impl(const uint8_t *w13_q, const uint8_t *w13_s, const uint8_t *w2_q,
                            const uint8_t *w2_s, int H, int I, const uint16_t *x, int n, uint16_t *y,
                            int qx, int qh) {
    double *xd = (double *)malloc(sizeof(double) * (size_t)n * H);
    float *h = (float *)malloc(sizeof(float) * (size_t)n * I);
    double *hd = (double *)malloc(sizeof(double) * (size_t)n * I);
    for (int64_t i = 0; i < (int64_t)n * H; ++i) xd[i] = (double)orc_bf16_to_f32(x[i]);
    if (qx)
        for (int t = 0; t < n; ++t) orc_mx8_quantize(xd + (int64_t)t * H, H, xd + (int64_t)t * H);

    /* gate/up: row i of W13 is the gate of unit i, row I+i its up projection */
#pragma omp parallel
    {
        double *wg = (double *)malloc(sizeof(double) * H);
        double *wu = (double *)malloc(sizeof(double) * H);
#pragma omp for schedule(static)
        for (int i = 0; i < I; ++i) {
            dequant_row(w13_q, w13_s, i, H, wg);
            dequant_row(w13_q, w13_s, (int64_t)I + i, H, wu);
            for (int t = 0; t < n; ++t) {
                double g = 0.0, u = 0.0;
                for (int c = 0; c < H; ++c) {
                    g += wg[c] * xd[(int64_t)t * H + c];
                    u += wu[c] * xd[(int64_t)t * H + c];
                }
                float gf = (float)g, uf = (float)u;
                h[(int64_t)t * I + i] = silu_f32(gf) * uf;
            }
        }
        free(wg);
        free(wu);
    }

    for (int64_t i = 0; i < (int64_t)n * I; ++i) hd[i] = (double)h[i];
    if (qh)
        for (int t = 0; t < n; ++t) orc_mx8_quantize(hd + (int64_t)t * I, I, hd + (int64_t)t * I);

    /* down: y_o = sum_i W2[o][i] h_i */
#pragma omp parallel
    {
        double *w2 = (double *)malloc(sizeof(double) * I);
#pragma omp for schedule(static)
        for (int o = 0; o < H; ++o) {
            dequant_row(w2_q, w2_s, o, I, w2);
            for (int t = 0; t < n; ++t) {
                double acc = 0.0;
                for (int i = 0; i < I; ++i) acc += w2[i] * hd[(int64_t)t * I + i];
                y[(int64_t)t * H + o] = orc_f32_to_bf16((float)acc);
            }
        }
        free(w2);
    }
    free(xd);
    free(h);
    free(hd);
}

/* ---------------------------------------------------------------- finalize */

void orc_finalize(const uint16_t *Y, const float *w, int T, int k, int H, uint16_t *out) {
    for (int t = 0; t < T; ++t) {
        for (int c = 0; c < H; ++c) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j)
                acc = fmaf(w[(int64_t)t * k + j], orc_bf16_to_f32(Y[((int64_t)t * k + j) * H + c]), acc);
            out[(int64_t)t * H + c] = orc_f32_to_bf16(acc);
        }
    }
}

/* -------------------------------------------------------------- layer step */

int64_t orc_expert_bytes(int H, int I) {
    int64_t n = 2LL * I * H + (int64_t)H * I;
    return n / 2 + n / 32;
}

static void expert_ptrs(const uint8_t *w13_q, const uint8_t *w13_s, const uint8_t *w2_q,
                        const uint8_t *w2_s, int H, int I, int e, const uint8_t **a,
                        const uint8_t **b, const uint8_t **c, const uint8_t **d) {
    *a = w13_q + (int64_t)e * 2 * I * (H / 2);
    *b = w13_s + (int64_t)e * 2 * I * (H / 32);
    *c = w2_q + (int64_t)e * H * (I / 2);
    *d = w2_s + (int64_t)e * H * (I / 32);
}

/* Evaluate expert rows for the listed slots: slots sharing an expert are
 * evaluated together (the per-token arithmetic does not depend on grouping). */
void orc_rows_for_slots(const uint8_t *w13_q, const uint8_t *w13_s, const uint8_t *w2_q,
                        const uint8_t *w2_s, int H, int I, int k, const int32_t *ids,
                        const uint16_t *x, const int32_t *slots, int n_slots,
                        uint16_t *Y_out) {
    orc_rows_for_slots_fmt(w13_q, w13_s, w2_q, w2_s, H, I, k, ids, x, slots, n_slots, Y_out, 0);
}

void orc_rows_for_slots_fmt(const uint8_t *w13_q, const uint8_t *w13_s, const uint8_t *w2_q,
                            const uint8_t *w2_s, int H, int I, int k, const int32_t *ids,
                            const uint16_t *x, const int32_t *slots, int n_slots,
                            uint16_t *Y_out, int mx8) {
    int *done = (int *)calloc((size_t)n_slots, sizeof(int));
    int *sel = (int *)malloc(sizeof(int) * (size_t)n_slots);
    uint16_t *xs = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)n_slots * H);
    uint16_t *ys = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)n_slots * H);
    for (int a = 0; a < n_slots; ++a) {
        if (done[a]) continue;
        int e = ids[slots[a]];
        int n = 0;
        for (int b = a; b < n_slots; ++b) {
            if (!done[b] && ids[slots[b]] == e) {
                sel[n] = b;
                memcpy(xs + (int64_t)n * H, x + (int64_t)(slots[b] / k) * H, sizeof(uint16_t) * H);
                ++n;
                done[b] = 1;
            }
        }
        const uint8_t *p13q, *p13s, *p2q, *p2s;
        expert_ptrs(w13_q, w13_s, w2_q, w2_s, H, I, e, &p13q, &p13s, &p2q, &p2s);
        expert_ffn_impl(p13q, p13s, p2q, p2s, H, I, xs, n, ys, mx8, mx8);
        for (int i = 0; i < n; ++i)
            memcpy(Y_out + (int64_t)sel[i] * H, ys + (int64_t)i * H, sizeof(uint16_t) * H);
    }
    free(done);
    free(sel);
    free(xs);
    free(ys);
}

void orc_layer_step(const uint8_t *w13_q, const uint8_t *w13_s, const uint8_t *w2_q,
                    const uint8_t *w2_s, int E, int k, int H, int I,
                    const float *logits, const uint16_t *x, int T,
                    int32_t *ids, float *w, uint16_t *Y, uint16_t *out,
                    int32_t *counts, int count_on, int count_tmax) {
    (void)E;
    orc_route(logits, T, E, k, ids, w);
    if (counts) orc_count(counts, E, ids, T, k, count_on, count_tmax);
    int P = T * k;
    int32_t *slots = (int32_t *)malloc(sizeof(int32_t) * (size_t)(P > 0 ? P : 1));
    for (int s = 0; s < P; ++s) slots[s] = s;
    orc_rows_for_slots(w13_q, w13_s, w2_q, w2_s, H, I, k, ids, x, slots, P, Y);
    free(slots);
    orc_finalize(Y, w, T, k, H, out);
}

/* ------------------------------------------------------------------- swaps */

int orc_swap(int32_t *row_map, int E, int n, const int32_t *promote, const int32_t *demote,
             int32_t *applied) {
    int done = 0;
    for (int i = 0; i < n; ++i) {
        int32_t c = promote[i], h = demote[i];
        int ok = c >= 0 && c < E && h >= 0 && h < E && c != h && row_map[c] < 0 && row_map[h] >= 0;
        if (ok) {
            int32_t hot_row = row_map[h];
            int32_t cold_code = row_map[c];
            row_map[c] = hot_row;
            row_map[h] = cold_code;
            ++done;
        }
        if (applied) applied[i] = ok;
    }
    return done;
}

/* ----------------------------------------------------------------- restore */

int orc_plan_restore(const int32_t *row_map, const int32_t *target, int E, int max_pairs,
                     int32_t *promote, int32_t *demote) {
    int hot_now = 0, hot_target = 0;
    for (int e = 0; e < E; ++e) {
        hot_now += row_map[e] >= 0;
        hot_target += target[e] >= 0;
    }
    if (hot_now != hot_target) return -1;
    /* the i-th expert to come in pairs with the i-th expert to go out */
    int n_in = 0, n_out = 0;
    for (int e = 0; e < E; ++e) {
        int was_hot = row_map[e] >= 0, want_hot = target[e] >= 0;
        if (!was_hot && want_hot && n_in < max_pairs) promote[n_in++] = e;
        if (was_hot && !want_hot && n_out < max_pairs) demote[n_out++] = e;
    }
    return n_in < n_out ? n_in : n_out;
}

/* ------------------------------------------------------------------ policy */

void orc_policy_init(orc_policy_t *p, int E, uint32_t *last, double *acc, const int32_t *counts) {
    p->E = E;
    p->last = last;
    p->acc = acc;
    p->wsum = 0.0;
    for (int e = 0; e < E; ++e) {
        last[e] = counts ? (uint32_t)counts[e] : 0u;
        acc[e] = 0.0;
    }
}

int orc_policy_read(orc_policy_t *p, const int32_t *counts, const int32_t *row_map,
                    double read_every, double half_life, double hysteresis, double min_avg,
                    int max_pairs, int32_t *promote, int32_t *demote) {
    int E = p->E;
    double d = pow(0.5, read_every / half_life);
    for (int e = 0; e < E; ++e) {
        uint32_t now = (uint32_t)counts[e];
        uint32_t delta = now - p->last[e];
        p->last[e] = now;
        p->acc[e] = d * p->acc[e] + (double)delta;
    }
    p->wsum = d * p->wsum + 1.0;

    /* cold candidates by average descending, hot by average ascending;
     * ties: lower expert id first.  Selection sort keeps it plain. */
    int *cold = (int *)malloc(sizeof(int) * E);
    int *hot = (int *)malloc(sizeof(int) * E);
    int nc = 0, nh = 0;
    for (int e = 0; e < E; ++e) {
        if (row_map[e] < 0) {
            if (p->acc[e] / p->wsum >= min_avg) cold[nc++] = e;
        } else {
            hot[nh++] = e;
        }
    }
    for (int a = 0; a < nc; ++a) {
        int best = a;
        for (int b = a + 1; b < nc; ++b) {
            double vb = p->acc[cold[b]] / p->wsum, vbest = p->acc[cold[best]] / p->wsum;
            if (vb > vbest || (vb == vbest && cold[b] < cold[best])) best = b;
        }
        int t = cold[a]; cold[a] = cold[best]; cold[best] = t;
    }
    for (int a = 0; a < nh; ++a) {
        int best = a;
        for (int b = a + 1; b < nh; ++b) {
            double vb = p->acc[hot[b]] / p->wsum, vbest = p->acc[hot[best]] / p->wsum;
            if (vb < vbest || (vb == vbest && hot[b] < hot[best])) best = b;
        }
        int t = hot[a]; hot[a] = hot[best]; hot[best] = t;
    }
    int n = 0;
    while (n < max_pairs && n < nc && n < nh) {
        double vc = p->acc[cold[n]] / p->wsum, vh = p->acc[hot[n]] / p->wsum;
        if (!(vc > hysteresis * vh)) break;
        promote[n] = cold[n];
        demote[n] = hot[n];
        ++n;
    }
    free(cold);
    free(hot);
    return n;
}

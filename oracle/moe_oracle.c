/*
 * CPU oracle of the routed-expert FFN of one MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file: it is used by tests/, by the smoke check and by the CPU baseline
 * leg of bench.py. It shares no code with the CUDA library (no headers, no
 * helpers, no tables); the two meet only in the input bytes.
 *
 * Plain, single-threaded, float64. Each function follows a passage of the
 * Strata pages (cited by page title and section) and, where the pages are
 * silent, the plainest reading of them:
 *
 *  - routing trace = k expert ids + k weights per token and layer
 *    ("extended-strata-moe reference", section "Routing trace format");
 *    top-10 of 512 experts (SGLang port post, header);
 *  - only the rows routed to an expert are computed ("expert-scoped layout",
 *    SGLang port post, section 2);
 *  - per expert: dequant -> gate/up -> SwiGLU -> down -> weighted scatter
 *    (the grouped expert kernel, SGLang port post, TL;DR and section 3);
 *  - the shared expert is applied to every row with weight 1
 *    (Strata BATCHING, "Several requests at once");
 *  - an expert-cache slot map says which experts are resident; the others are
 *    reported, counted as distinct experts per layer
 *    ("extended-strata-moe reference", sections "The mailbox" and "C API").
 *
 * Readings of silent points (all listed in the design notes):
 *  - top-k order: logit descending, ties to the lower expert id;
 *  - weights: softmax over the k selected logits (renormalised top-k),
 *    computed in float64 and rounded once to fp32;
 *  - permutation order inside an expert: pair index p = t*k + j ascending;
 *  - SwiGLU: h = silu(g) * u with silu(z) = z / (1 + exp(-z)); no gate on the
 *    shared expert; intermediates kept in float64.
 *
 * Build: gcc -O2 -ffp-contract=off -shared -fPIC moe_oracle.c -lm
 * (-ffp-contract=off keeps a*b+c unfused so results match across x86 and Arm).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* number formats                                                           */
/* ------------------------------------------------------------------------ */

/* IEEE 754 binary16 bit pattern -> double (exact). */
double orc_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 0x1F;
    int man = h & 0x3FF;
    double v;
    if (ex == 0)
        v = ldexp((double)man, -24);             /* subnormal: man * 2^-24 */
    else if (ex == 31)
        v = man ? NAN : INFINITY;
    else
        v = ldexp((double)(man | 0x400), ex - 25); /* (1024 + man) * 2^(e-15-10) */
    return sign ? -v : v;
}

/* bfloat16 bit pattern -> double (exact): the top half of an fp32. */
double orc_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* One stored weight of a block-quantised matrix with K columns:
 * code nibble n of column c (even column = low nibble), value n - 16*(n>=8),
 * times the fp16 scale of block c/32. */
double orc_weight(const uint8_t *q, const uint16_t *scale, int K, int r, int c)
{
    uint8_t byte = q[(size_t)r * (size_t)(K / 2) + (size_t)(c / 2)];
    int n = (byte >> (4 * (c & 1))) & 0xF;
    int v = n - 16 * (n >> 3);
    double s = orc_half_to_double(scale[(size_t)r * (size_t)(K / 32) + (size_t)(c / 32)]);
    return s * (double)v;
}

/* ------------------------------------------------------------------------ */
/* router                                                                   */
/* ------------------------------------------------------------------------ */

/* Tiny-case router: logits[t][e] = fp32( sum_h x[t][h] * Wg[h][e] ), summed in
 * h order in double and rounded once. */
void orc_router_logits(const float *x, const float *wg, int T, int H, int E, float *logits)
{
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            double s = 0.0;
            for (int h = 0; h < H; ++h)
                s += (double)x[(size_t)t * H + h] * (double)wg[(size_t)h * E + e];
            logits[(size_t)t * E + e] = (float)s;
        }
}

/* Top-k selection and renormalised softmax weights, row by row.
 * Selection: k passes, each taking the largest logit not yet taken; a strict
 * '>' while scanning ids upward keeps the lower id on ties.
 * Weights: m = logit of the first pick, e_j = exp(l_j - m), s = sum_j e_j in
 * j order, w_j = e_j / s rounded once to fp32 (w_exact keeps the double).
 * Returns 0, or 1 + the first row holding a non-finite logit. */
int orc_route(const float *logits, int T, int E, int k, int32_t *ids, float *w, double *w_exact)
{
    unsigned char *taken = (unsigned char *)malloc((size_t)E);
    double *ej = (double *)malloc(sizeof(double) * (size_t)k);
    int rc = 0;
    for (int t = 0; t < T && rc == 0; ++t) {
        const float *l = logits + (size_t)t * E;
        for (int e = 0; e < E; ++e)
            if (!isfinite(l[e])) { rc = t + 1; break; }
        if (rc) break;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || l[e] > l[best]))
                    best = e;
            taken[best] = 1;
            ids[(size_t)t * k + j] = best;
        }
        double m = (double)l[ids[(size_t)t * k]];
        double s = 0.0;
        for (int j = 0; j < k; ++j) {
            ej[j] = exp((double)l[ids[(size_t)t * k + j]] - m);
            s += ej[j];
        }
        for (int j = 0; j < k; ++j) {
            double v = ej[j] / s;
            w[(size_t)t * k + j] = (float)v;
            if (w_exact) w_exact[(size_t)t * k + j] = v;
        }
    }
    free(taken);
    free(ej);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* permutation                                                              */
/* ------------------------------------------------------------------------ */

/* Counting sort of the P = T*k (token, expert) pairs by expert.
 *  offsets[e]          first sorted position of expert e (offsets[E] = P)
 *  sorted_pair[pos]    pair p = t*k + j at sorted position pos (p ascending per expert)
 *  pair_pos[p]         inverse of sorted_pair
 *  miss_ids[0..n)      distinct touched experts with slot_map[e] < 0, ascending
 * slot_map may be NULL (every expert resident). Returns 0, or -1 on a bad id. */
int orc_permute(const int32_t *ids, int T, int E, int k, const int32_t *slot_map,
                int32_t *offsets, int32_t *sorted_pair, int32_t *pair_pos,
                int32_t *miss_ids, int32_t *n_miss)
{
    int P = T * k;
    int32_t *count = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int p = 0; p < P; ++p) {
        if (ids[p] < 0 || ids[p] >= E) { free(count); free(fill); return -1; }
        count[ids[p]] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + count[e];
    for (int p = 0; p < P; ++p) {
        int e = ids[p];
        int pos = offsets[e] + fill[e];
        fill[e] += 1;
        sorted_pair[pos] = p;
        pair_pos[p] = pos;
    }
    int nm = 0;
    for (int e = 0; e < E; ++e)
        if (count[e] > 0 && slot_map && slot_map[e] < 0)
            miss_ids[nm++] = e;
    *n_miss = nm;
    free(count);
    free(fill);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* expert FFN                                                               */
/* ------------------------------------------------------------------------ */

typedef struct {
    int32_t H, I, E, k, S, shared_I;
    const uint8_t *gate_q, *up_q, *down_q;      /* [S][I][H/2], [S][I][H/2], [S][H][I/2] */
    const uint16_t *gate_s, *up_s, *down_s;     /* [S][I][H/32], [S][I][H/32], [S][H][I/32] */
    const uint8_t *sh_gate_q, *sh_up_q, *sh_down_q;   /* shared expert, intermediate shared_I */
    const uint16_t *sh_gate_s, *sh_up_s, *sh_down_s;
} orc_layer;

static double orc_silu(double z) { return z / (1.0 + exp(-z)); }

/* One expert on one row: g = Wg x, u = Wu x, h = silu(g) u, o = Wd h. */
static void orc_expert_row(const uint8_t *gq, const uint16_t *gs,
                           const uint8_t *uq, const uint16_t *us,
                           const uint8_t *dq, const uint16_t *ds,
                           int H, int inter, const double *x, double *hbuf, double *o)
{
    for (int i = 0; i < inter; ++i) {
        double g = 0.0, u = 0.0;
        for (int c = 0; c < H; ++c) {
            g += orc_weight(gq, gs, H, i, c) * x[c];
            u += orc_weight(uq, us, H, i, c) * x[c];
        }
        hbuf[i] = orc_silu(g) * u;
    }
    for (int r = 0; r < H; ++r) {
        double acc = 0.0;
        for (int i = 0; i < inter; ++i)
            acc += orc_weight(dq, ds, inter, r, i) * hbuf[i];
        o[r] = acc;
    }
}

/* The activations of row t as doubles (x_is_bf16: bit patterns; else fp32). */
static void orc_load_row(const void *x, int x_is_bf16, int H, int t, double *out)
{
    for (int c = 0; c < H; ++c)
        out[c] = x_is_bf16 ? orc_bf16_to_double(((const uint16_t *)x)[(size_t)t * H + c])
                           : (double)((const float *)x)[(size_t)t * H + c];
}

/* Intermediate activations h (length I) of one (row, expert slot), for tests of
 * the gate/up stage alone. */
void orc_expert_h(const orc_layer *L, const void *x, int x_is_bf16, int t, int slot, double *h)
{
    int H = L->H, I = L->I;
    double *xd = (double *)malloc(sizeof(double) * (size_t)H);
    orc_load_row(x, x_is_bf16, H, t, xd);
    size_t gstride = (size_t)I * (size_t)(H / 2), sstride = (size_t)I * (size_t)(H / 32);
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int c = 0; c < H; ++c) {
            g += orc_weight(L->gate_q + slot * gstride, L->gate_s + slot * sstride, H, i, c) * xd[c];
            u += orc_weight(L->up_q + slot * gstride, L->up_s + slot * sstride, H, i, c) * xd[c];
        }
        h[i] = orc_silu(g) * u;
    }
    free(xd);
}

/* Layer output for the listed rows:
 *   y[t] = sum_{j=0}^{k-1} [slot(e_tj) >= 0] * w_tj * FFN_{e_tj}(x_t)  +  FFN_shared(x_t)
 * in double. slot_map NULL = expert e lives in slot e. Returns 0, or -1 on a
 * slot out of range. */
int orc_layer_rows(const orc_layer *L, const void *x, int x_is_bf16,
                   const int32_t *ids, const float *w, const int32_t *slot_map,
                   int n_rows, const int32_t *rows, double *y)
{
    int H = L->H, I = L->I, k = L->k;
    int Imax = L->shared_I > I ? L->shared_I : I;
    double *xd = (double *)malloc(sizeof(double) * (size_t)H);
    double *o = (double *)malloc(sizeof(double) * (size_t)H);
    double *hb = (double *)malloc(sizeof(double) * (size_t)Imax);
    size_t gq = (size_t)I * (size_t)(H / 2), gs = (size_t)I * (size_t)(H / 32);
    size_t dqs = (size_t)H * (size_t)(I / 2), dss = (size_t)H * (size_t)(I / 32);
    int rc = 0;
    for (int r = 0; r < n_rows && rc == 0; ++r) {
        int t = rows[r];
        double *yt = y + (size_t)r * H;
        for (int c = 0; c < H; ++c) yt[c] = 0.0;
        orc_load_row(x, x_is_bf16, H, t, xd);
        for (int j = 0; j < k; ++j) {
            int e = ids[(size_t)t * k + j];
            int slot = slot_map ? slot_map[e] : e;
            if (slot < 0) continue;               /* not resident: reported, not computed */
            if (slot >= L->S) { rc = -1; break; }
            orc_expert_row(L->gate_q + slot * gq, L->gate_s + slot * gs,
                           L->up_q + slot * gq, L->up_s + slot * gs,
                           L->down_q + slot * dqs, L->down_s + slot * dss,
                           H, I, xd, hb, o);
            double wj = (double)w[(size_t)t * k + j];
            for (int c = 0; c < H; ++c) yt[c] += wj * o[c];
        }
        if (rc == 0 && L->shared_I > 0) {
            orc_expert_row(L->sh_gate_q, L->sh_gate_s, L->sh_up_q, L->sh_up_s,
                           L->sh_down_q, L->sh_down_s, H, L->shared_I, xd, hb, o);
            for (int c = 0; c < H; ++c) yt[c] += o[c];
        }
    }
    free(xd);
    free(o);
    free(hb);
    return rc;
}

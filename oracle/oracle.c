/*
 * oracle.c -- plain, slow, CPU reference decoder for the paged-KV decode step.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference arm may load this library. The product path
 * (persistent_megakernel_05_b300) never calls it and shares no code with it.
 *
 * What it computes (the plainest reading of the pages; the pages print no
 * equations):
 *   "Cohere Megakernel" page, section "Megakernel ne demek": one decode step of a
 *     transformer LM = the whole forward pass for one new token per sequence.
 *   same page, section "Sinirlar acikca yazilmis": BF16 weights only, batch 1..8,
 *     paged KV cache, sliding-window attention, prefix cache, ragged lengths,
 *     continuous batching, greedy sampling.
 *   "Kog Inference Engine" page, section on memory bandwidth: every active weight
 *     crosses memory once per token (decode is a chain of matrix-vector products).
 *   The model: pre-norm decoder. x = E[tok]; per layer x += Attn(RMSNorm(x)),
 *   x += MLP(RMSNorm(x)) with MLP = SwiGLU or softmax-top-k MoE; final RMSNorm,
 *   untied LM head, greedy argmax (lowest index on ties).
 *
 * Precision: weights and the KV cache are BF16 values, upcast exactly to fp32.
 * All arithmetic is fp32 (products rounded, then summed, in natural index order;
 * built with -ffp-contract=off). RoPE angles are computed in double and rounded to
 * fp32. New K/V rows are rounded to BF16 (round-to-nearest-even) when written to
 * the cache and are read back from it, exactly like every older row.
 *
 * Parity pins (tests/test_oracle_pins.py): closed forms for RMSNorm and RoPE,
 * attention special cases (single key, uniform scores, one-hot), agreement with an
 * independent float64 NumPy twin and with torch library routines (rms_norm,
 * scaled_dot_product_attention with GQA, silu), cached decode == full recompute,
 * paged == contiguous, page-permutation invariance, MoE reductions, argmax ties,
 * Philox4x32-10 known-answer vectors, Gumbel-max sample frequencies = softmax(z / T).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_OK 0
#define OR_ERR_ARG 1
#define OR_ERR_PAGE 5

typedef struct or_model {
    int32_t n_layers, d_model, n_q_heads, n_kv_heads, head_dim, ffn_dim, vocab;
    int32_t n_experts, top_k, expert_ffn_dim;
    float rms_eps, rope_theta;
    int32_t sliding_window;
    const uint8_t *layer_is_sliding; /* [n_layers] or NULL */
    int32_t page_size;
    const uint16_t *embed, *final_norm, *lm_head;
    /* arrays of n_layers pointers */
    const uint16_t *const *attn_norm, *const *wq, *const *wk, *const *wv, *const *wo;
    const uint16_t *const *mlp_norm, *const *w_gate, *const *w_up, *const *w_down;
    const uint16_t *const *router, *const *exp_gate, *const *exp_up, *const *exp_down;
} or_model;

/* ---------- BF16 <-> fp32 (bit-level definitions) ---------- */

float or_bf16_to_f32(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

uint16_t or_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) /* NaN stays NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u; /* round to nearest, ties to even */
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* ---------- building blocks (each exported for the unit pins) ---------- */

/* RMSNorm: out[i] = x[i] / sqrt(mean(x^2) + eps) * g[i], fp32. */
void or_rmsnorm(const float *x, const uint16_t *g, int32_t n, float eps, float *out) {
    float ss = 0.0f;
    for (int32_t i = 0; i < n; i++) ss += x[i] * x[i];
    float r = 1.0f / sqrtf(ss / (float)n + eps);
    for (int32_t i = 0; i < n; i++) out[i] = (x[i] * r) * or_bf16_to_f32(g[i]);
}

/* y[r] = sum_k W[r][k] * x[k] for r in [0, rows), W BF16 [rows][cols] row-major. */
static void matvec(const uint16_t *W, const float *x, int32_t rows, int32_t cols, float *y,
                   int32_t nthreads) {
#pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int32_t r = 0; r < rows; r++) {
        const uint16_t *w = W + (int64_t)r * cols;
        float acc = 0.0f;
        for (int32_t k = 0; k < cols; k++) acc += or_bf16_to_f32(w[k]) * x[k];
        y[r] = acc;
    }
}

void or_matvec(const uint16_t *W, const float *x, int32_t rows, int32_t cols, float *y) {
    matvec(W, x, rows, cols, y, 1);
}

/* Rotate-half RoPE on one head vector v[hd] at absolute position pos:
 * pairs (i, i + hd/2), inv_freq_i = theta^(-2i/hd), angle = pos * inv_freq_i. */
void or_rope(float *v, int32_t hd, int32_t pos, float theta) {
    int32_t half = hd / 2;
    for (int32_t i = 0; i < half; i++) {
        double inv_freq = pow((double)theta, -2.0 * (double)i / (double)hd);
        double ang = (double)pos * inv_freq;
        float c = (float)cos(ang), s = (float)sin(ang);
        float a = v[i], b = v[i + half];
        v[i] = a * c - b * s;
        v[i + half] = b * c + a * s;
    }
}

/* One query head over n keys: out = sum_j softmax_j(q.k_j / sqrt(hd)) v_j. */
void or_attend(const float *q, const float *K, const float *V, int32_t n, int32_t hd,
               float *out) {
    float *s = (float *)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
    float scale = 1.0f / sqrtf((float)hd);
    float m = -INFINITY;
    for (int32_t j = 0; j < n; j++) {
        float dot = 0.0f;
        for (int32_t d = 0; d < hd; d++) dot += q[d] * K[(int64_t)j * hd + d];
        s[j] = dot * scale;
        if (s[j] > m) m = s[j];
    }
    float z = 0.0f;
    for (int32_t j = 0; j < n; j++) {
        s[j] = expf(s[j] - m);
        z += s[j];
    }
    for (int32_t d = 0; d < hd; d++) {
        float acc = 0.0f;
        for (int32_t j = 0; j < n; j++) acc += s[j] * V[(int64_t)j * hd + d];
        out[d] = acc / z;
    }
    free(s);
}

static float silu(float z) { return z / (1.0f + expf(-z)); }

/* Softmax over all E router logits, then the top-k (ties -> lower index), then the
 * k selected probabilities renormalised to sum to 1. ids[] ascending by rank. */
void or_route(const float *logits, int32_t E, int32_t k, int32_t *ids, float *w) {
    float m = -INFINITY;
    for (int32_t e = 0; e < E; e++)
        if (logits[e] > m) m = logits[e];
    float *p = (float *)malloc(sizeof(float) * (size_t)E);
    unsigned char *taken = (unsigned char *)calloc((size_t)E, 1);
    float z = 0.0f;
    for (int32_t e = 0; e < E; e++) {
        p[e] = expf(logits[e] - m);
        z += p[e];
    }
    for (int32_t e = 0; e < E; e++) p[e] = p[e] / z;
    float sel = 0.0f;
    for (int32_t i = 0; i < k; i++) {
        int32_t best = -1;
        for (int32_t e = 0; e < E; e++)
            if (!taken[e] && (best < 0 || p[e] > p[best])) best = e;
        taken[best] = 1;
        ids[i] = best;
        w[i] = p[best];
        sel += p[best];
    }
    for (int32_t i = 0; i < k; i++) w[i] = w[i] / sel;
    free(p);
    free(taken);
}

/* ---------- temperature sampling (Gumbel-max over a counter-based generator) ----------
 * Sampling from softmax(logits / T) equals taking argmax_i (logits_i / T + g_i) with g_i
 * independent standard Gumbel draws, g = -log(-log u), u uniform on (0, 1). The draws
 * come from Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
 * as 1, 2, 3", SC 2011), keyed by the 64-bit seed, with counter (token id, position,
 * batch row, 0): no state, so the kernel and this oracle draw the same u for the same
 * (seed, position, row, token). u = (top 24 bits of word 0 + 0.5) / 2^24, in fp32. */
void or_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; r++) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0, p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

float or_gumbel(uint64_t seed, int32_t token, int32_t pos, int32_t row) {
    const uint32_t ctr[4] = {(uint32_t)token, (uint32_t)pos, (uint32_t)row, 0u};
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t o[4];
    or_philox4x32_10(ctr, key, o);
    const float u = ((float)(o[0] >> 8) + 0.5f) * (1.0f / 16777216.0f);
    return -logf(-logf(u));
}

/* z_i = logits_i / T + g_i for every token i */
void or_gumbel_scores(const float *logits, int32_t n, float temperature, uint64_t seed, int32_t pos,
                      int32_t row, float *z) {
    for (int32_t i = 0; i < n; i++) z[i] = logits[i] / temperature + or_gumbel(seed, i, pos, row);
}

/* index of the largest logits_i / T + g_i (lowest index on ties) */
int32_t or_sample_gumbel(const float *logits, int32_t n, float temperature, uint64_t seed, int32_t pos,
                         int32_t row) {
    int32_t best = 0;
    float bv = -INFINITY;
    for (int32_t i = 0; i < n; i++) {
        const float z = logits[i] / temperature + or_gumbel(seed, i, pos, row);
        if (z > bv) { bv = z; best = i; }
    }
    return best;
}

/* Temperature sampling limited to the top_k largest logits (1 <= top_k <= n): the
 * candidate set is the top_k tokens in the order (larger logit first, lower index first
 * among equal logits); the draw is the candidate with the largest logits_i / T + g_i,
 * the lowest index among equal scores -- a draw from softmax(logits / T) renormalised
 * over the candidates (Gumbel-max restricted to a subset). Selection: a candidate is a
 * token with fewer than top_k tokens ahead of it in that order (a count, O(n^2) in the
 * worst case but fine for the sizes the tests use; tokens below the top_k-th largest
 * logit are rejected first). */
int32_t or_sample_gumbel_topk(const float *logits, int32_t n, float temperature, int32_t top_k,
                              uint64_t seed, int32_t pos, int32_t row) {
    if (top_k < 1 || top_k >= n) return or_sample_gumbel(logits, n, temperature, seed, pos, row);
    /* the top_k-th largest logit value (a lower bound for every candidate) */
    float *tmp = (float *)malloc(sizeof(float) * (size_t)n);
    if (!tmp) return -1;
    memcpy(tmp, logits, sizeof(float) * (size_t)n);
    for (int32_t k = 0; k < top_k; k++) {  /* partial selection sort, descending */
        int32_t best = k;
        for (int32_t i = k + 1; i < n; i++)
            if (tmp[i] > tmp[best]) best = i;
        const float t = tmp[k]; tmp[k] = tmp[best]; tmp[best] = t;
    }
    const float kth = tmp[top_k - 1];
    free(tmp);
    int32_t best = -1;
    float bv = -INFINITY;
    for (int32_t i = 0; i < n; i++) {
        if (logits[i] < kth) continue;
        int32_t ahead = 0;  /* tokens before i in (logit desc, index asc) order */
        for (int32_t j = 0; j < n && ahead < top_k; j++)
            if (logits[j] > logits[i] || (logits[j] == logits[i] && j < i)) ahead++;
        if (ahead >= top_k) continue;
        const float z = logits[i] / temperature + or_gumbel(seed, i, pos, row);
        if (best < 0 || z > bv) { bv = z; best = i; }
    }
    return best;
}

/* Greedy: index of the largest value, the lowest index among equal maxima. */
int32_t or_argmax(const float *v, int32_t n) {
    int32_t best = 0;
    for (int32_t i = 1; i < n; i++)
        if (v[i] > v[best]) best = i;
    return best;
}

/* ---------- paged KV addressing (the oracle's own index code) ---------- */

/* Element (layer l, page p, K or V, kv head g, slot s, dim d) of the pool
 * [n_layers][num_pages][2][n_kv_heads][page_size][head_dim]. */
static int64_t kv_index(const or_model *m, int32_t num_pages, int32_t l, int32_t p, int32_t kv,
                        int32_t g, int32_t s, int32_t d) {
    int64_t i = l;
    i = i * num_pages + p;
    i = i * 2 + kv;
    i = i * m->n_kv_heads + g;
    i = i * m->page_size + s;
    i = i * m->head_dim + d;
    return i;
}

static int layer_slides(const or_model *m, int32_t l) {
    return m->sliding_window > 0 && m->layer_is_sliding && m->layer_is_sliding[l];
}

/* MLP of one layer on xn -> adds into x. */
static void mlp_add(const or_model *m, int32_t l, const float *xn, float *x, int32_t nthreads) {
    int32_t d = m->d_model;
    if (m->n_experts == 0) {
        int32_t F = m->ffn_dim;
        float *g = (float *)malloc(sizeof(float) * (size_t)F);
        float *u = (float *)malloc(sizeof(float) * (size_t)F);
        float *y = (float *)malloc(sizeof(float) * (size_t)d);
        matvec(m->w_gate[l], xn, F, d, g, nthreads);
        matvec(m->w_up[l], xn, F, d, u, nthreads);
        for (int32_t i = 0; i < F; i++) g[i] = silu(g[i]) * u[i];
        matvec(m->w_down[l], g, d, F, y, nthreads);
        for (int32_t i = 0; i < d; i++) x[i] += y[i];
        free(g);
        free(u);
        free(y);
        return;
    }
    int32_t E = m->n_experts, k = m->top_k, Fe = m->expert_ffn_dim;
    float *r = (float *)malloc(sizeof(float) * (size_t)E);
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
    float *w = (float *)malloc(sizeof(float) * (size_t)k);
    float *g = (float *)malloc(sizeof(float) * (size_t)Fe);
    float *u = (float *)malloc(sizeof(float) * (size_t)Fe);
    float *y = (float *)malloc(sizeof(float) * (size_t)d);
    float *acc = (float *)calloc((size_t)d, sizeof(float));
    matvec(m->router[l], xn, E, d, r, nthreads);
    or_route(r, E, k, ids, w);
    /* sum over the selected experts in ascending expert id */
    for (int32_t e = 0; e < E; e++) {
        int32_t slot = -1;
        for (int32_t i = 0; i < k; i++)
            if (ids[i] == e) slot = i;
        if (slot < 0) continue;
        const uint16_t *Wg = m->exp_gate[l] + (int64_t)e * Fe * d;
        const uint16_t *Wu = m->exp_up[l] + (int64_t)e * Fe * d;
        const uint16_t *Wd = m->exp_down[l] + (int64_t)e * d * Fe;
        matvec(Wg, xn, Fe, d, g, nthreads);
        matvec(Wu, xn, Fe, d, u, nthreads);
        for (int32_t i = 0; i < Fe; i++) g[i] = silu(g[i]) * u[i];
        matvec(Wd, g, d, Fe, y, nthreads);
        for (int32_t i = 0; i < d; i++) acc[i] += w[slot] * y[i];
    }
    for (int32_t i = 0; i < d; i++) x[i] += acc[i];
    free(r); free(ids); free(w); free(g); free(u); free(y); free(acc);
}

/* ---------- one decode step over the paged cache ---------- */

int or_decode_step(const or_model *m, uint16_t *kv, int32_t num_pages, const int32_t *tokens,
                   const int32_t *positions, const int32_t *page_table, int32_t max_pages,
                   const int32_t *seq_lens, int32_t batch, float *logits, int32_t *next_tokens,
                   int32_t nthreads) {
    if (!m || !kv || !tokens || !positions || !page_table || !seq_lens || batch <= 0)
        return OR_ERR_ARG;
    if (nthreads <= 0) nthreads = 1;
    const int32_t d = m->d_model, Hq = m->n_q_heads, Hkv = m->n_kv_heads, hd = m->head_dim;
    const int32_t G = Hq / Hkv, ps = m->page_size, V = m->vocab;
    float *x = (float *)malloc(sizeof(float) * (size_t)d);
    float *xn = (float *)malloc(sizeof(float) * (size_t)d);
    float *q = (float *)malloc(sizeof(float) * (size_t)Hq * hd);
    float *kk = (float *)malloc(sizeof(float) * (size_t)Hkv * hd);
    float *vv = (float *)malloc(sizeof(float) * (size_t)Hkv * hd);
    float *o = (float *)malloc(sizeof(float) * (size_t)Hq * hd);
    float *y = (float *)malloc(sizeof(float) * (size_t)d);
    float *lg = (float *)malloc(sizeof(float) * (size_t)V);
    int rc = OR_OK;

    for (int32_t b = 0; b < batch && rc == OR_OK; b++) {
        const int32_t tok = tokens[b], pos = positions[b];
        const int32_t *pt = page_table + (int64_t)b * max_pages;
        if (tok < 0 || tok >= V || pos < 0 || seq_lens[b] != pos + 1 || pos / ps >= max_pages) {
            rc = OR_ERR_ARG;
            break;
        }
        for (int32_t i = 0; i < d; i++) x[i] = or_bf16_to_f32(m->embed[(int64_t)tok * d + i]);

        for (int32_t l = 0; l < m->n_layers && rc == OR_OK; l++) {
            or_rmsnorm(x, m->attn_norm[l], d, m->rms_eps, xn);
            matvec(m->wq[l], xn, Hq * hd, d, q, nthreads);
            matvec(m->wk[l], xn, Hkv * hd, d, kk, nthreads);
            matvec(m->wv[l], xn, Hkv * hd, d, vv, nthreads);
            for (int32_t h = 0; h < Hq; h++) or_rope(q + h * hd, hd, pos, m->rope_theta);
            for (int32_t g = 0; g < Hkv; g++) or_rope(kk + g * hd, hd, pos, m->rope_theta);

            /* append: BF16-rounded K and V at (page of pos, slot pos % ps) */
            const int32_t page = pt[pos / ps];
            if (page < 0 || page >= num_pages) {
                rc = OR_ERR_PAGE;
                break;
            }
            for (int32_t g = 0; g < Hkv; g++)
                for (int32_t dd = 0; dd < hd; dd++) {
                    kv[kv_index(m, num_pages, l, page, 0, g, pos % ps, dd)] =
                        or_f32_to_bf16(kk[g * hd + dd]);
                    kv[kv_index(m, num_pages, l, page, 1, g, pos % ps, dd)] =
                        or_f32_to_bf16(vv[g * hd + dd]);
                }

            /* keys j with lo <= j <= pos (a sliding layer keeps exactly W keys) */
            const int32_t lo = layer_slides(m, l) ? (pos - m->sliding_window + 1 > 0
                                                         ? pos - m->sliding_window + 1 : 0)
                                                  : 0;
            const int32_t n = pos - lo + 1;
            for (int32_t i = lo / ps; i <= pos / ps; i++)
                if (pt[i] < 0 || pt[i] >= num_pages) rc = OR_ERR_PAGE;
            if (rc != OR_OK) break;
#pragma omp parallel for num_threads(nthreads) schedule(static)
            for (int32_t h = 0; h < Hq; h++) {
                const int32_t g = h / G; /* GQA: query head h reads kv head h / G */
                float *K = (float *)malloc(sizeof(float) * (size_t)n * hd);
                float *Vv = (float *)malloc(sizeof(float) * (size_t)n * hd);
                for (int32_t j = lo; j <= pos; j++) {
                    const int32_t pg = pt[j / ps], s = j % ps;
                    for (int32_t dd = 0; dd < hd; dd++) {
                        K[(int64_t)(j - lo) * hd + dd] =
                            or_bf16_to_f32(kv[kv_index(m, num_pages, l, pg, 0, g, s, dd)]);
                        Vv[(int64_t)(j - lo) * hd + dd] =
                            or_bf16_to_f32(kv[kv_index(m, num_pages, l, pg, 1, g, s, dd)]);
                    }
                }
                or_attend(q + h * hd, K, Vv, n, hd, o + h * hd);
                free(K);
                free(Vv);
            }
            matvec(m->wo[l], o, d, Hq * hd, y, nthreads);
            for (int32_t i = 0; i < d; i++) x[i] += y[i];

            or_rmsnorm(x, m->mlp_norm[l], d, m->rms_eps, xn);
            mlp_add(m, l, xn, x, nthreads);
        }
        if (rc != OR_OK) break;
        or_rmsnorm(x, m->final_norm, d, m->rms_eps, xn);
        matvec(m->lm_head, xn, V, d, lg, nthreads);
        if (logits) memcpy(logits + (int64_t)b * V, lg, sizeof(float) * (size_t)V);
        if (next_tokens) next_tokens[b] = or_argmax(lg, V);
    }
    free(x); free(xn); free(q); free(kk); free(vv); free(o); free(y); free(lg);
    return rc;
}

/* ---------- full causal recompute without any cache (for the cache pins) ----------
 * Runs the whole model over tokens[0..T) at positions 0..T-1, layer by layer, keeping
 * all K/V rows in plain arrays (BF16-rounded, as a cache would store them).
 * logits: [T][vocab]. */
int or_forward_full(const or_model *m, const int32_t *tokens, int32_t T, float *logits,
                    int32_t nthreads) {
    if (!m || !tokens || T <= 0 || !logits) return OR_ERR_ARG;
    if (nthreads <= 0) nthreads = 1;
    const int32_t d = m->d_model, Hq = m->n_q_heads, Hkv = m->n_kv_heads, hd = m->head_dim;
    const int32_t G = Hq / Hkv, V = m->vocab;
    for (int32_t t = 0; t < T; t++)
        if (tokens[t] < 0 || tokens[t] >= V) return OR_ERR_ARG;
    float *X = (float *)malloc(sizeof(float) * (size_t)T * d);
    float *xn = (float *)malloc(sizeof(float) * (size_t)d);
    float *Q = (float *)malloc(sizeof(float) * (size_t)T * Hq * hd);
    float *K = (float *)malloc(sizeof(float) * (size_t)T * Hkv * hd);
    float *Vv = (float *)malloc(sizeof(float) * (size_t)T * Hkv * hd);
    float *o = (float *)malloc(sizeof(float) * (size_t)Hq * hd);
    float *y = (float *)malloc(sizeof(float) * (size_t)d);
    float *Kh = (float *)malloc(sizeof(float) * (size_t)T * hd);
    float *Vh = (float *)malloc(sizeof(float) * (size_t)T * hd);
    for (int32_t t = 0; t < T; t++) {
        for (int32_t i = 0; i < d; i++)
            X[(int64_t)t * d + i] = or_bf16_to_f32(m->embed[(int64_t)tokens[t] * d + i]);
    }
    for (int32_t l = 0; l < m->n_layers; l++) {
        for (int32_t t = 0; t < T; t++) {
            or_rmsnorm(X + (int64_t)t * d, m->attn_norm[l], d, m->rms_eps, xn);
            matvec(m->wq[l], xn, Hq * hd, d, Q + (int64_t)t * Hq * hd, nthreads);
            matvec(m->wk[l], xn, Hkv * hd, d, K + (int64_t)t * Hkv * hd, nthreads);
            matvec(m->wv[l], xn, Hkv * hd, d, Vv + (int64_t)t * Hkv * hd, nthreads);
            for (int32_t h = 0; h < Hq; h++) or_rope(Q + ((int64_t)t * Hq + h) * hd, hd, t, m->rope_theta);
            for (int32_t g = 0; g < Hkv; g++) or_rope(K + ((int64_t)t * Hkv + g) * hd, hd, t, m->rope_theta);
            for (int32_t i = 0; i < Hkv * hd; i++) {
                K[(int64_t)t * Hkv * hd + i] = or_bf16_to_f32(or_f32_to_bf16(K[(int64_t)t * Hkv * hd + i]));
                Vv[(int64_t)t * Hkv * hd + i] = or_bf16_to_f32(or_f32_to_bf16(Vv[(int64_t)t * Hkv * hd + i]));
            }
        }
        for (int32_t t = 0; t < T; t++) {
            const int32_t lo = layer_slides(m, l) ? (t - m->sliding_window + 1 > 0
                                                         ? t - m->sliding_window + 1 : 0)
                                                  : 0;
            for (int32_t h = 0; h < Hq; h++) {
                const int32_t g = h / G;
                for (int32_t j = lo; j <= t; j++)
                    for (int32_t dd = 0; dd < hd; dd++) {
                        Kh[(int64_t)(j - lo) * hd + dd] = K[((int64_t)j * Hkv + g) * hd + dd];
                        Vh[(int64_t)(j - lo) * hd + dd] = Vv[((int64_t)j * Hkv + g) * hd + dd];
                    }
                or_attend(Q + ((int64_t)t * Hq + h) * hd, Kh, Vh, t - lo + 1, hd, o + h * hd);
            }
            matvec(m->wo[l], o, d, Hq * hd, y, nthreads);
            for (int32_t i = 0; i < d; i++) X[(int64_t)t * d + i] += y[i];
            or_rmsnorm(X + (int64_t)t * d, m->mlp_norm[l], d, m->rms_eps, xn);
            mlp_add(m, l, xn, X + (int64_t)t * d, nthreads);
        }
    }
    for (int32_t t = 0; t < T; t++) {
        or_rmsnorm(X + (int64_t)t * d, m->final_norm, d, m->rms_eps, xn);
        matvec(m->lm_head, xn, V, d, logits + (int64_t)t * V, nthreads);
    }
    free(X); free(xn); free(Q); free(K); free(Vv); free(o); free(y); free(Kh); free(Vh);
    return OR_OK;
}

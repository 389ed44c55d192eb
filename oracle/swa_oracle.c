/*
 * swa_oracle.c -- fp64 CPU oracle for causal sliding-window attention with
 * attention sinks, SWA(w, s).
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library. The CUDA library never
 * links or calls it, and it shares no code, header or constant with it.
 *
 * It is deliberately plain and slow: every query row enumerates its key set
 * by testing each earlier position against the membership rule, then applies
 * the softmax-weighted sum in double precision. There is no tiling, no online
 * softmax, no reordering.
 *
 * Sources (web pages; cited by page and section):
 *  [P1] "滑动窗口注意力（SWA）配 sinks 比 post-training 线性注意力更划算"
 *       (papers.ananclaw.com explainer of arXiv 2608.28444), section
 *       "核心方法 / 1. 训练免费的 SWA(w, s)": the x_t equation (window of the
 *       last w tokens, softmax of q_t k_i^T / sqrt(d)) and the swa_mask
 *       pseudocode (window [max(0,t-w+1), t] plus the first s columns).
 *  [P4] wiblog.cn long-context SWA article, section
 *       "与 KV Cache 的配合：轮转替换策略": rolling KV cache, oldest entry
 *       evicted, slot located by index modulo the window.
 *
 * Readings taken where the pages are silent or disagree:
 *  - Key set K(t) = { j : 0 <= j <= t and (j >= t-w+1 or j < s) }. The
 *    pseudocode's sink columns are intersected with causality (j <= t); the
 *    x_t equation is the s = 0 case. w counts the query itself.
 *  - GQA: query head hq uses key/value head hq / (Hq / Hkv) (contiguous groups).
 *  - Inputs arrive as bf16 bit patterns and are widened exactly to double.
 *    The caller's float scale is widened to double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Membership rule of SWA(w, s) for query position t and key position j. */
static int key_in_set(int64_t t, int64_t j, int64_t w, int64_t s)
{
    if (j < 0 || j > t) return 0;          /* causal */
    if (j >= t - w + 1) return 1;          /* the last w tokens, t included */
    if (j < s) return 1;                   /* the first s tokens (sinks) */
    return 0;
}

/* Enumerate K(t) by testing every position 0..t. Writes the keys in
 * increasing order to keys[] when keys is not NULL; returns |K(t)|. */
int64_t oracle_keyset(int64_t t, int64_t w, int64_t s, int64_t *keys)
{
    int64_t n = 0;
    for (int64_t j = 0; j <= t; ++j) {
        if (key_in_set(t, j, w, s)) {
            if (keys) keys[n] = j;
            ++n;
        }
    }
    return n;
}

/* The L x L boolean key mask (row t, column j) built row by row from
 * oracle_keyset. */
void oracle_keymask(int64_t L, int64_t w, int64_t s, uint8_t *mask)
{
    int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * (size_t)(L > 0 ? L : 1));
    memset(mask, 0, (size_t)(L * L));
    for (int64_t t = 0; t < L; ++t) {
        int64_t n = oracle_keyset(t, w, s, keys);
        for (int64_t i = 0; i < n; ++i) mask[t * L + keys[i]] = 1;
    }
    free(keys);
}

/* Softmax attention of one query over n gathered key/value rows.
 *   x_i = scale * (q . k_i),  m = max_i x_i,  p_i = exp(x_i - m),
 *   out = sum_i p_i v_i / sum_i p_i,  lse = m + log(sum_i p_i).
 * Rows are bf16 bit patterns with element stride 1 and length d. */
static void attend_one(const uint16_t *q, const uint16_t *const *krows,
                       const uint16_t *const *vrows, int64_t n, int64_t d,
                       double scale, double *x, double *out, double *lse)
{
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c)
            dot += bf16_to_double(q[c]) * bf16_to_double(krows[i][c]);
        x[i] = scale * dot;
        if (x[i] > m) m = x[i];
    }
    double z = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        x[i] = exp(x[i] - m);
        z += x[i];
    }
    for (int64_t c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int64_t i = 0; i < n; ++i) acc += x[i] * bf16_to_double(vrows[i][c]);
        out[c] = acc / z;
    }
    if (lse) *lse = m + log(z);
}

/* Softmax weights p_i / sum p for one query row t, in key order; used by the
 * invariant tests (rows sum to one). Returns |K(t)|. */
int64_t oracle_weights(const uint16_t *q, const uint16_t *k, int64_t L,
                       int64_t Hq, int64_t Hkv, int64_t d, int64_t w, int64_t s,
                       double scale, int64_t b, int64_t hq, int64_t t,
                       double *weights)
{
    int64_t group = Hq / Hkv, kvh = hq / group;
    int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * (size_t)(t + 1));
    int64_t n = oracle_keyset(t, w, s, keys);
    const uint16_t *qrow = q + ((b * L + t) * Hq + hq) * d;
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
        const uint16_t *krow = k + ((b * L + keys[i]) * Hkv + kvh) * d;
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c) dot += bf16_to_double(qrow[c]) * bf16_to_double(krow[c]);
        weights[i] = scale * dot;
        if (weights[i] > m) m = weights[i];
    }
    double z = 0.0;
    for (int64_t i = 0; i < n; ++i) { weights[i] = exp(weights[i] - m); z += weights[i]; }
    for (int64_t i = 0; i < n; ++i) weights[i] /= z;
    free(keys);
    return n;
}

/* Prefill: for every batch b, every listed query position t and every query
 * head hq, attend over K(t).
 *   q [B, L, Hq, d], k and v [B, L, Hkv, d]   (bf16 bit patterns)
 *   rows: nrows query positions (NULL means all L positions, nrows = L)
 *   out [B, nrows, Hq, d] double; lse [B, nrows, Hq] double or NULL.
 * Returns 0, or -1 for an invalid argument. */
int oracle_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                   int64_t B, int64_t L, int64_t Hq, int64_t Hkv, int64_t d,
                   int64_t w, int64_t s, double scale,
                   const int64_t *rows, int64_t nrows,
                   double *out, double *lse, int nthreads)
{
    if (B < 0 || L < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || w < 1 || s < 0) return -1;
    if (Hq % Hkv != 0) return -1;
    if (rows == NULL) nrows = L;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t t = rows ? rows[r] : r;
        if (t < 0 || t >= L) return -1;
    }
    int64_t group = Hq / Hkv;
    int64_t nwork = B * nrows;
    (void)nthreads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
    for (int64_t wi = 0; wi < nwork; ++wi) {
        int64_t b = wi / nrows, r = wi % nrows;
        int64_t t = rows ? rows[r] : r;
        int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * (size_t)(t + 1));
        const uint16_t **kr = (const uint16_t **)malloc(sizeof(void *) * (size_t)(t + 1));
        const uint16_t **vr = (const uint16_t **)malloc(sizeof(void *) * (size_t)(t + 1));
        double *x = (double *)malloc(sizeof(double) * (size_t)(t + 1));
        int64_t n = oracle_keyset(t, w, s, keys);
        for (int64_t hq = 0; hq < Hq; ++hq) {
            int64_t kvh = hq / group;
            for (int64_t i = 0; i < n; ++i) {
                kr[i] = k + ((b * L + keys[i]) * Hkv + kvh) * d;
                vr[i] = v + ((b * L + keys[i]) * Hkv + kvh) * d;
            }
            const uint16_t *qrow = q + ((b * L + t) * Hq + hq) * d;
            double *orow = out + ((b * nrows + r) * Hq + hq) * d;
            double *lrow = lse ? lse + (b * nrows + r) * Hq + hq : NULL;
            attend_one(qrow, kr, vr, n, d, scale, x, orow, lrow);
        }
        free(keys); free(kr); free(vr); free(x);
    }
    return 0;
}

/* Backward of the prefill: the gradients of the outputs' definition above
 * with respect to q, k and v, for an upstream gradient dout. The pages give
 * no backward formulas (they mention SWA-aware fine-tuning only); this is the
 * chain rule applied to that definition, term by term:
 *   for every (b, hq, t), over j in K(t):
 *     x_j = scale q_t . k_j,  p = softmax(x),  dp_j = dout_t . v_j,
 *     delta = sum_j p_j dp_j,  ds_j = p_j (dp_j - delta),
 *     dq_t  = scale sum_j ds_j k_j,
 *     dk_j += scale ds_j q_t,  dv_j += p_j dout_t,
 * with k_j, v_j the rows of KV head hq / (Hq / Hkv), so dk and dv sum over the
 * query heads of a group.
 *   q, k, v bf16 bit patterns ([B, L, Hq, d], [B, L, Hkv, d]); dout double
 *   [B, L, Hq, d]; dq double [B, L, Hq, d]; dk, dv double [B, L, Hkv, d]
 *   (all three written). One work item per (b, KV head) owns its dk and dv
 *   rows and its group's dq rows. Returns 0, or -1 for an invalid argument. */
int oracle_prefill_backward(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            const double *dout, int64_t B, int64_t L, int64_t Hq,
                            int64_t Hkv, int64_t d, int64_t w, int64_t s, double scale,
                            double *dq, double *dk, double *dv, int nthreads)
{
    if (B < 0 || L < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || w < 1 || s < 0) return -1;
    if (Hq % Hkv != 0) return -1;
    int64_t group = Hq / Hkv;
    memset(dq, 0, sizeof(double) * (size_t)(B * L * Hq * d));
    memset(dk, 0, sizeof(double) * (size_t)(B * L * Hkv * d));
    memset(dv, 0, sizeof(double) * (size_t)(B * L * Hkv * d));
    (void)nthreads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
    for (int64_t wi = 0; wi < B * Hkv; ++wi) {
        int64_t b = wi / Hkv, kvh = wi % Hkv;
        int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * (size_t)(L > 0 ? L : 1));
        double *p = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        double *dp = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        for (int64_t hq = kvh * group; hq < (kvh + 1) * group; ++hq) {
            for (int64_t t = 0; t < L; ++t) {
                int64_t n = oracle_keyset(t, w, s, keys);
                const uint16_t *qrow = q + ((b * L + t) * Hq + hq) * d;
                const double *gout = dout + ((b * L + t) * Hq + hq) * d;
                double m = -INFINITY;
                for (int64_t i = 0; i < n; ++i) {
                    const uint16_t *krow = k + ((b * L + keys[i]) * Hkv + kvh) * d;
                    const uint16_t *vrow = v + ((b * L + keys[i]) * Hkv + kvh) * d;
                    double dot = 0.0, g = 0.0;
                    for (int64_t c = 0; c < d; ++c) {
                        dot += bf16_to_double(qrow[c]) * bf16_to_double(krow[c]);
                        g += gout[c] * bf16_to_double(vrow[c]);
                    }
                    p[i] = scale * dot;
                    dp[i] = g;
                    if (p[i] > m) m = p[i];
                }
                double z = 0.0;
                for (int64_t i = 0; i < n; ++i) { p[i] = exp(p[i] - m); z += p[i]; }
                double delta = 0.0;
                for (int64_t i = 0; i < n; ++i) { p[i] /= z; delta += p[i] * dp[i]; }
                double *dqrow = dq + ((b * L + t) * Hq + hq) * d;
                for (int64_t i = 0; i < n; ++i) {
                    const double ds = p[i] * (dp[i] - delta);
                    const uint16_t *krow = k + ((b * L + keys[i]) * Hkv + kvh) * d;
                    double *dkrow = dk + ((b * L + keys[i]) * Hkv + kvh) * d;
                    double *dvrow = dv + ((b * L + keys[i]) * Hkv + kvh) * d;
                    for (int64_t c = 0; c < d; ++c) {
                        dqrow[c] += scale * ds * bf16_to_double(krow[c]);
                        dkrow[c] += scale * ds * bf16_to_double(qrow[c]);
                        dvrow[c] += p[i] * gout[c];
                    }
                }
            }
        }
        free(keys); free(p); free(dp);
    }
    return 0;
}

/* Decode: one new query per head at position pos, attending over K(pos).
 * The caller passes a logical history: nh rows with positions hist_pos[i] and
 * key/value rows hist_k/hist_v [nh, Hkv, d] (bf16 bit patterns), holding at
 * least every position of K(pos). Positions outside K(pos) are ignored.
 *   q [Hq, d]; out [Hq, d]; lse [Hq] or NULL.
 * Returns 0; -1 for invalid arguments; -2 if a position of K(pos) is missing
 * from the history or present twice. */
int oracle_decode(const uint16_t *q, const int64_t *hist_pos,
                  const uint16_t *hist_k, const uint16_t *hist_v, int64_t nh,
                  int64_t pos, int64_t Hq, int64_t Hkv, int64_t d, int64_t w,
                  int64_t s, double scale, double *out, double *lse)
{
    if (pos < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || w < 1 || s < 0 || Hq % Hkv) return -1;
    int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * (size_t)(pos + 1));
    int64_t n = oracle_keyset(pos, w, s, keys);
    int64_t *where = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    int rc = 0;
    for (int64_t i = 0; i < n && rc == 0; ++i) {
        where[i] = -1;
        for (int64_t h = 0; h < nh; ++h) {
            if (hist_pos[h] == keys[i]) {
                if (where[i] >= 0) { rc = -2; break; }
                where[i] = h;
            }
        }
        if (where[i] < 0) rc = -2;
    }
    if (rc == 0) {
        int64_t group = Hq / Hkv;
        const uint16_t **kr = (const uint16_t **)malloc(sizeof(void *) * (size_t)n);
        const uint16_t **vr = (const uint16_t **)malloc(sizeof(void *) * (size_t)n);
        double *x = (double *)malloc(sizeof(double) * (size_t)n);
        for (int64_t hq = 0; hq < Hq; ++hq) {
            int64_t kvh = hq / group;
            for (int64_t i = 0; i < n; ++i) {
                kr[i] = hist_k + (where[i] * Hkv + kvh) * d;
                vr[i] = hist_v + (where[i] * Hkv + kvh) * d;
            }
            attend_one(q + hq * d, kr, vr, n, d, scale, x, out + hq * d, lse ? lse + hq : NULL);
        }
        free(kr); free(vr); free(x);
    }
    free(keys); free(where);
    return rc;
}

/* Rolling KV cache as a literal circular buffer [P4, "轮转替换策略"]: s pinned
 * sink slots that take positions 0..s-1, followed by w window slots filled by a
 * write pointer that advances by one and wraps to the first window slot.
 * Positions 0..last are appended in order. slot_pos[i] receives the position
 * held by slot i after the last append, or -1 if the slot was never written. */
void oracle_ring_contents(int64_t last, int64_t w, int64_t s, int64_t *slot_pos)
{
    for (int64_t i = 0; i < s + w; ++i) slot_pos[i] = -1;
    int64_t ptr = 0;
    for (int64_t p = 0; p <= last; ++p) {
        if (p < s) {
            slot_pos[p] = p;
        } else {
            slot_pos[s + ptr] = p;
            ptr = ptr + 1;
            if (ptr == w) ptr = 0;
        }
    }
}

/*
 * fp64 CPU oracle for context-parallel causal GQA prefill attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path (the CUDA library
 * and its Python binding) may include, link, load or call this file; only the
 * tests, the smoke check and the benchmark's CPU-baseline leg do.  It shares
 * no code, header, table or helper with the CUDA path.
 *
 * What it computes, and where that is defined:
 *
 *   Moreh, "Optimizing long-context prefill on multiple older-generation GPU
 *   nodes", section "Introduction to Context Parallelism": the prompt is split
 *   along the sequence; attention is the one op with cross-token dependence;
 *   Ring Attention computes attention on each device from a *partial* set of
 *   queries, keys and values while keys/values move between neighbours.
 *
 *   The pages give no formula.  The plainest reading, taken here, is that the
 *   method computes exactly ordinary softmax attention restricted by a causal
 *   (optionally sliding-window) mask, with grouped-query heads, and that each
 *   partial (queries against one block of keys) is reported as a normalised
 *   output plus the natural-log sum of exp of its scaled scores, so that
 *   partials over disjoint key blocks combine exactly (log-sum-exp merge).
 *
 * Definitions implemented (fp64 throughout, inputs are bf16 bit patterns
 * widened exactly):
 *
 *   g(h)      = floor(h / (Hq / Hkv))                 (grouped-query heads)
 *   visible   = (!causal || pos_k <= pos_q) && (W == 0 || pos_q - pos_k < W)
 *   s_j       = scale * sum_d q[i,h,d] * k[j,g,d]
 *   m         = max over visible j of s_j
 *   l         = sum over visible j of exp(s_j - m)
 *   out[i,h]  = sum over visible j of exp(s_j - m) * v[j,g,:] / l
 *   lse[h,i]  = m + ln l ;  no visible key: out = 0, lse = -inf
 *
 *   merge:  L = log sum_k exp(lse_k)   (shifted by the max; all -inf -> -inf)
 *           out = sum_k exp(lse_k - L) * out_k
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double widen_bf16(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Key at global position pk is visible to the query at global position pq. */
static int key_visible(int64_t pq, int64_t pk, int causal, int64_t window)
{
    if (causal && pk > pq)
        return 0;
    if (window > 0 && pq - pk >= window)
        return 0;
    return 1;
}

/*
 * Attention of a block of queries against a block of keys/values.
 *
 * q: bf16 bits, element (i, h, d) at q[i*q_srow + h*q_shead + d], i < Sq, h < Hq
 * k: bf16 bits, element (j, g, d) at k[j*k_srow + g*k_shead + d], j < Skv, g < Hkv
 * v: bf16 bits, element (j, g, e) at v[j*v_srow + g*v_shead + e], e < dv
 * q_pos0 / kv_pos0: global positions of q row 0 / k row 0 (masks use these).
 * rows (n_rows entries, or NULL = all Sq rows) and heads (n_heads entries, or
 * NULL = all Hq heads) select which outputs to compute.
 * out: [n_rows][n_heads][dv] fp64, lse: [n_heads][n_rows] fp64.
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int oracle_attention(const uint16_t *q, int64_t q_srow, int64_t q_shead,
                     const uint16_t *k, int64_t k_srow, int64_t k_shead,
                     const uint16_t *v, int64_t v_srow, int64_t v_shead,
                     int64_t Sq, int64_t Skv, int Hq, int Hkv, int dqk, int dv,
                     int64_t q_pos0, int64_t kv_pos0, int causal, int64_t window,
                     double scale, const int64_t *rows, int64_t n_rows,
                     const int *heads, int n_heads, double *out, double *lse)
{
    if ((!q && Sq > 0) || ((!k || !v) && Skv > 0) || Hq <= 0 || Hkv <= 0 ||
        Hq % Hkv != 0 || dqk <= 0 || dv <= 0 || Sq < 0 || Skv < 0)
        return -1;
    if (!rows)
        n_rows = Sq;
    if (!heads)
        n_heads = Hq;
    if ((!out || !lse) && n_rows * (int64_t)n_heads > 0)
        return -1;
    const int G = Hq / Hkv;
    const int64_t total = n_rows * (int64_t)n_heads;
    int failed = 0;

#pragma omp parallel reduction(| : failed)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Skv > 0 ? Skv : 1));
        double *qi = (double *)malloc(sizeof(double) * (size_t)dqk);
        double *acc = (double *)malloc(sizeof(double) * (size_t)dv);
        const int ok = s && qi && acc;
#pragma omp for schedule(dynamic, 16)
        for (int64_t t = 0; t < total; ++t) {
            if (!ok) {
                failed = 1;
                continue;
            }
            const int64_t hr = t / n_rows, rr = t % n_rows;
            const int h = heads ? heads[hr] : (int)hr;
            const int64_t i = rows ? rows[rr] : rr;
            const int g = h / G;
            double *o = out + (rr * n_heads + hr) * (int64_t)dv;
            double *ls = lse + hr * n_rows + rr;
            if (h < 0 || h >= Hq || i < 0 || i >= Sq) {
                failed = 1;
                continue;
            }
            const int64_t pq = q_pos0 + i;
            for (int d = 0; d < dqk; ++d)
                qi[d] = widen_bf16(q[i * q_srow + (int64_t)h * q_shead + d]);

            /* scores of visible keys and their maximum */
            double m = -INFINITY;
            for (int64_t j = 0; j < Skv; ++j) {
                if (!key_visible(pq, kv_pos0 + j, causal, window)) {
                    s[j] = -INFINITY;
                    continue;
                }
                const uint16_t *kj = k + j * k_srow + (int64_t)g * k_shead;
                double dot = 0.0;
                for (int d = 0; d < dqk; ++d)
                    dot += qi[d] * widen_bf16(kj[d]);
                s[j] = scale * dot;
                if (s[j] > m)
                    m = s[j];
            }
            if (m == -INFINITY) { /* no visible key */
                for (int e = 0; e < dv; ++e)
                    o[e] = 0.0;
                *ls = -INFINITY;
                continue;
            }
            /* exp-weights, their sum, and the weighted sum of values */
            double l = 0.0;
            for (int e = 0; e < dv; ++e)
                acc[e] = 0.0;
            for (int64_t j = 0; j < Skv; ++j) {
                if (s[j] == -INFINITY)
                    continue;
                const double p = exp(s[j] - m);
                l += p;
                const uint16_t *vj = v + j * v_srow + (int64_t)g * v_shead;
                for (int e = 0; e < dv; ++e)
                    acc[e] += p * widen_bf16(vj[e]);
            }
            for (int e = 0; e < dv; ++e)
                o[e] = acc[e] / l;
            *ls = m + log(l);
        }
        free(s);
        free(qi);
        free(acc);
    }
    return failed ? -1 : 0;
}

/*
 * Exact log-sum-exp merge of n partials over disjoint key sets.
 * outs[k]: [n_rows][n_heads][dv] fp64, lses[k]: [n_heads][n_rows] fp64.
 * out: [n_rows][n_heads][dv], lse: [n_heads][n_rows].
 */
int oracle_merge(const double *const *outs, const double *const *lses, int n,
                 int64_t n_rows, int n_heads, int dv, double *out, double *lse)
{
    if (!outs || !lses || !out || !lse || n < 0 || n_rows < 0 || n_heads < 0 || dv <= 0)
        return -1;
    const int64_t total = n_rows * (int64_t)n_heads;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < total; ++t) {
        const int64_t h = t / n_rows, r = t % n_rows;
        double mx = -INFINITY;
        for (int p = 0; p < n; ++p) {
            const double x = lses[p][h * n_rows + r];
            if (x > mx)
                mx = x;
        }
        double *o = out + (r * n_heads + h) * (int64_t)dv;
        if (mx == -INFINITY) {
            for (int e = 0; e < dv; ++e)
                o[e] = 0.0;
            lse[h * n_rows + r] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int p = 0; p < n; ++p)
            sum += exp(lses[p][h * n_rows + r] - mx);
        const double L = mx + log(sum);
        for (int e = 0; e < dv; ++e)
            o[e] = 0.0;
        for (int p = 0; p < n; ++p) {
            const double x = lses[p][h * n_rows + r];
            if (x == -INFINITY)
                continue;
            const double w = exp(x - L);
            const double *op = outs[p] + (r * n_heads + h) * (int64_t)dv;
            for (int e = 0; e < dv; ++e)
                o[e] += w * op[e];
        }
        lse[h * n_rows + r] = L;
    }
    return 0;
}

/* Number of OpenMP threads a parallel region of this library uses. */
int oracle_num_threads(void)
{
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        {
#ifdef _OPENMP
            n = omp_get_num_threads();
#endif
        }
    }
    return n;
}

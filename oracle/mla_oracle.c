/*
 * fp64 CPU oracle of the matrix-absorbed, NoPE, causal Gated MLA forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header or constant with the CUDA
 * library.
 *
 * Source: the course-notes page "Gated MLA（矩阵吸收版）" (Gated MLA, matrix
 * absorption), sections "矩阵吸收的核心思路" (core idea of absorption) and
 * "完整计算流（四步）" (the full four-step computation), steps 2-4, and the
 * symbol table page "符号表", table "MLA 变量".
 *
 * Every quantity is computed in double precision, in the order the page states
 * the steps, with no tiling, no online softmax and no fusion:
 *   step 2  q_abs[j]  = sum_d q[b,t,h,d] * W_UK[h,d,j]            (absorb)
 *           s[u]      = scale * sum_j q_abs[j] * c[b,u,j]   u <= t  (score)
 *           a[u]      = exp(s[u]-max s) / sum exp(s-max s)          (causal softmax)
 *   step 3  o_lat[j]  = sum_u a[u] * c[b,u,j]                       (latent weighting)
 *           o[v]      = sum_j o_lat[j] * W_UV[h,v,j]                (W_UV up-projection)
 *   step 4  out[b,t,h*d_v+v] = sigmoid(g[b,t,h*d_v+v]) * o[v]       (output gate)
 * Readings where the page is silent: the mask keeps u <= t (each token sees
 * itself and its past); a softmax scale multiplies the score before the mask
 * (1.0 reproduces the page's listing, which applies none); `g` is the gate's
 * pre-sigmoid logit W_g x, and a NULL g means no gate; the output's flat index
 * is h*d_v + v, the order of the listing's transpose-then-reshape.
 *
 * Parity: pinned by the tests against explicit decompression (k = c W_UK^T,
 * v = c W_UV^T under ordinary causal attention), softmax rows summing to one,
 * the T = 1 closed form, causality, prefix means under uniform attention and a
 * brute-force transcription on tiny inputs.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG -1
#define ORACLE_ERR_NOMEM -2

/* Step 2, absorb: q_abs = q_h . W_UK,h   ('bthd,hdj->bthj'). */
static void absorb_query(const double *q_row, const double *w_uk_h, int dq, int r, double *q_abs)
{
    for (int j = 0; j < r; ++j) {
        double acc = 0.0;
        for (int d = 0; d < dq; ++d) acc += q_row[d] * w_uk_h[(size_t)d * r + j];
        q_abs[j] = acc;
    }
}

/* Steps 2 (score, softmax), 3 and 4 for one (token, head) row whose absorbed
 * query is `q_abs`.  `c_rows` points at the first latent row of the sequence;
 * `n_keys` rows (row stride `ld_c`) are visible, every other key is masked. */
static void attend_latent_row(const double *q_abs, const double *c_rows, long long ld_c, long long n_keys,
                              const double *w_uv_h, const double *g_row, double scale, int dv, int r,
                              double *s, double *o_lat, double *out_row)
{
    /* step 2, score against the latent itself: s = q_abs . c^T  ('bthj,bsj->bhts') */
    for (long long u = 0; u < n_keys; ++u) {
        const double *cu = c_rows + u * ld_c;
        double acc = 0.0;
        for (int j = 0; j < r; ++j) acc += q_abs[j] * cu[j];
        s[u] = scale * acc;
    }
    /* step 2, softmax over the visible keys (masked keys carry weight 0) */
    double m = -INFINITY;
    for (long long u = 0; u < n_keys; ++u) if (s[u] > m) m = s[u];
    double z = 0.0;
    for (long long u = 0; u < n_keys; ++u) { s[u] = exp(s[u] - m); z += s[u]; }
    for (long long u = 0; u < n_keys; ++u) s[u] /= z;
    /* step 3, weight the latent rows first: o_lat = attn . c  ('bhts,bsj->bhtj') */
    for (int j = 0; j < r; ++j) o_lat[j] = 0.0;
    for (long long u = 0; u < n_keys; ++u) {
        const double *cu = c_rows + u * ld_c;
        for (int j = 0; j < r; ++j) o_lat[j] += s[u] * cu[j];
    }
    /* step 3, then up-project: o = o_lat . W_UV^T  ('bhtj,hvj->bhtv') */
    for (int v = 0; v < dv; ++v) {
        double acc = 0.0;
        for (int j = 0; j < r; ++j) acc += o_lat[j] * w_uv_h[(size_t)v * r + j];
        /* step 4, gate: sigmoid(W_g x) elementwise on the flattened heads */
        out_row[v] = g_row ? acc / (1.0 + exp(-g_row[v])) : acc;
    }
}

/*
 * Prefill (T queries against T keys, causal).
 *   q    [B,T,H,dq]   c [B,T,r]   w_uk [H,dq,r]   w_uv [H,dv,r]
 *   g    [B,T,H*dv] pre-sigmoid gate logits, or NULL (no gate)
 *   out  [n_out_rows, H*dv]
 * `rows` selects which flattened (b*T + t) token rows to compute (so a full-
 * size problem can be checked on a sample); NULL means all B*T rows in order.
 */
int mla_oracle_prefill(const double *q, const double *c, const double *w_uk, const double *w_uv,
                       const double *g, double scale, double *out,
                       int B, int T, int H, int dq, int dv, int r,
                       const long long *rows, long long n_rows)
{
    if (!q || !c || !w_uk || !w_uv || !out) return ORACLE_ERR_ARG;
    if (B < 0 || T < 0 || H <= 0 || dq <= 0 || dv <= 0 || r <= 0) return ORACLE_ERR_ARG;
    const long long total = rows ? n_rows : (long long)B * T;
    int err = ORACLE_OK;
#pragma omp parallel
    {
        double *q_abs = (double *)malloc(sizeof(double) * (size_t)r);
        double *o_lat = (double *)malloc(sizeof(double) * (size_t)r);
        double *s = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
        if (!q_abs || !o_lat || !s) {
#pragma omp atomic write
            err = ORACLE_ERR_NOMEM;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long long work = 0; work < total * H; ++work) {
                const long long i = work / H;
                const int h = (int)(work % H);
                const long long bt = rows ? rows[i] : i;
                if (bt < 0 || bt >= (long long)B * T) {
#pragma omp atomic write
                    err = ORACLE_ERR_ARG;
                    continue;
                }
                const long long b = bt / T, t = bt % T;
                absorb_query(q + ((size_t)bt * H + h) * dq, w_uk + (size_t)h * dq * r, dq, r, q_abs);
                attend_latent_row(q_abs, c + (size_t)b * T * r, r, t + 1, w_uv + (size_t)h * dv * r,
                                  g ? g + (size_t)bt * H * dv + (size_t)h * dv : NULL, scale, dv, r,
                                  s, o_lat, out + (size_t)i * H * dv + (size_t)h * dv);
            }
        }
        free(q_abs);
        free(o_lat);
        free(s);
    }
    return err;
}

/*
 * Cached-latent decode: one query per sequence, sequence b attends to cache
 * rows [0, lens[b]) with no mask (its own latent is the last cached row).
 * The query arrives already absorbed, so step 2 starts at the score.
 *   q_abs   [B,H,r]
 *   c_cache element (b,u,j) at b*max_len*ld_cache + u*ld_cache + j
 *   lens    [B], 0 <= lens[b] <= max_len; lens[b] == 0 gives an all-zero row
 *   w_uv    [H,dv,r]   g [B,H*dv] or NULL   out [B,H*dv]
 */
int mla_oracle_decode(const double *q_abs, const double *c_cache, long long ld_cache, long long max_len,
                      const int *lens, const double *w_uv, const double *g, double scale, double *out,
                      int B, int H, int dv, int r)
{
    if (!q_abs || !c_cache || !lens || !w_uv || !out) return ORACLE_ERR_ARG;
    if (B < 0 || H <= 0 || dv <= 0 || r <= 0 || ld_cache < r || max_len < 0) return ORACLE_ERR_ARG;
    for (int b = 0; b < B; ++b)
        if (lens[b] < 0 || lens[b] > max_len) return ORACLE_ERR_ARG;
    int err = ORACLE_OK;
#pragma omp parallel
    {
        double *o_lat = (double *)malloc(sizeof(double) * (size_t)r);
        double *s = (double *)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
        if (!o_lat || !s) {
#pragma omp atomic write
            err = ORACLE_ERR_NOMEM;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long long work = 0; work < (long long)B * H; ++work) {
                const int b = (int)(work / H), h = (int)(work % H);
                double *out_row = out + ((size_t)b * H + h) * dv;
                if (lens[b] == 0) {
                    for (int v = 0; v < dv; ++v) out_row[v] = 0.0;
                    continue;
                }
                attend_latent_row(q_abs + ((size_t)b * H + h) * r, c_cache + (size_t)b * max_len * ld_cache,
                                  ld_cache, lens[b], w_uv + (size_t)h * dv * r,
                                  g ? g + (size_t)b * H * dv + (size_t)h * dv : NULL, scale, dv, r,
                                  s, o_lat, out_row);
            }
        }
        free(o_lat);
        free(s);
    }
    return err;
}

/* Number of threads an OpenMP parallel region uses here (1 without OpenMP). */
int mla_oracle_num_threads(void)
{
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        {
#ifdef _OPENMP
            extern int omp_get_num_threads(void);
            n = omp_get_num_threads();
#endif
        }
    }
    return n;
}

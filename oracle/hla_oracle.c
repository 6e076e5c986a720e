/*
 * Oracle for the hybrid Gated-DeltaNet + sink/sliding-window softmax layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Plain, slow, sequential fp64 C.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load this
 * file's library.  It shares nothing with the CUDA path (no header, no table,
 * no helper).
 *
 * Sources (the pages are web summaries of the paper "The Key to Going Linear:
 * Analysis-Driven Transformer Linearization", Kuzina, Whatmough, Ehteshami
 * Bejnordi):
 *   - GDN state update: section "线性注意力替换机制" (linear attention
 *     replacement), the GDN equation S_t = (I - b_t k_t k_t^T) G_t S_{t-1}
 *     + b_t k_t^T v_t, with G_t = alpha_t I (scalar gate).
 *   - Cache budget: section "填补近似缺口的实用设计" (closing the
 *     approximation gap): 8 sink tokens keep full attention, a sliding window
 *     covers the rest of the budget, the linear path covers every other token.
 *   - Feature path: section "实践建议" item 3 (practical advice): a short
 *     convolution of kernel size 8 after RoPE and before L2 normalisation.
 *   - Softmax scale 1/sqrt(d): section "从 softmax 到 delta 规则的一阶近似",
 *     Lemma 1.
 *   - Weighted sum of the two branches: "Untangling Component Imbalance in
 *     Hybrid Linear Attention Conversion", section 关键设计 (1), inference-time
 *     hybridisation.
 *
 * Readings where the pages are silent (each one is listed in the design
 * notes): rotate-half RoPE with theta_i = base^(-2i/d); depthwise causal conv
 * with zero left padding, no bias, no activation, tap width-1 on the current
 * token; q is L2-normalised too; L2 eps 1e-6 inside the sqrt; token j enters
 * the state when it leaves the window (at position j + W) with its own gate
 * and beta, and no decay is applied while it waits; the softmax branch uses
 * the RoPE'd (not convolved) q, k and the raw v; o = o_sm + lambda * o_lin.
 *
 * Layouts: every array is row-major, one row per position of ONE sequence and
 * ONE head: x[p*d + c].  The state S is d_k x d_v, S[i*d + j], i = key dim.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

/* RoPE, rotate-half convention: channel pairs (i, i + d/2) of position p are
 * rotated by the angle p * base^(-2i/d). */
ORACLE_API void oracle_rope(int len, int d, double base, const double* x, double* y)
{
    int half = d / 2;
    for (int p = 0; p < len; ++p) {
        for (int i = 0; i < half; ++i) {
            double theta = pow(base, -2.0 * (double)i / (double)d);
            double angle = (double)p * theta;
            double c = cos(angle), s = sin(angle);
            double x1 = x[(size_t)p * d + i];
            double x2 = x[(size_t)p * d + i + half];
            y[(size_t)p * d + i] = x1 * c - x2 * s;
            y[(size_t)p * d + i + half] = x2 * c + x1 * s;
        }
    }
}

/* Causal depthwise short convolution, one filter per channel:
 *   y_p[c] = sum_{m=0}^{width-1} w[c][m] * x_{p-(width-1)+m}[c],
 * positions before the start of the sequence count as zero. */
ORACLE_API void oracle_short_conv(int len, int d, int width, const double* x,
                                  const double* w, double* y)
{
    for (int p = 0; p < len; ++p) {
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int m = 0; m < width; ++m) {
                int src = p - (width - 1) + m;
                if (src >= 0) acc += w[(size_t)c * width + m] * x[(size_t)src * d + c];
            }
            y[(size_t)p * d + c] = acc;
        }
    }
}

/* Row-wise L2 normalisation: y_p = x_p / sqrt(|x_p|^2 + eps). */
ORACLE_API void oracle_l2norm(int len, int d, double eps, const double* x, double* y)
{
    for (int p = 0; p < len; ++p) {
        double ss = 0.0;
        for (int c = 0; c < d; ++c) ss += x[(size_t)p * d + c] * x[(size_t)p * d + c];
        double inv = 1.0 / sqrt(ss + eps);
        for (int c = 0; c < d; ++c) y[(size_t)p * d + c] = x[(size_t)p * d + c] * inv;
    }
}

/* One GDN state update with token j (key k, value v, gate alpha, beta b):
 *   S <- alpha S - b alpha k (k^T S) + b k v^T        (erase on)
 *   S <- alpha S + k v^T                              (erase off: the GLA
 *                                                      update with scalar gate)
 */
ORACLE_API void oracle_gdn_update(int d, double* S, const double* k, const double* v,
                                  double alpha, double b, int erase_off, double* scratch)
{
    double* x = scratch; /* x = k^T S, a row over the value dim */
    for (int j = 0; j < d; ++j) {
        double acc = 0.0;
        for (int i = 0; i < d; ++i) acc += k[i] * S[(size_t)i * d + j];
        x[j] = acc;
    }
    for (int i = 0; i < d; ++i) {
        for (int j = 0; j < d; ++j) {
            double s = S[(size_t)i * d + j];
            if (erase_off)
                S[(size_t)i * d + j] = alpha * s + k[i] * v[j];
            else
                S[(size_t)i * d + j] = alpha * s - b * alpha * k[i] * x[j] + b * k[i] * v[j];
        }
    }
}

/* Linear branch with fixed-budget routing.  For each position p in order:
 * token j = p - window leaves the window now; if it is not a sink (j >=
 * n_sinks) it is absorbed into S with its own g_j (log alpha) and beta_j.
 * Then o_lin[p] = S^T qhat_p.  S_out receives the state after the last
 * absorption. */
ORACLE_API void oracle_gdn_delayed(int len, int d, int n_sinks, int window,
                                   const double* qhat, const double* khat, const double* vhat,
                                   const double* g, const double* beta, int erase_off,
                                   double* o_lin, double* S_out)
{
    double* S = (double*)calloc((size_t)d * d, sizeof(double));
    double* scratch = (double*)malloc((size_t)d * sizeof(double));
    for (int p = 0; p < len; ++p) {
        int j = p - window;
        if (j >= n_sinks) {
            oracle_gdn_update(d, S, khat + (size_t)j * d, vhat + (size_t)j * d,
                              exp(g[j]), beta[j], erase_off, scratch);
        }
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i) acc += qhat[(size_t)p * d + i] * S[(size_t)i * d + c];
            o_lin[(size_t)p * d + c] = acc;
        }
    }
    if (S_out) memcpy(S_out, S, (size_t)d * d * sizeof(double));
    free(scratch);
    free(S);
}

/* Is key position j visible to query position p?  Sinks are positions
 * 0..n_sinks-1; the window is the `window` most recent positions, the current
 * one included; the two sets are merged as a union. */
ORACLE_API int oracle_key_visible(int p, int j, int n_sinks, int window)
{
    if (j > p || j < 0) return 0;
    if (j < n_sinks) return 1;
    return j >= p - window + 1;
}

/* Exact softmax over the sink + window key set, scale 1/sqrt(d), with the
 * RoPE'd query/key and the raw value rows. */
ORACLE_API void oracle_window_softmax(int len, int d, int n_sinks, int window,
                                      const double* qr, const double* kr, const double* v,
                                      double* o_sm)
{
    double scale = 1.0 / sqrt((double)d);
    double* logit = (double*)malloc((size_t)(len > 0 ? len : 1) * sizeof(double));
    for (int p = 0; p < len; ++p) {
        double mx = -INFINITY;
        for (int j = 0; j <= p; ++j) {
            if (!oracle_key_visible(p, j, n_sinks, window)) continue;
            double acc = 0.0;
            for (int c = 0; c < d; ++c) acc += qr[(size_t)p * d + c] * kr[(size_t)j * d + c];
            logit[j] = acc * scale;
            if (logit[j] > mx) mx = logit[j];
        }
        double den = 0.0;
        for (int c = 0; c < d; ++c) o_sm[(size_t)p * d + c] = 0.0;
        for (int j = 0; j <= p; ++j) {
            if (!oracle_key_visible(p, j, n_sinks, window)) continue;
            double e = exp(logit[j] - mx);
            den += e;
            for (int c = 0; c < d; ++c) o_sm[(size_t)p * d + c] += e * v[(size_t)j * d + c];
        }
        for (int c = 0; c < d; ++c) o_sm[(size_t)p * d + c] /= den;
    }
    free(logit);
}

/* Configuration of one (sequence, query head) unit. */
typedef struct oracle_cfg {
    int d;           /* head dim */
    int n_sinks;
    int window;
    int conv_width;  /* 8 */
    double rope_base;
    double l2_eps;   /* 1e-6 */
    int l2norm_q;    /* 1: qhat = L2(conv(RoPE q)) */
    int erase_off;   /* test switch: GLA update instead of the delta rule */
    int softmax_off; /* test switch: drop the softmax branch */
} oracle_cfg;

/* The whole layer for one (sequence, query head): q, g, beta of that q-head,
 * k, v of its kv-head, conv filters [d][width] of the matching channels.
 * Optional outputs (NULL to skip): intermediates of the feature path and of
 * the two branches. */
ORACLE_API int oracle_layer_unit(const oracle_cfg* cfg, int len,
                                 const double* q, const double* k, const double* v,
                                 const double* g, const double* beta, double lambda,
                                 const double* wq, const double* wk, const double* wv,
                                 double* o, double* S_final,
                                 double* qr_out, double* kr_out,
                                 double* qhat_out, double* khat_out, double* vhat_out,
                                 double* o_sm_out, double* o_lin_out)
{
    int d = cfg->d;
    size_t n = (size_t)(len > 0 ? len : 1) * d;
    double* qr = (double*)malloc(n * sizeof(double));
    double* kr = (double*)malloc(n * sizeof(double));
    double* tq = (double*)malloc(n * sizeof(double));
    double* tk = (double*)malloc(n * sizeof(double));
    double* vh = (double*)malloc(n * sizeof(double));
    double* qh = (double*)malloc(n * sizeof(double));
    double* kh = (double*)malloc(n * sizeof(double));
    double* osm = (double*)malloc(n * sizeof(double));
    double* olin = (double*)malloc(n * sizeof(double));
    if (!qr || !kr || !tq || !tk || !vh || !qh || !kh || !osm || !olin) return 1;

    /* feature path: RoPE -> short conv -> L2 */
    oracle_rope(len, d, cfg->rope_base, q, qr);
    oracle_rope(len, d, cfg->rope_base, k, kr);
    oracle_short_conv(len, d, cfg->conv_width, qr, wq, tq);
    oracle_short_conv(len, d, cfg->conv_width, kr, wk, tk);
    oracle_short_conv(len, d, cfg->conv_width, v, wv, vh);
    if (cfg->l2norm_q)
        oracle_l2norm(len, d, cfg->l2_eps, tq, qh);
    else
        memcpy(qh, tq, n * sizeof(double));
    oracle_l2norm(len, d, cfg->l2_eps, tk, kh);

    /* linear branch (delayed absorption) and exact branch */
    oracle_gdn_delayed(len, d, cfg->n_sinks, cfg->window, qh, kh, vh, g, beta,
                       cfg->erase_off, olin, S_final);
    if (cfg->softmax_off)
        memset(osm, 0, n * sizeof(double));
    else
        oracle_window_softmax(len, d, cfg->n_sinks, cfg->window, qr, kr, v, osm);

    /* combine */
    for (size_t i = 0; i < (size_t)len * d; ++i) o[i] = osm[i] + lambda * olin[i];

    if (qr_out) memcpy(qr_out, qr, (size_t)len * d * sizeof(double));
    if (kr_out) memcpy(kr_out, kr, (size_t)len * d * sizeof(double));
    if (qhat_out) memcpy(qhat_out, qh, (size_t)len * d * sizeof(double));
    if (khat_out) memcpy(khat_out, kh, (size_t)len * d * sizeof(double));
    if (vhat_out) memcpy(vhat_out, vh, (size_t)len * d * sizeof(double));
    if (o_sm_out) memcpy(o_sm_out, osm, (size_t)len * d * sizeof(double));
    if (o_lin_out) memcpy(o_lin_out, olin, (size_t)len * d * sizeof(double));

    free(qr); free(kr); free(tq); free(tk); free(vh); free(qh); free(kh); free(osm); free(olin);
    return 0;
}

/* Key concentration and projection residual, the quantities of the analysis
 * in "迈向线性的关键：分析驱动的 Transformer 线性化", sections
 * 从 softmax 到 delta 规则的一阶近似 (Lemma 2 replaces "subtract the mean
 * key" by "project onto the orthogonal complement of the mean key", assuming
 * normalised, concentrated keys), 填补近似缺口的实用设计 (when keys do not
 * line up with one main direction the projection residual grows) and
 * 实验结果分析 (Fig. 3).  For the keys kr of one sequence and head (the
 * softmax branch's RoPE'd keys), at every position p, with u_i = kr_i/|kr_i|
 * and the prefix mean m_p = (1/(p+1)) sum_{i<=p} u_i:
 *   concentration[p] = |m_p|
 *   residual[p]      = |u_p - (mhat_p . u_p) mhat_p|,  mhat_p = m_p/|m_p|
 * (residual[p] = 1 where m_p = 0; a zero key counts as u = 0). */
ORACLE_API void oracle_key_stats(int len, int d, const double* kr, double* concentration, double* residual)
{
    double* m = (double*)calloc((size_t)(d > 0 ? d : 1), sizeof(double));
    double* u = (double*)malloc((size_t)(d > 0 ? d : 1) * sizeof(double));
    for (int p = 0; p < len; ++p) {
        double nk = 0.0;
        for (int c = 0; c < d; ++c) nk += kr[(size_t)p * d + c] * kr[(size_t)p * d + c];
        nk = sqrt(nk);
        for (int c = 0; c < d; ++c) {
            u[c] = nk > 0.0 ? kr[(size_t)p * d + c] / nk : 0.0;
            m[c] += u[c];
        }
        double nm = 0.0, dot = 0.0;
        for (int c = 0; c < d; ++c) {
            double mc = m[c] / (double)(p + 1);
            nm += mc * mc;
            dot += mc * u[c];
        }
        nm = sqrt(nm);
        concentration[p] = nm;
        if (nm == 0.0) {
            residual[p] = 1.0;
        } else {
            double proj = dot / nm, r = 0.0;
            for (int c = 0; c < d; ++c) {
                double e = u[c] - proj * (m[c] / (double)(p + 1)) / nm;
                r += e * e;
            }
            residual[p] = sqrt(r);
        }
    }
    free(u);
    free(m);
}


/*
 * GatedDeltaNet layer oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, sequential, obviously-correct fp64 C.  Only the test suite, the smoke
 * check and the CPU-baseline leg of the benchmark may load this file's library;
 * the CUDA product path never calls it and shares no code with it.
 *
 * What it computes, one (sequence, value-head) chain at a time.  The layer is
 * the one the pages name "GatedDeltaNet" with its "RMSNormGated" output norm
 * ("[Qwen3.5 MoE] Add hybrid decoder model (GatedDeltaNet + full attention +
 * MoE)", Summary, model.py bullet), its "depthwise conv1d" and "softplus"
 * (same page, parallelize.py bullet), run over packed variable-length
 * sequences ("Support Qwen35 SFT", XTuner changes: GatedDeltaNet in varlen
 * mode; "feat(models): dense Qwen3.5 custom attention", Summary: varlen
 * cu_seqlens, one packed row).  The pages name the pieces but print no
 * formula; the definitions written out below are the gated delta rule of
 * Yang, Kautz & Hatamizadeh, "Gated Delta Networks: Improving Mamba2 with
 * Delta Rule" (ICLR 2025):
 *
 *   conv     pre_t[c] = sum_{j=0..3} w[c][j] * x_{t-3+j}[c]   (x before the
 *            sequence start = 0 in prefill, = the carried cache in decode)
 *   SiLU     xh = pre * sigmoid(pre)
 *   L2       q <- q / sqrt(sum q^2 + eps_l2), same for k            (eps_l2 = 1e-6)
 *   gates    g_t = -exp(A_log) * softplus(a_t + dt_bias),  alpha_t = exp(g_t)
 *            beta_t = sigmoid(b_t)
 *   rule     S_t = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *            o_t = S_t q_t * dk^-1/2
 *   norm     y_t = o_t / sqrt(mean(o_t^2) + eps_rms) * w * silu(z_t)   (eps_rms = 1e-6)
 *
 * The state is stored as H = S^T (dk x dv, row i over dk, column j over dv),
 * the layout of the library's state tensors: element [i][j] = S[j][i].  In
 * that form one token is
 *   p = H^T k,   u = beta (v - alpha p),   H <- alpha H + k u^T,   o = H^T q * scale
 * which is S_t above multiplied out:
 *   alpha S_{t-1} - alpha beta S_{t-1} k k^T + beta v k^T
 *     = alpha S_{t-1} + beta (v - alpha S_{t-1} k) k^T,
 * transposed.
 *
 * A second, chunked formulation of the same recurrence (the WY/UT form of
 * Yang et al., "Parallelizing Linear Transformers with the Delta Rule over
 * Sequence Length", NeurIPS 2024, with the gate folded in as in the Gated
 * Delta Networks paper) is given in gdn_ref_recurrence_chunked; tests check
 * that the two agree.
 *
 * Every array is contiguous, row-major, fp64.  Nothing here allocates more
 * than O(dk*dv + C*C) scratch per call, and every function is re-entrant, so
 * callers may run independent chains on separate threads.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* softplus(x) = log(1 + e^x), written so that large x does not overflow. */
static double softplus(double x) { return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x)); }

/*
 * Causal depthwise convolution of width 4 followed by SiLU, for L tokens of
 * C channels.  x[t][c]; w[c][0..3] where w[c][3] multiplies the current token
 * and w[c][0] the token three steps back; hist[m][c] (m = 0, 1, 2) holds the
 * inputs at t = -3, -2, -1 (NULL = zeros, the start of a prefill sequence).
 * Writes y[t][c] = silu(pre_t[c]).
 */
void gdn_ref_conv_silu(int L, int C, const double *x, const double *w,
                       const double *hist, double *y) {
  for (int t = 0; t < L; ++t) {
    for (int c = 0; c < C; ++c) {
      double pre = 0.0;
      for (int j = 0; j < 4; ++j) {
        int tau = t - 3 + j; /* source token */
        double xv;
        if (tau >= 0)
          xv = x[(size_t)tau * C + c];
        else
          xv = hist ? hist[(size_t)(tau + 3) * C + c] : 0.0;
        pre += w[(size_t)c * 4 + j] * xv;
      }
      y[(size_t)t * C + c] = pre * sigmoid(pre);
    }
  }
}

/* In-place L2 normalisation of each of L rows of length D: x / sqrt(sum x^2 + eps). */
void gdn_ref_l2norm(int L, int D, double eps, double *x) {
  for (int t = 0; t < L; ++t) {
    double ss = 0.0;
    for (int i = 0; i < D; ++i) ss += x[(size_t)t * D + i] * x[(size_t)t * D + i];
    double inv = 1.0 / sqrt(ss + eps);
    for (int i = 0; i < D; ++i) x[(size_t)t * D + i] *= inv;
  }
}

/* Gates of one value head: g_t = -exp(A_log) softplus(a_t + dt_bias), beta_t = sigmoid(b_t). */
void gdn_ref_gates(int L, const double *a, const double *b, double A_log, double dt_bias,
                   double *g, double *beta) {
  for (int t = 0; t < L; ++t) {
    g[t] = -exp(A_log) * softplus(a[t] + dt_bias);
    beta[t] = sigmoid(b[t]);
  }
}

/*
 * The gated delta rule, token by token, for one chain.
 * q, k: [L][dk] (already normalised); v: [L][dv]; g, beta: [L];
 * H0: [dk][dv] entering state (NULL = zeros); o: [L][dv] output (scaled by
 * `scale`); Hf: [dk][dv] state after the last token.  Hf may alias H0.
 */
void gdn_ref_recurrence(int L, int dk, int dv, double scale, const double *q,
                        const double *k, const double *v, const double *g,
                        const double *beta, const double *H0, double *o, double *Hf) {
  double *H = (double *)malloc(sizeof(double) * (size_t)dk * dv);
  double *p = (double *)malloc(sizeof(double) * (size_t)dv);
  double *u = (double *)malloc(sizeof(double) * (size_t)dv);
  if (H0)
    memcpy(H, H0, sizeof(double) * (size_t)dk * dv);
  else
    memset(H, 0, sizeof(double) * (size_t)dk * dv);
  for (int t = 0; t < L; ++t) {
    const double *kt = k + (size_t)t * dk, *qt = q + (size_t)t * dk, *vt = v + (size_t)t * dv;
    double alpha = exp(g[t]);
    /* p = H^T k */
    for (int j = 0; j < dv; ++j) {
      double s = 0.0;
      for (int i = 0; i < dk; ++i) s += H[(size_t)i * dv + j] * kt[i];
      p[j] = s;
    }
    /* u = beta (v - alpha p) */
    for (int j = 0; j < dv; ++j) u[j] = beta[t] * (vt[j] - alpha * p[j]);
    /* H <- alpha H + k u^T */
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j)
        H[(size_t)i * dv + j] = alpha * H[(size_t)i * dv + j] + kt[i] * u[j];
    /* o = H^T q * scale */
    for (int j = 0; j < dv; ++j) {
      double s = 0.0;
      for (int i = 0; i < dk; ++i) s += H[(size_t)i * dv + j] * qt[i];
      o[(size_t)t * dv + j] = s * scale;
    }
  }
  memcpy(Hf, H, sizeof(double) * (size_t)dk * dv);
  free(H);
  free(p);
  free(u);
}

/*
 * The same recurrence in chunked (WY/UT) form, chunk length C; the last chunk
 * may be shorter.  Within a chunk of n rows r = 0..n-1 entering with state H:
 *   G_r   = g_0 + ... + g_r,            gamma_r = exp(G_r)
 *   A[r][s] = beta_r exp(G_r - G_s) (k_r . k_s)        for s < r, else 0
 *   T     = (I + A)^-1                  (unit lower triangular; forward substitution)
 *   W     = T diag(beta gamma) K,       U' = T diag(beta) V
 *   U     = U' - W H                    (row r of U is the u_r of the token form)
 *   O     = scale (diag(gamma) Q H + (Q K^T o D) U),  D[r][s] = exp(G_r - G_s) for s <= r
 *   H    <- gamma_{n-1} H + sum_s exp(G_{n-1} - G_s) k_s u_s^T
 * The decay between two rows is always formed as exp(G_r - G_s) with r >= s,
 * never as a ratio exp(G_r) / exp(G_s) (both factors can underflow to zero
 * inside one chunk); a decay from the chunk start, exp(G_r), may underflow to
 * zero, which is then its correctly rounded value.
 */
void gdn_ref_recurrence_chunked(int L, int dk, int dv, int C, double scale, const double *q,
                                const double *k, const double *v, const double *g,
                                const double *beta, const double *H0, double *o, double *Hf) {
  double *H = (double *)malloc(sizeof(double) * (size_t)dk * dv);
  double *G = (double *)malloc(sizeof(double) * (size_t)C);
  double *A = (double *)malloc(sizeof(double) * (size_t)C * C);
  double *T = (double *)malloc(sizeof(double) * (size_t)C * C);
  double *W = (double *)malloc(sizeof(double) * (size_t)C * dk);
  double *U = (double *)malloc(sizeof(double) * (size_t)C * dv);
  double *Hn = (double *)malloc(sizeof(double) * (size_t)dk * dv);
  double *QK = (double *)malloc(sizeof(double) * (size_t)C * C);
  if (H0)
    memcpy(H, H0, sizeof(double) * (size_t)dk * dv);
  else
    memset(H, 0, sizeof(double) * (size_t)dk * dv);

  for (int c0 = 0; c0 < L; c0 += C) {
    int n = (L - c0 < C) ? (L - c0) : C;
    const double *Kc = k + (size_t)c0 * dk, *Qc = q + (size_t)c0 * dk, *Vc = v + (size_t)c0 * dv;
    const double *gc = g + c0, *bc = beta + c0;
    double acc = 0.0;
    for (int r = 0; r < n; ++r) {
      acc += gc[r];
      G[r] = acc;
    }
    /* A (strictly lower) */
    for (int r = 0; r < n; ++r)
      for (int s = 0; s < n; ++s) {
        double val = 0.0;
        if (s < r) {
          double kk = 0.0;
          for (int i = 0; i < dk; ++i) kk += Kc[(size_t)r * dk + i] * Kc[(size_t)s * dk + i];
          val = bc[r] * exp(G[r] - G[s]) * kk;
        }
        A[(size_t)r * C + s] = val;
      }
    /* T = (I + A)^-1 by forward substitution, one column at a time */
    for (int s = 0; s < n; ++s)
      for (int r = 0; r < n; ++r) {
        double val = (r == s) ? 1.0 : 0.0;
        for (int m = 0; m < r; ++m) val -= A[(size_t)r * C + m] * T[(size_t)m * C + s];
        T[(size_t)r * C + s] = val;
      }
    /* W = T diag(beta gamma) K ;  U = T diag(beta) V - W H */
    for (int r = 0; r < n; ++r) {
      for (int i = 0; i < dk; ++i) {
        double s_ = 0.0;
        for (int m = 0; m < n; ++m) s_ += T[(size_t)r * C + m] * bc[m] * exp(G[m]) * Kc[(size_t)m * dk + i];
        W[(size_t)r * dk + i] = s_;
      }
      for (int j = 0; j < dv; ++j) {
        double s_ = 0.0;
        for (int m = 0; m < n; ++m) s_ += T[(size_t)r * C + m] * bc[m] * Vc[(size_t)m * dv + j];
        double wh = 0.0;
        for (int i = 0; i < dk; ++i) wh += W[(size_t)r * dk + i] * H[(size_t)i * dv + j];
        U[(size_t)r * dv + j] = s_ - wh;
      }
    }
    /* O = scale (diag(gamma) Q H + (Q K^T o D) U) */
    for (int r = 0; r < n; ++r)
      for (int s = 0; s <= r; ++s) {
        double qk = 0.0;
        for (int i = 0; i < dk; ++i) qk += Qc[(size_t)r * dk + i] * Kc[(size_t)s * dk + i];
        QK[(size_t)r * C + s] = qk * exp(G[r] - G[s]);
      }
    for (int r = 0; r < n; ++r)
      for (int j = 0; j < dv; ++j) {
        double inter = 0.0;
        for (int i = 0; i < dk; ++i) inter += Qc[(size_t)r * dk + i] * H[(size_t)i * dv + j];
        double intra = 0.0;
        for (int s = 0; s <= r; ++s) intra += QK[(size_t)r * C + s] * U[(size_t)s * dv + j];
        o[(size_t)(c0 + r) * dv + j] = scale * (exp(G[r]) * inter + intra);
      }
    /* H <- gamma_last H + sum_s exp(G_last - G_s) k_s u_s^T */
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) {
        double s_ = exp(G[n - 1]) * H[(size_t)i * dv + j];
        for (int m = 0; m < n; ++m) s_ += exp(G[n - 1] - G[m]) * Kc[(size_t)m * dk + i] * U[(size_t)m * dv + j];
        Hn[(size_t)i * dv + j] = s_;
      }
    memcpy(H, Hn, sizeof(double) * (size_t)dk * dv);
  }
  memcpy(Hf, H, sizeof(double) * (size_t)dk * dv);
  free(H);
  free(G);
  free(A);
  free(T);
  free(W);
  free(U);
  free(Hn);
  free(QK);
}

/* RMSNormGated on L rows of length dv: y = o / sqrt(mean(o^2) + eps) * w * silu(z). */
void gdn_ref_rmsnorm_gated(int L, int dv, double eps, const double *o, const double *z,
                           const double *w, double *y) {
  for (int t = 0; t < L; ++t) {
    double ss = 0.0;
    for (int j = 0; j < dv; ++j) ss += o[(size_t)t * dv + j] * o[(size_t)t * dv + j];
    double inv = 1.0 / sqrt(ss / dv + eps);
    for (int j = 0; j < dv; ++j) {
      double zz = z[(size_t)t * dv + j];
      y[(size_t)t * dv + j] = o[(size_t)t * dv + j] * inv * w[j] * (zz * sigmoid(zz));
    }
  }
}

/* ======================================================================
 * Backward pass (reverse mode) of each stage, for a scalar loss whose
 * gradient with respect to the layer output y is given (dy).  Each function
 * takes the stage's forward inputs again and the gradient of its outputs, and
 * returns (accumulates where noted) the gradient of its inputs.  They are the
 * chain rule applied to the definitions above, step by step in reverse order;
 * the tests pin them to central finite differences of the forward functions.
 * ====================================================================== */

/* RMSNormGated: y = o r w silu(z), r = 1 / sqrt(mean(o^2) + eps).
 *   dz  = dy o r w silu'(z),   silu'(z) = s (1 + z (1 - s)), s = sigmoid(z)
 *   dw += dy o r silu(z)       (accumulated over rows)
 *   do  = r c dy - o r^3 (sum_j dy_j o_j c_j) / dv,   c = w silu(z)       */
void gdn_ref_rmsnorm_gated_backward(int L, int dv, double eps, const double *o, const double *z,
                                    const double *w, const double *dy, double *d_o, double *dz,
                                    double *dw_acc) {
  for (int t = 0; t < L; ++t) {
    const double *ot = o + (size_t)t * dv, *zt = z + (size_t)t * dv, *gt = dy + (size_t)t * dv;
    double ss = 0.0;
    for (int j = 0; j < dv; ++j) ss += ot[j] * ot[j];
    double r = 1.0 / sqrt(ss / dv + eps);
    double dot = 0.0;
    for (int j = 0; j < dv; ++j) {
      double s = sigmoid(zt[j]);
      double c = w[j] * zt[j] * s;
      dot += gt[j] * ot[j] * c;
    }
    for (int j = 0; j < dv; ++j) {
      double s = sigmoid(zt[j]);
      double silu = zt[j] * s;
      double c = w[j] * silu;
      d_o[(size_t)t * dv + j] = r * c * gt[j] - ot[j] * r * r * r * dot / dv;
      dz[(size_t)t * dv + j] = gt[j] * ot[j] * r * w[j] * s * (1.0 + zt[j] * (1.0 - s));
      dw_acc[j] += gt[j] * ot[j] * r * silu;
    }
  }
}

/*
 * The gated delta rule in reverse, for one chain.  Forward (per token t, H
 * entering as H_{t-1}): p = H^T k, u = beta (v - alpha p), H_t = alpha H +
 * k u^T, o_t = scale H_t^T q, alpha = exp(g).  Given do [L][dv] (gradient of
 * o) and dHf [dk][dv] (gradient of the final state, NULL = 0), returns dq,
 * dk [L][dk], dv [L][dv], dg, dbeta [L] and dH0 [dk][dv] (gradient of the
 * entering state).  The states H_t are recomputed forward first (kept for all
 * t: L (dk dv) doubles of scratch).  Reverse step t, with G the gradient of H_t:
 *   G   += scale q_t do_t^T ;          dq_t = scale H_t do_t
 *   dalpha = <G, H_{t-1}> ;            du = G^T k ;       dk_t = G u
 *   dbeta = du . (v - alpha p) ;       dv_t = beta du ;   dalpha -= beta du . p
 *   dp = -alpha beta du ;              dk_t += H_{t-1} dp
 *   G <- alpha G + k dp^T   (the gradient of H_{t-1}) ;  dg_t = alpha dalpha
 */
void gdn_ref_recurrence_backward(int L, int dk, int dv, double scale, const double *q, const double *k,
                                 const double *v, const double *g, const double *beta, const double *H0,
                                 const double *d_o, const double *dHf, double *dq, double *dkk, double *dvv,
                                 double *dg, double *dbeta, double *dH0) {
  size_t S = (size_t)dk * dv;
  double *Hs = (double *)malloc(sizeof(double) * S * (size_t)(L + 1)); /* Hs[t] = state before token t */
  double *G = (double *)malloc(sizeof(double) * S);
  double *p = (double *)malloc(sizeof(double) * (size_t)dv);
  double *u = (double *)malloc(sizeof(double) * (size_t)dv);
  double *du = (double *)malloc(sizeof(double) * (size_t)dv);
  double *dp = (double *)malloc(sizeof(double) * (size_t)dv);
  if (H0)
    memcpy(Hs, H0, sizeof(double) * S);
  else
    memset(Hs, 0, sizeof(double) * S);
  for (int t = 0; t < L; ++t) { /* forward, keeping every state */
    const double *H = Hs + S * t;
    double *Hn = Hs + S * (t + 1);
    const double *kt = k + (size_t)t * dk, *vt = v + (size_t)t * dv;
    double alpha = exp(g[t]);
    for (int j = 0; j < dv; ++j) {
      double s = 0.0;
      for (int i = 0; i < dk; ++i) s += H[(size_t)i * dv + j] * kt[i];
      u[j] = beta[t] * (vt[j] - alpha * s);
    }
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) Hn[(size_t)i * dv + j] = alpha * H[(size_t)i * dv + j] + kt[i] * u[j];
  }
  if (dHf)
    memcpy(G, dHf, sizeof(double) * S);
  else
    memset(G, 0, sizeof(double) * S);
  for (int t = L - 1; t >= 0; --t) {
    const double *Hp = Hs + S * t, *Ht = Hs + S * (t + 1);
    const double *qt = q + (size_t)t * dk, *kt = k + (size_t)t * dk, *vt = v + (size_t)t * dv;
    const double *ot = d_o + (size_t)t * dv;
    double alpha = exp(g[t]);
    /* output: o_t = scale H_t^T q_t */
    for (int i = 0; i < dk; ++i) {
      double s = 0.0;
      for (int j = 0; j < dv; ++j) {
        G[(size_t)i * dv + j] += scale * qt[i] * ot[j];
        s += Ht[(size_t)i * dv + j] * ot[j];
      }
      dq[(size_t)t * dk + i] = scale * s;
    }
    /* recompute p and u of token t */
    for (int j = 0; j < dv; ++j) {
      double s = 0.0;
      for (int i = 0; i < dk; ++i) s += Hp[(size_t)i * dv + j] * kt[i];
      p[j] = s;
      u[j] = beta[t] * (vt[j] - alpha * s);
    }
    /* H_t = alpha H_{t-1} + k u^T */
    double dalpha = 0.0;
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) dalpha += G[(size_t)i * dv + j] * Hp[(size_t)i * dv + j];
    for (int j = 0; j < dv; ++j) {
      double s = 0.0;
      for (int i = 0; i < dk; ++i) s += G[(size_t)i * dv + j] * kt[i];
      du[j] = s;
    }
    for (int i = 0; i < dk; ++i) {
      double s = 0.0;
      for (int j = 0; j < dv; ++j) s += G[(size_t)i * dv + j] * u[j];
      dkk[(size_t)t * dk + i] = s;
    }
    /* u = beta (v - alpha p) */
    double db = 0.0, dup = 0.0;
    for (int j = 0; j < dv; ++j) {
      db += du[j] * (vt[j] - alpha * p[j]);
      dup += du[j] * p[j];
      dvv[(size_t)t * dv + j] = beta[t] * du[j];
      dp[j] = -alpha * beta[t] * du[j];
    }
    dalpha -= beta[t] * dup;
    dbeta[t] = db;
    /* p = H_{t-1}^T k */
    for (int i = 0; i < dk; ++i) {
      double s = 0.0;
      for (int j = 0; j < dv; ++j) s += Hp[(size_t)i * dv + j] * dp[j];
      dkk[(size_t)t * dk + i] += s;
    }
    /* the gradient of H_{t-1} */
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) G[(size_t)i * dv + j] = alpha * G[(size_t)i * dv + j] + kt[i] * dp[j];
    dg[t] = alpha * dalpha;
  }
  memcpy(dH0, G, sizeof(double) * S);
  free(Hs);
  free(G);
  free(p);
  free(u);
  free(du);
  free(dp);
}

/* L2 normalisation x / sqrt(sum x^2 + eps), row-wise, in reverse: with
 * n = sqrt(sum x^2 + eps) and y = x / n,  dx = (dy - y (y . dy)) / n.
 * x [L][D] is the forward input; dy in, dx out. */
void gdn_ref_l2norm_backward(int L, int D, double eps, const double *x, const double *dy, double *dx) {
  for (int t = 0; t < L; ++t) {
    const double *xt = x + (size_t)t * D, *gt = dy + (size_t)t * D;
    double ss = 0.0;
    for (int i = 0; i < D; ++i) ss += xt[i] * xt[i];
    double n = sqrt(ss + eps);
    double yg = 0.0;
    for (int i = 0; i < D; ++i) yg += (xt[i] / n) * gt[i];
    for (int i = 0; i < D; ++i) dx[(size_t)t * D + i] = (gt[i] - (xt[i] / n) * yg) / n;
  }
}

/* conv(4) + SiLU in reverse (see gdn_ref_conv_silu for the forward).  dy is
 * the gradient of silu(pre); with dpre = dy silu'(pre):
 *   dx[tau][c]   += dpre[t][c] w[c][j]     (tau = t - 3 + j >= 0)
 *   dhist[m][c]  += dpre[t][c] w[c][j]     (tau = m - 3 < 0; dhist may be NULL)
 *   dw[c][j]     += dpre[t][c] x_tau[c]    (x_tau from hist before the start)
 * dx, dhist and dw are accumulated. */
void gdn_ref_conv_silu_backward(int L, int C, const double *x, const double *w, const double *hist,
                                const double *dy, double *dx, double *dhist, double *dw) {
  for (int t = 0; t < L; ++t) {
    for (int c = 0; c < C; ++c) {
      double pre = 0.0;
      for (int j = 0; j < 4; ++j) {
        int tau = t - 3 + j;
        double xv = tau >= 0 ? x[(size_t)tau * C + c] : (hist ? hist[(size_t)(tau + 3) * C + c] : 0.0);
        pre += w[(size_t)c * 4 + j] * xv;
      }
      double s = sigmoid(pre);
      double dpre = dy[(size_t)t * C + c] * s * (1.0 + pre * (1.0 - s));
      for (int j = 0; j < 4; ++j) {
        int tau = t - 3 + j;
        double xv;
        if (tau >= 0) {
          xv = x[(size_t)tau * C + c];
          dx[(size_t)tau * C + c] += dpre * w[(size_t)c * 4 + j];
        } else {
          xv = hist ? hist[(size_t)(tau + 3) * C + c] : 0.0;
          if (dhist) dhist[(size_t)(tau + 3) * C + c] += dpre * w[(size_t)c * 4 + j];
        }
        dw[(size_t)c * 4 + j] += dpre * xv;
      }
    }
  }
}

/* Gates in reverse: g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b).
 *   da_t = dg_t (-exp(A_log)) sigmoid(a_t + dt_bias) ;  ddt_bias += da_t
 *   dA_log += dg_t g_t ;  db_t = dbeta_t beta_t (1 - beta_t)
 * da, db [L] out; dA_log, ddt_bias accumulated (one value head). */
void gdn_ref_gates_backward(int L, const double *a, const double *b, double A_log, double dt_bias,
                            const double *dg, const double *dbeta, double *da, double *db,
                            double *dA_log_acc, double *ddt_bias_acc) {
  for (int t = 0; t < L; ++t) {
    double x = a[t] + dt_bias;
    double g = -exp(A_log) * softplus(x);
    da[t] = dg[t] * (-exp(A_log)) * sigmoid(x);
    *ddt_bias_acc += da[t];
    *dA_log_acc += dg[t] * g;
    double be = sigmoid(b[t]);
    db[t] = dbeta[t] * be * (1.0 - be);
  }
}

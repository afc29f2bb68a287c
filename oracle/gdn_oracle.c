/*
 * gdn_oracle.c -- fp64 CPU oracle for the batched Gated-DeltaNet decode step.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this file. The CUDA library shares no code, header or
 * constant with it, and it never calls into the CUDA library.
 *
 * Sources (page title, then the section / equation it follows):
 *   [EVO]  "深度解析线性注意力机制演进与 AI Infra 实现" (linear-attention evolution
 *          article): sections "去掉分母引入卷积" (short conv + SiLU, conv_state),
 *          "DeltaNet：写门与残差写入", "GDN：增加遗忘门", "KDA: By Channel的遗忘门",
 *          "KDA实现逻辑概述" (decay first, residual, outer-product write, readout),
 *          appendix "附2: 为什么要L2 Norm" (L2 normalisation with an epsilon).
 *   [LOG]  "DeltaLog：延迟物化递归状态以加速线性注意力解码" (reading notes on the
 *          DeltaLog paper): Sec. 1.1 Eqs. (2)-(3) (diagonal decay plus outer
 *          product), Sec. 2.2 Eq. (7) (base + log invariant), Sec. 2.3
 *          Algorithm 1 and Eq. (6) (append / merge), Sec. 2.4 (delta-rule
 *          factors a_t = k_t, b_t = beta_t (v_t - vhat_t)).
 *
 * Conventions. The state of one (request, head) is S[dk][dv], row-major, dv
 * contiguous; the readout is o = S^T q ([LOG] Sec. 1.1 writes S in R^{dk x dv}
 * and o = q^T S). A log-decay lambda has width dlam: 1 for a per-head scalar
 * (GDN), dk for a per-key-channel vector (KDA); D(l) = diag(exp(l)) scales the
 * ROWS (key index) of S.
 *
 * Everything here is fp64 and written for a reader to check against the
 * pages, not for speed: no blocking, no fusion, no reordering.
 *
 * Readings where the pages are silent or disagree (each is also listed in the
 * design notes):
 *   - The delta correction reads the DECAYED previous state: [EVO] "GDN" says
 *     the old memory decays first and the reconstruction error is taken on the
 *     decayed memory, and its KDA pseudo-code decays S before computing
 *     v - S k. [LOG] Sec. 2.4 writes vhat = S_{t-1}^T k; here S_{t-1} is read
 *     as "the state that enters the correction", i.e. D(lambda_t) S_{t-1}.
 *   - L2 normalisation divides by sqrt(sum x^2 + eps); the value of eps is not
 *     printed and is a parameter.
 *   - q is multiplied by q_scale after normalisation ([EVO] "KDA实现逻辑概述"
 *     applies head_dim^{-1/2}); 1.0 reproduces o = S^T q exactly.
 *   - Conv taps: column 0 of conv_state is the oldest input; conv weight
 *     column j multiplies the input j steps before "current minus 3"; an
 *     optional per-channel bias is added before SiLU.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Flags (oracle-local; the CUDA library defines its own). */
#define ORC_CONV 1u         /* q,k,v come from the causal conv1d + SiLU of mixed_qkv */
#define ORC_L2NORM 2u       /* L2-normalise q and k per head */
#define ORC_PLAIN 4u        /* additive update: b = beta * v, no delta correction */
#define ORC_GATE_RAW 8u     /* lambda = logsigmoid(a), beta = sigmoid(b_raw) */
#define ORC_KLOG_PRENORM 16u /* log key factor = pre-normalisation key, value factor scaled */
#define ORC_GATE_KDA 32u     /* lambda from the KDA gate parametrisation, beta = sigmoid(logit) */
#define ORC_OUT_NORM_GATE 64u /* o <- RMSNorm(o) * w * sigmoid(g) per head */

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_SLOT 2
#define ORC_ERR_LOG 3

#define CONV_K 4 /* width of the causal short convolution */

typedef struct {
  int32_t batch, num_heads, dk, dv, num_slots;
  int32_t dlam;         /* 1: per-head scalar log-decay; dk: per-key-channel */
  int32_t log_capacity; /* C = M - 1 entries of the DeltaLog log */
  uint32_t flags;
  double q_scale, l2_eps;
} orc_cfg;

/* Optional per-head inputs of the KDA gate and output epilogue ([EVO] "KDA实现逻辑概述"). */
typedef struct {
  const double *a_log;      /* [H] */
  const double *dt_bias;    /* [H][dlam] */
  const double *out_gate;   /* [B][H][dv] output-gate logits */
  const double *out_norm_w; /* [dv] RMSNorm weight, or NULL (1) */
  double lower_bound;       /* lambda lies in (lower_bound, 0) */
  double out_eps;           /* RMSNorm epsilon */
} orc_kda;

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

static double orc_silu(double z) { return z / (1.0 + exp(-z)); }
static double orc_sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* KDA forget-gate parametrisation ([EVO] "KDA实现逻辑概述", the forget-gate block):
 *   x = f + dt_bias,  z = exp(A_log) * x,  lambda = lower_bound * sigmoid(z),
 * so lambda lies in (lower_bound, 0) and alpha = exp(lambda) in (e^lower_bound, 1). */
double orc_kda_log_decay(double f, double a_log, double dt_bias, double lower_bound) {
  const double x = f + dt_bias;
  const double z = exp(a_log) * x;
  return lower_bound * orc_sigmoid(z);
}

/* KDA output epilogue ([EVO] "KDA实现逻辑概述": o <- RMSNorm(o) (.) gamma with the output
 * gate gamma = sigmoid(g)): y_j = o_j / sqrt(mean_j(o_j^2) + eps) * w_j * sigmoid(g_j),
 * the mean over the dv channels of one head; w = NULL means w_j = 1. y may alias o. */
void orc_out_norm_gate(int dv, const double *o, const double *g, const double *w, double eps,
                       double *y) {
  double ss = 0.0;
  for (int j = 0; j < dv; ++j) ss += o[j] * o[j];
  const double inv = 1.0 / sqrt(ss / dv + eps);
  for (int j = 0; j < dv; ++j) y[j] = o[j] * inv * (w ? w[j] : 1.0) * orc_sigmoid(g[j]);
}
static double orc_log_sigmoid(double z) {
  return z < 0.0 ? z - log1p(exp(z)) : -log1p(exp(-z));
}

/* ---------------------------------------------------------------------------
 * Short causal convolution, one token, all channels of one request.
 * [EVO] "去掉分母引入卷积": output = SiLU(x_{t-3} w[:,0] + x_{t-2} w[:,1] +
 * x_{t-1} w[:,2] + x_t w[:,3]); the cache keeps the last conv_kernel-1 = 3
 * PRE-conv inputs (conv outputs are not stored).
 *   x    [nch]        current pre-conv input
 *   cs   [nch][3]     conv_state, column 0 oldest; updated in place
 *   w    [nch][4]     conv weight
 *   bias [nch] or NULL
 *   y    [nch]        SiLU(conv) output
 * ------------------------------------------------------------------------- */
void orc_conv1d_silu(int nch, const double *x, double *cs, const double *w,
                     const double *bias, double *y) {
  for (int c = 0; c < nch; ++c) {
    double acc = 0.0;
    for (int j = 0; j < CONV_K - 1; ++j) acc += cs[c * 3 + j] * w[c * CONV_K + j];
    acc += x[c] * w[c * CONV_K + 3];
    if (bias) acc += bias[c];
    y[c] = orc_silu(acc);
    cs[c * 3 + 0] = cs[c * 3 + 1];
    cs[c * 3 + 1] = cs[c * 3 + 2];
    cs[c * 3 + 2] = x[c];
  }
}

/* ---------------------------------------------------------------------------
 * Widened conv window of a speculative-decoding verify round, one request
 * ([HB] "推测解码：验证后如何恢复状态": the conv cache is widened to
 * conv_kernel - 1 + num_spec inputs, the round's candidates are appended at its
 * end, and the next round reads it at offset num_accepted - 1).
 * With T = 1 + num_spec positions the window holds W = (CONV_K - 1) + (T - 1)
 * PRE-conv inputs per channel, column 0 oldest. A round that enters with
 * na = num_accepted (1 <= na <= T) takes the CONV_K - 1 inputs before its first
 * position from columns na-1 .. na+1, convolves its T inputs with them
 * (orc_conv1d_silu, one token at a time), and leaves in the window the last W
 * inputs of that sequence: columns na and na+1, then its own T inputs.
 *   win  [nch][W]  updated in place
 *   x    [T][nch]  pre-conv inputs of the round
 *   w    [nch][4], bias [nch] or NULL
 *   y    [T][nch]  SiLU(conv) outputs
 * Returns ORC_OK, or ORC_ERR_ARG when na is outside [1, T].
 * ------------------------------------------------------------------------- */
int orc_verify_conv_window(int nch, int T, int na, double *win, const double *x,
                           const double *w, const double *bias, double *y) {
  if (T < 1 || na < 1 || na > T) return ORC_ERR_ARG;
  const int W = (CONV_K - 1) + (T - 1);
  const int off = na - 1;
  double *cs = (double *)malloc(sizeof(double) * (size_t)nch * 3);
  double *seq = (double *)malloc(sizeof(double) * (size_t)nch * (size_t)(T + CONV_K - 1));
  if (!cs || !seq) {
    free(cs);
    free(seq);
    return ORC_ERR_ARG;
  }
  /* the inputs the round sees, oldest first: the three before it, then its own */
  for (int c = 0; c < nch; ++c) {
    for (int j = 0; j < CONV_K - 1; ++j) {
      cs[c * 3 + j] = win[(size_t)c * W + off + j];
      seq[(size_t)c * (T + CONV_K - 1) + j] = win[(size_t)c * W + off + j];
    }
    for (int t = 0; t < T; ++t) seq[(size_t)c * (T + CONV_K - 1) + CONV_K - 1 + t] = x[(size_t)t * nch + c];
  }
  for (int t = 0; t < T; ++t) orc_conv1d_silu(nch, x + (size_t)t * nch, cs, w, bias, y + (size_t)t * nch);
  /* keep the last W of the T + 3 inputs */
  for (int c = 0; c < nch; ++c)
    for (int i = 0; i < W; ++i) win[(size_t)c * W + i] = seq[(size_t)c * (T + CONV_K - 1) + (T + CONV_K - 1 - W) + i];
  free(cs);
  free(seq);
  return ORC_OK;
}

/* L2 normalisation ([EVO] appendix 附2): y = scale * x / sqrt(sum x^2 + eps).
 * Returns 1/sqrt(sum x^2 + eps), the factor that maps x to its unit vector. */
double orc_l2norm(int n, const double *x, double eps, double scale, double *y) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss + eps);
  for (int i = 0; i < n; ++i) y[i] = scale * x[i] * inv;
  return inv;
}

/* ---------------------------------------------------------------------------
 * One dense gated delta-rule step for one head ([EVO] "GDN", "KDA",
 * "KDA实现逻辑概述"; [LOG] Eq. (2)-(3) with a_t = k_t):
 *   S    <- D(lambda) S                    forget (rows = key channels)
 *   vhat  = S^T k                          read on the decayed state
 *   b     = beta (v - vhat)                (plain mode: b = beta v)
 *   S    <- S + k b^T                      outer-product write
 *   o     = S^T q                          post-update readout
 * ------------------------------------------------------------------------- */
void orc_gdn_step(int dk, int dv, double *S, const double *q, const double *k,
                  const double *v, const double *lam, int dlam, double beta,
                  int plain, double *o) {
  double *b = (double *)malloc(sizeof(double) * (size_t)dv);
  for (int d = 0; d < dk; ++d) {
    double a = exp(lam[dlam == 1 ? 0 : d]);
    for (int j = 0; j < dv; ++j) S[(size_t)d * dv + j] *= a;
  }
  for (int j = 0; j < dv; ++j) {
    double vhat = 0.0;
    for (int d = 0; d < dk; ++d) vhat += S[(size_t)d * dv + j] * k[d];
    b[j] = plain ? beta * v[j] : beta * (v[j] - vhat);
  }
  for (int d = 0; d < dk; ++d)
    for (int j = 0; j < dv; ++j) S[(size_t)d * dv + j] += k[d] * b[j];
  for (int j = 0; j < dv; ++j) {
    double acc = 0.0;
    for (int d = 0; d < dk; ++d) acc += S[(size_t)d * dv + j] * q[d];
    o[j] = acc;
  }
  free(b);
}

/* ---------------------------------------------------------------------------
 * One DeltaLog step for one head, following [LOG] Algorithm 1 literally.
 *
 * Physical state ([LOG] Sec. 2.1): base Sbar[dk][dv], cumulative log-decay
 * ell[dlam], key log Klog[C][dk], value log Ulog[C][dv], decay snapshots
 * Lam[C][dlam], length *L with 0 <= L <= C.
 *
 * The logical state is Eq. (7):
 *   S = D(ell) Sbar + sum_{i<L} D(ell - Lam[i]) Klog[i] Ulog[i]^T.
 *
 *   1. ell' = ell + lambda           (closure: D(lambda) D(ell) = D(ell+lambda))
 *   2. P = D(ell') Sbar + sum_i D(ell'-Lam[i]) Klog[i] Ulog[i]^T
 *      -- Eq. (7) evaluated at ell': the decayed previous state, materialised
 *         here as a full matrix (the oracle does not use the Sec. 2.4
 *         coefficient form that a fast kernel would use).
 *   3. vhat = P^T k; b = beta (v - vhat)  (plain: b = beta v)
 *   4. o = (P + k b^T)^T q                post-update readout
 *   5. if L < C on entry: append (a, b * bscale, ell') at position L, ell = ell',
 *      L = L + 1, base unchanged; else merge, Eq. (6): Sbar = P + k b^T,
 *      ell = 0, L = 0 (the current update goes straight into the merge).
 *
 * The log keeps a factor pair (a, b') of the update k b^T. By default
 * a = k and b' = b ([LOG] Sec. 2.4). In the pre-normalisation variant
 * a = the raw key and b' = s b, where s is the factor that normalised it, so
 * a b'^T = k b^T still holds; the caller passes a and bscale = s.
 * Returns ORC_OK, or ORC_ERR_LOG if *L is outside [0, C].
 * ------------------------------------------------------------------------- */
int orc_deltalog_step(int dk, int dv, int dlam, int C, double *Sbar, double *ell,
                      double *Klog, double *Ulog, double *Lam, int32_t *L,
                      const double *q, const double *k, const double *v,
                      const double *lam, double beta, int plain, const double *a,
                      double bscale, double *o) {
  int n = *L;
  if (n < 0 || n > C) return ORC_ERR_LOG;
  double *ellp = (double *)malloc(sizeof(double) * (size_t)dlam);
  double *P = (double *)malloc(sizeof(double) * (size_t)dk * dv);
  double *b = (double *)malloc(sizeof(double) * (size_t)dv);

  for (int e = 0; e < dlam; ++e) ellp[e] = ell[e] + lam[e];

  for (int d = 0; d < dk; ++d) {
    double ed = ellp[dlam == 1 ? 0 : d];
    for (int j = 0; j < dv; ++j) {
      double acc = exp(ed) * Sbar[(size_t)d * dv + j];
      for (int i = 0; i < n; ++i) {
        double lamid = Lam[(size_t)i * dlam + (dlam == 1 ? 0 : d)];
        acc += exp(ed - lamid) * Klog[(size_t)i * dk + d] * Ulog[(size_t)i * dv + j];
      }
      P[(size_t)d * dv + j] = acc;
    }
  }

  for (int j = 0; j < dv; ++j) {
    double vhat = 0.0;
    for (int d = 0; d < dk; ++d) vhat += P[(size_t)d * dv + j] * k[d];
    b[j] = plain ? beta * v[j] : beta * (v[j] - vhat);
  }
  for (int j = 0; j < dv; ++j) {
    double acc = 0.0;
    for (int d = 0; d < dk; ++d) acc += (P[(size_t)d * dv + j] + k[d] * b[j]) * q[d];
    o[j] = acc;
  }

  if (n < C) {
    for (int d = 0; d < dk; ++d) Klog[(size_t)n * dk + d] = a[d];
    for (int j = 0; j < dv; ++j) Ulog[(size_t)n * dv + j] = b[j] * bscale;
    for (int e = 0; e < dlam; ++e) Lam[(size_t)n * dlam + e] = ellp[e];
    for (int e = 0; e < dlam; ++e) ell[e] = ellp[e];
    *L = n + 1;
  } else {
    for (int d = 0; d < dk; ++d)
      for (int j = 0; j < dv; ++j) Sbar[(size_t)d * dv + j] = P[(size_t)d * dv + j] + k[d] * b[j];
    for (int e = 0; e < dlam; ++e) ell[e] = 0.0;
    *L = 0;
  }
  free(ellp);
  free(P);
  free(b);
  return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * One decode step over a whole batch (OpenMP over requests, then over
 * (request, head) pairs). Layouts mirror the pools of a serving system:
 *   slot      [B]                 row of every pool used by request b; < 0 = padding
 *   q, k      [B][H][dk], v [B][H][dv]      (ignored with ORC_CONV)
 *   mixed     [B][nch], nch = 2*H*dk + H*dv; channel order [q heads | k heads | v heads]
 *   conv_w    [nch][4], conv_b [nch] or NULL, conv_pool [num_slots][nch][3]
 *   lam       [B][H][dlam] (raw gate logits with ORC_GATE_RAW, the forget pre-activation f
 *             with ORC_GATE_KDA), beta [B][H] (logits with either)
 *   S_pool    [num_slots][H][dk][dv]  dense: the state; deltalog: the base
 *   ell       [num_slots][H][dlam], klog [num_slots][H][C][dk],
 *   ulog      [num_slots][H][C][dv], lamlog [num_slots][H][C][dlam], len [num_slots][H]
 *   kda       optional KDA gate and epilogue inputs (ORC_GATE_KDA, ORC_OUT_NORM_GATE)
 *   o         [B][H][dv]           rows of padding requests are left untouched
 * mode 0 = dense, 1 = DeltaLog (append if the log has room, else merge).
 * ------------------------------------------------------------------------- */
int orc_step_batch_ex(const orc_cfg *cfg, int mode, const int32_t *slot,
                      const double *q, const double *k, const double *v,
                      const double *mixed, const double *conv_w, const double *conv_b,
                      double *conv_pool, const double *lam, const double *beta,
                      double *S_pool, double *ell, double *klog, double *ulog,
                      double *lamlog, int32_t *len, const orc_kda *kda, double *o) {
  const int B = cfg->batch, H = cfg->num_heads, dk = cfg->dk, dv = cfg->dv;
  const int dlam = cfg->dlam, C = cfg->log_capacity;
  const uint32_t fl = cfg->flags;
  if (B < 0 || H <= 0 || dk <= 0 || dv <= 0 || (dlam != 1 && dlam != dk) || C < 0)
    return ORC_ERR_ARG;
  if ((fl & ORC_KLOG_PRENORM) && ((fl & ORC_CONV) || !(fl & ORC_L2NORM))) return ORC_ERR_ARG;
  if ((fl & ORC_GATE_KDA) && ((fl & ORC_GATE_RAW) || !kda || !kda->a_log || !kda->dt_bias))
    return ORC_ERR_ARG;
  if ((fl & ORC_OUT_NORM_GATE) && (!kda || !kda->out_gate)) return ORC_ERR_ARG;
  for (int b = 0; b < B; ++b)
    if (slot[b] >= cfg->num_slots) return ORC_ERR_SLOT;
  if (mode == 1)
    for (int b = 0; b < B; ++b)
      if (slot[b] >= 0)
        for (int h = 0; h < H; ++h) {
          int32_t n = len[(size_t)slot[b] * H + h];
          if (n < 0 || n > C) return ORC_ERR_LOG;
        }

  const int nch = 2 * H * dk + H * dv;
  double *y = NULL; /* conv outputs [B][nch] */
  if (fl & ORC_CONV) {
    y = (double *)malloc(sizeof(double) * (size_t)B * nch);
#pragma omp parallel for schedule(static)
    for (int b = 0; b < B; ++b) {
      if (slot[b] < 0) continue;
      orc_conv1d_silu(nch, mixed + (size_t)b * nch, conv_pool + (size_t)slot[b] * nch * 3,
                      conv_w, conv_b, y + (size_t)b * nch);
    }
  }

  int err = ORC_OK;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int b = 0; b < B; ++b) {
    for (int h = 0; h < H; ++h) {
      const int s = slot[b];
      if (s < 0) continue;
      const double *qr, *kr, *vr;
      if (fl & ORC_CONV) {
        const double *yb = y + (size_t)b * nch;
        qr = yb + (size_t)h * dk;
        kr = yb + (size_t)H * dk + (size_t)h * dk;
        vr = yb + (size_t)2 * H * dk + (size_t)h * dv;
      } else {
        qr = q + ((size_t)b * H + h) * dk;
        kr = k + ((size_t)b * H + h) * dk;
        vr = v + ((size_t)b * H + h) * dv;
      }
      double *qh = (double *)malloc(sizeof(double) * (size_t)dk);
      double *kh = (double *)malloc(sizeof(double) * (size_t)dk);
      double *lh = (double *)malloc(sizeof(double) * (size_t)dlam);
      double kinv = 1.0;
      if (fl & ORC_L2NORM) {
        orc_l2norm(dk, qr, cfg->l2_eps, cfg->q_scale, qh);
        kinv = orc_l2norm(dk, kr, cfg->l2_eps, 1.0, kh);
      } else {
        for (int d = 0; d < dk; ++d) qh[d] = cfg->q_scale * qr[d];
        for (int d = 0; d < dk; ++d) kh[d] = kr[d];
      }
      const double *lr = lam + ((size_t)b * H + h) * dlam;
      double bh = beta[(size_t)b * H + h];
      if (fl & ORC_GATE_RAW) {
        for (int e = 0; e < dlam; ++e) lh[e] = orc_log_sigmoid(lr[e]);
        bh = orc_sigmoid(bh);
      } else if (fl & ORC_GATE_KDA) {
        for (int e = 0; e < dlam; ++e)
          lh[e] = orc_kda_log_decay(lr[e], kda->a_log[h], kda->dt_bias[(size_t)h * dlam + e],
                                    kda->lower_bound);
        bh = orc_sigmoid(bh);
      } else {
        for (int e = 0; e < dlam; ++e) lh[e] = lr[e];
      }
      const size_t sh = (size_t)s * H + h;
      double *oh = o + ((size_t)b * H + h) * dv;
      double *S = S_pool + sh * dk * dv;
      if (mode == 0) {
        orc_gdn_step(dk, dv, S, qh, kh, vr, lh, dlam, bh, (fl & ORC_PLAIN) != 0, oh);
      } else {
        const double *a = (fl & ORC_KLOG_PRENORM) ? kr : kh;
        double bscale = (fl & ORC_KLOG_PRENORM) ? kinv : 1.0;
        int rc = orc_deltalog_step(dk, dv, dlam, C, S, ell + sh * dlam, klog + sh * C * dk,
                                   ulog + sh * C * dv, lamlog + sh * C * dlam, len + sh, qh,
                                   kh, vr, lh, bh, (fl & ORC_PLAIN) != 0, a, bscale, oh);
        if (rc != ORC_OK) {
#pragma omp atomic write
          err = rc;
        }
      }
      if (fl & ORC_OUT_NORM_GATE)
        orc_out_norm_gate(dv, oh, kda->out_gate + ((size_t)b * H + h) * dv, kda->out_norm_w,
                          kda->out_eps, oh);
      free(qh);
      free(kh);
      free(lh);
    }
  }
  free(y);
  return err;
}

/* orc_step_batch_ex without the KDA gate / epilogue inputs. */
int orc_step_batch(const orc_cfg *cfg, int mode, const int32_t *slot,
                   const double *q, const double *k, const double *v,
                   const double *mixed, const double *conv_w, const double *conv_b,
                   double *conv_pool, const double *lam, const double *beta,
                   double *S_pool, double *ell, double *klog, double *ulog,
                   double *lamlog, int32_t *len, double *o) {
  return orc_step_batch_ex(cfg, mode, slot, q, k, v, mixed, conv_w, conv_b, conv_pool, lam, beta,
                           S_pool, ell, klog, ulog, lamlog, len, NULL, o);
}

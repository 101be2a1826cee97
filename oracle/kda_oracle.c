/*
 * kda_oracle.c -- fp64 CPU oracle of the fused KDA decode step.
 *
 * TEST INFRASTRUCTURE ONLY (see kda_oracle.h): loaded by the tests, the
 * smoke check and the benchmark's CPU-baseline leg, never by the product.
 *
 * "P1" is the page "[ROCm][Perf] Kimi-K3 Fused kernel for KDA decode"
 * (vLLM PR #50654 report).  Each function names the stage of that page it
 * restates; the equations are the standard KDA definition written out in
 * kda_oracle.h, since P1 prints none.
 *
 * Plain loops, no blocking or fusion: every step is evaluated in the order
 * the formulation states it.  Built with -ffp-contract=off so x86 and Arm
 * hosts produce the same bits.
 */
#include "kda_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

int kda_oracle_problem_size(void) { return (int)sizeof(kda_oracle_problem); }

/* ---------------------------------------------------------------- dtypes */

double kda_oracle_bf16_to_f64(uint16_t b) {
  /* bf16 is the top half of an IEEE binary32. */
  uint32_t bits = (uint32_t)b << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

uint16_t kda_oracle_round_bf16(double x) {
  /* Direct round-to-nearest-even of an fp64 value onto the bf16 grid
   * (8 significant bits, exponent range of binary32). */
  if (isnan(x)) return 0x7FC0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (a == 0.0) return sign;
  if (isinf(a)) return (uint16_t)(sign | 0x7F80);
  int e;
  frexp(a, &e);               /* a in [2^(e-1), 2^e) */
  int qe = e - 8;             /* spacing of 8-significant-bit numbers there */
  if (qe < -133) qe = -133;   /* bf16 subnormal spacing 2^-133 */
  double q = ldexp(a, -qe);   /* exact; q < 2^8 */
  double fl = floor(q);
  double rem = q - fl;        /* exact */
  if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
  double r = ldexp(fl, qe);
  if (r > 3.3895313892515355e38) return (uint16_t)(sign | 0x7F80); /* > max finite */
  float f = (float)r;         /* exact: r is on the bf16 grid */
  uint32_t bits;
  memcpy(&bits, &f, sizeof bits);
  return (uint16_t)(sign | (uint16_t)(bits >> 16));
}

/* ---------------------------------------------------------------- steps */

double kda_oracle_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* Stage "causal conv1d state advance" (P1 功能与动机; 实现拆解 #1).  The
 * window is oldest-first and its last tap is the current token. */
double kda_oracle_causal_conv(const double* x, const double* w, int W, double bias) {
  double y = 0.0;
  for (int t = 0; t < W; ++t) y += w[t] * x[t];
  return y + bias;
}

double kda_oracle_silu(double y) { return y * kda_oracle_sigmoid(y); }

/* q/k L2 normalisation ahead of the delta rule (standard KDA; not on P1). */
void kda_oracle_l2norm(const double* x, int n, double eps, double scale, double* y) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss + eps);
  for (int i = 0; i < n; ++i) y[i] = scale * x[i] * inv;
}

/* Stage "gated delta-rule recurrence" on the [K, V] fp32 state (P1
 * 功能与动机; 实现拆解 #1):
 *   S' = (I - beta k k^T) Diag(alpha) S + beta k v^T.
 * Evaluated as A = Diag(alpha) S, u = A^T k (= k^T A), then
 * S' = A - beta k u^T + beta k v^T. */
void kda_oracle_gated_delta_update(int K, int V, double* S, const double* alpha,
                                   double beta, const double* k, const double* v) {
  for (int i = 0; i < K; ++i)
    for (int j = 0; j < V; ++j) S[(size_t)i * V + j] *= alpha[i];
  double* u = (double*)calloc((size_t)V, sizeof(double));
  for (int j = 0; j < V; ++j) {
    double acc = 0.0;
    for (int i = 0; i < K; ++i) acc += k[i] * S[(size_t)i * V + j];
    u[j] = acc;
  }
  for (int i = 0; i < K; ++i)
    for (int j = 0; j < V; ++j)
      S[(size_t)i * V + j] = S[(size_t)i * V + j] - beta * k[i] * u[j] + beta * k[i] * v[j];
  free(u);
}

/* Readout o = S^T q. */
void kda_oracle_readout(int K, int V, const double* S, const double* q, double* o) {
  for (int j = 0; j < V; ++j) {
    double acc = 0.0;
    for (int i = 0; i < K; ++i) acc += S[(size_t)i * V + j] * q[i];
    o[j] = acc;
  }
}

/* Stage "gated RMSNorm" (P1 功能与动机; 实现拆解 #3 for the fp32 norm
 * weight; the op's output_gate / norm_weight / norm_eps arguments in
 * 关键源码片段). */
void kda_oracle_gated_rmsnorm(int V, const double* o, const double* w,
                              const double* gate, double eps, double* y) {
  double ss = 0.0;
  for (int j = 0; j < V; ++j) ss += o[j] * o[j];
  double r = 1.0 / sqrt(ss / (double)V + eps);
  for (int j = 0; j < V; ++j) y[j] = o[j] * r * w[j] * kda_oracle_sigmoid(gate[j]);
}

/* Gate activation ahead of the recurrence when the kernel fuses it (P1
 * 实现拆解 item 1 "safe gate"; formula is the standard KDA gate, not on P1). */
double kda_oracle_softplus(double z) {
  /* log(1 + e^z), written so that neither branch overflows */
  return (z > 0.0) ? z + log1p(exp(-z)) : log1p(exp(z));
}

double kda_oracle_kda_gate(double z, double A_log, double lower_bound) {
  if (lower_bound < 0.0) return lower_bound * kda_oracle_sigmoid(exp(A_log) * z);
  return -exp(A_log) * kda_oracle_softplus(z);
}

/* ---------------------------------------------------------------- step */

/* One (row n, head h).  Returns 1 if the slot was out of range. */
static int decode_unit(const kda_oracle_problem* p, int n, int h, double* work) {
  const int H = p->H, K = p->K, V = p->V, W = p->W;
  const int64_t Dq = (int64_t)H * K, Dv = (int64_t)H * V, C = 2 * Dq + Dv;
  const int32_t s = p->slot_idx[n];
  uint16_t* out = p->out + (int64_t)n * Dv + (int64_t)h * V;
  double* out64 = p->out_f64 ? p->out_f64 + (int64_t)n * Dv + (int64_t)h * V : NULL;

  /* 0. Padding rows (P1 实现拆解 #1; kernel excerpt in 关键源码片段): zero
   *    output, no state or conv-state access. */
  if (s <= 0 || s >= p->num_slots) {
    for (int j = 0; j < V; ++j) {
      out[j] = 0;
      if (out64) out64[j] = 0.0;
    }
    return s >= p->num_slots;
  }

  double* qt = work;            /* K */
  double* kt = qt + K;          /* K */
  double* vt = kt + K;          /* V */
  double* qh = vt + V;          /* K */
  double* kh = qh + K;          /* K */
  double* alpha = kh + K;       /* K */
  double* o = alpha + K;        /* V */
  double* y = o + V;            /* V */
  double* gt = y + V;           /* V */
  double* nw = gt + V;          /* V */
  double* x = nw + V;           /* W */
  double* wt = x + W;           /* W */
  double* S = wt + W;           /* K*V */

  /* 1. Conv + SiLU per channel of the q, k, v blocks, then the shift. */
  for (int c = 0; c < 3; ++c) {
    const int dim_c = (c < 2) ? K : V;
    const int64_t D_c = (c < 2) ? Dq : Dv;
    const int64_t off_c = (c == 0) ? 0 : (c == 1) ? Dq : 2 * Dq;
    const float* wc = p->conv_weight + ((c == 0) ? 0 : (c == 1) ? (int64_t)W * Dq : 2 * (int64_t)W * Dq);
    double* dst = (c == 0) ? qt : (c == 1) ? kt : vt;
    for (int j = 0; j < dim_c; ++j) {
      const int64_t ch = off_c + (int64_t)h * dim_c + j;
      /* element (s, ch, t) of the conv state, in either layout */
      uint16_t* cs0 = p->conv_state + (int64_t)s * C * (W - 1);
      const int64_t cs_ch = p->conv_state_sd ? 1 : (W - 1);
      const int64_t cs_t = p->conv_state_sd ? C : 1;
#define CS(t) cs0[ch * cs_ch + (int64_t)(t) * cs_t]
      const uint16_t xin = p->qkv[(int64_t)n * p->qkv_row_stride + ch];
      for (int t = 0; t < W - 1; ++t) x[t] = kda_oracle_bf16_to_f64(CS(t));
      x[W - 1] = kda_oracle_bf16_to_f64(xin);
      for (int t = 0; t < W; ++t) wt[t] = (double)wc[(int64_t)t * D_c + (int64_t)h * dim_c + j];
      const double bias = p->conv_bias ? (double)p->conv_bias[ch] : 0.0;
      dst[j] = kda_oracle_silu(kda_oracle_causal_conv(x, wt, W, bias));
      if (p->update_conv_state && W > 1) {
        for (int t = 0; t < W - 2; ++t) CS(t) = CS(t + 1);
        CS(W - 2) = xin;
      }
#undef CS
    }
  }

  /* 2. L2 norms. */
  const double scale = (p->q_scale != 0.0) ? p->q_scale : 1.0 / sqrt((double)K);
  kda_oracle_l2norm(qt, K, p->l2_eps, scale, qh);
  kda_oracle_l2norm(kt, K, p->l2_eps, 1.0, kh);

  /* 3. Gated delta rule on the slot's state. */
  float* Sg = p->state + (((int64_t)s * H + h) * K) * V;
  for (int64_t e = 0; e < (int64_t)K * V; ++e) S[e] = (double)Sg[e];
  double beta = kda_oracle_bf16_to_f64(p->beta[(int64_t)n * H + h]);
  if (p->fused_gate) {
    /* the gate activation replaces the pre-activated g and beta */
    const double a_log = (double)p->A_log[h];
    for (int i = 0; i < K; ++i) {
      double z = (double)p->g[((int64_t)n * H + h) * K + i];
      if (p->dt_bias) z += (double)p->dt_bias[(int64_t)h * K + i];
      alpha[i] = exp(kda_oracle_kda_gate(z, a_log, p->lower_bound));
    }
    beta = kda_oracle_sigmoid(beta);
  } else {
    for (int i = 0; i < K; ++i) alpha[i] = exp((double)p->g[((int64_t)n * H + h) * K + i]);
  }
  kda_oracle_gated_delta_update(K, V, S, alpha, beta, kh, vt);

  /* 4. Readout from the updated state. */
  kda_oracle_readout(K, V, S, qh, o);

  /* 5. Gated RMSNorm, or the raw readout. */
  if (p->out_norm) {
    for (int j = 0; j < V; ++j) {
      gt[j] = kda_oracle_bf16_to_f64(p->gate[(int64_t)n * Dv + (int64_t)h * V + j]);
      nw[j] = (double)p->norm_weight[j];
    }
    kda_oracle_gated_rmsnorm(V, o, nw, gt, p->eps, y);
  } else {
    for (int j = 0; j < V; ++j) y[j] = o[j];
  }

  /* 6. Round and store. */
  for (int j = 0; j < V; ++j) {
    out[j] = kda_oracle_round_bf16(y[j]);
    if (out64) out64[j] = y[j];
  }
  for (int64_t e = 0; e < (int64_t)K * V; ++e) Sg[e] = (float)S[e];
  return 0;
}

int kda_oracle_decode(const kda_oracle_problem* p, int num_threads) {
  if (!p || p->N < 0 || p->H < 1 || p->K < 1 || p->V < 1 || p->W < 1 || p->num_slots < 1) return -1;
  if (p->N == 0) return 0;
  if (!p->qkv || !p->conv_weight || !p->conv_state || !p->state || !p->g || !p->beta ||
      !p->slot_idx || !p->out)
    return -1;
  if (p->out_norm && (!p->gate || !p->norm_weight)) return -1;
  if (p->fused_gate && !p->A_log) return -1;
  const int64_t C = 2 * (int64_t)p->H * p->K + (int64_t)p->H * p->V;
  if (p->qkv_row_stride < C) return -1;

  const int64_t units = (int64_t)p->N * p->H;
  const size_t work_len = (size_t)(5 * p->K + 5 * p->V + 2 * p->W) + (size_t)p->K * p->V;
  int oob = 0;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#else
  (void)num_threads;
#endif
#pragma omp parallel reduction(+ : oob)
  {
    double* work = (double*)malloc(work_len * sizeof(double));
#pragma omp for schedule(dynamic, 16)
    for (int64_t u = 0; u < units; ++u) {
      const int n = (int)(u / p->H), h = (int)(u % p->H);
      const int r = decode_unit(p, n, h, work);
      if (h == 0) oob += r; /* count rows, not (row, head) pairs */
    }
    free(work);
  }
  return oob;
}

/* ---------------------------------------------------------------- prefill */

int kda_oracle_prefill_problem_size(void) { return (int)sizeof(kda_oracle_prefill_problem); }

/* One (sequence b, head h) of the prefill: the decode steps token by token,
 * the window and the state carried along (P2 实现拆解 #2-#3 for the varlen
 * batch; steps as in the decode formulation).  Returns 1 if the slot was out
 * of range. */
static int prefill_unit(const kda_oracle_prefill_problem* p, int b, int h, double* work) {
  const int H = p->H, K = p->K, V = p->V, W = p->W;
  const int64_t Dq = (int64_t)H * K, Dv = (int64_t)H * V, C = 2 * Dq + Dv;
  const int32_t r0 = p->cu_seqlens[b], r1 = p->cu_seqlens[b + 1];
  const int32_t s = p->slot_idx[b];
  if (r1 <= r0) return 0; /* empty sequence: nothing to do */

  if (s < 1 || s >= p->num_slots) { /* padding or out of range */
    for (int32_t r = r0; r < r1; ++r)
      for (int j = 0; j < V; ++j) {
        p->out[(int64_t)r * Dv + (int64_t)h * V + j] = 0;
        if (p->out_f64) p->out_f64[(int64_t)r * Dv + (int64_t)h * V + j] = 0.0;
      }
    return s >= p->num_slots;
  }

  double* qt = work;            /* K */
  double* kt = qt + K;          /* K */
  double* vt = kt + K;          /* V */
  double* qh = vt + V;          /* K */
  double* kh = qh + K;          /* K */
  double* alpha = kh + K;       /* K */
  double* o = alpha + K;        /* V */
  double* y = o + V;            /* V */
  double* gt = y + V;           /* V */
  double* nw = gt + V;          /* V */
  double* x = nw + V;           /* W */
  double* wt = x + W;           /* W */
  double* S = wt + W;           /* K*V */
  uint16_t* win = (uint16_t*)(S + (size_t)K * V); /* (2K+V) channels x (W-1) taps, oldest first */

  /* the head's channels of the three blocks, in q | k | v order */
  const int dims[3] = {K, K, V};
  const int64_t offs[3] = {0, Dq, 2 * Dq};
  const int64_t Ds[3] = {Dq, Dq, Dv};
  const float* wbase[3] = {p->conv_weight, p->conv_weight + (int64_t)W * Dq, p->conv_weight + 2 * (int64_t)W * Dq};
  uint16_t* cs0 = p->conv_state + (int64_t)s * C * (W - 1);

  /* element (ch, t) of the slot's conv state in either layout */
  const int64_t cs_ch = p->conv_state_sd ? 1 : (W - 1);
  const int64_t cs_t = p->conv_state_sd ? C : 1;
  /* window <- the slot's conv state */
  for (int c = 0, m = 0; c < 3; ++c)
    for (int j = 0; j < dims[c]; ++j, ++m) {
      const int64_t ch = offs[c] + (int64_t)h * dims[c] + j;
      for (int t = 0; t < W - 1; ++t) win[(size_t)m * (W - 1) + t] = cs0[ch * cs_ch + t * cs_t];
    }

  float* Sg = p->state + (((int64_t)s * H + h) * K) * V;
  for (int64_t e = 0; e < (int64_t)K * V; ++e) S[e] = (double)Sg[e];
  const double scale = (p->q_scale != 0.0) ? p->q_scale : pow((double)K, -0.5);

  for (int32_t r = r0; r < r1; ++r) {
    /* 1. conv + SiLU with the window, then slide the window */
    for (int c = 0, m = 0; c < 3; ++c) {
      double* dst = (c == 0) ? qt : (c == 1) ? kt : vt;
      for (int j = 0; j < dims[c]; ++j, ++m) {
        const int64_t ch = offs[c] + (int64_t)h * dims[c] + j;
        uint16_t* wm = win + (size_t)m * (W - 1);
        const uint16_t xin = p->qkv[(int64_t)r * p->qkv_row_stride + ch];
        for (int t = 0; t < W - 1; ++t) x[t] = kda_oracle_bf16_to_f64(wm[t]);
        x[W - 1] = kda_oracle_bf16_to_f64(xin);
        for (int t = 0; t < W; ++t) wt[t] = (double)wbase[c][(int64_t)t * Ds[c] + (int64_t)h * dims[c] + j];
        const double bias = p->conv_bias ? (double)p->conv_bias[ch] : 0.0;
        dst[j] = kda_oracle_silu(kda_oracle_causal_conv(x, wt, W, bias));
        if (W > 1) {
          for (int t = 0; t < W - 2; ++t) wm[t] = wm[t + 1];
          wm[W - 2] = xin;
        }
      }
    }
    /* 2. L2 norms */
    kda_oracle_l2norm(qt, K, p->l2_eps, scale, qh);
    kda_oracle_l2norm(kt, K, p->l2_eps, 1.0, kh);
    /* 3. gated delta rule, state kept in fp64 */
    double beta = kda_oracle_bf16_to_f64(p->beta[(int64_t)r * H + h]);
    if (p->fused_gate) {
      const double a_log = (double)p->A_log[h];
      for (int i = 0; i < K; ++i) {
        double zz = (double)p->g[((int64_t)r * H + h) * K + i];
        if (p->dt_bias) zz += (double)p->dt_bias[(int64_t)h * K + i];
        alpha[i] = exp(kda_oracle_kda_gate(zz, a_log, p->lower_bound));
      }
      beta = kda_oracle_sigmoid(beta);
    } else {
      for (int i = 0; i < K; ++i) alpha[i] = exp((double)p->g[((int64_t)r * H + h) * K + i]);
    }
    kda_oracle_gated_delta_update(K, V, S, alpha, beta, kh, vt);
    /* 4. readout, 5. gated RMSNorm or raw */
    kda_oracle_readout(K, V, S, qh, o);
    if (p->out_norm) {
      for (int j = 0; j < V; ++j) {
        gt[j] = kda_oracle_bf16_to_f64(p->gate[(int64_t)r * Dv + (int64_t)h * V + j]);
        nw[j] = (double)p->norm_weight[j];
      }
      kda_oracle_gated_rmsnorm(V, o, nw, gt, p->eps, y);
    } else {
      for (int j = 0; j < V; ++j) y[j] = o[j];
    }
    for (int j = 0; j < V; ++j) {
      p->out[(int64_t)r * Dv + (int64_t)h * V + j] = kda_oracle_round_bf16(y[j]);
      if (p->out_f64) p->out_f64[(int64_t)r * Dv + (int64_t)h * V + j] = y[j];
    }
  }

  /* store the final state and window */
  for (int64_t e = 0; e < (int64_t)K * V; ++e) Sg[e] = (float)S[e];
  for (int c = 0, m = 0; c < 3; ++c)
    for (int j = 0; j < dims[c]; ++j, ++m) {
      const int64_t ch = offs[c] + (int64_t)h * dims[c] + j;
      for (int t = 0; t < W - 1; ++t) cs0[ch * cs_ch + t * cs_t] = win[(size_t)m * (W - 1) + t];
    }
  return 0;
}

int kda_oracle_prefill(const kda_oracle_prefill_problem* p, int num_threads) {
  if (!p || p->B < 0 || p->H < 1 || p->K < 1 || p->V < 1 || p->W < 2 || p->num_slots < 1) return -1;
  if (p->B == 0) return 0;
  if (!p->cu_seqlens || !p->conv_weight || !p->conv_state || !p->state || !p->slot_idx) return -1;
  if (p->cu_seqlens[0] != 0) return -1;
  for (int b = 0; b < p->B; ++b)
    if (p->cu_seqlens[b + 1] < p->cu_seqlens[b]) return -1;
  if (p->cu_seqlens[p->B] > 0 && (!p->qkv || !p->g || !p->beta || !p->out)) return -1;
  if (p->out_norm && p->cu_seqlens[p->B] > 0 && (!p->gate || !p->norm_weight)) return -1;
  if (p->fused_gate && !p->A_log) return -1;
  const int64_t C = 2 * (int64_t)p->H * p->K + (int64_t)p->H * p->V;
  if (p->qkv_row_stride < C) return -1;

  const int64_t units = (int64_t)p->B * p->H;
  const size_t work_len = (size_t)(5 * p->K + 5 * p->V + 2 * p->W) + (size_t)p->K * p->V +
                          ((size_t)(2 * p->K + p->V) * (p->W - 1) * sizeof(uint16_t) + sizeof(double) - 1) / sizeof(double);
  int oob = 0;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#else
  (void)num_threads;
#endif
#pragma omp parallel reduction(+ : oob)
  {
    double* work = (double*)malloc(work_len * sizeof(double));
#pragma omp for schedule(dynamic, 1)
    for (int64_t u = 0; u < units; ++u) {
      const int b = (int)(u / p->H), h = (int)(u % p->H);
      const int r = prefill_unit(p, b, h, work);
      if (h == 0) oob += r;
    }
    free(work);
  }
  return oob;
}

/* ---------------------------------------------------------------- multi-token decode */

int kda_oracle_multi_problem_size(void) { return (int)sizeof(kda_oracle_multi_problem); }

/* One (sequence n, head h) of the multi-token decode: the decode steps token
 * by token from the source slot's window and state, each present token's
 * state and window stored to its own destination slot (formulation in
 * kda_oracle.h, MULTI-TOKEN DECODE; P1 实现拆解 items 3-4 for the excluded
 * speculative batches).  Returns the number of out-of-range slots met. */
static int multi_unit(const kda_oracle_multi_problem* p, int n, int h, double* work) {
  const int H = p->H, K = p->K, V = p->V, W = p->W, T = p->T;
  const int64_t Dq = (int64_t)H * K, Dv = (int64_t)H * V, C = 2 * Dq + Dv;
  const int32_t src = p->src_slot[n];

  if (src <= 0 || src >= p->num_slots) { /* padding or out-of-range sequence */
    for (int t = 0; t < T; ++t) {
      const int64_t r = (int64_t)n * T + t;
      for (int j = 0; j < V; ++j) {
        p->out[r * Dv + (int64_t)h * V + j] = 0;
        if (p->out_f64) p->out_f64[r * Dv + (int64_t)h * V + j] = 0.0;
      }
    }
    return src >= p->num_slots;
  }

  double* qt = work;            /* K */
  double* kt = qt + K;          /* K */
  double* vt = kt + K;          /* V */
  double* qh = vt + V;          /* K */
  double* kh = qh + K;          /* K */
  double* alpha = kh + K;       /* K */
  double* o = alpha + K;        /* V */
  double* y = o + V;            /* V */
  double* gt = y + V;           /* V */
  double* nw = gt + V;          /* V */
  double* x = nw + V;           /* W */
  double* wt = x + W;           /* W */
  double* S = wt + W;           /* K*V */
  uint16_t* win = (uint16_t*)(S + (size_t)K * V); /* (2K+V) channels x (W-1) taps, oldest first */

  const int dims[3] = {K, K, V};
  const int64_t offs[3] = {0, Dq, 2 * Dq};
  const int64_t Ds[3] = {Dq, Dq, Dv};
  const float* wbase[3] = {p->conv_weight, p->conv_weight + (int64_t)W * Dq, p->conv_weight + 2 * (int64_t)W * Dq};
  /* element (ch, t) of a slot's conv state in either layout */
  const int64_t cs_ch = p->conv_state_sd ? 1 : (W - 1);
  const int64_t cs_t = p->conv_state_sd ? C : 1;

  /* the source: window and state, read in full before anything is stored */
  const uint16_t* cs_src = p->conv_state + (int64_t)src * C * (W - 1);
  for (int c = 0, m = 0; c < 3; ++c)
    for (int j = 0; j < dims[c]; ++j, ++m) {
      const int64_t ch = offs[c] + (int64_t)h * dims[c] + j;
      for (int t = 0; t < W - 1; ++t) win[(size_t)m * (W - 1) + t] = cs_src[ch * cs_ch + t * cs_t];
    }
  const float* S_src = p->state + (((int64_t)src * H + h) * K) * V;
  for (int64_t e = 0; e < (int64_t)K * V; ++e) S[e] = (double)S_src[e];
  const double scale = (p->q_scale != 0.0) ? p->q_scale : 1.0 / sqrt((double)p->K);

  int oob = 0;
  for (int t = 0; t < T; ++t) {
    const int64_t r = (int64_t)n * T + t;
    const int32_t dst = p->dst_slots[r];
    uint16_t* out = p->out + r * Dv + (int64_t)h * V;
    double* out64 = p->out_f64 ? p->out_f64 + r * Dv + (int64_t)h * V : NULL;
    if (dst <= 0 || dst >= p->num_slots) { /* absent token */
      for (int j = 0; j < V; ++j) {
        out[j] = 0;
        if (out64) out64[j] = 0.0;
      }
      oob += dst >= p->num_slots;
      continue;
    }
    /* 1. conv + SiLU over the window and this token's input; the window slides */
    for (int c = 0, m = 0; c < 3; ++c) {
      double* dstv = (c == 0) ? qt : (c == 1) ? kt : vt;
      for (int j = 0; j < dims[c]; ++j, ++m) {
        const int64_t ch = offs[c] + (int64_t)h * dims[c] + j;
        uint16_t* wm = win + (size_t)m * (W - 1);
        const uint16_t xin = p->qkv[r * p->qkv_row_stride + ch];
        for (int k = 0; k < W - 1; ++k) x[k] = kda_oracle_bf16_to_f64(wm[k]);
        x[W - 1] = kda_oracle_bf16_to_f64(xin);
        for (int k = 0; k < W; ++k) wt[k] = (double)wbase[c][(int64_t)k * Ds[c] + (int64_t)h * dims[c] + j];
        const double bias = p->conv_bias ? (double)p->conv_bias[ch] : 0.0;
        dstv[j] = kda_oracle_silu(kda_oracle_causal_conv(x, wt, W, bias));
        for (int k = 0; k < W - 2; ++k) wm[k] = wm[k + 1];
        wm[W - 2] = xin;
      }
    }
    /* 2. L2 norms */
    kda_oracle_l2norm(qt, K, p->l2_eps, scale, qh);
    kda_oracle_l2norm(kt, K, p->l2_eps, 1.0, kh);
    /* 3. gated delta rule on the carried fp64 state */
    double beta = kda_oracle_bf16_to_f64(p->beta[r * H + h]);
    if (p->fused_gate) {
      const double a_log = (double)p->A_log[h];
      for (int i = 0; i < K; ++i) {
        double zi = (double)p->g[(r * H + h) * K + i];
        if (p->dt_bias) zi += (double)p->dt_bias[(int64_t)h * K + i];
        alpha[i] = exp(kda_oracle_kda_gate(zi, a_log, p->lower_bound));
      }
      beta = kda_oracle_sigmoid(beta); /* raw logit */
    } else {
      for (int i = 0; i < K; ++i) alpha[i] = exp((double)p->g[(r * H + h) * K + i]);
    }
    kda_oracle_gated_delta_update(K, V, S, alpha, beta, kh, vt);
    /* 4. readout, 5. gated RMSNorm or raw */
    kda_oracle_readout(K, V, S, qh, o);
    if (p->out_norm) {
      for (int j = 0; j < V; ++j) {
        gt[j] = kda_oracle_bf16_to_f64(p->gate[r * Dv + (int64_t)h * V + j]);
        nw[j] = (double)p->norm_weight[j];
      }
      kda_oracle_gated_rmsnorm(V, o, nw, gt, p->eps, y);
    } else {
      for (int j = 0; j < V; ++j) y[j] = o[j];
    }
    for (int j = 0; j < V; ++j) {
      out[j] = kda_oracle_round_bf16(y[j]);
      if (out64) out64[j] = y[j];
    }
    /* 6. store the state (rounded) and the window after this token */
    float* S_dst = p->state + (((int64_t)dst * H + h) * K) * V;
    for (int64_t e = 0; e < (int64_t)K * V; ++e) S_dst[e] = (float)S[e];
    if (p->update_conv_state) {
      uint16_t* cs_dst = p->conv_state + (int64_t)dst * C * (W - 1);
      for (int c = 0, m = 0; c < 3; ++c)
        for (int j = 0; j < dims[c]; ++j, ++m) {
          const int64_t ch = offs[c] + (int64_t)h * dims[c] + j;
          for (int k = 0; k < W - 1; ++k) cs_dst[ch * cs_ch + k * cs_t] = win[(size_t)m * (W - 1) + k];
        }
    }
  }
  return oob;
}

int kda_oracle_decode_multi(const kda_oracle_multi_problem* p, int num_threads) {
  if (!p || p->N < 0 || p->T < 1 || p->H < 1 || p->K < 1 || p->V < 1 || p->W < 2 || p->num_slots < 1)
    return -1;
  if (p->N == 0) return 0;
  if (!p->src_slot || !p->dst_slots || !p->qkv || !p->conv_weight || !p->conv_state || !p->state || !p->g ||
      !p->beta || !p->out)
    return -1;
  if (p->out_norm && (!p->gate || !p->norm_weight)) return -1;
  if (p->fused_gate && !p->A_log) return -1;
  const int64_t C = 2 * (int64_t)p->H * p->K + (int64_t)p->H * p->V;
  if (p->qkv_row_stride < C) return -1;

  const int64_t units = (int64_t)p->N * p->H;
  const size_t work_len = (size_t)(5 * p->K + 5 * p->V + 2 * p->W) + (size_t)p->K * p->V +
                          ((size_t)(2 * p->K + p->V) * (p->W - 1) * sizeof(uint16_t) + sizeof(double) - 1) / sizeof(double);
  int oob = 0;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#else
  (void)num_threads;
#endif
#pragma omp parallel reduction(+ : oob)
  {
    double* work = (double*)malloc(work_len * sizeof(double));
#pragma omp for schedule(dynamic, 4)
    for (int64_t u = 0; u < units; ++u) {
      const int n = (int)(u / p->H), h = (int)(u % p->H);
      const int r = multi_unit(p, n, h, work);
      if (h == 0) oob += r; /* count per sequence, not per (sequence, head) */
    }
    free(work);
  }
  return oob;
}

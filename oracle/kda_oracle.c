/*
 * kda_oracle.c -- plain FP64 CPU reference of the recurrent KDA (Kimi Delta
 * Attention) training recurrence, forward and backward.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark may load this library. It shares no code, header, table
 * or constant with the CUDA path.
 *
 * Sources followed (flashinfer documentation pages):
 *  - "flashinfer.kda_backward.recurrent_kda_backward", description: Q and K are
 *    L2-normalised with epsilon 1e-6; decay = exp(lower_bound * sigmoid(
 *    exp(A_log) * (g + dt_bias))); beta passes through a sigmoid; adjoints are
 *    `do` (token output) and `dfinal_state` (final state); the gradients are
 *    (dq, dk, dv, dg, dbeta, dA_log, ddt_bias, dinitial_state), taken with
 *    respect to the raw gate and the raw beta logits.
 *  - "flashinfer.kda_training.recurrent_kda_training_forward", parameters:
 *    value-first FP32 state [N, Hv, V, K]; v, g, beta and the state carry Hv
 *    heads, q and k carry Hqk heads with Hv an integer multiple of Hqk.
 *  - "flashinfer.kda.recurrent_kda", parameter `lower_bound`: the same gate
 *    formula lower_bound * sigmoid(exp(A_log) * (g + dt_bias)); parameters g
 *    and beta: g may come precomputed in log space (the decay is then exp(g))
 *    and beta may come already passed through the sigmoid. Those two inference
 *    modes are kda_oracle_forward_modes below.
 * The pages name the method (a gated delta rule with per-key-dimension decay)
 * but print no update equations. This file takes the plain reading, per token:
 *     S' = S diag(d);  u = v - S' k^;  S = S' + beta u k^T;  o = scale S q^
 * i.e. decay, delta correction, rank-1 write, output read from the post-update
 * state.  GQA: value head h reads query/key head h / (Hv/Hqk).
 *
 * Layouts (all row-major, packed token axis; a fixed [B,T] layout is passed as
 * B sequences with cu = 0, T, 2T, ...):
 *   q, k      [Ttot, Hqk, DK]     v [Ttot, Hv, DV]     g [Ttot, Hv, DK]
 *   beta      [Ttot, Hv]          A_log [Hv]           dt_bias [Hv, DK]
 *   h0, hT    [N, Hv, DV, DK]     o, do [Ttot, Hv, DV]
 * `qk_mask` (may be NULL) selects which query/key heads (and so which value
 * heads) are computed; outputs of unselected heads are not written.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define NORM_EPS 1e-6 /* epsilon of the L2 normalisation of q and k */

int kda_oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* x^ = x / sqrt(sum x^2 + eps); returns the factor r = (sum x^2 + eps)^-1/2. */
static double l2norm(const double* x, int64_t n, double* xhat) {
  double ss = 0.0;
  for (int64_t i = 0; i < n; ++i) ss += x[i] * x[i];
  double r = 1.0 / sqrt(ss + NORM_EPS);
  for (int64_t i = 0; i < n; ++i) xhat[i] = x[i] * r;
  return r;
}

typedef struct {
  int64_t nseq;
  const int64_t* cu;
  int64_t hqk, hv, dk, dv;
  const double *q, *k, *v, *g, *beta, *A_log, *dt_bias, *h0;
  double scale, lb;
  /* inference gate modes (flashinfer.kda.recurrent_kda, parameters g and beta):
   * 0 (the default) computes the gate in the kernel and passes beta through a
   * sigmoid; log_space_g = 1 takes g as the log decay itself, presigmoid_beta =
   * 1 takes beta as already passed through the sigmoid */
  int log_space_g, presigmoid_beta;
} problem;

/* Per-token quantities shared by the forward and backward steps. */
typedef struct {
  double *qhat, *khat, *z, *d;
  double rq, rk, b;
} token_terms;

static void token_prepare(const problem* P, int64_t t, int64_t h, token_terms* tt) {
  const int64_t r = P->hv / P->hqk;
  const int64_t qh = h / r;
  const int64_t DK = P->dk;
  tt->rq = l2norm(P->q + (t * P->hqk + qh) * DK, DK, tt->qhat);
  tt->rk = l2norm(P->k + (t * P->hqk + qh) * DK, DK, tt->khat);
  if (P->log_space_g) {
    for (int64_t j = 0; j < DK; ++j) {
      tt->z[j] = 0.0;
      tt->d[j] = exp(P->g[(t * P->hv + h) * DK + j]);
    }
  } else {
    const double ea = exp(P->A_log[h]);
    for (int64_t j = 0; j < DK; ++j) {
      tt->z[j] = ea * (P->g[(t * P->hv + h) * DK + j] + P->dt_bias[h * DK + j]);
      tt->d[j] = exp(P->lb * sigmoid(tt->z[j]));
    }
  }
  const double braw = P->beta[t * P->hv + h];
  tt->b = P->presigmoid_beta ? braw : sigmoid(braw);
}

static void token_alloc(const problem* P, token_terms* tt) {
  tt->qhat = (double*)malloc(sizeof(double) * P->dk);
  tt->khat = (double*)malloc(sizeof(double) * P->dk);
  tt->z = (double*)malloc(sizeof(double) * P->dk);
  tt->d = (double*)malloc(sizeof(double) * P->dk);
}

static void token_free(token_terms* tt) {
  free(tt->qhat); free(tt->khat); free(tt->z); free(tt->d);
}

/* One step of the recurrence on S (DV x DK, in place). Writes u (DV) and, if
 * o is non-NULL, the output o = scale * S q^ read after the update. */
static void step(const problem* P, int64_t t, int64_t h, const token_terms* tt, double* S,
                 double* u, double* o) {
  const int64_t DK = P->dk, DV = P->dv;
  const double* vt = P->v + (t * P->hv + h) * DV;
  for (int64_t i = 0; i < DV; ++i) {
    double* row = S + i * DK;
    double p = 0.0;
    for (int64_t j = 0; j < DK; ++j) {
      row[j] *= tt->d[j];          /* S' = S diag(d) */
      p += row[j] * tt->khat[j];   /* p = S' k^      */
    }
    u[i] = vt[i] - p;              /* u = v - S' k^  */
    const double bu = tt->b * u[i];
    double acc = 0.0;
    for (int64_t j = 0; j < DK; ++j) {
      row[j] += bu * tt->khat[j];  /* S = S' + beta u k^T */
      acc += row[j] * tt->qhat[j];
    }
    if (o) o[i] = P->scale * acc;  /* o = scale S q^ */
  }
}

static int head_selected(const problem* P, const uint8_t* qk_mask, int64_t h) {
  return qk_mask == NULL || qk_mask[h / (P->hv / P->hqk)];
}

static int forward_impl(const problem* PP, const uint8_t* qk_mask, double* o, double* hT);

int kda_oracle_forward(int64_t nseq, const int64_t* cu, int64_t hqk, int64_t hv, int64_t dk,
                       int64_t dv, const double* q, const double* k, const double* v,
                       const double* g, const double* beta, const double* A_log,
                       const double* dt_bias, const double* h0, double scale, double lower_bound,
                       const uint8_t* qk_mask, double* o, double* hT) {
  if (nseq <= 0 || hqk <= 0 || hv <= 0 || hv % hqk != 0 || dk <= 0 || dv <= 0) return 1;
  problem P = {nseq, cu, hqk, hv, dk, dv, q, k, v, g, beta, A_log, dt_bias, h0, scale, lower_bound, 0, 0};
  return forward_impl(&P, qk_mask, o, hT);
}

/* The same forward with the inference page's gate modes: log_space_g = 1 reads
 * g as the per-key log decay (d = exp(g); A_log, dt_bias and lower_bound are
 * not used), presigmoid_beta = 1 reads beta as the learning rate itself. */
int kda_oracle_forward_modes(int64_t nseq, const int64_t* cu, int64_t hqk, int64_t hv, int64_t dk,
                             int64_t dv, const double* q, const double* k, const double* v,
                             const double* g, const double* beta, const double* A_log,
                             const double* dt_bias, const double* h0, double scale, double lower_bound,
                             int log_space_g, int presigmoid_beta, double* o, double* hT) {
  if (nseq <= 0 || hqk <= 0 || hv <= 0 || hv % hqk != 0 || dk <= 0 || dv <= 0) return 1;
  problem P = {nseq, cu, hqk, hv, dk, dv, q, k, v, g, beta, A_log, dt_bias, h0, scale, lower_bound,
               log_space_g != 0, presigmoid_beta != 0};
  return forward_impl(&P, NULL, o, hT);
}

static int forward_impl(const problem* PP, const uint8_t* qk_mask, double* o, double* hT) {
  const problem P = *PP;
  const int64_t nseq = P.nseq, hv = P.hv, dk = P.dk, dv = P.dv;
  const int64_t* cu = P.cu;
  const double* h0 = P.h0;
  const int64_t units = nseq * hv;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t un = 0; un < units; ++un) {
    const int64_t n = un / hv, h = un % hv;
    if (!head_selected(&P, qk_mask, h)) continue;
    token_terms tt;
    token_alloc(&P, &tt);
    double* S = (double*)malloc(sizeof(double) * dv * dk);
    double* u = (double*)malloc(sizeof(double) * dv);
    memcpy(S, h0 + (n * hv + h) * dv * dk, sizeof(double) * dv * dk);
    for (int64_t t = cu[n]; t < cu[n + 1]; ++t) {
      token_prepare(&P, t, h, &tt);
      step(&P, t, h, &tt, S, u, o + (t * hv + h) * dv);
    }
    memcpy(hT + (n * hv + h) * dv * dk, S, sizeof(double) * dv * dk);
    free(S); free(u);
    token_free(&tt);
  }
  return 0;
}

/*
 * Chunked restatement of the same forward, for the chunk-equals-sequential
 * check. Within a chunk of C tokens starting from state S0, with
 * Gam_i = sum_{j<=i} a_j (a = log decay, per key dim):
 *   A_ij = sum_k k^_i k^_j exp(Gam_i - Gam_j)            (j < i)
 *   B_ij = sum_k q^_i k^_j exp(Gam_i - Gam_j)            (j <= i)
 *   Y_i  = beta_i (v_i - S0 (k^_i * exp(Gam_i)))
 *   W    solves (I + diag(beta) A) W = Y by forward substitution
 *   o_i  = scale (S0 (q^_i * exp(Gam_i)) + sum_{j<=i} B_ij W_j)
 *   S_C  = S0 diag(exp(Gam_C)) + sum_j W_j (k^_j * exp(Gam_C - Gam_j))^T
 * where W_j = beta_j u_j are the rank-1 write vectors of the sequential form.
 */
int kda_oracle_forward_chunked(int64_t nseq, const int64_t* cu, int64_t hqk, int64_t hv,
                               int64_t dk, int64_t dv, const double* q, const double* k,
                               const double* v, const double* g, const double* beta,
                               const double* A_log, const double* dt_bias, const double* h0,
                               double scale, double lower_bound, int64_t chunk, double* o,
                               double* hT) {
  if (nseq <= 0 || hqk <= 0 || hv <= 0 || hv % hqk != 0 || chunk <= 0) return 1;
  problem P = {nseq, cu, hqk, hv, dk, dv, q, k, v, g, beta, A_log, dt_bias, h0, scale, lower_bound, 0, 0};
  const int64_t units = nseq * hv;
  const int64_t C = chunk;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t un = 0; un < units; ++un) {
    const int64_t n = un / hv, h = un % hv;
    token_terms tt;
    token_alloc(&P, &tt);
    double* S = (double*)malloc(sizeof(double) * dv * dk);
    double* Qh = (double*)malloc(sizeof(double) * C * dk);
    double* Kh = (double*)malloc(sizeof(double) * C * dk);
    double* Gm = (double*)malloc(sizeof(double) * C * dk);
    double* bt = (double*)malloc(sizeof(double) * C);
    double* A = (double*)malloc(sizeof(double) * C * C);
    double* Bm = (double*)malloc(sizeof(double) * C * C);
    double* W = (double*)malloc(sizeof(double) * C * dv);
    memcpy(S, h0 + (n * hv + h) * dv * dk, sizeof(double) * dv * dk);
    for (int64_t c0 = cu[n]; c0 < cu[n + 1]; c0 += C) {
      const int64_t nc = (cu[n + 1] - c0 < C) ? cu[n + 1] - c0 : C;
      for (int64_t i = 0; i < nc; ++i) {
        token_prepare(&P, c0 + i, h, &tt);
        for (int64_t j = 0; j < dk; ++j) {
          Qh[i * dk + j] = tt.qhat[j];
          Kh[i * dk + j] = tt.khat[j];
          Gm[i * dk + j] = log(tt.d[j]) + (i > 0 ? Gm[(i - 1) * dk + j] : 0.0);
        }
        bt[i] = tt.b;
      }
      for (int64_t i = 0; i < nc; ++i)
        for (int64_t j = 0; j < nc; ++j) {
          double a = 0.0, bb = 0.0;
          if (j <= i)
            for (int64_t x = 0; x < dk; ++x) {
              const double e = exp(Gm[i * dk + x] - Gm[j * dk + x]);
              a += Kh[i * dk + x] * Kh[j * dk + x] * e;
              bb += Qh[i * dk + x] * Kh[j * dk + x] * e;
            }
          A[i * C + j] = (j < i) ? a : 0.0;
          Bm[i * C + j] = (j <= i) ? bb : 0.0;
        }
      /* Y, then forward substitution for W */
      for (int64_t i = 0; i < nc; ++i) {
        const double* vt = v + ((c0 + i) * hv + h) * dv;
        for (int64_t y = 0; y < dv; ++y) {
          double sk = 0.0;
          for (int64_t x = 0; x < dk; ++x) sk += S[y * dk + x] * Kh[i * dk + x] * exp(Gm[i * dk + x]);
          double w = bt[i] * (vt[y] - sk);
          for (int64_t j = 0; j < i; ++j) w -= bt[i] * A[i * C + j] * W[j * dv + y];
          W[i * dv + y] = w;
        }
      }
      for (int64_t i = 0; i < nc; ++i) {
        double* ot = o + ((c0 + i) * hv + h) * dv;
        for (int64_t y = 0; y < dv; ++y) {
          double acc = 0.0;
          for (int64_t x = 0; x < dk; ++x) acc += S[y * dk + x] * Qh[i * dk + x] * exp(Gm[i * dk + x]);
          for (int64_t j = 0; j <= i; ++j) acc += Bm[i * C + j] * W[j * dv + y];
          ot[y] = scale * acc;
        }
      }
      const double* GC = Gm + (nc - 1) * dk;
      for (int64_t y = 0; y < dv; ++y)
        for (int64_t x = 0; x < dk; ++x) {
          double s = S[y * dk + x] * exp(GC[x]);
          for (int64_t j = 0; j < nc; ++j) s += W[j * dv + y] * Kh[j * dk + x] * exp(GC[x] - Gm[j * dk + x]);
          S[y * dk + x] = s;
        }
    }
    memcpy(hT + (n * hv + h) * dv * dk, S, sizeof(double) * dv * dk);
    free(S); free(Qh); free(Kh); free(Gm); free(bt); free(A); free(Bm); free(W);
    token_free(&tt);
  }
  return 0;
}

/*
 * Backward: reverse-mode differentiation of the sequential forward, per token,
 * last to first. With G = dL/dS_t accumulated from later tokens:
 *   G     += scale do_t q^T            dq^ = scale S_t^T do_t
 *   w      = G k^                      dbeta_act = u . w      du = beta w
 *   dv     = du                        dk^ = beta G^T u - S'^T du
 *   dS'    = G - du k^T                da[k] = sum_v dS'[v,k] S'[v,k]
 *   G      = dS' diag(d)               (gradient w.r.t. S_{t-1})
 * then through the gate, sigmoid and L2 norm:
 *   dz = da lb sig(z)(1-sig(z));  dg = dz exp(A_log);  ddt_bias += dz exp(A_log);
 *   dA_log += sum_k dz z;  dbeta_raw = dbeta_act beta (1-beta);
 *   dq += r_q (dq^ - q^ (q^ . dq^))  (summed over the value heads of a query head),
 * and dinitial_state = G after the first token. States inside a block of BLK
 * tokens are recomputed from a stored state at the block start.
 * dA_log and ddt_bias are summed per (sequence, head) and then over sequences
 * in index order, so the result does not depend on the thread count.
 */
#define BLK 64

int kda_oracle_backward(int64_t nseq, const int64_t* cu, int64_t hqk, int64_t hv, int64_t dk,
                        int64_t dv, const double* q, const double* k, const double* v,
                        const double* g, const double* beta, const double* A_log,
                        const double* dt_bias, const double* h0, const double* d_o,
                        const double* dhT, double scale, double lower_bound,
                        const uint8_t* qk_mask, double* dq, double* dk_out, double* dv_out,
                        double* dg, double* dbeta, double* dA_log, double* ddt_bias,
                        double* dh0) {
  if (nseq <= 0 || hqk <= 0 || hv <= 0 || hv % hqk != 0 || dk <= 0 || dv <= 0) return 1;
  problem P = {nseq, cu, hqk, hv, dk, dv, q, k, v, g, beta, A_log, dt_bias, h0, scale, lower_bound, 0, 0};
  const int64_t r = hv / hqk;
  const int64_t DK = dk, DV = dv;
  const int64_t SZ = DV * DK;
  /* per (sequence, head) partial sums: [nseq][hv][DK + 1], last slot dA_log */
  double* part = (double*)calloc((size_t)(nseq * hv * (DK + 1)), sizeof(double));
  const int64_t groups = nseq * hqk;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t gi = 0; gi < groups; ++gi) {
    const int64_t n = gi / hqk, qh = gi % hqk;
    if (qk_mask && !qk_mask[qh]) continue;
    const int64_t t0 = cu[n], t1 = cu[n + 1], T = t1 - t0;
    for (int64_t t = t0; t < t1; ++t) {
      memset(dq + (t * hqk + qh) * DK, 0, sizeof(double) * DK);
      memset(dk_out + (t * hqk + qh) * DK, 0, sizeof(double) * DK);
    }
    const int64_t nblk = (T + BLK - 1) / BLK;
    token_terms tt;
    token_alloc(&P, &tt);
    double* ck = (double*)malloc(sizeof(double) * SZ * (nblk > 0 ? nblk : 1));
    double* Sb = (double*)malloc(sizeof(double) * SZ * BLK);  /* S_{t-1} per token of a block */
    double* S = (double*)malloc(sizeof(double) * SZ);
    double* Sp = (double*)malloc(sizeof(double) * SZ);        /* S' */
    double* G = (double*)malloc(sizeof(double) * SZ);
    double* u = (double*)malloc(sizeof(double) * DV);
    double* w = (double*)malloc(sizeof(double) * DV);
    double* du = (double*)malloc(sizeof(double) * DV);
    double* dqh = (double*)malloc(sizeof(double) * DK);
    double* dkh = (double*)malloc(sizeof(double) * DK);
    double* da = (double*)malloc(sizeof(double) * DK);
    for (int64_t hh = 0; hh < r; ++hh) {
      const int64_t h = qh * r + hh;
      double* pp = part + (n * hv + h) * (DK + 1);
      /* forward pass, storing the state at each block start */
      memcpy(S, h0 + (n * hv + h) * SZ, sizeof(double) * SZ);
      for (int64_t t = t0; t < t1; ++t) {
        if ((t - t0) % BLK == 0) memcpy(ck + ((t - t0) / BLK) * SZ, S, sizeof(double) * SZ);
        token_prepare(&P, t, h, &tt);
        step(&P, t, h, &tt, S, u, NULL);
      }
      memcpy(G, dhT + (n * hv + h) * SZ, sizeof(double) * SZ);
      const double ea = exp(A_log[h]);
      for (int64_t blk = nblk - 1; blk >= 0; --blk) {
        const int64_t b0 = t0 + blk * BLK;
        const int64_t b1 = (b0 + BLK < t1) ? b0 + BLK : t1;
        memcpy(S, ck + blk * SZ, sizeof(double) * SZ);
        for (int64_t t = b0; t < b1; ++t) {
          memcpy(Sb + (t - b0) * SZ, S, sizeof(double) * SZ);
          token_prepare(&P, t, h, &tt);
          step(&P, t, h, &tt, S, u, NULL);
        }
        for (int64_t t = b1 - 1; t >= b0; --t) {
          token_prepare(&P, t, h, &tt);
          /* rebuild S' and S_t from S_{t-1} */
          memcpy(S, Sb + (t - b0) * SZ, sizeof(double) * SZ);
          const double* vt = v + (t * hv + h) * DV;
          const double* dot = d_o + (t * hv + h) * DV;
          for (int64_t i = 0; i < DV; ++i) {
            double p = 0.0;
            for (int64_t j = 0; j < DK; ++j) {
              Sp[i * DK + j] = S[i * DK + j] * tt.d[j];
              p += Sp[i * DK + j] * tt.khat[j];
            }
            u[i] = vt[i] - p;
            for (int64_t j = 0; j < DK; ++j) S[i * DK + j] = Sp[i * DK + j] + tt.b * u[i] * tt.khat[j];
          }
          /* output adjoint */
          for (int64_t i = 0; i < DV; ++i)
            for (int64_t j = 0; j < DK; ++j) G[i * DK + j] += scale * dot[i] * tt.qhat[j];
          for (int64_t j = 0; j < DK; ++j) {
            double acc = 0.0;
            for (int64_t i = 0; i < DV; ++i) acc += S[i * DK + j] * dot[i];
            dqh[j] = scale * acc;
          }
          /* rank-1 write and delta correction */
          double dbeta_act = 0.0;
          for (int64_t i = 0; i < DV; ++i) {
            double acc = 0.0;
            for (int64_t j = 0; j < DK; ++j) acc += G[i * DK + j] * tt.khat[j];
            w[i] = acc;
            dbeta_act += u[i] * acc;
            du[i] = tt.b * acc;
            dv_out[(t * hv + h) * DV + i] = du[i];
          }
          for (int64_t j = 0; j < DK; ++j) {
            double a1 = 0.0, a2 = 0.0;
            for (int64_t i = 0; i < DV; ++i) {
              a1 += G[i * DK + j] * u[i];
              a2 += Sp[i * DK + j] * du[i];
            }
            dkh[j] = tt.b * a1 - a2;
          }
          /* dS' = G - du k^T; da = sum_v dS' * S'; G <- dS' diag(d) */
          for (int64_t j = 0; j < DK; ++j) da[j] = 0.0;
          for (int64_t i = 0; i < DV; ++i)
            for (int64_t j = 0; j < DK; ++j) {
              const double dsp = G[i * DK + j] - du[i] * tt.khat[j];
              da[j] += dsp * Sp[i * DK + j];
              G[i * DK + j] = dsp * tt.d[j];
            }
          /* gate, beta and norm backward */
          double dA = 0.0;
          for (int64_t j = 0; j < DK; ++j) {
            const double sg = sigmoid(tt.z[j]);
            const double dz = da[j] * lower_bound * sg * (1.0 - sg);
            dg[(t * hv + h) * DK + j] = dz * ea;
            pp[j] += dz * ea;
            dA += dz * tt.z[j];
          }
          pp[DK] += dA;
          dbeta[t * hv + h] = dbeta_act * tt.b * (1.0 - tt.b);
          double qd = 0.0, kd = 0.0;
          for (int64_t j = 0; j < DK; ++j) {
            qd += tt.qhat[j] * dqh[j];
            kd += tt.khat[j] * dkh[j];
          }
          double* dqt = dq + (t * hqk + qh) * DK;
          double* dkt = dk_out + (t * hqk + qh) * DK;
          for (int64_t j = 0; j < DK; ++j) {
            dqt[j] += tt.rq * (dqh[j] - tt.qhat[j] * qd);
            dkt[j] += tt.rk * (dkh[j] - tt.khat[j] * kd);
          }
        }
      }
      memcpy(dh0 + (n * hv + h) * SZ, G, sizeof(double) * SZ);
    }
    free(ck); free(Sb); free(S); free(Sp); free(G); free(u); free(w); free(du);
    free(dqh); free(dkh); free(da);
    token_free(&tt);
  }
  for (int64_t h = 0; h < hv; ++h) {
    if (!head_selected(&P, qk_mask, h)) continue;
    double sA = 0.0;
    for (int64_t j = 0; j < DK; ++j) {
      double s = 0.0;
      for (int64_t n = 0; n < nseq; ++n) s += part[(n * hv + h) * (DK + 1) + j];
      ddt_bias[h * DK + j] = s;
    }
    for (int64_t n = 0; n < nseq; ++n) sA += part[(n * hv + h) * (DK + 1) + DK];
    dA_log[h] = sA;
  }
  free(part);
  return 0;
}

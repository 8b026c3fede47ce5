/*
 * fp64 token-by-token KDA forward in plain C, threaded over (sequence, head).
 *
 * TEST INFRASTRUCTURE ONLY: the same plain definition as oracle/kda_ref.py,
 * written in C so that the large workloads finish in seconds on the host
 * cores. Nothing in the product path links or calls this file; only tests,
 * the smoke check and the bench's CPU-baseline leg do.
 *
 * Definition (Kimi Delta Attention, arXiv:2510.26692, cited on the cuLA
 * overview page, section "cuLA 소개"; parameter meanings and the [N,H,V,K]
 * state layout from the FlashKDA page, section "FlashKDA의 KDA 연산 구조"):
 *
 *   log alpha_k = lower_bound * sigmoid(exp(A_log[h]) * (g[t,h,k] + dt_bias[h,k]))
 *   q_hat = q / sqrt(|q|^2 + eps),  k_hat = k / sqrt(|k|^2 + eps)
 *   beta  = sigmoid(beta_logit[t,h])
 *   S     = Diag(alpha) S;  S += beta k_hat (v - S^T k_hat)^T;  o = scale S^T q_hat
 *
 * bf16 inputs arrive as their raw 16-bit patterns and are widened exactly
 * (the bf16 bits are the top half of an IEEE binary32).
 */
#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_to_f64(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* 1/(1+exp(-x)) without overflow; exactly 1 at +inf and 0 at -inf. */
static double sigmoid(double x) {
  if (x >= 0.0) return 1.0 / (1.0 + exp(-x));
  double e = exp(x);
  return e / (1.0 + e);
}

typedef struct {
  const uint16_t *q, *k, *v, *g, *beta;
  const float *A_log, *dt_bias;
  const double *init;
  const int32_t *cu, *pairs;
  double lb, scale, eps;
  int B, T, H, K, V, N, n_pairs;
  const int64_t *o_offset; /* per pair: first row of its output block */
  double *o_out, *final_out;
  atomic_int next;
} job_t;

static void run_pair(job_t *J, int p, double *S, double *alpha, double *qh,
                     double *kh, double *pred, double *tmp_v) {
  const int K = J->K, V = J->V, H = J->H;
  int s = J->pairs ? J->pairs[2 * p] : p / H;
  int h = J->pairs ? J->pairs[2 * p + 1] : p % H;
  int b, t0, t1;
  if (J->cu) { b = 0; t0 = J->cu[s]; t1 = J->cu[s + 1]; }
  else { b = s; t0 = 0; t1 = J->T; }
  /* S[k*V + v] = state[s,h,v,k] */
  for (int kk = 0; kk < K; ++kk)
    for (int vv = 0; vv < V; ++vv)
      S[kk * V + vv] = J->init ? J->init[(((int64_t)s * H + h) * V + vv) * K + kk] : 0.0;
  const double ea = exp((double)J->A_log[h]);
  double *o_base = J->o_out + J->o_offset[p];
  for (int t = t0; t < t1; ++t) {
    const int64_t row = ((int64_t)b * J->T + t) * H + h;
    const uint16_t *qr = J->q + row * K, *kr = J->k + row * K, *gr = J->g + row * K;
    const uint16_t *vr = J->v + row * V;
    double qs = 0.0, ks = 0.0;
    for (int kk = 0; kk < K; ++kk) {
      double db = J->dt_bias ? (double)J->dt_bias[(int64_t)h * K + kk] : 0.0;
      double a = ea * (bf16_to_f64(gr[kk]) + db);
      alpha[kk] = exp(J->lb * sigmoid(a));
      double x = bf16_to_f64(qr[kk]), y = bf16_to_f64(kr[kk]);
      qh[kk] = x; kh[kk] = y;
      qs += x * x; ks += y * y;
    }
    const double qn = 1.0 / sqrt(qs + J->eps), kn = 1.0 / sqrt(ks + J->eps);
    for (int kk = 0; kk < K; ++kk) { qh[kk] *= qn; kh[kk] *= kn; }
    const double bt = sigmoid(bf16_to_f64(J->beta[(int64_t)b * J->T * H + (int64_t)t * H + h]));
    /* decay, then prediction S^T k_hat */
    for (int vv = 0; vv < V; ++vv) pred[vv] = 0.0;
    for (int kk = 0; kk < K; ++kk) {
      double *Sr = S + (int64_t)kk * V;
      const double al = alpha[kk], kv = kh[kk];
      for (int vv = 0; vv < V; ++vv) { Sr[vv] *= al; pred[vv] += Sr[vv] * kv; }
    }
    for (int vv = 0; vv < V; ++vv) tmp_v[vv] = bt * (bf16_to_f64(vr[vv]) - pred[vv]);
    /* write, then o = scale S^T q_hat */
    for (int vv = 0; vv < V; ++vv) pred[vv] = 0.0;
    for (int kk = 0; kk < K; ++kk) {
      double *Sr = S + (int64_t)kk * V;
      const double kv = kh[kk], qv = qh[kk];
      for (int vv = 0; vv < V; ++vv) { Sr[vv] += kv * tmp_v[vv]; pred[vv] += Sr[vv] * qv; }
    }
    double *orow = o_base + (int64_t)(t - t0) * V;
    for (int vv = 0; vv < V; ++vv) orow[vv] = J->scale * pred[vv];
  }
  double *fo = J->final_out + (int64_t)p * V * K;
  for (int vv = 0; vv < V; ++vv)
    for (int kk = 0; kk < K; ++kk) fo[(int64_t)vv * K + kk] = S[(int64_t)kk * V + vv];
}

static void *worker(void *arg) {
  job_t *J = (job_t *)arg;
  const int K = J->K, V = J->V;
  double *S = (double *)malloc(sizeof(double) * ((size_t)K * V + 3 * K + 2 * V));
  if (!S) return (void *)1;
  double *alpha = S + (size_t)K * V, *qh = alpha + K, *kh = qh + K, *pred = kh + K,
         *tmp_v = pred + V;
  for (;;) {
    int p = atomic_fetch_add(&J->next, 1);
    if (p >= J->n_pairs) break;
    run_pair(J, p, S, alpha, qh, kh, pred, tmp_v);
  }
  free(S);
  return NULL;
}

/*
 * q,k,g: bf16 bits [B,T,H,K]; v: [B,T,H,V]; beta: [B,T,H]; A_log fp32 [H];
 * dt_bias fp32 [H,K] or NULL; init fp64 [N,H,V,K] or NULL; cu_seqlens int32
 * [N+1] or NULL (then N == B and every sequence has length T).
 * pairs: int32 [n_pairs][2] of (sequence, head), or NULL for all N*H pairs in
 * order s*H + h. o_out receives, for pair p, its sequence's rows [len][V]
 * starting at row offset o_rows[p] (caller computes); final_out [n_pairs][V][K].
 * Returns 0 on success, 1 on a bad argument, 2 if a thread failed.
 */
int kda_oracle_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                   const uint16_t *g, const uint16_t *beta, const float *A_log,
                   const float *dt_bias, double lower_bound, double scale,
                   const double *init, const int32_t *cu_seqlens, int B, int T,
                   int H, int K, int V, int N, const int32_t *pairs,
                   int n_pairs, const int64_t *o_rows, double *o_out,
                   double *final_out, double eps, int n_threads) {
  if (!q || !k || !v || !g || !beta || !A_log || !o_out || !final_out || !o_rows)
    return 1;
  if (B <= 0 || T < 0 || H <= 0 || K <= 0 || V <= 0 || N < 0 || n_pairs < 0) return 1;
  if (n_threads < 1) n_threads = 1;
  int64_t *offs = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_pairs + 1));
  if (!offs) return 2;
  for (int p = 0; p < n_pairs; ++p) offs[p] = o_rows[p] * (int64_t)V;
  job_t J;
  memset(&J, 0, sizeof J);
  J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta;
  J.A_log = A_log; J.dt_bias = dt_bias; J.init = init;
  J.cu = cu_seqlens; J.pairs = pairs;
  J.lb = lower_bound; J.scale = scale; J.eps = eps;
  J.B = B; J.T = T; J.H = H; J.K = K; J.V = V; J.N = N; J.n_pairs = n_pairs;
  J.o_offset = offs; J.o_out = o_out; J.final_out = final_out;
  atomic_init(&J.next, 0);
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
  if (!th) { free(offs); return 2; }
  int started = 0, rc = 0;
  for (int i = 0; i < n_threads; ++i) {
    if (pthread_create(&th[i], NULL, worker, &J) != 0) break;
    ++started;
  }
  if (started == 0) rc = 2;
  for (int i = 0; i < started; ++i) {
    void *ret = NULL;
    pthread_join(th[i], &ret);
    if (ret) rc = 2;
  }
  free(th);
  free(offs);
  return rc;
}

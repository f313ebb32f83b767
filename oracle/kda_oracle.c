/*
 * kda_oracle.c -- plain fp64 CPU oracle for Kimi Delta Attention (KDA).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the libkda CUDA
 * library and its Python binding) includes, links or calls this file.  It is
 * loaded by the tests, by __graft_entry__.smoke() and by the CPU-baseline leg
 * of bench.py, and shares no code with the CUDA path.
 *
 * What it computes, token by token, in double precision:
 *
 *   Gate  (blog.higcp.com "猜想：K3 可能是最适合 TPU 的 MoE 架构",
 *          section "下界衰减：一个纯粹为硬件让步的算法改动"):
 *       g = gmin * sigmoid(e^{A_h} z),  alpha = exp(g),  gmin = -5,
 *       with A the per-head log-scale (optional argument; A = 0 when absent,
 *       i.e. any scale already folded into z by the caller).
 *
 *   Q/K preprocessing (mhpq.cn/news/56770, the paragraph on Q/K
 *   preprocessing after "KDA 到底在算什么"): q and k are L2-normalised
 *   before the recurrence; here x / sqrt(sum(x^2) + eps).  The page gives
 *   no eps; the library fixes eps = 1e-6 and the oracle takes it as an
 *   argument so that closed-form pins can set it to 0.
 *
 *   Recurrence and read-out (mhpq.cn/news/56770, section "KDA 到底在算什么"):
 *       S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *       o_t = S_t^T q_t
 *   S is dk x dv; alpha_t scales the rows of S (one retention per key
 *   channel).  Written out as the three steps it is made of:
 *       decay:  S <- Diag(alpha_t) S
 *       erase + write:  e = v_t - S^T k_t ;  S <- S + beta_t k_t e^T
 *       read:   o_t = S^T q_t            (after the update, so token t is seen)
 *   This is exactly the product above, expanded: (I - b k k^T) S' + b k v^T
 *   = S' + b k (v - S'^T k)^T.
 *
 * Layouts (row-major, packed over the variable-length batch):
 *   q, k  [T_tot, H, dk]     v, out [T_tot, H, dv]     z (or raw g) [T_tot, H, dk]
 *   beta  [T_tot, H]         state  [N, H, dk, dv]      cu_seqlens [N + 1]
 *
 * Sequences (n) and heads (h) are independent; a plain thread pool walks the
 * (n, h) pairs.  Inside one pair the loop is the per-token recurrence above,
 * with no blocking, fusion or reordering.
 */
#define _GNU_SOURCE
#include <math.h>
#include <pthread.h>
#include <sched.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define KDA_ORACLE_GMIN (-5.0)

/* log-decay g = gmin * sigmoid(z), sigmoid(z) = 1 / (1 + e^{-z}). */
double kda_oracle_log_decay(double z) {
  return KDA_ORACLE_GMIN / (1.0 + exp(-z));
}

/* x / sqrt(sum x^2 + eps), n entries, out may alias x. */
void kda_oracle_l2norm(const double* x, double* out, int n, double eps) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  const double inv = 1.0 / sqrt(ss + eps);
  for (int i = 0; i < n; ++i) out[i] = x[i] * inv;
}

typedef struct {
  int num_seqs, num_heads, dk, dv;
  const int64_t* cu_seqlens;
  const double *q, *k, *v, *z, *beta, *initial_state;
  double *out, *final_state;
  int z_is_raw_log_decay;
  const double* a_log;
  double eps;
  /* work distribution */
  int64_t next_task;
  pthread_mutex_t lock;
} job_t;

static void run_pair(job_t* J, int n, int h) {
  const int H = J->num_heads, dk = J->dk, dv = J->dv;
  double* S = (double*)malloc(sizeof(double) * (size_t)dk * dv);
  double* qh = (double*)malloc(sizeof(double) * dk);
  double* kh = (double*)malloc(sizeof(double) * dk);
  double* a = (double*)malloc(sizeof(double) * dk);
  double* e = (double*)malloc(sizeof(double) * dv);
  const size_t sidx = ((size_t)n * H + h) * dk * dv;
  const double zscale = J->a_log ? exp(J->a_log[h]) : 1.0; /* e^{A_h} */
  if (J->initial_state)
    memcpy(S, J->initial_state + sidx, sizeof(double) * (size_t)dk * dv);
  else
    memset(S, 0, sizeof(double) * (size_t)dk * dv);

  for (int64_t t = J->cu_seqlens[n]; t < J->cu_seqlens[n + 1]; ++t) {
    const size_t th = (size_t)t * H + h;
    kda_oracle_l2norm(J->q + th * dk, qh, dk, J->eps);
    kda_oracle_l2norm(J->k + th * dk, kh, dk, J->eps);
    for (int c = 0; c < dk; ++c) {
      const double zc = J->z[th * dk + c];
      const double g = J->z_is_raw_log_decay ? zc : kda_oracle_log_decay(zscale * zc);
      a[c] = exp(g);
    }
    const double b = J->beta[th];
    const double* vt = J->v + th * dv;
    /* decay: S <- Diag(alpha) S (row c scaled by alpha_c) */
    for (int c = 0; c < dk; ++c)
      for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] *= a[c];
    /* erase + write: e = v - S^T k ; S <- S + beta k e^T */
    for (int j = 0; j < dv; ++j) {
      double acc = 0.0;
      for (int c = 0; c < dk; ++c) acc += S[(size_t)c * dv + j] * kh[c];
      e[j] = vt[j] - acc;
    }
    for (int c = 0; c < dk; ++c)
      for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] += b * kh[c] * e[j];
    /* read: o = S^T q */
    double* ot = J->out + th * dv;
    for (int j = 0; j < dv; ++j) {
      double acc = 0.0;
      for (int c = 0; c < dk; ++c) acc += S[(size_t)c * dv + j] * qh[c];
      ot[j] = acc;
    }
  }
  if (J->final_state)
    memcpy(J->final_state + sidx, S, sizeof(double) * (size_t)dk * dv);
  free(S); free(qh); free(kh); free(a); free(e);
}

static void* worker(void* arg) {
  job_t* J = (job_t*)arg;
  const int64_t total = (int64_t)J->num_seqs * J->num_heads;
  for (;;) {
    pthread_mutex_lock(&J->lock);
    const int64_t task = J->next_task++;
    pthread_mutex_unlock(&J->lock);
    if (task >= total) break;
    run_pair(J, (int)(task / J->num_heads), (int)(task % J->num_heads));
  }
  return NULL;
}

/* Number of CPUs this process may run on. */
int kda_oracle_available_cpus(void) {
  cpu_set_t set;
  CPU_ZERO(&set);
  if (sched_getaffinity(0, sizeof(set), &set) == 0) {
    const int c = CPU_COUNT(&set);
    if (c > 0) return c;
  }
  const long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

/*
 * Run the recurrence over a packed batch.  Returns the number of threads
 * used, or -1 on a bad argument.  initial_state may be NULL (zeros);
 * final_state may be NULL (not written).  z holds logits (gate applied
 * here) unless z_is_raw_log_decay != 0, in which case it holds g itself.
 * a_log ([num_heads], may be NULL = zeros) is the gate's per-head log-scale.
 */
int kda_oracle_recurrent(int num_seqs, int num_heads, int dk, int dv,
                         const int64_t* cu_seqlens, const double* q,
                         const double* k, const double* v, const double* z,
                         const double* beta, const double* initial_state,
                         double* out, double* final_state,
                         int z_is_raw_log_decay, double eps, int num_threads,
                         const double* a_log) {
  if (num_seqs < 0 || num_heads <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens)
    return -1;
  for (int n = 0; n < num_seqs; ++n)
    if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
  job_t J;
  J.num_seqs = num_seqs; J.num_heads = num_heads; J.dk = dk; J.dv = dv;
  J.cu_seqlens = cu_seqlens; J.q = q; J.k = k; J.v = v; J.z = z;
  J.beta = beta; J.initial_state = initial_state; J.out = out;
  J.final_state = final_state; J.z_is_raw_log_decay = z_is_raw_log_decay;
  J.a_log = a_log;
  J.eps = eps; J.next_task = 0;
  pthread_mutex_init(&J.lock, NULL);
  int nt = num_threads > 0 ? num_threads : kda_oracle_available_cpus();
  const int64_t total = (int64_t)num_seqs * num_heads;
  if (nt > total) nt = total > 0 ? (int)total : 1;
  if (nt <= 1) {
    worker(&J);
    nt = 1;
  } else {
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nt);
    for (int i = 0; i < nt; ++i) pthread_create(&th[i], NULL, worker, &J);
    for (int i = 0; i < nt; ++i) pthread_join(th[i], NULL);
    free(th);
  }
  pthread_mutex_destroy(&J.lock);
  return nt;
}

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
#define KDA_ORACLE_BWD_BLOCK 64 /* tokens between stored states in the backward */

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

/* ------------------------------------------------------------------------
 * Backward (reverse mode) of the same per-token recurrence, for one loss L
 * whose gradients with respect to every output o_t (d_out) and to the final
 * state (d_final, may be NULL = 0) are given.  Each step is differentiated
 * as written above, in reverse token order:
 *   o = S_t^T q^          ->  dS_t += q^ do^T,  dq^ = S_t do
 *   S_t = Sb + b k^ e^T   ->  w = dS_t^T k^,  de = b w,  db = e . w,
 *                             dk^ = b dS_t e,  dSb = dS_t
 *   e = v - Sb^T k^       ->  dv = de,  dSb -= k^ de^T,  dk^ -= Sb de
 *   Sb = Diag(alpha) S    ->  dalpha = rowsum(dSb * S),  dS = Diag(alpha) dSb
 *   alpha = exp(g), g = gmin sigmoid(s z), s = e^{A_h}
 *                         ->  dz = dalpha alpha gmin sigmoid (1 - sigmoid) s
 *   x^ = x r, r = (|x|^2 + eps)^{-1/2}  ->  dx = r dx^ - r^3 (x . dx^) x
 * The states S_{t-1} are rebuilt block by block: the forward stores the
 * state before every KDA_ORACLE_BWD_BLOCK tokens and each block is run
 * again, keeping its states, before it is differentiated.
 * ---------------------------------------------------------------------- */

typedef struct {
  int num_seqs, num_heads, dk, dv;
  const int64_t* cu_seqlens;
  const double *q, *k, *v, *z, *beta, *initial_state, *a_log, *d_out, *d_final;
  double *dq, *dk_out, *dv_out, *dz, *dbeta, *d_initial;
  double eps;
  int64_t next_task;
  pthread_mutex_t lock;
} bjob_t;

/* alpha, q^, k^ and the norms of token th */
static void token_inputs(const bjob_t* J, size_t th, double zscale, double* qh, double* kh,
                         double* al, double* rq, double* rk) {
  const int dk = J->dk;
  double sq = 0.0, sk = 0.0;
  for (int c = 0; c < dk; ++c) {
    sq += J->q[th * dk + c] * J->q[th * dk + c];
    sk += J->k[th * dk + c] * J->k[th * dk + c];
  }
  *rq = 1.0 / sqrt(sq + J->eps);
  *rk = 1.0 / sqrt(sk + J->eps);
  for (int c = 0; c < dk; ++c) {
    qh[c] = J->q[th * dk + c] * *rq;
    kh[c] = J->k[th * dk + c] * *rk;
    al[c] = exp(kda_oracle_log_decay(zscale * J->z[th * dk + c]));
  }
}

/* S <- the state after token th, from S (the state before it) */
static void forward_token(const bjob_t* J, size_t th, double zscale, double* S, double* qh,
                          double* kh, double* al, double* e) {
  const int dk = J->dk, dv = J->dv;
  double rq, rk;
  token_inputs(J, th, zscale, qh, kh, al, &rq, &rk);
  for (int c = 0; c < dk; ++c)
    for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] *= al[c];
  for (int j = 0; j < dv; ++j) {
    double acc = 0.0;
    for (int c = 0; c < dk; ++c) acc += S[(size_t)c * dv + j] * kh[c];
    e[j] = J->v[th * dv + j] - acc;
  }
  const double b = J->beta[th];
  for (int c = 0; c < dk; ++c)
    for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] += b * kh[c] * e[j];
}

static void backward_pair(bjob_t* J, int n, int h) {
  const int H = J->num_heads, dk = J->dk, dv = J->dv;
  const size_t ss = (size_t)dk * dv;
  const int64_t t0 = J->cu_seqlens[n], t1 = J->cu_seqlens[n + 1], L = t1 - t0;
  const int nb = (int)((L + KDA_ORACLE_BWD_BLOCK - 1) / KDA_ORACLE_BWD_BLOCK);
  const double zscale = J->a_log ? exp(J->a_log[h]) : 1.0;
  double* ckpt = (double*)malloc(sizeof(double) * ss * (size_t)(nb + 1));
  double* blk = (double*)malloc(sizeof(double) * ss * (KDA_ORACLE_BWD_BLOCK + 1));
  double* S = (double*)malloc(sizeof(double) * ss);
  double* dS = (double*)malloc(sizeof(double) * ss);
  double* dSb = (double*)malloc(sizeof(double) * ss);
  double* qh = (double*)malloc(sizeof(double) * dk);
  double* kh = (double*)malloc(sizeof(double) * dk);
  double* al = (double*)malloc(sizeof(double) * dk);
  double* dqh = (double*)malloc(sizeof(double) * dk);
  double* dkh = (double*)malloc(sizeof(double) * dk);
  double* dal = (double*)malloc(sizeof(double) * dk);
  double* e = (double*)malloc(sizeof(double) * dv);
  double* w = (double*)malloc(sizeof(double) * dv);
  const size_t sidx = ((size_t)n * H + h) * ss;
  if (J->initial_state) memcpy(S, J->initial_state + sidx, sizeof(double) * ss);
  else memset(S, 0, sizeof(double) * ss);
  /* forward: the state before each block */
  for (int b = 0; b < nb; ++b) {
    memcpy(ckpt + (size_t)b * ss, S, sizeof(double) * ss);
    const int64_t e1 = t0 + (int64_t)(b + 1) * KDA_ORACLE_BWD_BLOCK < t1
                           ? t0 + (int64_t)(b + 1) * KDA_ORACLE_BWD_BLOCK : t1;
    for (int64_t t = t0 + (int64_t)b * KDA_ORACLE_BWD_BLOCK; t < e1; ++t)
      forward_token(J, (size_t)t * H + h, zscale, S, qh, kh, al, e);
  }
  if (J->d_final) memcpy(dS, J->d_final + sidx, sizeof(double) * ss);
  else memset(dS, 0, sizeof(double) * ss);
  for (int b = nb - 1; b >= 0; --b) {
    const int64_t b0 = t0 + (int64_t)b * KDA_ORACLE_BWD_BLOCK;
    const int64_t b1 = b0 + KDA_ORACLE_BWD_BLOCK < t1 ? b0 + KDA_ORACLE_BWD_BLOCK : t1;
    /* blk[i] = state before token b0 + i, for i = 0 .. b1 - b0 */
    memcpy(blk, ckpt + (size_t)b * ss, sizeof(double) * ss);
    for (int64_t t = b0; t < b1; ++t) {
      double* nxt = blk + (size_t)(t - b0 + 1) * ss;
      memcpy(nxt, blk + (size_t)(t - b0) * ss, sizeof(double) * ss);
      forward_token(J, (size_t)t * H + h, zscale, nxt, qh, kh, al, e);
    }
    for (int64_t t = b1 - 1; t >= b0; --t) {
      const size_t th = (size_t)t * H + h;
      const double* Sp = blk + (size_t)(t - b0) * ss;     /* S_{t-1} */
      const double* St = blk + (size_t)(t - b0 + 1) * ss; /* S_t */
      double rq, rk;
      token_inputs(J, th, zscale, qh, kh, al, &rq, &rk);
      const double bt = J->beta[th];
      /* e = v - (Diag(alpha) S_{t-1})^T k^ */
      for (int j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int c = 0; c < dk; ++c) acc += al[c] * Sp[(size_t)c * dv + j] * kh[c];
        e[j] = J->v[th * dv + j] - acc;
      }
      const double* dout = J->d_out + th * dv;
      /* read-out */
      for (int c = 0; c < dk; ++c) {
        double acc = 0.0;
        for (int j = 0; j < dv; ++j) {
          dS[(size_t)c * dv + j] += qh[c] * dout[j];
          acc += St[(size_t)c * dv + j] * dout[j];
        }
        dqh[c] = acc;
      }
      /* write: w = dS^T k^, de = b w, db = e . w, dk^ = b dS e */
      double db = 0.0;
      for (int j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int c = 0; c < dk; ++c) acc += dS[(size_t)c * dv + j] * kh[c];
        w[j] = acc;
        db += e[j] * acc;
      }
      for (int c = 0; c < dk; ++c) {
        double acc = 0.0;
        for (int j = 0; j < dv; ++j) acc += dS[(size_t)c * dv + j] * e[j];
        dkh[c] = bt * acc;
      }
      /* erase: dv = de, dSb = dS - k^ de^T, dk^ -= Sb de */
      for (int j = 0; j < dv; ++j) J->dv_out[th * dv + j] = bt * w[j];
      for (int c = 0; c < dk; ++c) {
        double acc = 0.0;
        for (int j = 0; j < dv; ++j) {
          const double de = bt * w[j];
          dSb[(size_t)c * dv + j] = dS[(size_t)c * dv + j] - kh[c] * de;
          acc += al[c] * Sp[(size_t)c * dv + j] * de;
        }
        dkh[c] -= acc;
      }
      /* decay: dalpha = rowsum(dSb * S_{t-1}), dS_{t-1} = Diag(alpha) dSb */
      for (int c = 0; c < dk; ++c) {
        double acc = 0.0;
        for (int j = 0; j < dv; ++j) {
          acc += dSb[(size_t)c * dv + j] * Sp[(size_t)c * dv + j];
          dS[(size_t)c * dv + j] = al[c] * dSb[(size_t)c * dv + j];
        }
        dal[c] = acc;
      }
      /* gate, norms */
      double qd = 0.0, kd = 0.0;
      for (int c = 0; c < dk; ++c) {
        qd += J->q[th * dk + c] * dqh[c];
        kd += J->k[th * dk + c] * dkh[c];
      }
      for (int c = 0; c < dk; ++c) {
        const double zc = zscale * J->z[th * dk + c];
        const double sg = 1.0 / (1.0 + exp(-zc));
        J->dz[th * dk + c] = dal[c] * al[c] * KDA_ORACLE_GMIN * sg * (1.0 - sg) * zscale;
        J->dq[th * dk + c] = rq * dqh[c] - rq * rq * rq * qd * J->q[th * dk + c];
        J->dk_out[th * dk + c] = rk * dkh[c] - rk * rk * rk * kd * J->k[th * dk + c];
      }
      J->dbeta[th] = db;
    }
  }
  if (J->d_initial) memcpy(J->d_initial + sidx, dS, sizeof(double) * ss);
  free(ckpt); free(blk); free(S); free(dS); free(dSb); free(qh); free(kh); free(al);
  free(dqh); free(dkh); free(dal); free(e); free(w);
}

static void* bworker(void* arg) {
  bjob_t* J = (bjob_t*)arg;
  const int64_t total = (int64_t)J->num_seqs * J->num_heads;
  for (;;) {
    pthread_mutex_lock(&J->lock);
    const int64_t task = J->next_task++;
    pthread_mutex_unlock(&J->lock);
    if (task >= total) break;
    backward_pair(J, (int)(task / J->num_heads), (int)(task % J->num_heads));
  }
  return NULL;
}

/*
 * Gradients of L with respect to q, k, v, z, beta and the initial state,
 * given dL/d out (d_out, [T_tot, H, dv]) and dL/d final_state (d_final, may
 * be NULL).  Layouts as kda_oracle_recurrent; every output array is
 * written in full (d_initial may be NULL).  Returns the number of threads
 * used, or -1 on a bad argument.
 */
int kda_oracle_backward(int num_seqs, int num_heads, int dk, int dv,
                        const int64_t* cu_seqlens, const double* q, const double* k,
                        const double* v, const double* z, const double* beta,
                        const double* initial_state, const double* a_log, const double* d_out,
                        const double* d_final, double* dq, double* dkk, double* dvv,
                        double* dz, double* dbeta, double* d_initial, double eps,
                        int num_threads) {
  if (num_seqs < 0 || num_heads <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens) return -1;
  for (int n = 0; n < num_seqs; ++n)
    if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
  bjob_t J;
  J.num_seqs = num_seqs; J.num_heads = num_heads; J.dk = dk; J.dv = dv;
  J.cu_seqlens = cu_seqlens; J.q = q; J.k = k; J.v = v; J.z = z; J.beta = beta;
  J.initial_state = initial_state; J.a_log = a_log; J.d_out = d_out; J.d_final = d_final;
  J.dq = dq; J.dk_out = dkk; J.dv_out = dvv; J.dz = dz; J.dbeta = dbeta;
  J.d_initial = d_initial; J.eps = eps; J.next_task = 0;
  pthread_mutex_init(&J.lock, NULL);
  int nt = num_threads > 0 ? num_threads : kda_oracle_available_cpus();
  const int64_t total = (int64_t)num_seqs * num_heads;
  if (nt > total) nt = total > 0 ? (int)total : 1;
  if (nt <= 1) {
    bworker(&J);
    nt = 1;
  } else {
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nt);
    for (int i = 0; i < nt; ++i) pthread_create(&th[i], NULL, bworker, &J);
    for (int i = 0; i < nt; ++i) pthread_join(th[i], NULL);
    free(th);
  }
  pthread_mutex_destroy(&J.lock);
  return nt;
}

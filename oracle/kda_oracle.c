/*
 * kda_oracle.c -- plain, slow, token-serial fp64 CPU oracle for the
 * Kimi-Delta-Attention (KDA) forward recurrence and its reverse-mode backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may link,
 * load or call this file: only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA path.
 *
 * What it computes (per sequence s and head h, tokens t = 1..L):
 *
 *   q^_t = q_t / sqrt(|q_t|^2 + eps),  k^_t = k_t / sqrt(|k_t|^2 + eps)
 *       (the in-kernel L2 norm whose backward the kernel-B guide inlines in
 *        its B3 epilogue: "bwd-kernelB-beginner-guide-full", Part 2, B3,
 *        optimisation 4 and 7)
 *   gk_t = -exp(A_log[h]) * softplus(g_t + dt_bias[h])   (per channel, K values)
 *       (A_log is a learned per-head scalar and dt_bias a learned per-channel
 *        bias of the gate: same guide, B3 optimisation 7, where the reverse
 *        cumulative sum accumulates dA_log, one scalar per head, and
 *        ddt_bias, one value per channel; dt_bias is nullable = 0)
 *   a_t  = exp(gk_t)
 *   S'_t = Diag(a_t) S_{t-1}
 *   delta_t = v_t - S'_t^T k^_t
 *   S_t  = S'_t + beta_t k^_t delta_t^T
 *        = (I - beta_t k^_t k^_t^T) Diag(a_t) S_{t-1} + beta_t k^_t v_t^T
 *   o_t  = scale * S_t^T q^_t,      S_0 = h0,   S_L = hT
 *
 * S is K x V.  The backward is the hand-derived vector-Jacobian product of
 * exactly these steps, taken token by token in reverse, for the loss
 *   sum_t <dO_t, o_t> + <dh_T, S_L>.
 *
 * Memory: the reverse sweep needs S_{t-1} for every token; states are
 * checkpointed every `chunk` tokens on the forward sweep and the `chunk`
 * states of one segment are recomputed from the checkpoint before that
 * segment is walked backwards.  The checkpoint spacing changes nothing in
 * the arithmetic (the recomputation repeats the same operations in the
 * same order), it only bounds memory.
 *
 * Test hooks (never used by the library): gate_mode = 1 takes g as the
 * per-channel log-decay gk directly; erase = 0 drops the -beta k k^T term
 * (gated linear attention); normalize = 0 skips the L2 norm.
 *
 * Layout: every per-token tensor is token-major [Ttot, H, D] (D = K or V),
 * sequences packed back to back as given by cu_seqlens[num_seqs + 1];
 * beta is [Ttot, H]; A_log is [H]; h0, hT, dh_T, dh0 are [num_seqs, H, K, V].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
  int num_seqs;
  const int64_t *cu_seqlens; /* [num_seqs + 1], cu_seqlens[0] == 0 */
  int H, K, V;
  double scale;              /* read-out scale */
  double eps;                /* added to |x|^2 inside the L2-norm sqrt */
  int gate_mode;             /* 0: gk = -exp(A_log) softplus(g); 1: gk = g */
  int erase;                 /* 1: delta rule; 0: erase term dropped */
  int normalize;             /* 1: L2-normalise q and k; 0: use them as given */
  int chunk;                 /* checkpoint spacing and chunk size of the
                                optional per-chunk state outputs (> 0) */
  int nthreads;              /* OpenMP threads (<= 0: runtime default) */
  const double *dt_bias;     /* nullable [H, K]: bias added to g inside softplus */
} kda_oracle_cfg;

/* the gate pre-activation g_t[i] + dt_bias[h][i] of token element `off` */
static double gate_x(const kda_oracle_cfg *c, const double *g, size_t off, int h, int i) {
  return g[off + i] + (c->dt_bias ? c->dt_bias[(size_t)h * c->K + i] : 0.0);
}

static double softplus(double x) {
  /* log(1 + e^x) written without overflow */
  return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* Per-token preparation shared by the forward and the backward sweep:
 * normalised q, k (and the norms), and the log-decay gk. */
typedef struct {
  int L, K, V;
  double *qn, *kn;   /* [L, K] */
  double *nq, *nk;   /* [L] the norms sqrt(|x|^2 + eps) */
  double *gk;        /* [L, K] */
} unit_prep;

static void prep_unit(const kda_oracle_cfg *c, int s, int h, const double *q,
                      const double *k, const double *g, const double *A_log,
                      unit_prep *p) {
  const int H = c->H, K = c->K;
  const int64_t t0 = c->cu_seqlens[s];
  const int L = (int)(c->cu_seqlens[s + 1] - t0);
  p->L = L;
  p->K = K;
  p->V = c->V;
  p->qn = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * K);
  p->kn = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * K);
  p->gk = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * K);
  p->nq = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
  p->nk = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
  const double A = c->gate_mode == 0 ? exp(A_log[h]) : 0.0;
  for (int t = 0; t < L; ++t) {
    const size_t off = ((size_t)(t0 + t) * H + h) * K;
    double sq = 0.0, sk = 0.0;
    for (int i = 0; i < K; ++i) {
      sq += q[off + i] * q[off + i];
      sk += k[off + i] * k[off + i];
    }
    const double nq = c->normalize ? sqrt(sq + c->eps) : 1.0;
    const double nk = c->normalize ? sqrt(sk + c->eps) : 1.0;
    p->nq[t] = nq;
    p->nk[t] = nk;
    for (int i = 0; i < K; ++i) {
      p->qn[(size_t)t * K + i] = q[off + i] / nq;
      p->kn[(size_t)t * K + i] = k[off + i] / nk;
      p->gk[(size_t)t * K + i] =
          c->gate_mode == 0 ? -A * softplus(gate_x(c, g, off, h, i)) : g[off + i];
    }
  }
}

static void free_prep(unit_prep *p) {
  free(p->qn); free(p->kn); free(p->gk); free(p->nq); free(p->nk);
}

/* One forward token step: S (K x V) holds S_{t-1} on entry and S_t on exit.
 * Sp receives S'_t, delta receives delta_t. */
static void token_step(int K, int V, int erase, const double *kn,
                       const double *gk, const double *v, double beta,
                       double *S, double *Sp, double *delta) {
  for (int i = 0; i < K; ++i) {
    const double a = exp(gk[i]);
    for (int j = 0; j < V; ++j) Sp[(size_t)i * V + j] = a * S[(size_t)i * V + j];
  }
  for (int j = 0; j < V; ++j) {
    double acc = 0.0;
    if (erase)
      for (int i = 0; i < K; ++i) acc += Sp[(size_t)i * V + j] * kn[i];
    delta[j] = v[j] - acc;
  }
  for (int i = 0; i < K; ++i)
    for (int j = 0; j < V; ++j)
      S[(size_t)i * V + j] = Sp[(size_t)i * V + j] + beta * kn[i] * delta[j];
}

static void gather_v(const kda_oracle_cfg *c, const double *v, int64_t tok,
                     int h, double *out) {
  memcpy(out, v + ((size_t)tok * c->H + h) * c->V, sizeof(double) * c->V);
}

/* ------------------------------------------------------------------------ */
/* Forward: o, the final state hT and, optionally, the state at the start of */
/* every chunk of `chunk` tokens ([NTc, H, K, V], NTc = sum ceil(L/chunk)).  */
/* ------------------------------------------------------------------------ */
int kda_oracle_forward(const kda_oracle_cfg *c, const double *q,
                       const double *k, const double *v, const double *g,
                       const double *beta, const double *A_log,
                       const double *h0, double *o, double *hT,
                       double *chunk_states) {
  const int H = c->H, K = c->K, V = c->V, N = c->num_seqs, C = c->chunk;
  if (N < 0 || H <= 0 || K <= 0 || V <= 0 || C <= 0) return 1;
  int64_t *chunk_base = (int64_t *)malloc(sizeof(int64_t) * (N + 1));
  chunk_base[0] = 0;
  for (int s = 0; s < N; ++s) {
    const int64_t L = c->cu_seqlens[s + 1] - c->cu_seqlens[s];
    if (L < 0) { free(chunk_base); return 2; }
    chunk_base[s + 1] = chunk_base[s] + (L + C - 1) / C;
  }
#ifdef _OPENMP
  if (c->nthreads > 0) omp_set_num_threads(c->nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int u = 0; u < N * H; ++u) {
    const int s = u / H, h = u % H;
    unit_prep p;
    prep_unit(c, s, h, q, k, g, A_log, &p);
    const int64_t t0 = c->cu_seqlens[s];
    double *S = (double *)calloc((size_t)K * V, sizeof(double));
    double *Sp = (double *)malloc(sizeof(double) * (size_t)K * V);
    double *delta = (double *)malloc(sizeof(double) * V);
    double *vt = (double *)malloc(sizeof(double) * V);
    if (h0) memcpy(S, h0 + (size_t)u * K * V, sizeof(double) * (size_t)K * V);
    for (int t = 0; t < p.L; ++t) {
      if (chunk_states && t % C == 0) {
        const int64_t n = chunk_base[s] + t / C;
        memcpy(chunk_states + ((size_t)n * H + h) * K * V, S,
               sizeof(double) * (size_t)K * V);
      }
      gather_v(c, v, t0 + t, h, vt);
      token_step(K, V, c->erase, p.kn + (size_t)t * K, p.gk + (size_t)t * K,
                 vt, beta[(size_t)(t0 + t) * H + h], S, Sp, delta);
      if (o) {
        const double *qt = p.qn + (size_t)t * K;
        double *ot = o + ((size_t)(t0 + t) * H + h) * V;
        for (int j = 0; j < V; ++j) {
          double acc = 0.0;
          for (int i = 0; i < K; ++i) acc += S[(size_t)i * V + j] * qt[i];
          ot[j] = c->scale * acc;
        }
      }
    }
    if (hT) memcpy(hT + (size_t)u * K * V, S, sizeof(double) * (size_t)K * V);
    free(S); free(Sp); free(delta); free(vt);
    free_prep(&p);
  }
  free(chunk_base);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Backward.  Outputs (all overwritten): dq, dk, dg [Ttot,H,K]; dv [Ttot,H,V];*/
/* dbeta [Ttot,H]; dA_log [H] (summed over sequences and tokens); ddt_bias  */
/* [H,K] (nullable; summed over sequences and tokens); dh0                   */
/* [N,H,K,V] (nullable); chunk_dstates (nullable) [NTc,H,K,V]: the gradient  */
/* with respect to the state at the END of each chunk, i.e. the adjoint that */
/* enters that chunk's reverse walk.                                         */
/* ------------------------------------------------------------------------ */
int kda_oracle_backward(const kda_oracle_cfg *c, const double *q,
                        const double *k, const double *v, const double *g,
                        const double *beta, const double *A_log,
                        const double *h0, const double *dO, const double *dhT,
                        double *dq, double *dk, double *dv, double *dg,
                        double *dbeta, double *dA_log, double *ddt_bias,
                        double *dh0, double *chunk_dstates) {
  const int H = c->H, K = c->K, V = c->V, N = c->num_seqs, C = c->chunk;
  if (N < 0 || H <= 0 || K <= 0 || V <= 0 || C <= 0) return 1;
  int64_t *chunk_base = (int64_t *)malloc(sizeof(int64_t) * (N + 1));
  chunk_base[0] = 0;
  for (int s = 0; s < N; ++s) {
    const int64_t L = c->cu_seqlens[s + 1] - c->cu_seqlens[s];
    if (L < 0) { free(chunk_base); return 2; }
    chunk_base[s + 1] = chunk_base[s] + (L + C - 1) / C;
  }
  /* per-unit dA_log contributions, summed in a fixed order afterwards */
  double *dA_unit = (double *)calloc((size_t)(N > 0 ? N : 1) * H, sizeof(double));
  /* per-unit ddt_bias contributions, the same way */
  double *db_unit = (double *)calloc((size_t)(N > 0 ? N : 1) * H * K, sizeof(double));
#ifdef _OPENMP
  if (c->nthreads > 0) omp_set_num_threads(c->nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int u = 0; u < N * H; ++u) {
    const int s = u / H, h = u % H;
    unit_prep p;
    prep_unit(c, s, h, q, k, g, A_log, &p);
    const int L = p.L;
    const int64_t t0 = c->cu_seqlens[s];
    const size_t KV = (size_t)K * V;
    const int nck = (L + C - 1) / C;

    /* forward sweep: checkpoint S_{t-1} at the start of every chunk */
    double *ckpt = (double *)malloc(sizeof(double) * KV * (nck > 0 ? nck : 1));
    double *S = (double *)calloc(KV, sizeof(double));
    double *Sp = (double *)malloc(sizeof(double) * KV);
    double *delta = (double *)malloc(sizeof(double) * V);
    double *vt = (double *)malloc(sizeof(double) * V);
    if (h0) memcpy(S, h0 + (size_t)u * KV, sizeof(double) * KV);
    for (int t = 0; t < L; ++t) {
      if (t % C == 0) memcpy(ckpt + (size_t)(t / C) * KV, S, sizeof(double) * KV);
      gather_v(c, v, t0 + t, h, vt);
      token_step(K, V, c->erase, p.kn + (size_t)t * K, p.gk + (size_t)t * K,
                 vt, beta[(size_t)(t0 + t) * H + h], S, Sp, delta);
    }

    /* reverse sweep */
    double *Sprev = (double *)malloc(sizeof(double) * KV * (size_t)(C + 1));
    double *dS = (double *)calloc(KV, sizeof(double));
    double *dSp = (double *)malloc(sizeof(double) * KV);
    double *dqn = (double *)calloc((size_t)(L > 0 ? L : 1) * K, sizeof(double));
    double *dkn = (double *)calloc((size_t)(L > 0 ? L : 1) * K, sizeof(double));
    double *dgk = (double *)calloc((size_t)(L > 0 ? L : 1) * K, sizeof(double));
    double *x = (double *)malloc(sizeof(double) * K);
    double *ddelta = (double *)malloc(sizeof(double) * V);
    if (dhT) memcpy(dS, dhT + (size_t)u * KV, sizeof(double) * KV);
    for (int n = nck - 1; n >= 0; --n) {
      const int ta = n * C, tb = (ta + C < L) ? ta + C : L;
      if (chunk_dstates)
        memcpy(chunk_dstates + ((size_t)(chunk_base[s] + n) * H + h) * KV, dS,
               sizeof(double) * KV);
      /* recompute S_{t-1} for t in [ta, tb] from the checkpoint:
         Sprev[j] = state after token ta + j - 1, i.e. before token ta + j */
      memcpy(Sprev, ckpt + (size_t)n * KV, sizeof(double) * KV);
      for (int t = ta; t < tb; ++t) {
        double *Sn = Sprev + (size_t)(t - ta + 1) * KV;
        memcpy(Sn, Sprev + (size_t)(t - ta) * KV, sizeof(double) * KV);
        gather_v(c, v, t0 + t, h, vt);
        token_step(K, V, c->erase, p.kn + (size_t)t * K, p.gk + (size_t)t * K,
                   vt, beta[(size_t)(t0 + t) * H + h], Sn, Sp, delta);
      }
      for (int t = tb - 1; t >= ta; --t) {
        const double *Sold = Sprev + (size_t)(t - ta) * KV;   /* S_{t-1} */
        const double *Snew = Sprev + (size_t)(t - ta + 1) * KV; /* S_t */
        const double *qt = p.qn + (size_t)t * K;
        const double *kt = p.kn + (size_t)t * K;
        const double *gt = p.gk + (size_t)t * K;
        const double bt = beta[(size_t)(t0 + t) * H + h];
        const double *dOt = dO + ((size_t)(t0 + t) * H + h) * V;
        gather_v(c, v, t0 + t, h, vt);
        /* S'_t and delta_t */
        for (int i = 0; i < K; ++i) {
          const double a = exp(gt[i]);
          for (int j = 0; j < V; ++j) Sp[(size_t)i * V + j] = a * Sold[(size_t)i * V + j];
        }
        for (int j = 0; j < V; ++j) {
          double acc = 0.0;
          if (c->erase)
            for (int i = 0; i < K; ++i) acc += Sp[(size_t)i * V + j] * kt[i];
          delta[j] = vt[j] - acc;
        }
        /* 1. read-out: o_t = scale S_t^T q^_t */
        for (int i = 0; i < K; ++i)
          for (int j = 0; j < V; ++j) dS[(size_t)i * V + j] += c->scale * qt[i] * dOt[j];
        /* 2. dq^_t = scale S_t dO_t */
        for (int i = 0; i < K; ++i) {
          double acc = 0.0;
          for (int j = 0; j < V; ++j) acc += Snew[(size_t)i * V + j] * dOt[j];
          dqn[(size_t)t * K + i] = c->scale * acc;
        }
        /* 3. write term S_t = S'_t + beta k delta^T */
        for (int i = 0; i < K; ++i) {
          double acc = 0.0;
          for (int j = 0; j < V; ++j) acc += dS[(size_t)i * V + j] * delta[j];
          x[i] = acc;                                    /* dS delta */
        }
        double db = 0.0;
        for (int i = 0; i < K; ++i) db += kt[i] * x[i];
        dbeta[(size_t)(t0 + t) * H + h] = db;             /* k^T dS delta */
        for (int j = 0; j < V; ++j) {
          double acc = 0.0;
          for (int i = 0; i < K; ++i) acc += dS[(size_t)i * V + j] * kt[i];
          ddelta[j] = bt * acc;                          /* beta dS^T k */
        }
        double *dvt = dv + ((size_t)(t0 + t) * H + h) * V;
        for (int j = 0; j < V; ++j) dvt[j] = ddelta[j];  /* delta = v - ... */
        /* 4. dk^_t = beta dS delta - S'_t ddelta (second term: erase) */
        for (int i = 0; i < K; ++i) {
          double acc = 0.0;
          if (c->erase)
            for (int j = 0; j < V; ++j) acc += Sp[(size_t)i * V + j] * ddelta[j];
          dkn[(size_t)t * K + i] = bt * x[i] - acc;
        }
        /* 5. dS' = dS - k ddelta^T (erase only) */
        for (int i = 0; i < K; ++i)
          for (int j = 0; j < V; ++j)
            dSp[(size_t)i * V + j] =
                dS[(size_t)i * V + j] - (c->erase ? kt[i] * ddelta[j] : 0.0);
        /* 6. S'_t = Diag(a_t) S_{t-1}: gate and carry */
        for (int i = 0; i < K; ++i) {
          const double a = exp(gt[i]);
          double acc = 0.0;
          for (int j = 0; j < V; ++j) acc += dSp[(size_t)i * V + j] * Sold[(size_t)i * V + j];
          dgk[(size_t)t * K + i] = a * acc;              /* da * da/dgk */
          for (int j = 0; j < V; ++j) dS[(size_t)i * V + j] = a * dSp[(size_t)i * V + j];
        }
      }
    }
    if (dh0) memcpy(dh0 + (size_t)u * KV, dS, sizeof(double) * KV);

    /* L2-norm backward and gate chain */
    const double A = c->gate_mode == 0 ? exp(A_log[h]) : 0.0;
    double dA = 0.0;
    for (int t = 0; t < L; ++t) {
      const size_t off = ((size_t)(t0 + t) * H + h) * K;
      const double *qt = p.qn + (size_t)t * K, *kt = p.kn + (size_t)t * K;
      const double *dqt = dqn + (size_t)t * K, *dkt = dkn + (size_t)t * K;
      double pq = 0.0, pk = 0.0;
      for (int i = 0; i < K; ++i) { pq += qt[i] * dqt[i]; pk += kt[i] * dkt[i]; }
      for (int i = 0; i < K; ++i) {
        if (c->normalize) {
          dq[off + i] = (dqt[i] - qt[i] * pq) / p.nq[t];
          dk[off + i] = (dkt[i] - kt[i] * pk) / p.nk[t];
        } else {
          dq[off + i] = dqt[i];
          dk[off + i] = dkt[i];
        }
        const double d = dgk[(size_t)t * K + i];
        if (c->gate_mode == 0) {
          /* d softplus = sigmoid; the bias enters like g */
          dg[off + i] = d * (-A) * sigmoid(gate_x(c, g, off, h, i));
          db_unit[(size_t)u * K + i] += dg[off + i];
          dA += d * p.gk[(size_t)t * K + i];             /* d gk / d A_log = gk */
        } else {
          dg[off + i] = d;
        }
      }
    }
    dA_unit[u] = dA;

    free(ckpt); free(S); free(Sp); free(delta); free(vt);
    free(Sprev); free(dS); free(dSp); free(dqn); free(dkn); free(dgk);
    free(x); free(ddelta);
    free_prep(&p);
  }
  if (dA_log)
    for (int h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int s = 0; s < N; ++s) acc += dA_unit[(size_t)s * H + h];
      dA_log[h] = acc;
    }
  if (ddt_bias)
    for (int h = 0; h < H; ++h)
      for (int i = 0; i < K; ++i) {
        double acc = 0.0;
        for (int s = 0; s < N; ++s) acc += db_unit[((size_t)s * H + h) * K + i];
        ddt_bias[(size_t)h * K + i] = acc;
      }
  free(dA_unit);
  free(db_unit);
  free(chunk_base);
  return 0;
}

int kda_oracle_abi_version(void) { return 2; }

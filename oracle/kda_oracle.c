/*
 * kda_oracle.c -- plain, slow, fp64 CPU reference of the Kimi Delta Attention
 * (KDA) forward pass, and of its backward pass (reverse mode of the same token
 * recurrence, at the end of this file).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path calls, links or loads
 * this file; only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark do.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes (for every sequence n and head h, in any order):
 *
 *   prep, per token t and channel c   (flags use_gate_in_kernel,
 *   use_qk_l2norm_in_kernel, use_beta_sigmoid_in_kernel, safe_gate with
 *   lower_bound in [-5, 0]: "How to Use FlashKDA as a Backend for
 *   flash-linear-attention", sections "Running Inference with chunk_kda" and
 *   "Kernel API and Tensor Requirements"):
 *       a        = exp(A_log[h]) * (g[t,h,c] + dt_bias[h,c])
 *       log a_c  = lower_bound * sigmoid(a)            in [lower_bound, 0]
 *       qn       = q / sqrt(sum q^2 + 1e-6),  kn likewise
 *       beta_t   = sigmoid(beta[t,h]),  sigmoid(x) = 1 / (1 + exp(-x))
 *   The pages give the flags and the bound but not the elementwise form; the
 *   form above is this project's stated reading, used identically on the GPU.
 *
 *   recurrence (the KDA gated delta rule that the GEMMs drive: "How FlashKDA
 *   Integrates with CUTLASS ...", section "Kernel Launch Pipeline and Template
 *   Dispatching"; K = V = 128):
 *       S_t = (I - beta_t kn_t kn_t^T) Diag(alpha_t) S_{t-1} + beta_t kn_t v_t^T
 *       o_t = scale * S_t^T qn_t
 *   evaluated as  S <- Diag(alpha) S;  u = beta (v - S^T kn);  S <- S + kn u^T,
 *   which is the same expression with the product expanded.
 *
 *   state layout: the state tensors are [N, H, V, K], i.e. element
 *   (n, h, v, k) holds S[k][v] ("How to Use FlashKDA ...", section "State
 *   Handling and Variable-Length Batches"; transpose_state_layout=True in
 *   "Running Inference with chunk_kda").  A missing initial state is zero.
 *
 *   varlen: sequence n covers packed tokens [cu[n], cu[n+1]) ("How FlashKDA
 *   Integrates with CUTLASS ...", section "Variable-Length Sequence Support").
 *
 *   grouped value heads (HV > H, named as a variant the SM90 kernel leaves to
 *   the fused CUDA path: "feat(kda): SM90 FlashKDA prefill, intracard CP, and
 *   backend dispatch", description): the pages give no formula, so this is the
 *   project's reading.  Everything that belongs to one state -- v, g, beta,
 *   A_log, dt_bias, out and the states -- has HV heads; q and k have HK heads
 *   with HV a multiple of HK, and value head h reads q/k head h / (HV / HK)
 *   (consecutive value heads share a key head).  HK = HV is the plain case.
 *
 * The chunked function restates the same result in the chunked WY/UT form the
 * pages describe for the GPU kernels ("feat(kda): SM90 FlashKDA prefill,
 * intracard CP, and backend dispatch", commit notes: K1 prepares decayed q/k,
 * beta and the WY inverse per chunk; K2 runs the inter-chunk recurrence).  It is
 * written from the algebra, without blocking, and serves only as a second,
 * independent check of the token loop.
 *
 * All inputs arrive as fp64 values that are exact copies of the bf16 / fp32
 * tensors the GPU reads.  Arithmetic is IEEE fp64; build without -ffast-math.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define KD 128 /* head dimension K = V = 128 */

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* Elementwise preparation of one (token, head) row. */
static void prep_row(const double* q, const double* k, const double* g, double beta_raw,
                     double A_log_h, const double* dt_bias_h, double lower_bound,
                     double* qn, double* kn, double* log_alpha, double* beta) {
  double sq = 0.0, sk = 0.0;
  for (int c = 0; c < KD; ++c) {
    sq += q[c] * q[c];
    sk += k[c] * k[c];
  }
  const double rq = 1.0 / sqrt(sq + 1e-6);
  const double rk = 1.0 / sqrt(sk + 1e-6);
  const double ea = exp(A_log_h);
  for (int c = 0; c < KD; ++c) {
    qn[c] = q[c] * rq;
    kn[c] = k[c] * rk;
    log_alpha[c] = lower_bound * sigmoid(ea * (g[c] + dt_bias_h[c]));
  }
  *beta = sigmoid(beta_raw);
}

/* Public: prep over n_tok packed tokens x H heads, [tok][H][128] layouts. */
void kda_oracle_prep(int64_t n_tok, int32_t H, const double* q, const double* k,
                     const double* g, const double* beta_raw, const double* A_log,
                     const double* dt_bias, double lower_bound, double* qn, double* kn,
                     double* log_alpha, double* beta) {
  for (int64_t t = 0; t < n_tok; ++t)
    for (int32_t h = 0; h < H; ++h) {
      const int64_t r = (t * H + h) * KD;
      prep_row(q + r, k + r, g + r, beta_raw[t * H + h], A_log[h], dt_bias + (int64_t)h * KD,
               lower_bound, qn + r, kn + r, log_alpha + r, beta + t * H + h);
    }
}

typedef struct {
  int64_t T_total;
  int32_t H, N; /* H: value heads (one state each) */
  int32_t HK;   /* q/k heads; value head h reads q/k head h / (H / HK) */
  const int64_t* cu;
  const double *q, *k, *v, *g, *beta_raw, *A_log, *dt_bias;
  double lower_bound, scale;
  const double* init; /* [N][H][V][K] or NULL */
  double* out;        /* [T_total][H][V] */
  double* fin;        /* [N][H][V][K] or NULL */
  int32_t chunk;      /* 0: token loop; >0: chunked WY form with this chunk length */
  int32_t nthreads;
  int32_t tid;
} job_t;

/* ---- token-by-token recurrence for one (sequence, head) ---------------- */
static void run_unit_token(const job_t* J, int32_t n, int32_t h) {
  double* S = (double*)calloc((size_t)KD * KD, sizeof(double)); /* S[k][v] */
  double qn[KD], kn[KD], la[KD], a[KD], sk[KD], u[KD], beta;
  if (J->init)
    for (int vv = 0; vv < KD; ++vv)
      for (int kk = 0; kk < KD; ++kk)
        S[kk * KD + vv] = J->init[(((int64_t)n * J->H + h) * KD + vv) * KD + kk];
  const int32_t hk = h / (J->H / J->HK);
  for (int64_t t = J->cu[n]; t < J->cu[n + 1]; ++t) {
    const int64_t r = (t * J->H + h) * KD, rk = (t * J->HK + hk) * KD;
    prep_row(J->q + rk, J->k + rk, J->g + r, J->beta_raw[t * J->H + h], J->A_log[h],
             J->dt_bias + (int64_t)h * KD, J->lower_bound, qn, kn, la, &beta);
    for (int kk = 0; kk < KD; ++kk) a[kk] = exp(la[kk]);
    /* S <- Diag(alpha) S */
    for (int kk = 0; kk < KD; ++kk)
      for (int vv = 0; vv < KD; ++vv) S[kk * KD + vv] *= a[kk];
    /* u = beta (v - S^T kn) */
    for (int vv = 0; vv < KD; ++vv) sk[vv] = 0.0;
    for (int kk = 0; kk < KD; ++kk)
      for (int vv = 0; vv < KD; ++vv) sk[vv] += S[kk * KD + vv] * kn[kk];
    for (int vv = 0; vv < KD; ++vv) u[vv] = beta * (J->v[r + vv] - sk[vv]);
    /* S <- S + kn u^T */
    for (int kk = 0; kk < KD; ++kk)
      for (int vv = 0; vv < KD; ++vv) S[kk * KD + vv] += kn[kk] * u[vv];
    /* o = scale S^T qn */
    for (int vv = 0; vv < KD; ++vv) sk[vv] = 0.0;
    for (int kk = 0; kk < KD; ++kk)
      for (int vv = 0; vv < KD; ++vv) sk[vv] += S[kk * KD + vv] * qn[kk];
    for (int vv = 0; vv < KD; ++vv) J->out[r + vv] = J->scale * sk[vv];
  }
  if (J->fin)
    for (int vv = 0; vv < KD; ++vv)
      for (int kk = 0; kk < KD; ++kk)
        J->fin[(((int64_t)n * J->H + h) * KD + vv) * KD + kk] = S[kk * KD + vv];
  free(S);
}

/* ---- chunked WY / UT formulation for one (sequence, head) ---------------
 * For a chunk of c tokens with start state S, cumulative in-chunk log-decay
 * gam_r = sum_{s<=r} log alpha_s (per channel) and Gam_r = exp(gam_r):
 *   A[i][j] = beta_i sum_k kn_i[k] exp(gam_i[k]-gam_j[k]) kn_j[k]   (i > j)
 *   L = I + A (unit lower triangular),  Linv = L^{-1}
 *   W  = Linv Diag(beta) (Kn o Gam),   Ut = Linv Diag(beta) V
 *   U  = Ut - W S
 *   P[i][j] = sum_k qn_i[k] exp(gam_i[k]-gam_j[k]) kn_j[k]          (j <= i)
 *   O  = scale ((Qn o Gam) S + P U)
 *   S' = Diag(Gam_{c-1}) S + sum_j Diag(exp(gam_{c-1}-gam_j)) kn_j u_j^T
 */
static void run_unit_chunked(const job_t* J, int32_t n, int32_t h) {
  const int C = J->chunk;
  const int64_t bos = J->cu[n], eos = J->cu[n + 1];
  double* S = (double*)calloc((size_t)KD * KD, sizeof(double));
  double* qn = (double*)malloc(sizeof(double) * C * KD);
  double* kn = (double*)malloc(sizeof(double) * C * KD);
  double* gam = (double*)malloc(sizeof(double) * C * KD);
  double* bt = (double*)malloc(sizeof(double) * C);
  double* A = (double*)malloc(sizeof(double) * C * C);
  double* Li = (double*)malloc(sizeof(double) * C * C);
  double* W = (double*)malloc(sizeof(double) * C * KD);
  double* Ut = (double*)malloc(sizeof(double) * C * KD);
  double* U = (double*)malloc(sizeof(double) * C * KD);
  double* P = (double*)malloc(sizeof(double) * C * C);
  double* Sn = (double*)malloc(sizeof(double) * KD * KD);
  double la[KD];
  const int32_t hk = h / (J->H / J->HK);
  if (J->init)
    for (int vv = 0; vv < KD; ++vv)
      for (int kk = 0; kk < KD; ++kk)
        S[kk * KD + vv] = J->init[(((int64_t)n * J->H + h) * KD + vv) * KD + kk];
  for (int64_t t0 = bos; t0 < eos; t0 += C) {
    const int c = (int)((eos - t0) < C ? (eos - t0) : C);
    for (int r = 0; r < c; ++r) {
      const int64_t row = ((t0 + r) * J->H + h) * KD, rowk = ((t0 + r) * J->HK + hk) * KD;
      prep_row(J->q + rowk, J->k + rowk, J->g + row, J->beta_raw[(t0 + r) * J->H + h],
               J->A_log[h], J->dt_bias + (int64_t)h * KD, J->lower_bound, qn + r * KD,
               kn + r * KD, la, bt + r);
      for (int kk = 0; kk < KD; ++kk)
        gam[r * KD + kk] = la[kk] + (r ? gam[(r - 1) * KD + kk] : 0.0);
    }
    /* A (strictly lower) and P (lower incl. diagonal) */
    for (int i = 0; i < c; ++i)
      for (int j = 0; j < c; ++j) {
        double sa = 0.0, sp = 0.0;
        if (j <= i)
          for (int kk = 0; kk < KD; ++kk) {
            const double d = exp(gam[i * KD + kk] - gam[j * KD + kk]);
            sa += kn[i * KD + kk] * d * kn[j * KD + kk];
            sp += qn[i * KD + kk] * d * kn[j * KD + kk];
          }
        A[i * C + j] = (j < i) ? bt[i] * sa : 0.0;
        P[i * C + j] = (j <= i) ? sp : 0.0;
      }
    /* Linv by forward substitution, one column at a time: (I + A) x = e_j */
    for (int j = 0; j < c; ++j)
      for (int i = 0; i < c; ++i) {
        double x = (i == j) ? 1.0 : 0.0;
        for (int m = 0; m < i; ++m) x -= A[i * C + m] * Li[m * C + j];
        Li[i * C + j] = x;
      }
    /* W, Ut */
    for (int i = 0; i < c; ++i)
      for (int kk = 0; kk < KD; ++kk) {
        double sw = 0.0, su = 0.0;
        for (int j = 0; j < c; ++j) {
          const double lb = Li[i * C + j] * bt[j];
          sw += lb * kn[j * KD + kk] * exp(gam[j * KD + kk]);
          su += lb * J->v[((t0 + j) * J->H + h) * KD + kk];
        }
        W[i * KD + kk] = sw;
        Ut[i * KD + kk] = su;
      }
    /* U = Ut - W S */
    for (int i = 0; i < c; ++i)
      for (int vv = 0; vv < KD; ++vv) {
        double s = 0.0;
        for (int kk = 0; kk < KD; ++kk) s += W[i * KD + kk] * S[kk * KD + vv];
        U[i * KD + vv] = Ut[i * KD + vv] - s;
      }
    /* O = scale ((Qn o Gam) S + P U) */
    for (int i = 0; i < c; ++i)
      for (int vv = 0; vv < KD; ++vv) {
        double s = 0.0;
        for (int kk = 0; kk < KD; ++kk)
          s += qn[i * KD + kk] * exp(gam[i * KD + kk]) * S[kk * KD + vv];
        for (int j = 0; j <= i; ++j) s += P[i * C + j] * U[j * KD + vv];
        J->out[((t0 + i) * J->H + h) * KD + vv] = J->scale * s;
      }
    /* S' = Diag(Gam_last) S + sum_j Diag(exp(gam_last - gam_j)) kn_j u_j^T */
    for (int kk = 0; kk < KD; ++kk) {
      const double gl = gam[(c - 1) * KD + kk];
      for (int vv = 0; vv < KD; ++vv) {
        double s = exp(gl) * S[kk * KD + vv];
        for (int j = 0; j < c; ++j)
          s += exp(gl - gam[j * KD + kk]) * kn[j * KD + kk] * U[j * KD + vv];
        Sn[kk * KD + vv] = s;
      }
    }
    memcpy(S, Sn, sizeof(double) * KD * KD);
  }
  if (J->fin)
    for (int vv = 0; vv < KD; ++vv)
      for (int kk = 0; kk < KD; ++kk)
        J->fin[(((int64_t)n * J->H + h) * KD + vv) * KD + kk] = S[kk * KD + vv];
  free(S); free(qn); free(kn); free(gam); free(bt); free(A); free(Li);
  free(W); free(Ut); free(U); free(P); free(Sn);
}

static void* worker(void* arg) {
  const job_t* J = (const job_t*)arg;
  const int64_t units = (int64_t)J->N * J->H;
  for (int64_t u = J->tid; u < units; u += J->nthreads) {
    const int32_t n = (int32_t)(u / J->H), h = (int32_t)(u % J->H);
    if (J->chunk > 0)
      run_unit_chunked(J, n, h);
    else
      run_unit_token(J, n, h);
  }
  return NULL;
}

static int run_all(job_t* base) {
  int nt = base->nthreads < 1 ? 1 : base->nthreads;
  const int64_t units = (int64_t)base->N * base->H;
  if (units < nt) nt = (int)(units > 0 ? units : 1);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nt);
  job_t* jobs = (job_t*)malloc(sizeof(job_t) * nt);
  for (int i = 0; i < nt; ++i) {
    jobs[i] = *base;
    jobs[i].nthreads = nt;
    jobs[i].tid = i;
  }
  for (int i = 1; i < nt; ++i) pthread_create(&th[i], NULL, worker, &jobs[i]);
  worker(&jobs[0]);
  for (int i = 1; i < nt; ++i) pthread_join(th[i], NULL);
  free(th);
  free(jobs);
  return nt;
}

/*
 * Public: forward over packed tokens.  q, k: [T_total][HK][128]; v, g:
 * [T_total][H][128]; beta: [T_total][H]; A_log: [H]; dt_bias: [H][128]; H a
 * multiple of HK (value head h reads q/k head h / (H / HK)); cu: [N+1] prefix sums
 * with cu[0] = 0 and cu[N] = T_total; init/fin: [N][H][V][K] or NULL;
 * out: [T_total][H][V].  chunk = 0 runs the token loop, chunk > 0 the chunked
 * WY form.  Returns the number of threads used.
 */
int kda_oracle_fwd(int64_t T_total, int32_t H, int32_t HK, int32_t N, const int64_t* cu,
                   const double* q,
                   const double* k, const double* v, const double* g, const double* beta_raw,
                   const double* A_log, const double* dt_bias, double lower_bound, double scale,
                   const double* init, double* out, double* fin, int32_t chunk,
                   int32_t nthreads) {
  job_t J;
  memset(&J, 0, sizeof(J));
  J.T_total = T_total;
  J.H = H;
  J.HK = (HK > 0 && H % HK == 0) ? HK : H;
  J.N = N;
  J.cu = cu;
  J.q = q;
  J.k = k;
  J.v = v;
  J.g = g;
  J.beta_raw = beta_raw;
  J.A_log = A_log;
  J.dt_bias = dt_bias;
  J.lower_bound = lower_bound;
  J.scale = scale;
  J.init = init;
  J.out = out;
  J.fin = fin;
  J.chunk = chunk;
  J.nthreads = nthreads;
  return run_all(&J);
}

/* ======================================================================
 * Backward pass (reverse mode of the token recurrence above), fp64.
 *
 * Given dL/do_t for every token and dL/dS_final for every sequence (either
 * may be zero), returns dL/d(every input).  Per token, in reverse order, with
 * S' = Diag(alpha) S_{t-1}, d = S'^T kn, u = beta (v - d), S_t = S' + kn u^T,
 * o_t = scale S_t^T qn and dS = dL/dS_t:
 *   dS  += scale qn do^T               dqn  = scale S_t do
 *   du   = dS^T kn                     dkn += dS u
 *   dbeta = du . (v - d)               dv   = beta du          dd = -beta du
 *   dS'  = dS + kn dd^T                dkn += S' dd
 *   dalpha[k] = sum_v dS'[k][v] S_{t-1}[k][v]                  dS_{t-1} = Diag(alpha) dS'
 * then the prep chain back to the raw inputs:
 *   dla = dalpha alpha;  da = dla lb s (1 - s), s = sigmoid(a), a = e (g + dt_bias), e = exp(A_log)
 *   dg = da e;  ddt_bias += da e;  dA_log += sum_k da a
 *   dq = r dqn - r^3 (q . dqn) q,  r = (|q|^2 + 1e-6)^(-1/2)  (k likewise)
 *   dbeta_raw = dbeta beta (1 - beta)
 * States S_{t-1} are recomputed from checkpoints every 64 tokens, so memory is
 * bounded by 64 states per worker.  Work is split over key heads: a worker owns
 * the key head's dq / dk rows and the dA_log / dt_bias sums of its value heads.
 * ====================================================================== */
#define BWD_CK 64

typedef struct {
  int64_t T_total;
  int32_t H, HK, N;
  const int64_t* cu;
  const double *q, *k, *v, *g, *beta_raw, *A_log, *dt_bias;
  double lower_bound, scale;
  const double *init, *dout, *dfin; /* init / dfin: [N][H][V][K] or NULL */
  double *dq, *dk, *dv, *dg, *dbeta, *dA_log, *ddt_bias, *dinit;
  int32_t nthreads, tid;
} bwd_job_t;

/* one (sequence, value head) unit */
static void bwd_unit(const bwd_job_t* J, int32_t n, int32_t h) {
  const int32_t hk = h / (J->H / J->HK);
  const int64_t bos = J->cu[n], eos = J->cu[n + 1], len = eos - bos;
  const size_t SS = (size_t)KD * KD;
  double* S = (double*)calloc(SS, sizeof(double));          /* running state S[k][v] */
  double* ck = (double*)malloc(sizeof(double) * SS * (size_t)((len + BWD_CK - 1) / BWD_CK + 1));
  double* blk = (double*)malloc(sizeof(double) * SS * BWD_CK); /* S_{t-1} of one block */
  double* dS = (double*)calloc(SS, sizeof(double));
  double* Sp = (double*)malloc(sizeof(double) * SS);
  double qn[KD], kn[KD], la[KD], al[KD], d[KD], u[KD], beta;
  if (J->init)
    for (int vv = 0; vv < KD; ++vv)
      for (int kk = 0; kk < KD; ++kk)
        S[kk * KD + vv] = J->init[(((int64_t)n * J->H + h) * KD + vv) * KD + kk];
  /* forward: checkpoints S at t = bos + 64 m */
  for (int64_t t = bos; t < eos; ++t) {
    if ((t - bos) % BWD_CK == 0) memcpy(ck + SS * (size_t)((t - bos) / BWD_CK), S, sizeof(double) * SS);
    const int64_t r = (t * J->H + h) * KD, rk = (t * J->HK + hk) * KD;
    prep_row(J->q + rk, J->k + rk, J->g + r, J->beta_raw[t * J->H + h], J->A_log[h],
             J->dt_bias + (int64_t)h * KD, J->lower_bound, qn, kn, la, &beta);
    for (int kk = 0; kk < KD; ++kk) {
      const double a = exp(la[kk]);
      for (int vv = 0; vv < KD; ++vv) S[kk * KD + vv] *= a;
    }
    for (int vv = 0; vv < KD; ++vv) d[vv] = 0.0;
    for (int kk = 0; kk < KD; ++kk)
      for (int vv = 0; vv < KD; ++vv) d[vv] += S[kk * KD + vv] * kn[kk];
    for (int vv = 0; vv < KD; ++vv) u[vv] = beta * (J->v[r + vv] - d[vv]);
    for (int kk = 0; kk < KD; ++kk)
      for (int vv = 0; vv < KD; ++vv) S[kk * KD + vv] += kn[kk] * u[vv];
  }
  /* dS = dL/dS_final */
  if (J->dfin)
    for (int vv = 0; vv < KD; ++vv)
      for (int kk = 0; kk < KD; ++kk)
        dS[kk * KD + vv] = J->dfin[(((int64_t)n * J->H + h) * KD + vv) * KD + kk];
  const double ea = exp(J->A_log[h]);
  const int64_t nblk = (len + BWD_CK - 1) / BWD_CK;
  for (int64_t b = nblk - 1; b >= 0; --b) {
    const int64_t t0 = bos + b * BWD_CK, t1 = (t0 + BWD_CK < eos) ? t0 + BWD_CK : eos;
    /* recompute S_{t-1} for t in [t0, t1) */
    memcpy(S, ck + SS * (size_t)b, sizeof(double) * SS);
    for (int64_t t = t0; t < t1; ++t) {
      memcpy(blk + SS * (size_t)(t - t0), S, sizeof(double) * SS);
      const int64_t r = (t * J->H + h) * KD, rk = (t * J->HK + hk) * KD;
      prep_row(J->q + rk, J->k + rk, J->g + r, J->beta_raw[t * J->H + h], J->A_log[h],
               J->dt_bias + (int64_t)h * KD, J->lower_bound, qn, kn, la, &beta);
      for (int kk = 0; kk < KD; ++kk) {
        const double a = exp(la[kk]);
        for (int vv = 0; vv < KD; ++vv) S[kk * KD + vv] *= a;
      }
      for (int vv = 0; vv < KD; ++vv) d[vv] = 0.0;
      for (int kk = 0; kk < KD; ++kk)
        for (int vv = 0; vv < KD; ++vv) d[vv] += S[kk * KD + vv] * kn[kk];
      for (int vv = 0; vv < KD; ++vv) u[vv] = beta * (J->v[r + vv] - d[vv]);
      for (int kk = 0; kk < KD; ++kk)
        for (int vv = 0; vv < KD; ++vv) S[kk * KD + vv] += kn[kk] * u[vv];
    }
    for (int64_t t = t1 - 1; t >= t0; --t) {
      const double* Sm = blk + SS * (size_t)(t - t0); /* S_{t-1} */
      const int64_t r = (t * J->H + h) * KD, rk = (t * J->HK + hk) * KD;
      prep_row(J->q + rk, J->k + rk, J->g + r, J->beta_raw[t * J->H + h], J->A_log[h],
               J->dt_bias + (int64_t)h * KD, J->lower_bound, qn, kn, la, &beta);
      for (int kk = 0; kk < KD; ++kk) al[kk] = exp(la[kk]);
      /* recompute S' = Diag(alpha) S_{t-1}, d, u and S_t */
      for (int kk = 0; kk < KD; ++kk)
        for (int vv = 0; vv < KD; ++vv) Sp[kk * KD + vv] = al[kk] * Sm[kk * KD + vv];
      for (int vv = 0; vv < KD; ++vv) d[vv] = 0.0;
      for (int kk = 0; kk < KD; ++kk)
        for (int vv = 0; vv < KD; ++vv) d[vv] += Sp[kk * KD + vv] * kn[kk];
      for (int vv = 0; vv < KD; ++vv) u[vv] = beta * (J->v[r + vv] - d[vv]);
      const double* dout = J->dout + r;
      double dqn[KD], dkn[KD], du[KD], dd[KD], dal[KD], dbeta = 0.0;
      /* o = scale S_t^T qn, S_t = S' + kn u^T */
      for (int kk = 0; kk < KD; ++kk) {
        double s = 0.0;
        for (int vv = 0; vv < KD; ++vv) s += (Sp[kk * KD + vv] + kn[kk] * u[vv]) * dout[vv];
        dqn[kk] = J->scale * s;
        for (int vv = 0; vv < KD; ++vv) dS[kk * KD + vv] += J->scale * qn[kk] * dout[vv];
      }
      for (int vv = 0; vv < KD; ++vv) {
        double s = 0.0;
        for (int kk = 0; kk < KD; ++kk) s += dS[kk * KD + vv] * kn[kk];
        du[vv] = s;
      }
      for (int kk = 0; kk < KD; ++kk) {
        double s = 0.0;
        for (int vv = 0; vv < KD; ++vv) s += dS[kk * KD + vv] * u[vv];
        dkn[kk] = s;
      }
      for (int vv = 0; vv < KD; ++vv) {
        dbeta += du[vv] * (J->v[r + vv] - d[vv]);
        J->dv[r + vv] = beta * du[vv];
        dd[vv] = -beta * du[vv];
      }
      /* dS' = dS + kn dd^T ; dkn += S' dd ; dalpha ; dS_{t-1} = Diag(alpha) dS' */
      for (int kk = 0; kk < KD; ++kk) {
        double s = 0.0, sa = 0.0;
        for (int vv = 0; vv < KD; ++vv) {
          const double dsp = dS[kk * KD + vv] + kn[kk] * dd[vv];
          s += Sp[kk * KD + vv] * dd[vv];
          sa += dsp * Sm[kk * KD + vv];
          dS[kk * KD + vv] = al[kk] * dsp;
        }
        dkn[kk] += s;
        dal[kk] = sa;
      }
      /* prep chain */
      double qq = 0.0, kk2 = 0.0, qd = 0.0, kd = 0.0;
      const double* qr = J->q + rk;
      const double* kr = J->k + rk;
      for (int c = 0; c < KD; ++c) {
        qq += qr[c] * qr[c];
        kk2 += kr[c] * kr[c];
        qd += qr[c] * dqn[c];
        kd += kr[c] * dkn[c];
      }
      const double rq = 1.0 / sqrt(qq + 1e-6), rkn = 1.0 / sqrt(kk2 + 1e-6);
      for (int c = 0; c < KD; ++c) {
        J->dq[rk + c] += rq * dqn[c] - rq * rq * rq * qd * qr[c];
        J->dk[rk + c] += rkn * dkn[c] - rkn * rkn * rkn * kd * kr[c];
        const double a = ea * (J->g[r + c] + J->dt_bias[(int64_t)h * KD + c]);
        const double sg = sigmoid(a);
        const double da = dal[c] * al[c] * J->lower_bound * sg * (1.0 - sg);
        J->dg[r + c] = da * ea;
        J->ddt_bias[(int64_t)h * KD + c] += da * ea;
        J->dA_log[h] += da * a;
      }
      J->dbeta[t * J->H + h] = dbeta * beta * (1.0 - beta);
    }
  }
  if (J->dinit)
    for (int vv = 0; vv < KD; ++vv)
      for (int kk = 0; kk < KD; ++kk)
        J->dinit[(((int64_t)n * J->H + h) * KD + vv) * KD + kk] = dS[kk * KD + vv];
  free(S); free(ck); free(blk); free(dS); free(Sp);
}

static void* bwd_worker(void* arg) {
  const bwd_job_t* J = (const bwd_job_t*)arg;
  const int32_t G = J->H / J->HK;
  for (int32_t hk = J->tid; hk < J->HK; hk += J->nthreads)
    for (int32_t n = 0; n < J->N; ++n)
      for (int32_t h = hk * G; h < (hk + 1) * G; ++h) bwd_unit(J, n, h);
  return NULL;
}

/*
 * Public: backward over packed tokens (layouts as kda_oracle_fwd; dout
 * [T_total][H][V]; dfin, init, dinit [N][H][V][K] or NULL).  Outputs dq, dk
 * [T_total][HK][K], dv, dg [T_total][H][K], dbeta [T_total][H], dA_log [H],
 * ddt_bias [H][K] must be zeroed by the caller (dq, dk, dA_log and ddt_bias
 * accumulate).  Returns the number of threads used.
 */
int kda_oracle_bwd(int64_t T_total, int32_t H, int32_t HK, int32_t N, const int64_t* cu,
                   const double* q, const double* k, const double* v, const double* g,
                   const double* beta_raw, const double* A_log, const double* dt_bias,
                   double lower_bound, double scale, const double* init, const double* dout,
                   const double* dfin, double* dq, double* dk, double* dv, double* dg,
                   double* dbeta, double* dA_log, double* ddt_bias, double* dinit,
                   int32_t nthreads) {
  bwd_job_t J;
  memset(&J, 0, sizeof(J));
  J.T_total = T_total; J.H = H; J.HK = (HK > 0 && H % HK == 0) ? HK : H; J.N = N; J.cu = cu;
  J.q = q; J.k = k; J.v = v; J.g = g; J.beta_raw = beta_raw; J.A_log = A_log;
  J.dt_bias = dt_bias; J.lower_bound = lower_bound; J.scale = scale; J.init = init;
  J.dout = dout; J.dfin = dfin; J.dq = dq; J.dk = dk; J.dv = dv; J.dg = dg; J.dbeta = dbeta;
  J.dA_log = dA_log; J.ddt_bias = ddt_bias; J.dinit = dinit;
  int nt = nthreads < 1 ? 1 : nthreads;
  if (nt > J.HK) nt = J.HK;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nt);
  bwd_job_t* jobs = (bwd_job_t*)malloc(sizeof(bwd_job_t) * nt);
  for (int i = 0; i < nt; ++i) {
    jobs[i] = J;
    jobs[i].nthreads = nt;
    jobs[i].tid = i;
  }
  for (int i = 1; i < nt; ++i) pthread_create(&th[i], NULL, bwd_worker, &jobs[i]);
  bwd_worker(&jobs[0]);
  for (int i = 1; i < nt; ++i) pthread_join(th[i], NULL);
  free(th);
  free(jobs);
  return nt;
}

/*
 * Plain fp64 CPU oracle for the selective state-space scan.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark may load or call this library; the product path never does.
 * It shares no code, header or constant with the CUDA implementation.
 *
 * Everything is computed in double precision, one channel at a time, in the order
 * the pages write the method.  Channels are independent, so they are spread over
 * POSIX threads; that changes no arithmetic.
 *
 * Sources (page title, section):
 *  [S1] "Mamba и State Space Models", sections "Mamba: Selective State Space Model"
 *       and "Selective Scan (core algorithm)": the selective recurrence
 *       h_t = exp(Δ_t A) h_{t-1} + Δ_t B_t x_t, y_t = C_t h_t, with Δ = softplus(dt_proj(.)),
 *       and the block's output gate y * SiLU(res) (section "Реализация MambaBlock").
 *  [S2] "Модуль 8. Альтернативы Transformer: SSM, Mamba и гибриды":
 *       §4 (discrete SSM, exact ZOH input term A^{-1}(e^{ΔA}-I)B and its a→0 limit Δ),
 *       §6 (Δ_t = softplus(.), softplus(u) = log(1+e^u); the depthwise causal conv and
 *       its cache), §7 (affine pairs (a,b), composition (a2,b2)∘(a1,b1) = (a2 a1, a2 b1 + b2)),
 *       §14 (conv_state and ssm_state caches of a Mamba-1 layer).
 *  [S3] "State Space Models: Mamba и альтернатива Transformer", section
 *       "Mamba: Selective State Space" (D skip y = C·h + D·x, SiLU after the conv,
 *       y * SiLU(res)) and "SSM Scan Algorithm" (recurrent form, closed-form prefix).
 *
 * Readings where the pages are silent or disagree (each also listed in the design notes):
 *  - input term is Δ·B·x (the Mamba parameterisation, [S1], [S2] §4/§14); the exact ZOH
 *    term is a separate option (discretization = 1);
 *  - Δ = softplus(Δ_raw + bias) with a per-channel bias added before softplus;
 *  - the D skip is included and the gate multiplies (C·h + D·x);
 *  - the conv has no bias, kernel width K, and conv_state holds the last K-1 raw inputs,
 *    oldest first; a SiLU follows the conv ([S3]).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>
#include <unistd.h>

#define ORACLE_API __attribute__((visibility("default")))

/* softplus(v) = log(1 + e^v) ([S2] §6), written in the overflow-free form. */
static double softplus(double v) {
  return v > 0.0 ? v + log1p(exp(-v)) : log1p(exp(v));
}

/* SiLU(z) = z * sigmoid(z) = z / (1 + e^{-z}). */
static double silu(double z) { return z / (1.0 + exp(-z)); }

/* The affine step h -> a h + b, composed "later after earlier" ([S2] §7). */
ORACLE_API void oracle_compose_affine(double a2, double b2, double a1, double b1,
                                      double* a_out, double* b_out) {
  *a_out = a2 * a1;
  *b_out = a2 * b1 + b2;
}

/* Discrete coefficients for one state coordinate and one step:
 *   abar = exp(Δ a)
 *   bbar = Δ b                         (discretization 0, the Mamba input term)
 *   bbar = (exp(Δ a) - 1) / a * b      (discretization 1, exact ZOH, [S2] §4),
 *          with the a -> 0 limit Δ b. */
static void discretize(double delta, double a, double b, int discretization,
                       double* abar, double* bbar) {
  *abar = exp(delta * a);
  if (discretization == 1 && a != 0.0)
    *bbar = expm1(delta * a) / a * b;
  else
    *bbar = delta * b;
}

/* ------------------------------------------------------------------------------------
 * Channel-list problem description.  A "channel" is one (batch b, inner channel d) pair.
 * Per-channel arrays are indexed by the channel's position c in the list; B and C stay
 * in their (batch, dstate, L) layout and are read through bidx[c].
 * ---------------------------------------------------------------------------------- */
typedef struct {
  const double* u;          /* (n, L) */
  const double* delta;      /* (n, L)  Δ_raw */
  const double* A;          /* (n, N) */
  const double* B;          /* (batch, N, L) */
  const double* C;          /* (batch, N, L) */
  const double* D;          /* (n) or NULL */
  const double* z;          /* (n, L) or NULL: no gate */
  const double* bias;       /* (n) or NULL */
  const double* h0;         /* (n, N) or NULL: zero initial state */
  const int64_t* bidx;      /* (n) batch index of each channel */
  double* y;                /* (n, L) */
  double* hL;               /* (n, N) or NULL */
  int64_t n, L;
  int N;
  int softplus_flag;
  int discretization;
  int64_t chunk;            /* chunked variant: chunk length (>0) */
} scan_problem;

static double delta_at(const scan_problem* p, int64_t c, int64_t t) {
  double v = p->delta[c * p->L + t] + (p->bias ? p->bias[c] : 0.0);
  return p->softplus_flag ? softplus(v) : v;
}

/* Readout for step t: y = C_t·h + D x_t, then the gate y * SiLU(z_t). */
static double readout(const scan_problem* p, int64_t c, int64_t t, const double* h) {
  const int N = p->N;
  const double* Cb = p->C + p->bidx[c] * (int64_t)N * p->L;
  double y = 0.0;
  for (int n = 0; n < N; ++n) y += Cb[(int64_t)n * p->L + t] * h[n];
  double x = p->u[c * p->L + t];
  if (p->D) y += p->D[c] * x;
  if (p->z) y *= silu(p->z[c * p->L + t]);
  return y;
}

/* One recurrence step h <- abar ⊙ h + bbar x for step t ([S1] "Selective Scan"). */
static void step(const scan_problem* p, int64_t c, int64_t t, double* h) {
  const int N = p->N;
  const double* Bb = p->B + p->bidx[c] * (int64_t)N * p->L;
  double dlt = delta_at(p, c, t);
  double x = p->u[c * p->L + t];
  for (int n = 0; n < N; ++n) {
    double abar, bbar;
    discretize(dlt, p->A[c * N + n], Bb[(int64_t)n * p->L + t], p->discretization, &abar, &bbar);
    h[n] = abar * h[n] + bbar * x;
  }
}

/* Sequential scan of one channel: the plain recurrence, update then read ([S1], [S3]). */
static void scan_channel(const scan_problem* p, int64_t c) {
  double h[64];
  const int N = p->N;
  for (int n = 0; n < N; ++n) h[n] = p->h0 ? p->h0[c * N + n] : 0.0;
  for (int64_t t = 0; t < p->L; ++t) {
    step(p, c, t, h);
    p->y[c * p->L + t] = readout(p, c, t, h);
  }
  if (p->hL)
    for (int n = 0; n < N; ++n) p->hL[c * N + n] = h[n];
}

/* Chunked scan of one channel, the two-level form of [S2] §7:
 *  1. for every chunk, its aggregate affine pair per state coordinate: (Π abar, h_end from 0);
 *  2. the carry into chunk k is the composition of the aggregates of chunks < k applied
 *     to the initial state;
 *  3. every chunk is re-run from its carried-in state to produce y. */
static void chunked_scan_channel(const scan_problem* p, int64_t c) {
  const int N = p->N;
  const int64_t T = p->chunk, L = p->L;
  const int64_t nchunks = (L + T - 1) / T;
  double carry[64], agg_a[64], agg_b[64], h[64];
  for (int n = 0; n < N; ++n) carry[n] = p->h0 ? p->h0[c * N + n] : 0.0;
  const double* Bb = p->B + p->bidx[c] * (int64_t)N * L;
  for (int64_t k = 0; k < nchunks; ++k) {
    int64_t t0 = k * T, t1 = t0 + T < L ? t0 + T : L;
    /* 1. aggregate of chunk k, built step by step with the composition operator */
    for (int n = 0; n < N; ++n) { agg_a[n] = 1.0; agg_b[n] = 0.0; }
    for (int64_t t = t0; t < t1; ++t) {
      double dlt = delta_at(p, c, t);
      double x = p->u[c * L + t];
      for (int n = 0; n < N; ++n) {
        double abar, bbar;
        discretize(dlt, p->A[c * N + n], Bb[(int64_t)n * L + t], p->discretization, &abar, &bbar);
        oracle_compose_affine(abar, bbar * x, agg_a[n], agg_b[n], &agg_a[n], &agg_b[n]);
      }
    }
    /* 3. re-run chunk k from the carried-in state */
    for (int n = 0; n < N; ++n) h[n] = carry[n];
    for (int64_t t = t0; t < t1; ++t) {
      step(p, c, t, h);
      p->y[c * L + t] = readout(p, c, t, h);
    }
    /* 2. carry into chunk k+1 = aggregate_k applied to carry_k */
    for (int n = 0; n < N; ++n) {
      double a_unused;
      oracle_compose_affine(agg_a[n], agg_b[n], 1.0, carry[n], &a_unused, &carry[n]);
    }
  }
  if (p->hL)
    for (int n = 0; n < N; ++n) p->hL[c * N + n] = carry[n];
}

/* ------------------------------------------------------------------------------------
 * A minimal thread pool over channels.
 * ---------------------------------------------------------------------------------- */
typedef struct {
  void (*fn)(const void*, int64_t);
  const void* problem;
  int64_t n;
  int64_t next;
  pthread_mutex_t mu;
} pool;

static void* pool_worker(void* arg) {
  pool* q = (pool*)arg;
  for (;;) {
    pthread_mutex_lock(&q->mu);
    int64_t c = q->next++;
    pthread_mutex_unlock(&q->mu);
    if (c >= q->n) break;
    q->fn(q->problem, c);
  }
  return NULL;
}

static void run_channels(void (*fn)(const void*, int64_t), const void* problem, int64_t n,
                         int threads) {
  if (threads <= 0) threads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  if ((int64_t)threads > n) threads = (int)(n > 0 ? n : 1);
  pool q;
  q.fn = fn; q.problem = problem; q.n = n; q.next = 0;
  pthread_mutex_init(&q.mu, NULL);
  if (threads == 1) {
    pool_worker(&q);
  } else {
    pthread_t tid[256];
    for (int i = 0; i < threads; ++i) pthread_create(&tid[i], NULL, pool_worker, &q);
    for (int i = 0; i < threads; ++i) pthread_join(tid[i], NULL);
  }
  pthread_mutex_destroy(&q.mu);
}

static void scan_fn(const void* p, int64_t c) { scan_channel((const scan_problem*)p, c); }
static void chunked_fn(const void* p, int64_t c) { chunked_scan_channel((const scan_problem*)p, c); }

/* Returns 0 on success, -1 on a bad argument. */
static int fill_problem(scan_problem* p, const double* u, const double* delta, const double* A,
                        const double* B, const double* C, const double* D, const double* z,
                        const double* bias, int softplus_flag, int discretization,
                        const double* h0, const int64_t* bidx, double* y, double* hL,
                        int64_t n, int N, int64_t L) {
  if (!u || !delta || !A || !B || !C || !bidx || !y) return -1;
  if (n < 0 || L < 0 || N < 1 || N > 64) return -1;
  if (discretization != 0 && discretization != 1) return -1;
  p->u = u; p->delta = delta; p->A = A; p->B = B; p->C = C; p->D = D; p->z = z;
  p->bias = bias; p->h0 = h0; p->bidx = bidx; p->y = y; p->hL = hL;
  p->n = n; p->L = L; p->N = N; p->softplus_flag = softplus_flag;
  p->discretization = discretization; p->chunk = 0;
  return 0;
}

ORACLE_API int oracle_selective_scan(const double* u, const double* delta, const double* A,
                                     const double* B, const double* C, const double* D,
                                     const double* z, const double* bias, int softplus_flag,
                                     int discretization, const double* h0, const int64_t* bidx,
                                     double* y, double* hL, int64_t n, int N, int64_t L,
                                     int threads) {
  scan_problem p;
  if (fill_problem(&p, u, delta, A, B, C, D, z, bias, softplus_flag, discretization, h0, bidx,
                   y, hL, n, N, L))
    return -1;
  run_channels(scan_fn, &p, n, threads);
  return 0;
}

ORACLE_API int oracle_chunked_scan(const double* u, const double* delta, const double* A,
                                   const double* B, const double* C, const double* D,
                                   const double* z, const double* bias, int softplus_flag,
                                   int discretization, const double* h0, const int64_t* bidx,
                                   double* y, double* hL, int64_t n, int N, int64_t L,
                                   int64_t chunk, int threads) {
  scan_problem p;
  if (fill_problem(&p, u, delta, A, B, C, D, z, bias, softplus_flag, discretization, h0, bidx,
                   y, hL, n, N, L))
    return -1;
  if (chunk < 1) return -1;
  p.chunk = chunk;
  run_channels(chunked_fn, &p, n, threads);
  return 0;
}

/* ------------------------------------------------------------------------------------
 * Causal depthwise conv1d of width K followed (optionally) by SiLU, per channel:
 *   out[t] = SiLU( Σ_{k=0}^{K-1} w[k] · xpad[t + k] ),  xpad = [state (K-1 values), x_0 .. x_{L-1}]
 * i.e. a cross-correlation with K-1 leading pad values, keeping the first L outputs
 * ("Mamba и State Space Models", "Реализация MambaBlock"; "State Space Models: Mamba и
 * альтернатива Transformer", "Mamba: Selective State Space").  With a NULL state the pad
 * is zero.  state_out receives the last K-1 entries of xpad, oldest first.
 * ---------------------------------------------------------------------------------- */
ORACLE_API int oracle_causal_conv1d(const double* x, const double* w, const double* state_in,
                                    double* out, double* state_out, int64_t n, int64_t L,
                                    int K, int apply_silu) {
  if (!x || !w || !out || n < 0 || L < 0 || K < 1 || K > 64) return -1;
  double* xpad = (double*)malloc(sizeof(double) * (size_t)(L + K - 1));
  if (!xpad) return -1;
  for (int64_t c = 0; c < n; ++c) {
    for (int k = 0; k < K - 1; ++k) xpad[k] = state_in ? state_in[c * (K - 1) + k] : 0.0;
    for (int64_t t = 0; t < L; ++t) xpad[K - 1 + t] = x[c * L + t];
    for (int64_t t = 0; t < L; ++t) {
      double s = 0.0;
      for (int k = 0; k < K; ++k) s += w[c * K + k] * xpad[t + k];
      out[c * L + t] = apply_silu ? silu(s) : s;
    }
    if (state_out)
      for (int k = 0; k < K - 1; ++k) state_out[c * (K - 1) + k] = xpad[L + k];
  }
  free(xpad);
  return 0;
}

/* ------------------------------------------------------------------------------------
 * One decode step of a Mamba-1 layer with its two caches ([S2] §6 and §14):
 *   window  = [conv_state[0..K-2], x_t]
 *   u       = SiLU(Σ_k w[k] window[k]);  conv_state <- window[1..K-1]
 *   Δ       = softplus(Δ_raw + bias)
 *   h       <- exp(Δ A) ⊙ h + Δ B_t u
 *   y_t     = (C_t·h + D u) · SiLU(z_t)
 * Per-channel arrays are indexed by channel c; B_t and C_t are (batch, N) via bidx.
 * ---------------------------------------------------------------------------------- */
ORACLE_API int oracle_state_update(const double* x_t, const double* delta_t, const double* A,
                                   const double* B_t, const double* C_t, const double* D,
                                   const double* z_t, const double* bias, int softplus_flag,
                                   double* state, double* conv_state, const double* conv_w,
                                   double* y_t, const int64_t* bidx, int64_t n, int N, int K) {
  if (!x_t || !delta_t || !A || !B_t || !C_t || !state || !conv_state || !conv_w || !y_t ||
      !bidx || n < 0 || N < 1 || N > 64 || K < 1 || K > 64)
    return -1;
  for (int64_t c = 0; c < n; ++c) {
    double window[64];
    for (int k = 0; k < K - 1; ++k) window[k] = conv_state[c * (K - 1) + k];
    window[K - 1] = x_t[c];
    double s = 0.0;
    for (int k = 0; k < K; ++k) s += conv_w[c * K + k] * window[k];
    double u = silu(s);
    for (int k = 0; k < K - 1; ++k) conv_state[c * (K - 1) + k] = window[k + 1];

    double v = delta_t[c] + (bias ? bias[c] : 0.0);
    double dlt = softplus_flag ? softplus(v) : v;
    const double* Bb = B_t + bidx[c] * N;
    const double* Cb = C_t + bidx[c] * N;
    double y = 0.0;
    for (int nn = 0; nn < N; ++nn) {
      double* h = &state[c * N + nn];
      *h = exp(dlt * A[c * N + nn]) * *h + dlt * Bb[nn] * u;
      y += Cb[nn] * *h;
    }
    if (D) y += D[c] * u;
    if (z_t) y *= silu(z_t[c]);
    y_t[c] = y;
  }
  return 0;
}

/* ------------------------------------------------------------------------------------
 * Backward of the selective scan (reverse-mode differentiation of the recurrence above).
 * For one channel, with v_t = Δ_raw_t + bias, Δ_t = softplus(v_t) (or v_t), Ā = exp(Δ A),
 * b_t = Δ_t B_t x_t, h_t = Ā_t ⊙ h_{t-1} + b_t, s_t = C_t·h_t + D x_t, y_t = s_t SiLU(z_t), and an
 * upstream gradient dy:
 *   ds_t   = dy_t SiLU(z_t);            dz_t = dy_t s_t SiLU'(z_t),  SiLU'(z) = σ(z)(1 + z(1 - σ(z)))
 *   dh_t   = ds_t C_t + Ā_{t+1} ⊙ dh_{t+1}   (from the last step backwards; nothing after L-1)
 *   dC_t  += ds_t h_t;   dB_t += dh_t Δ_t x_t
 *   dΔ_t   = Σ_n dh_{t,n} (h_{t-1,n} Ā_{t,n} A_n + B_{t,n} x_t)
 *   dA_n  += Σ_t dh_{t,n} h_{t-1,n} Ā_{t,n} Δ_t
 *   dx_t   = ds_t D + Σ_n dh_{t,n} Δ_t B_{t,n};   dD += ds_t x_t
 *   dv_t   = dΔ_t σ(v_t) (softplus' = sigmoid), or dΔ_t without softplus;  dΔ_raw_t = dv_t;  dbias += dv_t
 * The Δ·B input term is differentiated (the ZOH variant is not).  Per channel c the results are
 * dx, dΔ_raw, dz (n, L); dA (n, N); dD, dbias (n); and this channel's contributions to dB and dC,
 * (n, N, L) -- the caller sums those over the channels of each batch row.
 * ---------------------------------------------------------------------------------- */
typedef struct {
  const scan_problem* fwd;
  const double* dy;   /* (n, L) */
  double* du;         /* (n, L) */
  double* ddelta;     /* (n, L) */
  double* dz;         /* (n, L) or NULL when there is no gate */
  double* dA;         /* (n, N) */
  double* dD;         /* (n) */
  double* dbias;      /* (n) */
  double* dB;         /* (n, N, L) per-channel contribution */
  double* dC;         /* (n, N, L) per-channel contribution */
} bwd_problem;

static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

static void backward_channel(const bwd_problem* q, int64_t c) {
  const scan_problem* p = q->fwd;
  const int N = p->N;
  const int64_t L = p->L;
  const double* Bb = p->B + p->bidx[c] * (int64_t)N * L;
  const double* Cb = p->C + p->bidx[c] * (int64_t)N * L;
  /* forward, keeping every state (h[t] = state after step t; hs[0] = initial) */
  double* hs = (double*)malloc(sizeof(double) * (size_t)(L + 1) * N);
  double* sv = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
  for (int n = 0; n < N; ++n) hs[n] = p->h0 ? p->h0[c * N + n] : 0.0;
  for (int64_t t = 0; t < L; ++t) {
    double dlt = delta_at(p, c, t);
    double x = p->u[c * L + t];
    double s = 0.0;
    for (int n = 0; n < N; ++n) {
      double abar = exp(dlt * p->A[c * N + n]);
      double h = abar * hs[t * N + n] + dlt * Bb[(int64_t)n * L + t] * x;
      hs[(t + 1) * N + n] = h;
      s += Cb[(int64_t)n * L + t] * h;
    }
    if (p->D) s += p->D[c] * x;
    sv[t] = s;
  }
  /* backward */
  double dh[64], dAacc[64];
  for (int n = 0; n < N; ++n) { dh[n] = 0.0; dAacc[n] = 0.0; }
  double dD = 0.0, dbias = 0.0;
  for (int64_t t = L - 1; t >= 0; --t) {
    double dlt = delta_at(p, c, t);
    double x = p->u[c * L + t];
    double dyt = q->dy[c * L + t];
    double ds = dyt;
    if (p->z) {
      double zz = p->z[c * L + t];
      double sg = sigmoid(zz);
      ds = dyt * silu(zz);
      q->dz[c * L + t] = dyt * sv[t] * sg * (1.0 + zz * (1.0 - sg));
    }
    double dx = p->D ? ds * p->D[c] : 0.0;
    dD += ds * x;
    double ddl = 0.0;
    for (int n = 0; n < N; ++n) {
      double a = p->A[c * N + n];
      double abar = exp(dlt * a);
      double bn = Bb[(int64_t)n * L + t];
      double cn = Cb[(int64_t)n * L + t];
      /* dh_t = ds_t C_t + (Ā_{t+1} dh_{t+1}); the second term was folded into dh at step t+1 */
      dh[n] += ds * cn;
      q->dC[(c * N + n) * L + t] = ds * hs[(t + 1) * N + n];
      q->dB[(c * N + n) * L + t] = dh[n] * dlt * x;
      double hprev = hs[t * N + n];
      ddl += dh[n] * (hprev * abar * a + bn * x);
      dAacc[n] += dh[n] * hprev * abar * dlt;
      dx += dh[n] * dlt * bn;
      dh[n] *= abar;   /* carried to step t-1: Ā_t ⊙ dh_t */
    }
    double v = p->delta[c * L + t] + (p->bias ? p->bias[c] : 0.0);
    double dv = p->softplus_flag ? ddl * sigmoid(v) : ddl;
    q->du[c * L + t] = dx;
    q->ddelta[c * L + t] = dv;
    dbias += dv;
  }
  for (int n = 0; n < N; ++n) q->dA[c * N + n] = dAacc[n];
  q->dD[c] = dD;
  q->dbias[c] = dbias;
  free(hs);
  free(sv);
}

static void backward_fn(const void* q, int64_t c) { backward_channel((const bwd_problem*)q, c); }

ORACLE_API int oracle_scan_backward(const double* u, const double* delta, const double* A, const double* B,
                                    const double* C, const double* D, const double* z, const double* bias,
                                    int softplus_flag, const double* h0, const int64_t* bidx, const double* dy,
                                    double* du, double* ddelta, double* dz, double* dA, double* dD,
                                    double* dbias, double* dB, double* dC, int64_t n, int N, int64_t L,
                                    int threads) {
  scan_problem p;
  /* the forward outputs are not written here; du stands in for the y pointer the check wants */
  if (fill_problem(&p, u, delta, A, B, C, D, z, bias, softplus_flag, 0, h0, bidx, du, NULL, n, N, L))
    return -1;
  if (!dy || !du || !ddelta || !dA || !dD || !dbias || !dB || !dC || (z && !dz)) return -1;
  bwd_problem q;
  q.fwd = &p; q.dy = dy; q.du = du; q.ddelta = ddelta; q.dz = dz; q.dA = dA; q.dD = dD; q.dbias = dbias;
  q.dB = dB; q.dC = dC;
  run_channels(backward_fn, &q, n, threads);
  return 0;
}

/* ------------------------------------------------------------------------------------------
 * Mamba-2 state space duality (SSD): scalar decay per head, matrix state per head.
 *  [S1] "Mamba и State Space Models", "Mamba-2: State Space Duality (SSD)": A is a scalar
 *       (A = -exp(A_log)), d_state 128, y = SS(A)·(B ⊗ X)·C.
 *  [S2] "Модуль 8", §7: with transition a_t·I and a zero initial state the weight of input j in
 *       output i ≥ j is M_ij = C_i^T B_j Π_{r=j+1..i} a_r; inside a chunk the block is computed as
 *       a masked matrix product, between chunks only the state is passed; §14: the state has the
 *       shape [batch, nheads, headdim, d_state] and the input term is Δ·B·x.
 * Per batch b and head h, with P = headdim, N = dstate and the head's group g:
 *   Δ_t = softplus(dt[b,t,h] + dt_bias[h]),  a_t = exp(Δ_t A[h])
 *   H_t[p][n] = a_t H_{t-1}[p][n] + Δ_t x[b,t,h,p] B[b,t,g,n]
 *   y[b,t,h,p] = Σ_n C[b,t,g,n] H_t[p][n] + D[h] x[b,t,h,p]
 * Layouts: x, y (batch, L, nheads, headdim); dt (batch, L, nheads); B, C (batch, L, ngroups, dstate);
 * A, D, dt_bias (nheads); h0, hT (batch, nheads, headdim, dstate).  Heads split evenly over groups.
 * ------------------------------------------------------------------------------------------ */
typedef struct {
  const double *x, *dt, *A, *B, *C, *D, *dt_bias, *h0;
  double *y, *hT;
  int softplus_flag;
  int64_t batch, L, chunk;
  int nheads, headdim, dstate, ngroups;
} ssd_problem;

static double ssd_delta(const ssd_problem* p, int64_t b, int64_t t, int h) {
  double v = p->dt[(b * p->L + t) * p->nheads + h];
  if (p->dt_bias) v += p->dt_bias[h];
  return p->softplus_flag ? softplus(v) : v;
}

static const double* ssd_x(const ssd_problem* p, int64_t b, int64_t t, int h) {
  return p->x + ((b * p->L + t) * p->nheads + h) * p->headdim;
}

static const double* ssd_bc(const ssd_problem* p, const double* base, int64_t b, int64_t t, int h) {
  const int g = h / (p->nheads / p->ngroups);
  return base + ((b * p->L + t) * p->ngroups + g) * p->dstate;
}

static void ssd_init_state(const ssd_problem* p, int64_t b, int h, double* H) {
  const int64_t PN = (int64_t)p->headdim * p->dstate;
  for (int64_t i = 0; i < PN; ++i) H[i] = p->h0 ? p->h0[(b * p->nheads + h) * PN + i] : 0.0;
}

static void ssd_store_state(const ssd_problem* p, int64_t b, int h, const double* H) {
  const int64_t PN = (int64_t)p->headdim * p->dstate;
  if (p->hT)
    for (int64_t i = 0; i < PN; ++i) p->hT[(b * p->nheads + h) * PN + i] = H[i];
}

/* the recurrence, one step at a time ([S2] §7, form 1) */
static void ssd_sequential_pair(const ssd_problem* p, int64_t pair) {
  const int64_t b = pair / p->nheads;
  const int h = (int)(pair % p->nheads);
  const int P = p->headdim, N = p->dstate;
  double* H = (double*)malloc(sizeof(double) * (size_t)P * N);
  ssd_init_state(p, b, h, H);
  for (int64_t t = 0; t < p->L; ++t) {
    const double dl = ssd_delta(p, b, t, h);
    const double a = exp(dl * p->A[h]);
    const double* x = ssd_x(p, b, t, h);
    const double* Bt = ssd_bc(p, p->B, b, t, h);
    const double* Ct = ssd_bc(p, p->C, b, t, h);
    for (int i = 0; i < P; ++i)
      for (int n = 0; n < N; ++n) H[i * N + n] = a * H[i * N + n] + dl * x[i] * Bt[n];
    double* y = p->y + ((b * p->L + t) * p->nheads + h) * P;
    for (int i = 0; i < P; ++i) {
      double s = 0.0;
      for (int n = 0; n < N; ++n) s += Ct[n] * H[i * N + n];
      y[i] = s + (p->D ? p->D[h] * x[i] : 0.0);
    }
  }
  ssd_store_state(p, b, h, H);
  free(H);
}

/* the chunked block form ([S2] §7, form 3): inside a chunk, y_i = Σ_{j≤i} (C_i·B_j) Π_{r=j+1..i} a_r Δ_j x_j
 * plus the state entering the chunk read through (Π_{r=start..i} a_r) C_i; between chunks only the
 * state is passed: H_end = (Π_chunk a) H_start + Σ_j (Π_{r=j+1..end} a_r) Δ_j x_j B_j^T. */
static void ssd_chunked_pair(const ssd_problem* p, int64_t pair) {
  const int64_t b = pair / p->nheads;
  const int h = (int)(pair % p->nheads);
  const int P = p->headdim, N = p->dstate;
  const int64_t Q = p->chunk;
  double* H = (double*)malloc(sizeof(double) * (size_t)P * N);
  double* Hn = (double*)malloc(sizeof(double) * (size_t)P * N);
  double* a = (double*)malloc(sizeof(double) * (size_t)Q);
  double* dl = (double*)malloc(sizeof(double) * (size_t)Q);
  ssd_init_state(p, b, h, H);
  for (int64_t s0 = 0; s0 < p->L; s0 += Q) {
    const int64_t q = p->L - s0 < Q ? p->L - s0 : Q;
    for (int64_t i = 0; i < q; ++i) {
      dl[i] = ssd_delta(p, b, s0 + i, h);
      a[i] = exp(dl[i] * p->A[h]);
    }
    for (int64_t i = 0; i < q; ++i) {
      const double* Ci = ssd_bc(p, p->C, b, s0 + i, h);
      double* y = p->y + ((b * p->L + s0 + i) * p->nheads + h) * P;
      for (int k = 0; k < P; ++k) y[k] = 0.0;
      double decay = 1.0;                       /* Π_{r=j+1..i} a_r */
      for (int64_t j = i; j >= 0; --j) {
        if (j < i) decay *= a[j + 1];
        const double* Bj = ssd_bc(p, p->B, b, s0 + j, h);
        double cb = 0.0;
        for (int n = 0; n < N; ++n) cb += Ci[n] * Bj[n];
        const double m = cb * decay * dl[j];
        const double* xj = ssd_x(p, b, s0 + j, h);
        for (int k = 0; k < P; ++k) y[k] += m * xj[k];
      }
      double into = 1.0;                        /* Π_{r=start..i} a_r */
      for (int64_t r = 0; r <= i; ++r) into *= a[r];
      const double* xi = ssd_x(p, b, s0 + i, h);
      for (int k = 0; k < P; ++k) {
        double s = 0.0;
        for (int n = 0; n < N; ++n) s += Ci[n] * H[k * N + n];
        y[k] += into * s + (p->D ? p->D[h] * xi[k] : 0.0);
      }
    }
    double total = 1.0;
    for (int64_t r = 0; r < q; ++r) total *= a[r];
    for (int64_t i = 0; i < (int64_t)P * N; ++i) Hn[i] = total * H[i];
    for (int64_t j = 0; j < q; ++j) {
      double decay = 1.0;                       /* Π_{r=j+1..end} a_r */
      for (int64_t r = j + 1; r < q; ++r) decay *= a[r];
      const double* Bj = ssd_bc(p, p->B, b, s0 + j, h);
      const double* xj = ssd_x(p, b, s0 + j, h);
      for (int k = 0; k < P; ++k)
        for (int n = 0; n < N; ++n) Hn[k * N + n] += decay * dl[j] * xj[k] * Bj[n];
    }
    memcpy(H, Hn, sizeof(double) * (size_t)P * N);
  }
  ssd_store_state(p, b, h, H);
  free(H);
  free(Hn);
  free(a);
  free(dl);
}

static void ssd_fn(const void* q, int64_t pair) {
  const ssd_problem* p = (const ssd_problem*)q;
  if (p->chunk > 0) ssd_chunked_pair(p, pair);
  else ssd_sequential_pair(p, pair);
}

/* chunk = 0: the recurrence; chunk > 0: the chunked block form with that chunk length */
ORACLE_API int oracle_ssd_scan(const double* x, const double* dt, const double* A, const double* B,
                               const double* C, const double* D, const double* dt_bias, int softplus_flag,
                               const double* h0, double* y, double* hT, int64_t batch, int64_t L, int nheads,
                               int headdim, int dstate, int ngroups, int64_t chunk, int threads) {
  if (!x || !dt || !A || !B || !C || !y || batch < 1 || L < 0 || nheads < 1 || headdim < 1 || dstate < 1 ||
      ngroups < 1 || nheads % ngroups != 0 || chunk < 0)
    return -1;
  ssd_problem p;
  p.x = x; p.dt = dt; p.A = A; p.B = B; p.C = C; p.D = D; p.dt_bias = dt_bias; p.h0 = h0;
  p.y = y; p.hT = hT; p.softplus_flag = softplus_flag;
  p.batch = batch; p.L = L; p.chunk = chunk;
  p.nheads = nheads; p.headdim = headdim; p.dstate = dstate; p.ngroups = ngroups;
  run_channels(ssd_fn, &p, batch * nheads, threads);
  return 0;
}

/*
 * CPU oracle for the state-passing mixer forward and the decode update.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check
 * and the benchmark's CPU-baseline leg may load this library.  The product
 * path never calls it and shares no code with it.
 *
 * Everything is float64, computed literally in the order the method states,
 * from the exact values of the (bf16 or fp32) inputs, with no intermediate
 * rounding and no blocking, chunking or reordering:
 *
 *   orc_conv_state_fwd  causal depthwise conv with an explicit (K-1)-sample
 *                       state, in the extended-sequence form of
 *                       "Chapter 7: state, chunking and incremental inference"
 *                       (section "define the state with the extended
 *                       sequence"):  u = [S_0..S_{K-2}, x_0..x_{L-1}],
 *                       z_t = beta + sum_k w_k u_{t+k},  F = u[L : L+K-1],
 *                       output SiLU(z) = z / (1 + exp(-z)).
 *   orc_conv_state_bwd  its gradient with state, as derived in the same
 *                       chapter (section "unified derivation of the backward
 *                       pass with state"): with delta_t = dL/dz_t and
 *                       q = dL/dF, dL/du_j = sum_{t,k: t+k=j} delta_t w_k
 *                       + [L <= j < L+K-1] q_{j-L}, dS = du[0 : K-1],
 *                       dx = du[K-1 : K-1+L], dw_k = sum_t delta_t u_{t+k},
 *                       dbeta = sum_t delta_t (summed over the batch too).
 *   orc_ssm_scan        the linear recurrence of "Understanding and Improving
 *                       Length Generalization in Recurrent Models" section 2
 *                       Eq. (1), h_t = A_t h_{t-1} + B_t x_t, y_t = C_t^T h_t,
 *                       specialised to one scalar decay per head,
 *                       A_t = exp(dt_t * A_h), run from the initial state
 *                       h_{-1} (Eq. (4)'s non-zero initial state), one token
 *                       at a time.
 *   orc_ssm_scan_bwd    the gradient of orc_ssm_scan with state, for
 *                       state-passing and truncated-backpropagation training
 *                       ("Understanding and Improving Length Generalization
 *                       in Recurrent Models" sections 4.4-4.5; the causal-conv
 *                       chapter's "chunked training and truncated backward"
 *                       section on passing the state gradient across
 *                       chunks): with g_t = dL/dh_t (every later use
 *                       included) and a_t = exp(dt_t A_h), token by token
 *                       in reverse, g_t = a_{t+1} g_{t+1} + dy_t C_t^T (the
 *                       gradient of the final state dhT entering at t = L-1),
 *                       dC_t = h_t^T dy_t, dx_t = g_t B_t, dB_t = g_t^T x_t,
 *                       dl_t = a_t <g_t, h_{t-1}> for l_t = dt_t A_h, so
 *                       ddt_t = dl_t A_h and dA_h = sum dl_t dt_t, and
 *                       dh0 = a_0 g_0; dB and dC sum over the heads of a
 *                       group, dA over the batch.
 *   orc_mamba2_scan     the recurrence of the full Mamba-2 mixer wiring
 *                       (the Mamba-2 layers of "Understanding and Improving
 *                       Length Generalization in Recurrent Models" sections 1
 *                       and 4.4, with the causal-conv chapter's xBC conv): on
 *                       the conv + SiLU output of all D + 2 G N channels of
 *                       xBC (channels [0, D) are x, then B and C),
 *                       dt_t = softplus(dt_raw_t + dt_bias_h),
 *                       a_t = exp(dt_t A_h), h_t = a_t h_{t-1} + dt_t x_t B_t^T,
 *                       y_t = (h_t C_t + D_h x_t) SiLU(z_t), one token at a
 *                       time from the initial state.
 *   orc_mixer_update    the single- and multi-token update of the same
 *                       chapter (sections "single-token update", "the
 *                       physical cache can be longer", "circular mode",
 *                       "continuous batching"): history j of a request at
 *                       length p is read from slot (p - j) mod S_len, token i
 *                       is written to slot (p + i) mod S_len after every
 *                       read, the stored value is the input x (not the
 *                       output), rows are addressed through
 *                       conv_state_indices, cache_seqlens is not advanced;
 *                       without cache_seqlens, the non-circular mode of
 *                       "the physical cache can be longer": a row keeps its
 *                       newest S_len >= K-1 inputs oldest first, the conv
 *                       reads the last K-1 of them, and the row drops its
 *                       oldest L_new inputs and appends the new ones;
 *                       then the same recurrence on the pool's SSM state.
 *
 * Threads split only independent (batch, channel) / (batch, head) / request
 * work; each item is computed by one thread in sequential order, so the
 * result does not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef void (*item_fn)(void* ctx, long item);

typedef struct {
  item_fn fn;
  void* ctx;
  long n_items;
  long tid;
  long nthreads;
} worker_arg;

static void* worker_main(void* p) {
  worker_arg* a = (worker_arg*)p;
  for (long i = a->tid; i < a->n_items; i += a->nthreads) a->fn(a->ctx, i);
  return NULL;
}

static long resolve_threads(int nthreads, long n_items) {
  long t = nthreads;
  if (t <= 0) t = sysconf(_SC_NPROCESSORS_ONLN);
  if (t < 1) t = 1;
  if (t > n_items) t = n_items;
  if (t > 256) t = 256;
  return t < 1 ? 1 : t;
}

/* run fn(ctx, i) for i in [0, n_items), items interleaved over threads */
static void parallel_for(long n_items, int nthreads, item_fn fn, void* ctx) {
  if (n_items <= 0) return;
  long T = resolve_threads(nthreads, n_items);
  if (T == 1) {
    for (long i = 0; i < n_items; ++i) fn(ctx, i);
    return;
  }
  pthread_t th[256];
  worker_arg args[256];
  for (long t = 0; t < T; ++t) {
    args[t].fn = fn;
    args[t].ctx = ctx;
    args[t].n_items = n_items;
    args[t].tid = t;
    args[t].nthreads = T;
    pthread_create(&th[t], NULL, worker_main, &args[t]);
  }
  for (long t = 0; t < T; ++t) pthread_join(th[t], NULL);
}

int orc_num_threads(int nthreads) { return (int)resolve_threads(nthreads, 1L << 30); }

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* ------------------------------------------------------------------------ */
/* causal conv with state                                                   */
/* ------------------------------------------------------------------------ */

typedef struct {
  const double *x, *w, *bias, *S;
  double *u, *F;
  long Bz, L, D;
  int K, act;
} conv_ctx;

static void conv_item(void* p, long item) {
  conv_ctx* c = (conv_ctx*)p;
  const long b = item / c->D, d = item % c->D;
  const int K = c->K;
  const long L = c->L, D = c->D, E = L + K - 1;
  /* the extended sequence u = [S, x] for this (batch, channel) */
  double* ext = (double*)malloc(sizeof(double) * (size_t)(E > 0 ? E : 1));
  for (int j = 0; j < K - 1; ++j)
    ext[j] = c->S ? c->S[(b * D + d) * (K - 1) + j] : 0.0;
  for (long t = 0; t < L; ++t) ext[K - 1 + t] = c->x[(b * L + t) * D + d];
  const double beta = c->bias ? c->bias[d] : 0.0;
  for (long t = 0; t < L; ++t) {
    double z = beta;
    for (int k = 0; k < K; ++k) z += c->w[d * K + k] * ext[t + k];
    c->u[(b * L + t) * D + d] = c->act ? silu(z) : z;
  }
  /* final state: the K-1 newest entries of the extended sequence */
  for (int j = 0; j < K - 1; ++j) c->F[(b * D + d) * (K - 1) + j] = ext[L + j];
  free(ext);
}

int orc_conv_state_fwd(const double* x, const double* w, const double* bias,
                       const double* S, double* u, double* F, long Bz, long L,
                       long D, int K, int apply_silu, int nthreads) {
  if (Bz < 0 || L < 0 || D < 0 || K < 1) return -1;
  conv_ctx c = {x, w, bias, S, u, F, Bz, L, D, K, apply_silu};
  parallel_for(Bz * D, nthreads, conv_item, &c);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* its gradient with state                                                  */
/* ------------------------------------------------------------------------ */

/* d/dz of z / (1 + exp(-z)) = s (1 + z (1 - s)) with s the logistic function */
static double dsilu(double z) {
  const double s = 1.0 / (1.0 + exp(-z));
  return s * (1.0 + z * (1.0 - s));
}

typedef struct {
  const double *x, *w, *bias, *S, *dy, *q;
  double *dx, *dS, *dw, *dbias;
  long Bz, L, D;
  int K, act;
} convb_ctx;

/* one channel d, every sequence of the batch in order (dw and dbeta sum
   over the batch, so one thread owns the channel) */
static void convb_item(void* p, long d) {
  convb_ctx* c = (convb_ctx*)p;
  const int K = c->K;
  const long L = c->L, D = c->D, E = L + K - 1;
  double* ext = (double*)malloc(sizeof(double) * (size_t)(E > 0 ? E : 1));
  double* du = (double*)malloc(sizeof(double) * (size_t)(E > 0 ? E : 1));
  double* delta = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
  const double beta = c->bias ? c->bias[d] : 0.0;
  double dbeta = 0.0;
  for (int k = 0; k < K; ++k) c->dw[d * K + k] = 0.0;
  for (long b = 0; b < c->Bz; ++b) {
    /* forward again: the extended sequence and z_t */
    for (int j = 0; j < K - 1; ++j)
      ext[j] = c->S ? c->S[(b * D + d) * (K - 1) + j] : 0.0;
    for (long t = 0; t < L; ++t) ext[K - 1 + t] = c->x[(b * L + t) * D + d];
    for (long t = 0; t < L; ++t) {
      double z = beta;
      for (int k = 0; k < K; ++k) z += c->w[d * K + k] * ext[t + k];
      const double g = c->dy[(b * L + t) * D + d];
      delta[t] = c->act ? g * dsilu(z) : g;
    }
    /* dL/du: the convolution term, then the direct path of the tail slice */
    for (long j = 0; j < E; ++j) du[j] = 0.0;
    for (long t = 0; t < L; ++t)
      for (int k = 0; k < K; ++k) du[t + k] += delta[t] * c->w[d * K + k];
    for (int r = 0; r < K - 1; ++r)
      du[L + r] += c->q ? c->q[(b * D + d) * (K - 1) + r] : 0.0;
    for (int j = 0; j < K - 1; ++j) c->dS[(b * D + d) * (K - 1) + j] = du[j];
    for (long t = 0; t < L; ++t) c->dx[(b * L + t) * D + d] = du[K - 1 + t];
    for (int k = 0; k < K; ++k) {
      double acc = 0.0;
      for (long t = 0; t < L; ++t) acc += delta[t] * ext[t + k];
      c->dw[d * K + k] += acc;
    }
    for (long t = 0; t < L; ++t) dbeta += delta[t];
  }
  if (c->dbias) c->dbias[d] = dbeta;
  free(ext);
  free(du);
  free(delta);
}

int orc_conv_state_bwd(const double* x, const double* w, const double* bias,
                       const double* S, const double* dy, const double* q, double* dx,
                       double* dS, double* dw, double* dbias, long Bz, long L, long D, int K,
                       int apply_silu, int nthreads) {
  if (Bz < 0 || L < 0 || D < 0 || K < 1) return -1;
  convb_ctx c = {x, w, bias, S, dy, q, dx, dS, dw, dbias, Bz, L, D, K, apply_silu};
  parallel_for(D, nthreads, convb_item, &c);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* scalar-decay selective scan from an initial state                        */
/* ------------------------------------------------------------------------ */

typedef struct {
  const double *u, *dt, *A, *B, *C, *h0;
  double *y, *hT;
  long Bz, L, H, P, N, G;
} scan_ctx;

static void scan_item(void* p, long item) {
  scan_ctx* c = (scan_ctx*)p;
  const long H = c->H, P = c->P, N = c->N, G = c->G, L = c->L;
  const long b = item / H, hd = item % H;
  const long g = hd / (H / G);
  double* h = (double*)malloc(sizeof(double) * (size_t)(P * N > 0 ? P * N : 1));
  for (long i = 0; i < P * N; ++i)
    h[i] = c->h0 ? c->h0[(b * H + hd) * P * N + i] : 0.0;
  for (long t = 0; t < L; ++t) {
    const double a = exp(c->dt[(b * L + t) * H + hd] * c->A[hd]);
    const double* Bt = c->B + ((b * L + t) * G + g) * N;
    const double* Ct = c->C + ((b * L + t) * G + g) * N;
    const double* xt = c->u + ((b * L + t) * H + hd) * P;
    double* yt = c->y + ((b * L + t) * H + hd) * P;
    for (long pp = 0; pp < P; ++pp) {
      double acc = 0.0;
      for (long n = 0; n < N; ++n) {
        double v = a * h[pp * N + n] + xt[pp] * Bt[n];
        h[pp * N + n] = v;
        acc += v * Ct[n];
      }
      yt[pp] = acc;
    }
  }
  if (c->hT)
    for (long i = 0; i < P * N; ++i) c->hT[(b * H + hd) * P * N + i] = h[i];
  free(h);
}

int orc_ssm_scan(const double* u, const double* dt, const double* A,
                 const double* B, const double* C, const double* h0, double* y,
                 double* hT, long Bz, long L, long H, long P, long N, long G,
                 int nthreads) {
  if (Bz < 0 || L < 0 || H < 1 || P < 1 || N < 1 || G < 1 || H % G) return -1;
  scan_ctx c = {u, dt, A, B, C, h0, y, hT, Bz, L, H, P, N, G};
  parallel_for(Bz * H, nthreads, scan_item, &c);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* gradient of the scan, with the initial and final states                  */
/* ------------------------------------------------------------------------ */

typedef struct {
  const double *u, *dt, *A, *B, *C, *h0, *dy, *dhT;
  double *du, *ddt, *dA_part, *dB, *dC, *dh0;
  long Bz, L, H, P, N, G;
} scanb_ctx;

/* one (batch row, group): its heads in order, so the group sums of dB and dC
 * have one writer and a fixed order */
static void scanb_item(void* p, long item) {
  scanb_ctx* c = (scanb_ctx*)p;
  const long H = c->H, P = c->P, N = c->N, G = c->G, L = c->L, PN = c->P * c->N;
  const long b = item / G, g = item % G, hpg = H / G;
  for (long t = 0; t < L; ++t)
    for (long n = 0; n < N; ++n) {
      c->dB[((b * L + t) * G + g) * N + n] = 0.0;
      c->dC[((b * L + t) * G + g) * N + n] = 0.0;
    }
  /* hs[t + 1] = h_t, hs[0] = h_{-1} */
  double* hs = (double*)malloc(sizeof(double) * (size_t)((L + 1) * PN > 0 ? (L + 1) * PN : 1));
  double* gr = (double*)malloc(sizeof(double) * (size_t)(PN > 0 ? PN : 1));
  for (long hd = g * hpg; hd < (g + 1) * hpg; ++hd) {
    for (long i = 0; i < PN; ++i) hs[i] = c->h0 ? c->h0[(b * H + hd) * PN + i] : 0.0;
    for (long t = 0; t < L; ++t) {
      const double a = exp(c->dt[(b * L + t) * H + hd] * c->A[hd]);
      const double* Bt = c->B + ((b * L + t) * G + g) * N;
      const double* xt = c->u + ((b * L + t) * H + hd) * P;
      for (long pp = 0; pp < P; ++pp)
        for (long n = 0; n < N; ++n)
          hs[(t + 1) * PN + pp * N + n] = a * hs[t * PN + pp * N + n] + xt[pp] * Bt[n];
    }
    for (long i = 0; i < PN; ++i) gr[i] = c->dhT ? c->dhT[(b * H + hd) * PN + i] : 0.0;
    double dA_acc = 0.0;
    for (long t = L - 1; t >= 0; --t) {
      const double dtt = c->dt[(b * L + t) * H + hd];
      const double a = exp(dtt * c->A[hd]);
      const double* Bt = c->B + ((b * L + t) * G + g) * N;
      const double* Ct = c->C + ((b * L + t) * G + g) * N;
      const double* xt = c->u + ((b * L + t) * H + hd) * P;
      const double* dyt = c->dy + ((b * L + t) * H + hd) * P;
      const double* ht = hs + (t + 1) * PN;
      const double* hp = hs + t * PN;
      double* dBt = c->dB + ((b * L + t) * G + g) * N;
      double* dCt = c->dC + ((b * L + t) * G + g) * N;
      /* g = dL/dh_t: the later tokens' part already in gr, plus y_t's */
      for (long pp = 0; pp < P; ++pp)
        for (long n = 0; n < N; ++n) gr[pp * N + n] += dyt[pp] * Ct[n];
      for (long n = 0; n < N; ++n) {
        double sc = 0.0, sb = 0.0;
        for (long pp = 0; pp < P; ++pp) {
          sc += dyt[pp] * ht[pp * N + n];
          sb += gr[pp * N + n] * xt[pp];
        }
        dCt[n] += sc;
        dBt[n] += sb;
      }
      double da = 0.0;
      for (long pp = 0; pp < P; ++pp) {
        double sx = 0.0;
        for (long n = 0; n < N; ++n) {
          sx += gr[pp * N + n] * Bt[n];
          da += gr[pp * N + n] * hp[pp * N + n];
        }
        c->du[((b * L + t) * H + hd) * P + pp] = sx;
      }
      const double dl = a * da;
      c->ddt[(b * L + t) * H + hd] = dl * c->A[hd];
      dA_acc += dl * dtt;
      for (long i = 0; i < PN; ++i) gr[i] *= a; /* now dL/dh_{t-1} */
    }
    if (c->dh0)
      for (long i = 0; i < PN; ++i) c->dh0[(b * H + hd) * PN + i] = gr[i];
    c->dA_part[b * H + hd] = dA_acc;
  }
  free(gr);
  free(hs);
}

int orc_ssm_scan_bwd(const double* u, const double* dt, const double* A,
                     const double* B, const double* C, const double* h0,
                     const double* dy, const double* dhT, double* du, double* ddt,
                     double* dA, double* dB, double* dC, double* dh0, long Bz,
                     long L, long H, long P, long N, long G, int nthreads) {
  if (Bz < 0 || L < 0 || H < 1 || P < 1 || N < 1 || G < 1 || H % G) return -1;
  double* part = (double*)malloc(sizeof(double) * (size_t)(Bz * H > 0 ? Bz * H : 1));
  scanb_ctx c = {u, dt, A, B, C, h0, dy, dhT, du, ddt, part, dB, dC, dh0, Bz, L, H, P, N, G};
  parallel_for(Bz * G, nthreads, scanb_item, &c);
  for (long hd = 0; hd < H; ++hd) {
    double s = 0.0;
    for (long b = 0; b < Bz; ++b) s += part[b * H + hd];
    dA[hd] = s;
  }
  free(part);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* decode update over a circular conv-state pool                            */
/* ------------------------------------------------------------------------ */

typedef struct {
  const double *x, *w, *bias, *dt, *A, *B, *C;
  double *conv_pool, *ssm_pool, *y;
  const int32_t *seqlens, *idx;
  long Bz, Lnew, H, P, N, G, pool, S_len;
  int K;
  int* bad; /* per row: 1 if the row was skipped */
} upd_ctx;

static long pos_mod(long a, long m) {
  long r = a % m;
  return r < 0 ? r + m : r;
}

static void upd_item(void* p, long b) {
  upd_ctx* c = (upd_ctx*)p;
  const long H = c->H, P = c->P, N = c->N, G = c->G, D = H * P;
  const long Lnew = c->Lnew, S_len = c->S_len;
  const int K = c->K;
  const long r = c->idx ? (long)c->idx[b] : b;
  /* no lengths: the non-circular mode, the row holds the newest S_len
     inputs oldest first (as if its write pointer were always at S_len) */
  const int circular = c->seqlens != NULL;
  const long pl = circular ? (long)c->seqlens[b] : S_len;
  if (r < 0 || r >= c->pool || pl < 0) {
    c->bad[b] = 1;
    for (long i = 0; i < Lnew * D; ++i) c->y[b * Lnew * D + i] = 0.0;
    return;
  }
  double* u = (double*)malloc(sizeof(double) * (size_t)(Lnew * D > 0 ? Lnew * D : 1));
  double* ext = (double*)malloc(sizeof(double) * (size_t)(K - 1 + Lnew));
  double* row = c->conv_pool + r * D * S_len;
  for (long d = 0; d < D; ++d) {
    /* read every history value this call needs before any slot is written:
       logical position p - (K-1) + j lives in slot (p - (K-1) + j) mod S_len */
    for (int j = 0; j < K - 1; ++j)
      ext[j] = row[d * S_len + pos_mod(pl - (K - 1) + j, S_len)];
    for (long i = 0; i < Lnew; ++i) ext[K - 1 + i] = c->x[(b * Lnew + i) * D + d];
    const double beta = c->bias ? c->bias[d] : 0.0;
    for (long i = 0; i < Lnew; ++i) {
      double z = beta;
      for (int k = 0; k < K; ++k) z += c->w[d * K + k] * ext[i + k];
      u[i * D + d] = silu(z);
    }
    if (circular) {
      /* store the inputs (not the outputs) at the write pointer */
      for (long i = 0; i < Lnew; ++i)
        row[d * S_len + pos_mod(pl + i, S_len)] = c->x[(b * Lnew + i) * D + d];
    } else {
      /* drop the oldest L_new inputs, append the new ones: the row becomes
         the last S_len entries of [row, x_0 .. x_{L_new-1}] */
      double* seq = (double*)malloc(sizeof(double) * (size_t)(S_len + Lnew));
      for (long j = 0; j < S_len; ++j) seq[j] = row[d * S_len + j];
      for (long i = 0; i < Lnew; ++i) seq[S_len + i] = c->x[(b * Lnew + i) * D + d];
      for (long j = 0; j < S_len; ++j) row[d * S_len + j] = seq[Lnew + j];
      free(seq);
    }
  }
  for (long hd = 0; hd < H; ++hd) {
    const long g = hd / (H / G);
    double* h = c->ssm_pool + (r * H + hd) * P * N;
    for (long i = 0; i < Lnew; ++i) {
      const double a = exp(c->dt[(b * Lnew + i) * H + hd] * c->A[hd]);
      const double* Bt = c->B + ((b * Lnew + i) * G + g) * N;
      const double* Ct = c->C + ((b * Lnew + i) * G + g) * N;
      for (long pp = 0; pp < P; ++pp) {
        const double xv = u[i * D + hd * P + pp];
        double acc = 0.0;
        for (long n = 0; n < N; ++n) {
          double v = a * h[pp * N + n] + xv * Bt[n];
          h[pp * N + n] = v;
          acc += v * Ct[n];
        }
        c->y[((b * Lnew + i) * H + hd) * P + pp] = acc;
      }
    }
  }
  free(ext);
  free(u);
}

/* Returns the number of skipped rows (row index outside [0, pool) or a
   negative length: pools untouched, y row set to zero), or -1 on bad sizes.
   Rows whose slot appears twice are a caller contract violation; the oracle
   then applies rows one after another in batch order (single thread). */
int orc_mixer_update(const double* x, const double* w, const double* bias,
                     double* conv_pool, long pool, long S_len,
                     const int32_t* cache_seqlens, const int32_t* idx,
                     const double* dt, const double* A, const double* B,
                     const double* C, double* ssm_pool, double* y, long Bz,
                     long Lnew, long H, long P, long N, long G, int K,
                     int nthreads) {
  if (Bz < 0 || Lnew < 0 || H < 1 || P < 1 || N < 1 || G < 1 || H % G ||
      K < 1 || S_len < K - 1 || S_len < 1 || pool < 0)
    return -1;
  int* bad = (int*)calloc((size_t)(Bz > 0 ? Bz : 1), sizeof(int));
  int dup = 0;
  if (idx) {
    char* seen = (char*)calloc((size_t)(pool > 0 ? pool : 1), 1);
    for (long b = 0; b < Bz; ++b) {
      long r = idx[b];
      if (r >= 0 && r < pool) {
        if (seen[r]) dup = 1;
        seen[r] = 1;
      }
    }
    free(seen);
  }
  upd_ctx c = {x, w, bias, dt, A, B, C, conv_pool, ssm_pool, y, cache_seqlens, idx,
               Bz, Lnew, H, P, N, G, pool, S_len, K, bad};
  parallel_for(Bz, dup ? 1 : nthreads, upd_item, &c);
  int nbad = 0;
  for (long b = 0; b < Bz; ++b) nbad += bad[b];
  free(bad);
  return nbad;
}

/* ------------------------------------------------------------------------ */
/* the full Mamba-2 mixer wiring                                            */
/* ------------------------------------------------------------------------ */

/* log(1 + e^v), without overflow for large v */
static double softplus(double v) { return v > 30.0 ? v + log1p(exp(-v)) : log1p(exp(v)); }

typedef struct {
  const double *u, *z, *dtr, *dtb, *A, *Dsk, *h0;
  double *y, *hT;
  long Bz, L, H, P, N, G;
} m2_ctx;

static void m2_item(void* p, long item) {
  m2_ctx* c = (m2_ctx*)p;
  const long H = c->H, P = c->P, N = c->N, G = c->G, L = c->L;
  const long Dx = H * P, Dt = Dx + 2 * G * N;
  const long b = item / H, hd = item % H;
  const long g = hd / (H / G);
  const double Dh = c->Dsk ? c->Dsk[hd] : 0.0;
  double* h = (double*)malloc(sizeof(double) * (size_t)(P * N > 0 ? P * N : 1));
  for (long i = 0; i < P * N; ++i)
    h[i] = c->h0 ? c->h0[(b * H + hd) * P * N + i] : 0.0;
  for (long t = 0; t < L; ++t) {
    /* the conv output of token t: x of this head, B and C of its group */
    const double* ut = c->u + (b * L + t) * Dt;
    const double* xt = ut + hd * P;
    const double* Bt = ut + Dx + g * N;
    const double* Ct = ut + Dx + G * N + g * N;
    const double dt = softplus(c->dtr[(b * L + t) * H + hd] + (c->dtb ? c->dtb[hd] : 0.0));
    const double a = exp(dt * c->A[hd]);
    double* yt = c->y + ((b * L + t) * H + hd) * P;
    for (long pp = 0; pp < P; ++pp) {
      double acc = 0.0;
      for (long n = 0; n < N; ++n) {
        double v = a * h[pp * N + n] + dt * xt[pp] * Bt[n];
        h[pp * N + n] = v;
        acc += v * Ct[n];
      }
      const double gate = c->z ? silu(c->z[(b * L + t) * Dx + hd * P + pp]) : 1.0;
      yt[pp] = (acc + Dh * xt[pp]) * gate;
    }
  }
  if (c->hT)
    for (long i = 0; i < P * N; ++i) c->hT[(b * H + hd) * P * N + i] = h[i];
  free(h);
}

int orc_mamba2_scan(const double* u, const double* z, const double* dt_raw,
                    const double* dt_bias, const double* A, const double* D_skip,
                    const double* h0, double* y, double* hT, long Bz, long L, long H,
                    long P, long N, long G, int nthreads) {
  if (Bz < 0 || L < 0 || H < 1 || P < 1 || N < 1 || G < 1 || H % G) return -1;
  m2_ctx c = {u, z, dt_raw, dt_bias, A, D_skip, h0, y, hT, Bz, L, H, P, N, G};
  parallel_for(Bz * H, nthreads, m2_item, &c);
  return 0;
}

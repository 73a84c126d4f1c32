/*
 * Float64 CPU oracle of the Mamba-2 SSD core: forward recurrence and its
 * reverse-time analytic backward.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * definition the CUDA library is checked against.  Only the tests, the
 * smoke check and the benchmark's CPU-baseline leg load it; the library
 * never does.  It shares no code, header or constant with the CUDA path.
 *
 * What it restates (burn_dragon_kernel 0.5.0, page
 * src/sequence/mamba2/backward.rs):
 *   - forward: `ssd_forward_state_history_reference` — per step,
 *       decay = exp(dt_t * A_h),  h <- h * decay + dt_t * x_t (outer) B_t,
 *     with h starting from the initial state or zeros;
 *   - output: the `y_grouped` expression of `tensorized_mamba2_backward_impl`
 *       y_t = sum_n h_t[:, n] * C_t[n] + D_h * x_t;
 *   - backward: `ssd_backward_reference` — walking t from T-1 down to 0 with
 *     a carried state gradient:
 *       gS   = dy_t (outer) C_t + carry
 *       dC_t = sum over the group's heads and p of dy_t[p] * h_t[p, :]
 *       gda  = <gS, h_{t-1}>
 *       ddt  = <gS, x_t (outer) B_t> + gda * decay_t * A_h
 *       dA  += gda * decay_t * dt_t        (the page returns this times
 *                                           -exp(a_log) as grad_a_log)
 *       dB_t = sum over heads and p of gS[p, :] * dt_t * x_t[p]
 *       dx_t = D_h * dy_t + dt_t * gS B_t
 *       carry = gS * decay_t
 *     and dD = sum dy * x.
 * Readings where the page is silent:
 *   - dh0 (not returned on the page) is the carry left after t = 0;
 *   - the per-chunk history entry c is the state *before* step c * Q, so
 *     entry 0 is h0 (or zeros); the final state is the state after T - 1.
 *
 * Heads map to groups as h = g * (H / G) + j (the page reshapes nheads into
 * [ngroups, heads_per_group]).  Layouts (row-major): x, dy [B][T][H][P];
 * dt [B][T][H]; A, D [H]; Bm, Cm [B][T][G][N]; h0 [B][H][P][N];
 * chunk_states [B][nc][H][P][N].
 *
 * Memory: the backward never divides by a decay.  Each (b, h) task stores
 * the state every SEG steps on a forward sweep and recomputes one segment
 * at a time while walking back, so its memory is O(T/SEG + SEG) states.
 *
 * Determinism: one task per (b, h); the sums over heads (dB, dC) and over
 * batch (dA, dD) are taken after all tasks finish, in a fixed order, so the
 * result does not depend on the number of threads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SEG 64

typedef struct {
  int64_t B, T, H, P, N, G, Q;
  const double *x, *dt, *A, *Bm, *Cm, *D, *h0, *dy;
  double *y, *final_state, *chunk_states;
  /* backward outputs / per-task partials */
  double *dx, *ddt, *dh0;
  double *dB_part, *dC_part; /* [B][H][T][N] per-head contributions */
  double *dA_part, *dD_part; /* [B][H] */
  int64_t next_task;         /* atomic work counter */
  int failed;
} octx;

static inline int64_t nchunks_of(const octx* c) { return (c->T + c->Q - 1) / c->Q; }
static inline int64_t group_of(const octx* c, int64_t h) { return h / (c->H / c->G); }

/* One recurrence step on a P x N state. */
static void state_step(const octx* c, int64_t b, int64_t h, int64_t t, double* s) {
  const int64_t P = c->P, N = c->N, g = group_of(c, h);
  const double dtv = c->dt[(b * c->T + t) * c->H + h];
  const double decay = exp(dtv * c->A[h]);
  const double* xv = c->x + ((b * c->T + t) * c->H + h) * P;
  const double* Bv = c->Bm + ((b * c->T + t) * c->G + g) * N;
  for (int64_t p = 0; p < P; ++p) {
    const double u = dtv * xv[p];
    double* row = s + p * N;
    for (int64_t n = 0; n < N; ++n) row[n] = row[n] * decay + u * Bv[n];
  }
}

static void load_h0(const octx* c, int64_t b, int64_t h, double* s) {
  const int64_t PN = c->P * c->N;
  if (c->h0)
    memcpy(s, c->h0 + (b * c->H + h) * PN, (size_t)PN * sizeof(double));
  else
    memset(s, 0, (size_t)PN * sizeof(double));
}

static int forward_task(octx* c, int64_t b, int64_t h) {
  const int64_t P = c->P, N = c->N, PN = P * N, T = c->T, H = c->H, g = group_of(c, h);
  const int64_t nc = nchunks_of(c);
  double* s = (double*)malloc((size_t)PN * sizeof(double));
  if (!s) return -1;
  load_h0(c, b, h, s);
  for (int64_t t = 0; t < T; ++t) {
    if (c->chunk_states && t % c->Q == 0)
      memcpy(c->chunk_states + ((b * nc + t / c->Q) * H + h) * PN, s, (size_t)PN * sizeof(double));
    state_step(c, b, h, t, s);
    if (c->y) {
      const double* xv = c->x + ((b * T + t) * H + h) * P;
      const double* Cv = c->Cm + ((b * T + t) * c->G + g) * N;
      double* yv = c->y + ((b * T + t) * H + h) * P;
      for (int64_t p = 0; p < P; ++p) {
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) acc += s[p * N + n] * Cv[n];
        yv[p] = acc + c->D[h] * xv[p];
      }
    }
  }
  if (c->final_state) memcpy(c->final_state + (b * H + h) * PN, s, (size_t)PN * sizeof(double));
  free(s);
  return 0;
}

static int backward_task(octx* c, int64_t b, int64_t h) {
  const int64_t P = c->P, N = c->N, PN = P * N, T = c->T, H = c->H, G = c->G;
  const int64_t g = group_of(c, h);
  const int64_t nseg = (T + SEG - 1) / SEG;
  double* ckpt = (double*)malloc((size_t)(nseg * PN) * sizeof(double)); /* h_{t0-1} per segment */
  double* hs = (double*)malloc((size_t)(SEG * PN) * sizeof(double));    /* h_t inside a segment */
  double* carry = (double*)calloc((size_t)PN, sizeof(double));
  double* gS = (double*)malloc((size_t)PN * sizeof(double));
  if (!ckpt || !hs || !carry || !gS) {
    free(ckpt); free(hs); free(carry); free(gS);
    return -1;
  }
  double* s = hs; /* scratch for the checkpoint sweep */
  load_h0(c, b, h, s);
  for (int64_t t = 0; t < T; ++t) {
    if (t % SEG == 0) memcpy(ckpt + (t / SEG) * PN, s, (size_t)PN * sizeof(double));
    state_step(c, b, h, t, s);
  }

  double dA_acc = 0.0, dD_acc = 0.0;
  double* dBh = c->dB_part + (b * H + h) * T * N;
  double* dCh = c->dC_part + (b * H + h) * T * N;
  for (int64_t seg = nseg - 1; seg >= 0; --seg) {
    const int64_t t0 = seg * SEG;
    const int64_t t1 = (t0 + SEG < T) ? t0 + SEG : T;
    /* recompute h_t for t in [t0, t1) from h_{t0-1} */
    memcpy(hs, ckpt + seg * PN, (size_t)PN * sizeof(double));
    state_step(c, b, h, t0, hs);
    for (int64_t t = t0 + 1; t < t1; ++t) {
      memcpy(hs + (t - t0) * PN, hs + (t - t0 - 1) * PN, (size_t)PN * sizeof(double));
      state_step(c, b, h, t, hs + (t - t0) * PN);
    }
    for (int64_t t = t1 - 1; t >= t0; --t) {
      const double* cur = hs + (t - t0) * PN;
      const double* prev = (t > t0) ? hs + (t - t0 - 1) * PN : ckpt + seg * PN;
      const int64_t tok = (b * T + t) * H + h;
      const double dtv = c->dt[tok];
      const double decay = exp(dtv * c->A[h]);
      const double* xv = c->x + tok * P;
      const double* dyv = c->dy + tok * P;
      const double* Bv = c->Bm + ((b * T + t) * G + g) * N;
      const double* Cv = c->Cm + ((b * T + t) * G + g) * N;
      double* dBt = dBh + t * N;
      double* dCt = dCh + t * N;
      double gda = 0.0, drive = 0.0;
      for (int64_t n = 0; n < N; ++n) { dBt[n] = 0.0; dCt[n] = 0.0; }
      for (int64_t p = 0; p < P; ++p) {
        double gx = 0.0; /* sum_n gS[p, n] * B[n] */
        for (int64_t n = 0; n < N; ++n) {
          const double v = dyv[p] * Cv[n] + carry[p * N + n];
          gS[p * N + n] = v;
          dCt[n] += dyv[p] * cur[p * N + n];
          gda += v * prev[p * N + n];
          gx += v * Bv[n];
          dBt[n] += v * dtv * xv[p];
        }
        drive += gx * xv[p];
        c->dx[tok * P + p] = c->D[h] * dyv[p] + dtv * gx;
        dD_acc += dyv[p] * xv[p];
      }
      c->ddt[tok] = drive + gda * decay * c->A[h];
      dA_acc += gda * decay * dtv;
      for (int64_t i = 0; i < PN; ++i) carry[i] = gS[i] * decay;
    }
  }
  if (c->dh0) memcpy(c->dh0 + (b * H + h) * PN, carry, (size_t)PN * sizeof(double));
  c->dA_part[b * H + h] = dA_acc;
  c->dD_part[b * H + h] = dD_acc;
  free(ckpt); free(hs); free(carry); free(gS);
  return 0;
}

typedef struct { octx* c; int which; } worker_arg;

static void* worker(void* argp) {
  worker_arg* a = (worker_arg*)argp;
  octx* c = a->c;
  const int64_t ntask = c->B * c->H;
  for (;;) {
    const int64_t k = __atomic_fetch_add(&c->next_task, 1, __ATOMIC_RELAXED);
    if (k >= ntask) break;
    const int64_t b = k / c->H, h = k % c->H;
    const int rc = a->which == 0 ? forward_task(c, b, h) : backward_task(c, b, h);
    if (rc) __atomic_store_n(&c->failed, 1, __ATOMIC_RELAXED);
  }
  return NULL;
}

static int run_tasks(octx* c, int which, int nthreads) {
  const int64_t ntask = c->B * c->H;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > ntask) nthreads = (int)ntask;
  c->next_task = 0;
  c->failed = 0;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  worker_arg wa = {c, which};
  if (!th) return -1;
  int started = 0;
  for (int i = 1; i < nthreads; ++i) {
    if (pthread_create(&th[i], NULL, worker, &wa) != 0) break;
    started = i;
  }
  worker(&wa);
  for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
  free(th);
  return c->failed ? -1 : 0;
}

static int check_dims(int64_t B, int64_t T, int64_t H, int64_t P, int64_t N, int64_t G, int64_t Q) {
  if (B < 1 || T < 1 || H < 1 || P < 1 || N < 1 || G < 1 || Q < 1) return -2;
  if (H % G) return -2;
  return 0;
}

/* Returns 0 on success, -1 on allocation failure, -2 on bad dimensions.
 * y, final_state and chunk_states may be NULL (not computed). */
int oracle_ssd_forward(int64_t B, int64_t T, int64_t H, int64_t P, int64_t N, int64_t G,
                       int64_t Q, const double* x, const double* dt, const double* A,
                       const double* Bm, const double* Cm, const double* D, const double* h0,
                       double* y, double* final_state, double* chunk_states, int nthreads) {
  if (check_dims(B, T, H, P, N, G, Q)) return -2;
  octx c;
  memset(&c, 0, sizeof c);
  c.B = B; c.T = T; c.H = H; c.P = P; c.N = N; c.G = G; c.Q = Q;
  c.x = x; c.dt = dt; c.A = A; c.Bm = Bm; c.Cm = Cm; c.D = D; c.h0 = h0;
  c.y = y; c.final_state = final_state; c.chunk_states = chunk_states;
  return run_tasks(&c, 0, nthreads);
}

/* Gradients of L = sum(dy * y) w.r.t. x, dt, A, B, C, D and h0.
 * dh0 may be NULL.  Outputs are overwritten. */
int oracle_ssd_backward(int64_t B, int64_t T, int64_t H, int64_t P, int64_t N, int64_t G,
                        int64_t Q, const double* x, const double* dt, const double* A,
                        const double* Bm, const double* Cm, const double* D, const double* h0,
                        const double* dy, double* dx, double* ddt, double* dA, double* dBm,
                        double* dCm, double* dD, double* dh0, int nthreads) {
  if (check_dims(B, T, H, P, N, G, Q)) return -2;
  octx c;
  memset(&c, 0, sizeof c);
  c.B = B; c.T = T; c.H = H; c.P = P; c.N = N; c.G = G; c.Q = Q;
  c.x = x; c.dt = dt; c.A = A; c.Bm = Bm; c.Cm = Cm; c.D = D; c.h0 = h0; c.dy = dy;
  c.dx = dx; c.ddt = ddt; c.dh0 = dh0;
  const size_t part = (size_t)(B * H * T * N);
  c.dB_part = (double*)malloc(part * sizeof(double));
  c.dC_part = (double*)malloc(part * sizeof(double));
  c.dA_part = (double*)malloc((size_t)(B * H) * sizeof(double));
  c.dD_part = (double*)malloc((size_t)(B * H) * sizeof(double));
  int rc = -1;
  if (c.dB_part && c.dC_part && c.dA_part && c.dD_part) rc = run_tasks(&c, 1, nthreads);
  if (rc == 0) {
    const int64_t hpg = H / G;
    /* fixed-order sums: heads of a group in head order, batch in batch order */
    for (int64_t b = 0; b < B; ++b)
      for (int64_t t = 0; t < T; ++t)
        for (int64_t g = 0; g < G; ++g) {
          double* oB = dBm + ((b * T + t) * G + g) * N;
          double* oC = dCm + ((b * T + t) * G + g) * N;
          for (int64_t n = 0; n < N; ++n) { oB[n] = 0.0; oC[n] = 0.0; }
          for (int64_t j = 0; j < hpg; ++j) {
            const int64_t h = g * hpg + j;
            const double* pB = c.dB_part + ((b * H + h) * T + t) * N;
            const double* pC = c.dC_part + ((b * H + h) * T + t) * N;
            for (int64_t n = 0; n < N; ++n) { oB[n] += pB[n]; oC[n] += pC[n]; }
          }
        }
    for (int64_t h = 0; h < H; ++h) {
      double sa = 0.0, sd = 0.0;
      for (int64_t b = 0; b < B; ++b) { sa += c.dA_part[b * H + h]; sd += c.dD_part[b * H + h]; }
      dA[h] = sa;
      dD[h] = sd;
    }
  }
  free(c.dB_part); free(c.dC_part); free(c.dA_part); free(c.dD_part);
  return rc;
}

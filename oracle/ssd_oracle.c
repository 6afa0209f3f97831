/*
 * ssd_oracle.c -- float64 CPU oracle of the Mamba-2 selective state-space
 * (SSD) layer, forward and reverse mode.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link or call
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg use it.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes (the plain definition, evaluated token by token):
 *
 *   Page "llm-mamba-200" (gigipick.blogspot.com), section 1 ("the core
 *   bottleneck of Mamba/S4: the recurrence") defines the layer as a linear
 *   recurrence h_t = f(h_{t-1}, x_t) with input-dependent (selective) A and B;
 *   the equation itself is lost from the extracted text, so the recurrence is
 *   read in its Mamba-2 form with a scalar decay per head:
 *
 *     dt_eff_t = softplus(dt_t + dt_bias_h)
 *     a_t      = exp(dt_eff_t * A_h)
 *     h_t      = a_t * h_{t-1} + dt_eff_t * x_t (outer) B_t        (P x N)
 *     y_t      = h_t . C_t + D_h * x_t                              (P)
 *
 *   with h_{-1} = initial_states (or 0).  When seq_idx is given, a token whose
 *   segment id differs from its predecessor's starts a new sequence: the state
 *   entering it is zero (the initial state feeds only the first segment).
 *
 * The reverse mode is derived by hand from the recurrence above (the pages
 * name the backward only as the state-passing backward of the same scan, page
 * "B200 Helion Mamba-2" (aitrends.kr/articles/109906), section "Helion based
 * B200 kernel redesign"):
 *
 *   g_t  = dL/dh_t = dy_t (outer) C_t + [t+1 < L and no reset at t+1] a_{t+1} g_{t+1}
 *          (+ dfinal_states at t = L-1)
 *   hp_t = state entering step t (0 after a reset)
 *   dx_t = D_h dy_t + dt_eff_t * g_t B_t
 *   dB_t += dt_eff_t * g_t^T x_t          dC_t += h_t^T dy_t   (summed over the
 *                                                              heads of a group)
 *   ddt_eff_t = <g_t, x_t (outer) B_t> + A_h a_t <g_t, hp_t>
 *   dA_h  += dt_eff_t a_t <g_t, hp_t>       dD_h += <dy_t, x_t>
 *   ddt_t = ddt_eff_t * sigmoid(dt_t + dt_bias_h),   ddt_bias_h += ddt_t
 *   dinitial_states = a_0 g_0
 *
 * Layouts (row-major, dense): x, y, dx, dy (b,L,H,P); dt, ddt (b,L,H);
 * B, C, dB, dC (b,L,G,N); states (b,H,P,N); seq_idx (b,L) int32; A, D,
 * dt_bias and their gradients (H).  Head h belongs to group floor(h*G/H).
 *
 * The backward keeps a checkpoint of h every S ~ sqrt(L) steps and recomputes
 * each span forward while walking it backward (recomputation is bit-identical
 * in float64).  Work is spread over OpenMP threads: forward by (b, h), backward
 * by (b, group) so that the group sums of dB and dC, and every other sum, are
 * taken in one fixed order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int g_threads = 0;      /* 0: OpenMP default */
static int g_last_threads = 1; /* threads used by the last parallel region */

void oracle_set_threads(int n) { g_threads = n; }
int oracle_last_threads(void) { return g_last_threads; }
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

static int pick_threads(long units) {
  int n = g_threads > 0 ? g_threads : oracle_max_threads();
  if (units < n) n = (int)units;
  if (n < 1) n = 1;
  return n;
}

/* softplus in a form that neither overflows nor loses digits for large |z|. */
static double softplus(double z) { return (z > 0.0 ? z : 0.0) + log1p(exp(-fabs(z))); }
static double sigmoid(double z) {
  if (z >= 0.0) return 1.0 / (1.0 + exp(-z));
  double e = exp(z);
  return e / (1.0 + e);
}

typedef struct {
  long b, L, H, P, N, G;
} dims_t;

static long group_of(const dims_t* d, long h) { return h * d->G / d->H; }

/* Does token t of row bi start a new sequence (segment id differs from t-1)? */
static int is_reset(const int32_t* seq_idx, const dims_t* d, long bi, long t) {
  if (!seq_idx || t == 0) return 0;
  return seq_idx[bi * d->L + t] != seq_idx[bi * d->L + t - 1];
}

/* One recurrence step for head (bi, h) at token t: state hs (P*N) is updated in
 * place from the state entering the step.  Returns a_t; *de gets dt_eff_t. */
static double step_fwd(const dims_t* d, long bi, long h, long t, const double* x, const double* dt,
                       const double* dt_bias, const double* A, const double* B,
                       const int32_t* seq_idx, double* hs, double* de_out) {
  const long P = d->P, N = d->N, g = group_of(d, h);
  double de = softplus(dt[(bi * d->L + t) * d->H + h] + dt_bias[h]);
  double a = exp(de * A[h]);
  double a_eff = is_reset(seq_idx, d, bi, t) ? 0.0 : a;
  const double* xt = x + ((bi * d->L + t) * d->H + h) * P;
  const double* Bt = B + ((bi * d->L + t) * d->G + g) * N;
  for (long p = 0; p < P; ++p)
    for (long n = 0; n < N; ++n) hs[p * N + n] = a_eff * hs[p * N + n] + de * xt[p] * Bt[n];
  if (de_out) *de_out = de;
  return a;
}

int oracle_ssd_fwd(long batch, long seqlen, long nheads, long headdim, long dstate, long ngroups,
                   const double* x, const double* dt, const double* dt_bias, const double* A,
                   const double* B, const double* C, const double* D,
                   const double* initial_states, const int32_t* seq_idx, double* y,
                   double* final_states) {
  dims_t d = {batch, seqlen, nheads, headdim, dstate, ngroups};
  if (batch < 1 || seqlen < 1 || nheads < 1 || headdim < 1 || dstate < 1 || ngroups < 1 ||
      nheads % ngroups != 0)
    return 1;
  const long P = headdim, N = dstate, units = batch * nheads;
  int nth = pick_threads(units);
  g_last_threads = nth;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nth)
  for (long u = 0; u < units; ++u) {
    long bi = u / d.H, h = u % d.H, g = group_of(&d, h);
    double* hs = (double*)calloc((size_t)(P * N), sizeof(double));
    if (!hs) {
#pragma omp atomic write
      err = 2;
      continue;
    }
    if (initial_states) memcpy(hs, initial_states + (bi * d.H + h) * P * N, sizeof(double) * P * N);
    for (long t = 0; t < d.L; ++t) {
      step_fwd(&d, bi, h, t, x, dt, dt_bias, A, B, seq_idx, hs, NULL);
      const double* Ct = C + ((bi * d.L + t) * d.G + g) * N;
      const double* xt = x + ((bi * d.L + t) * d.H + h) * P;
      double* yt = y + ((bi * d.L + t) * d.H + h) * P;
      for (long p = 0; p < P; ++p) {
        double acc = 0.0;
        for (long n = 0; n < N; ++n) acc += hs[p * N + n] * Ct[n];
        yt[p] = acc + D[h] * xt[p];
      }
    }
    if (final_states) memcpy(final_states + (bi * d.H + h) * P * N, hs, sizeof(double) * P * N);
    free(hs);
  }
  return err;
}

/* Reverse mode.  Every gradient output is overwritten.  dfinal_states and
 * dinitial_states may be NULL (zero upstream / not wanted). */
int oracle_ssd_bwd(long batch, long seqlen, long nheads, long headdim, long dstate, long ngroups,
                   const double* x, const double* dt, const double* dt_bias, const double* A,
                   const double* B, const double* C, const double* D,
                   const double* initial_states, const int32_t* seq_idx, const double* dy,
                   const double* dfinal_states, double* dx, double* ddt, double* ddt_bias,
                   double* dA, double* dB, double* dC, double* dD, double* dinitial_states) {
  dims_t d = {batch, seqlen, nheads, headdim, dstate, ngroups};
  if (batch < 1 || seqlen < 1 || nheads < 1 || headdim < 1 || dstate < 1 || ngroups < 1 ||
      nheads % ngroups != 0)
    return 1;
  const long P = headdim, N = dstate, L = seqlen, H = nheads, G = ngroups, PN = headdim * dstate;
  long S = (long)ceil(sqrt((double)L));
  if (S < 1) S = 1;
  const long nck = (L + S - 1) / S;
  /* Per-(b,h) partial sums of the per-head parameter gradients, folded over b
   * in a fixed order after the parallel region. */
  double* pdA = (double*)calloc((size_t)(batch * H), sizeof(double));
  double* pdD = (double*)calloc((size_t)(batch * H), sizeof(double));
  double* pdb = (double*)calloc((size_t)(batch * H), sizeof(double));
  if (!pdA || !pdD || !pdb) {
    free(pdA); free(pdD); free(pdb);
    return 2;
  }
  memset(dB, 0, sizeof(double) * batch * L * G * N);
  memset(dC, 0, sizeof(double) * batch * L * G * N);
  const long units = batch * G;
  int nth = pick_threads(units);
  g_last_threads = nth;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nth)
  for (long u = 0; u < units; ++u) {
    long bi = u / G, gi = u % G;
    double* ck = (double*)malloc(sizeof(double) * nck * PN);   /* state before token k*S */
    double* hs = (double*)malloc(sizeof(double) * S * PN);     /* states h_t of one span */
    double* gcur = (double*)malloc(sizeof(double) * PN);
    double* hrun = (double*)malloc(sizeof(double) * PN);
    if (!ck || !hs || !gcur || !hrun) {
      free(ck); free(hs); free(gcur); free(hrun);
#pragma omp atomic write
      err = 2;
      continue;
    }
    for (long h = 0; h < H; ++h) {
      if (group_of(&d, h) != gi) continue;
      /* forward sweep, keeping a checkpoint every S tokens */
      if (initial_states) memcpy(hrun, initial_states + (bi * H + h) * PN, sizeof(double) * PN);
      else memset(hrun, 0, sizeof(double) * PN);
      for (long t = 0; t < L; ++t) {
        if (t % S == 0) memcpy(ck + (t / S) * PN, hrun, sizeof(double) * PN);
        step_fwd(&d, bi, h, t, x, dt, dt_bias, A, B, seq_idx, hrun, NULL);
      }
      /* gnext = dL/dh_t arriving from later tokens; at t = L-1 it is dfinal */
      if (dfinal_states) memcpy(gcur, dfinal_states + (bi * H + h) * PN, sizeof(double) * PN);
      else memset(gcur, 0, sizeof(double) * PN);
      for (long k = nck - 1; k >= 0; --k) {
        long t0 = k * S, t1 = t0 + S < L ? t0 + S : L;
        memcpy(hrun, ck + k * PN, sizeof(double) * PN);
        for (long t = t0; t < t1; ++t) {
          step_fwd(&d, bi, h, t, x, dt, dt_bias, A, B, seq_idx, hrun, NULL);
          memcpy(hs + (t - t0) * PN, hrun, sizeof(double) * PN);
        }
        for (long t = t1 - 1; t >= t0; --t) {
          const double* ht = hs + (t - t0) * PN;
          const double* hprev = (t == t0) ? ck + k * PN : hs + (t - 1 - t0) * PN;
          const int reset = is_reset(seq_idx, &d, bi, t);
          const double z = dt[(bi * L + t) * H + h] + dt_bias[h];
          const double de = softplus(z), a = exp(de * A[h]);
          const double* xt = x + ((bi * L + t) * H + h) * P;
          const double* dyt = dy + ((bi * L + t) * H + h) * P;
          const double* Bt = B + ((bi * L + t) * G + gi) * N;
          const double* Ct = C + ((bi * L + t) * G + gi) * N;
          double* dxt = dx + ((bi * L + t) * H + h) * P;
          double* dBt = dB + ((bi * L + t) * G + gi) * N;
          double* dCt = dC + ((bi * L + t) * G + gi) * N;
          /* g_t = (gradient from later tokens) + dy_t (outer) C_t */
          for (long p = 0; p < P; ++p)
            for (long n = 0; n < N; ++n) gcur[p * N + n] += dyt[p] * Ct[n];
          double s_xb = 0.0, s_hp = 0.0, s_dyx = 0.0;
          for (long p = 0; p < P; ++p) {
            double acc = 0.0;
            for (long n = 0; n < N; ++n) {
              acc += gcur[p * N + n] * Bt[n];
              s_xb += gcur[p * N + n] * xt[p] * Bt[n];
              if (!reset) s_hp += gcur[p * N + n] * hprev[p * N + n];
            }
            dxt[p] = D[h] * dyt[p] + de * acc;
            s_dyx += dyt[p] * xt[p];
          }
          for (long n = 0; n < N; ++n) {
            double accb = 0.0, accc = 0.0;
            for (long p = 0; p < P; ++p) {
              accb += gcur[p * N + n] * xt[p];
              accc += ht[p * N + n] * dyt[p];
            }
            dBt[n] += de * accb;
            dCt[n] += accc;
          }
          const double ddt_eff = s_xb + A[h] * a * s_hp;
          const double ddt_t = ddt_eff * sigmoid(z);
          ddt[(bi * L + t) * H + h] = ddt_t;
          pdA[bi * H + h] += de * a * s_hp;
          pdD[bi * H + h] += s_dyx;
          pdb[bi * H + h] += ddt_t;
          /* hand the gradient to h_{t-1}: it flows only through a_t, and not
           * at all across a sequence reset */
          const double carry = reset ? 0.0 : a;
          for (long e = 0; e < PN; ++e) gcur[e] *= carry;
        }
      }
      if (dinitial_states) memcpy(dinitial_states + (bi * H + h) * PN, gcur, sizeof(double) * PN);
    }
    free(ck); free(hs); free(gcur); free(hrun);
  }
  for (long h = 0; h < H; ++h) {
    double sa = 0.0, sd = 0.0, sb = 0.0;
    for (long bi = 0; bi < batch; ++bi) {
      sa += pdA[bi * H + h];
      sd += pdD[bi * H + h];
      sb += pdb[bi * H + h];
    }
    dA[h] = sa;
    dD[h] = sd;
    ddt_bias[h] = sb;
  }
  free(pdA); free(pdD); free(pdb);
  return err;
}

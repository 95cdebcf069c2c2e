/*
 * CPU oracle for the fused scaled linear layer -- TEST INFRASTRUCTURE ONLY.
 * The definition it follows, and its sources on the pages, are in
 * eg_oracle.h.  Build: gcc -O2 -ffp-contract=off -fPIC -shared -pthread
 * (no FMA contraction, so x86 and Arm hosts give the same bits).
 */
#define _GNU_SOURCE
#include "eg_oracle.h"

#include <math.h>
#include <pthread.h>
#include <sched.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------ codecs --- */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
double orc_bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP 8-bit floating point, E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa
 * bits; exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there
 * is no infinity, so the largest finite magnitude is 1.75 * 2^8 = 448. */
double orc_e4m3_to_double(uint8_t code) {
  int sign = code >> 7;
  int e = (code >> 3) & 0xF;
  int m = code & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -mag : mag;
}

/* Round a float64 to bf16 (8 significant bits, exponent range of binary32)
 * with ties to even, in one step (not through float32). */
uint16_t orc_bf16_from_double(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7F80;
  int e;
  frexp(a, &e); /* a = f * 2^e, f in [0.5, 1): leading bit weight 2^(e-1) */
  int lead = e - 1;
  if (lead < -126) lead = -126;         /* subnormal bf16 share one quantum */
  double q = ldexp(1.0, lead - 7);      /* spacing of bf16 values near a */
  double n = nearbyint(a / q);          /* a/q is exact; ties to even */
  double r = n * q;
  if (r >= 0x1p128) return sign | 0x7F80; /* rounds past the largest finite */
  float f = (float)r;                   /* exact: r is a bf16 value */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return sign | (uint16_t)(u >> 16);
}

/* Activations, written out from their definitions: ReLU max(v, 0); GELU with
 * the Gaussian CDF 0.5*(1 + erf(v/sqrt 2)); its tanh approximation
 * 0.5*v*(1 + tanh(sqrt(2/pi)*(v + 0.044715 v^3))) (the constant printed on
 * the page, 0.79788456, is sqrt(2/pi) rounded); SiLU v * sigmoid(v). */
double orc_act(int32_t act, double v) {
  switch (act) {
    case ORC_ACT_NONE: return v;
    case ORC_ACT_RELU: return v > 0.0 ? v : 0.0;
    case ORC_ACT_GELU_ERF: return 0.5 * v * (1.0 + erf(v / sqrt(2.0)));
    case ORC_ACT_GELU_TANH: {
      double c = sqrt(2.0 / M_PI);
      return 0.5 * v * (1.0 + tanh(c * (v + 0.044715 * v * v * v)));
    }
    case ORC_ACT_SILU: return v / (1.0 + exp(-v));
    default: return NAN;
  }
}

/* ------------------------------------------------------------ helpers --- */

static double decode(int32_t dtype, const void* base, int64_t idx) {
  switch (dtype) {
    case ORC_IN_BF16: return orc_bf16_to_double(((const uint16_t*)base)[idx]);
    case ORC_IN_E4M3: return orc_e4m3_to_double(((const uint8_t*)base)[idx]);
    case ORC_IN_INT8: return (double)((const int8_t*)base)[idx];
    default: return NAN;
  }
}

static int check(const orc_problem* p, const void* A, const void* W,
                 const float* sa, const float* sw, const uint16_t* bias,
                 const uint16_t* R) {
  if (!p || p->M < 0 || p->N < 0 || p->K < 0) return -1;
  if (p->M && p->N && (!A || !W)) return -1;
  if (p->dtype < ORC_IN_BF16 || p->dtype > ORC_IN_INT8) return -1;
  if (p->scale == ORC_SCALE_NONE) {
    if (p->dtype != ORC_IN_BF16) return -1;
  } else if (p->scale == ORC_SCALE_TOKEN_CHANNEL) {
    if (!sa || !sw) return -1;
  } else if (p->scale == ORC_SCALE_BLOCK) {
    if (!sa || !sw || p->dtype != ORC_IN_E4M3 || p->K % 128) return -1;
  } else {
    return -1;
  }
  if ((p->flags & ORC_BIAS) && !bias) return -1;
  if ((p->flags & (ORC_RESIDUAL | ORC_RESIDUAL_PRE_ACT)) && !R) return -1;
  if (p->act < ORC_ACT_NONE || p->act > ORC_ACT_SILU) return -1;
  if ((p->flags & ORC_OUT_F16) && (p->flags & ORC_OUT_E4M3)) return -1;
  if ((p->flags & ORC_OUT_E4M3) && !(p->s_y > 0.0f && isfinite(p->s_y))) return -1;
  return 0;
}

/* The epilogue for one output element, steps in the order given above. */
static uint16_t epilogue(const orc_problem* p, int64_t m, int64_t n, double acc,
                         const float* sa, const float* sw, const uint16_t* bias,
                         const uint16_t* R) {
  double v = acc;
  if (p->scale == ORC_SCALE_TOKEN_CHANNEL) v = v * ((double)sa[m] * (double)sw[n]);
  if (p->flags & ORC_BIAS) v = v + orc_bf16_to_double(bias[n]);
  if (p->flags & ORC_RESIDUAL_PRE_ACT) {
    v = v + orc_bf16_to_double(R[m * p->N + n]);
    v = orc_act(p->act, v);
  } else {
    v = orc_act(p->act, v);
    if (p->flags & ORC_RESIDUAL) v = v + orc_bf16_to_double(R[m * p->N + n]);
  }
  if (p->flags & ORC_OUT_F16) return orc_f16_from_double(v);
  if (p->flags & ORC_OUT_E4M3) return orc_e4m3_from_double(v / (double)p->s_y);
  return orc_bf16_from_double(v);
}

/* Accumulator of one output from decoded rows a[K] and w[K]. */
static double accum_row(const orc_problem* p, const double* a, const double* w,
                        int64_t m, int64_t n, const float* sa, const float* sw,
                        int64_t* exact) {
  const int64_t K = p->K;
  if (p->scale == ORC_SCALE_BLOCK) {
    const int64_t KB = K / 128;
    double acc = 0.0;
    for (int64_t kb = 0; kb < KB; kb++) {
      double part = 0.0;
      for (int64_t k = kb * 128; k < kb * 128 + 128; k++) part += a[k] * w[k];
      acc += ((double)sa[m * KB + kb] * (double)sw[(n / 128) * KB + kb]) * part;
    }
    return acc;
  }
  if (p->dtype == ORC_IN_INT8) {
    int64_t s = 0;
    for (int64_t k = 0; k < K; k++) s += (int64_t)a[k] * (int64_t)w[k];
    if (exact) *exact = s;
    return (double)s;
  }
  double acc = 0.0;
  for (int64_t k = 0; k < K; k++) acc += a[k] * w[k];
  return acc;
}

int orc_default_threads(void) {
  cpu_set_t set;
  if (sched_getaffinity(0, sizeof set, &set) == 0) {
    int c = CPU_COUNT(&set);
    if (c > 0) return c;
  }
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

/* --------------------------------------------------------- full / naive --- */

typedef struct {
  const orc_problem* p;
  const void *A, *W;
  const float *sa, *sw;
  const uint16_t *bias, *R;
  uint16_t* Y;
  double* acc;
  int64_t* acc_i64;
  const double* Ad; /* decoded A, [M][K] */
  int64_t n0, n1;
} full_job;

static void* full_worker(void* arg) {
  full_job* j = (full_job*)arg;
  const orc_problem* p = j->p;
  const int64_t K = p->K, N = p->N;
  double* w = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
  if (!w) return (void*)1;
  for (int64_t n = j->n0; n < j->n1; n++) {
    for (int64_t k = 0; k < K; k++) w[k] = decode(p->dtype, j->W, n * K + k);
    for (int64_t m = 0; m < p->M; m++) {
      int64_t ex = 0;
      double acc = accum_row(p, j->Ad + m * K, w, m, n, j->sa, j->sw, &ex);
      if (j->acc) j->acc[m * N + n] = acc;
      if (j->acc_i64 && p->dtype == ORC_IN_INT8) j->acc_i64[m * N + n] = ex;
      if (j->Y) j->Y[m * N + n] = epilogue(p, m, n, acc, j->sa, j->sw, j->bias, j->R);
    }
  }
  free(w);
  return NULL;
}

int orc_linear(const orc_problem* p, const void* A, const void* W,
               const float* sa, const float* sw, const uint16_t* bias,
               const uint16_t* R, uint16_t* Y, double* acc, int64_t* acc_i64,
               int nthreads) {
  if (check(p, A, W, sa, sw, bias, R)) return -1;
  if (p->M == 0 || p->N == 0) return 0;
  const int64_t M = p->M, K = p->K;
  double* Ad = (double*)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
  if (!Ad) return -1;
  for (int64_t i = 0; i < M * K; i++) Ad[i] = decode(p->dtype, A, i);
  int T = nthreads > 0 ? nthreads : orc_default_threads();
  if (T > p->N) T = (int)p->N;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)T);
  full_job* jobs = (full_job*)malloc(sizeof(full_job) * (size_t)T);
  int rc = 0;
  for (int t = 0; t < T; t++) {
    full_job j = {p, A, W, sa, sw, bias, R, Y, acc, acc_i64, Ad,
                  p->N * t / T, p->N * (t + 1) / T};
    jobs[t] = j;
    if (pthread_create(&th[t], NULL, full_worker, &jobs[t])) { rc = -1; T = t; break; }
  }
  for (int t = 0; t < T; t++) {
    void* r = NULL;
    pthread_join(th[t], &r);
    if (r) rc = -1;
  }
  free(th);
  free(jobs);
  free(Ad);
  return rc;
}

int orc_linear_naive(const orc_problem* p, const void* A, const void* W,
                     const float* sa, const float* sw, const uint16_t* bias,
                     const uint16_t* R, uint16_t* Y, double* acc,
                     int64_t* acc_i64) {
  if (check(p, A, W, sa, sw, bias, R)) return -1;
  const int64_t M = p->M, N = p->N, K = p->K;
  for (int64_t m = 0; m < M; m++) {
    for (int64_t n = 0; n < N; n++) {
      double s = 0.0;
      int64_t si = 0;
      if (p->scale == ORC_SCALE_BLOCK) {
        for (int64_t kb = 0; kb < K / 128; kb++) {
          double part = 0.0;
          for (int64_t k = kb * 128; k < kb * 128 + 128; k++)
            part += decode(p->dtype, A, m * K + k) * decode(p->dtype, W, n * K + k);
          s += ((double)sa[m * (K / 128) + kb] * (double)sw[(n / 128) * (K / 128) + kb]) * part;
        }
      } else {
        for (int64_t k = 0; k < K; k++) {
          if (p->dtype == ORC_IN_INT8)
            si += (int64_t)((const int8_t*)A)[m * K + k] * (int64_t)((const int8_t*)W)[n * K + k];
          else
            s += decode(p->dtype, A, m * K + k) * decode(p->dtype, W, n * K + k);
        }
        if (p->dtype == ORC_IN_INT8) s = (double)si;
      }
      if (acc) acc[m * N + n] = s;
      if (acc_i64 && p->dtype == ORC_IN_INT8) acc_i64[m * N + n] = si;
      if (Y) Y[m * N + n] = epilogue(p, m, n, s, sa, sw, bias, R);
    }
  }
  return 0;
}

/* ------------------------------------------------------------- points --- */

typedef struct {
  const orc_problem* p;
  const void *A, *W;
  const float *sa, *sw;
  const uint16_t *bias, *R;
  const int64_t *ms, *ns;
  uint16_t* Y;
  double* acc;
  int64_t i0, i1;
} pts_job;

static void* pts_worker(void* arg) {
  pts_job* j = (pts_job*)arg;
  const orc_problem* p = j->p;
  const int64_t K = p->K;
  double* a = (double*)malloc(sizeof(double) * (size_t)(2 * (K > 0 ? K : 1)));
  if (!a) return (void*)1;
  double* w = a + (K > 0 ? K : 1);
  for (int64_t i = j->i0; i < j->i1; i++) {
    int64_t m = j->ms[i], n = j->ns[i];
    for (int64_t k = 0; k < K; k++) {
      a[k] = decode(p->dtype, j->A, m * K + k);
      w[k] = decode(p->dtype, j->W, n * K + k);
    }
    double acc = accum_row(p, a, w, m, n, j->sa, j->sw, NULL);
    if (j->acc) j->acc[i] = acc;
    if (j->Y) j->Y[i] = epilogue(p, m, n, acc, j->sa, j->sw, j->bias, j->R);
  }
  free(a);
  return NULL;
}

int orc_linear_points(const orc_problem* p, const void* A, const void* W,
                      const float* sa, const float* sw, const uint16_t* bias,
                      const uint16_t* R, const int64_t* ms, const int64_t* ns,
                      int64_t npts, uint16_t* Y, double* acc, int nthreads) {
  if (check(p, A, W, sa, sw, bias, R) || npts < 0 || (npts && (!ms || !ns))) return -1;
  for (int64_t i = 0; i < npts; i++)
    if (ms[i] < 0 || ms[i] >= p->M || ns[i] < 0 || ns[i] >= p->N) return -1;
  if (npts == 0) return 0;
  int T = nthreads > 0 ? nthreads : orc_default_threads();
  if (T > npts) T = (int)npts;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)T);
  pts_job* jobs = (pts_job*)malloc(sizeof(pts_job) * (size_t)T);
  int rc = 0;
  for (int t = 0; t < T; t++) {
    pts_job j = {p, A, W, sa, sw, bias, R, ms, ns, Y, acc,
                 npts * t / T, npts * (t + 1) / T};
    jobs[t] = j;
    if (pthread_create(&th[t], NULL, pts_worker, &jobs[t])) { rc = -1; T = t; break; }
  }
  for (int t = 0; t < T; t++) {
    void* r = NULL;
    pthread_join(th[t], &r);
    if (r) rc = -1;
  }
  free(th);
  free(jobs);
  return rc;
}

/* ------------------------------------------------------------ split-K --- */

int orc_accum_splitk(const orc_problem* p, const void* A, const void* W,
                     const float* sa, const float* sw, int64_t S, int64_t kunit,
                     double* acc, int64_t* acc_i64) {
  if (check(p, A, W, sa, sw, NULL, NULL) || S < 1 || kunit < 1 || !acc) return -1;
  if (p->scale == ORC_SCALE_BLOCK && kunit % 128) return -1;
  const int64_t M = p->M, N = p->N, K = p->K;
  const int64_t T = (K + kunit - 1) / kunit;
  if (S > T && T > 0) return -1;
  const int64_t KB = K / 128;
  for (int64_t m = 0; m < M; m++) {
    for (int64_t n = 0; n < N; n++) {
      double total = 0.0;
      int64_t itotal = 0;
      for (int64_t s = 0; s < S; s++) {
        int64_t k0 = (s * T / S) * kunit, k1 = ((s + 1) * T / S) * kunit;
        if (k1 > K) k1 = K;
        double part = 0.0;
        int64_t ipart = 0;
        if (p->scale == ORC_SCALE_BLOCK) {
          for (int64_t kb = k0 / 128; kb < k1 / 128; kb++) {
            double blk = 0.0;
            for (int64_t k = kb * 128; k < kb * 128 + 128; k++)
              blk += decode(p->dtype, A, m * K + k) * decode(p->dtype, W, n * K + k);
            part += ((double)sa[m * KB + kb] * (double)sw[(n / 128) * KB + kb]) * blk;
          }
        } else if (p->dtype == ORC_IN_INT8) {
          for (int64_t k = k0; k < k1; k++)
            ipart += (int64_t)((const int8_t*)A)[m * K + k] * (int64_t)((const int8_t*)W)[n * K + k];
        } else {
          for (int64_t k = k0; k < k1; k++)
            part += decode(p->dtype, A, m * K + k) * decode(p->dtype, W, n * K + k);
        }
        total += part;
        itotal += ipart;
      }
      if (p->dtype == ORC_IN_INT8 && p->scale != ORC_SCALE_BLOCK) total = (double)itotal;
      acc[m * N + n] = total;
      if (acc_i64 && p->dtype == ORC_IN_INT8) acc_i64[m * N + n] = itotal;
    }
  }
  return 0;
}


/* ---------------------------------------------------------------------- */
/* Per-token dynamic quantisation.                                         */

/* E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent field 0 holds
 * the subnormals m * 2^-9; the all-ones pattern S.1111.111 is NaN, so the
 * largest finite magnitude is 1.75 * 2^8 = 448.  The magnitude is rounded
 * on the grid of its binade (the subnormal grid 2^-9 below 2^-6), ties to
 * even; a result past 448 saturates. */
uint8_t orc_e4m3_from_float(float v) { return orc_e4m3_from_double((double)v); }

uint8_t orc_e4m3_from_double(double v) {
  const uint8_t sign = signbit(v) ? 0x80 : 0;
  if (isnan(v)) return sign | 0x7F;
  const double a = fabs(v);
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);          /* a = f * 2^e, f in [0.5, 1) */
  int lead = e - 1;      /* a in [2^lead, 2^(lead+1)) */
  if (lead < -6) lead = -6;                 /* subnormals share the 2^-9 grid */
  const double quantum = ldexp(1.0, lead - 3);
  const double n = nearbyint(a / quantum);  /* exact quotient; ties to even */
  const double r = n * quantum;             /* the rounded magnitude */
  if (r >= 448.0) return sign | 0x7E;       /* 448 or beyond: saturate */
  if (r < 0x1p-6) return sign | (uint8_t)nearbyint(r / 0x1p-9);  /* subnormal (or 0) */
  int er;
  const double fr = frexp(r, &er);          /* r = fr * 2^er, fr in [0.5, 1) */
  const int exp_field = er - 1 + 7;
  const int mant = (int)((fr * 2.0 - 1.0) * 8.0);  /* exact: r is on the grid */
  return sign | (uint8_t)((exp_field << 3) | mant);
}

int orc_quant_rows(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, int32_t dtype,
                   uint8_t* q, int64_t ldq, float* s) {
  if (M < 0 || K < 0 || (M > 0 && (!s || (K > 0 && (!x || !q)))) || ldx < K || ldq < K) return -1;
  if (dtype != ORC_IN_E4M3 && dtype != ORC_IN_INT8) return -1;
  const float qmax = dtype == ORC_IN_E4M3 ? 448.0f : 127.0f;
  for (int64_t m = 0; m < M; ++m) {
    const uint16_t* row = x + m * ldx;
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      const float v = fabsf((float)orc_bf16_to_double(row[k]));  /* exact */
      if (v > amax) amax = v;
    }
    const float sm = amax > 0.0f ? amax / qmax : 1.0f;
    s[m] = sm;
    for (int64_t k = 0; k < K; ++k) {
      const float t = (float)orc_bf16_to_double(row[k]) / sm;   /* float32 division */
      uint8_t code;
      if (dtype == ORC_IN_E4M3) {
        code = orc_e4m3_from_float(t);
      } else {
        float r = nearbyintf(t);  /* ties to even */
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        code = (uint8_t)(int8_t)r;
      }
      q[m * ldq + k] = code;
    }
  }
  return 0;
}


/* ---------------------------------------------------------------------- */
/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits; exponent
 * field 0 holds the subnormals m * 2^-24; field 31 is infinity / NaN. */
double orc_f16_to_double(uint16_t bits) {
  const int sign = bits >> 15;
  const int e = (bits >> 10) & 0x1F;
  const int m = bits & 0x3FF;
  double mag;
  if (e == 31) mag = m ? NAN : INFINITY;
  else if (e == 0) mag = ldexp((double)m, -24);
  else mag = ldexp(1.0 + (double)m / 1024.0, e - 15);
  return sign ? -mag : mag;
}

uint16_t orc_f16_from_double(double v) {
  const uint16_t sign = signbit(v) ? 0x8000 : 0;
  if (isnan(v)) return 0x7E00;
  const double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7C00;
  int e;
  frexp(a, &e);
  int lead = e - 1;
  if (lead < -14) lead = -14;                /* subnormals share the 2^-24 grid */
  const double quantum = ldexp(1.0, lead - 10);
  const double n = nearbyint(a / quantum);   /* exact quotient; ties to even */
  const double r = n * quantum;
  if (r >= 65536.0) return sign | 0x7C00;    /* past the largest finite: infinity */
  if (r < 0x1p-14) return sign | (uint16_t)nearbyint(r / 0x1p-24);
  int er;
  const double fr = frexp(r, &er);
  const int exp_field = er - 1 + 15;
  const int mant = (int)((fr * 2.0 - 1.0) * 1024.0);
  return sign | (uint16_t)((exp_field << 10) | mant);
}


/* ---------------------------------------------------------------------- */
/* Gated linear unit over the two W halves.                                */

static uint16_t round_out(const orc_problem* p, double v) {
  if (p->flags & ORC_OUT_F16) return orc_f16_from_double(v);
  if (p->flags & ORC_OUT_E4M3) return orc_e4m3_from_double(v / (double)p->s_y);
  return orc_bf16_from_double(v);
}

int orc_linear_gated(const orc_problem* p, const void* A, const void* W, const float* sa,
                     const float* sw, const uint16_t* bias, const uint16_t* R, uint16_t* Y,
                     int nthreads) {
  if (!p || (p->flags & ORC_RESIDUAL_PRE_ACT)) return -1;
  if ((p->flags & ORC_BIAS) && !bias) return -1;
  if ((p->flags & ORC_RESIDUAL) && !R) return -1;
  if (p->scale == ORC_SCALE_BLOCK && p->N % 128) return -1;
  const int64_t M = p->M, N = p->N;
  if (M == 0 || N == 0) return 0;
  /* the accumulators of all 2N weight rows, from the plain accumulation */
  orc_problem inner = *p;
  inner.N = 2 * N;
  inner.flags = 0;
  inner.act = ORC_ACT_NONE;
  double* acc = (double*)malloc(sizeof(double) * (size_t)(M * 2 * N));
  if (!acc) return -1;
  int rc = orc_linear(&inner, A, W, sa, sw, NULL, NULL, NULL, acc, NULL, nthreads);
  if (rc == 0) {
    for (int64_t m = 0; m < M; m++) {
      for (int64_t n = 0; n < N; n++) {
        double g = acc[m * 2 * N + n], u = acc[m * 2 * N + N + n];
        if (p->scale == ORC_SCALE_TOKEN_CHANNEL) {
          g = g * ((double)sa[m] * (double)sw[n]);
          u = u * ((double)sa[m] * (double)sw[N + n]);
        }
        if (p->flags & ORC_BIAS) {
          g = g + orc_bf16_to_double(bias[n]);
          u = u + orc_bf16_to_double(bias[N + n]);
        }
        double y = orc_act(p->act, g) * u;
        if (p->flags & ORC_RESIDUAL) y = y + orc_bf16_to_double(R[m * N + n]);
        Y[m * N + n] = round_out(p, y);
      }
    }
  }
  free(acc);
  return rc;
}

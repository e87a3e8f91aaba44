/*
 * lean_oracle.c -- plain float64 CPU oracle for LeanAttention decode-phase
 * attention.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library. It shares no code,
 * header, table or constant with the CUDA library, and nothing here is used
 * to produce a product result.
 *
 * What it computes, and where the pages define it:
 *
 *   attention (xllm-io paper review, "3.1 standard attention"):
 *       S = Q K^T,  P = softmax(S / sqrt(d)),  O = P V
 *     with one query token per (request, head) in the decode phase
 *     (same review, "2.1 problem background" table: decode has N_q = 1).
 *     The scale is passed in explicitly ("scale" below; 1/sqrt(d) in every
 *     workload) and applied to every score before the softmax.
 *
 *   partial result of a block of keys (same review, "3.2 softmax rescaling
 *   as a reduction", part 1):
 *       m = rowmax(S),  l = rowsum(exp(S - m)),  Obar = exp(S - m) V
 *
 *   the rescaling reduction f (same section, part 2):
 *       m_xy = max(m_x, m_y)
 *       l_xy = exp(m_x - m_xy) l_x + exp(m_y - m_xy) l_y
 *       Obar_xy = exp(m_x - m_xy) Obar_x + exp(m_y - m_xy) Obar_y
 *       O = Obar_xy / l_xy
 *
 * The full-context result is the definition written out: a two-pass
 * softmax (pass 1: the maximum score; pass 2: the exponential sums),
 * nothing blocked, fused or reordered. Rows (request, query head) are
 * independent and are spread over threads; each row's arithmetic is
 * sequential in token order.
 *
 * Element decoding: fp16 and bf16 inputs are decoded from their bit
 * patterns into doubles from the IEEE 754 binary16 definition and from the
 * bfloat16 definition (the upper half of an IEEE binary32), so every input
 * value is used exactly.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1, ORACLE_F64 = 2 };

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double mag;
  if (e == 0) {
    mag = ldexp((double)f, -24); /* subnormal: f/1024 * 2^-14 */
  } else if (e == 31) {
    mag = (f == 0) ? INFINITY : NAN;
  } else {
    mag = ldexp(1024.0 + (double)f, e - 25); /* (1 + f/1024) * 2^(e-15) */
  }
  return sign ? -mag : mag;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_double(uint16_t b) {
  int sign = (b >> 15) & 1;
  int e = (b >> 7) & 0xff;
  int f = b & 0x7f;
  double mag;
  if (e == 0) {
    mag = ldexp((double)f, -133); /* subnormal: f/128 * 2^-126 */
  } else if (e == 255) {
    mag = (f == 0) ? INFINITY : NAN;
  } else {
    mag = ldexp(128.0 + (double)f, e - 134); /* (1 + f/128) * 2^(e-127) */
  }
  return sign ? -mag : mag;
}

void oracle_decode_array(int dtype, const uint16_t* src, double* dst, long n) {
  for (long i = 0; i < n; ++i)
    dst[i] = dtype == ORACLE_F16 ? oracle_half_to_double(src[i]) : oracle_bf16_to_double(src[i]);
}

/* Element i of an input array, as a double. */
static double elem(const void* base, long i, int dtype) {
  if (dtype == ORACLE_F16) return oracle_half_to_double(((const uint16_t*)base)[i]);
  if (dtype == ORACLE_BF16) return oracle_bf16_to_double(((const uint16_t*)base)[i]);
  return ((const double*)base)[i];
}

/*
 * One row of attention over keys/values [t0, t1) of a slab.
 * q: d elements at element offset q_off; keys and values of token t at
 * element offset kv_off + t*d. Writes the partial triple of part 1 of
 * "3.2 softmax rescaling as a reduction": m, l and the unscaled Obar[d].
 * The scores are computed once into s[] (pass 1 takes their maximum,
 * pass 2 the exponential sums), so the arithmetic is the definition itself.
 * An empty range gives the identity triple (-inf, 0, 0).
 */
static int partial_row(int d, int dtype, const void* q, long q_off, const void* k, const void* v,
                       long kv_off, long t0, long t1, double scale, double* m_out, double* l_out,
                       double* obar) {
  long n = t1 - t0;
  for (int c = 0; c < d; ++c) obar[c] = 0.0;
  if (n <= 0) {
    *m_out = -INFINITY;
    *l_out = 0.0;
    return 0;
  }
  double* s = (double*)malloc(sizeof(double) * (size_t)n);
  if (!s) return -1;
  /* S = scale * q K^T over the block */
  for (long t = 0; t < n; ++t) {
    long krow = kv_off + (t0 + t) * (long)d;
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc += elem(q, q_off + c, dtype) * elem(k, krow + c, dtype);
    s[t] = scale * acc;
  }
  /* pass 1: m = rowmax(S) */
  double m = -INFINITY;
  for (long t = 0; t < n; ++t)
    if (s[t] > m) m = s[t];
  /* pass 2: l = rowsum(exp(S - m)), Obar = exp(S - m) V */
  double l = 0.0;
  for (long t = 0; t < n; ++t) {
    double p = exp(s[t] - m);
    long vrow = kv_off + (t0 + t) * (long)d;
    l += p;
    for (int c = 0; c < d; ++c) obar[c] += p * elem(v, vrow + c, dtype);
  }
  free(s);
  *m_out = m;
  *l_out = l;
  return 0;
}

/*
 * The rescaling reduction f of "3.2 softmax rescaling as a reduction",
 * part 2, on triples laid out as [m, l, Obar[0..d)]. The identity triple
 * (-inf, 0, 0) is handled explicitly: exp(-inf - (-inf)) is undefined, and
 * merging with an empty block must return the other operand.
 */
void oracle_merge_f(int d, const double* x, const double* y, double* out) {
  double mx = x[0], my = y[0];
  if (mx == -INFINITY) {
    memmove(out, y, sizeof(double) * (size_t)(d + 2));
    return;
  }
  if (my == -INFINITY) {
    memmove(out, x, sizeof(double) * (size_t)(d + 2));
    return;
  }
  double m = mx > my ? mx : my;
  double ax = exp(mx - m), ay = exp(my - m);
  double l = ax * x[1] + ay * y[1];
  for (int c = 0; c < d; ++c) out[2 + c] = ax * x[2 + c] + ay * y[2 + c];
  out[0] = m;
  out[1] = l;
}

/* O = diag(l)^-1 Obar: the final scaling of part 2. */
void oracle_normalise(int d, const double* x, double* o) {
  for (int c = 0; c < d; ++c) o[c] = x[2 + c] / x[1];
}

/* Partial triple [m, l, Obar[d]] of one row over tokens [t0, t1). */
int oracle_partial(int d, int dtype, const void* q, const void* k, const void* v, long t0, long t1,
                   double scale, double* triple) {
  return partial_row(d, dtype, q, 0, k, v, 0, t0, t1, scale, &triple[0], &triple[1], triple + 2);
}

/*
 * Layout of the batched inputs (decode phase, ragged batch):
 *   q   [batch, nq, hq, d]  (nq = 1: one query token per request)
 *   k,v per request b: a [hkv, L_b, d] slab at element offset hkv*cu[b]*d,
 *       L_b = cu[b+1] - cu[b]; token t of kv head h at (hkv*cu[b] + h*L_b + t)*d.
 *   query head h reads kv head h / (hq/hkv).
 *   With nq > 1 (verification of speculative tokens) the queries are the
 *   last nq tokens of the context: query i sits at position L_b - nq + i and
 *   sees keys 0 .. L_b - nq + i (causal).
 *   out [nrows, d] for the requested rows (row index r = (b*nq + i)*hq + h).
 */
typedef struct {
  int batch, nq, hq, hkv, d, dtype;
  const int32_t* cu;
  const void *q, *k, *v;
  double scale;
  long nrows;
  const int64_t* rows;
  double* out;
  int nthreads, tid;
  int status;
} job_t;

static void* attend_worker(void* arg) {
  job_t* j = (job_t*)arg;
  int grp = j->hq / j->hkv;
  double* tri = (double*)malloc(sizeof(double) * (size_t)(j->d + 2));
  if (!tri) {
    j->status = -1;
    return NULL;
  }
  for (long i = j->tid; i < j->nrows; i += j->nthreads) {
    long r = j->rows ? (long)j->rows[i] : i;
    long h = r % j->hq, bq = r / j->hq, b = bq / j->nq, qi = bq % j->nq, kvh = h / grp;
    long L = (long)j->cu[b + 1] - (long)j->cu[b];
    long kv_off = ((long)j->hkv * j->cu[b] + kvh * L) * (long)j->d;
    long visible = L - (j->nq - 1 - qi); /* keys 0 .. L - nq + qi */
    if (partial_row(j->d, j->dtype, j->q, r * (long)j->d, j->k, j->v, kv_off, 0, visible, j->scale,
                    &tri[0], &tri[1], tri + 2) != 0) {
      j->status = -1;
      break;
    }
    oracle_normalise(j->d, tri, j->out + i * (long)j->d);
  }
  free(tri);
  return NULL;
}

/*
 * Full-context decode attention for the listed rows (rows == NULL: all
 * batch*hq rows in order). Returns 0, or -1 on bad arguments or allocation
 * failure.
 */
int oracle_attend_spec(int batch, int nq, int hq, int hkv, int d, const int32_t* cu, int dtype,
                       const void* q, const void* k, const void* v, double scale, long nrows,
                       const int64_t* rows, double* out, int nthreads) {
  if (batch <= 0 || nq <= 0 || hq <= 0 || hkv <= 0 || d <= 0 || hq % hkv != 0) return -1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  for (long i = 0; i < nrows; ++i) {
    long r = rows ? (long)rows[i] : i;
    if (r < 0 || r >= (long)batch * nq * hq) return -1;
  }
  for (int b = 0; b < batch; ++b)
    if (cu[b + 1] - cu[b] < nq) return -1; /* the query tokens are part of the context */
  job_t jobs[256];
  pthread_t th[256];
  for (int t = 0; t < nthreads; ++t) {
    job_t j = {batch, nq, hq, hkv, d, dtype, cu, q, k, v, scale, nrows, rows, out, nthreads, t, 0};
    jobs[t] = j;
  }
  if (nthreads == 1) {
    attend_worker(&jobs[0]);
    return jobs[0].status;
  }
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, attend_worker, &jobs[t]) != 0) break;
    ++started;
  }
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  /* rows of threads that could not start are computed here */
  for (int t = started; t < nthreads; ++t) attend_worker(&jobs[t]);
  for (int t = 0; t < nthreads; ++t)
    if (jobs[t].status != 0) return -1;
  return 0;
}

/* Decode attention with one query token per request: the definition of
   "3.1 standard attention" with N_q = 1. */
int oracle_attend(int batch, int hq, int hkv, int d, const int32_t* cu, int dtype, const void* q,
                  const void* k, const void* v, double scale, long nrows, const int64_t* rows,
                  double* out, int nthreads) {
  return oracle_attend_spec(batch, 1, hq, hkv, d, cu, dtype, q, k, v, scale, nrows, rows, out,
                            nthreads);
}

/*
 * Brute-force checkers that pin the oracle's element codecs (test code only).
 *
 * The oracle's encoders are written as a decision table (E2M1) and as an
 * exponent/mantissa rounding (E4M3).  These checkers instead search the table of
 * representable values for the nearest one (ties to the even code), and sweep every
 * float32 bit pattern.  The value tables are passed in by the caller (the E4M3
 * table comes from torch's float8_e4m3fn decoding; the E2M1 magnitudes from the
 * OCP definition), so nothing here shares arithmetic with the oracle.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

typedef uint8_t (*enc_fn)(float);

static float as_f32(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Exact comparison of |a - m1| against |a - m2| (m1 < m2, both small table values):
 * returns <0 if m1 is nearer, >0 if m2 is nearer, 0 on a tie.  When a lies outside
 * [m1, m2] the nearer value is the one on a's side; inside, both differences are
 * exact in double because a is then a float32 no larger than the table's maximum. */
static int closer(double a, double m1, double m2) {
  if (a <= m1) return -1;
  if (a >= m2) return 1;
  double d1 = a - m1, d2 = m2 - a;
  return (d1 < d2) ? -1 : (d1 > d2) ? 1 : 0;
}

/* ---------- E2M1: nearest of the 8 magnitudes, every candidate compared ---------- */
static uint8_t brute_e2m1(const double* mag, float y) {
  double a = fabs((double)y);
  int best = 0;
  for (int i = 1; i < 8; ++i) {
    int c = closer(a, mag[best], mag[i]);
    if (c > 0 || (c == 0 && (i % 2) == 0 && (best % 2) != 0)) best = i;
  }
  return (uint8_t)((signbit(y) ? 8 : 0) | best);
}

typedef struct {
  enc_fn enc;
  const double* table;
  uint64_t lo, hi;
  int64_t bad;
  uint32_t first_bad;
} job_t;

static void* e2m1_worker(void* p) {
  job_t* j = (job_t*)p;
  for (uint64_t u = j->lo; u < j->hi; ++u) {
    uint32_t b = (uint32_t)u;
    if ((b & 0x7F800000u) == 0x7F800000u) continue; /* inf / nan: out of contract */
    float y = as_f32(b);
    if (j->enc(y) != brute_e2m1(j->table, y)) {
      if (j->bad == 0) j->first_bad = b;
      j->bad++;
    }
  }
  return NULL;
}

/* ---------- E4M3: nearest of the 127 finite non-negative values ---------- */
static int nearest_e4m3(const double* val, int j, double v) {
  /* val ascending (code order); val[j] <= v; returns the nearest code, ties to even */
  if (j >= 126) return 126;
  double dl = v - val[j], dh = val[j + 1] - v;
  if (dl < dh) return j;
  if (dh < dl) return j + 1;
  return (j % 2 == 0) ? j : j + 1;
}

static void* e4m3_worker(void* p) {
  job_t* jb = (job_t*)p;
  const double* val = jb->table;
  double v0 = (double)as_f32((uint32_t)jb->lo);
  int j = 0;
  while (j < 126 && val[j + 1] <= v0) ++j;
  for (uint64_t u = jb->lo; u < jb->hi; ++u) {
    double v = (double)as_f32((uint32_t)u);
    while (j < 126 && val[j + 1] <= v) ++j;
    int want = nearest_e4m3(val, j, v);
    if (jb->enc((float)v) != (uint8_t)want) {
      if (jb->bad == 0) jb->first_bad = (uint32_t)u;
      jb->bad++;
    }
  }
  return NULL;
}

static int64_t run(void* (*fn)(void*), enc_fn enc, const double* table, uint64_t lo, uint64_t hi,
                   int nthreads, uint32_t* first_bad) {
  job_t jobs[64];
  pthread_t th[64];
  if (nthreads > 64) nthreads = 64;
  if (nthreads < 1) nthreads = 1;
  uint64_t span = (hi - lo + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].enc = enc;
    jobs[t].table = table;
    jobs[t].lo = lo + span * t;
    jobs[t].hi = jobs[t].lo + span < hi ? jobs[t].lo + span : hi;
    if (jobs[t].lo > hi) jobs[t].lo = hi;
    jobs[t].bad = 0;
    jobs[t].first_bad = 0;
    pthread_create(&th[t], NULL, fn, &jobs[t]);
  }
  int64_t bad = 0;
  *first_bad = 0;
  for (int t = 0; t < nthreads; ++t) {
    pthread_join(th[t], NULL);
    if (jobs[t].bad && bad == 0) *first_bad = jobs[t].first_bad;
    bad += jobs[t].bad;
  }
  return bad;
}

/* Every float32 bit pattern except inf/nan. */
int64_t pin_e2m1_sweep(enc_fn enc, const double* mag8, int nthreads, uint32_t* first_bad) {
  return run(e2m1_worker, enc, mag8, 0, 1ull << 32, nthreads, first_bad);
}

/* Every finite non-negative float32 (patterns 0 .. 0x7F7FFFFF). */
int64_t pin_e4m3_sweep(enc_fn enc, const double* val127, int nthreads, uint32_t* first_bad) {
  return run(e4m3_worker, enc, val127, 0, 0x7F800000ull, nthreads, first_bad);
}

/* Full brute force (all 127 candidates compared) on given patterns; sign mirrored. */
int64_t pin_e4m3_brute(enc_fn enc, const double* val127, const uint32_t* patterns, int64_t n,
                       uint32_t* first_bad) {
  int64_t bad = 0;
  *first_bad = 0;
  for (int64_t i = 0; i < n; ++i) {
    float f = as_f32(patterns[i]);
    if (!isfinite(f)) continue;
    double a = fabs((double)f);
    int best = 0;
    for (int c = 1; c < 127; ++c) {
      int cmp = closer(a, val127[best], val127[c]);
      if (cmp > 0 || (cmp == 0 && (c % 2) == 0 && (best % 2) != 0)) best = c;
    }
    uint8_t want = (uint8_t)((signbit(f) ? 0x80 : 0) | best);
    if (enc(f) != want) {
      if (bad == 0) *first_bad = patterns[i];
      bad++;
    }
  }
  return bad;
}

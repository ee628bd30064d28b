/*
 * Seeded synthetic input generator for the DSA layer workloads.
 *
 * This file draws random numbers and nothing else: it holds none of the
 * indexer / top-k / attention arithmetic. Both the fp64 oracle and the CUDA
 * path are fed from what it writes, so the two sides see identical inputs.
 *
 * Every value is a pure function of (seed, stream, flat index): a counter-based
 * generator built on the SplitMix64 finaliser (Steele, Lea, Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014). There is no
 * hidden state, so any slice of a tensor can be regenerated on its own and the
 * output does not depend on the thread count.
 *
 *   word(seed, stream, i) = mix64(base(seed, stream) + i)
 *   base(seed, stream)    = mix64((seed << 20) ^ stream)
 *
 * Integer draws on [lo, hi] use the high 32 bits of a word (multiply-shift).
 * Normal draws use the Box-Muller transform on two 53-bit uniforms and are
 * rounded to bfloat16 with round-to-nearest-even directly from double.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t mix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static inline uint64_t stream_base(uint64_t seed, uint64_t stream) {
  return mix64((seed << 20) ^ stream);
}

uint64_t synth_word(uint64_t seed, uint64_t stream, uint64_t i) {
  return mix64(stream_base(seed, stream) + i);
}

/* integer uniform on [lo, hi] */
static inline int64_t draw_int(uint64_t w, int64_t lo, int64_t hi) {
  uint64_t span = (uint64_t)(hi - lo + 1);
  return lo + (int64_t)(((w >> 32) * span) >> 32);
}

/* bfloat16 bit pattern of x, rounded to nearest, ties to even, from double */
static uint16_t bf16_rne(double x) {
  if (x == 0.0) return signbit(x) ? 0x8000u : 0u;
  if (isnan(x)) return 0x7FC0u;
  int e;
  double m = frexp(fabs(x), &e);       /* |x| = m * 2^e, m in [0.5, 1) */
  double q = ldexp(m, 8);              /* 8 significant bits in [128, 256) */
  double r = nearbyint(q);             /* default mode: ties to even */
  double y = ldexp(r, e - 8);
  if (signbit(x)) y = -y;
  float f = (float)y;                  /* exact: y has <= 9 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

typedef struct {
  int kind;            /* 0 normal bf16, 1 dyadic bf16, 2 dyadic f32, 3 signed nonzero f32 */
  void* out;
  int64_t begin, end;  /* element range */
  uint64_t seed, stream;
  int64_t lo, hi;
  int denom_log2;
} job_t;

static void run_job(job_t* j) {
  uint64_t base = stream_base(j->seed, j->stream);
  double scale = ldexp(1.0, -j->denom_log2);
  if (j->kind == 0) {
    uint16_t* o = (uint16_t*)j->out;
    /* element 2p uses cos, element 2p+1 uses sin of the same pair p */
    for (int64_t i = j->begin; i < j->end; ++i) {
      int64_t p = i >> 1;
      uint64_t w1 = mix64(base + 2 * (uint64_t)p);
      uint64_t w2 = mix64(base + 2 * (uint64_t)p + 1);
      double u1 = ((double)(w1 >> 11) + 1.0) * 0x1.0p-53; /* (0, 1] */
      double u2 = (double)(w2 >> 11) * 0x1.0p-53;         /* [0, 1) */
      double r = sqrt(-2.0 * log(u1));
      double a = 6.283185307179586476925286766559 * u2;
      double z = (i & 1) ? r * sin(a) : r * cos(a);
      o[i] = bf16_rne(z);
    }
  } else if (j->kind == 1) {
    uint16_t* o = (uint16_t*)j->out;
    for (int64_t i = j->begin; i < j->end; ++i)
      o[i] = bf16_rne((double)draw_int(mix64(base + (uint64_t)i), j->lo, j->hi) * scale);
  } else if (j->kind == 2) {
    float* o = (float*)j->out;
    for (int64_t i = j->begin; i < j->end; ++i)
      o[i] = (float)((double)draw_int(mix64(base + (uint64_t)i), j->lo, j->hi) * scale);
  } else {
    /* uniform over {+-1, ..., +-hi} / 2^denom_log2 (zero excluded) */
    float* o = (float*)j->out;
    for (int64_t i = j->begin; i < j->end; ++i) {
      int64_t r = draw_int(mix64(base + (uint64_t)i), 0, 2 * j->hi - 1);
      int64_t v = r < j->hi ? r - j->hi : r - j->hi + 1;
      o[i] = (float)((double)v * scale);
    }
  }
}

static void* thread_main(void* arg) {
  run_job((job_t*)arg);
  return NULL;
}

static void run_parallel(job_t proto, int64_t n, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (n < 65536) nthreads = 1;
  job_t jobs[256];
  pthread_t th[256];
  int64_t per = (n + nthreads - 1) / nthreads;
  per = (per + 1) & ~(int64_t)1; /* keep Box-Muller pairs inside one job */
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = proto;
    jobs[t].begin = (int64_t)t * per;
    jobs[t].end = jobs[t].begin + per < n ? jobs[t].begin + per : n;
    if (jobs[t].begin >= n) break;
    if (pthread_create(&th[t], NULL, thread_main, &jobs[t]) != 0) {
      run_job(&jobs[t]);
      th[t] = 0;
    }
    started = t + 1;
  }
  for (int t = 0; t < started; ++t)
    if (th[t]) pthread_join(th[t], NULL);
}

/* N(0,1) rounded to bf16 (bit patterns) */
void synth_normal_bf16(uint16_t* out, int64_t n, uint64_t seed, uint64_t stream, int nthreads) {
  job_t j = {0, out, 0, n, seed, stream, 0, 0, 0};
  run_parallel(j, n, nthreads);
}

/* i / 2^denom_log2 with i uniform on [lo, hi], as bf16 bit patterns */
void synth_dyadic_bf16(uint16_t* out, int64_t n, uint64_t seed, uint64_t stream, int64_t lo,
                       int64_t hi, int denom_log2, int nthreads) {
  job_t j = {1, out, 0, n, seed, stream, lo, hi, denom_log2};
  run_parallel(j, n, nthreads);
}

/* i / 2^denom_log2 with i uniform on [lo, hi], as float32 */
void synth_dyadic_f32(float* out, int64_t n, uint64_t seed, uint64_t stream, int64_t lo, int64_t hi,
                      int denom_log2, int nthreads) {
  job_t j = {2, out, 0, n, seed, stream, lo, hi, denom_log2};
  run_parallel(j, n, nthreads);
}

/* i / 2^denom_log2 with i uniform on {-hi..-1, 1..hi}, as float32 */
void synth_signed_nonzero_f32(float* out, int64_t n, uint64_t seed, uint64_t stream, int64_t hi,
                              int denom_log2, int nthreads) {
  job_t j = {3, out, 0, n, seed, stream, 0, hi, denom_log2};
  run_parallel(j, n, nthreads);
}

/*
 * Document packing: each of the B rows of length S is cut into ndocs
 * contiguous documents of length >= 1 that cover the row. The ndocs-1 cut
 * points are distinct uniform draws on [1, S-1], sorted; tokens before the
 * first cut get id 0, and so on. Requires S >= ndocs.
 */
int synth_segments(int32_t* seg, int B, int S, int ndocs, uint64_t seed, uint64_t stream) {
  if (ndocs < 1 || S < ndocs || ndocs > 64) return -1;
  for (int b = 0; b < B; ++b) {
    int cuts[64];
    int nc = 0;
    uint64_t ctr = 0;
    while (nc < ndocs - 1) {
      int c = (int)draw_int(synth_word(seed, stream + (uint64_t)b, ctr++), 1, S - 1);
      int dup = 0;
      for (int i = 0; i < nc; ++i) dup |= (cuts[i] == c);
      if (!dup) cuts[nc++] = c;
    }
    for (int i = 1; i < nc; ++i) /* insertion sort */
      for (int j2 = i; j2 > 0 && cuts[j2 - 1] > cuts[j2]; --j2) {
        int tmp = cuts[j2];
        cuts[j2] = cuts[j2 - 1];
        cuts[j2 - 1] = tmp;
      }
    int d = 0;
    for (int s = 0; s < S; ++s) {
      while (d < nc && s >= cuts[d]) ++d;
      seg[(int64_t)b * S + s] = d;
    }
  }
  return 0;
}

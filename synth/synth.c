/*
 * Seeded synthetic inputs for the NVFP4 linear layer: bf16 weight and
 * activation matrices with the shapes and value distributions of the
 * workloads (Gaussian and Student-t weights, all-zero weight blocks,
 * outlier activation channels).
 *
 * This module is shared by the oracle side (tests) and the device side
 * (tests, bench).  It holds none of the quantization arithmetic: it only
 * draws numbers and rounds them to bf16.
 *
 * Every element is a pure function of (seed, stream, row, col), so any
 * subset of rows can be regenerated on its own and the result does not
 * depend on the number of threads.
 *
 * Generator: splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014) on a counter; 53-bit uniforms in (0,1];
 * Box-Muller for N(0,1); Student-t with nu=4 as Z / sqrt(chi2_4 / 4) with
 * chi2_4 = 2 (E1 + E2), E = -ln U.  Rounding to bf16 is round-to-nearest-even.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static uint64_t splitmix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* Key for one (seed, stream) pair; counters are mixed in afterwards. */
static uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return splitmix64(splitmix64(seed) ^ (stream * 0xD1B54A32D192ED03ull));
}

/* Uniform in (0, 1]: 53 random bits, never exactly zero. */
static double uniform01(uint64_t key, uint64_t ctr) {
  uint64_t r = splitmix64(key ^ splitmix64(ctr));
  return ((double)(r >> 11) + 1.0) * (1.0 / 9007199254740992.0);
}

static const double kTwoPi = 6.283185307179586476925286766559;

static double normal01(uint64_t key, uint64_t ctr) {
  double u1 = uniform01(key, 4 * ctr + 0);
  double u2 = uniform01(key, 4 * ctr + 1);
  return sqrt(-2.0 * log(u1)) * cos(kTwoPi * u2);
}

static double student_t4(uint64_t key, uint64_t ctr) {
  double z = normal01(key, ctr);
  double e1 = -log(uniform01(key, 4 * ctr + 2));
  double e2 = -log(uniform01(key, 4 * ctr + 3));
  return z / sqrt(0.5 * (e1 + e2));
}

/* fp32 -> bf16 bits, round to nearest even (inputs here are finite). */
static uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

enum { DIST_NORMAL = 0, DIST_STUDENT_T4 = 1 };

typedef struct {
  int dist;
  uint64_t seed, stream;
  int64_t row0, rows, cols, ld;
  double scale;
  double zero_block_p;     /* probability that a 16-wide block along cols is zeroed */
  const uint8_t *outlier;  /* [cols] 1 = multiply by outlier_mult, or NULL */
  double outlier_mult;
  uint16_t *out;
  int64_t r_begin, r_end;  /* thread slice, relative to row0 */
} job_t;

static void *run_job(void *arg) {
  job_t *j = (job_t *)arg;
  uint64_t key = stream_key(j->seed, j->stream);
  uint64_t zkey = stream_key(j->seed, j->stream ^ 0x5A5A5A5A5A5A5A5Aull);
  int64_t nblk = j->cols / 16;
  for (int64_t r = j->r_begin; r < j->r_end; ++r) {
    int64_t grow = j->row0 + r;
    uint16_t *dst = j->out + r * j->ld;
    for (int64_t c = 0; c < j->cols; ++c) {
      uint64_t ctr = (uint64_t)grow * (uint64_t)j->cols + (uint64_t)c;
      double v = (j->dist == DIST_STUDENT_T4) ? student_t4(key, ctr) : normal01(key, ctr);
      v *= j->scale;
      if (j->outlier && j->outlier[c]) v *= j->outlier_mult;
      dst[c] = f32_to_bf16((float)v);
    }
    if (j->zero_block_p > 0.0) {
      for (int64_t b = 0; b < nblk; ++b) {
        uint64_t ctr = (uint64_t)grow * (uint64_t)nblk + (uint64_t)b;
        if (uniform01(zkey, ctr) <= j->zero_block_p) memset(dst + 16 * b, 0, 32);
      }
    }
  }
  return NULL;
}

/*
 * Fill rows [row0, row0+rows) of a logical [*, cols] bf16 matrix into
 * out[rows][ld].  dist: 0 = N(0,1), 1 = Student-t(4).  Each value is
 * multiplied by `scale` (and by outlier_mult where outlier[col] != 0)
 * before rounding to bf16.  With zero_block_p > 0 each 16-wide block along
 * cols is set to zero with that probability (cols must then be a multiple
 * of 16).  Returns 0, or -1 on bad arguments.
 */
int synth_fill_bf16(int dist, uint64_t seed, uint64_t stream, int64_t row0, int64_t rows,
                    int64_t cols, int64_t ld, double scale, double zero_block_p,
                    const uint8_t *outlier, double outlier_mult, uint16_t *out,
                    int nthreads) {
  if (rows < 0 || cols < 0 || ld < cols || !out) return -1;
  if (zero_block_p > 0.0 && (cols % 16) != 0) return -1;
  if (dist != DIST_NORMAL && dist != DIST_STUDENT_T4) return -1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (rows < nthreads) nthreads = rows > 0 ? (int)rows : 1;
  job_t jobs[256];
  pthread_t th[256];
  for (int t = 0; t < nthreads; ++t) {
    job_t *j = &jobs[t];
    j->dist = dist; j->seed = seed; j->stream = stream; j->row0 = row0; j->rows = rows;
    j->cols = cols; j->ld = ld; j->scale = scale; j->zero_block_p = zero_block_p;
    j->outlier = outlier; j->outlier_mult = outlier_mult; j->out = out;
    j->r_begin = rows * t / nthreads;
    j->r_end = rows * (t + 1) / nthreads;
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, run_job, &jobs[t]) != 0) break;
    started = t;
  }
  run_job(&jobs[0]);
  for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
  for (int t = started + 1; t < nthreads; ++t) run_job(&jobs[t]);
  return 0;
}

/*
 * Choose exactly `count` distinct channels out of `cols` with a seeded
 * Fisher-Yates shuffle; mask[c] = 1 for the chosen ones.
 */
int synth_pick_channels(uint64_t seed, uint64_t stream, int64_t cols, int64_t count,
                        uint8_t *mask) {
  if (cols < 0 || count < 0 || count > cols || !mask) return -1;
  int64_t *perm = (int64_t *)malloc(sizeof(int64_t) * (size_t)(cols > 0 ? cols : 1));
  if (!perm) return -1;
  for (int64_t i = 0; i < cols; ++i) perm[i] = i;
  uint64_t key = stream_key(seed, stream ^ 0xC3C3C3C3C3C3C3C3ull);
  for (int64_t i = 0; i < count; ++i) {
    uint64_t r = splitmix64(key ^ splitmix64((uint64_t)i));
    int64_t j = i + (int64_t)(r % (uint64_t)(cols - i));
    int64_t tmp = perm[i]; perm[i] = perm[j]; perm[j] = tmp;
  }
  memset(mask, 0, (size_t)cols);
  for (int64_t i = 0; i < count; ++i) mask[perm[i]] = 1;
  free(perm);
  return 0;
}

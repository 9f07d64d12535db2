/*
 * Seeded synthetic inputs, host side.
 *
 * This file draws random numbers and nothing else: it holds none of the MoE
 * layer's arithmetic.  Its twin synth_cuda.cu draws the same numbers on the
 * GPU, bit for bit, from the same definition:
 *
 *   splitmix64      Vigna's published SplitMix64 finaliser (mix of x + golden
 *                   gamma), used here as a counter-based generator.
 *   stream key      key = splitmix64(splitmix64(seed) ^ (tid * GOLDEN)) for
 *                   a tensor id tid.
 *   element i       twelve 24-bit uniforms u_j = splitmix64(key + 12 i + j) >> 40,
 *                   z = (sum_j u_j - 6 * 2^24) / 2^24  (Irwin-Hall with n = 12:
 *                   mean 0, variance 1, exact in double),
 *                   v = z * scale[col]  (one rounded double multiply),
 *                   stored rounded to nearest-even in the storage type.
 *
 * Every step is integer arithmetic or one IEEE double multiply followed by
 * one IEEE rounding, so both sides agree exactly.
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <math.h>

#define SYNTH_GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + SYNTH_GOLDEN;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t synth_splitmix64(uint64_t x) { return splitmix64(x); }

uint64_t synth_stream_key(uint64_t seed, uint64_t tid) {
  return splitmix64(splitmix64(seed) ^ (tid * SYNTH_GOLDEN));
}

/* Standard-normal-like draw of element i (exact double). */
static inline double draw_z(uint64_t key, uint64_t i) {
  uint64_t base = key + 12ULL * i;
  int64_t acc = 0;
  for (int j = 0; j < 12; ++j) acc += (int64_t)(splitmix64(base + (uint64_t)j) >> 40);
  return (double)(acc - 6LL * 16777216LL) * (1.0 / 16777216.0);
}

double synth_draw_z(uint64_t key, uint64_t i) { return draw_z(key, i); }

/* IEEE binary64 -> binary16, round to nearest, ties to even. */
static uint16_t double_to_half_rn(double v) {
  uint16_t sign = signbit(v) ? 0x8000u : 0u;
  double a = fabs(v);
  if (isnan(v)) return (uint16_t)(sign | 0x7E00u);
  if (a >= 65520.0) return (uint16_t)(sign | 0x7C00u); /* rounds to inf */
  if (a < ldexp(1.0, -14)) {
    /* subnormal range: units of 2^-24 */
    double q = a * 16777216.0;            /* exact (power-of-two scale) */
    double r = nearbyint(q);              /* default rounding mode: nearest-even */
    return (uint16_t)(sign | (uint16_t)r); /* r == 1024 becomes the smallest normal */
  }
  int e;
  double m = frexp(a, &e);                /* a = m * 2^e, m in [0.5, 1) */
  /* 11 significant bits: scale mantissa to [1024, 2048) */
  double q = ldexp(m, 11);
  double r = nearbyint(q);
  int ex = e - 1;                          /* a = (r/1024) * 2^ex */
  if (r >= 2048.0) { r = 1024.0; ex += 1; }
  if (ex > 15) return (uint16_t)(sign | 0x7C00u);
  return (uint16_t)(sign | (uint16_t)((ex + 15) << 10) | (uint16_t)((int)r - 1024));
}

uint16_t synth_double_to_half(double v) { return double_to_half_rn(v); }

/*
 * Fill n elements starting at flat index `first` of tensor (seed, tid).
 * scale: per-column scale array (length ncols) or NULL; sigma used when NULL.
 * dtype 0 = float32, 1 = float16 (bits).
 */
void synth_fill(void* out, int dtype, uint64_t first, uint64_t n, uint64_t seed, uint64_t tid,
                double sigma, const double* scale, uint64_t ncols) {
  uint64_t key = synth_stream_key(seed, tid);
#pragma omp parallel for schedule(static)
  for (long long q = 0; q < (long long)n; ++q) {
    uint64_t i = first + (uint64_t)q;
    double s = scale ? scale[i % ncols] : sigma;
    double v = draw_z(key, i) * s;
    if (dtype == 0) ((float*)out)[q] = (float)v;
    else ((uint16_t*)out)[q] = double_to_half_rn(v);
  }
}

/*
 * Fill a sub-block of a row-major [rows, cols] tensor: rows [r0, r0+nr) and all
 * columns, as one contiguous run (a convenience for per-expert slices).
 */
void synth_fill_rows(void* out, int dtype, uint64_t cols, uint64_t r0, uint64_t nr, uint64_t seed,
                     uint64_t tid, double sigma, const double* scale) {
  synth_fill(out, dtype, r0 * cols, nr * cols, seed, tid, sigma, scale, cols);
}

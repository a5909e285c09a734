/*
 * synthgen.c -- seeded synthetic inputs for the MoE verify layer.
 *
 * This module only draws random numbers and stores them in the formats the
 * workload asks for (bf16 activations and weights, uniform 4-bit codes, E4M3
 * block scales, a Zipf log-prior).  It contains none of the layer's
 * arithmetic; both the CUDA path and the CPU oracle receive their inputs from
 * here and from nowhere else.
 *
 * Random numbers: a counter-based SplitMix64 stream.  SplitMix64 (Steele, Lea
 * and Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014)
 * advances a 64-bit state by the golden-ratio increment and mixes it with the
 * variant-13 finalizer; the i-th output of a stream that starts from state s
 * is therefore mix(s + (i + 1) * gamma), which lets any element be generated
 * on its own.  Each tensor gets its own stream whose start state is derived
 * from (seed, layer, tensor id).
 *
 * Plain C11, no platform intrinsics; results are identical on x86-64 and
 * aarch64 except for normal draws, which go through libm's log/cos.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SG_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sg_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* i-th draw (i >= 0) of the stream whose start state is `key`. */
static inline uint64_t sg_draw(uint64_t key, uint64_t i) {
  return sg_mix(key + (i + 1) * SG_GAMMA);
}

uint64_t sg_key(uint64_t seed, uint32_t layer, uint32_t tensor) {
  uint64_t k = sg_mix(seed * SG_GAMMA + 0x5EED5EED12345ULL);
  k = sg_mix(k ^ ((uint64_t)layer * 0xD1B54A32D192ED03ULL));
  k = sg_mix(k ^ ((uint64_t)tensor * 0xABC98388FB8FAC03ULL));
  return k;
}

uint64_t sg_u64(uint64_t key, uint64_t i) { return sg_draw(key, i); }

/* Uniform in [0, 1) with 53 random bits. */
static inline double sg_unit(uint64_t z) { return (double)(z >> 11) * 0x1.0p-53; }

/* Round a double to the nearest bf16 (ties to even), returning the bit
 * pattern.  Handles subnormals and overflow to infinity. */
static uint16_t sg_bf16_rne(double v) {
  if (v != v) return 0x7FC0;
  uint16_t sign = (uint16_t)(signbit(v) ? 0x8000 : 0);
  double a = fabs(v);
  if (a == 0.0) return sign;
  int e;
  (void)frexp(a, &e);                 /* a = m * 2^e, m in [0.5, 1) */
  int q = e - 8;                      /* quantum of an 8-bit significand */
  if (q < -133) q = -133;             /* bf16 subnormal quantum 2^-133 */
  double n = rint(ldexp(a, -q));      /* integer significand, RNE */
  double r = ldexp(n, q);
  if (r >= 0x1.0p128) return (uint16_t)(sign | 0x7F80);
  float f = (float)r;                 /* exact: r has <= 8 significant bits */
  uint32_t bits;
  memcpy(&bits, &f, 4);
  return (uint16_t)(sign | (uint16_t)((bits >> 16) & 0x7FFF));
}

/* Round a positive double to the nearest E4M3 (OCP E4M3FN, bias 7) code,
 * ties to even, saturating at 448.  Used only to quantise the randomly
 * drawn block scales. */
static uint8_t sg_e4m3_rne_pos(double v) {
  if (!(v > 0.0)) return 0;
  if (v >= 448.0) return 0x7E;
  if (v < 0x1.0p-6) {                 /* subnormal range, quantum 2^-9 */
    double n = rint(v * 512.0);       /* n in 0..8; 8 is the smallest normal */
    return (uint8_t)n;
  }
  int e;
  double m = frexp(v, &e);            /* v = m * 2^e, m in [0.5,1) */
  int ex = e - 1;                     /* v = (2m) * 2^ex, 2m in [1,2) */
  double frac = rint((2.0 * m - 1.0) * 8.0);
  if (frac >= 8.0) { frac = 0.0; ex += 1; }
  int field = ex + 7;
  if (field > 15 || (field == 15 && frac > 6.0)) return 0x7E;
  return (uint8_t)((field << 3) | (int)frac);
}

/* Bytes of uniformly random 4-bit codes.  Draw j supplies bytes 8j..8j+7
 * (little-endian), so `byte_off` must be a multiple of 8. */
void sg_fill_codes(uint64_t key, uint64_t byte_off, uint64_t n, uint8_t* out) {
  uint64_t j0 = byte_off >> 3;
  uint64_t nw = (n + 7) >> 3;
  #pragma omp parallel for schedule(static)
  for (int64_t jj = 0; jj < (int64_t)nw; ++jj) {
    uint64_t z = sg_draw(key, j0 + (uint64_t)jj);
    uint64_t base = (uint64_t)jj << 3;
    for (int b = 0; b < 8; ++b) {
      if (base + b < n) out[base + b] = (uint8_t)(z >> (8 * b));
    }
  }
}

/* E4M3 block scales drawn uniformly in [lo, hi] and rounded to E4M3.
 * Element i uses draw (off + i). */
void sg_fill_scales(uint64_t key, uint64_t off, uint64_t n, double lo, double hi,
                    uint8_t* out) {
  #pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) {
    double u = sg_unit(sg_draw(key, off + (uint64_t)i));
    out[i] = sg_e4m3_rne_pos(lo + u * (hi - lo));
  }
}

/* bf16 values mu + sigma * N(0,1) (Box-Muller on draws 2(off+i), 2(off+i)+1). */
void sg_fill_normal_bf16(uint64_t key, uint64_t off, uint64_t n, double mu, double sigma,
                         uint16_t* out) {
  const double two_pi = 6.283185307179586476925286766559;
  #pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) {
    uint64_t c = 2 * (off + (uint64_t)i);
    double u1 = ((double)(sg_draw(key, c) >> 11) + 1.0) * 0x1.0p-53;  /* (0,1] */
    double u2 = sg_unit(sg_draw(key, c + 1));
    double g = sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
    out[i] = sg_bf16_rne(mu + sigma * g);
  }
}

/* Uniform integers in [0, bound) (Lemire-free modulo; bound << 2^64). */
void sg_fill_uniform_int(uint64_t key, uint64_t off, uint64_t n, uint64_t bound,
                         int32_t* out) {
  for (uint64_t i = 0; i < n; ++i) out[i] = (int32_t)(sg_draw(key, off + i) % bound);
}

/* Zipf(s) log-prior over n experts: b[e] = -s * ln(e + 1), as float. */
void sg_zipf_log_prior(double s, int n, float* out) {
  for (int e = 0; e < n; ++e) out[e] = (float)(-s * log((double)e + 1.0));
}

/*
 * Counter-based generator for the synthetic inputs of the head-chunked attention layer.
 *
 * This header is the only code shared by the test oracle and the CUDA path: it makes the
 * seeded inputs (X, Wqkv, Wo, dY) and nothing else.  It holds none of the attention
 * arithmetic.  The same functions compile for the host (gcc, with -ffp-contract=off) and for
 * the device (nvcc; device arithmetic goes through explicitly rounded intrinsics), so element
 * `idx` of tensor `tid` has the same bits wherever it is produced.
 *
 * Definition
 *   key(seed, tid)      = mix64(seed + (tid + 1) * GAMMA)
 *   draw(key, n)        = mix64(key + (n + 1) * GAMMA)      -- output n of a SplitMix64 stream
 *   U(r)                = ((r >> 12) + 0.5) * 2^-52            -- uniform on (0, 1)
 *   normal(seed,tid,i)  : Marsaglia-Bray polar method on draws n = 64*i + 2a, 64*i + 2a + 1,
 *                         attempt a = 0..31: u1 = 2U-1, u2 = 2U-1, s = u1^2 + u2^2,
 *                         accept 0 < s < 1, z = u1 * sqrt(-2 ln(s) / s); after 32 rejected
 *                         attempts (probability ~1e-21) z = 0.
 *   value               = bf16_rne(mean + std * z)  (fp64 arithmetic, one rounding to bf16)
 * mix64 is the SplitMix64 finaliser (Steele, Lea, Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014; constants as published by Vigna).  ln is computed here from the
 * identity ln(m 2^e) = e ln2 + 2 atanh((m-1)/(m+1)) and the atanh power series, in plain
 * IEEE double operations, so no libm result enters the bits.
 */
#ifndef UPIPE_INPUTS_GEN_H
#define UPIPE_INPUTS_GEN_H

#include <stdint.h>

#if defined(__CUDACC__)
#define UG_FN static __host__ __device__ __forceinline__
#else
#define UG_FN static inline
#endif

#if defined(__CUDA_ARCH__)
#define UG_ADD(a, b) __dadd_rn((a), (b))
#define UG_SUB(a, b) __dsub_rn((a), (b))
#define UG_MUL(a, b) __dmul_rn((a), (b))
#define UG_DIV(a, b) __ddiv_rn((a), (b))
#define UG_SQRT(a) __dsqrt_rn((a))
#else
#include <math.h>
#define UG_ADD(a, b) ((a) + (b))
#define UG_SUB(a, b) ((a) - (b))
#define UG_MUL(a, b) ((a) * (b))
#define UG_DIV(a, b) ((a) / (b))
#define UG_SQRT(a) sqrt((a))
#endif

#define UG_GAMMA 0x9E3779B97F4A7C15ULL

UG_FN uint64_t ug_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

UG_FN uint64_t ug_key(uint64_t seed, uint64_t tid) { return ug_mix64(seed + (tid + 1) * UG_GAMMA); }

UG_FN uint64_t ug_draw(uint64_t key, uint64_t n) { return ug_mix64(key + (n + 1) * UG_GAMMA); }

UG_FN double ug_bits_to_double(uint64_t b) {
  union { uint64_t u; double d; } v;
  v.u = b;
  return v.d;
}

UG_FN uint64_t ug_double_to_bits(double d) {
  union { uint64_t u; double d; } v;
  v.d = d;
  return v.u;
}

/* uniform on (0,1): 52 random bits plus one half, times 2^-52; every step is exact */
UG_FN double ug_uniform(uint64_t r) {
  return UG_MUL(UG_ADD((double)(r >> 12), 0.5), 2.220446049250313080847263336181640625e-16);
}

/* natural log of x in (0, 1], plain double arithmetic (see header comment) */
UG_FN double ug_log(double x) {
  uint64_t b = ug_double_to_bits(x);
  int e = (int)((b >> 52) & 0x7FF) - 1022;           /* x = m * 2^e with m in [0.5, 1) */
  double m = ug_bits_to_double((b & 0x000FFFFFFFFFFFFFULL) | 0x3FE0000000000000ULL);
  if (m < 0.70710678118654752440) {                  /* move m into [1/sqrt2, sqrt2) */
    m = UG_MUL(m, 2.0);
    e -= 1;
  }
  double t = UG_DIV(UG_SUB(m, 1.0), UG_ADD(m, 1.0)); /* |t| <= 0.1716 */
  double t2 = UG_MUL(t, t);
  double sum = 0.0;
  /* atanh(t) = t * sum_{k>=0} t^(2k) / (2k+1); 16 terms leave < 1e-26 relative */
  for (int k = 15; k >= 0; --k) sum = UG_ADD(UG_DIV(1.0, (double)(2 * k + 1)), UG_MUL(sum, t2));
  double at = UG_MUL(t, sum);
  return UG_ADD(UG_MUL((double)e, 0.69314718055994530942), UG_MUL(2.0, at));
}

/* round-to-nearest-even of a double to bfloat16 bits; magnitudes below 2^-126 become +-0 */
UG_FN uint16_t ug_bf16_rne(double x) {
  uint64_t b = ug_double_to_bits(x);
  uint16_t sign = (uint16_t)((b >> 48) & 0x8000);
  int ex = (int)((b >> 52) & 0x7FF);
  if (ex == 0x7FF) return (uint16_t)(sign | 0x7FC0);
  int eb = ex - 1023 + 127;
  if (eb <= 0) return sign;
  uint64_t mant = (b & 0x000FFFFFFFFFFFFFULL) | 0x0010000000000000ULL; /* 53 bits */
  uint64_t kept = mant >> 45;                                              /* 8 bits  */
  uint64_t rem = mant & ((1ULL << 45) - 1);
  const uint64_t half = 1ULL << 44;
  if (rem > half || (rem == half && (kept & 1))) kept += 1;
  if (kept == 0x100) {
    kept = 0x80;
    eb += 1;
  }
  if (eb >= 0xFF) return (uint16_t)(sign | 0x7F80);
  return (uint16_t)(sign | (uint16_t)(eb << 7) | (uint16_t)(kept & 0x7F));
}

/* standard normal for element idx of tensor tid */
UG_FN double ug_normal(uint64_t key, uint64_t idx) {
  for (uint64_t a = 0; a < 32; ++a) {
    double u1 = UG_SUB(UG_MUL(2.0, ug_uniform(ug_draw(key, idx * 64 + 2 * a))), 1.0);
    double u2 = UG_SUB(UG_MUL(2.0, ug_uniform(ug_draw(key, idx * 64 + 2 * a + 1))), 1.0);
    double s = UG_ADD(UG_MUL(u1, u1), UG_MUL(u2, u2));
    if (s > 0.0 && s < 1.0) return UG_MUL(u1, UG_SQRT(UG_DIV(UG_MUL(-2.0, ug_log(s)), s)));
  }
  return 0.0;
}

UG_FN uint16_t ug_normal_bf16(uint64_t key, uint64_t idx, double mean, double stddev) {
  return ug_bf16_rne(UG_ADD(mean, UG_MUL(stddev, ug_normal(key, idx))));
}

#endif /* UPIPE_INPUTS_GEN_H */

/*
 * gen.h -- seeded, counter-based synthetic input generator.
 *
 * This header is the ONE piece of code that both the CPU oracle's callers and
 * the CUDA tests/bench use: it makes inputs and holds none of the indexer's
 * arithmetic (no dot products, no ReLU, no weighting, no sigmoid, no select).
 * Every element is a pure function of (seed, tensor tag, two coordinates,
 * element counter), so any sample of a multi-GB tensor can be regenerated on
 * the host bit for bit, and the CUDA fill kernels (gen_cuda.cu) compile these
 * same functions for the device.
 *
 * Bit-exactness across x86 host, Arm host and GPU: only integer operations
 * and single IEEE round-to-nearest float operations are used (one multiply,
 * one fused multiply-add, one division), each spelled out explicitly so that
 * no compiler may contract or reassociate them.
 *
 * Building blocks (published definitions, written out here):
 *   - SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
 *     generators", OOPSLA 2014): output i of a stream with state `key` is the
 *     finaliser applied to key + (i+1)*0x9E3779B97F4A7C15.
 *   - Irwin-Hall approximation of a normal variate: the sum of eight
 *     independent uniform 16-bit integers, centred (an exact integer) and
 *     scaled to the target standard deviation with one fp32 multiply.
 *     Support is +-4.9 sigma; mean and variance are exact.
 *   - OCP 8-bit floating point E4M3 (OCP FP8 spec v1.0): bias 7, 3 mantissa
 *     bits, max finite 448, no infinities, 0x7F/0xFF are NaN.  Encoding here is
 *     round-to-nearest-even with saturation to +-448.
 *   - bfloat16: upper 16 bits of an IEEE binary32, round-to-nearest-even.
 */
#ifndef FM_GEN_H
#define FM_GEN_H

#include <stdint.h>

#ifdef __CUDACC__
#define GEN_FN __host__ __device__ static inline
#else
#define GEN_FN static inline
#endif

#if defined(__CUDA_ARCH__)
#define GEN_FMUL(a, b) __fmul_rn((a), (b))
#define GEN_FDIV(a, b) __fdiv_rn((a), (b))
#define GEN_FMA(a, b, c) __fmaf_rn((a), (b), (c))
#else
#include <math.h>
#define GEN_FMUL(a, b) ((float)(a) * (float)(b))
#define GEN_FDIV(a, b) ((float)(a) / (float)(b))
#define GEN_FMA(a, b, c) fmaf((a), (b), (c))
#endif

/* Tensor tags: each tensor of a workload draws from its own stream. */
enum {
  GEN_TAG_Q = 1,      /* query vectors q[.., h, d]                      */
  GEN_TAG_K = 2,      /* compressed chunk keys K[.., s, d]              */
  GEN_TAG_PLANT = 3,  /* which chunks are planted hot                   */
  GEN_TAG_W = 4,      /* head weights w (prefill workload)              */
  GEN_TAG_PAGES = 5,  /* resident page draw                             */
  GEN_TAG_PLACE = 6,  /* physical placement of pages in the pool        */
  GEN_TAG_MISC = 7
};

#define GEN_GAMMA 0x9E3779B97F4A7C15ull

/* Fp32 scale constants c = sigma / sd(sum of 8 uniform u16), sd = sqrt(8*(65536^2-1)/12). */
#define GEN_C_SIGMA_1 0x1.3988e2p-16f            /* sigma = 1            */
#define GEN_C_SIGMA_INV_SQRT128 0x1.bb67aep-20f  /* sigma = 1/sqrt(128)  */
#define GEN_C_SIGMA_INV8 0x1.3988e2p-19f         /* sigma = 1/8          */

GEN_FN uint64_t gen_fin(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* Output `ctr` of the SplitMix64 stream whose state starts at `key`. */
GEN_FN uint64_t gen_bits(uint64_t key, uint64_t ctr) {
  return gen_fin(key + (ctr + 1ull) * GEN_GAMMA);
}

/* Stream key of tensor `tag` at coordinates (a, b) for run seed `seed`. */
GEN_FN uint64_t gen_key(uint64_t seed, uint64_t tag, uint64_t a, uint64_t b) {
  uint64_t k = gen_bits(seed, tag);
  k = gen_bits(k, a);
  return gen_bits(k, b);
}

/* Centred Irwin-Hall(8) integer in [-262140, 262140] for element `e`. */
GEN_FN int32_t gen_ih8(uint64_t key, uint64_t e) {
  uint64_t h0 = gen_bits(key, 2ull * e);
  uint64_t h1 = gen_bits(key, 2ull * e + 1ull);
  int32_t s = 0;
  for (int j = 0; j < 4; ++j) {
    s += (int32_t)((h0 >> (16 * j)) & 0xFFFFu);
    s += (int32_t)((h1 >> (16 * j)) & 0xFFFFu);
  }
  return s - 262140;
}

/* Approximately normal fp32 value: mean 0, standard deviation sigma(c). */
GEN_FN float gen_normal(uint64_t key, uint64_t e, float c) {
  return GEN_FMUL((float)gen_ih8(key, e), c);
}

GEN_FN uint32_t gen_f32_bits(float f) {
  union { float f; uint32_t u; } v;
  v.f = f;
  return v.u;
}

GEN_FN float gen_bits_f32(uint32_t u) {
  union { float f; uint32_t u; } v;
  v.u = u;
  return v.f;
}

/* fp32 -> bfloat16 bits, round to nearest even (inputs are finite). */
GEN_FN uint16_t gen_bf16_rne(float f) {
  uint32_t u = gen_f32_bits(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* fp32 -> OCP E4M3 code, round to nearest even, saturating to +-448. */
GEN_FN uint8_t gen_e4m3_rne_sat(float f) {
  uint32_t u = gen_f32_bits(f);
  uint8_t sign = (uint8_t)((u >> 24) & 0x80u);
  uint32_t ebits = (u >> 23) & 0xFFu;
  if (ebits == 0xFFu) return (uint8_t)(sign | 0x7Eu); /* inf/nan: saturate (never produced) */
  if (ebits == 0u) return sign;                         /* fp32 zero/subnormal -> zero */
  int32_t E = (int32_t)ebits - 127;                     /* |f| = m24 * 2^(E-23) */
  uint32_t m24 = (u & 0x7FFFFFu) | 0x800000u;
  if (E > 8) return (uint8_t)(sign | 0x7Eu);
  /* quantum: 2^(E-3) for normals (E >= -6), 2^-9 below */
  int32_t qexp = E >= -6 ? E - 3 : -9;
  int32_t shift = 23 - (E - qexp);                      /* m24 >> shift = |f| / 2^qexp */
  uint32_t q;
  if (shift >= 32) {
    q = 0;
  } else {
    uint32_t qt = m24 >> shift;
    uint32_t rem = m24 & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    q = qt + ((rem > half || (rem == half && (qt & 1u))) ? 1u : 0u);
  }
  uint32_t code;
  if (qexp == -9) {
    code = q; /* 0..8; q == 8 is the smallest normal 2^-6 (code 0x08) */
  } else {
    code = ((uint32_t)(E + 7) << 3) + (q - 8u); /* q in [8,16]; 16 carries into the exponent */
  }
  if (code > 0x7Eu) code = 0x7Eu;
  return (uint8_t)(sign | code);
}

/* Bernoulli draw: true with probability thr32 / 2^32. */
GEN_FN int gen_bernoulli(uint64_t key, uint64_t e, uint32_t thr32) {
  return (uint32_t)(gen_bits(key, e) >> 32) < thr32;
}

/* ---------------------------------------------------------------------------
 * Element recipes (each function returns one element; fill loops live in
 * gen_host.c and gen_cuda.cu).
 * ------------------------------------------------------------------------- */

/* bf16 query element q[a][b][h][d], a/b = (request, layer) or (token, 0). */
GEN_FN uint16_t gen_q_bf16(uint64_t seed, uint64_t a, uint64_t b, uint32_t h, uint32_t d,
                           uint32_t head_dim) {
  uint64_t key = gen_key(seed, GEN_TAG_Q, a, b);
  return gen_bf16_rne(gen_normal(key, (uint64_t)h * head_dim + d, GEN_C_SIGMA_1));
}

/* Is chunk s of stream (a, b) planted hot? */
GEN_FN int gen_is_planted(uint64_t seed, uint64_t a, uint64_t b, uint64_t s, uint32_t thr32) {
  return gen_bernoulli(gen_key(seed, GEN_TAG_PLANT, a, b), s, thr32);
}

/* fp32 key element before any rounding: cold N(0, 1/128) noise, plus
 * 3 * hot[d] when the chunk is planted (hot = unit(mean q_0..7), given). */
GEN_FN float gen_k_f32(uint64_t seed, uint64_t a, uint64_t b, uint64_t s, uint32_t d,
                       uint32_t head_dim, int planted, float hot_d) {
  uint64_t key = gen_key(seed, GEN_TAG_K, a, b);
  float noise = gen_normal(key, s * head_dim + d, GEN_C_SIGMA_INV_SQRT128);
  return planted ? GEN_FMA(3.0f, hot_d, noise) : noise;
}

/* Per-chunk fp8 quantisation: scale = max|K_s| / 448 (1 if all zero). */
GEN_FN float gen_fp8_scale(float absmax) {
  return absmax > 0.0f ? GEN_FDIV(absmax, 448.0f) : 1.0f;
}

GEN_FN uint8_t gen_fp8_code(float k, float scale) {
  return gen_e4m3_rne_sat(GEN_FDIV(k, scale));
}

/* N(0, 1/64) fp32 head weight w[t][h] (prefill workload). */
GEN_FN float gen_w_normal(uint64_t seed, uint64_t t, uint32_t h) {
  return gen_normal(gen_key(seed, GEN_TAG_W, t, 0), (uint64_t)h, GEN_C_SIGMA_INV8);
}

#endif /* FM_GEN_H */

/*
 * gen_host.c -- host fill loops for the synthetic workloads (see gen.h).
 *
 * Input generation only: nothing here computes an indexer score.  Built with
 * -ffp-contract=off so that the fp32 operations in gen.h round exactly as
 * written, identically on x86-64, AArch64 and the GPU.
 */
#include "gen.h"

#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define GEN_API __attribute__((visibility("default")))

/* q[a][b][h][d] bf16 for a < A, b < Bc. */
GEN_API void gen_fill_q_bf16(uint64_t seed, int64_t A, int64_t Bc, int32_t n_h, int32_t d,
                             uint16_t* out) {
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t a = 0; a < A; ++a)
    for (int64_t b = 0; b < Bc; ++b) {
      uint16_t* o = out + ((size_t)a * Bc + b) * (size_t)n_h * d;
      for (int32_t h = 0; h < n_h; ++h)
        for (int32_t x = 0; x < d; ++x) o[(size_t)h * d + x] = gen_q_bf16(seed, a, b, h, x, d);
    }
}

/* Planted direction hot[a][b][:] = unit(mean over heads 0..7 of q[a][b][h][:]),
 * in double, rounded once to fp32.  Used only to build planted keys. */
GEN_API void gen_hot_dirs(const uint16_t* q, int64_t A, int64_t Bc, int32_t n_h, int32_t d,
                          float* hot) {
  int32_t nh8 = n_h < 8 ? n_h : 8;
  for (int64_t ab = 0; ab < A * Bc; ++ab) {
    const uint16_t* qa = q + (size_t)ab * n_h * d;
    double m[1024];
    double nn = 0.0;
    for (int32_t x = 0; x < d && x < 1024; ++x) {
      double s = 0.0;
      for (int32_t h = 0; h < nh8; ++h) s += (double)gen_bits_f32((uint32_t)qa[(size_t)h * d + x] << 16);
      m[x] = s / (double)nh8;
    }
    for (int32_t x = 0; x < d && x < 1024; ++x) nn += m[x] * m[x];
    nn = sqrt(nn);
    for (int32_t x = 0; x < d; ++x) hot[(size_t)ab * d + x] = nn > 0.0 ? (float)(m[x] / nn) : 0.0f;
  }
}

/* bf16 keys of stream (a, b) for the listed chunk ids (planted per thr32). */
GEN_API void gen_k_bf16_rows(uint64_t seed, int64_t a, int64_t b, const int64_t* s_list, int64_t n,
                             int32_t d, uint32_t thr32, const float* hot, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    int64_t s = s_list[i];
    int planted = thr32 ? gen_is_planted(seed, a, b, s, thr32) : 0;
    for (int32_t x = 0; x < d; ++x)
      out[(size_t)i * d + x] = gen_bf16_rne(gen_k_f32(seed, a, b, s, x, d, planted, hot ? hot[x] : 0.0f));
  }
}

/* Dense bf16 keys K[a][b][s][d], s < S, for all (a, b). */
GEN_API void gen_fill_k_bf16(uint64_t seed, int64_t A, int64_t Bc, int64_t S, int32_t d,
                             uint32_t thr32, const float* hot, uint16_t* out) {
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t ab = 0; ab < A * Bc; ++ab)
    for (int64_t s = 0; s < S; ++s) {
      int64_t a = ab / Bc, b = ab % Bc;
      int planted = thr32 ? gen_is_planted(seed, a, b, s, thr32) : 0;
      const float* hd = hot ? hot + (size_t)ab * d : NULL;
      uint16_t* o = out + ((size_t)ab * S + s) * d;
      for (int32_t x = 0; x < d; ++x)
        o[x] = gen_bf16_rne(gen_k_f32(seed, a, b, s, x, d, planted, hd ? hd[x] : 0.0f));
    }
}

GEN_API void gen_planted_list(uint64_t seed, int64_t a, int64_t b, int64_t S, uint32_t thr32,
                              uint8_t* out) {
  for (int64_t s = 0; s < S; ++s) out[s] = (uint8_t)gen_is_planted(seed, a, b, s, thr32);
}

/* fp8-e4m3 keys (+ per-chunk fp32 scale) of stream (a, b) for listed chunk ids. */
GEN_API void gen_k_fp8_rows(uint64_t seed, int64_t a, int64_t b, const int64_t* s_list, int64_t n,
                            int32_t d, uint32_t thr32, const float* hot, uint8_t* k8, float* scale) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    int64_t s = s_list[i];
    int planted = thr32 ? gen_is_planted(seed, a, b, s, thr32) : 0;
    float v[1024];
    float amax = 0.0f;
    for (int32_t x = 0; x < d && x < 1024; ++x) {
      v[x] = gen_k_f32(seed, a, b, s, x, d, planted, hot ? hot[x] : 0.0f);
      float av = fabsf(v[x]);
      if (av > amax) amax = av;
    }
    float sc = gen_fp8_scale(amax);
    scale[i] = sc;
    for (int32_t x = 0; x < d && x < 1024; ++x) k8[(size_t)i * d + x] = gen_fp8_code(v[x], sc);
  }
}

/* w[t][h] ~ N(0, 1/64) fp32. */
GEN_API void gen_fill_w_normal(uint64_t seed, int64_t T, int32_t n_h, float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t)
    for (int32_t h = 0; h < n_h; ++h) out[(size_t)t * n_h + h] = gen_w_normal(seed, t, h);
}

/* Uniform integer in [0, n) from a counter stream, by rejection (unbiased). */
static uint32_t gen_uniform_below(uint64_t key, uint64_t* ctr, uint32_t n) {
  uint64_t limit = (0x100000000ull / n) * n;
  for (;;) {
    uint64_t x = gen_bits(key, (*ctr)++) >> 32;
    if (x < limit) return (uint32_t)(x % n);
  }
}

/* R distinct ids from [0, n) (partial Fisher-Yates), in draw order. */
GEN_API int gen_sample_distinct(uint64_t seed, uint64_t tag, int64_t a, int64_t b, int32_t n,
                                int32_t R, int32_t* scratch /*[n]*/, int32_t* out /*[R]*/) {
  if (R > n || n <= 0) return -1;
  uint64_t key = gen_key(seed, tag, a, b);
  uint64_t ctr = 0;
  for (int32_t i = 0; i < n; ++i) scratch[i] = i;
  for (int32_t i = 0; i < R; ++i) {
    uint32_t j = (uint32_t)i + gen_uniform_below(key, &ctr, (uint32_t)(n - i));
    int32_t t = scratch[i];
    scratch[i] = scratch[j];
    scratch[j] = t;
    out[i] = scratch[i];
  }
  return 0;
}

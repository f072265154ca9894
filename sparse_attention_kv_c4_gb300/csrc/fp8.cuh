// fp8.cuh -- building blocks for scoring against E4M3 keys (the compressed_k
// format of the "FlashMemory-DeepSeek-V4" README: 128 E4M3 bytes + an fp32
// scale per chunk): E4M3 conversion, the query split below, the tcgen05
// kind::f8f6f4 MMA and a 3-D TMA load.
//
// Query split.  For head h: q_h = 2^e_h * (t1 + t2) with e_h the power of two that puts
// max|q_h| in (224, 448] (E4M3's top binades), t1 = RNE_e4m3(q_h 2^-e_h) and
// t2 = RNE_e4m3(q_h 2^-e_h - t1).  The pair reproduces every bf16 element
// whose residual stays inside E4M3's range; elements below max|q_h| 2^-13
// lose low bits (at most 2^-10 of the head's scale).  2^e_h is folded into
// the head weight, so the MMA's two dots (t1 . k, t2 . k) summed and scaled
// by w_h 2^e_h give w_h (q_h . k).
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>

#include "fm_common.cuh"

namespace fm {

// fp32 -> E4M3 code, round to nearest even (|f| <= 448 here).
FM_DEV uint32_t e4m3_rne(float f) {
  return (uint32_t)__nv_cvt_float_to_fp8(f, __NV_SATFINITE, __NV_E4M3);
}
FM_DEV float e4m3_value(uint32_t code) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)code, __NV_E4M3);
  return __half2float(__half(h));
}

// 2^n as an fp32 built from its exponent field (-126 <= n <= 127).
FM_DEV float pow2f(int n) { return __int_as_float((n + 127) << 23); }

// One head of the query split.  `raw` holds the lane's four bf16 elements
// 4l .. 4l+3 of the head (the low half of raw.x is element 4l); r1 / r2 are
// the head's t1 / t2 rows (128 bytes each); wq_h receives w_h * 2^e_h.  All
// lanes of the warp call it.
// Scaling by 2^-e_h is a multiply by that power of two built from its
// exponent field: an exact power of two, so the product is x 2^-e_h rounded
// once, as ldexpf gives it, whenever 2^-e_h and 2^e_h are normal floats
// (max|q_h| >= 2^-118).  Heads below that take ldexpf.
FM_DEV void split_head(uint2 raw, float w_h, uint8_t* __restrict__ r1, uint8_t* __restrict__ r2,
                       float* __restrict__ wq_h) {
  const int lane = threadIdx.x & 31;
  const float v[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                      __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
  float amax = 0.f;
  for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fabsf(v[j]));
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  int e = 0;
  bool pow2 = true;  // warp-uniform: amax is the warp's maximum
  if (amax > 0.f && isfinite(amax)) {
    const int be = (int)(__float_as_uint(amax) >> 23);  // biased exponent (amax > 0)
    if (be >= 9) {                                      // e and e + 1 within [-126, 126]
      e = be - 127 - 8;
      if (amax * pow2f(-e) > 448.f) e += 1;
    } else {
      pow2 = false;
      e = ilogbf(amax) - 8;
      if (ldexpf(amax, -e) > 448.f) e += 1;
    }
  }
  const float down = pow2 ? pow2f(-e) : 0.f;
  uint32_t c1w = 0, c2w = 0;
  for (int j = 0; j < 4; ++j) {
    const float s = pow2 ? v[j] * down : ldexpf(v[j], -e);
    const uint32_t c1 = e4m3_rne(s);
    const float r = s - e4m3_value(c1);
    c1w |= c1 << (8 * j);
    c2w |= e4m3_rne(r) << (8 * j);
  }
  reinterpret_cast<uint32_t*>(r1)[lane] = c1w;
  reinterpret_cast<uint32_t*>(r2)[lane] = c2w;
  if (lane == 0) *wq_h = pow2 ? w_h * pow2f(e) : ldexpf(w_h, e);
}

// The lane's slice of head h of a query block (16-byte aligned rows of 128
// bf16 elements), as split_head takes it.
FM_DEV uint2 load_head_slice(const uint16_t* __restrict__ q, int h) {
  return __ldg(reinterpret_cast<const uint2*>(q + (int64_t)h * 128) + (threadIdx.x & 31));
}

// Split the n_heads x 128 bf16 query block q into t1 (rows 0..n_heads-1) and
// t2 (rows n_heads..2 n_heads-1), 128 bytes per row, and write
// wq[h] = w[h] * 2^e_h.  Called by every thread of a CTA of `nthreads`
// threads; warp i takes heads i, i + nthreads/32, ...; lane l takes
// elements 4l .. 4l+3.
FM_DEV void split_query(const uint16_t* __restrict__ q, const float* __restrict__ w, int n_heads, int nthreads,
                        uint8_t* __restrict__ t1, uint8_t* __restrict__ t2, float* __restrict__ wq) {
  const int warp = threadIdx.x >> 5, nw = nthreads / 32;
  // four heads' loads in flight at a time: one memory round trip per four heads
  for (int h0 = warp; h0 < n_heads; h0 += 4 * nw) {
    uint2 raw[4];
    float wv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int h = h0 + u * nw;
      if (h < n_heads) {
        raw[u] = load_head_slice(q, h);
        wv[u] = __ldg(w + h);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int h = h0 + u * nw;
      if (h < n_heads) split_head(raw[u], wv[u], t1 + (int64_t)h * 128, t2 + (int64_t)h * 128, wq + h);
    }
  }
}

// Instruction descriptor, kind::f8f6f4 with E4M3 A/B, fp32 accumulate, K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

FM_DEV void umma_e4m3_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, one M x N x 32 E4M3 step; A's row r is
// TMEM lane r, its 32 E4M3 values four to a 32-bit column, in K order.
FM_DEV void umma_e4m3_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

FM_DEV void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

}  // namespace fm

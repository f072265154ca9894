// gen_cuda.cu -- device fill kernels for the synthetic workloads.
//
// The element recipes are the ones in gen.h, compiled for the device, so a
// device-filled tensor equals the host-filled one bit for bit (checked by the
// generator tests on samples).  Input generation only: no indexer arithmetic.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gen.h"

#define GEN_API extern "C" __attribute__((visibility("default")))

// K[a][b][s][d] bf16 at out + a*stride_a + b*stride_b + s*d + x (element strides).
__global__ void gen_k_bf16_kernel(uint64_t seed, int64_t A, int64_t Bc, int64_t S, int32_t d,
                                  uint32_t thr32, const float* __restrict__ hot,
                                  uint16_t* __restrict__ out, int64_t stride_a, int64_t stride_b) {
  int64_t rows = A * Bc * S;
  for (int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; row < rows;
       row += (int64_t)gridDim.x * (blockDim.x / 32)) {
    int64_t s = row % S;
    int64_t ab = row / S;
    int64_t a = ab / Bc, b = ab % Bc;
    int planted = thr32 ? gen_is_planted(seed, a, b, s, thr32) : 0;
    const float* hd = hot ? hot + ab * d : nullptr;
    uint16_t* o = out + a * stride_a + b * stride_b + s * d;
    for (int32_t x = threadIdx.x % 32; x < d; x += 32)
      o[x] = gen_bf16_rne(gen_k_f32(seed, a, b, s, x, d, planted, hd ? hd[x] : 0.0f));
  }
}

// One warp per chunk of a physical pool page: owner[p] = (a, b, logical page).
__global__ void gen_k_fp8_pool_kernel(uint64_t seed, int64_t P, int32_t d, int32_t page_size,
                                      uint32_t thr32, const int32_t* __restrict__ owner,
                                      const float* __restrict__ hot, int64_t hot_stride_a,
                                      int64_t hot_stride_b, uint8_t* __restrict__ k8,
                                      float* __restrict__ scale) {
  int64_t rows = P * page_size;
  int lane = threadIdx.x % 32;
  for (int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; row < rows;
       row += (int64_t)gridDim.x * (blockDim.x / 32)) {
    int64_t p = row / page_size;
    int64_t o = row % page_size;
    int64_t a = owner[3 * p + 0], b = owner[3 * p + 1], lp = owner[3 * p + 2];
    int64_t s = lp * page_size + o;
    int planted = thr32 ? gen_is_planted(seed, a, b, s, thr32) : 0;
    const float* hd = hot ? hot + a * hot_stride_a + b * hot_stride_b : nullptr;
    float v[8];
    float amax = 0.0f;
    int nv = 0;
    for (int32_t x = lane; x < d && nv < 8; x += 32, ++nv) {
      v[nv] = gen_k_f32(seed, a, b, s, x, d, planted, hd ? hd[x] : 0.0f);
      amax = fmaxf(amax, fabsf(v[nv]));
    }
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    float sc = gen_fp8_scale(amax);
    if (lane == 0) scale[row] = sc;
    nv = 0;
    for (int32_t x = lane; x < d && nv < 8; x += 32, ++nv) k8[row * d + x] = gen_fp8_code(v[nv], sc);
  }
}

// bf16 keys of a pool: one warp per chunk of a physical page, owner[p] =
// (a, b, logical page); cold keys only (the paged recipe plants nothing).
__global__ void gen_k_bf16_pool_kernel(uint64_t seed, int64_t P, int32_t d, int32_t page_size,
                                       const int32_t* __restrict__ owner, uint16_t* __restrict__ out) {
  int64_t rows = P * page_size;
  int lane = threadIdx.x % 32;
  for (int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; row < rows;
       row += (int64_t)gridDim.x * (blockDim.x / 32)) {
    int64_t p = row / page_size;
    int64_t o = row % page_size;
    int64_t a = owner[3 * p + 0], b = owner[3 * p + 1], lp = owner[3 * p + 2];
    int64_t s = lp * page_size + o;
    for (int32_t x = lane; x < d; x += 32) out[row * d + x] = gen_bf16_rne(gen_k_f32(seed, a, b, s, x, d, 0, 0.0f));
  }
}

__global__ void gen_q_bf16_kernel(uint64_t seed, int64_t A, int64_t Bc, int32_t n_h, int32_t d,
                                  uint16_t* __restrict__ out) {
  int64_t n = A * Bc * n_h * d;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    int64_t x = i % d;
    int64_t h = (i / d) % n_h;
    int64_t ab = i / ((int64_t)d * n_h);
    out[i] = gen_q_bf16(seed, ab / Bc, ab % Bc, (uint32_t)h, (uint32_t)x, (uint32_t)d);
  }
}

static int gen_grid(int64_t work, int per_block) {
  int64_t g = (work + per_block - 1) / per_block;
  if (g > 152 * 64) g = 152 * 64;
  if (g < 1) g = 1;
  return (int)g;
}

GEN_API int gen_cuda_fill_k_bf16(uint64_t seed, int64_t A, int64_t Bc, int64_t S, int32_t d,
                                 uint32_t thr32, const float* hot_dev, uint16_t* out_dev,
                                 int64_t stride_a, int64_t stride_b, cudaStream_t stream) {
  gen_k_bf16_kernel<<<gen_grid(A * Bc * S, 8), 256, 0, stream>>>(seed, A, Bc, S, d, thr32, hot_dev,
                                                                   out_dev, stride_a, stride_b);
  return (int)cudaGetLastError();
}

GEN_API int gen_cuda_fill_k_fp8_pool(uint64_t seed, int64_t P, int32_t d, int32_t page_size,
                                     uint32_t thr32, const int32_t* owner_dev, const float* hot_dev,
                                     int64_t hot_stride_a, int64_t hot_stride_b, uint8_t* k8_dev,
                                     float* scale_dev, cudaStream_t stream) {
  if (d > 256) return (int)cudaErrorInvalidValue;
  gen_k_fp8_pool_kernel<<<gen_grid(P * page_size, 8), 256, 0, stream>>>(
      seed, P, d, page_size, thr32, owner_dev, hot_dev, hot_stride_a, hot_stride_b, k8_dev, scale_dev);
  return (int)cudaGetLastError();
}

GEN_API int gen_cuda_fill_k_bf16_pool(uint64_t seed, int64_t P, int32_t d, int32_t page_size,
                                      const int32_t* owner_dev, uint16_t* out_dev, cudaStream_t stream) {
  gen_k_bf16_pool_kernel<<<gen_grid(P * page_size, 8), 256, 0, stream>>>(seed, P, d, page_size, owner_dev, out_dev);
  return (int)cudaGetLastError();
}

GEN_API int gen_cuda_fill_q_bf16(uint64_t seed, int64_t A, int64_t Bc, int32_t n_h, int32_t d,
                                 uint16_t* out_dev, cudaStream_t stream) {
  gen_q_bf16_kernel<<<gen_grid(A * Bc * n_h * d, 256), 256, 0, stream>>>(seed, A, Bc, n_h, d, out_dev);
  return (int)cudaGetLastError();
}

// query_chain.cu -- the query side of a CSA layer's indexer: from a token's
// hidden state to the query heads and head weights the Memory Indexer scores
// with ("FlashMemory-DeepSeek-V4" README, "Retriever architecture" and
// "Hyperparameters"):
//     a = wq_a . h                         Linear dim -> r (no bias)
//     c = RMSNorm(a; q_norm, eps)
//     u = wq_b . c                         Linear r -> n_h * 128
//     q_h = Hadamard(RoPE_yarn(u_h, pos))  per head: rotary on the last 64 of
//                                          128 entries, then the normalised
//                                          Walsh-Hadamard transform
//     w = (w_proj . h) * 128^-1/2 * n_h^-1/2
//
// GB300 mapping.  For a decode batch (tens of tokens) the three projections
// stream 81 MB of bf16 weights per layer and are plain GEMMs: they run in
// cuBLAS (bf16 inputs, fp32 accumulate and fp32 outputs).  The rest are two
// small kernels:
//   rmsnorm_kernel        one CTA per token: sum of squares in fp32, the
//                         normalised row rounded to bf16 (wq_b's input type).
//   rope_hadamard_kernel  one warp per (token, head), four entries per lane:
//                         the rotary angles pos * theta'_i are formed and
//                         reduced in fp64 (positions reach 2^20, where an
//                         fp32 angle would lose whole radians), the
//                         Walsh-Hadamard butterflies run in registers (strides
//                         1 and 2 inside a lane, 4..64 across lanes by
//                         shuffles), and q is written as bf16 (and fp32 when
//                         asked).
#include <cublas_v2.h>
#include <cuda_bf16.h>
#include <math.h>

#include <mutex>

#include "fm_common.cuh"
#include "fm_internal.h"

#define FM_API extern "C" __attribute__((visibility("default")))

namespace fm {
namespace {

constexpr int kHeadDim = 128;
constexpr int kRopeDim = 64;
constexpr int kNormThreads = 256;

__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }

struct RopeCfg {
  double base, factor, orig_len, beta_fast, beta_slow;
};

__global__ void __launch_bounds__(kNormThreads)
    rmsnorm_kernel(const float* __restrict__ a, const uint16_t* __restrict__ g, int r, float eps,
                   uint16_t* __restrict__ out) {
  __shared__ float warp_ss[kNormThreads / 32];
  const int t = blockIdx.x, tid = threadIdx.x;
  const float* row = a + (int64_t)t * r;
  float ss = 0.f;
  for (int i = tid; i < r; i += kNormThreads) ss = fmaf(row[i], row[i], ss);
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((tid & 31) == 0) warp_ss[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < kNormThreads / 32; ++i) tot += warp_ss[i];
  const float inv = rsqrtf(tot / (float)r + eps);
  for (int i = tid; i < r; i += kNormThreads) {
    const float gv = __uint_as_float((uint32_t)g[i] << 16);
    out[(int64_t)t * r + i] = f32_to_bf16_rne(row[i] * inv * gv);
  }
}

// YaRN NTK-by-parts frequency of rotary pair i (see the oracle's reading).
__device__ double yarn_freq(int i, const RopeCfg& c) {
  const double two_pi = 6.283185307179586476925286766559;
  const double theta = pow(c.base, -2.0 * (double)i / (double)kRopeDim);
  const double turns = c.orig_len * theta / two_pi;
  double gamma = (turns - c.beta_slow) / (c.beta_fast - c.beta_slow);
  gamma = gamma < 0.0 ? 0.0 : (gamma > 1.0 ? 1.0 : gamma);
  return (1.0 - gamma) * theta / c.factor + gamma * theta;
}

__global__ void __launch_bounds__(256)
    rope_hadamard_kernel(const float* __restrict__ u, const int64_t* __restrict__ pos, int64_t rows, int n_h,
                         RopeCfg rc, uint16_t* __restrict__ q_out, float* __restrict__ q_out_f32) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);  // (token, head)
  if (row >= rows) return;
  const int64_t t = row / n_h;
  const float4 in = *reinterpret_cast<const float4*>(u + row * kHeadDim + 4 * lane);
  float v[4] = {in.x, in.y, in.z, in.w};
  // rotary on entries 64..127 (lanes 16..31): pairs (2i, 2i+1), i = 2 lane - 32 + {0, 1}
  if (lane >= 16) {
    const double p = (double)pos[t];
    const double two_pi = 6.283185307179586476925286766559;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int i = 2 * lane - 32 + k;
      double a = p * yarn_freq(i, rc);
      a -= two_pi * floor(a / two_pi);
      double s, c;
      sincos(a, &s, &c);
      const float x0 = v[2 * k], x1 = v[2 * k + 1];
      v[2 * k] = (float)((double)x0 * c - (double)x1 * s);
      v[2 * k + 1] = (float)((double)x0 * s + (double)x1 * c);
    }
  }
  // Walsh-Hadamard butterflies: strides 1, 2 inside the lane, 4..64 across lanes
  {
    const float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
    v[0] = a0 + a2;
    v[1] = a1 + a3;
    v[2] = a0 - a2;
    v[3] = a1 - a3;
  }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float other = __shfl_xor_sync(0xffffffffu, v[j], m);
      v[j] = upper ? other - v[j] : v[j] + other;
    }
  }
  const float norm = 0.08838834764831845f;  // 1 / sqrt(128)
#pragma unroll
  for (int j = 0; j < 4; ++j) v[j] *= norm;
  uint2 packed;
  packed.x = (uint32_t)f32_to_bf16_rne(v[0]) | ((uint32_t)f32_to_bf16_rne(v[1]) << 16);
  packed.y = (uint32_t)f32_to_bf16_rne(v[2]) | ((uint32_t)f32_to_bf16_rne(v[3]) << 16);
  *reinterpret_cast<uint2*>(q_out + row * kHeadDim + 4 * lane) = packed;
  if (q_out_f32 != nullptr)
    *reinterpret_cast<float4*>(q_out_f32 + row * kHeadDim + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
}

// One cuBLAS handle per device, created on first use; calls that enqueue on
// it are serialised (the handle's stream is set per call).
std::mutex g_blas_mu;
cublasHandle_t g_blas[64] = {};

fm_status blas_for(int device, cublasHandle_t* out) {
  if (device < 0 || device >= 64) return set_error(FM_ERR_UNSUPPORTED, "query chain: device %d", device);
  if (g_blas[device] == nullptr) {
    cublasHandle_t h = nullptr;
    if (cublasCreate(&h) != CUBLAS_STATUS_SUCCESS) return set_error(FM_ERR_CUDA, "query chain: cublasCreate failed");
    g_blas[device] = h;
  }
  *out = g_blas[device];
  return FM_OK;
}

// Y[T, N] (ldy = N, row-major) = alpha * X[T, K] . W[N, K]^T (both bf16, row-major).
fm_status gemm_xwt(cublasHandle_t h, const uint16_t* X, const uint16_t* W, int T, int N, int K, float alpha,
                   float* Y) {
  const float beta = 0.f;
  const cublasStatus_t st =
      cublasGemmEx(h, CUBLAS_OP_T, CUBLAS_OP_N, N, T, K, &alpha, W, CUDA_R_16BF, K, X, CUDA_R_16BF, K, &beta, Y,
                   CUDA_R_32F, N, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
  if (st != CUBLAS_STATUS_SUCCESS) return set_error(FM_ERR_CUDA, "query chain: cublasGemmEx status %d", (int)st);
  return FM_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t chain_ws_bytes(int T, int r, int n_h) {
  return align256((size_t)T * r * 4) + align256((size_t)T * r * 2) + align256((size_t)T * n_h * kHeadDim * 4);
}

}  // namespace
}  // namespace fm

FM_API size_t fm_query_chain_workspace(int T, int r, int n_h) {
  if (T < 0 || r < 1 || n_h < 1) return 0;
  return fm::chain_ws_bytes(T, r, n_h);
}

FM_API fm_status fm_query_chain(const uint16_t* hidden, const uint16_t* wq_a, const uint16_t* q_norm,
                                const uint16_t* wq_b, const uint16_t* w_proj, const int64_t* pos, int T, int dim,
                                int r, int n_h, int head_dim, int rope_dim, double rope_base, double rope_factor,
                                double rope_orig_len, double rope_beta_fast, double rope_beta_slow, float eps,
                                uint16_t* q_out, float* q_out_f32, float* w_out, void* workspace,
                                size_t workspace_bytes, fm_stream_t stream) {
  using namespace fm;
  if (head_dim != kHeadDim || rope_dim != kRopeDim)
    return set_error(FM_ERR_INVALID_ARG, "fm_query_chain: head_dim=%d rope_dim=%d (need 128, 64)", head_dim,
                     rope_dim);
  if (T < 0 || dim < 8 || r < 8 || n_h < 1 || dim % 8 != 0 || r % 8 != 0 || n_h > 1024)
    return set_error(FM_ERR_INVALID_ARG, "fm_query_chain: bad sizes T=%d dim=%d r=%d n_h=%d (dim, r: multiples of 8)",
                     T, dim, r, n_h);
  if (!(rope_base > 1.0) || !(rope_factor >= 1.0) || !(rope_orig_len > 0.0) || !(rope_beta_fast > rope_beta_slow) ||
      !(eps >= 0.0f))
    return set_error(FM_ERR_INVALID_ARG, "fm_query_chain: bad rotary or norm parameters");
  if (T == 0) return FM_OK;
  if (!hidden || !wq_a || !q_norm || !wq_b || !w_proj || !pos || !q_out || !w_out)
    return set_error(FM_ERR_INVALID_ARG, "fm_query_chain: required pointer is NULL");
  if (!aligned(hidden, 16) || !aligned(wq_a, 16) || !aligned(wq_b, 16) || !aligned(w_proj, 16) ||
      !aligned(q_norm, 2) || !aligned(pos, 8) || !aligned(q_out, 8) || !aligned(w_out, 4) ||
      (q_out_f32 && !aligned(q_out_f32, 16)))
    return set_error(FM_ERR_INVALID_ARG, "fm_query_chain: misaligned pointer");
  const size_t need = chain_ws_bytes(T, r, n_h);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need)
    return set_error(FM_ERR_WORKSPACE, "fm_query_chain: workspace needs %zu bytes, 256-byte aligned", need);
  int sms = 0;
  fm_status st = check_device(&sms);
  if (st != FM_OK) return st;
  int dev = 0;
  cudaGetDevice(&dev);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float* a = static_cast<float*>(workspace);
  uint16_t* c = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + align256((size_t)T * r * 4));
  float* u = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(c) + align256((size_t)T * r * 2));
  {
    std::lock_guard<std::mutex> lock(g_blas_mu);
    cublasHandle_t h = nullptr;
    if ((st = blas_for(dev, &h)) != FM_OK) return st;
    if (cublasSetStream(h, s) != CUBLAS_STATUS_SUCCESS) return set_error(FM_ERR_CUDA, "fm_query_chain: cublasSetStream");
    if ((st = gemm_xwt(h, hidden, wq_a, T, r, dim, 1.0f, a)) != FM_OK) return st;
    // head weights: w_proj . h scaled by head_dim^-1/2 n_h^-1/2
    const float ws = (float)(1.0 / sqrt((double)head_dim) / sqrt((double)n_h));
    if ((st = gemm_xwt(h, hidden, w_proj, T, n_h, dim, ws, w_out)) != FM_OK) return st;
    rmsnorm_kernel<<<T, kNormThreads, 0, s>>>(a, q_norm, r, eps, c);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "fm_query_chain: rmsnorm launch: %s", cudaGetErrorString(e));
    if ((st = gemm_xwt(h, c, wq_b, T, n_h * kHeadDim, r, 1.0f, u)) != FM_OK) return st;
  }
  RopeCfg rc{rope_base, rope_factor, rope_orig_len, rope_beta_fast, rope_beta_slow};
  const int64_t rows = (int64_t)T * n_h;
  rope_hadamard_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(u, pos, rows, n_h, rc, q_out, q_out_f32);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "fm_query_chain: rope launch: %s", cudaGetErrorString(e));
  return FM_OK;
}

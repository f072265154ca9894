// topk.cu -- standalone exact top-k over rows of fp32 scores (one CTA per row).
#include "fm_internal.h"
#include "topk.cuh"

namespace fm {
namespace {

constexpr int kTopkThreads = 512;

struct IdentityMap {
  FM_DEV int32_t operator()(int i) const { return i; }
};

// Candidate i of a paged row is chunk page_ids[i / 64] * 64 + i % 64.
struct PageMap {
  const int32_t* ids;
  FM_DEV int32_t operator()(int i) const { return __ldg(ids + (i >> 6)) * 64 + (i & 63); }
};

__global__ void __launch_bounds__(kTopkThreads)
    topk_rows_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ n_valid, int n, int k,
                     const int32_t* __restrict__ page_ids, int64_t page_ld, int32_t* __restrict__ idx_out,
                     float* __restrict__ score_out) {
  extern __shared__ uint8_t topk_smem_raw[];
  TopkFastSmem<kTopkThreads>& sm = *reinterpret_cast<TopkFastSmem<kTopkThreads>*>(topk_smem_raw);
  const int64_t r = blockIdx.x;
  int nr = n;
  if (n_valid != nullptr) {
    const int v = __ldg(n_valid + r);
    nr = v < 0 ? 0 : (v > n ? n : v);
  }
  const float* row = scores + r * ld;
  int32_t* io = idx_out + r * k;
  float* so = score_out != nullptr ? score_out + r * k : nullptr;
  if (page_ids != nullptr)
    block_topk<kTopkThreads>(row, nr, k, PageMap{page_ids + r * page_ld}, io, so, sm);
  else
    block_topk<kTopkThreads>(row, nr, k, IdentityMap{}, io, so, sm);
}

}  // namespace

fm_status launch_topk_rows(const float* scores, int64_t ld, const int32_t* n_valid, int rows, int n, int k,
                           const int32_t* page_ids, int64_t page_ld, int32_t* idx_out, float* score_out,
                           cudaStream_t stream) {
  if (rows == 0) return FM_OK;
  const int smem = (int)sizeof(TopkFastSmem<kTopkThreads>);
  cudaError_t e0 = cudaFuncSetAttribute(topk_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e0 != cudaSuccess) return set_error(FM_ERR_CUDA, "topk: cudaFuncSetAttribute: %s", cudaGetErrorString(e0));
  topk_rows_kernel<<<rows, kTopkThreads, smem, stream>>>(scores, ld, n_valid, n, k, page_ids, page_ld, idx_out,
                                                       score_out);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "topk: launch: %s", cudaGetErrorString(e));
  return FM_OK;
}

}  // namespace fm

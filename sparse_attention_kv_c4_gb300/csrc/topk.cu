// topk.cu -- exact top-k over rows of fp32 scores: one CTA of 256 threads
// per row runs block_topk (topk.cuh): sample threshold, one filtering pass
// from HBM with eight float4 loads in flight per thread, exact select among
// the candidates, ids in index order through a bitmap.
#include "fm_internal.h"
#include "topk.cuh"

namespace fm {
namespace {

constexpr int kTopkThreads = 256;

struct IdentityMap {
  FM_DEV int32_t operator()(int i) const { return i; }
};

// Candidate i of a paged row is chunk page_ids[i / 64] * 64 + i % 64.
struct PageMap {
  const int32_t* ids;
  FM_DEV int32_t operator()(int i) const { return __ldg(ids + (i >> 6)) * 64 + (i & 63); }
};

FM_DEV int row_len(const int32_t* __restrict__ n_valid, int64_t r, int n) {
  if (n_valid == nullptr) return n;
  const int v = __ldg(n_valid + r);
  return v < 0 ? 0 : (v > n ? n : v);
}

__global__ void __launch_bounds__(kTopkThreads)
    topk_rows_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ n_valid, int n, int k,
                     const int32_t* __restrict__ page_ids, int64_t page_ld, int32_t* __restrict__ idx_out,
                     float* __restrict__ score_out) {
  extern __shared__ uint8_t topk_smem_raw[];
  TopkFastSmem<kTopkThreads>& sm = *reinterpret_cast<TopkFastSmem<kTopkThreads>*>(topk_smem_raw);
  const int64_t r = blockIdx.x;
  const int nr = row_len(n_valid, r, n);
  const float* row = scores + r * ld;
  int32_t* io = idx_out + r * k;
  float* so = score_out != nullptr ? score_out + r * k : nullptr;
  if (page_ids != nullptr)
    block_topk<kTopkThreads>(row, nr, k, PageMap{page_ids + r * page_ld}, io, so, sm);
  else
    block_topk<kTopkThreads>(row, nr, k, IdentityMap{}, io, so, sm);
}


}  // namespace

size_t topk_workspace_bytes(int rows, int n) {
  (void)rows;
  (void)n;
  return 0;
}

fm_status launch_topk_rows(const float* scores, int64_t ld, const int32_t* n_valid, int rows, int n, int k,
                           const int32_t* page_ids, int64_t page_ld, int32_t* idx_out, float* score_out,
                           cudaStream_t stream) {
  if (rows == 0) return FM_OK;
  const int smem = (int)sizeof(TopkFastSmem<kTopkThreads>);
  cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "topk: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  topk_rows_kernel<<<rows, kTopkThreads, smem, stream>>>(scores, ld, n_valid, n, k, page_ids, page_ld, idx_out,
                                                       score_out);
  e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "topk: launch: %s", cudaGetErrorString(e));
  return FM_OK;
}

}  // namespace fm

// topk.cu -- exact top-k over rows of fp32 scores: one CTA of 256 threads
// per row runs block_topk (topk.cuh): sample threshold, one filtering pass
// from HBM with eight float4 loads in flight per thread, exact select among
// the candidates, ids in index order through a bitmap.
#include "fm_internal.h"
#include "topk.cuh"

namespace fm {
namespace {

constexpr int kTopkThreads = 256;

// Programmatic dependent launch: a top-k kernel may start while the kernel
// before it on the stream (the scorer that wrote its rows) finishes; every
// thread waits for that kernel's completion, and its memory, before reading.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename Kernel, typename... Args>
cudaError_t launch_pdl(Kernel kernel, int grid, int block, int smem, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)block);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

struct IdentityMap {
  FM_DEV int32_t operator()(int i) const { return i; }
};

// Candidate i of a paged row is chunk page_ids[i / 64] * 64 + i % 64.
struct PageMap {
  static constexpr bool kPageIds = true;  // the emit may stage ids[] in shared memory
  const int32_t* ids;
  FM_DEV int32_t operator()(int i) const { return __ldg(ids + (i >> 6)) * 64 + (i & 63); }
};

// A paged row compacted to its resident chunks: page j holds candidates
// prefix[j] .. prefix[j+1]-1, which are the set bits of mask[j] in increasing
// order.  Candidate i is found by a binary search for the last page whose
// prefix is <= i (an empty page shares its prefix with the next page, so the
// last such page holds i) and the (i - prefix[j])-th set bit of its mask.
struct MaskedPageMap {
  const int32_t* ids;
  const int32_t* prefix;
  const unsigned long long* mask;
  int n_pages;
  FM_DEV int32_t operator()(int i) const {
    int lo = 0, hi = n_pages - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(prefix + mid) <= i) lo = mid;
      else hi = mid - 1;
    }
    const unsigned long long m = __ldg(mask + lo);
    int r = i - __ldg(prefix + lo);
    const uint32_t m_lo = (uint32_t)m, m_hi = (uint32_t)(m >> 32);
    const int c_lo = __popc(m_lo);
    const int o = r < c_lo ? (int)__fns(m_lo, 0, r + 1) : 32 + (int)__fns(m_hi, 0, r - c_lo + 1);
    return __ldg(ids + lo) * 64 + o;
  }
};

FM_DEV int row_len(const int32_t* __restrict__ n_valid, int64_t r, int n) {
  if (n_valid == nullptr) return n;
  const int v = __ldg(n_valid + r);
  return v < 0 ? 0 : (v > n ? n : v);
}

// kMap: 0 = candidate index, 1 = paged rows (PageMap), 2 = paged rows
// compacted to resident chunks (MaskedPageMap); one instantiation each so the
// id maps do not share a register allocation.  kShort: rows of at most
// kTopkShortN scores (every row up to a 1M-token history) take a smaller
// candidate list (kTopkCapShort), which lets five CTAs share an SM instead of
// four (760 rows per wave on 152 SMs, so the 630 queries of a 1M-context
// decode batch run in one wave); a list that overflows falls back to the
// exact radix path, so the cap affects only speed.
template <int kMap, bool kShort>
__global__ void __launch_bounds__(kTopkThreads, kShort ? 5 : 4)
    topk_rows_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ n_valid, int n, int k,
                     const int32_t* __restrict__ page_ids, int64_t page_ld, const int32_t* __restrict__ page_prefix,
                     const unsigned long long* __restrict__ page_mask, int32_t* __restrict__ idx_out,
                     float* __restrict__ score_out) {
  constexpr int kCap = kShort ? kTopkCapShort : kTopkCap;
  grid_dep_wait();
  extern __shared__ uint8_t topk_smem_raw[];
  TopkFastSmem<kTopkThreads, kCap>& sm = *reinterpret_cast<TopkFastSmem<kTopkThreads, kCap>*>(topk_smem_raw);
  const int64_t r = blockIdx.x;
  const int nr = row_len(n_valid, r, n);
  const float* row = scores + r * ld;
  int32_t* io = idx_out + r * k;
  float* so = score_out != nullptr ? score_out + r * k : nullptr;
  if constexpr (kMap == 2) {
    // all page_ld pages are searched: pages past the listed ones are empty
    const MaskedPageMap map{page_ids + r * page_ld, page_prefix + r * (page_ld + 1), page_mask + r * page_ld,
                            (int)page_ld};
    block_topk<kTopkThreads, kCap>(row, nr, k, map, io, so, sm);
  } else if constexpr (kMap == 1) {
    block_topk<kTopkThreads, kCap>(row, nr, k, PageMap{page_ids + r * page_ld}, io, so, sm);
  } else {
    block_topk<kTopkThreads, kCap>(row, nr, k, IdentityMap{}, io, so, sm);
  }
}


// Rows of at most kTopkTinyN scores with k <= 512 (a 512K-context decode
// batch: 1260 queries x 192 pages = 12288 chunks each): 128 threads, a
// 1536-entry candidate list, a 1024-score sample and a bitmap for 16384 ids
// (24 KB of shared memory), so nine CTAs share an SM and a 1260-query batch
// runs in one wave rather than two.  The sample aims at 1024 candidates; a
// row where it misses is re-aimed once (block_topk) before the exact path.
constexpr int kTopkTinyThreads = 128;
constexpr int kTopkTinyN = 16384;
constexpr int kTopkTinyK = 512;
constexpr int kTopkTinyCap = 1536;
constexpr int kTopkTinyRuns = 16;
using TinySmem = TopkFastSmem<kTopkTinyThreads, kTopkTinyCap, kTopkTinyRuns, kTopkTinyN>;

template <int kMap>
__global__ void __launch_bounds__(kTopkTinyThreads, 9)
    topk_rows_tiny_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ n_valid, int n,
                          int k, const int32_t* __restrict__ page_ids, int64_t page_ld,
                          const int32_t* __restrict__ page_prefix, const unsigned long long* __restrict__ page_mask,
                          int32_t* __restrict__ idx_out, float* __restrict__ score_out) {
  grid_dep_wait();
  extern __shared__ uint8_t topk_smem_raw[];
  TinySmem& sm = *reinterpret_cast<TinySmem*>(topk_smem_raw);
  const int64_t r = blockIdx.x;
  const int nr = row_len(n_valid, r, n);
  const float* row = scores + r * ld;
  int32_t* io = idx_out + r * k;
  float* so = score_out != nullptr ? score_out + r * k : nullptr;
  if constexpr (kMap == 2) {
    const MaskedPageMap map{page_ids + r * page_ld, page_prefix + r * (page_ld + 1), page_mask + r * page_ld,
                            (int)page_ld};
    block_topk<kTopkTinyThreads, kTopkTinyCap, MaskedPageMap, kTopkTinyRuns, kTopkTinyN>(row, nr, k, map, io, so, sm);
  } else if constexpr (kMap == 1) {
    block_topk<kTopkTinyThreads, kTopkTinyCap, PageMap, kTopkTinyRuns, kTopkTinyN>(
        row, nr, k, PageMap{page_ids + r * page_ld}, io, so, sm);
  } else {
    block_topk<kTopkTinyThreads, kTopkTinyCap, IdentityMap, kTopkTinyRuns, kTopkTinyN>(row, nr, k, IdentityMap{}, io,
                                                                                        so, sm);
  }
}

// Prefill rows with segment entries (block_topk_segmax): read the entries,
// then only the segments that can hold a top-k score.  Same shared memory and
// occupancy as the short-row kernel (five CTAs per SM), whose select it falls
// back on for a row it cannot prune.
constexpr int kSegMaxN = kTopkBitmapN;  // rows of at most this many scores
using SegSmem = TopkFastSmem<kTopkThreads, kTopkCapShort>;

__global__ void __launch_bounds__(kTopkThreads, 5)
    topk_rows_segmax_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ n_valid,
                            const int32_t* __restrict__ segmax, int64_t seg_ld, int n, int k,
                            int32_t* __restrict__ idx_out, float* __restrict__ score_out) {
  grid_dep_wait();
  extern __shared__ uint8_t topk_smem_raw[];
  SegSmem& sm = *reinterpret_cast<SegSmem*>(topk_smem_raw);
  const int64_t r = blockIdx.x;
  const int nr = row_len(n_valid, r, n);
  block_topk_segmax<kTopkThreads, kTopkCapShort>(scores + r * ld, nr, k, segmax + r * seg_ld, ld % 4 == 0,
                                                 IdentityMap{}, idx_out + r * k,
                                                 score_out != nullptr ? score_out + r * k : nullptr, sm);
}
}  // namespace

size_t topk_workspace_bytes(int rows, int n) {
  (void)rows;
  (void)n;
  return 0;
}

fm_status launch_topk_rows(const float* scores, int64_t ld, const int32_t* n_valid, int rows, int n, int k,
                           const int32_t* page_ids, int64_t page_ld, const int32_t* page_prefix,
                           const unsigned long long* page_mask, int32_t* idx_out, float* score_out,
                           cudaStream_t stream) {
  if (rows == 0) return FM_OK;
  if (n <= kTopkTinyN && k <= kTopkTinyK && rows > 5 * 152) {
    // more rows than one wave of 256-thread CTAs (five per SM on GB300's 152
    // SMs): the 128-thread kernel runs nine per SM
    auto* kernel = page_mask != nullptr ? topk_rows_tiny_kernel<2>
                                        : (page_ids != nullptr ? topk_rows_tiny_kernel<1> : topk_rows_tiny_kernel<0>);
    const int smem = (int)sizeof(TinySmem);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "topk: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    e = launch_pdl(kernel, rows, kTopkTinyThreads, smem, stream, scores, ld, n_valid, n, k, page_ids, page_ld,
                   page_prefix, page_mask, idx_out, score_out);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "topk: launch: %s", cudaGetErrorString(e));
    return FM_OK;
  }
  const bool short_rows = n <= kTopkShortN;
  const int smem = short_rows ? (int)sizeof(TopkFastSmem<kTopkThreads, kTopkCapShort>)
                              : (int)sizeof(TopkFastSmem<kTopkThreads, kTopkCap>);
  void (*kernel)(const float*, int64_t, const int32_t*, int, int, const int32_t*, int64_t, const int32_t*,
                 const unsigned long long*, int32_t*, float*);
  if (short_rows)
    kernel = page_mask != nullptr ? topk_rows_kernel<2, true>
                                  : (page_ids != nullptr ? topk_rows_kernel<1, true> : topk_rows_kernel<0, true>);
  else
    kernel = page_mask != nullptr ? topk_rows_kernel<2, false>
                                  : (page_ids != nullptr ? topk_rows_kernel<1, false> : topk_rows_kernel<0, false>);
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "topk: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  // the whole shared-memory carveout, so that the occupancy shared memory
  // allows (four or five CTAs) is not cut by a smaller L1 split
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "topk: carveout: %s", cudaGetErrorString(e));
  e = launch_pdl(kernel, rows, kTopkThreads, smem, stream, scores, ld, n_valid, n, k, page_ids, page_ld, page_prefix,
                 page_mask, idx_out, score_out);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "topk: launch: %s", cudaGetErrorString(e));
  return FM_OK;
}

fm_status launch_topk_rows_segmax(const float* scores, int64_t ld, const int32_t* n_valid, const int32_t* segmax,
                                  int64_t seg_ld, int rows, int n, int k, int32_t* idx_out, float* score_out,
                                  cudaStream_t stream) {
  if (rows == 0) return FM_OK;
  // rows too short to prune (fewer than 2k segments) or longer than the
  // short-row kernel takes: the plain select
  if ((n + 31) / 32 < 2 * k || n > kSegMaxN)
    return launch_topk_rows(scores, ld, n_valid, rows, n, k, nullptr, 0, nullptr, nullptr, idx_out, score_out,
                            stream);
  const int smem = (int)sizeof(SegSmem);
  cudaError_t e = cudaFuncSetAttribute(topk_rows_segmax_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(topk_rows_segmax_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "topk segmax: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  e = launch_pdl(topk_rows_segmax_kernel, rows, kTopkThreads, smem, stream, scores, ld, n_valid, segmax, seg_ld, n, k,
                 idx_out, score_out);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "topk segmax: launch: %s", cudaGetErrorString(e));
  return FM_OK;
}

}  // namespace fm

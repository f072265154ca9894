// recall.cu -- page recall: the densest resident pages of each request.
//
// Computes ("FlashMemory-DeepSeek-V4" README, "Two-level recall algorithm",
// Level 1: resident_set = threshold mask + recency tail + attention sink;
// "Page-recall": 64-chunk pages; KMAX note under "Reference performance": each
// request recalls the KMAX densest pages, 256K -> 96, 512K -> 192, 1M -> 384):
//     resident(s) = mask bit s  or  s < sink  or  s >= S - recent   (s < S)
//     density(p)  = number of resident chunks in [64p, 64p + 64)
// and the kmax pages of highest density (density > 0; ties to the lower page
// id), written in ascending page order and padded with -1.  This turns the
// Memory-Indexer bitmask (fm_memindex_score_mask) into the page table the
// native paged scorer (fm_native_topk_paged) reads.
//
// GB300 mapping.  The input is tiny (one bit per chunk: 32 KB per request at
// 1M context) and the selection is over small integers, so this is one CTA per
// request and no tensor work: a 65-bin density histogram in shared memory
// gives the cut density D and how many pages of density D are taken; a
// block-wide prefix sum of (pages above D, pages at D) over contiguous page
// ranges gives every thread its output slots, so the output is in page order
// with ties resolved to the lower id without any sort.
#include "fm_common.cuh"
#include "fm_internal.h"

#define FM_API extern "C" __attribute__((visibility("default")))

namespace fm {
namespace {

constexpr int kRecallThreads = 1024;  // four 64-chunk pages per thread at 1M context
constexpr int kPageChunks = 64;

// Bits [lo, hi) of the 64-chunk window starting at chunk a, as a mask.
FM_DEV uint64_t range_bits(int64_t a, int64_t lo, int64_t hi) {
  const int64_t l = (lo > a ? lo : a) - a;
  const int64_t h = (hi < a + 64 ? hi : a + 64) - a;
  if (h <= l) return 0ull;
  const uint64_t width = h - l == 64 ? ~0ull : ((1ull << (h - l)) - 1ull);
  return width << l;
}

FM_DEV int page_density(const uint32_t* __restrict__ row, int64_t words, int64_t p, int64_t S, int64_t sink,
                        int64_t recent) {
  const int64_t a = p * kPageChunks;
  const uint64_t w0 = 2 * p < words ? __ldg(row + 2 * p) : 0u;
  const uint64_t w1 = 2 * p + 1 < words ? __ldg(row + 2 * p + 1) : 0u;
  uint64_t m = w0 | (w1 << 32);
  m |= range_bits(a, 0, sink) | range_bits(a, S - recent, S);
  m &= range_bits(a, 0, S);  // bits past S never count
  return __popcll(m);
}

struct RecallSmem {
  uint32_t hist[kPageChunks + 1];
  uint32_t warp_tot[kRecallThreads / 32];
  int cut;          // cut density D (>= 1)
  uint32_t above;   // pages with density > D
  uint32_t take_eq; // pages of density D that are taken (lowest ids)
};

// Exclusive block prefix sum of 32-bit values (all threads call it).
FM_DEV uint32_t excl_scan(uint32_t v, uint32_t* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t t = lane < kRecallThreads / 32 ? warp_tot[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < kRecallThreads / 32) warp_tot[lane] = t;
  }
  __syncthreads();
  const uint32_t before = warp == 0 ? 0u : warp_tot[warp - 1];
  __syncthreads();
  return before + x - v;
}

__global__ void __launch_bounds__(kRecallThreads)
    page_recall_kernel(const uint32_t* __restrict__ mask, int64_t S, int64_t sink, int64_t recent, int kmax,
                       int32_t* __restrict__ pages_out, int32_t* __restrict__ density_out,
                       int32_t* __restrict__ n_out) {
  __shared__ RecallSmem sm;
  const int tid = threadIdx.x;
  const int64_t b = blockIdx.x;
  const int64_t words = (S + 31) / 32;
  const int64_t n_pages = (S + kPageChunks - 1) / kPageChunks;
  const uint32_t* row = mask + b * words;
  int32_t* po = pages_out + b * kmax;
  int32_t* dn = density_out != nullptr ? density_out + b * kmax : nullptr;

  // ---- 1. density histogram (coalesced: consecutive threads, consecutive pages)
  for (int i = tid; i <= kPageChunks; i += kRecallThreads) sm.hist[i] = 0u;
  __syncthreads();
  for (int64_t p = tid; p < n_pages; p += kRecallThreads)
    atomicAdd(&sm.hist[page_density(row, words, p, S, sink, recent)], 1u);
  __syncthreads();
  if (tid == 0) {
    // Walk densities from 64 down: the cut D is the first density at which
    // the pages so far reach kmax; pages above D are all taken and the
    // lowest-id kmax - above pages of density D fill up.  If every non-empty
    // page fits, all of them are taken (D = 1, every page of density 1).
    uint32_t above = 0;  // pages of density > d
    int cut = 0;
    uint32_t take_eq = 0;
    for (int d = kPageChunks; d >= 1; --d) {
      const uint32_t c = sm.hist[d];
      if (above + c >= (uint32_t)kmax) {
        cut = d;
        take_eq = (uint32_t)kmax - above;
        break;
      }
      above += c;
    }
    if (cut == 0) {
      cut = 1;
      take_eq = sm.hist[1];
      above -= sm.hist[1];
    }
    sm.cut = cut;
    sm.above = above;
    sm.take_eq = take_eq;
  }
  __syncthreads();
  const int cut = sm.cut;
  const uint32_t take_eq = sm.take_eq;
  const uint32_t n_taken = sm.above + take_eq;

  // ---- 2. ordered emission over contiguous page ranges
  const int64_t per = (n_pages + kRecallThreads - 1) / kRecallThreads;
  const int64_t p0 = tid * per;
  const int64_t p1 = p0 + per < n_pages ? p0 + per : n_pages;
  uint32_t gt = 0, eq = 0;
  for (int64_t p = p0; p < p1; ++p) {
    const int d = page_density(row, words, p, S, sink, recent);
    gt += d > cut;
    eq += d == cut;
  }
  const uint32_t gt_before = excl_scan(gt, sm.warp_tot);
  const uint32_t eq_before = excl_scan(eq, sm.warp_tot);
  uint32_t g = gt_before, e = eq_before;
  for (int64_t p = p0; p < p1; ++p) {
    const int d = page_density(row, words, p, S, sink, recent);
    bool take = false;
    uint32_t pos = 0;
    if (d > cut) {
      take = true;
      pos = g + (e < take_eq ? e : take_eq);
      ++g;
    } else if (d == cut) {
      if (e < take_eq) {
        take = true;
        pos = g + e;
      }
      ++e;
    }
    if (take) {
      po[pos] = (int32_t)p;
      if (dn) dn[pos] = d;
    }
  }
  for (uint32_t i = n_taken + tid; i < (uint32_t)kmax; i += kRecallThreads) {
    po[i] = -1;
    if (dn) dn[i] = -1;
  }
  if (tid == 0 && n_out != nullptr) n_out[b] = (int32_t)n_taken;
}

}  // namespace
}  // namespace fm

FM_API fm_status fm_page_recall(const uint32_t* mask, int B, int64_t S, int64_t sink, int64_t recent, int kmax,
                                int32_t* pages_out, int32_t* density_out, int32_t* n_out, fm_stream_t stream) {
  using namespace fm;
  if (B < 0 || S < 0 || S >= (int64_t(1) << 31) || sink < 0 || recent < 0 || kmax < 1 || kmax > 65536)
    return set_error(FM_ERR_INVALID_ARG, "fm_page_recall: bad sizes B=%d S=%lld sink=%lld recent=%lld kmax=%d", B,
                     (long long)S, (long long)sink, (long long)recent, kmax);
  if (B == 0) return FM_OK;
  if (!pages_out || (S > 0 && !mask))
    return set_error(FM_ERR_INVALID_ARG, "fm_page_recall: mask and pages_out must be non-NULL");
  if (!aligned(mask, 4) || !aligned(pages_out, 4) || (density_out && !aligned(density_out, 4)) ||
      (n_out && !aligned(n_out, 4)))
    return set_error(FM_ERR_INVALID_ARG, "fm_page_recall: pointers need 4-byte alignment");
  int sms = 0;
  fm_status st = check_device(&sms);
  if (st != FM_OK) return st;
  const int64_t sink_c = sink < S ? sink : S, recent_c = recent < S ? recent : S;
  page_recall_kernel<<<B, kRecallThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      mask, S, sink_c, recent_c, kmax, pages_out, density_out, n_out);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "page recall: launch: %s", cudaGetErrorString(e));
  return FM_OK;
}

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
// request and no tensor work: each thread computes the densities of its
// contiguous run of pages once (two popcounts per page away from the sink,
// the recency tail and a partial last page) and keeps them in registers; a
// 65-bin density histogram in shared memory gives the cut density D (one warp
// finds it from suffix sums) and how many pages of density D are taken; one
// block-wide prefix sum of (pages above D, pages at D) gives every thread its
// output slots, so the output is in page order with ties resolved to the
// lower id without any sort.
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
  unsigned long long warp_tot64[kRecallThreads / 32];
  int cut;          // cut density D (>= 1)
  uint32_t above;   // pages with density > D
  uint32_t take_eq; // pages of density D that are taken (lowest ids)
};

// Exclusive block prefix sum of 64-bit values (all threads call it): two
// 32-bit counts side by side, neither carrying into the other while each
// stays below 2^32.
FM_DEV unsigned long long excl_scan64(unsigned long long v, unsigned long long* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    unsigned long long t = lane < kRecallThreads / 32 ? warp_tot[lane] : 0ull;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < kRecallThreads / 32) warp_tot[lane] = t;
  }
  __syncthreads();
  const unsigned long long before = warp == 0 ? 0ull : warp_tot[warp - 1];
  __syncthreads();
  return before + x - v;
}

// Pages per thread whose densities stay in registers between the passes
// (4096 pages at 1M context: four per thread); longer histories recompute.
constexpr int kKeep = 8;

__global__ void __launch_bounds__(kRecallThreads)
    page_recall_kernel(const uint32_t* __restrict__ mask, int64_t S, int64_t sink, int64_t recent, int kmax,
                       int32_t* __restrict__ pages_out, int32_t* __restrict__ density_out,
                       int32_t* __restrict__ n_out) {
  __shared__ RecallSmem sm;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t b = blockIdx.x;
  const int64_t words = (S + 31) / 32;
  const int64_t n_pages = (S + kPageChunks - 1) / kPageChunks;
  const uint32_t* row = mask + b * words;
  int32_t* po = pages_out + b * kmax;
  int32_t* dn = density_out != nullptr ? density_out + b * kmax : nullptr;
  // Each thread owns a contiguous run of pages, so the output can be written
  // in page order from one prefix sum; its densities are computed once.
  const int64_t per = (n_pages + kRecallThreads - 1) / kRecallThreads;
  const int64_t p0 = tid * per;
  const int64_t p1 = p0 + per < n_pages ? p0 + per : n_pages;
  // pages wholly inside [sink, S - recent) and below S need no range masks
  const int64_t plain_lo = (sink + kPageChunks - 1) / kPageChunks;
  const int64_t plain_hi = (S - recent) / kPageChunks;  // pages [plain_lo, plain_hi)
  auto density = [&](int64_t p) -> int {
    if (p >= plain_lo && p < plain_hi) {
      return __popc(__ldg(row + 2 * p)) + __popc(__ldg(row + 2 * p + 1));
    }
    return page_density(row, words, p, S, sink, recent);
  };
  int dens[kKeep];
  for (int i = tid; i <= kPageChunks; i += kRecallThreads) sm.hist[i] = 0u;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kKeep; ++i) {
    dens[i] = 0;
    if (p0 + i < p1) {
      dens[i] = density(p0 + i);
      atomicAdd(&sm.hist[dens[i]], 1u);
    }
  }
  for (int64_t p = p0 + kKeep; p < p1; ++p) atomicAdd(&sm.hist[density(p)], 1u);
  __syncthreads();
  if (warp == 0) {
    // The cut D is the largest density at which the pages of density >= D
    // reach kmax; pages above D are all taken and the lowest-id kmax - above
    // pages of density D fill up.  If every non-empty page fits, all are
    // taken (D = 1).  Lane l holds densities 2l + 1, 2l + 2 (and 64 on lane
    // 31); suffix sums over lanes give the count at or above each density.
    const uint32_t c1 = sm.hist[2 * lane + 1], c2 = sm.hist[2 * lane + 2];
    uint32_t suf = c1 + c2;  // this lane's pages, then those of higher lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_down_sync(0xffffffffu, suf, o);
      if (lane + o < 32) suf += y;
    }
    const uint32_t above_lane = suf - c1 - c2;  // pages with density > 2l + 2
    // density 2l + 2 reaches kmax?  else 2l + 1?
    const bool hit2 = above_lane + c2 >= (uint32_t)kmax;
    const bool hit1 = above_lane + c2 + c1 >= (uint32_t)kmax;
    const uint32_t ball = __ballot_sync(0xffffffffu, hit1);
    if (ball == 0u) {  // every non-empty page fits
      if (lane == 0) {
        sm.cut = 1;
        sm.take_eq = c1;
        sm.above = suf - c1;
      }
    } else {
      const int top = 31 - __clz((int)ball);  // highest lane whose densities reach kmax
      if (lane == top) {
        if (hit2) {
          sm.cut = 2 * lane + 2;
          sm.above = above_lane;
          sm.take_eq = (uint32_t)kmax - above_lane;
        } else {
          sm.cut = 2 * lane + 1;
          sm.above = above_lane + c2;
          sm.take_eq = (uint32_t)kmax - above_lane - c2;
        }
      }
    }
  }
  __syncthreads();
  const int cut = sm.cut;
  const uint32_t take_eq = sm.take_eq;
  const uint32_t n_taken = sm.above + take_eq;

  // ---- ordered emission: one prefix sum of (pages above D, pages at D)
  uint32_t gt = 0, eq = 0;
#pragma unroll
  for (int i = 0; i < kKeep; ++i)
    if (p0 + i < p1) {
      gt += dens[i] > cut;
      eq += dens[i] == cut;
    }
  for (int64_t p = p0 + kKeep; p < p1; ++p) {
    const int d = density(p);
    gt += d > cut;
    eq += d == cut;
  }
  // one scan of both counts, 32 bits each
  const unsigned long long packed = excl_scan64(((unsigned long long)gt << 32) | eq, sm.warp_tot64);
  uint32_t g = (uint32_t)(packed >> 32), e = (uint32_t)packed;
  auto emit = [&](int64_t p, int d) {
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
  };
#pragma unroll
  for (int i = 0; i < kKeep; ++i)
    if (p0 + i < p1) emit(p0 + i, dens[i]);
  for (int64_t p = p0 + kKeep; p < p1; ++p) emit(p, density(p));
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

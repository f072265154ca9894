// topk.cuh -- exact block-level top-k select over one row of fp32 scores.
//
// Semantics ("FlashMemory-DeepSeek-V4: Lightning Index ...", sec. 3: the
// native selector keeps the Top-k of Score_native inside the resident set;
// "DeepSeek-V4 CSA + HCA explained", sec. 3, CSA-2: top-512 of the C4Indexer
// score, sec. 8: fewer than 512 chunks -> all of them): the min(k, n) best
// candidates by (score desc, index asc), emitted in ascending index order.
//
// Algorithm: scores map to order-preserving uint32 keys; four 8-bit radix
// passes (most significant digit first) find the exact k-th key T and how many
// of the keys equal to T are needed; one final pass over the row in index
// order writes every key > T and the first `need` keys == T, with output
// positions from a block-wide prefix sum -- so the output is already sorted
// by index and ties resolve to the lower index.  Histograms use warp-
// aggregated shared-memory atomics (__match_any_sync).
#pragma once

#include "fm_common.cuh"

namespace fm {

template <int THREADS>
struct TopkSmem {
  uint32_t hist[256];
  uint32_t warp_tot[THREADS / 32];
  uint32_t sel_prefix, sel_mask, need, digit_above;
};

// Block-wide exclusive prefix sum of `v` (all THREADS threads call it).
template <int THREADS>
FM_DEV uint32_t block_excl_scan(uint32_t v, uint32_t* warp_tot, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t t = lane < THREADS / 32 ? warp_tot[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < THREADS / 32) warp_tot[lane] = t;  // inclusive warp totals
  }
  __syncthreads();
  const uint32_t before = warp == 0 ? 0u : warp_tot[warp - 1];
  *total = warp_tot[THREADS / 32 - 1];
  __syncthreads();
  return before + x - v;
}

// Exact select over row[0..n) (n >= 0) straight from global memory (four
// radix passes + one ordered output pass).  idx_map(i) gives the id written
// for candidate i.  Writes k entries of idx_out / score_out (score_out may be
// null).  All THREADS threads of the block must call this.
template <int THREADS, typename IdxMap>
FM_DEV void block_topk_radix(const float* __restrict__ row, int n, int k, IdxMap idx_map, int32_t* __restrict__ idx_out,
                       float* __restrict__ score_out, TopkSmem<THREADS>& sm) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int kk = n < k ? n : k;
  uint32_t prefix = 0, pmask = 0, need = (uint32_t)kk;

  if (n > k) {
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += THREADS) sm.hist[i] = 0;
      __syncthreads();
      for (int i0 = 0; i0 < n; i0 += THREADS) {
        const int i = i0 + tid;
        uint32_t key = 0;
        bool act = false;
        if (i < n) {
          key = float_key(__ldg(row + i));
          act = (key & pmask) == prefix;
        }
        if (act) atomicAdd(&sm.hist[(key >> shift) & 0xFFu], 1u);
      }
      __syncthreads();
      if (tid < 32) {
        // lane l owns digits 255-8l .. 248-8l (descending)
        uint32_t c[8], s = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = sm.hist[255 - 8 * lane - j];
          s += c[j];
        }
        uint32_t incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        uint32_t above = incl - s;  // count in digits above this lane's range
        // the lane whose range contains the need-th key
        const bool mine = above < need && need <= incl;
        if (mine) {
          uint32_t acc = above;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (acc + c[j] >= need) {
              sm.sel_prefix = 255u - 8u * (uint32_t)lane - (uint32_t)j;
              sm.digit_above = acc;
              break;
            }
            acc += c[j];
          }
        }
      }
      __syncthreads();
      const uint32_t d = sm.sel_prefix;
      need -= sm.digit_above;
      prefix |= d << shift;
      pmask |= 0xFFu << shift;
      __syncthreads();
    }
  }

  // Final pass: keys > T always, keys == T while fewer than `need` taken.
  // (When n <= k, pmask == 0 and every candidate is "== T": all are taken.)
  uint32_t out_base = 0, eq_seen = 0;
  const uint32_t T = prefix;
  for (int i0 = 0; i0 < n && out_base < (uint32_t)kk; i0 += THREADS) {
    const int i = i0 + tid;
    float v = 0.f;
    uint32_t gt = 0, eq = 0;
    if (i < n) {
      v = __ldg(row + i);
      const uint32_t key = float_key(v) & pmask;
      gt = key > T;
      eq = key == T;
    }
    uint32_t tot;
    const uint32_t packed = block_excl_scan<THREADS>((eq << 16) | gt, sm.warp_tot, &tot);
    const uint32_t gt_before = packed & 0xFFFFu, eq_before = packed >> 16;
    const uint32_t eq_tile = tot >> 16, gt_tile = tot & 0xFFFFu;
    const uint32_t taken_before = min(eq_seen + eq_before, need) - min(eq_seen, need);
    const bool take = gt || (eq && eq_seen + eq_before < need);
    if (take) {
      const uint32_t pos = out_base + gt_before + taken_before;
      idx_out[pos] = idx_map(i);
      if (score_out) score_out[pos] = v;
    }
    out_base += gt_tile + (min(eq_seen + eq_tile, need) - min(eq_seen, need));
    eq_seen += eq_tile;
  }
  for (int p = kk + tid; p < k; p += THREADS) {
    idx_out[p] = -1;
    if (score_out) score_out[p] = -INFINITY;
  }
}

}  // namespace fm

namespace fm {

// Fast path: a threshold from a sample, one filtering pass into shared memory,
// an exact select among the candidates, output positions from a bitmap.
//
//  Every candidate is ranked by its unique composite key (key << 32 | ~index),
//  which orders (score desc, index asc).
//  1. Sample 32 evenly spaced runs of 64 consecutive scores (coalesced) and
//     take theta = about the r-th largest sampled score key, r chosen so that
//     about 2 min(k, n) candidates (3 min(k, n) for rows long enough that r
//     would fall below 64; at most 2/3 of the list) are expected at or above
//     it.
//  2. One vectorised pass compares each score with theta's score as a plain
//     fp32 compare; the scores that reach it (a few percent, ties with
//     theta's score included) are appended with their composites to a
//     shared-memory list (one shared-memory atomic per warp and pass); the
//     largest appended composite is tracked too.
//  3. If the list holds at least min(k, n) entries and did not overflow, the
//     true top-k is inside it (the k-th largest composite is >= the lowest
//     composite with theta's key): a block-wide radix select over the
//     composites, starting at the first bit where that bound and the largest
//     candidate differ, finds the min(k, n)-th largest T.  A list that
//     overflows (rows flooded by ties at the threshold) or falls short takes
//     one re-aimed sample, then the exact global-memory radix path
//     (block_topk_radix).
//  4. The selected indices are marked in a bitmap; one block-wide prefix sum
//     over the bitmap words gives each thread's word range its first output
//     slot, and each selected candidate computes its own slot (rank by index)
//     from it, so the output is in ascending index order with no sort and no
//     second read of the row (longer rows sort the selection instead).
// Scores are reported from their keys: -0 reads as +0 and NaN as -inf.
constexpr int kTopkCap = 4096;       // candidate slots (32 KB of shared memory)
constexpr int kTopkCapShort = 3072;  // for rows of at most kTopkShortN scores (24 KB: five CTAs per SM)
constexpr int kTopkShortN = 1 << 18;  // every row up to a 1M-token history (262144 chunks)
constexpr int kTopkRuns = 32;        // sample: 32 runs x 64 scores
constexpr int kTopkSample = kTopkRuns * 64;
constexpr int kTopkBitmapN = 131072;  // rows up to this length emit ids via a bitmap

template <int THREADS>
struct SelectSmem {
  uint32_t hist[2][256];
  uint32_t digit[2], above[2], in_digit[2];
};

// RUNS: sampled runs of 64 scores; BITMAP_N: rows up to this length emit ids
// through a bitmap (a CTA instantiated for shorter rows only needs that much).
template <int THREADS, int CAP = kTopkCap, int RUNS = kTopkRuns, int BITMAP_N = kTopkBitmapN>
struct TopkFastSmem {
  unsigned long long cand[CAP];
  unsigned long long cmax;
  union {
    unsigned long long sample[RUNS * 64];
    uint32_t sample32[2 * RUNS * 64];  // rows longer than BITMAP_N: twice the sample, keys only
    unsigned long long sel[1024];
    uint32_t bitmap[BITMAP_N / 32];
  } u;
  uint32_t tpre[THREADS];
  uint32_t count;
  int overflow;
  uint32_t klo, khi, nlist;  // block_topk_segmax: range of the segment keys, list length
  SelectSmem<THREADS> sel;
  TopkSmem<THREADS> radix;
};

// Bitonic sort of s[0..P2) descending (P2 a power of two), all threads.
template <int THREADS>
FM_DEV void bitonic_desc(unsigned long long* s, int P2) {
  for (int size = 2; size <= P2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < P2 / 2; i += THREADS) {
        const int lo = 2 * stride * (i / stride) + (i % stride);
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const unsigned long long a = s[lo], b = s[hi];
        if ((a < b) == desc) {
          s[lo] = b;
          s[hi] = a;
        }
      }
      __syncthreads();
    }
  }
}

FM_DEV int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

// Radix select of the r-th largest (1 <= r <= n) of the values a[0..n)
// (32- or 64-bit) in shared memory, all of which lie in [lo, hi]: 8-bit digits, most
// significant first, starting at the highest bit where lo and hi differ (the
// bits above it are common to every value, so they need no pass).  It stops
// once the deciding digit holds exactly the remaining need (then the result T
// has count(a >= T) == r) or at most `loose` values (then r <= count(a >= T)
// <= r + loose); always count(a >= T) >= r.  Digit counts are plain
// shared-memory atomics (cheaper here than aggregating them per warp with
// __match_any_sync); the two histograms alternate so that each digit costs two
// block barriers.  All threads call it.
template <int THREADS, typename T>
FM_DEV T block_select(const T* a, int n, int r, T lo, T hi, uint32_t loose, SelectSmem<THREADS>& sm) {
  constexpr int kBits = 8 * (int)sizeof(T);
  const int tid = threadIdx.x, lane = tid & 31;
  if (lo == hi) return lo;
  const int hb = kBits == 64 ? 63 - __clzll((long long)(lo ^ hi)) : 31 - __clz((int)(lo ^ hi));
  T pmask = hb == kBits - 1 ? T(0) : (~T(0) << (hb + 1));
  T prefix = lo & pmask;
  uint32_t need = (uint32_t)r;
  for (int i = tid; i < 256; i += THREADS) sm.hist[0][i] = 0u;
  __syncthreads();
  int b = 0;
  for (int s = hb - 7;; s -= 8, b ^= 1) {
    const int shift = s > 0 ? s : 0;
    uint32_t* hist = sm.hist[b];
    for (int i = tid; i < 256; i += THREADS) sm.hist[b ^ 1][i] = 0u;  // for the next digit
    for (int i = tid; i < n; i += THREADS) {
      const T v = a[i];
      if ((v & pmask) == prefix) atomicAdd(&hist[(uint32_t)(v >> shift) & 0xFFu], 1u);
    }
    __syncthreads();
    if (tid < 32) {
      // lane l owns digits 255-8l .. 248-8l (descending)
      uint32_t c[8], s8 = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - 8 * lane - j];
        s8 += c[j];
      }
      uint32_t incl = s8;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t above = incl - s8;
      if (above < need && need <= incl) {
        uint32_t acc = above;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (acc + c[j] >= need) {
            sm.digit[b] = 255u - 8u * (uint32_t)lane - (uint32_t)j;
            sm.above[b] = acc;
            sm.in_digit[b] = c[j];
            break;
          }
          acc += c[j];
        }
      }
    }
    __syncthreads();
    const uint32_t d = sm.digit[b], in_digit = sm.in_digit[b];
    need -= sm.above[b];
    prefix |= (T)d << shift;  // bits already decided agree with d
    pmask |= (T)0xFFu << shift;
    if (shift == 0 || in_digit == need || in_digit <= loose) break;
  }
  return prefix;
}

// An id map that reads page ids (candidate i -> ids[i / 64] * 64 + i % 64)
// declares kPageIds; the emit then stages the row's page ids in shared memory
// (past the bitmap words it uses) before the select, so the ids it writes
// cost no global load on the way out.
template <typename M, typename = void>
struct has_page_ids {
  static constexpr bool value = false;
};
template <typename M>
struct has_page_ids<M, decltype((void)M::kPageIds)> {
  static constexpr bool value = M::kPageIds;
};

// Steps 3 and 4 of the select, shared by block_topk and block_topk_segmax:
// the exact kk-th largest composite T among the cnt candidates in sm.cand
// (every one of them in [theta, sm.cmax]), then every candidate >= T written
// in index order, and -1 / -inf in positions kk .. k-1.  Rows of at most
// BITMAP_N scores emit through sm.u.bitmap, whose first (n + 31) / 32 words
// the caller has cleared.  All threads call it.
template <int THREADS, int CAP, typename IdxMap, int RUNS, int BITMAP_N>
FM_DEV void block_topk_emit(TopkFastSmem<THREADS, CAP, RUNS, BITMAP_N>& sm, int cnt, unsigned long long theta, int n,
                            int kk, int k, IdxMap idx_map, int32_t* __restrict__ idx_out,
                            float* __restrict__ score_out) {
  constexpr int kTopkBitmapN = BITMAP_N;
  const int tid = threadIdx.x;
  // ---- 3. exact select among the candidates -------------------------------------
  const int words = (n + 31) >> 5;
  const int npages = (n + 63) >> 6;
  uint32_t* staged = sm.u.bitmap + words;  // page ids past the bitmap words in use
  bool use_staged = false;
  if constexpr (has_page_ids<IdxMap>::value) {
    use_staged = n <= kTopkBitmapN && words + npages <= kTopkBitmapN / 32;
    if (use_staged)
      for (int i = tid; i < npages; i += THREADS) staged[i] = (uint32_t)__ldg(idx_map.ids + i);
  }
  // every candidate lies in [theta, cmax] (the select's barriers also publish
  // the staged ids)
  const unsigned long long T = block_select<THREADS>(sm.cand, cnt, kk, theta, sm.cmax, 0u, sm.sel);
  // ---- 4. emit in index order -------------------------------------------------
  if (n <= kTopkBitmapN) {
    for (int i = tid; i < cnt; i += THREADS) {
      const unsigned long long c = sm.cand[i];
      if (c >= T) {
        const uint32_t idx = ~(uint32_t)c;
        atomicOr(&sm.u.bitmap[idx >> 5], 1u << (idx & 31));
      }
    }
    __syncthreads();
    const int per = (words + THREADS - 1) / THREADS;  // consecutive words per thread
    const int w0 = tid * per;
    uint32_t mine = 0;
    for (int j = 0; j < per; ++j)
      if (w0 + j < words) mine += (uint32_t)__popc(sm.u.bitmap[w0 + j]);
    uint32_t tot;
    sm.tpre[tid] = block_excl_scan<THREADS>(mine, sm.radix.warp_tot, &tot);
    __syncthreads();
    for (int i = tid; i < cnt; i += THREADS) {
      const unsigned long long c = sm.cand[i];
      if (c >= T) {
        const uint32_t idx = ~(uint32_t)c;
        const int w = (int)(idx >> 5), owner = w / per;
        uint32_t pos = sm.tpre[owner] + (uint32_t)__popc(sm.u.bitmap[w] & ((1u << (idx & 31)) - 1u));
        for (int w2 = owner * per; w2 < w; ++w2) pos += (uint32_t)__popc(sm.u.bitmap[w2]);
        idx_out[pos] = use_staged ? (int32_t)staged[idx >> 6] * 64 + (int32_t)(idx & 63) : idx_map((int)idx);
        if (score_out) score_out[pos] = key_float((uint32_t)(c >> 32));
      }
    }
  } else {
    if (tid == 0) sm.count = 0;
    __syncthreads();
    for (int i = tid; i < cnt; i += THREADS) {
      const unsigned long long c = sm.cand[i];
      if (c >= T) {
        // re-key by index: ascending index == descending ~index
        const uint32_t slot = atomicAdd(&sm.count, 1u);
        sm.u.sel[slot] = ((unsigned long long)(uint32_t)c << 32) | (c >> 32);
      }
    }
    __syncthreads();
    const int K2 = next_pow2(kk);
    for (int i = kk + tid; i < K2; i += THREADS) sm.u.sel[i] = 0ull;
    __syncthreads();
    bitonic_desc<THREADS>(sm.u.sel, K2);
    for (int p = tid; p < kk; p += THREADS) {
      const unsigned long long c = sm.u.sel[p];
      const int i = (int)(~(uint32_t)(c >> 32));
      idx_out[p] = idx_map(i);
      if (score_out) score_out[p] = key_float((uint32_t)c);
    }
  }
  for (int p = kk + tid; p < k; p += THREADS) {
    idx_out[p] = -1;
    if (score_out) score_out[p] = -INFINITY;
  }
}

template <int THREADS, int CAP, typename IdxMap, int RUNS = kTopkRuns, int BITMAP_N = kTopkBitmapN>
FM_DEV void block_topk(const float* __restrict__ row, int n, int k, IdxMap idx_map, int32_t* __restrict__ idx_out,
                       float* __restrict__ score_out, TopkFastSmem<THREADS, CAP, RUNS, BITMAP_N>& sm) {
  constexpr int kTopkRuns = RUNS;  // this instantiation's sample and bitmap sizes
  constexpr int kTopkSample = RUNS * 64;
  constexpr int kTopkBitmapN = BITMAP_N;
  const int tid = threadIdx.x;
  const int kk = n < k ? n : k;
  if (kk == 0) {
    for (int p = tid; p < k; p += THREADS) {
      idx_out[p] = -1;
      if (score_out) score_out[p] = -INFINITY;
    }
    return;
  }
  // ---- 1. threshold from a sample --------------------------------------------
  // A sample that misjudges the row (fewer than min(k, n) candidates reach
  // theta, or more than the list holds) is re-aimed once: the survivor count
  // c observed at sample rank r gives the rank r * want / c, and the sample and
  // the filter pass run again (the row is in L2 by then).  Only a second miss
  // takes the exact global-memory path, whose four radix passes and ordered
  // output pass over the row cost a multiple of the fast path.
  // expected candidates: 2 min(k, n) where the sample rank of theta is at
  // least 64 (the survivor count then stays within about half of its aim at
  // four standard deviations), else 3 min(k, n); at most 2/3 of the list
  const long long aim = 2LL * kk * kTopkSample >= 64LL * n ? 2LL * kk : 3LL * kk;
  const long long want = aim < 2 * CAP / 3 ? aim : 2 * CAP / 3;
  long long r_aim = -1;  // sample rank of theta (-1: from `want`)
  unsigned long long theta = 0ull;
  for (int attempt = 0;; ++attempt) {
  theta = 0ull;
  if (n > CAP) {
    if (n <= kTopkBitmapN) {
      // every thread's samples are loaded before any is stored, so their
      // loads overlap (run * (n - 64) < 2^31 for these rows).  The filter
      // thresholds at theta's score key, so the sample is kept as 32-bit
      // keys and theta's index part is zero.
      constexpr int kPerT = kTopkSample / THREADS;
      static_assert(kPerT * THREADS == kTopkSample, "sample entries per thread");
      float sv[kPerT];
#pragma unroll
      for (int t = 0; t < kPerT; ++t) {
        const int i = tid + t * THREADS, run = i >> 6, off = i & 63;
        sv[t] = __ldg(row + run * (n - 64) / (kTopkRuns - 1) + off);
      }
#pragma unroll
      for (int t = 0; t < kPerT; ++t) sm.u.sample32[tid + t * THREADS] = float_key(sv[t]);
      __syncthreads();
      long long r = r_aim >= 0 ? r_aim : (want * kTopkSample) / (long long)n;
      r = r < 1 ? 1 : (r > kTopkSample ? kTopkSample : r);
      r_aim = r;
      theta = (unsigned long long)block_select<THREADS>(sm.u.sample32, kTopkSample, (int)r, 0u, ~0u, 4u, sm.sel)
              << 32;
    } else {
      // Long rows (a whole 1M-token history is 262144 scores): with 2048
      // samples only ~12 would lie above the threshold and about one row in
      // a thousand would fall short of k candidates.  Twice the sample as
      // plain 32-bit keys (same shared memory) keeps ~24 above it; the
      // threshold then admits every score >= the sampled key (ties at it
      // are not split by index).
      for (int i = tid; i < 2 * kTopkSample; i += THREADS) {
        const int run = i >> 6, off = i & 63;
        const int j = (int)(((long long)run * (n - 64)) / (2 * kTopkRuns - 1)) + off;
        sm.u.sample32[i] = float_key(__ldg(row + j));
      }
      __syncthreads();
      long long r = r_aim >= 0 ? r_aim : (want * 2 * kTopkSample) / (long long)n;
      r = r < 1 ? 1 : (r > 2 * kTopkSample ? 2 * kTopkSample : r);
      r_aim = r;
      theta = (unsigned long long)block_select<THREADS>(sm.u.sample32, 2 * kTopkSample, (int)r, 0u, ~0u, 4u, sm.sel)
              << 32;
    }
  }
  // the sample is dead from here: its space becomes the (cleared) bitmap
  if (n <= kTopkBitmapN) {
    const int words = (n + 31) >> 5;
    for (int i = tid; i < words; i += THREADS) sm.u.bitmap[i] = 0u;
  }
  if (tid == 0) {
    sm.count = 0;
    sm.overflow = 0;
    sm.cmax = 0ull;
  }
  __syncthreads();
  // ---- 2. filter pass ---------------------------------------------------------
  // Every score keyed at or above theta's score key survives: the threshold
  // drops from theta to the lowest composite with that key, so all scores
  // tied with theta's are kept.  The list then holds every composite at or
  // above that bound; with at least min(k, n) of them (checked below) the
  // top min(k, n) of the row are all among them, so the select is exact.
  // A key test is a plain fp32 compare (-0 == +0 like their keys, NaN below
  // every threshold); a threshold at or below the key of -inf (rows
  // dominated by -inf/NaN, where NaN ranks as -inf) takes every score.
  const uint32_t theta_key = (uint32_t)(theta >> 32);
  const bool take_all = theta_key <= 0x007FFFFFu;
  const float theta_f = take_all ? -INFINITY : key_float(theta_key);
  const int lane = tid & 31;
  auto composite_of = [](float v, int i) -> unsigned long long {
    return ((unsigned long long)float_key(v) << 32) | (uint32_t)(~(uint32_t)i);
  };
  // Each warp counts its survivors and reserves their slots with one
  // shared-memory atomic (all lanes call it).
  auto reserve = [&](uint32_t mine) -> uint32_t {
    uint32_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
    uint32_t base = 0;
    if (lane == 31 && total > 0u) base = atomicAdd(&sm.count, total);
    return __shfl_sync(0xffffffffu, base, 31) + incl - mine;
  };
  unsigned long long tmax = 0ull;  // this thread's largest stored composite
  auto store = [&](uint32_t slot, float v, int i) {
    const unsigned long long c = composite_of(v, i);
    if (slot < (uint32_t)CAP) {
      sm.cand[slot] = c;
      tmax = c > tmax ? c : tmax;
    } else {
      sm.overflow = 1;
    }
  };
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  const int n4 = vec ? n / 4 : 0;
  const float4* row4 = reinterpret_cast<const float4*>(row);
  constexpr int kVec = 8;  // float4 loads in flight per thread
  for (int i40 = 0; i40 < n4; i40 += THREADS * kVec) {  // same trip count in every thread
    float4 v[kVec];
#pragma unroll
    for (int u = 0; u < kVec; ++u) {
      const int i4 = i40 + u * THREADS + tid;
      v[u] = i4 < n4 ? __ldg(row4 + i4) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
    uint32_t mask = 0;  // bit 4u + e: element e of v[u] survives
#pragma unroll
    for (int u = 0; u < kVec; ++u) {
      const float4 x = v[u];
      const uint32_t m4 = take_all ? 15u
                                   : (uint32_t)(x.x >= theta_f) | ((uint32_t)(x.y >= theta_f) << 1) |
                                         ((uint32_t)(x.z >= theta_f) << 2) | ((uint32_t)(x.w >= theta_f) << 3);
      if (i40 + u * THREADS + tid < n4) mask |= m4 << (4 * u);
    }
    uint32_t slot = reserve((uint32_t)__popc(mask));
    // survivors are few (~6% of a row): each lane walks its own, re-reading
    // the score (a cache hit) rather than indexing v[] at run time, which
    // would put v in local memory
    while (mask) {
      const int b = __ffs(mask) - 1;
      mask &= mask - 1u;
      const int i = 4 * (i40 + (b >> 2) * THREADS + tid) + (b & 3);
      store(slot++, __ldg(row + i), i);
    }
  }
  for (int i0 = 4 * n4; i0 < n; i0 += THREADS) {  // scalar rest (all of an unaligned row)
    const int i = i0 + tid;
    const float v = i < n ? __ldg(row + i) : -INFINITY;
    const bool p = i < n && (take_all || v >= theta_f);
    const uint32_t slot = reserve((uint32_t)p);
    if (p) store(slot, v, i);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long y = __shfl_xor_sync(0xffffffffu, tmax, o);
    tmax = y > tmax ? y : tmax;
  }
  if (lane == 0 && tmax != 0ull) atomicMax(&sm.cmax, tmax);
  __syncthreads();
  const int survivors = (int)sm.count;  // every survivor, also those past the list
  if (!sm.overflow && survivors >= kk) break;
  __syncthreads();
  // a miss: re-aim the sample rank once (n > CAP here: a row that fits the
  // list takes every score and cannot miss), else the exact path
  long long r_next = r_aim * want / (survivors > 0 ? survivors : 1);
  r_next = r_next < 1 ? 1 : r_next;
  if (attempt > 0 || n <= CAP || r_next == r_aim) {
    block_topk_radix<THREADS>(row, n, k, idx_map, idx_out, score_out, sm.radix);
    return;
  }
  r_aim = r_next;
  }  // attempts
  block_topk_emit(sm, (int)sm.count, (unsigned long long)(uint32_t)(theta >> 32) << 32, n, kk, k, idx_map, idx_out,
                  score_out);
}

// A segment entry e -- of the 32 scores 32g .. 32g+31 of a row that lie below
// its length, the largest bit pattern read as a signed integer (what the
// prefill score kernel writes) -- gives two keys:
//  - seg_floor_key: the key of one of those scores.  Unless e is a NaN it is
//    one of their bit patterns; a NaN gives 0, below every score's key.
//  - seg_ceil_key: a key no smaller than any of theirs.  With e >= 0 (not
//    NaN), no pattern with the sign bit clear exceeds e, so e is the largest
//    score and every negative score, -0 and NaN (which float_key ranks as
//    -inf) keys lower.  With e < 0 every score has its sign bit set, so none
//    keys above +0.  A NaN entry bounds nothing: ~0.
FM_DEV uint32_t seg_floor_key(int32_t e) {
  const float f = __int_as_float(e);
  return f != f ? 0u : float_key(f);
}
FM_DEV uint32_t seg_ceil_key(int32_t e) {
  const float f = __int_as_float(e);
  if (f != f) return ~0u;
  return float_key(e < 0 ? 0.0f : f);
}

// Exact top-k of a row of n scores that comes with its segment entries
// segmax[0 .. ceil(n/32)) (above): same output as block_topk.
//   1. tau = the kk-th largest floor key over the segments.  kk distinct
//      segments each hold a score keyed >= tau, so the kk-th largest score
//      keys >= tau: no score below tau can be selected.
//   2. Every score keyed >= tau lies in a segment whose ceiling key is
//      >= tau; those segments are listed (for kk = 512 of 2048 segments,
//      about a quarter of the row).
//   3. One pass over the listed segments keeps every score keyed >= tau as a
//      candidate (for independent scores, ~1.15 kk of them).
//   4. The exact select and the emission of block_topk among the candidates
//      (ties resolve to the lower index as there: all tied scores are in).
// Rows with fewer than 2 kk segments, more segments than the sample space
// holds, or more candidates than the list, take block_topk on the whole row.
template <int THREADS, int CAP, typename IdxMap, int RUNS = kTopkRuns, int BITMAP_N = kTopkBitmapN>
FM_DEV void block_topk_segmax(const float* __restrict__ row, int n, int k, const int32_t* __restrict__ segmax,
                              bool ld4, IdxMap idx_map, int32_t* __restrict__ idx_out, float* __restrict__ score_out,
                              TopkFastSmem<THREADS, CAP, RUNS, BITMAP_N>& sm) {
  constexpr int kSegCap = 2 * RUNS * 64;   // entries of sm.u.sample32
  constexpr int kPer = kSegCap / THREADS;  // segment entries per thread
  constexpr int kU = 16;                   // segments in flight per warp
  constexpr int kWarps = THREADS / 32;
  static_assert(kPer <= 32 && kPer * THREADS == kSegCap, "segment entries per thread");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kk = n < k ? n : k;
  const int nseg = (n + 31) >> 5;
  if (kk == 0 || nseg < 2 * kk || nseg > kSegCap || n > BITMAP_N) {
    block_topk<THREADS, CAP, IdxMap, RUNS, BITMAP_N>(row, n, k, idx_map, idx_out, score_out, sm);
    return;
  }
  // ---- 1. tau -------------------------------------------------------------------
  // thread t holds the entries of segments t, t + THREADS, ...
  uint32_t* keys = sm.u.sample32;
  if (tid == 0) {
    sm.klo = ~0u;
    sm.khi = 0u;
    sm.nlist = 0u;
  }
  int32_t e[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int g = tid + j * THREADS;
    e[j] = g < nseg ? __ldg(segmax + g) : 0;
  }
  uint32_t lo = ~0u, hi = 0u;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int g = tid + j * THREADS;
    if (g < nseg) {
      const uint32_t f = seg_floor_key(e[j]);
      keys[g] = f;
      lo = f < lo ? f : lo;
      hi = f > hi ? f : hi;
    }
  }
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
  __syncthreads();  // klo / khi / nlist initialised
  if (lane == 0) {
    atomicMin(&sm.klo, lo);
    atomicMax(&sm.khi, hi);
  }
  __syncthreads();
  // loose: a tau a little below the exact kk-th key is still a bound (a few
  // more segments listed); the select skips the bits that every key shares
  const uint32_t tau = block_select<THREADS>(keys, nseg, kk, sm.klo, sm.khi, 64u, sm.sel);
  // ---- 2. the listed segments (in no particular order: ids leave in index
  // order through the bitmap) ---------------------------------------------------
  const bool vec = ld4 && (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  uint32_t flags = 0;  // bit j: segment tid + j * THREADS is listed
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int g = tid + j * THREADS;
    if (g < nseg && seg_ceil_key(e[j]) >= tau) flags |= 1u << j;
  }
  {
    // one warp scan and one shared-memory atomic per warp place the entries;
    // no thread reads keys[] once the select has returned
    const uint32_t c = (uint32_t)__popc(flags);
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
    uint32_t base = 0;
    if (lane == 31 && total > 0u) base = atomicAdd(&sm.nlist, total);
    uint32_t pos = __shfl_sync(0xffffffffu, base, 31) + incl - c;
    while (flags) {
      const int j = __ffs(flags) - 1;
      flags &= flags - 1u;
      const int g = tid + j * THREADS;
      keys[pos++] = (uint32_t)g;
    }
  }
  if (tid == 0) {
    sm.count = 0;
    sm.overflow = 0;
    sm.cmax = 0ull;
  }
  __syncthreads();
  // ---- 3. candidates: every score of a listed segment keyed >= tau --------------
  // A score keys >= tau exactly when it is >= tau's float (-0 == +0 as their
  // keys); with tau at or below the key of -inf (where NaN ranks) the keys are
  // compared instead.  With ld4 (the row's allocated length a multiple of 4)
  // and the row on a 16-byte boundary, four segments are read per float4 load
  // (eight lanes each), else one per scalar load.
  const int m = (int)sm.nlist;
  const bool take_all = tau <= 0x007FFFFFu;
  const float tau_f = take_all ? -INFINITY : key_float(tau);
  unsigned long long tmax = 0ull;
  auto passes = [&](float x, int i) -> bool {
    return i < n && (take_all ? float_key(x) >= tau : x >= tau_f);
  };
  // `c` list slots for this lane (most lanes have none: one shared-memory
  // atomic each for the rest beats a warp scan's chain of shuffles)
  auto reserve = [&](uint32_t c) -> uint32_t { return c ? atomicAdd(&sm.count, c) : 0u; };
  auto store = [&](uint32_t slot, float x, int i) {
    const unsigned long long cv = ((unsigned long long)float_key(x) << 32) | (uint32_t)(~(uint32_t)i);
    if (slot < (uint32_t)CAP) {
      sm.cand[slot] = cv;
      tmax = cv > tmax ? cv : tmax;
    } else {
      sm.overflow = 1;
    }
  };
  if (vec) {
    // a float4 starting at a multiple of 4 below n stays inside the row
    constexpr int kLoads = kU / 4;
    const int sub = lane >> 3, part = (lane & 7) * 4;
    for (int j0 = warp * kU; j0 < m; j0 += kWarps * kU) {  // warp-uniform trip count
      float4 v[kLoads];
      int base[kLoads];
#pragma unroll
      for (int u = 0; u < kLoads; ++u) {
        const int j = j0 + 4 * u + sub;
        base[u] = j < m ? (int)keys[j] * 32 + part : n;
        v[u] = base[u] < n ? __ldg(reinterpret_cast<const float4*>(row + base[u]))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      uint32_t mask = 0;  // bit 4u + e: element e of v[u] is a candidate
#pragma unroll
      for (int u = 0; u < kLoads; ++u)
        mask |= ((uint32_t)passes(v[u].x, base[u]) | ((uint32_t)passes(v[u].y, base[u] + 1) << 1) |
                 ((uint32_t)passes(v[u].z, base[u] + 2) << 2) | ((uint32_t)passes(v[u].w, base[u] + 3) << 3))
                << (4 * u);
      // candidates are rare (~4% of the listed scores): each lane walks its
      // own, re-reading the score (a cache hit) rather than indexing v[] at run
      // time, which would put v in local memory
      uint32_t slot = reserve((uint32_t)__popc(mask));
      while (mask) {
        const int b = __ffs(mask) - 1;
        mask &= mask - 1u;
        const int i = (int)keys[j0 + 4 * (b >> 2) + sub] * 32 + part + (b & 3);
        store(slot++, __ldg(row + i), i);
      }
    }
  } else {
    for (int j0 = warp * kU; j0 < m; j0 += kWarps * kU) {  // warp-uniform trip count
      float v[kU];
      int idx[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int j = j0 + u;
        idx[u] = j < m ? (int)keys[j] * 32 + lane : n;
        v[u] = idx[u] < n ? __ldg(row + idx[u]) : 0.f;
      }
      uint32_t mask = 0;
#pragma unroll
      for (int u = 0; u < kU; ++u) mask |= (uint32_t)passes(v[u], idx[u]) << u;
      uint32_t slot = reserve((uint32_t)__popc(mask));
      while (mask) {
        const int u = __ffs(mask) - 1;
        mask &= mask - 1u;
        const int i = (int)keys[j0 + u] * 32 + lane;
        store(slot++, __ldg(row + i), i);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long y = __shfl_xor_sync(0xffffffffu, tmax, o);
    tmax = y > tmax ? y : tmax;
  }
  if (lane == 0 && tmax != 0ull) atomicMax(&sm.cmax, tmax);
  __syncthreads();
  const int cnt = (int)sm.count;
  if (sm.overflow || cnt < kk) {  // cnt >= kk always holds (step 1); overflow: a row of clustered maxima
    __syncthreads();
    block_topk<THREADS, CAP, IdxMap, RUNS, BITMAP_N>(row, n, k, idx_map, idx_out, score_out, sm);
    return;
  }
  // ---- 4. the list is dead: its space becomes the (cleared) bitmap ---------------
  const int words = (n + 31) >> 5;
  for (int i = tid; i < words; i += THREADS) sm.u.bitmap[i] = 0u;
  __syncthreads();
  block_topk_emit(sm, cnt, (unsigned long long)tau << 32, n, kk, k, idx_map, idx_out, score_out);
}

}  // namespace fm

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
        const uint32_t digit = act ? ((key >> shift) & 0xFFu) : (0x100u + (uint32_t)lane);
        const uint32_t peers = __match_any_sync(0xffffffffu, digit);
        if (act && lane == __ffs(peers) - 1) atomicAdd(&sm.hist[digit], (uint32_t)__popc(peers));
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
// an exact select among the candidates.
//
//  Every candidate is ranked by its unique composite key (key << 32 | ~index),
//  which orders (score desc, index asc).
//  1. Sample 16 evenly spaced runs of 64 consecutive scores (coalesced) and
//     take theta = about the r-th largest sample composite, r chosen so that
//     about 2.5k candidates of the row are expected at or above it (equal
//     scores are thresholded by index, so ties cannot flood the list).
//  2. One vectorised pass compares each score with theta's score as a plain
//     fp32 compare; only scores that reach it (a few percent) build their
//     composite and are appended, when composite >= theta, to a shared-memory
//     list (one shared-memory atomic per appended candidate).
//  3. If the list holds at least min(k, n) entries and did not overflow, the
//     true top-k is inside it (the k-th largest composite is >= theta): a radix
//     select over the composites finds the min(k, n)-th largest; the selected
//     indices are marked in a bitmap and emitted in index order by one
//     block-wide prefix sum (longer rows gather and sort instead).  Otherwise
//     the exact global-memory radix path (block_topk_radix) runs.
// Scores are reported from their keys: -0 reads as +0 and NaN as -inf.
constexpr int kTopkCap = 4096;        // candidate slots (32 KB of shared memory)
constexpr int kTopkRuns = 16;         // sample: 16 runs x 64 scores
constexpr int kTopkSample = kTopkRuns * 64;
constexpr int kTopkBitmapN = 131072;  // rows up to this length emit ids via a bitmap

template <int THREADS>
struct TopkFastSmem {
  unsigned long long cand[kTopkCap];
  uint32_t whist[256];
  unsigned long long wsel;
  union {
    unsigned long long sample[kTopkSample];
    unsigned long long sel[1024];
    uint32_t bitmap[kTopkBitmapN / 32];
  } u;
  uint32_t count;
  int overflow;
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

// Radix select over a[0..n) in shared memory, most significant 8-bit digit
// first, at most max_passes digits.  Returns T with count(a >= T) >= r
// (1 <= r <= n).  It stops early when the deciding digit holds exactly the
// remaining need (then count(a >= T) == r for distinct values) or at most
// `loose` values (then count(a >= T) <= r + loose).  All threads call it.
template <int THREADS, typename V>
FM_DEV V smem_radix_select(const V* a, int n, int r, int max_passes, uint32_t loose, TopkSmem<THREADS>& sm) {
  const int tid = threadIdx.x, lane = tid & 31;
  constexpr int kBits = 8 * (int)sizeof(V);
  V prefix = 0, pmask = 0;
  uint32_t need = (uint32_t)r;
  for (int pass = 0; pass < max_passes && pass < kBits / 8; ++pass) {
    const int shift = kBits - 8 * (pass + 1);
    for (int i = tid; i < 256; i += THREADS) sm.hist[i] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += THREADS) {
      const int i = i0 + tid;
      bool act = false;
      uint32_t digit = 0x100u + (uint32_t)lane;
      if (i < n) {
        const V v = a[i];
        act = (v & pmask) == prefix;
        if (act) digit = (uint32_t)((v >> shift) & 0xFFu);
      }
      const uint32_t peers = __match_any_sync(0xffffffffu, digit);
      if (act && lane == __ffs(peers) - 1) atomicAdd(&sm.hist[digit], (uint32_t)__popc(peers));
    }
    __syncthreads();
    if (tid < 32) {
      uint32_t c[8], s8 = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = sm.hist[255 - 8 * lane - j];
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
            sm.sel_prefix = 255u - 8u * (uint32_t)lane - (uint32_t)j;
            sm.digit_above = acc;
            sm.need = c[j];
            break;
          }
          acc += c[j];
        }
      }
    }
    __syncthreads();
    const uint32_t d = sm.sel_prefix;
    const uint32_t in_digit = sm.need;
    need -= sm.digit_above;
    prefix |= (V)d << shift;
    pmask |= (V)0xFFu << shift;
    __syncthreads();
    if (in_digit == need || in_digit <= loose) break;  // lower bits cannot matter (or need not)
  }
  return prefix;
}

// The same select run by one warp (no block barriers): for the short lists of
// samples and candidates a single warp is faster than the whole block.
template <typename V>
FM_DEV V warp_radix_select(const V* a, int n, int r, int max_passes, uint32_t loose, uint32_t* hist) {
  const int lane = threadIdx.x & 31;
  constexpr int kBits = 8 * (int)sizeof(V);
  V prefix = 0, pmask = 0;
  uint32_t need = (uint32_t)r;
  for (int pass = 0; pass < max_passes && pass < kBits / 8; ++pass) {
    const int shift = kBits - 8 * (pass + 1);
#pragma unroll
    for (int j = 0; j < 8; ++j) hist[lane + 32 * j] = 0u;
    __syncwarp();
    for (int i = lane; i < n; i += 32) {
      const V v = a[i];
      if ((v & pmask) == prefix) atomicAdd(&hist[(uint32_t)((v >> shift) & 0xFFu)], 1u);
    }
    __syncwarp();
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
    uint32_t d = 0, dabove = 0, din = 0;
    const bool mine = above < need && need <= incl;
    if (mine) {
      uint32_t acc = above;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (acc + c[j] >= need) {
          d = 255u - 8u * (uint32_t)lane - (uint32_t)j;
          dabove = acc;
          din = c[j];
          break;
        }
        acc += c[j];
      }
    }
    const int src = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
    d = __shfl_sync(0xffffffffu, d, src);
    dabove = __shfl_sync(0xffffffffu, dabove, src);
    din = __shfl_sync(0xffffffffu, din, src);
    need -= dabove;
    prefix |= (V)d << shift;
    pmask |= (V)0xFFu << shift;
    __syncwarp();
    if (din == need || din <= loose) break;
  }
  return prefix;
}

template <int THREADS, typename IdxMap>
FM_DEV void block_topk(const float* __restrict__ row, int n, int k, IdxMap idx_map, int32_t* __restrict__ idx_out,
                       float* __restrict__ score_out, TopkFastSmem<THREADS>& sm) {
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
  unsigned long long theta = 0ull;
  if (n > kTopkCap) {
    for (int i = tid; i < kTopkSample; i += THREADS) {
      const int run = i >> 6, off = i & 63;
      const int j = (int)(((long long)run * (n - 64)) / (kTopkRuns - 1)) + off;
      sm.u.sample[i] = ((unsigned long long)float_key(__ldg(row + j)) << 32) | (uint32_t)(~(uint32_t)j);
    }
    __syncthreads();
    int r = (int)(((long long)5 * kk * kTopkSample) / (2 * (long long)n));  // ~2.5 k candidates
    r = r < 1 ? 1 : (r > kTopkSample ? kTopkSample : r);
    if (tid < 32) {
      const unsigned long long t = warp_radix_select<unsigned long long>(sm.u.sample, kTopkSample, r, 8, 8u, sm.whist);
      if (tid == 0) sm.wsel = t;
    }
    __syncthreads();
    theta = sm.wsel;
  }
  if (tid == 0) {
    sm.count = 0;
    sm.overflow = 0;
  }
  __syncthreads();
  // ---- 2. filter pass ---------------------------------------------------------
  // A score can only pass if score >= theta's score (as floats: -0 compares
  // equal to +0 like its key); the composite then decides ties by index.  A
  // threshold at -inf (rows dominated by -inf/NaN) cannot be tested as a float
  // because NaN ranks as -inf: then every score goes to the composite test.
  const uint32_t theta_key = (uint32_t)(theta >> 32);
  const bool take_all = theta == 0ull || theta_key <= 0x007FFFFFu;
  const float theta_f = take_all ? -INFINITY : key_float(theta_key);
  auto push = [&](bool maybe, float v, int i) {
    if (maybe) {
      const unsigned long long c = ((unsigned long long)float_key(v) << 32) | (uint32_t)(~(uint32_t)i);
      if (c >= theta) {
        const uint32_t slot = atomicAdd(&sm.count, 1u);
        if (slot < (uint32_t)kTopkCap)
          sm.cand[slot] = c;
        else
          sm.overflow = 1;
      }
    }
  };
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  const int n4 = vec ? n / 4 : 0;
  const float4* row4 = reinterpret_cast<const float4*>(row);
  for (int i40 = 0; i40 < n4; i40 += THREADS * 4) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i4 = i40 + u * THREADS + tid;
      v[u] = i4 < n4 ? __ldg(row4 + i4) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i4 = i40 + u * THREADS + tid;
      const bool in = i4 < n4;
      push(in && (take_all || v[u].x >= theta_f), v[u].x, 4 * i4);
      push(in && (take_all || v[u].y >= theta_f), v[u].y, 4 * i4 + 1);
      push(in && (take_all || v[u].z >= theta_f), v[u].z, 4 * i4 + 2);
      push(in && (take_all || v[u].w >= theta_f), v[u].w, 4 * i4 + 3);
    }
  }
  for (int i = 4 * n4 + tid; i < n; i += THREADS) {
    const float v = __ldg(row + i);
    push(take_all || v >= theta_f, v, i);
  }
  __syncthreads();
  const int cnt = (int)sm.count;
  if (sm.overflow || cnt < kk) {
    __syncthreads();
    block_topk_radix<THREADS>(row, n, k, idx_map, idx_out, score_out, sm.radix);
    return;
  }
  // ---- 3. exact select among the candidates -------------------------------------
  if (tid < 32) {
    const unsigned long long t = warp_radix_select<unsigned long long>(sm.cand, cnt, kk, 8, 0u, sm.whist);
    if (tid == 0) sm.wsel = t;
  }
  __syncthreads();
  const unsigned long long T = sm.wsel;
  if (n <= kTopkBitmapN) {
    // mark the selected indices in a bitmap, then emit them in index order
    // with one block-wide prefix sum over the bitmap words
    const int words = (n + 31) >> 5;
    for (int i = tid; i < words; i += THREADS) sm.u.bitmap[i] = 0u;
    __syncthreads();
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
    uint32_t pos = block_excl_scan<THREADS>(mine, sm.radix.warp_tot, &tot);
    for (int j = 0; j < per && w0 + j < words; ++j) {
      uint32_t bits = sm.u.bitmap[w0 + j];
      while (bits) {
        const int b = __ffs(bits) - 1;
        bits &= bits - 1;
        const int i = ((w0 + j) << 5) + b;
        idx_out[pos] = idx_map(i);
        if (score_out) score_out[pos] = key_float(float_key(__ldg(row + i)));
        ++pos;
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

}  // namespace fm

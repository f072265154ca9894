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

// Select over row[0..n) (n >= 0).  idx_map(i) gives the id written for
// candidate i.  Writes k entries of idx_out / score_out (score_out may be
// null).  All THREADS threads of the block must call this.
template <int THREADS, typename IdxMap>
FM_DEV void block_topk(const float* __restrict__ row, int n, int k, IdxMap idx_map, int32_t* __restrict__ idx_out,
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

// paged.cu -- native lightning-indexer scoring over the resident 64-chunk
// pages, followed by the top-k select.
//
// Computes, for query qi and resident page-table entry r (the "FlashMemory-
// DeepSeek-V4" README, "Two-level recall algorithm" Level 2 and the
// "compressed_k format"; "DeepSeek-V4 CSA + HCA explained", sec. 3 CSA-1):
//     y[qi, chunk] = sum_h w[qi,h] * ReLU( scale[p,o] * (q[qi,h,:] . e4m3(k[p,o,:])) )
// with p = page_phys[qi,r], chunk id = page_logical[qi,r] * 64 + o, then the
// top-k of y by (y desc, id asc) (CSA-2), ids ascending.
//
// GB300 mapping (three launches):
//  1. paged_prep_kernel (one CTA per query): sorts the query's page-table
//     entries by logical page id (so candidate order == chunk-id order and the
//     result cannot depend on the table's row order), drops out-of-range and
//     repeated entries (flagging the device status word), and splits the bf16
//     query into two E4M3 terms per head: q_h = 2^e_h * (t1 + t2), with e_h a
//     power of two putting max|q_h| in (224, 448].  t1 = RNE_e4m3(q_h 2^-e_h),
//     t2 = RNE_e4m3(q_h 2^-e_h - t1); the pair reproduces every bf16 element
//     whose residual stays inside E4M3's range.  2^e_h is folded into w.
//  2. paged_score_kernel (persistent, one CTA per SM): TMA loads two E4M3 pages
//     (2 x 8 KB, SWIZZLE_128B) per 128-chunk tile straight into the UMMA A
//     operand -- no conversion pass; tcgen05.mma kind::f8f6f4 M=128 chunks x
//     N=64 heads x K=32, four K steps against t1 and four against t2 into
//     the same accumulator, so TMEM holds (t1 + t2).k per head.  The
//     producer warp issues a batch of tiles at once (lane i fills the stage
//     of tile i), four issuing threads and four epilogue warp groups take
//     tiles in turn.  The epilogue (thread = chunk) reads its 64 dots, applies
//     the chunk's scale, ReLU and w (from a per-warp shared-memory copy), and
//     writes y to the workspace.  Key copies carry an L2 evict-first hint and
//     score stores an evict-last hint, so the scores are still in L2 when
//     the top-k reads them.
//  3. the block top-k (topk.cuh), mapping candidate i to its chunk id.
#include <math.h>

#include "fm_common.cuh"
#include "fm_internal.h"
#include "fp8.cuh"

namespace fm {
namespace {

constexpr int kPage = 64;
constexpr int kM = 128;                  // chunks per tile = 2 pages
constexpr int kHeads = 64;
constexpr int kDim = 128;                // bytes per E4M3 key row
constexpr int kPageBytes = kPage * kDim; // 8 KB
constexpr int kTileBytes = kM * kDim;    // 16 KB
constexpr int kQBytes = 2 * kHeads * kDim;  // t1 rows 0..63, t2 rows 64..127
constexpr int kMaxR = FM_PAGED_MAX_R;  // 4096 pages: a 1M-token request's whole history
constexpr int kMaxStages = 12;
constexpr int kEpiGroups = 4;          // epilogue warp groups, taking tiles in turn
constexpr int kMmaWarps = 4;           // UMMA issuers, taking tiles in turn (issuer m owns accumulator m)
constexpr int kFirstEpiWarp = 1 + kMmaWarps;
constexpr int kThreads = kFirstEpiWarp * 32 + kEpiGroups * 128;
constexpr int kAccBufs = 4;
constexpr int kAccCols = kHeads;  // one column per head: the t1 and t2 MMAs accumulate into it
constexpr uint32_t kTmemCols = kAccBufs * kAccCols;
constexpr int kPrepThreads = 256;

// L2 priorities.  The keys are read once per call and the scores are read
// back by the top-k right after: the key copies go in as evict-first and the
// score stores as evict-last, so the [Q, R*64] score block (62 MB for 630
// queries x 384 pages) stays in the 129 MB L2 for the top-k instead of being
// evicted by the key stream.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t x,
                                                 int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, "
      "%4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                               uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// Programmatic dependent launch: the prep kernel lets the scorer launch
// once every prep CTA has started; the scorer sets up its barriers, TMEM and
// tensor-map prefetches, then waits for the prep grid's completion (and its
// memory) before any role reads the prep's output.  The top-k launched after
// the scorer waits the same way.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void st_f32_hint(float* addr, float v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(addr), "f"(v), "l"(policy) : "memory");
}

// --------------------------------------------------------------------------
// 1. prep: sort pages, validate, split q
// --------------------------------------------------------------------------

// THREADS: 256; 1024 for tables longer than 1024 entries when the queries
// fit one wave of such CTAs (the bitonic sort's passes then take four
// elements per thread instead of sixteen); 128 for tables of at most 256
// entries when the queries exceed one wave of 256-thread CTAs (ten such CTAs
// share an SM: 1520 queries per wave, so a 512K-context batch of 1260
// queries runs in one wave; each thread still has one compare-exchange per
// sorting stage).  The keys live in dynamic shared memory sized to the
// table (Rpow2 entries).
template <int THREADS>
constexpr int prep_ctas_per_sm() { return THREADS <= 128 ? 10 : (THREADS <= 256 ? 5 : 1); }

// Ascending bitonic sort of keys[0 .. 2 THREADS) with thread t holding
// elements 2t and 2t+1 in registers: a compare-exchange at distance j joins
// them inside the thread (j = 1), with lane t ^ j/2 of the same warp through
// shuffles (j <= 32), or through shared memory (j >= 64), so only the
// stages at distance 64 and more (six of 45 for 512 keys) pay block
// barriers.  The lower element of a pair keeps the minimum where the block
// of k2 elements it sits in is ascending.  Ends with keys[] sorted.
template <int THREADS>
__device__ __forceinline__ void bitonic_sort_pairs(unsigned long long* keys) {
  constexpr int N = 2 * THREADS;
  const int e0 = 2 * (int)threadIdx.x;
  unsigned long long v0 = keys[e0], v1 = keys[e0 + 1];
  for (int k2 = 2; k2 <= N; k2 <<= 1) {
    const bool asc = (e0 & k2) == 0;
    for (int j = k2 >> 1; j > 0; j >>= 1) {
      if (j == 1) {
        const unsigned long long lo = v0 < v1 ? v0 : v1, hi = v0 < v1 ? v1 : v0;
        v0 = asc ? lo : hi;
        v1 = asc ? hi : lo;
        continue;
      }
      unsigned long long p0, p1;
      if (j <= 32) {
        p0 = __shfl_xor_sync(0xffffffffu, v0, j >> 1);
        p1 = __shfl_xor_sync(0xffffffffu, v1, j >> 1);
      } else {
        keys[e0] = v0;
        keys[e0 + 1] = v1;
        __syncthreads();
        p0 = keys[e0 ^ j];
        p1 = keys[(e0 + 1) ^ j];
        __syncthreads();
      }
      const bool keep_min = ((e0 & j) == 0) == asc;  // both elements share bit j (j >= 2)
      v0 = keep_min ? (v0 < p0 ? v0 : p0) : (v0 < p0 ? p0 : v0);
      v1 = keep_min ? (v1 < p1 ? v1 : p1) : (v1 < p1 ? p1 : v1);
    }
  }
  keys[e0] = v0;
  keys[e0 + 1] = v1;
  __syncthreads();
}

template <int THREADS>
__global__ void __launch_bounds__(THREADS, prep_ctas_per_sm<THREADS>())
    paged_prep_kernel(const uint16_t* __restrict__ q, const float* __restrict__ w,
                      const int32_t* __restrict__ page_phys, const int32_t* __restrict__ page_logical,
                      const int32_t* __restrict__ n_res, int R, int64_t P, int Rpow2,
                      const uint32_t* __restrict__ res_mask, int64_t mask_ld, int mask_group,
                      int32_t* __restrict__ s_logical, int32_t* __restrict__ s_phys,
                      int32_t* __restrict__ nres_eff, int32_t* __restrict__ n_valid,
                      unsigned long long* __restrict__ pmask, int32_t* __restrict__ pprefix,
                      uint8_t* __restrict__ qsplit, float* __restrict__ wq, unsigned int* __restrict__ status,
                      bool split) {
  extern __shared__ unsigned long long keys[];  // [Rpow2]
  __shared__ uint32_t warp_tot[THREADS / 32];
  grid_dep_launch_dependents();
  const int qi = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the query and head weights are loaded first, so that their latency
  // overlaps the page-table sort (warp i splits heads i, i + THREADS/32, ...;
  // at most eight heads' loads in flight per warp, the rest after the sort)
  constexpr int kWarps = THREADS / 32, kHeadsPerWarp = kHeads / kWarps;
  constexpr int kEarly = kHeadsPerWarp < 8 ? kHeadsPerWarp : 8;
  uint2 qraw[kEarly];
  float wraw[kEarly];
#pragma unroll
  for (int i = 0; i < kEarly; ++i) {
    if (split) qraw[i] = load_head_slice(q + (int64_t)qi * kHeads * kDim, warp + i * kWarps);
    wraw[i] = __ldg(w + (int64_t)qi * kHeads + warp + i * kWarps);
  }
  int nr = R;
  if (n_res != nullptr) {
    const int v = n_res[qi];
    nr = v < 0 ? 0 : (v > R ? R : v);
  }
  for (int i = tid; i < Rpow2; i += THREADS)
    keys[i] = i < nr ? (((unsigned long long)(uint32_t)page_logical[(int64_t)qi * R + i] << 32) | (uint32_t)i)
                     : ~0ull;
  __syncthreads();
  // bitonic sort, ascending: with two keys per thread in registers where the
  // table fits that exactly, else each stage's Rpow2 / 2 compare-exchange
  // pairs indexed directly in shared memory (pair t joins element lo =
  // 2j (t / j) + t % j with lo + j, so no thread idles on the upper element)
  if (Rpow2 == 2 * THREADS) {
    bitonic_sort_pairs<THREADS>(keys);
  } else {
    for (int k2 = 2; k2 <= Rpow2; k2 <<= 1)
      for (int j = k2 >> 1; j > 0; j >>= 1) {
        for (int t = tid; t < Rpow2 / 2; t += THREADS) {
          const int lo = ((t & ~(j - 1)) << 1) | (t & (j - 1)), hi = lo + j;  // j is a power of two
          const unsigned long long a = keys[lo], b = keys[hi];
          if ((a > b) == ((lo & k2) == 0)) {
            keys[lo] = b;
            keys[hi] = a;
          }
        }
        __syncthreads();
      }
  }
  uint32_t base = 0;
  for (int i0 = 0; i0 < Rpow2; i0 += THREADS) {
    const int i = i0 + tid;
    uint32_t valid = 0;
    int32_t lg = 0, ph = 0;
    if (i < nr) {
      lg = (int32_t)(keys[i] >> 32);
      ph = page_phys[(int64_t)qi * R + (uint32_t)keys[i]];
      const bool dup = i > 0 && (keys[i - 1] >> 32) == (keys[i] >> 32);
      const bool range_ok = ph >= 0 && ph < P && lg >= 0 && lg < (1 << 25);
      if (dup) atomicOr(status, FM_DEV_DUP_PAGE);
      if (!range_ok) atomicOr(status, FM_DEV_PAGE_RANGE);
      valid = (!dup && range_ok) ? 1u : 0u;
    }
    // block exclusive scan of `valid`
    uint32_t x = valid;
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    uint32_t before = 0, total = 0;
    for (int wi = 0; wi < THREADS / 32; ++wi) {
      if (wi < warp) before += warp_tot[wi];
      total += warp_tot[wi];
    }
    if (valid) {
      s_logical[(int64_t)qi * R + base + before + x - 1] = lg;
      s_phys[(int64_t)qi * R + base + before + x - 1] = ph;
    }
    base += total;
    __syncthreads();
  }
  if (res_mask == nullptr) {
    if (tid == 0) {
      nres_eff[qi] = (int32_t)base;
      n_valid[qi] = (int32_t)base * kPage;
    }
  } else {
    // Level-2 resident set: page j's 64-bit mask of resident chunks (words
    // past the mask row read as 0) and the prefix count of resident chunks
    // before it; the scorer writes only resident chunks, compacted.  Pages
    // past the listed ones get an empty mask and the final count.
    const uint32_t* mrow = res_mask + (int64_t)(qi / mask_group) * mask_ld;
    uint32_t run = 0;
    for (int j0 = 0; j0 < R; j0 += THREADS) {
      const int j = j0 + tid;
      unsigned long long m = 0ull;
      if (j < (int)base) {
        const int64_t wd = 2 * (int64_t)s_logical[(int64_t)qi * R + j];
        const uint32_t lo = wd < mask_ld ? __ldg(mrow + wd) : 0u;
        const uint32_t hi = wd + 1 < mask_ld ? __ldg(mrow + wd + 1) : 0u;
        m = ((unsigned long long)hi << 32) | lo;
      }
      const uint32_t c = (uint32_t)__popcll(m);
      uint32_t x = c;
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) warp_tot[warp] = x;
      __syncthreads();
      uint32_t before = 0, total = 0;
      for (int wi = 0; wi < THREADS / 32; ++wi) {
        if (wi < warp) before += warp_tot[wi];
        total += warp_tot[wi];
      }
      if (j < R) {
        pmask[(int64_t)qi * R + j] = m;
        pprefix[(int64_t)qi * (R + 1) + j] = (int32_t)(run + before + x - c);
      }
      run += total;
      __syncthreads();
    }
    if (tid == 0) {
      pprefix[(int64_t)qi * (R + 1) + R] = (int32_t)run;
      nres_eff[qi] = (int32_t)base;
      n_valid[qi] = (int32_t)run;
    }
  }
  // q split (E4M3 pool): q_h = 2^e_h (t1 + t2), 2^e_h folded into w; a bf16
  // pool takes q as it is and w unchanged
  uint8_t* t1 = qsplit + (int64_t)qi * 2 * kHeads * kDim;
#pragma unroll
  for (int i0 = 0; i0 < kHeadsPerWarp; i0 += kEarly) {
    if (i0 > 0) {
#pragma unroll
      for (int i = 0; i < kEarly; ++i) {
        if (split) qraw[i] = load_head_slice(q + (int64_t)qi * kHeads * kDim, warp + (i0 + i) * kWarps);
        wraw[i] = __ldg(w + (int64_t)qi * kHeads + warp + (i0 + i) * kWarps);
      }
    }
#pragma unroll
    for (int i = 0; i < kEarly; ++i) {
      const int h = warp + (i0 + i) * kWarps;
      if (split)
        split_head(qraw[i], wraw[i], t1 + (int64_t)h * kDim, t1 + (int64_t)(kHeads + h) * kDim,
                   wq + (int64_t)qi * kHeads + h);
      else if (lane == 0)
        wq[(int64_t)qi * kHeads + h] = wraw[i];
    }
  }
}

// --------------------------------------------------------------------------
// 2. persistent tcgen05 scorer
// --------------------------------------------------------------------------

struct ScoreParams {
  const int32_t* s_phys;
  const int32_t* nres_eff;
  const unsigned long long* pmask;  // resident-chunk masks per listed page, or null (every chunk)
  const int32_t* pprefix;           // resident chunks before each page (compacted write positions)
  const float* k_scale;
  const float* wq;
  float* scores;  // [Q, R*64]
  unsigned int* status;
  int64_t total_tiles;
  int tiles_per_q;
  int R;
  int stages;
};

// kMasked: write only the resident chunks of each page, compacted (the
// Level-2 resident mask); a separate instantiation so that the unmasked
// kernel's code is unchanged by it.
// kBf16: the pool holds bf16 keys (no scale).  A stage is then two 16 KB
// K-halves of the 128-chunk tile (elements 0-63 and 64-127 of every key, one
// SWIZZLE_128B box of 64 rows per page and half), q is the caller's bf16
// query in two 8 KB K-halves, and each tile is eight tcgen05.mma kind::f16
// M128 N64 K16 into the head accumulator; the epilogue is the E4M3 one with
// the scale fixed at 1.
template <bool kMasked, bool kBf16>
__global__ void __launch_bounds__(kThreads, 1)
    paged_score_kernel(const __grid_constant__ CUtensorMap tmap_pool, const __grid_constant__ CUtensorMap tmap_q,
                       const ScoreParams p) {
  constexpr int kStageBytes = kBf16 ? 2 * kTileBytes : kTileBytes;  // key bytes per stage
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_smem = smem;                       // 16 KB
  uint8_t* a_smem = smem + kQBytes;             // stages x kStageBytes
  float* scale_smem = reinterpret_cast<float*>(a_smem + p.stages * kStageBytes);          // stages x 128 (E4M3)

  __shared__ __align__(8) uint64_t bar_full[kMaxStages], bar_empty[kMaxStages];
  __shared__ __align__(8) uint64_t bar_tfull[kAccBufs], bar_tempty[kAccBufs], bar_qfull, bar_qempty, bar_drain;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int stages = p.stages;
  const int64_t t_begin = p.total_tiles * blockIdx.x / gridDim.x;
  const int64_t t_end = p.total_tiles * (blockIdx.x + 1) / gridDim.x;
  const int64_t ld = (int64_t)p.R * kPage;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 128);  // the epilogue read the scales after the MMA finished
    }
    for (int i = 0; i < kAccBufs; ++i) {
      mbar_init(&bar_tfull[i], 1);
      mbar_init(&bar_tempty[i], 128);
    }
    mbar_init(&bar_qfull, 1);
    mbar_init(&bar_qempty, kMmaWarps);
    mbar_init(&bar_drain, kMmaWarps);  // each issuer arrives once its MMAs are done
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tmap_pool);
    tma_prefetch(&tmap_q);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dep_wait();  // the page tables, split query and weights come from the prep kernel
  const uint32_t tmem_base = tmem_slot;

  if (warp == 0) {
    // -------------------------------- producer (whole warp) ------------------
    // Tiles are issued in batches of up to kBatch consecutive tiles of one
    // query: lane i waits for the stage of the batch's i-th tile and issues its
    // copies, so the per-copy issue latency is paid once per batch.
    constexpr int kBatch = 8;
    const uint64_t stream_policy = l2_policy_evict_first();
    __shared__ int issued_ph[kMaxStages];
    for (int s = lane; s < kMaxStages; s += 32) issued_ph[s] = -1;
    uint32_t seq = 0, q_phase = 0;
    int q_issued = -1;
    int64_t cur_q = -1;
    int nres = 0;
    bool ok = true;
    int64_t qi = t_begin / p.tiles_per_q;
    int tile = (int)(t_begin % p.tiles_per_q);
    int64_t t = t_begin;
    __syncwarp();
    while (t < t_end) {
      // A new query's q is loaded after its first batch of key copies has
      // been issued: the copies wait only for stages the old query's
      // epilogues free, while the q slot waits until every issuer is done
      // with the old q, so issuing them first keeps the ring filling across
      // the query boundary instead of draining it.
      bool load_q = false;
      if (qi != cur_q) {
        nres = p.nres_eff[qi];
        cur_q = qi;
        load_q = nres > 0;
      }
      int nb = p.tiles_per_q - tile;
      if ((int64_t)nb > t_end - t) nb = (int)(t_end - t);
      if (nb > kBatch) nb = kBatch;
      // A batch never holds two uses of one stage: each lane's parity wait
      // on its stage's empty barrier is exact only if the stage's previous
      // use was issued (and its wait passed) in an earlier batch.  (With four
      // stages of bf16 tiles, lanes i and i + 4 of an eight-tile batch would
      // wait for consecutive uses of the same stage at once, and the later
      // wait could pass on the phase two uses back.)
      if (nb > stages) nb = stages;
      const int my_tile = tile + lane;
      const bool valid = lane < nb && 2 * my_tile < nres;
      const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
      if (valid) {
        const uint32_t sq = seq + (uint32_t)__popc(vmask & ((1u << lane) - 1u));
        const uint32_t stage = sq % (uint32_t)stages, phase = (sq / (uint32_t)stages) & 1u;
        if (!mbar_wait(&bar_empty[stage], phase ^ 1u, &abort_flag, p.status)) {
          ok = false;
        } else {
          const int npg = nres - 2 * my_tile >= 2 ? 2 : 1;
          mbar_arrive_expect_tx(&bar_full[stage],
                                (uint32_t)(npg * (kBf16 ? 2 * kPageBytes : kPageBytes + kPage * 4)));
          for (int h = 0; h < npg; ++h) {
            // the sorted page table is in the workspace (L2-resident): one
            // load per page, issued by all lanes of the batch in parallel
            const int32_t ph = __ldg(p.s_phys + qi * p.R + 2 * my_tile + h);
            uint8_t* dst = a_smem + stage * kStageBytes + h * kPageBytes;
            if constexpr (kBf16) {  // rows h*64.. of both K-halves
              tma_load_2d_hint(dst, &tmap_pool, &bar_full[stage], 0, ph * kPage, stream_policy);
              tma_load_2d_hint(dst + kTileBytes, &tmap_pool, &bar_full[stage], 64, ph * kPage, stream_policy);
            } else {
              tma_load_2d_hint(dst, &tmap_pool, &bar_full[stage], 0, ph * kPage, stream_policy);
              bulk_load_hint(scale_smem + stage * kM + h * kPage, p.k_scale + (int64_t)ph * kPage, kPage * 4,
                             &bar_full[stage], stream_policy);
            }
          }
          issued_ph[stage] = (int)phase;
        }
      }
      seq += (uint32_t)__popc(vmask);
      if (load_q && lane == 0 && ok) {
        if (q_issued >= 0) {  // every issuer has committed its last MMA on the old q
          if (!mbar_wait(&bar_qempty, q_phase, &abort_flag, p.status)) ok = false;
          q_phase ^= 1;
        }
        if (ok) {
          mbar_arrive_expect_tx(&bar_qfull, (uint32_t)kQBytes);
          if constexpr (kBf16) {  // the two K-halves of the query's 64 head rows
            tma_load_2d(q_smem, &tmap_q, &bar_qfull, 0, (int32_t)(qi * kHeads));
            tma_load_2d(q_smem + kQBytes / 2, &tmap_q, &bar_qfull, 64, (int32_t)(qi * kHeads));
          } else {
            tma_load_2d(q_smem, &tmap_q, &bar_qfull, 0, (int32_t)(qi * 2 * kHeads));
          }
          q_issued = (q_issued + 1) & 1;
        }
      }
      if (__any_sync(0xffffffffu, !ok)) break;
      t += nb;
      tile += nb;
      if (tile == p.tiles_per_q) {
        tile = 0;
        ++qi;
      }
    }
    __syncwarp();
    if (lane == 0 && abort_flag) {  // let copies already in flight land before the CTA exits
      for (int s = 0; s < stages; ++s)
        if (issued_ph[s] >= 0) mbar_wait_drain(&bar_full[s], (uint32_t)issued_ph[s]);
      if (q_issued >= 0) mbar_wait_drain(&bar_qfull, (uint32_t)q_issued);
    }
  } else if (warp < kFirstEpiWarp) {
    if (lane == 0) {
      // ---------------------------- UMMA issuers ------------------------------
      // Issuer m takes the tiles with sequence number = m (mod 4) and owns
      // accumulator m, so the issuers' barrier waits and commits overlap each
      // other's MMAs.
      const uint32_t me = (uint32_t)(warp - 1);
      const uint32_t idesc = kBf16 ? idesc_bf16_f32(kM, kHeads) : idesc_e4m3_f32(kM, kHeads);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0, q_phase = 0, seq = 0;
      int64_t cur_q = -1;
      int nres = 0;
      bool have_q = false, ok = true;
      const uint64_t a_desc0 = sdesc_sw128(smem_u32(a_smem));
      const uint64_t b_desc0 = sdesc_sw128(smem_u32(q_smem));
      int64_t qi = t_begin / p.tiles_per_q;
      int tile = (int)(t_begin % p.tiles_per_q) - 1;
      for (int64_t t = t_begin; t < t_end && ok; ++t) {
        if (++tile == p.tiles_per_q) {
          tile = 0;
          ++qi;
        }
        if (qi != cur_q) {
          nres = p.nres_eff[qi];
          cur_q = qi;
          if (nres > 0) {
            if (have_q) umma_commit(&bar_qempty);
            if (!mbar_wait(&bar_qfull, q_phase, &abort_flag, p.status)) break;
            q_phase ^= 1;
            have_q = true;
            tc_fence_after();
          }
        }
        if (2 * tile >= nres) continue;
        if ((seq++ % kMmaWarps) == me) {
          if (!mbar_wait(&bar_tempty[acc], acc_phase ^ 1u, &abort_flag, p.status)) break;
          if (!mbar_wait(&bar_full[stage], phase, &abort_flag, p.status)) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * kAccCols;
          // descriptor start-address field counts 16-byte units
          const uint64_t a_desc = a_desc0 + (uint64_t)(stage * (kStageBytes >> 4));
          if constexpr (kBf16) {
            // K steps of 16 elements (32 bytes): four in each K-half; the
            // halves are 16 KB (keys) and 8 KB (query) apart
#pragma unroll
            for (int k = 0; k < 8; ++k)
              umma_bf16_ss(d_tmem, a_desc + (k >> 2) * (kTileBytes >> 4) + (k & 3) * 2,
                           b_desc0 + (k >> 2) * ((kQBytes / 2) >> 4) + (k & 3) * 2, idesc, k != 0 ? 1u : 0u);
          } else {
            // the t2 rows start 8 KB (eight 1 KB swizzle atoms) after the t1 rows
            constexpr uint64_t kT2 = (kHeads * kDim) >> 4;
#pragma unroll
            for (int k = 0; k < kDim / 32; ++k)
              umma_e4m3_ss(d_tmem, a_desc + 2 * k, b_desc0 + 2 * k, idesc, k != 0 ? 1u : 0u);
#pragma unroll
            for (int k = 0; k < kDim / 32; ++k)
              umma_e4m3_ss(d_tmem, a_desc + 2 * k, b_desc0 + kT2 + 2 * k, idesc, 1u);
          }
          umma_commit(&bar_tfull[acc]);  // also frees the stage: its epilogue releases it
        }
        if (++stage == (uint32_t)stages) {
          stage = 0;
          phase ^= 1u;
        }
        if (++acc == (uint32_t)kAccBufs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      umma_commit(&bar_drain);
      mbar_wait_drain(&bar_drain, 0);
    }
  } else {
    // -------------------------------- epilogue -------------------------------
    // Four groups of four warps (one per TMEM lane quadrant) take the tiles in
    // turn, group g always reading accumulator g; every thread owns one chunk
    // row of its group's tiles.
    const int quad = warp & 3;
    const int group = (warp - kFirstEpiWarp) >> 2;
    const int row = quad * 32 + lane;
    // one copy of the current query's head weights per epilogue warp, so a
    // warp refreshes its own copy with __syncwarp alone
    __shared__ __align__(16) float w_smem[kEpiGroups * 4][kHeads];
    float* w_mine = w_smem[warp - kFirstEpiWarp];
    // Group g takes the CTA's live tiles (those with 2 tile < n_res) with
    // sequence number g, g + 4, ..., so its accumulator is g, and its stage
    // and the two phases step by four tiles each time (the stage count is a
    // multiple of four).  It walks each query's own tiles with an int32 loop;
    // the weights and the query's live range are set once per query.
    const uint32_t acc = (uint32_t)group;
    uint32_t acc_phase = 0, stage = (uint32_t)group, phase = 0;
    uint32_t seq_base = 0;  // live tiles of the CTA before the current query's
    bool aborted = false;
    const uint64_t keep_policy = l2_policy_evict_last();
    for (int64_t it = t_begin; it < t_end && !aborted;) {
      const int64_t qi = it / p.tiles_per_q;
      const int tile0 = (int)(it - qi * p.tiles_per_q);
      const int tile_end = (t_end - it < (int64_t)(p.tiles_per_q - tile0)) ? tile0 + (int)(t_end - it) : p.tiles_per_q;
      it += tile_end - tile0;
      const int nres = p.nres_eff[qi];
      const int live_end = tile_end < (nres + 1) / 2 ? tile_end : (nres + 1) / 2;
      const int live = live_end > tile0 ? live_end - tile0 : 0;
      if (live == 0) continue;
      __syncwarp();
      for (int i = lane; i < kHeads; i += 32) w_mine[i] = __ldg(p.wq + qi * kHeads + i);
      __syncwarp();
      for (int k = (int)(((uint32_t)group - seq_base) & (kEpiGroups - 1)); k < live; k += kEpiGroups) {
        const int tile = tile0 + k;
        const int j = 2 * tile + (row >> 6);
        const bool valid = j < nres;
        if (!mbar_wait(&bar_tfull[acc], acc_phase, &abort_flag, p.status) ||
            // the stage's scales landed with its full barrier (already complete)
            !mbar_wait(&bar_full[stage], phase, &abort_flag, p.status)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const float sc = valid ? (kBf16 ? 1.f : scale_smem[stage * kM + row]) : 0.f;
        mbar_arrive(&bar_empty[stage]);
        const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * kAccCols;
        const float4* wl = reinterpret_cast<const float4*>(w_mine);
        float y = 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {  // 32 heads at a time keeps the thread within 80 registers
          uint32_t r[32];
          tmem_ld32(taddr + half * 32, r);
          tmem_ld_wait();
          if (half == 1) {
            tc_fence_before();
            mbar_arrive(&bar_tempty[acc]);  // the dots are in registers: the MMA may reuse the accumulator
          }
          // q_h . k = 2^e_h (t1 + t2) . k; 2^e_h is folded into w
          float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
          if (sc > 0.f) {  // ReLU(sc d) = sc ReLU(d): one multiply per chunk
#pragma unroll
            for (int h = 0; h < 32; h += 4) {
              const float4 wv = wl[half * 8 + h / 4];
              x0 = fmaf(wv.x, fmaxf(__uint_as_float(r[h]), 0.f), x0);
              x1 = fmaf(wv.y, fmaxf(__uint_as_float(r[h + 1]), 0.f), x1);
              x2 = fmaf(wv.z, fmaxf(__uint_as_float(r[h + 2]), 0.f), x2);
              x3 = fmaf(wv.w, fmaxf(__uint_as_float(r[h + 3]), 0.f), x3);
            }
            y += sc * ((x0 + x1) + (x2 + x3));
          } else {
#pragma unroll
            for (int h = 0; h < 32; h += 4) {
              const float4 wv = wl[half * 8 + h / 4];
              x0 = fmaf(wv.x, fmaxf(sc * __uint_as_float(r[h]), 0.f), x0);
              x1 = fmaf(wv.y, fmaxf(sc * __uint_as_float(r[h + 1]), 0.f), x1);
              x2 = fmaf(wv.z, fmaxf(sc * __uint_as_float(r[h + 2]), 0.f), x2);
              x3 = fmaf(wv.w, fmaxf(sc * __uint_as_float(r[h + 3]), 0.f), x3);
            }
            y += (x0 + x1) + (x2 + x3);
          }
        }
        if constexpr (kMasked) {
          if (valid) {
            const unsigned long long m = __ldg(p.pmask + qi * p.R + j);
            const int o = row & (kPage - 1);
            if ((m >> o) & 1ull)
              st_f32_hint(
                  p.scores + qi * ld + __ldg(p.pprefix + qi * (p.R + 1) + j) + __popcll(m & ((1ull << o) - 1ull)), y,
                  keep_policy);
          }
        } else {
          if (valid) st_f32_hint(p.scores + qi * ld + (int64_t)tile * kM + row, y, keep_policy);
        }
        acc_phase ^= 1u;
        stage += kEpiGroups;
        if (stage >= (uint32_t)stages) {
          stage -= (uint32_t)stages;
          phase ^= 1u;
        }
      }
      seq_base += (uint32_t)live;
    }
  }

  grid_dep_launch_dependents();  // the top-k may launch; it waits for this grid's completion
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct PagedWs {
  int32_t *s_logical, *s_phys, *nres_eff, *n_valid, *pprefix;
  unsigned long long* pmask;
  uint8_t* qsplit;
  float *wq, *scores;
  size_t bytes;
};

PagedWs paged_ws_layout(void* base, int Q, int R) {
  PagedWs w;
  uint8_t* b = static_cast<uint8_t*>(base);
  size_t off = 0;
  auto take = [&](size_t n) {
    uint8_t* p = b ? b + off : nullptr;
    off += align256(n);
    return p;
  };
  w.s_logical = reinterpret_cast<int32_t*>(take((size_t)Q * R * 4));
  w.s_phys = reinterpret_cast<int32_t*>(take((size_t)Q * R * 4));
  w.nres_eff = reinterpret_cast<int32_t*>(take((size_t)Q * 4));
  w.n_valid = reinterpret_cast<int32_t*>(take((size_t)Q * 4));
  w.pmask = reinterpret_cast<unsigned long long*>(take((size_t)Q * R * 8));
  w.pprefix = reinterpret_cast<int32_t*>(take((size_t)Q * (R + 1) * 4));
  w.qsplit = take((size_t)Q * kQBytes);
  w.wq = reinterpret_cast<float*>(take((size_t)Q * kHeads * 4));
  w.scores = reinterpret_cast<float*>(take((size_t)Q * R * kPage * 4));
  w.bytes = off;
  return w;
}

}  // namespace

size_t paged_workspace_bytes(int Q, int R) { return paged_ws_layout(nullptr, Q, R).bytes; }

fm_status launch_paged(const PagedArgs& a, int num_sms, unsigned int* status, cudaStream_t stream) {
  if (a.Q == 0) return FM_OK;
  PagedWs ws = paged_ws_layout(a.workspace, a.Q, a.R);
  int Rpow2 = 1;
  while (Rpow2 < a.R) Rpow2 <<= 1;
  // Tables longer than 1024 entries sort faster per query with 1024 threads,
  // but only two such CTAs fit an SM: when the queries exceed one wave of
  // them, 256 threads (five per SM) finish the batch sooner.
  const bool wide = a.R > 1024 && a.Q <= 2 * num_sms;
  const bool bf16 = a.key_dtype == FM_DTYPE_BF16;
  // Tables of at most 256 entries: 128-thread CTAs when the queries exceed
  // one wave of 256-thread CTAs.
  const bool narrow = !wide && Rpow2 <= 256 && a.Q > prep_ctas_per_sm<kPrepThreads>() * num_sms;
  auto prep = wide ? paged_prep_kernel<1024> : (narrow ? paged_prep_kernel<128> : paged_prep_kernel<kPrepThreads>);
  const int prep_threads = wide ? 1024 : (narrow ? 128 : kPrepThreads);
  prep<<<a.Q, prep_threads, (size_t)Rpow2 * 8, stream>>>(a.q, a.w, a.page_phys, a.page_logical, a.n_res, a.R, a.P,
                                                      Rpow2, a.res_mask, a.mask_ld, a.mask_group, ws.s_logical,
                                                      ws.s_phys, ws.nres_eff, ws.n_valid, ws.pmask, ws.pprefix,
                                                      ws.qsplit, ws.wq, status, !bf16);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "paged prep: launch: %s", cudaGetErrorString(e));

  CUtensorMap tmap_pool, tmap_q;
  if (bf16) {
    // pool rows of 128 bf16 (256 bytes); boxes of 64 elements x 64 rows, one
    // per page and K-half; the caller's q [Q*64, 128] bf16 the same way
    const uint64_t strides[1] = {(uint64_t)kDim * 2};
    const uint32_t box[2] = {64u, (uint32_t)kPage};
    const uint64_t pdims[2] = {(uint64_t)kDim, (uint64_t)a.P * kPage};
    fm_status st = make_tmap(&tmap_pool, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.k_pool, pdims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != FM_OK) return st;
    const uint64_t qdims[2] = {(uint64_t)kDim, (uint64_t)a.Q * kHeads};
    const uint32_t qbox[2] = {64u, (uint32_t)kHeads};
    st = make_tmap(&tmap_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, qdims, strides, qbox,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != FM_OK) return st;
  } else {
    {
      const uint64_t dims[2] = {(uint64_t)kDim, (uint64_t)a.P * kPage};
      const uint64_t strides[1] = {(uint64_t)kDim};
      const uint32_t box[2] = {(uint32_t)kDim, (uint32_t)kPage};
      fm_status st = make_tmap(&tmap_pool, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.k_pool, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_128B);
      if (st != FM_OK) return st;
    }
    {
      const uint64_t dims[2] = {(uint64_t)kDim, (uint64_t)a.Q * 2 * kHeads};
      const uint64_t strides[1] = {(uint64_t)kDim};
      const uint32_t box[2] = {(uint32_t)kDim, (uint32_t)(2 * kHeads)};
      fm_status st = make_tmap(&tmap_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, ws.qsplit, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_128B);
      if (st != FM_OK) return st;
    }
  }
  const int tiles_per_q = (a.R + 1) / 2;
  const int64_t total = (int64_t)a.Q * tiles_per_q;
  const int smem_cap = 227 * 1024 - 6 * 1024;  // less the kernel's static shared memory
  const int fixed = 1024 + kQBytes;
  const int per_stage = bf16 ? 2 * kTileBytes : kTileBytes + kM * 4;
  int stages = (smem_cap - fixed) / per_stage;
  if (stages > kMaxStages) stages = kMaxStages;
  // Tile i uses stage i % stages and is consumed by issuer / epilogue group
  // i % 4.  With stages a multiple of 4 every stage has a single consumer, so
  // a consumer's parity wait on a stage's full barrier can only see that
  // stage's previous fill completed (it consumed that fill itself).  Key
  // copies may complete out of order; with another consumer's fill as the
  // previous use, a wait could pass on the previous phase while that fill is
  // still in flight.
  stages -= stages % kMmaWarps;
  const int smem = fixed + stages * per_stage;

  ScoreParams p;
  p.s_phys = ws.s_phys;
  p.nres_eff = ws.nres_eff;
  p.pmask = a.res_mask != nullptr ? ws.pmask : nullptr;
  p.pprefix = ws.pprefix;
  p.k_scale = a.k_scale;
  p.wq = ws.wq;
  p.scores = ws.scores;
  p.status = status;
  p.total_tiles = total;
  p.tiles_per_q = tiles_per_q;
  p.R = a.R;
  p.stages = stages;
  auto* score_kernel = a.res_mask != nullptr ? (bf16 ? paged_score_kernel<true, true> : paged_score_kernel<true, false>)
                                             : (bf16 ? paged_score_kernel<false, true> : paged_score_kernel<false, false>);
  e = cudaFuncSetAttribute(score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "paged: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  const int grid = (int)(total < num_sms ? total : num_sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, score_kernel, tmap_pool, tmap_q, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "paged score: launch: %s", cudaGetErrorString(e));

  // ids: logical chunk ids, or reserve cells (the fused remap)
  const int32_t* ids = a.id_mode == 1 ? ws.s_phys : ws.s_logical;
  return launch_topk_rows(ws.scores, (int64_t)a.R * kPage, ws.n_valid, a.Q, a.R * kPage, a.k, ids, a.R,
                          a.res_mask != nullptr ? ws.pprefix : nullptr, a.res_mask != nullptr ? ws.pmask : nullptr,
                          a.idx_out, a.score_out, stream);
}

}  // namespace fm

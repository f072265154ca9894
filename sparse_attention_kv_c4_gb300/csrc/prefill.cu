// prefill.cu -- many-query indexer scoring against dense chunk keys under the
// causal chunk limit, followed by the top-k select.
//
// Computes ("DeepSeek-V4 CSA + HCA explained", sec. 3 CSA-1 / CSA-2; c4 chunk
// s covers tokens 4s..4s+3, sec. 1 and 8):
//     Y[t,s] = sum_h w[t,h] * ReLU(q[t,h,:] . K[s,:]),
//     candidates of query t: s < min(S, floor(pos[t] / ratio)),
// then the top-k of each row by (Y desc, s asc), ids ascending.
//
// GB300 mapping.  This is the one real dense contraction of the indexer
// (T x 64 heads against S chunks, K = 128), so it runs on the 5th-generation
// tensor cores: a persistent CTA per SM owns a contiguous range of
// (query block of 4 tokens, 128-chunk tile) work items, keeps the block's
// q [256 rows = 4 tokens x 64 heads, 128] resident in shared memory (B
// operand) and streams key tiles [128 chunks x 128] (A operand, L2-resident
// after first touch) through a TMA ring; tcgen05.mma M=128 x N=256 x K=16
// accumulates D [128 chunks x 256] in TMEM, double-buffered (512 columns);
// two issuing threads alternate tiles so barrier latency overlaps MMAs.
// Sixteen epilogue warps (four per TMEM lane quadrant, one token each) load
// their row of D with both 32-column TMEM loads in flight, release the
// accumulator, and turn it into Y with fp32 max/FMA against the token's head
// weights (kept in shared memory per query block); tiles wholly past a
// block's causal limit are skipped.  The block top-k then reads
// each row up to its causal limit.  Called for the scores alone, a second
// small kernel writes -inf wherever s >= the token's limit (the score kernel
// itself is the same either way).
#include <math.h>

#include "fm_common.cuh"
#include "fm_internal.h"

namespace fm {
namespace {

constexpr int kM = 128;                   // chunks per tile
constexpr int kHeads = 64;
constexpr int kTok = 4;                   // query tokens per block
constexpr int kN = kTok * kHeads;         // 256
constexpr int kDim = 128;
constexpr int kTileBytes = kM * kDim * 2;    // 32 KB
constexpr int kAtomA = kM * 64 * 2;          // 16 KB
constexpr int kQBytes = kN * kDim * 2;       // 64 KB
constexpr int kAtomB = kN * 64 * 2;          // 32 KB
constexpr int kMaxStages = 8;
constexpr int kEpiWarps = 16;               // four per TMEM lane quadrant, one token each
constexpr int kMmaWarps = 2;                // two UMMA issuers, alternating tiles
constexpr int kFirstEpiWarp = 1 + kMmaWarps;
constexpr int kThreads = (kFirstEpiWarp + kEpiWarps) * 32;
constexpr uint32_t kTmemCols = 512;

struct Params {
  const float* w;
  const int64_t* pos;
  float* logits;
  int32_t* segmax;  // [T, seg_ld] segment maxima for the top-k, or null
  int64_t seg_ld;
  unsigned int* status;
  int64_t S;
  int64_t total_items;
  int T;
  int tiles_per_qb;
  int ratio;
  int stages;
};

FM_DEV int64_t causal_limit(int64_t pos, int64_t S, int ratio) {
  if (pos < 0) return 0;
  const int64_t l = pos / ratio;
  return l < S ? l : S;
}

// Largest causal limit among the tokens of query block qb.
FM_DEV int64_t block_limit(const Params& p, int64_t qb) {
  int64_t lim = 0;
  for (int j = 0; j < kTok; ++j) {
    const int64_t t = qb * kTok + j;
    if (t < p.T) {
      const int64_t l = causal_limit(__ldg(p.pos + t), p.S, p.ratio);
      lim = l > lim ? l : lim;
    }
  }
  return lim;
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_score_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                         const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_smem = smem;
  uint8_t* k_smem = smem + kQBytes;

  __shared__ __align__(8) uint64_t bar_full[kMaxStages], bar_empty[kMaxStages];
  __shared__ __align__(8) uint64_t bar_tfull[2], bar_tempty[2], bar_qfull, bar_qempty, bar_drain;
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(16) float w_smem[kEpiWarps][kHeads];  // each epilogue warp's token weights
  __shared__ int abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int stages = p.stages;
  const int64_t t_begin = p.total_items * blockIdx.x / gridDim.x;
  const int64_t t_end = p.total_items * (blockIdx.x + 1) / gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_tfull[i], 1);
      mbar_init(&bar_tempty[i], kEpiWarps * 32);
    }
    mbar_init(&bar_qfull, 1);
    mbar_init(&bar_qempty, kMmaWarps);
    mbar_init(&bar_drain, kMmaWarps);  // each issuer arrives once its MMAs are done
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tmap_k);
    tma_prefetch(&tmap_q);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------ TMA producer ------------------------------
      uint32_t stage = 0, phase = 0, q_phase = 0;
      int issued[kMaxStages];
      for (int s = 0; s < kMaxStages; ++s) issued[s] = -1;
      int q_issued = -1;
      int64_t cur_qb = -1, lim = 0;
      int64_t qb = t_begin / p.tiles_per_qb;
      int ct = (int)(t_begin % p.tiles_per_qb) - 1;
      for (int64_t it = t_begin; it < t_end; ++it) {
        if (++ct == p.tiles_per_qb) {
          ct = 0;
          ++qb;
        }
        if (qb != cur_qb) {
          cur_qb = qb;
          lim = block_limit(p, qb);
          if (lim > 0) {
            if (q_issued >= 0) {
              if (!mbar_wait(&bar_qempty, q_phase, &abort_flag, p.status)) break;
              q_phase ^= 1;
            }
            mbar_arrive_expect_tx(&bar_qfull, (uint32_t)kQBytes);
            for (int a = 0; a < 2; ++a)
              tma_load_2d(q_smem + a * kAtomB, &tmap_q, &bar_qfull, a * 64, (int32_t)(qb * kN));
            q_issued = (q_issued + 1) & 1;
          }
        }
        if ((int64_t)ct * kM >= lim) continue;
        if (!mbar_wait(&bar_empty[stage], phase ^ 1u, &abort_flag, p.status)) break;
        mbar_arrive_expect_tx(&bar_full[stage], (uint32_t)kTileBytes);
        for (int a = 0; a < 2; ++a)
          tma_load_2d(k_smem + stage * kTileBytes + a * kAtomA, &tmap_k, &bar_full[stage], a * 64, ct * kM);
        issued[stage] = (int)phase;
        if (++stage == (uint32_t)stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (abort_flag) {
        for (int s = 0; s < stages; ++s)
          if (issued[s] >= 0) mbar_wait_drain(&bar_full[s], (uint32_t)issued[s]);
        if (q_issued >= 0) mbar_wait_drain(&bar_qfull, (uint32_t)q_issued);
      }
    }
  } else if (warp < kFirstEpiWarp) {
    if (lane == 0) {
      // ---------------------------- UMMA issuers --------------------------------
      // Issuer m takes the tiles with sequence number = m (mod 2) and always
      // accumulates into TMEM buffer m, so one issuer's barrier waits and
      // commits overlap the other's MMAs.
      const uint32_t me = (uint32_t)(warp - 1);
      const uint32_t idesc = idesc_bf16_f32(kM, kN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0, q_phase = 0, seq = 0;
      int64_t cur_qb = -1, lim = 0;
      bool have_q = false;
      const uint64_t a_desc0 = sdesc_sw128(smem_u32(k_smem));
      const uint64_t b_desc0 = sdesc_sw128(smem_u32(q_smem));
      int64_t qb = t_begin / p.tiles_per_qb;
      int ct = (int)(t_begin % p.tiles_per_qb) - 1;
      for (int64_t it = t_begin; it < t_end; ++it) {
        if (++ct == p.tiles_per_qb) {
          ct = 0;
          ++qb;
        }
        if (qb != cur_qb) {
          cur_qb = qb;
          lim = block_limit(p, qb);
          if (lim > 0) {
            if (have_q) umma_commit(&bar_qempty);
            if (!mbar_wait(&bar_qfull, q_phase, &abort_flag, p.status)) break;
            q_phase ^= 1;
            have_q = true;
            tc_fence_after();
          }
        }
        if ((int64_t)ct * kM >= lim) continue;
        if ((seq++ & 1u) == me) {
          if (!mbar_wait(&bar_tempty[acc], acc_phase ^ 1u, &abort_flag, p.status)) break;
          if (!mbar_wait(&bar_full[stage], phase, &abort_flag, p.status)) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * kN;
          // descriptor start-address field counts 16-byte units
          const uint64_t a_desc = a_desc0 + (uint64_t)(stage * (kTileBytes >> 4));
#pragma unroll
          for (int k = 0; k < kDim / 16; ++k)
            umma_bf16_ss(d_tmem, a_desc + (k >> 2) * (kAtomA >> 4) + (k & 3) * 2,
                         b_desc0 + (k >> 2) * (kAtomB >> 4) + (k & 3) * 2, idesc, k > 0 ? 1u : 0u);
          umma_commit(&bar_empty[stage]);
          umma_commit(&bar_tfull[acc]);
        }
        if (++stage == (uint32_t)stages) {
          stage = 0;
          phase ^= 1u;
        }
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      umma_commit(&bar_drain);
      mbar_wait_drain(&bar_drain, 0);
    }
  } else {
    // -------------------------------- epilogue ----------------------------------
    const int quad = warp & 3;
    const int j = (warp - kFirstEpiWarp) >> 2;  // token of the block handled by this warp
    const int row = quad * 32 + lane;
    uint32_t acc = 0, acc_phase = 0;
    bool aborted = false;
    // The same tile sequence as the producer and the issuers, walked one query
    // block at a time: an int32 loop over the block's tiles in this CTA's
    // range that lie below the block's causal limit (the skipped ones advance
    // no barrier), with the token's causal limit and its rows of logits and
    // segment entries set once per block.
    for (int64_t it = t_begin; it < t_end && !aborted;) {
      const int64_t qb = it / p.tiles_per_qb;
      const int ct0 = (int)(it - qb * p.tiles_per_qb);
      const int ct_end = (t_end - it < (int64_t)(p.tiles_per_qb - ct0)) ? ct0 + (int)(t_end - it) : p.tiles_per_qb;
      it += ct_end - ct0;
      const int64_t lim = block_limit(p, qb);
      const int ct_live = (int)((lim + kM - 1) / kM);  // tiles with ct * kM < lim
      const int ct_stop = ct_end < ct_live ? ct_end : ct_live;
      // the warp's token weights stay in shared memory for the whole block
      const int64_t tw = qb * kTok + j;
      const bool live = tw < p.T;
      const int lim_t = live ? (int)causal_limit(__ldg(p.pos + tw), p.S, p.ratio) : 0;  // S < 2^31
      float* const lrow = p.logits + (live ? tw : 0) * p.S + row;
      int32_t* const srow = p.segmax != nullptr ? p.segmax + (live ? tw : 0) * p.seg_ld + quad : nullptr;
      const float* wsrc = p.w + (live ? tw : 0) * kHeads;
      __syncwarp();
      w_smem[warp - kFirstEpiWarp][lane] = __ldg(wsrc + lane);
      w_smem[warp - kFirstEpiWarp][lane + 32] = __ldg(wsrc + lane + 32);
      __syncwarp();
      // tiles in pairs, so the accumulator index (and with it the barrier and
      // TMEM addresses) is a constant in each copy of the body
      auto tile_body = [&](const int ct, const uint32_t ai, const uint32_t ph) -> bool {
        if (!mbar_wait(&bar_tfull[ai], ph, &abort_flag, p.status)) return false;
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + ai * kN + j * kHeads;
        // both halves of the row in flight at once, one wait, then the
        // accumulator is released before the arithmetic
        uint32_t r0[32], r1[32];
        tmem_ld32(taddr, r0);
        tmem_ld32(taddr + 32, r1);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&bar_tempty[ai]);
        const float4* w4 = reinterpret_cast<const float4*>(w_smem[warp - kFirstEpiWarp]);
        float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f, x4 = 0.f, x5 = 0.f, x6 = 0.f, x7 = 0.f;
#pragma unroll
        for (int h4 = 0; h4 < 8; ++h4) {
          const float4 a = w4[h4];
          const float4 c = w4[8 + h4];
          x0 = fmaf(a.x, fmaxf(__uint_as_float(r0[4 * h4]), 0.f), x0);
          x1 = fmaf(a.y, fmaxf(__uint_as_float(r0[4 * h4 + 1]), 0.f), x1);
          x2 = fmaf(a.z, fmaxf(__uint_as_float(r0[4 * h4 + 2]), 0.f), x2);
          x3 = fmaf(a.w, fmaxf(__uint_as_float(r0[4 * h4 + 3]), 0.f), x3);
          x4 = fmaf(c.x, fmaxf(__uint_as_float(r1[4 * h4]), 0.f), x4);
          x5 = fmaf(c.y, fmaxf(__uint_as_float(r1[4 * h4 + 1]), 0.f), x5);
          x6 = fmaf(c.z, fmaxf(__uint_as_float(r1[4 * h4 + 2]), 0.f), x6);
          x7 = fmaf(c.w, fmaxf(__uint_as_float(r1[4 * h4 + 3]), 0.f), x7);
        }
        const float y = ((x0 + x1) + (x2 + x3)) + ((x4 + x5) + (x6 + x7));
        // only the token's own candidates (s below its causal limit) are written
        const bool valid = ct * kM + row < lim_t;
        if (valid) lrow[ct * kM] = y;
        if (srow != nullptr) {
          // the warp's 32 scores are one segment: its entry is the largest bit
          // pattern read as a signed integer (the largest score when any is
          // >= +0; see topk.cuh, block_topk_segmax, for how the select reads
          // it).  Lane 0's score is the segment's first, so its `valid` says
          // whether the segment starts below the limit.
          const int m = __reduce_max_sync(0xffffffffu, valid ? __float_as_int(y) : INT_MIN);
          if (lane == 0 && valid) srow[ct * 4] = m;
        }
        return true;
      };
      int ct = ct0;
      if (acc == 1u && ct < ct_stop) {  // the second tile of a pair begun in an earlier block
        if (!tile_body(ct, 1u, acc_phase)) {
          aborted = true;
          break;
        }
        ++ct;
        acc = 0u;
        acc_phase ^= 1u;
      }
      for (; ct + 1 < ct_stop; ct += 2) {
        if (!tile_body(ct, 0u, acc_phase) || !tile_body(ct + 1, 1u, acc_phase)) {
          aborted = true;
          break;
        }
        acc_phase ^= 1u;
      }
      if (!aborted && ct < ct_stop) {
        if (!tile_body(ct, 0u, acc_phase))
          aborted = true;
        else
          acc = 1u;
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

__global__ void causal_limits_kernel(const int64_t* __restrict__ pos, int T, int64_t S, int ratio,
                                     int32_t* __restrict__ n_valid) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < T) n_valid[t] = (int32_t)causal_limit(pos[t], S, ratio);
}

// logits[t, s] = -inf for s >= the causal limit of token t (one CTA per row).
__global__ void causal_fill_kernel(const int64_t* __restrict__ pos, int64_t S, int ratio, float* __restrict__ logits) {
  const int64_t t = blockIdx.x;
  float* row = logits + t * S;
  for (int64_t s = causal_limit(__ldg(pos + t), S, ratio) + threadIdx.x; s < S; s += blockDim.x) row[s] = -INFINITY;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
int64_t seg_count(int64_t S) { return (S + 31) / 32; }

}  // namespace

// logits [T, S], the causal limits [T], the segment maxima [T, ceil(S / 32)]
size_t prefill_workspace_bytes(int T, int64_t S) {
  return align256((size_t)T * S * 4) + align256((size_t)T * 4) + align256((size_t)T * seg_count(S) * 4);
}

fm_status launch_prefill_scores(const PrefillArgs& a, float* logits, int32_t* segmax, bool fill_masked, int num_sms,
                                unsigned int* status, cudaStream_t stream) {
  cudaError_t e = cudaSuccess;
  if (a.T > 0 && a.S > 0) {
    CUtensorMap tmap_k, tmap_q;
    {
      const uint64_t dims[2] = {(uint64_t)kDim, (uint64_t)a.S};
      const uint64_t strides[1] = {(uint64_t)kDim * 2};
      const uint32_t box[2] = {64, (uint32_t)kM};
      fm_status st = make_tmap(&tmap_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.keys, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_128B);
      if (st != FM_OK) return st;
    }
    {
      const uint64_t dims[2] = {(uint64_t)kDim, (uint64_t)a.T * kHeads};
      const uint64_t strides[1] = {(uint64_t)kDim * 2};
      const uint32_t box[2] = {64, (uint32_t)kN};
      fm_status st = make_tmap(&tmap_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_128B);
      if (st != FM_OK) return st;
    }
    const int tiles_per_qb = (int)((a.S + kM - 1) / kM);
    const int64_t n_qb = (a.T + kTok - 1) / kTok;
    const int64_t total = n_qb * tiles_per_qb;
    const int smem_cap = 227 * 1024 - (int)sizeof(float) * kEpiWarps * kHeads;  // minus the static w_smem
    const int fixed = 1024 + kQBytes;
    int stages = (smem_cap - fixed) / kTileBytes;
    if (stages > kMaxStages) stages = kMaxStages;
    // tile i uses stage i % stages and issuer i % 2: with an even stage count
    // each stage has one consumer, whose parity wait on the stage's full
    // barrier then cannot pass on a previous fill still in flight (key copies
    // may complete out of order)
    stages -= stages % kMmaWarps;
    const int smem = fixed + stages * kTileBytes;
    Params p;
    p.w = a.w;
    p.pos = a.pos;
    p.logits = logits;
    p.segmax = segmax;
    p.seg_ld = seg_count(a.S);
    p.status = status;
    p.S = a.S;
    p.total_items = total;
    p.T = a.T;
    p.tiles_per_qb = tiles_per_qb;
    p.ratio = a.ratio;
    p.stages = stages;
    e = cudaFuncSetAttribute(prefill_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "prefill: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    const int grid = (int)(total < num_sms ? total : num_sms);
    prefill_score_kernel<<<grid, kThreads, smem, stream>>>(tmap_k, tmap_q, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "prefill score: launch: %s", cudaGetErrorString(e));
    if (fill_masked) {
      causal_fill_kernel<<<a.T, 256, 0, stream>>>(a.pos, a.S, a.ratio, logits);
      e = cudaGetLastError();
      if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "prefill fill: launch: %s", cudaGetErrorString(e));
    }
  }
  return FM_OK;
}

fm_status launch_prefill(const PrefillArgs& a, int num_sms, unsigned int* status, cudaStream_t stream) {
  if (a.T == 0) return FM_OK;
  float* logits = static_cast<float*>(a.workspace);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  const size_t logits_bytes = align256((size_t)a.T * a.S * 4);
  int32_t* n_valid = reinterpret_cast<int32_t*>(ws + logits_bytes);
  int32_t* segmax = reinterpret_cast<int32_t*>(ws + logits_bytes + align256((size_t)a.T * 4));
  causal_limits_kernel<<<(a.T + 255) / 256, 256, 0, stream>>>(a.pos, a.T, a.S, a.ratio, n_valid);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "prefill limits: launch: %s", cudaGetErrorString(e));
  fm_status st = launch_prefill_scores(a, logits, segmax, false, num_sms, status, stream);
  if (st != FM_OK) return st;
  return launch_topk_rows_segmax(logits, a.S, n_valid, segmax, seg_count(a.S), a.T, (int)a.S, a.k, a.idx_out,
                                 a.score_out, stream);
}

}  // namespace fm

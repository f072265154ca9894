// memindex.cu -- Memory Indexer scoring, OR-union over layers, resident mask.
//
// Computes, for request b, layer l, chunk s (see "FlashMemory-DeepSeek-V4:
// Lightning Index Ultra-Long Context via Lookahead Sparse Attention", sec. 3
// "Memory Indexer scoring function", and the "FlashMemory-DeepSeek-V4" README,
// "Retriever architecture"):
//     x[b,l,s] = sum_h w[b,l,h] * ReLU(q[b,l,h,:] . K[b,l,s,:])
//     resident[b,s] = max_l x[b,l,s] >= logit(threshold)
// (sigmoid is monotone, so max_l sigmoid(x) >= thr  <=>  max_l x >= logit(thr)).
//
// GB300 mapping.  The work is a stream over the keys (256 B per chunk per
// layer, 64 FLOP/B), so it is HBM-bound only if the dot products run on the
// tensor cores.  A persistent CTA per SM owns a contiguous range of 128-chunk
// tiles and runs a warp-specialised pipeline:
//   warp 0  TMA producer: K tiles [128 chunks x 128 d] bf16 (SWIZZLE_128B) into
//           an N-stage ring; the request's q [L x 64 x 128] once per request.
//   warp 1  UMMA issuer: per layer, 8 x tcgen05.mma M=128 (chunks) x N=64
//           (heads) x K=16 into a TMEM accumulator [128 lanes x 64 cols];
//           two accumulator sets (2 x 4 layers x 64 cols = 512 TMEM columns)
//           so the epilogue of one tile overlaps the MMAs of the next.
//   warps 2-5  epilogue: thread = chunk row; tcgen05.ld its 64 head dots per
//           layer, sum_h w_h * max(dot, 0) in fp32 registers, max over layers,
//           compare, __ballot_sync -> one mask word per warp; optional
//           max-sigmoid and per-layer logits.
#include <math.h>

#include "fm_common.cuh"
#include "fm_internal.h"

namespace fm {
namespace {

constexpr int kM = 128;                         // chunks per tile (UMMA M)
constexpr int kHeads = 64;                      // UMMA N
constexpr int kDim = 128;                       // reduction length
constexpr int kMaxL = 4;                        // indexer layers
constexpr int kMaxStages = 8;
constexpr int kTileBytes = kM * kDim * 2;       // 32 KB of keys per layer-tile
constexpr int kAtomA = kM * 64 * 2;             // one 128-byte-wide K atom of A
constexpr int kQLayerBytes = kHeads * kDim * 2; // 16 KB of q per layer
constexpr int kAtomB = kHeads * 64 * 2;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;

struct Params {
  const float* w;
  uint32_t* mask;
  float* maxsig;
  float* logits;
  unsigned int* status;
  int64_t S;
  int64_t total_tiles;
  int tiles_per_b;
  int L;
  int stages;
  float thr_logit;
};

__global__ void __launch_bounds__(kThreads, 1)
    memindex_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                    const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_smem = smem;
  uint8_t* k_smem = smem + p.L * kQLayerBytes;

  __shared__ __align__(8) uint64_t bar_full[kMaxStages], bar_empty[kMaxStages];
  __shared__ __align__(8) uint64_t bar_tfull[2], bar_tempty[2], bar_qfull, bar_qempty, bar_drain;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int L = p.L, stages = p.stages;
  const int64_t t_begin = p.total_tiles * blockIdx.x / gridDim.x;
  const int64_t t_end = p.total_tiles * (blockIdx.x + 1) / gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_tfull[i], 1);
      mbar_init(&bar_tempty[i], 128);
    }
    mbar_init(&bar_qfull, 1);
    mbar_init(&bar_qempty, 1);
    mbar_init(&bar_drain, 1);
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
      int64_t cur_b = -1;
      bool ok = true;
      int64_t b = t_begin / p.tiles_per_b;
      int tile = (int)(t_begin % p.tiles_per_b) - 1;
      for (int64_t t = t_begin; t < t_end && ok; ++t) {
        if (++tile == p.tiles_per_b) {
          tile = 0;
          ++b;
        }
        if (b != cur_b) {
          if (cur_b >= 0) {
            if (!mbar_wait(&bar_qempty, q_phase, &abort_flag, p.status)) break;
            q_phase ^= 1;
          }
          mbar_arrive_expect_tx(&bar_qfull, (uint32_t)(L * kQLayerBytes));
          for (int l = 0; l < L; ++l)
            for (int a = 0; a < 2; ++a)
              tma_load_2d(q_smem + l * kQLayerBytes + a * kAtomB, &tmap_q, &bar_qfull, a * 64,
                          (int32_t)((b * L + l) * kHeads));
          q_issued = (q_issued + 1) & 1;
          cur_b = b;
        }
        for (int l = 0; l < L; ++l) {
          if (!mbar_wait(&bar_empty[stage], phase ^ 1u, &abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bar_full[stage], (uint32_t)kTileBytes);
          for (int a = 0; a < 2; ++a)
            tma_load_4d(k_smem + stage * kTileBytes + a * kAtomA, &tmap_k, &bar_full[stage], a * 64, tile * kM, l,
                        (int32_t)b);
          issued[stage] = (int)phase;
          if (++stage == (uint32_t)stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (abort_flag) {  // let copies already in flight land before the CTA exits
        for (int s = 0; s < stages; ++s)
          if (issued[s] >= 0) mbar_wait_drain(&bar_full[s], (uint32_t)issued[s]);
        if (q_issued >= 0) mbar_wait_drain(&bar_qfull, (uint32_t)q_issued);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------ UMMA issuer -------------------------------
      const uint32_t idesc = idesc_bf16_f32(kM, kHeads);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0, q_phase = 0;
      int64_t cur_b = -1;
      bool ok = true;
      const uint64_t a_desc0 = sdesc_sw128(smem_u32(k_smem));
      const uint64_t b_desc0 = sdesc_sw128(smem_u32(q_smem));
      int64_t b = t_begin / p.tiles_per_b;
      int tile = (int)(t_begin % p.tiles_per_b) - 1;
      for (int64_t t = t_begin; t < t_end && ok; ++t) {
        if (++tile == p.tiles_per_b) {
          tile = 0;
          ++b;
        }
        if (b != cur_b) {
          if (cur_b >= 0) umma_commit(&bar_qempty);
          if (!mbar_wait(&bar_qfull, q_phase, &abort_flag, p.status)) break;
          q_phase ^= 1;
          tc_fence_after();
          cur_b = b;
        }
        if (!mbar_wait(&bar_tempty[acc], acc_phase ^ 1u, &abort_flag, p.status)) break;
        tc_fence_after();
        for (int l = 0; l < L; ++l) {
          if (!mbar_wait(&bar_full[stage], phase, &abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * (kMaxL * kHeads) + l * kHeads;
          // descriptor start-address field counts 16-byte units
          const uint64_t a_desc = a_desc0 + (uint64_t)(stage * (kTileBytes >> 4));
          const uint64_t b_desc = b_desc0 + (uint64_t)(l * (kQLayerBytes >> 4));
#pragma unroll
          for (int k = 0; k < kDim / 16; ++k)
            umma_bf16_ss(d_tmem, a_desc + (k >> 2) * (kAtomA >> 4) + (k & 3) * 2,
                         b_desc + (k >> 2) * (kAtomB >> 4) + (k & 3) * 2, idesc, k > 0 ? 1u : 0u);
          umma_commit(&bar_empty[stage]);
          if (++stage == (uint32_t)stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&bar_tfull[acc]);
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      umma_commit(&bar_drain);  // every MMA issued above has finished before TMEM is freed
      mbar_wait_drain(&bar_drain, 0);
    }
  } else {
    // -------------------------------- epilogue ----------------------------------
    const int quad = warp & 3;  // TMEM lane quadrant this warp can access
    const int row = quad * 32 + lane;
    const int64_t words = (p.S + 31) / 32;
    uint32_t acc = 0, acc_phase = 0;
    int64_t b = t_begin / p.tiles_per_b;
    int tile = (int)(t_begin % p.tiles_per_b) - 1;
    for (int64_t t = t_begin; t < t_end; ++t) {
      if (++tile == p.tiles_per_b) {
        tile = 0;
        ++b;
      }
      if (!mbar_wait(&bar_tfull[acc], acc_phase, &abort_flag, p.status)) break;
      tc_fence_after();
      const int64_t s = (int64_t)tile * kM + row;
      const bool valid = s < p.S;
      float m = -INFINITY;
      for (int l = 0; l < L; ++l) {
        uint32_t r0[32], r1[32];
        const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * (kMaxL * kHeads) + l * kHeads;
        tmem_ld32(taddr, r0);
        tmem_ld32(taddr + 32, r1);
        // head weights: warp-uniform addresses, served by L1 as broadcasts
        const float4* wl = reinterpret_cast<const float4*>(p.w + (b * L + l) * kHeads);
        float wr[kHeads];
#pragma unroll
        for (int i = 0; i < kHeads / 4; ++i) {
          const float4 v = __ldg(wl + i);
          wr[4 * i] = v.x;
          wr[4 * i + 1] = v.y;
          wr[4 * i + 2] = v.z;
          wr[4 * i + 3] = v.w;
        }
        tmem_ld_wait();
        float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
#pragma unroll
        for (int h = 0; h < 32; h += 2) {
          x0 = fmaf(wr[h], fmaxf(__uint_as_float(r0[h]), 0.f), x0);
          x1 = fmaf(wr[h + 1], fmaxf(__uint_as_float(r0[h + 1]), 0.f), x1);
          x2 = fmaf(wr[32 + h], fmaxf(__uint_as_float(r1[h]), 0.f), x2);
          x3 = fmaf(wr[33 + h], fmaxf(__uint_as_float(r1[h + 1]), 0.f), x3);
        }
        const float x = (x0 + x1) + (x2 + x3);
        if (p.logits != nullptr && valid) p.logits[(b * L + l) * p.S + s] = x;
        m = fmaxf(m, x);
      }
      tc_fence_before();
      mbar_arrive(&bar_tempty[acc]);
      const uint32_t bits = __ballot_sync(0xffffffffu, valid && m >= p.thr_logit);
      const int64_t word = (int64_t)tile * (kM / 32) + quad;
      if (lane == 0 && word < words) p.mask[b * words + word] = bits;
      if (p.maxsig != nullptr && valid) p.maxsig[b * p.S + s] = 1.0f / (1.0f + expf(-m));
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

fm_status launch_memindex(const MemindexArgs& a, int num_sms, unsigned int* status, cudaStream_t stream) {
  const int tiles_per_b = (int)((a.S + kM - 1) / kM);
  const int64_t total = (int64_t)a.B * tiles_per_b;
  if (total == 0) return FM_OK;

  CUtensorMap tmap_k, tmap_q;
  {
    // keys: dims (d, S, L, B), box (64, 128, 1, 1), 128-byte swizzle
    const uint64_t dims[4] = {(uint64_t)kDim, (uint64_t)a.S, (uint64_t)a.L, (uint64_t)a.B};
    const uint64_t strides[3] = {(uint64_t)kDim * 2, (uint64_t)a.key_stride_l * 2, (uint64_t)a.key_stride_b * 2};
    const uint32_t box[4] = {64, (uint32_t)kM, 1, 1};
    fm_status st = make_tmap(&tmap_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.keys, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != FM_OK) return st;
  }
  {
    // q: rows (B*L*64) x 128, box (64, 64)
    const uint64_t dims[2] = {(uint64_t)kDim, (uint64_t)a.B * a.L * kHeads};
    const uint64_t strides[1] = {(uint64_t)kDim * 2};
    const uint32_t box[2] = {64, (uint32_t)kHeads};
    fm_status st = make_tmap(&tmap_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != FM_OK) return st;
  }

  const int smem_cap = 227 * 1024;
  const int fixed = 1024 + a.L * kQLayerBytes;
  int stages = (smem_cap - fixed) / kTileBytes;
  if (stages > 6) stages = 6;
  const int smem = fixed + stages * kTileBytes;

  Params p;
  p.w = a.w;
  p.mask = a.mask;
  p.maxsig = a.maxsig;
  p.logits = a.logits;
  p.status = status;
  p.S = a.S;
  p.total_tiles = total;
  p.tiles_per_b = tiles_per_b;
  p.L = a.L;
  p.stages = stages;
  p.thr_logit = a.thr_logit;

  cudaError_t e = cudaFuncSetAttribute(memindex_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "memindex: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  const int grid = (int)(total < num_sms ? total : num_sms);
  memindex_kernel<<<grid, kThreads, smem, stream>>>(tmap_k, tmap_q, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "memindex: launch: %s", cudaGetErrorString(e));
  return FM_OK;
}

}  // namespace fm

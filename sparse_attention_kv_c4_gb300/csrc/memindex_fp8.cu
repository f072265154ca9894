// memindex_fp8.cu -- the Memory Indexer over compressed E4M3 keys.
//
// Computes the same scores as memindex.cu ("FlashMemory-DeepSeek-V4: Lightning
// Index Ultra-Long Context via Lookahead Sparse Attention", sec. 3 "Memory
// Indexer scoring function"), with each chunk's key in the compressed_k
// format the retriever reads (sec. 6; "FlashMemory-DeepSeek-V4" README,
// "compressed_k format": 128 E4M3 bytes plus an fp32 scale, dequantised as
// fp8.float() * scale):
//     x[b,l,s] = sum_h w[b,l,h] * ReLU(q[b,l,h,:] . (scale[b,l,s] * e4m3(k8[b,l,s,:])))
//     resident[b,s] = max_l x[b,l,s] >= logit(threshold)
// The scale is applied to each head's dot instead of to each key element
// (mathematically equal; the difference is one fp32 rounding per element).
//
// GB300 mapping.  At 132 B per chunk-layer the stream is half the bf16 path's,
// so the dots run on the tensor cores in E4M3 (kind::f8f6f4) to stay
// HBM-bound:
//   prep    one CTA per (request, layer): q split into two E4M3 terms per head
//           (fp8.cuh), 2^e_h folded into w; the weighted query sum q_w in
//           four E4M3 terms in two more rows (the ReLU's linear half, below).
//   warp 0  TMA producer: the request's split q (L x 20 KB) once per request,
//           then per layer a key tile [128 chunks x 128 B] (SWIZZLE_128B)
//           into the stage ring of the pair (below) that takes the tile.
//   warps 1-2  UMMA issuers: per layer-tile 8 x tcgen05.mma M=128 (chunks)
//           x N=80 (64 heads, the q_w rows, zeros) x K=32: four K steps
//           against the t1 block, then four against the t2 block into the
//           same accumulator, so TMEM holds (t1 + t2).k directly.  One issuing
//           thread alone cannot keep up with the key stream (each MMA costs it
//           tens of cycles), so two issue in parallel.
//   warps 3-10  epilogue, two groups of four warps (one warp per SM
//           sub-partition would leave every latency exposed).  Issuer m and
//           group m form pair m: the pair takes the CTA's tiles with local
//           index = m (mod 2) and owns three of the six 80-column
//           accumulators.  Thread = chunk row; its chunk's scales are fetched
//           with cp.async two of its pair's tiles ahead into a shared-memory
//           ring (a load from HBM per layer-tile would stall the warp for its
//           full latency), the head weights come from a per-warp shared copy.
//           With ReLU(d) = (d + |d|) / 2 a chunk's logit is
//           (sc q_w.k + |sc| sum_h w'_h |d_h|) / 2, w'_h = w_h 2^e_h and
//           d_h = (t1 + t2).k: one FFMA per head (the absolute value folds
//           into it), q_w.k from two accumulator columns.  Then the running
//           max over the tile's layers, the ballot of the mask word,
//           max-sigmoid (and per-layer logits when asked).
#include <math.h>

#include "fm_common.cuh"
#include "fm_internal.h"
#include "fp8.cuh"

#define FM_API extern "C" __attribute__((visibility("default")))

namespace fm {
namespace {

constexpr int kM = 128;                      // chunks per tile (UMMA M)
constexpr int kHeads = 64;                   // t1.k + t2.k accumulate in one column per head
// The split query of a layer: a t1 block and a t2 block of kQTermRows rows
// each (the 64 heads, then the weighted query sum's terms and zeros: the
// ReLU's linear half on the tensor core, below); kQTermRows is the MMA's N.
constexpr int kQTermRows = kHeads + 16;
constexpr int kQRows = 2 * kQTermRows;
constexpr int kDim = 128;                    // E4M3 bytes per key (UMMA K, 4 steps of 32)
constexpr int kMaxL = 4;
constexpr int kTileBytes = kM * kDim;        // 16 KB of keys per layer-tile
constexpr int kQTermBytes = kQTermRows * kDim;  // 10 KB
constexpr int kQLayerBytes = kQRows * kDim;  // 20 KB of split query per layer
constexpr int kWStride = kHeads + 4;         // floats per (request, layer) of wq: w', then 2^e1, 2^e2
constexpr int kAccBufs = 6;                  // accumulators of kQTermRows columns (480 of 512)
constexpr int kMaxStages = 12;
// Issuer m and epilogue group m form pair m: the pair takes the CTA's tiles
// with local index i = m (mod kPairs) and owns accumulators
// [m * kRingAccs, (m + 1) * kRingAccs), a ring with one filler and one
// reader, so every parity wait on it is unambiguous.  (Rings shared between
// issuers or between epilogue groups let a waiter run two uses ahead of an
// accumulator and pass a parity wait on a stale phase.)
constexpr int kPairs = 2;
constexpr int kMmaWarps = kPairs;
constexpr int kEpiGroups = kPairs;
constexpr int kRingAccs = kAccBufs / kPairs;
constexpr int kFirstEpiWarp = 1 + kMmaWarps;
constexpr int kThreads = kFirstEpiWarp * 32 + kEpiGroups * 128;
constexpr int kPrepThreads = 256;
constexpr uint32_t kTmemCols = 512;          // kAccBufs x kQTermRows, as a power of two
constexpr int kScDepth = 2;                  // a group's tiles of scales in flight ahead of it
constexpr int kScSlots = kScDepth + 1;
constexpr int kScRingBytes = kEpiGroups * kScSlots * kMaxL * kM * 4;  // 12 KB

// 4-byte asynchronous global -> shared copy; src_bytes = 0 writes a zero
__device__ __forceinline__ void cp_async4(float* dst, const float* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

struct Params {
  const float* wq;            // [B*L, kWStride]: head weights with 2^e_h folded in, then q_w's two scales
  const float* k_scale;
  int64_t sstride_b, sstride_l;
  uint32_t* mask;
  float* maxsig;
  float* logits;
  unsigned int* status;
  int64_t S;
  int64_t total_tiles;
  int tiles_per_b;
  int L;
  int stages;  // key stages per pair
  float thr_logit;
};

__global__ void __launch_bounds__(kPrepThreads)
    memindex_fp8_prep_kernel(const uint16_t* __restrict__ q, const float* __restrict__ w,
                             uint8_t* __restrict__ qsplit, float* __restrict__ wq) {
  const int64_t bl = blockIdx.x;
  uint8_t* t1 = qsplit + bl * kQLayerBytes;
  uint8_t* t2 = t1 + kQTermBytes;
  float* wl = wq + bl * kWStride;
  split_query(q + bl * kHeads * kDim, w + bl * kHeads, kHeads, kPrepThreads, t1, t2, wl);
  // The ReLU's linear half: with ReLU(d) = (d + |d|) / 2 a chunk's logit is
  // (sc q_w.k + |sc| sum_h w'_h |d_h|) / 2, where q_w = sum_h w_h q_h.  q_w
  // (fp32, heads in order) goes into four E4M3 terms: with 2^e1 putting
  // max|q_w| in (224, 448], u1 = RNE(q_w 2^-e1), u2 = RNE(rest), then the
  // rest times 2^8 the same way (u3, u4), within 2^-18 of max|q_w|.  Rows
  // 64 (u1 | u2) and 65 (u3 | u4) of the t1 | t2 blocks, zeros in 66 .. 79.
  __shared__ float red[kPrepThreads / 32];
  const int j = threadIdx.x;
  float qw = 0.f;
  if (j < kDim) {
    const uint16_t* qb = q + bl * kHeads * kDim + j;
    for (int h = 0; h < kHeads; ++h)
      qw = fmaf(__ldg(w + bl * kHeads + h), __uint_as_float((uint32_t)__ldg(qb + h * kDim) << 16), qw);
  }
  float m = fabsf(qw);
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((j & 31) == 0) red[j >> 5] = m;
  __syncthreads();
  float amax = 0.f;
  for (int i = 0; i < kPrepThreads / 32; ++i) amax = fmaxf(amax, red[i]);
  int e = 0;
  if (amax > 0.f && isfinite(amax)) {
    e = ilogbf(amax) - 8;
    if (ldexpf(amax, -e) > 448.f) e += 1;
  }
  if (j < kDim) {
    const float s1 = ldexpf(qw, -e);
    const uint32_t u1 = e4m3_rne(s1);
    const float r1 = s1 - e4m3_value(u1);
    const uint32_t u2 = e4m3_rne(r1);
    const float s2 = (r1 - e4m3_value(u2)) * 256.f;
    const uint32_t u3 = e4m3_rne(s2);
    t1[kHeads * kDim + j] = (uint8_t)u1;
    t2[kHeads * kDim + j] = (uint8_t)u2;
    t1[(kHeads + 1) * kDim + j] = (uint8_t)u3;
    t2[(kHeads + 1) * kDim + j] = (uint8_t)e4m3_rne(s2 - e4m3_value(u3));
  }
  for (int i = threadIdx.x; i < 14 * kDim; i += kPrepThreads) {
    t1[(kHeads + 2) * kDim + i] = 0;
    t2[(kHeads + 2) * kDim + i] = 0;
  }
  if (threadIdx.x == 0) {
    wl[kHeads] = ldexpf(1.f, e);
    wl[kHeads + 1] = ldexpf(1.f, e - 8);
    wl[kHeads + 2] = 0.f;
    wl[kHeads + 3] = 0.f;
  }
}

// Two consecutive 32-bit TMEM columns: thread i gets lane (base + i).
__device__ __forceinline__ void tmem_ld2(uint32_t taddr, uint32_t (&r)[2]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(taddr)
               : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    memindex_fp8_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                        const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_smem = smem;
  float* sc_ring = reinterpret_cast<float*>(smem + p.L * kQLayerBytes);  // [group][slot][layer][row]
  uint8_t* k_smem = smem + p.L * kQLayerBytes + kScRingBytes;

  __shared__ __align__(8) uint64_t bar_full[kMaxStages], bar_empty[kMaxStages];
  __shared__ __align__(8) uint64_t bar_tfull[kAccBufs], bar_tempty[kAccBufs], bar_qfull, bar_qempty, bar_drain;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  // one copy of the current request's head weights per epilogue warp, so a
  // warp refreshes its own copy with __syncwarp alone
  __shared__ __align__(16) float w_smem[kEpiGroups * 4][kMaxL * kWStride];

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int L = p.L, ring = p.stages;  // key stages per pair; pair m owns [m * ring, (m + 1) * ring)
  const int64_t t_begin = p.total_tiles * blockIdx.x / gridDim.x;
  const int64_t t_end = p.total_tiles * (blockIdx.x + 1) / gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairs * ring; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
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
      // Each pair has its own ring of key stages, filled in the order its
      // issuer consumes them.  (Key copies may complete out of order: with a
      // ring shared by both issuers, an issuer could wait on a stage whose
      // previous fill -- the other issuer's -- is still in flight and pass
      // its parity wait on that older phase.)
      uint32_t rstage[kPairs] = {}, rphase[kPairs] = {}, q_phase = 0;
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
            tma_load_2d(q_smem + l * kQLayerBytes, &tmap_q, &bar_qfull, 0, (int32_t)((b * L + l) * kQRows));
          q_issued = (q_issued + 1) & 1;
          cur_b = b;
        }
        const int m = (int)((t - t_begin) % kPairs);
        for (int l = 0; l < L; ++l) {
          const uint32_t stage = m * ring + rstage[m], phase = rphase[m];
          if (!mbar_wait(&bar_empty[stage], phase ^ 1u, &abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bar_full[stage], (uint32_t)kTileBytes);
          tma_load_4d(k_smem + stage * kTileBytes, &tmap_k, &bar_full[stage], 0, tile * kM, l, (int32_t)b);
          issued[stage] = (int)phase;
          if (++rstage[m] == (uint32_t)ring) {
            rstage[m] = 0;
            rphase[m] ^= 1u;
          }
        }
      }
      if (abort_flag) {  // let copies already in flight land before the CTA exits
        for (int s = 0; s < kPairs * ring; ++s)
          if (issued[s] >= 0) mbar_wait_drain(&bar_full[s], (uint32_t)issued[s]);
        if (q_issued >= 0) mbar_wait_drain(&bar_qfull, (uint32_t)q_issued);
      }
    }
  } else if (warp < kFirstEpiWarp) {
    if (lane == 0) {
      // ------------------------------ UMMA issuers ------------------------------
      // Issuer m takes its pair's tiles (all layers of each) from its pair's
      // stage ring, so one issuer's barrier waits and commits overlap the
      // other's MMAs.
      const int me = warp - 1;
      const uint32_t idesc = idesc_e4m3_f32(kM, kQTermRows);
      uint32_t rstage = 0, phase = 0, racc = 0, acc_phase = 0, q_phase = 0;
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
        if ((int)((t - t_begin) % kPairs) != me) continue;  // the other pair's tile
        for (int l = 0; l < L; ++l) {
          const uint32_t acc = me * kRingAccs + racc;
          const uint32_t stage = me * ring + rstage;
          if (!mbar_wait(&bar_tempty[acc], acc_phase ^ 1u, &abort_flag, p.status) ||
              !mbar_wait(&bar_full[stage], phase, &abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * kQTermRows;
          // descriptor start-address field counts 16-byte units; K steps of
          // 32 bytes advance it by 2 inside the 128-byte swizzle atom
          const uint64_t a_desc = a_desc0 + (uint64_t)(stage * (kTileBytes >> 4));
          const uint64_t b_desc = b_desc0 + (uint64_t)(l * (kQLayerBytes >> 4));
          // the t2 block starts 10 KB (ten 1 KB swizzle atoms) after the t1 block
          constexpr uint64_t kT2 = kQTermBytes >> 4;
#pragma unroll
          for (int k = 0; k < kDim / 32; ++k)
            umma_e4m3_ss(d_tmem, a_desc + 2 * k, b_desc + 2 * k, idesc, k != 0 ? 1u : 0u);
#pragma unroll
          for (int k = 0; k < kDim / 32; ++k) umma_e4m3_ss(d_tmem, a_desc + 2 * k, b_desc + kT2 + 2 * k, idesc, 1u);
          umma_commit(&bar_empty[stage]);
          umma_commit(&bar_tfull[acc]);
          if (++rstage == (uint32_t)ring) {
            rstage = 0;
            phase ^= 1u;
          }
          if (++racc == (uint32_t)kRingAccs) {
            racc = 0;
            acc_phase ^= 1u;
          }
        }
      }
      umma_commit(&bar_drain);  // every MMA issued above has finished before TMEM is freed
      mbar_wait_drain(&bar_drain, 0);
    }
  } else {
    // -------------------------------- epilogue ----------------------------------
    // Group g (four warps, one per TMEM lane quadrant) is pair g's reader: it
    // takes the CTA's tiles with local index i = g (mod kPairs).
    const int group = (warp - kFirstEpiWarp) >> 2;
    const int quad = warp & 3;  // TMEM lane quadrant this warp can access
    const int row = quad * 32 + lane;
    const int64_t words = (p.S + 31) / 32;
    // The scales of the group's j-th tile go to its ring slot j % kScSlots.
    // Each thread copies and later reads only its own row, so its own
    // cp.async.wait_group is the only ordering needed.
    float* ring = sc_ring + group * (kScSlots * kMaxL * kM);
    int64_t pf_t = t_begin + group, pf_b = pf_t / p.tiles_per_b;
    int pf_tile = (int)(pf_t % p.tiles_per_b), pf_slot = 0;
    auto prefetch = [&]() {
      if (pf_t < t_end) {
        const int64_t s = (int64_t)pf_tile * kM + row;
        const bool v = s < p.S;
        const float* src = p.k_scale + pf_b * p.sstride_b + (v ? s : 0);
        for (int l = 0; l < L; ++l)
          cp_async4(ring + (pf_slot * kMaxL + l) * kM + row, src + l * p.sstride_l, v ? 4u : 0u);
        pf_t += kEpiGroups;
        pf_tile += kEpiGroups;
        while (pf_tile >= p.tiles_per_b) {
          pf_tile -= p.tiles_per_b;
          ++pf_b;
        }
      }
      cp_async_commit();  // an empty group past the end keeps the group count uniform
      if (++pf_slot == kScSlots) pf_slot = 0;
    };
    for (int d = 0; d < kScDepth; ++d) prefetch();

    // the pair's accumulator ring, read in the order its issuer fills it
    uint32_t racc = 0, acc_phase = 0;
    int slot = 0;
    bool ok = true;
    int64_t b = t_begin / p.tiles_per_b, w_b = -1;
    int tile = (int)(t_begin % p.tiles_per_b) - 1;
    float* w_mine = w_smem[warp - kFirstEpiWarp];
    for (int64_t t = t_begin; t < t_end && ok; ++t) {
      if (++tile == p.tiles_per_b) {
        tile = 0;
        ++b;
      }
      if ((int)((t - t_begin) % kPairs) != group) continue;  // the other pair's tile
      if (b != w_b) {  // a new request: its weights into this warp's copy
        __syncwarp();
        for (int i = lane; i < L * kWStride; i += 32) w_mine[i] = __ldg(p.wq + b * L * kWStride + i);
        __syncwarp();
        w_b = b;
      }
      prefetch();                  // the group's tile kScDepth ahead
      cp_async_wait<kScDepth>();   // this tile's scales have landed
      const float* sc_t = ring + slot * kMaxL * kM + row;
      if (++slot == kScSlots) slot = 0;
      const int64_t s = (int64_t)tile * kM + row;
      const bool valid = s < p.S;  // rows past S read a zero scale and score 0
      float m = -INFINITY;
      for (int l = 0; l < L; ++l) {
        const float sc = sc_t[l * kM];
        const uint32_t acc = group * kRingAccs + racc;
        if (!mbar_wait(&bar_tfull[acc], acc_phase, &abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * kQTermRows;
        uint32_t r0[32], r1[32], lin[2];
        tmem_ld32(taddr, r0);
        tmem_ld32(taddr + 32, r1);
        tmem_ld2(taddr + kHeads, lin);  // q_w . k in two powers of two
        const float* wlayer = w_mine + l * kWStride;
        const float4* wl = reinterpret_cast<const float4*>(wlayer);
        float wr[kHeads];
#pragma unroll
        for (int i = 0; i < kHeads / 4; ++i) {
          const float4 v = wl[i];
          wr[4 * i] = v.x;
          wr[4 * i + 1] = v.y;
          wr[4 * i + 2] = v.z;
          wr[4 * i + 3] = v.w;
        }
        const float e1 = wlayer[kHeads], e2 = wlayer[kHeads + 1];
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&bar_tempty[acc]);  // the dots are in registers: the MMA may reuse the accumulator
        // q_h . k = 2^e_h (t1 + t2) . k with 2^e_h folded into w', and
        // ReLU(sc d) = (sc d + |sc| |d|) / 2 for either sign of sc: here
        // sum_h w'_h |d_h| (the absolute value folds into the FFMA), then the
        // linear half sc q_w.k
        float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
#pragma unroll
        for (int h = 0; h < 32; h += 4) {
          x0 = fmaf(wr[h], fabsf(__uint_as_float(r0[h])), x0);
          x1 = fmaf(wr[h + 1], fabsf(__uint_as_float(r0[h + 1])), x1);
          x2 = fmaf(wr[h + 2], fabsf(__uint_as_float(r0[h + 2])), x2);
          x3 = fmaf(wr[h + 3], fabsf(__uint_as_float(r0[h + 3])), x3);
        }
#pragma unroll
        for (int h = 0; h < 32; h += 4) {
          x0 = fmaf(wr[32 + h], fabsf(__uint_as_float(r1[h])), x0);
          x1 = fmaf(wr[33 + h], fabsf(__uint_as_float(r1[h + 1])), x1);
          x2 = fmaf(wr[34 + h], fabsf(__uint_as_float(r1[h + 2])), x2);
          x3 = fmaf(wr[35 + h], fabsf(__uint_as_float(r1[h + 3])), x3);
        }
        const float qwk = fmaf(e1, __uint_as_float(lin[0]), e2 * __uint_as_float(lin[1]));
        const float y = 0.5f * fmaf(sc, qwk, fabsf(sc) * ((x0 + x1) + (x2 + x3)));
        if (p.logits != nullptr && valid) p.logits[(b * L + l) * p.S + s] = y;
        m = fmaxf(m, y);
        if (++racc == (uint32_t)kRingAccs) {
          racc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) break;
      const uint32_t bits = __ballot_sync(0xffffffffu, valid && m >= p.thr_logit);
      const int64_t word = (int64_t)tile * (kM / 32) + quad;
      if (lane == 0 && word < words) p.mask[b * words + word] = bits;
      if (p.maxsig != nullptr && valid) p.maxsig[b * p.S + s] = 1.0f / (1.0f + expf(-m));
    }
    cp_async_wait<0>();  // no copy may still target shared memory when the CTA exits
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

size_t memindex_fp8_workspace_bytes(int B, int L) {
  return align256((size_t)B * L * kQLayerBytes) + align256((size_t)B * L * kWStride * 4);
}

namespace {

struct Fp8Args {
  const uint16_t* q;
  const float* w;
  const uint8_t* k8;
  const float* k_scale;
  int64_t key_stride_b, key_stride_l, sstride_b, sstride_l;
  int B, L;
  int64_t S;
  float thr_logit;
  uint32_t* mask;
  float* maxsig;
  float* logits;
  void* workspace;
};

fm_status launch_memindex_fp8(const Fp8Args& a, int num_sms, unsigned int* status, cudaStream_t stream) {
  const int tiles_per_b = (int)((a.S + kM - 1) / kM);
  const int64_t total = (int64_t)a.B * tiles_per_b;
  if (total == 0) return FM_OK;
  uint8_t* qsplit = static_cast<uint8_t*>(a.workspace);
  float* wq = reinterpret_cast<float*>(qsplit + align256((size_t)a.B * a.L * kQLayerBytes));
  memindex_fp8_prep_kernel<<<a.B * a.L, kPrepThreads, 0, stream>>>(a.q, a.w, qsplit, wq);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "memindex fp8 prep: launch: %s", cudaGetErrorString(e));

  CUtensorMap tmap_k, tmap_q;
  {
    // keys: dims (128 B, S, L, B), box (128, 128, 1, 1), 128-byte swizzle
    const uint64_t dims[4] = {(uint64_t)kDim, (uint64_t)a.S, (uint64_t)a.L, (uint64_t)a.B};
    const uint64_t strides[3] = {(uint64_t)kDim, (uint64_t)a.key_stride_l, (uint64_t)a.key_stride_b};
    const uint32_t box[4] = {(uint32_t)kDim, (uint32_t)kM, 1, 1};
    fm_status st = make_tmap(&tmap_k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, a.k8, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != FM_OK) return st;
  }
  {
    // split query: rows (B*L*kQRows) x 128 B, one box of kQRows rows per layer
    const uint64_t dims[2] = {(uint64_t)kDim, (uint64_t)a.B * a.L * kQRows};
    const uint64_t strides[1] = {(uint64_t)kDim};
    const uint32_t box[2] = {(uint32_t)kDim, (uint32_t)kQRows};
    fm_status st = make_tmap(&tmap_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, qsplit, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != FM_OK) return st;
  }
  const int smem_cap = 227 * 1024 - 10 * 1024;  // less the kernel's static shared memory
  const int fixed = 1024 + a.L * kQLayerBytes + kScRingBytes;
  int stages = (smem_cap - fixed) / kTileBytes;
  if (stages > kMaxStages) stages = kMaxStages;
  const int ring = stages / kPairs;  // each pair's own stage ring
  if (ring < 2) return set_error(FM_ERR_UNSUPPORTED, "memindex fp8: %d key stages per pair are too few", ring);
  const int smem = fixed + kPairs * ring * kTileBytes;

  Params p;
  p.wq = wq;
  p.k_scale = a.k_scale;
  p.sstride_b = a.sstride_b;
  p.sstride_l = a.sstride_l;
  p.mask = a.mask;
  p.maxsig = a.maxsig;
  p.logits = a.logits;
  p.status = status;
  p.S = a.S;
  p.total_tiles = total;
  p.tiles_per_b = tiles_per_b;
  p.L = a.L;
  p.stages = ring;
  p.thr_logit = a.thr_logit;
  e = cudaFuncSetAttribute(memindex_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "memindex fp8: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  const int grid = (int)(total < num_sms ? total : num_sms);
  memindex_fp8_kernel<<<grid, kThreads, smem, stream>>>(tmap_k, tmap_q, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "memindex fp8: launch: %s", cudaGetErrorString(e));
  return FM_OK;
}

}  // namespace
}  // namespace fm

FM_API size_t fm_memindex_fp8_workspace(int B, int L) {
  if (B < 0 || L < 1 || L > 4) return 0;
  return fm::memindex_fp8_workspace_bytes(B, L);
}

FM_API fm_status fm_memindex_score_mask_fp8(const uint16_t* q, const float* w, const uint8_t* k8, const float* k_scale,
                                            int64_t key_stride_b, int64_t key_stride_l, int64_t scale_stride_b,
                                            int64_t scale_stride_l, int B, int L, int64_t S, int n_h, int d,
                                            float threshold, uint32_t* mask_out, float* maxsig_out, float* logits_out,
                                            void* workspace, size_t workspace_bytes, fm_stream_t stream) {
  using namespace fm;
  if (n_h != 64 || d != 128)
    return set_error(FM_ERR_INVALID_ARG, "fm_memindex_score_mask_fp8: n_h=%d d=%d (need 64, 128)", n_h, d);
  if (B < 0 || L < 1 || L > 4 || S < 0 || S >= (int64_t(1) << 31))
    return set_error(FM_ERR_INVALID_ARG, "fm_memindex_score_mask_fp8: bad sizes B=%d L=%d S=%lld", B, L,
                     (long long)S);
  if (!(threshold > 0.0f && threshold < 1.0f))
    return set_error(FM_ERR_INVALID_ARG, "fm_memindex_score_mask_fp8: threshold %g not in (0, 1)", (double)threshold);
  if (B == 0 || S == 0) return FM_OK;
  if (!q || !w || !k8 || !k_scale || !mask_out)
    return set_error(FM_ERR_INVALID_ARG, "fm_memindex_score_mask_fp8: required pointer is NULL");
  if (!aligned(q, 16) || !aligned(w, 16) || !aligned(k8, 16) || !aligned(k_scale, 4) || !aligned(mask_out, 4) ||
      (maxsig_out && !aligned(maxsig_out, 4)) || (logits_out && !aligned(logits_out, 4)))
    return set_error(FM_ERR_INVALID_ARG, "fm_memindex_score_mask_fp8: misaligned pointer (q, w, k8: 16 bytes)");
  // key rows are 128 contiguous bytes; layer and request strides must be
  // multiples of 16 bytes and must not make rows of different (b, l) overlap
  if (key_stride_l % 16 != 0 || key_stride_b % 16 != 0 || (L > 1 && key_stride_l < S * d) ||
      (B > 1 && key_stride_b < (L > 1 ? key_stride_l * L : S * d)))
    return set_error(FM_ERR_INVALID_ARG, "fm_memindex_score_mask_fp8: bad key strides b=%lld l=%lld",
                     (long long)key_stride_b, (long long)key_stride_l);
  if ((L > 1 && scale_stride_l < S) || (B > 1 && scale_stride_b < (L > 1 ? scale_stride_l * L : S)) ||
      scale_stride_l < 0 || scale_stride_b < 0)
    return set_error(FM_ERR_INVALID_ARG, "fm_memindex_score_mask_fp8: bad scale strides b=%lld l=%lld",
                     (long long)scale_stride_b, (long long)scale_stride_l);
  const size_t need = memindex_fp8_workspace_bytes(B, L);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need)
    return set_error(FM_ERR_WORKSPACE, "fm_memindex_score_mask_fp8: workspace needs %zu bytes, 256-byte aligned",
                     need);
  int sms = 0;
  fm_status st = check_device(&sms);
  if (st != FM_OK) return st;
  unsigned int* status = nullptr;
  st = status_word(&status);
  if (st != FM_OK) return st;
  Fp8Args a;
  a.q = q;
  a.w = w;
  a.k8 = k8;
  a.k_scale = k_scale;
  a.key_stride_b = key_stride_b;
  a.key_stride_l = key_stride_l;
  a.sstride_b = scale_stride_b;
  a.sstride_l = scale_stride_l;
  a.B = B;
  a.L = L;
  a.S = S;
  a.thr_logit = (float)log((double)threshold / (1.0 - (double)threshold));
  a.mask = mask_out;
  a.maxsig = maxsig_out;
  a.logits = logits_out;
  a.workspace = workspace;
  return launch_memindex_fp8(a, sms, status, reinterpret_cast<cudaStream_t>(stream));
}

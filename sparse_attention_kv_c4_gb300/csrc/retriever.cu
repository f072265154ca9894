// retriever.cu -- the trained retriever's Memory Indexer, reading the packed
// compressed_k rows directly.
//
// Computes ("FlashMemory-DeepSeek-V4" README, "Retriever architecture",
// "compressed_k format", "Joint checkpoint + ensemble"; "FlashMemory-
// DeepSeek-V4: Lightning Index Ultra-Long Context via Lookahead Sparse
// Attention", sec. 3 "Memory Indexer scoring function"):
//     x[b,l,s] = sum_{h < n_h} w[b,l,h] * ReLU(q[b,l,h,:] . (scale * e4m3(k8)))
// where chunk s of (request b, layer l) is one 132-byte row: its 128 E4M3
// key bytes, then its fp32 dequant scale; then per chunk the layers' sigmoid
// scores are ensembled, e[b,s] = max_l sigma(x) (the union) or mean_l
// sigma(x), and the chunk is resident iff e >= threshold.  n_h is 128 (the
// retriever's heads) or 64.
//
// GB300 mapping.  A 132-byte row pitch is not a multiple of 16 bytes, so no
// tensor map can describe the keys and no UMMA shared-memory layout can use
// them in place.  Instead:
//   warp 0  producer: per request the split query (L x 2 n_h rows of 128 B,
//           SWIZZLE_128B TMA); per layer-tile one bulk copy of its 128 packed
//           rows (16,896 contiguous bytes) into the stage ring of the pair
//           (below) that takes the tile.
//   warps 11-14  the unpack group (one warp per TMEM lane quadrant): for
//           every layer-tile, thread = chunk row reads its 33 words from
//           shared memory (a 33-word row stride spreads a warp over all 32
//           banks) and writes the 128 key bytes into the owning pair's TMEM A
//           slot (tcgen05.st, lane = row): the MMA's A operand, with no
//           shared-memory re-layout; the scale goes to a shared-memory scale
//           ring of the pair.  A negative scale becomes positive with every
//           key sign bit flipped (the same dequantised key), so the scoring
//           needs only ReLU(sc d) = sc ReLU(d).
//   warps 3-10  two scoring groups of four warps (one per TMEM lane
//           quadrant): a group reads its layer-tile's n_h dots and scales and
//           computes y = sum_h w_h 2^e_h ReLU(scale (t1 + t2).k), the
//           per-layer logits, the ensemble, the mask word (ballot) and the
//           ensembled score.  (With the unpack in the same warps, the
//           shared-memory reads and TMEM stores sat on the scoring's
//           critical path.)
//   warps 1-2  UMMA issuers: per layer-tile 8 x tcgen05.mma kind::f8f6f4
//           M=128 N=n_h K=32 with A from TMEM, four K steps against the
//           query's t1 rows and four against its t2 rows into one
//           accumulator (the query split of fp8.cuh).
// Issuer m and scoring group m form pair m: the pair takes the CTA's tiles
// with local index = m (mod 2) and owns its stage ring, two TMEM A slots,
// four scale slots and its accumulators (256 TMEM columns).  Every ring has
// a single filler and a single reader (the producer / the unpack group / the
// issuer / the scoring group), so each parity wait is exact.
#include <math.h>

#include "fm_common.cuh"
#include "fm_internal.h"
#include "fp8.cuh"

#define FM_API extern "C" __attribute__((visibility("default")))

namespace fm {
namespace {

constexpr int kM = 128;                    // chunks per tile (UMMA M, TMEM lanes)
constexpr int kDim = 128;                  // E4M3 key bytes per chunk
constexpr int kRowBytes = kDim + 4;        // packed compressed_k row
constexpr int kRowWords = kRowBytes / 4;   // 33
constexpr int kTileBytes = kM * kRowBytes;  // 16,896 bytes per layer-tile
constexpr int kPairs = 2;
constexpr int kMmaWarps = kPairs;
constexpr int kFirstEpiWarp = 1 + kMmaWarps;
constexpr int kFirstUnpackWarp = kFirstEpiWarp + kPairs * 4;  // four unpack warps, one per TMEM lane quadrant
constexpr int kThreads = (kFirstUnpackWarp + 4) * 32;
constexpr int kSSlots = 4;                 // scale slots per pair (shared memory), handed from unpack to scoring
constexpr int kASlots = 2;                 // TMEM A slots per pair
constexpr int kACols = kDim / 4;           // 32 columns: 128 E4M3 bytes per lane
constexpr int kPairCols = 256;             // TMEM columns per pair
constexpr uint32_t kTmemCols = kPairs * kPairCols;
constexpr int kMaxRing = 6;                // key stages per pair
constexpr int kMaxDAccs = 3;
constexpr int kPrepThreads = 256;

// kLin: the linear half of the ReLU on the tensor core.  With ReLU(d) =
// (d + |d|) / 2 a chunk's score is sc/2 (q_w . k + sum_h w'_h |d_h|), where
// q_w = sum_h w_h q_h; q_w is split into four E4M3 terms (two per power of
// two) in four more rows of the t1 block of B, so the t1 MMAs (N = NH + 16)
// leave the four terms' dots in four more accumulator columns, the t2 MMAs
// keep N = NH, and the epilogue has one FFMA (|d| folded in) per head.
template <int NH, bool kLin>
struct Cfg {
  static constexpr int kBRows = NH + (kLin ? 16 : 0);                  // B rows per term block: the MMA's N
  static constexpr int kQTermBytes = kBRows * kDim;                   // the t1 block, then the t2 block
  static constexpr int kQLayerBytes = 2 * kQTermBytes;
  static constexpr int kDAccs = (kPairCols - kASlots * kACols) / kBRows;  // 1 for 128 heads, 3 for 64
  static constexpr int kWStride = NH + (kLin ? 4 : 0);  // floats per (request, layer) of wq: w', then 2^e1, 2^e2
  static constexpr int kMaxL = kLin ? 3 : 4;             // layers the launch takes (the launcher picks kLin by L)
};

// Programmatic dependent launch between the prep kernel and the scoring
// kernel: the prep lets the scoring kernel start at once, whose producer sends
// its first key copies (inputs of the call, which no kernel of the call
// writes) before griddepcontrol.wait; every read of the prep's output (the
// split query, the weights) comes after a wait.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Four consecutive 32-bit TMEM columns: thread i gets lane (base + i).
FM_DEV void tmem_ld4(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr)
               : "memory");
}

struct Params {
  const uint8_t* ck;         // packed rows
  int64_t ck_stride_b, ck_stride_l;  // bytes
  const float* wq;           // [B*L, n_h] head weights with 2^e_h folded in
  uint32_t* mask;
  float* ens;                // [B, S] ensembled score, or null
  float* logits;             // [B, L, S], or null
  unsigned int* status;
  int64_t S;
  int64_t total_tiles;
  int tiles_per_b;
  int L;
  int ring;                  // key stages per pair
  int mode;                  // 0 max, 1 mean
  float thr, thr_logit;
};

template <int NH, bool kLin>
__global__ void __launch_bounds__(kPrepThreads)
    retriever_prep_kernel(const uint16_t* __restrict__ q, const float* __restrict__ w, uint8_t* __restrict__ qsplit,
                          float* __restrict__ wq) {
  using C = Cfg<NH, kLin>;
  grid_dep_launch_dependents();
  const int64_t bl = blockIdx.x;
  uint8_t* t1 = qsplit + bl * C::kQLayerBytes;
  uint8_t* t2 = t1 + C::kQTermBytes;
  float* wl = wq + bl * C::kWStride;
  split_query(q + bl * NH * kDim, w + bl * NH, NH, kPrepThreads, t1, t2, wl);
  if constexpr (kLin) {
    // q_w[j] = sum_h w_h q_h[j] (fp32, heads in order); with 2^e1 putting
    // max|q_w| in (224, 448]: u1 = RNE(q_w 2^-e1), u2 = RNE(rest), then the
    // rest after those two times 2^8 the same way (u3, u4), so q_w =
    // 2^e1 (u1 + u2) + 2^(e1-8) (u3 + u4) to within 2^-18 of max|q_w|.
    // Rows NH .. NH+3 of the t1 block hold u1, u2, u3, u4, zeros in rows
    // NH+4 .. NH+15 (and in the t2 block's rows NH .., which no MMA reads).
    __shared__ float red[kPrepThreads / 32];
    const int j = threadIdx.x;
    float qw = 0.f;
    if (j < kDim) {
      const uint16_t* qb = q + bl * NH * kDim + j;
      for (int h = 0; h < NH; ++h)
        qw = fmaf(__ldg(w + bl * NH + h), __uint_as_float((uint32_t)__ldg(qb + (int64_t)h * kDim) << 16), qw);
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
      const uint32_t u4 = e4m3_rne(s2 - e4m3_value(u3));
      t1[NH * kDim + j] = (uint8_t)u1;
      t1[(NH + 1) * kDim + j] = (uint8_t)u2;
      t1[(NH + 2) * kDim + j] = (uint8_t)u3;
      t1[(NH + 3) * kDim + j] = (uint8_t)u4;
    }
    for (int i = threadIdx.x; i < 12 * kDim; i += kPrepThreads) t1[(NH + 4) * kDim + i] = 0;
    for (int i = threadIdx.x; i < 16 * kDim; i += kPrepThreads) t2[NH * kDim + i] = 0;
    if (threadIdx.x == 0) {
      wl[NH] = ldexpf(1.f, e);
      wl[NH + 1] = ldexpf(1.f, e - 8);
      wl[NH + 2] = 0.f;
      wl[NH + 3] = 0.f;
    }
  }
}

template <int NH, bool kLin>
__global__ void __launch_bounds__(kThreads, 1)
    retriever_kernel(const __grid_constant__ CUtensorMap tmap_q, const Params p) {
  using C = Cfg<NH, kLin>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_smem = smem;
  uint8_t* k_smem = smem + p.L * C::kQLayerBytes;  // [pair][ring] stages of kTileBytes

  __shared__ __align__(8) uint64_t bar_full[kPairs * kMaxRing], bar_empty[kPairs * kMaxRing];
  __shared__ __align__(8) uint64_t bar_afull[kPairs * kASlots], bar_aempty[kPairs * kASlots];
  __shared__ __align__(8) uint64_t bar_tfull[kPairs * kMaxDAccs], bar_tempty[kPairs * kMaxDAccs];
  __shared__ __align__(8) uint64_t bar_sfull[kPairs * kSSlots], bar_sempty[kPairs * kSSlots];
  __shared__ __align__(8) uint64_t bar_qfull, bar_qempty, bar_drain;
  __shared__ float scale_ring[kPairs * kSSlots][kM];  // each chunk's (non-negative) scale, per layer-tile
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  // one copy of the current request's weights per scoring warp, so a warp
  // refreshes its own copy with __syncwarp alone (a static array: copies in
  // dynamic shared memory measured 2.6% slower)
  __shared__ __align__(16) float w_smem[kPairs * 4][C::kMaxL * C::kWStride];

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int L = p.L, ring = p.ring;
  const int64_t t_begin = p.total_tiles * blockIdx.x / gridDim.x;
  const int64_t t_end = p.total_tiles * (blockIdx.x + 1) / gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairs * ring; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 128);  // the group read the stage's rows
    }
    for (int i = 0; i < kPairs * kASlots; ++i) {
      mbar_init(&bar_afull[i], 128);  // the group wrote the A slot
      mbar_init(&bar_aempty[i], 1);   // the MMAs reading it finished
    }
    for (int i = 0; i < kPairs * C::kDAccs; ++i) {
      mbar_init(&bar_tfull[i], 1);
      mbar_init(&bar_tempty[i], 128);
    }
    for (int i = 0; i < kPairs * kSSlots; ++i) {
      mbar_init(&bar_sfull[i], 128);   // the unpack group wrote the slot's scales
      mbar_init(&bar_sempty[i], 128);  // the scoring group read them
    }
    mbar_init(&bar_qfull, 1);
    mbar_init(&bar_qempty, kMmaWarps);
    mbar_init(&bar_drain, kMmaWarps);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) tma_prefetch(&tmap_q);
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
      // ------------------------------ producer ---------------------------------
      uint32_t rstage[kPairs] = {}, rphase[kPairs] = {}, q_phase = 0;
      int issued[kPairs * kMaxRing];
      for (int s = 0; s < kPairs * kMaxRing; ++s) issued[s] = -1;
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
        // the request's split query: t1 block, then t2 block (one box of
        // kBRows rows each) per layer
        auto load_q = [&](int64_t rb) {
          mbar_arrive_expect_tx(&bar_qfull, (uint32_t)(L * C::kQLayerBytes));
          for (int l = 0; l < L; ++l)
            for (int tb = 0; tb < 2; ++tb)
              tma_load_2d(q_smem + l * C::kQLayerBytes + tb * C::kQTermBytes, &tmap_q, &bar_qfull, 0,
                          (int32_t)(((rb * L + l) * 2 + tb) * C::kBRows));
          q_issued = (q_issued + 1) & 1;
        };
        bool q_after_keys = false;  // the first request: its key copies go out before the wait for the prep
        if (b != cur_b) {
          if (cur_b >= 0) {
            if (!mbar_wait(&bar_qempty, q_phase, &abort_flag, p.status)) break;
            q_phase ^= 1;
            load_q(b);
          } else {
            q_after_keys = true;
          }
          cur_b = b;
        }
        const int m = (int)((t - t_begin) % kPairs);
        const int64_t rows = p.S - (int64_t)tile * kM < kM ? p.S - (int64_t)tile * kM : kM;
        const uint32_t bytes = (uint32_t)(rows * kRowBytes);  // S % 4 == 0: a multiple of 16
        for (int l = 0; l < L; ++l) {
          const uint32_t stage = m * ring + rstage[m], phase = rphase[m];
          if (!mbar_wait(&bar_empty[stage], phase ^ 1u, &abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bar_full[stage], bytes);
          bulk_load(k_smem + stage * kTileBytes,
                    p.ck + b * p.ck_stride_b + l * p.ck_stride_l + (int64_t)tile * kTileBytes, bytes,
                    &bar_full[stage]);
          issued[stage] = (int)phase;
          if (++rstage[m] == (uint32_t)ring) {
            rstage[m] = 0;
            rphase[m] ^= 1u;
          }
        }
        if (q_after_keys && ok) {
          grid_dep_wait();
          load_q(b);
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
      const int me = warp - 1;
      const uint32_t idesc = idesc_e4m3_f32(kM, C::kBRows), idesc2 = idesc_e4m3_f32(kM, NH);
      uint32_t aslot = 0, a_phase = 0, dacc = 0, d_phase = 0, q_phase = 0;
      int64_t cur_b = -1;
      bool ok = true;
      const uint64_t b_desc0 = sdesc_sw128(smem_u32(q_smem));
      const uint32_t pair_base = tmem_base + (uint32_t)(me * kPairCols);
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
          const int ai = me * kASlots + (int)aslot, di = me * C::kDAccs + (int)dacc;
          if (!mbar_wait(&bar_afull[ai], a_phase, &abort_flag, p.status) ||
              !mbar_wait(&bar_tempty[di], d_phase ^ 1u, &abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_tmem = pair_base + aslot * kACols;
          const uint32_t d_tmem = pair_base + kASlots * kACols + dacc * C::kBRows;
          // B: the layer's t1 block, then its t2 block kQTermBytes later
          // (descriptor addresses count 16-byte units); A: 8 TMEM columns
          // (32 E4M3 values per lane) per K step
          const uint64_t b_desc = b_desc0 + (uint64_t)(l * (C::kQLayerBytes >> 4));
          constexpr uint64_t kT2 = (uint64_t)C::kQTermBytes >> 4;
#pragma unroll
          for (int k = 0; k < kDim / 32; ++k)
            umma_e4m3_ts(d_tmem, a_tmem + 8 * k, b_desc + 2 * k, idesc, k != 0 ? 1u : 0u);
#pragma unroll
          for (int k = 0; k < kDim / 32; ++k) umma_e4m3_ts(d_tmem, a_tmem + 8 * k, b_desc + kT2 + 2 * k, idesc2, 1u);
          umma_commit(&bar_aempty[ai]);
          umma_commit(&bar_tfull[di]);
          if (++aslot == (uint32_t)kASlots) {
            aslot = 0;
            a_phase ^= 1u;
          }
          if (++dacc == (uint32_t)C::kDAccs) {
            dacc = 0;
            d_phase ^= 1u;
          }
        }
      }
      umma_commit(&bar_drain);  // every MMA issued above has finished before TMEM is freed
      mbar_wait_drain(&bar_drain, 0);
    }
  } else if (warp < kFirstUnpackWarp) {
    // ------------------------------ scoring groups ------------------------------
    const int group = (warp - kFirstEpiWarp) >> 2;
    const int quad = warp & 3;  // TMEM lane quadrant this warp can access
    const int row = quad * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(group * kPairCols);
    const int64_t words = (p.S + 31) / 32;
    float* w_mine = w_smem[warp - kFirstEpiWarp];
    const int64_t span = t_end - t_begin;
    const int64_t n_tiles = span > group ? (span - group + kPairs - 1) / kPairs : 0;  // the pair's tiles

    // The pair's tiles t_begin + group + 2i in order, each scored layer by
    // layer: the request, the tile's rows and output pointers are set once per
    // tile, so a layer-tile carries little besides its own waits and dots.
    int64_t b = (t_begin + group) / p.tiles_per_b;
    int tile = (int)((t_begin + group) % p.tiles_per_b);
    uint32_t dacc = 0, d_phase = 0, sslot = 0, s_phase = 0;
    int64_t w_b = -1;
    bool ok = true;
    grid_dep_wait();  // the weights come from the prep kernel
    for (int64_t i = 0; i < n_tiles && ok; ++i) {
      if (b != w_b) {  // a new request: its weights into this warp's copy
        __syncwarp();
        for (int k = lane; k < L * C::kWStride; k += 32) w_mine[k] = __ldg(p.wq + b * L * C::kWStride + k);
        __syncwarp();
        w_b = b;
      }
      const int64_t s = (int64_t)tile * kM + row;
      const bool valid = s < p.S;
      float* const lg = p.logits != nullptr ? p.logits + b * L * p.S + s : nullptr;
      float acc_m = -INFINITY, acc_sum = 0.f;
      for (int l = 0; l < L; ++l) {
        // the chunk's scale, from the unpack group (>= 0: a negative scale's
        // sign went into the key bytes)
        const int si = group * kSSlots + (int)sslot;
        if (!mbar_wait(&bar_sfull[si], s_phase, &abort_flag, p.status)) {
          ok = false;
          break;
        }
        const float sc = scale_ring[si][row];
        mbar_arrive(&bar_sempty[si]);
        if (++sslot == (uint32_t)kSSlots) {
          sslot = 0;
          s_phase ^= 1u;
        }
        const int di = group * C::kDAccs + (int)dacc;
        if (!mbar_wait(&bar_tfull[di], d_phase, &abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = lane_base + kASlots * kACols + dacc * C::kBRows;
        const float4* wl = reinterpret_cast<const float4*>(w_mine + l * C::kWStride);
        float y = 0.f;
        uint32_t lin[4] = {0u, 0u, 0u, 0u};
        const float scc = kLin ? 0.5f * sc : sc;  // each chunk's partial sum times the scale as it lands
        // 32 heads at a time, double-buffered: the load of chunk c + 1 is in
        // flight while chunk c is summed, so the accumulator is released one
        // load latency earlier
        uint32_t r[2][32];
        tmem_ld32(taddr, r[0]);
        if constexpr (kLin) tmem_ld4(taddr + NH, lin);  // q_w . k as four terms' dots
#pragma unroll
        for (int c = 0; c < NH / 32; ++c) {
          tmem_ld_wait();
          if (c + 1 < NH / 32) {
            tmem_ld32(taddr + (c + 1) * 32, r[(c + 1) & 1]);
          } else {
            tc_fence_before();
            mbar_arrive(&bar_tempty[di]);  // the dots are in registers: the MMA may reuse the accumulator
          }
          const uint32_t* rc = r[c & 1];
          // q_h . k = 2^e_h (t1 + t2) . k; 2^e_h is folded into w, and
          // ReLU(sc d) = sc ReLU(d) for sc >= 0: one multiply per chunk
          float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
#pragma unroll
          for (int h = 0; h < 32; h += 4) {
            const float4 wv = wl[c * 8 + h / 4];
            if constexpr (kLin) {  // w |d| (the absolute value folds into the FFMA)
              x0 = fmaf(wv.x, fabsf(__uint_as_float(rc[h])), x0);
              x1 = fmaf(wv.y, fabsf(__uint_as_float(rc[h + 1])), x1);
              x2 = fmaf(wv.z, fabsf(__uint_as_float(rc[h + 2])), x2);
              x3 = fmaf(wv.w, fabsf(__uint_as_float(rc[h + 3])), x3);
            } else {
              x0 = fmaf(wv.x, fmaxf(__uint_as_float(rc[h]), 0.f), x0);
              x1 = fmaf(wv.y, fmaxf(__uint_as_float(rc[h + 1]), 0.f), x1);
              x2 = fmaf(wv.z, fmaxf(__uint_as_float(rc[h + 2]), 0.f), x2);
              x3 = fmaf(wv.w, fmaxf(__uint_as_float(rc[h + 3]), 0.f), x3);
            }
          }
          y = fmaf(scc, (x0 + x1) + (x2 + x3), y);
        }
        if constexpr (kLin) {
          const float* we = w_mine + l * C::kWStride + NH;  // 2^e1, 2^e2
          const float hi = __uint_as_float(lin[0]) + __uint_as_float(lin[1]);
          const float lo = __uint_as_float(lin[2]) + __uint_as_float(lin[3]);
          y = fmaf(scc, fmaf(we[0], hi, we[1] * lo), y);
        }
        if (++dacc == (uint32_t)C::kDAccs) {
          dacc = 0;
          d_phase ^= 1u;
        }
        if (lg != nullptr && valid) lg[l * p.S] = y;
        if (p.mode == 0)
          acc_m = fmaxf(acc_m, y);
        else
          acc_sum += 1.0f / (1.0f + expf(-y));
      }
      if (!ok) break;
      // the ensemble over the tile's layers
      float e;
      bool res;
      if (p.mode == 0) {  // max of sigmoids = sigmoid of the max: compare the logit
        e = 1.0f / (1.0f + expf(-acc_m));
        res = valid && acc_m >= p.thr_logit;
      } else {
        e = acc_sum / (float)L;
        res = valid && e >= p.thr;
      }
      const uint32_t bits = __ballot_sync(0xffffffffu, res);
      const int64_t word = (int64_t)tile * (kM / 32) + quad;
      if (lane == 0 && word < words) p.mask[b * words + word] = bits;
      if (p.ens != nullptr && valid) p.ens[b * p.S + s] = e;
      tile += kPairs;
      while (tile >= p.tiles_per_b) {
        tile -= p.tiles_per_b;
        ++b;
      }
    }
  } else {
    // ------------------------------ unpack group --------------------------------
    // Every layer-tile of the CTA, in order (tile i belongs to pair i % 2):
    // thread = chunk row reads its 33 words from the pair's stage (a 33-word
    // row stride spreads a warp over all 32 banks), frees the stage, moves a
    // negative scale's sign into the key bytes, writes the 128 key bytes into
    // the pair's next TMEM A slot (tcgen05.st, lane = row) and the scale into
    // the pair's next scale slot.  Doing this in warps of its own takes the
    // row unpack off the scoring warps' critical path.
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    // each pair's ring positions, in registers (a runtime-indexed array of
    // them would live in local memory)
    struct Ring {
      uint32_t lstage, lphase, aslot, a_phase, sslot, s_phase;
    };
    Ring r0 = {}, r1 = {};
    // one layer-tile of pair m
    auto unpack = [&](Ring& c, const int m, const bool valid) -> bool {
      const uint32_t stage = m * ring + c.lstage;
      if (!mbar_wait(&bar_full[stage], c.lphase, &abort_flag, p.status)) return false;
      const uint32_t* src = reinterpret_cast<const uint32_t*>(k_smem + stage * kTileBytes) + row * kRowWords;
      uint32_t kw[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) kw[i] = valid ? src[i] : 0u;
      float sc = valid ? __uint_as_float(src[32]) : 0.f;
      mbar_arrive(&bar_empty[stage]);
      if (++c.lstage == (uint32_t)ring) {
        c.lstage = 0;
        c.lphase ^= 1u;
      }
      if (sc < 0.f) {  // scale * e4m3(k) == (-scale) * e4m3(-k): flip every sign bit, keep the scale positive
        sc = -sc;
#pragma unroll
        for (int i = 0; i < 32; ++i) kw[i] ^= 0x80808080u;
      }
      const int ai = m * kASlots + (int)c.aslot;
      if (!mbar_wait(&bar_aempty[ai], c.a_phase ^ 1u, &abort_flag, p.status)) return false;
      tc_fence_after();
      tmem_st32(tmem_base + lane_off + (uint32_t)(m * kPairCols) + c.aslot * kACols, kw);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar_afull[ai]);
      if (++c.aslot == (uint32_t)kASlots) {
        c.aslot = 0;
        c.a_phase ^= 1u;
      }
      const int si = m * kSSlots + (int)c.sslot;
      if (!mbar_wait(&bar_sempty[si], c.s_phase ^ 1u, &abort_flag, p.status)) return false;
      scale_ring[si][row] = sc;
      mbar_arrive(&bar_sfull[si]);
      if (++c.sslot == (uint32_t)kSSlots) {
        c.sslot = 0;
        c.s_phase ^= 1u;
      }
      return true;
    };
    int tile = (int)(t_begin % p.tiles_per_b) - 1;
    bool ok = true;
    for (int64_t t = t_begin; t < t_end && ok; ++t) {
      if (++tile == p.tiles_per_b) tile = 0;
      const bool valid = (int64_t)tile * kM + row < p.S;  // rows past S hold stale bytes
      const bool pair1 = ((t - t_begin) & 1) != 0;
      for (int l = 0; l < L && ok; ++l) ok = pair1 ? unpack(r1, 1, valid) : unpack(r0, 0, valid);
    }
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// The split query [B*L][2 term blocks][rows][128] and the weights
// [B*L][stride]; at 128 heads sized for the linear half's wider layout (16
// more rows per term block, 4 more weights), which either launch fits in.
size_t retriever_ws_bytes(int B, int L, int n_h) {
  const int rows = n_h == 128 ? n_h + 16 : n_h, stride = n_h == 128 ? n_h + 4 : n_h;
  return align256((size_t)B * L * 2 * rows * kDim) + align256((size_t)B * L * stride * 4);
}

struct RetrieverArgs {
  const uint16_t* q;
  const float* w;
  const uint8_t* ck;
  int64_t ck_stride_b, ck_stride_l;
  int B, L, n_h, mode;
  int64_t S;
  float thr;
  uint32_t* mask;
  float* ens;
  float* logits;
  void* workspace;
};

// Key stages per pair that fit beside L layers of the split query (less the
// static shared memory: the weight copies, the scale ring, the barriers); 0
// for more layers than the configuration takes.
template <int NH, bool kLin>
int retriever_ring(int L) {
  using C = Cfg<NH, kLin>;
  if (L > C::kMaxL) return 0;
  const int smem_cap = 227 * 1024 - (int)sizeof(float) * kPairs * 4 * C::kMaxL * C::kWStride -
                       (int)sizeof(float) * kPairs * kSSlots * kM - 2048;
  const int ring = (smem_cap - 1024 - L * C::kQLayerBytes) / (kPairs * kTileBytes);
  return ring > kMaxRing ? kMaxRing : ring;
}

template <int NH, bool kLin>
fm_status launch_retriever_cfg(const RetrieverArgs& a, int num_sms, unsigned int* status, cudaStream_t stream) {
  using C = Cfg<NH, kLin>;
  const int tiles_per_b = (int)((a.S + kM - 1) / kM);
  const int64_t total = (int64_t)a.B * tiles_per_b;
  if (total == 0) return FM_OK;
  uint8_t* qsplit = static_cast<uint8_t*>(a.workspace);
  float* wq = reinterpret_cast<float*>(qsplit + align256((size_t)a.B * a.L * C::kQLayerBytes));
  retriever_prep_kernel<NH, kLin><<<a.B * a.L, kPrepThreads, 0, stream>>>(a.q, a.w, qsplit, wq);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "retriever prep: launch: %s", cudaGetErrorString(e));

  CUtensorMap tmap_q;
  {
    // split query: rows (B*L*2*kBRows) x 128 B, one box per term block
    const uint64_t dims[2] = {(uint64_t)kDim, (uint64_t)a.B * a.L * 2 * C::kBRows};
    const uint64_t strides[1] = {(uint64_t)kDim};
    const uint32_t box[2] = {(uint32_t)kDim, (uint32_t)C::kBRows};
    fm_status st = make_tmap(&tmap_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, qsplit, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != FM_OK) return st;
  }
  const int ring = retriever_ring<NH, kLin>(a.L);
  if (ring < 2) return set_error(FM_ERR_UNSUPPORTED, "retriever: %d key stages per pair are too few", ring);
  const int smem = 1024 + a.L * C::kQLayerBytes + kPairs * ring * kTileBytes;

  Params p;
  p.ck = a.ck;
  p.ck_stride_b = a.ck_stride_b;
  p.ck_stride_l = a.ck_stride_l;
  p.wq = wq;
  p.mask = a.mask;
  p.ens = a.ens;
  p.logits = a.logits;
  p.status = status;
  p.S = a.S;
  p.total_tiles = total;
  p.tiles_per_b = tiles_per_b;
  p.L = a.L;
  p.ring = ring;
  p.mode = a.mode;
  p.thr = a.thr;
  p.thr_logit = logf(a.thr / (1.0f - a.thr));
  e = cudaFuncSetAttribute(retriever_kernel<NH, kLin>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "retriever: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  const int grid = (int)(total < num_sms ? total : num_sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, retriever_kernel<NH, kLin>, tmap_q, p);
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "retriever: launch: %s", cudaGetErrorString(e));
  return FM_OK;
}

// The linear half on the tensor core wherever it still leaves three key
// stages per pair (128 heads, up to three layers); else the ReLU in the
// epilogue (two stages cost 7% at three layers).
template <int NH>
fm_status launch_retriever(const RetrieverArgs& a, int num_sms, unsigned int* status, cudaStream_t stream) {
  if constexpr (NH == 128)
    if (retriever_ring<NH, true>(a.L) >= 3) return launch_retriever_cfg<NH, true>(a, num_sms, status, stream);
  return launch_retriever_cfg<NH, false>(a, num_sms, status, stream);
}

}  // namespace
}  // namespace fm

FM_API size_t fm_retriever_workspace(int B, int L, int n_h) {
  if (B < 0 || L < 1 || L > 4 || (n_h != 64 && n_h != 128)) return 0;
  return fm::retriever_ws_bytes(B, L, n_h);
}

FM_API fm_status fm_retriever_score_mask(const uint16_t* q, const float* w, const uint8_t* compressed_k,
                                         int64_t ck_stride_b, int64_t ck_stride_l, int B, int L, int64_t S, int n_h,
                                         int d, int ensemble, float threshold, uint32_t* mask_out, float* ens_out,
                                         float* logits_out, void* workspace, size_t workspace_bytes,
                                         fm_stream_t stream) {
  using namespace fm;
  if ((n_h != 64 && n_h != 128) || d != 128)
    return set_error(FM_ERR_INVALID_ARG, "fm_retriever_score_mask: n_h=%d d=%d (need 64 or 128, 128)", n_h, d);
  if (B < 0 || L < 1 || L > 4 || S < 0 || S >= (int64_t(1) << 31) || S % 4 != 0)
    return set_error(FM_ERR_INVALID_ARG, "fm_retriever_score_mask: bad sizes B=%d L=%d S=%lld (S %% 4 == 0)", B, L,
                     (long long)S);
  if (ensemble != FM_ENSEMBLE_MAX && ensemble != FM_ENSEMBLE_MEAN)
    return set_error(FM_ERR_INVALID_ARG, "fm_retriever_score_mask: ensemble %d is not max (0) or mean (1)", ensemble);
  if (!(threshold > 0.0f && threshold < 1.0f))
    return set_error(FM_ERR_INVALID_ARG, "fm_retriever_score_mask: threshold %g not in (0, 1)", (double)threshold);
  if (B == 0 || S == 0) return FM_OK;
  if (!q || !w || !compressed_k || !mask_out)
    return set_error(FM_ERR_INVALID_ARG, "fm_retriever_score_mask: required pointer is NULL");
  if (!aligned(q, 16) || !aligned(w, 16) || !aligned(compressed_k, 16) || !aligned(mask_out, 4) ||
      (ens_out && !aligned(ens_out, 4)) || (logits_out && !aligned(logits_out, 4)))
    return set_error(FM_ERR_INVALID_ARG, "fm_retriever_score_mask: misaligned pointer (q, w, compressed_k: 16 bytes)");
  // packed rows are 132 contiguous bytes; layer and request strides must be
  // multiples of 16 bytes and must not make rows of different (b, l) overlap
  const int64_t rows_bytes = S * (d + 4);
  if (ck_stride_l % 16 != 0 || ck_stride_b % 16 != 0 || (L > 1 && ck_stride_l < rows_bytes) ||
      (B > 1 && ck_stride_b < (L > 1 ? ck_stride_l * L : rows_bytes)))
    return set_error(FM_ERR_INVALID_ARG, "fm_retriever_score_mask: bad strides b=%lld l=%lld",
                     (long long)ck_stride_b, (long long)ck_stride_l);
  const size_t need = retriever_ws_bytes(B, L, n_h);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need)
    return set_error(FM_ERR_WORKSPACE, "fm_retriever_score_mask: workspace needs %zu bytes, 256-byte aligned", need);
  int sms = 0;
  fm_status st = check_device(&sms);
  if (st != FM_OK) return st;
  unsigned int* status = nullptr;
  st = status_word(&status);
  if (st != FM_OK) return st;
  RetrieverArgs a;
  a.q = q;
  a.w = w;
  a.ck = compressed_k;
  a.ck_stride_b = ck_stride_b;
  a.ck_stride_l = ck_stride_l;
  a.B = B;
  a.L = L;
  a.n_h = n_h;
  a.mode = ensemble;
  a.S = S;
  a.thr = threshold;
  a.mask = mask_out;
  a.ens = ens_out;
  a.logits = logits_out;
  a.workspace = workspace;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return n_h == 128 ? launch_retriever<128>(a, sms, status, s) : launch_retriever<64>(a, sms, status, s);
}

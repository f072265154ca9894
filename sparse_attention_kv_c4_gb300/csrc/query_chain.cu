// query_chain.cu -- the query side of a CSA layer's indexer: from a token's
// hidden state to the query heads and head weights the Memory Indexer scores
// with ("FlashMemory-DeepSeek-V4" README, "Retriever architecture" and
// "Hyperparameters"):
//     a = wq_a . h                         Linear dim -> r (no bias)
//     c = RMSNorm(a; q_norm, eps)
//     u = wq_b . c                         Linear r -> n_h * 128
//     q_h = Hadamard(RoPE_yarn(u_h, pos))  per head: rotary on the last 64 of
//                                          128 entries, then the normalised
//                                          Walsh-Hadamard transform
//     w = (w_proj . h) * 128^-1/2 * n_h^-1/2
//
// GB300 mapping.  For a decode batch (tens of tokens) the three projections
// stream 86 MB of bf16 weights per layer against a few kilobytes of
// activations: HBM-bound matrix products with 30 to 60 FLOP per weight byte,
// more than the CUDA cores can sustain at full bandwidth.  They run on the
// tensor cores with the weights as the streamed operand:
//   proj_gemm_kernel      one CTA per (128-row weight tile, K split): a TMA
//                         producer streams [128 rows x 128] weight chunks as
//                         two SWIZZLE_128B atoms (the UMMA A operand) and the
//                         matching [tokens x 128] activation chunks (B, tokens
//                         padded to a multiple of 16 by the copy's zero fill);
//                         one thread issues 8 tcgen05.mma kind::f16 M=128
//                         N=tokens K=16 per chunk into a TMEM accumulator;
//                         four epilogue warps write the fp32 partial sums
//                         (thread = weight row).  wq_a and
//                         w_proj share the hidden state, so they are one launch
//                         (w_proj's tile after wq_a's).  Each GEMM is split
//                         along K so that tiles x splits fills the SMs once.
//   rmsnorm_kernel        one CTA per (token, layer): sums the K-split
//                         partials of a in a fixed order, RMSNorm in fp32,
//                         the normalised row rounded to bf16 (wq_b's input
//                         type); the head weights w from w_proj's partials;
//                         and, once per token, the rotary (cos, sin) of its
//                         32 pairs: the angle pos * theta'_i formed and
//                         reduced modulo 2 pi in fp64 (positions reach 2^20
//                         and beyond, where an fp32 angle would lose whole
//                         radians), sine and cosine of the reduced angle in
//                         fp32.
//   rope_hadamard_kernel  one warp per (layer, token, head), four entries per
//                         lane: sums u's partials, rotates the last 64 entries
//                         with the token's (cos, sin), runs the Walsh-Hadamard
//                         butterflies in registers (strides 1 and 2 inside a
//                         lane, 4..64 across lanes by shuffles), and writes q
//                         as bf16 (and fp32 when asked).
// Partial sums are reduced in a fixed order, so results do not depend on
// scheduling.
#include <cuda_bf16.h>
#include <math.h>

#include <cmath>

#include "fm_common.cuh"
#include "fm_internal.h"

#define FM_API extern "C" __attribute__((visibility("default")))

namespace fm {
namespace {

constexpr int kHeadDim = 128;
constexpr int kRopeDim = 64;

__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }

// Programmatic dependent launch.  The chain's kernels are launched with
// programmatic stream serialisation: each may start while its predecessor
// finishes, and waits (griddepcontrol.wait) for the predecessor's completion
// and memory before it reads or writes global memory -- except that the
// second GEMM issues its first weight chunks before its wait (the weights are
// inputs of the call, never written by the kernels it can overlap: the
// chain's own RMSNorm and first GEMM).  A predecessor that does not trigger
// early (any kernel outside the chain) completes before the chain's first
// GEMM starts; the rotary kernel triggers early, so a following call's first
// GEMM sets up while it runs.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, unsigned block, size_t smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// One device pointer per layer (by value).
struct LayerPtrs {
  const uint16_t* p[4];
};

// Rotary frequencies theta'_i of the 32 pairs, computed once per call on the
// host (fp64) and passed by value.
struct RopeFreqs {
  double f[kRopeDim / 2];
};

// ---------------------------------------------------------------------------
// Projection GEMM for a few tokens, over up to kGMaxMats weight matrices of
// up to kGMaxLayers layers in one launch:
//     part[layer][split][t][col] = sum_{k in split} X_layer[t, k] * W_m[row, k]
// with matrix m's 128-row tiles numbered from mat_tile0[m], its rows placed at
// column (mat_col_tile[m] + tile) * 128 + row of its layer's part rows.
// ---------------------------------------------------------------------------
constexpr int kGM = 128;                  // weight rows per tile (UMMA M, TMEM lanes)
constexpr int kGK = 64;                   // K elements of one 128-byte swizzle atom
constexpr int kGAtomA = kGM * kGK * 2;    // 16 KB of weights per atom
constexpr int kGAtoms = 2;                // atoms per stage: a chunk is 128 K elements (8 MMAs per barrier round trip)
constexpr int kGKStage = kGK * kGAtoms;
constexpr int kGThreads = 192;            // producer warp, issuer warp, four epilogue warps
constexpr int kGMaxStages = 8;
constexpr int kGMaxTokens = 256;          // tokens per launch (UMMA N <= 256)
constexpr int kGMaxSplits = 16;
constexpr int kGSizingSms = 160;          // workspace sizing bound on the SM count (GB300: 152)
constexpr int kGMaxLayers = 4;
constexpr int kGMaxMats = 2 * kGMaxLayers;

struct GemmMaps {
  CUtensorMap w[kGMaxMats];   // weight matrices [rows, K] bf16
  CUtensorMap x[kGMaxLayers]; // each layer's activations [T, K] bf16
};

struct GemmParams {
  float* part;
  unsigned int* status;
  int64_t ld_part;     // columns of one layer's part rows
  int64_t t_rows;      // rows of one (layer, split) block of part (all tokens of the call)
  int t_base;          // first token of this launch
  int T;               // tokens in this launch (<= kGMaxTokens)
  int tpad;            // UMMA N: T rounded up to 16
  int kc;              // K chunks
  int n_mats;
  int mat_tile0[kGMaxMats + 1];  // first tile of each matrix (prefix over the matrices)
  int mat_layer[kGMaxMats];
  int mat_col_tile[kGMaxMats];   // the matrix's first column tile in its layer's part rows
  int splits;
  int stages;
  uint32_t tmem_cols;
  int prefetch_weights;  // issue the first stages' weight chunks before the dependency wait
};

__global__ void __launch_bounds__(kGThreads, 1)
    proj_gemm_kernel(const __grid_constant__ GemmMaps maps, const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int b_bytes = p.tpad * 128;                  // one activation atom
  const int stage_bytes = kGAtoms * (kGAtomA + b_bytes);  // A atoms, then B atoms; all multiples of 1 KB

  __shared__ __align__(8) uint64_t bar_full[kGMaxStages], bar_empty[kGMaxStages], bar_tfull, bar_drain;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int tile = blockIdx.x / p.splits, split = blockIdx.x % p.splits;
  const int c_begin = (int)((int64_t)p.kc * split / p.splits);
  const int c_end = (int)((int64_t)p.kc * (split + 1) / p.splits);  // > c_begin: splits <= kc
  int m = 0;
  while (m + 1 < p.n_mats && tile >= p.mat_tile0[m + 1]) ++m;
  const int tile_in = tile - p.mat_tile0[m];
  const int layer = p.mat_layer[m];
  const int row0 = tile_in * kGM;
  const CUtensorMap* wmap = &maps.w[m];
  const CUtensorMap* xmap = &maps.x[layer];
  const int stages = p.stages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    mbar_init(&bar_tfull, 1);
    mbar_init(&bar_drain, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(wmap);
    tma_prefetch(xmap);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_slot;
  grid_dep_launch_dependents();  // the next kernel may start (it waits for this one's completion)

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------ TMA producer ------------------------------
      int issued[kGMaxStages];
      for (int s = 0; s < kGMaxStages; ++s) issued[s] = -1;
      // The first stages' weight chunks go out before the dependency wait:
      // weights are never written by the kernels this one may overlap.  The
      // activation chunks (the previous kernel's output) follow the wait.
      const int pre = !p.prefetch_weights ? 0 : (c_end - c_begin < stages ? c_end - c_begin : stages);
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&bar_full[i], (uint32_t)stage_bytes);
        for (int a = 0; a < kGAtoms; ++a)
          tma_load_2d(smem + i * stage_bytes + a * kGAtomA, wmap, &bar_full[i], (c_begin + i) * kGKStage + a * kGK,
                      row0);
        issued[i] = 0;
      }
      grid_dep_wait();
      for (int i = 0; i < pre; ++i)
        for (int a = 0; a < kGAtoms; ++a)
          tma_load_2d(smem + i * stage_bytes + kGAtoms * kGAtomA + a * b_bytes, xmap, &bar_full[i],
                      (c_begin + i) * kGKStage + a * kGK, p.t_base);
      uint32_t stage = (uint32_t)(pre % stages), phase = pre == stages ? 1u : 0u;
      for (int c = c_begin + pre; c < c_end; ++c) {
        if (!mbar_wait(&bar_empty[stage], phase ^ 1u, &abort_flag, p.status)) break;
        mbar_arrive_expect_tx(&bar_full[stage], (uint32_t)stage_bytes);
        uint8_t* st = smem + stage * stage_bytes;
        for (int a = 0; a < kGAtoms; ++a) {
          tma_load_2d(st + a * kGAtomA, wmap, &bar_full[stage], c * kGKStage + a * kGK, row0);
          tma_load_2d(st + kGAtoms * kGAtomA + a * b_bytes, xmap, &bar_full[stage], c * kGKStage + a * kGK, p.t_base);
        }
        issued[stage] = (int)phase;
        if (++stage == (uint32_t)stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (abort_flag) {  // let copies already in flight land before the CTA exits
        for (int s = 0; s < stages; ++s)
          if (issued[s] >= 0) mbar_wait_drain(&bar_full[s], (uint32_t)issued[s]);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------ UMMA issuer -------------------------------
      const uint32_t idesc = idesc_bf16_f32(kGM, p.tpad);
      const uint64_t desc0 = sdesc_sw128(smem_u32(smem));
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int c = c_begin; c < c_end; ++c) {
        if (!mbar_wait(&bar_full[stage], phase, &abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // descriptor start-address field counts 16-byte units; K=16 steps are
        // 32 bytes apart inside the 128-byte swizzle atom
        const uint64_t s_desc = desc0 + (uint64_t)(stage * (stage_bytes >> 4));
#pragma unroll
        for (int a = 0; a < kGAtoms; ++a) {
          const uint64_t a_desc = s_desc + (uint64_t)((a * kGAtomA) >> 4);
          const uint64_t b_desc = s_desc + (uint64_t)((kGAtoms * kGAtomA + a * b_bytes) >> 4);
#pragma unroll
          for (int k = 0; k < kGK / 16; ++k)
            umma_bf16_ss(tmem_base, a_desc + 2 * k, b_desc + 2 * k, idesc, (c > c_begin || a > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(&bar_empty[stage]);
        if (++stage == (uint32_t)stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) umma_commit(&bar_tfull);
      umma_commit(&bar_drain);
      mbar_wait_drain(&bar_drain, 0);
    }
  } else {
    // ------------------------------ epilogue -------------------------------------
    // warp w reads TMEM lanes 32 (w % 4) ..: thread = weight row of the tile
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    if (mbar_wait(&bar_tfull, 0, &abort_flag, p.status)) {
      tc_fence_after();
      float* out = p.part + (((int64_t)layer * p.splits + split) * p.t_rows + p.t_base) * p.ld_part +
                   (int64_t)(p.mat_col_tile[m] + tile_in) * kGM + row;
      for (int t0 = 0; t0 < p.tpad; t0 += 16) {
        uint32_t r[16];
        tmem_ld16(tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)t0, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (t0 + j < p.T) out[(int64_t)(t0 + j) * p.ld_part] = __uint_as_float(r[j]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

// K splits of a projection with `tiles` weight tiles: enough that
// tiles x splits fills the SMs once, at most one per K chunk.
int gemm_splits(int tiles, int kc, int num_sms) {
  int s = num_sms / tiles;
  const int cap = kGSizingSms / tiles < kGMaxSplits ? kGSizingSms / tiles : kGMaxSplits;
  if (s > cap) s = cap;
  if (s > kc) s = kc;
  return s < 1 ? 1 : s;
}
// Upper bound of gemm_splits over devices and K (sizes the workspace).
int gemm_splits_max(int tiles) {
  const int cap = kGSizingSms / tiles < kGMaxSplits ? kGSizingSms / tiles : kGMaxSplits;
  return cap < 1 ? 1 : cap;
}

// One projection launch set: up to kGMaxMats weight matrices [rows, K] (matrix
// m of layer mats[m].layer, its tiles at column tile mats[m].col_tile of that
// layer's part rows) against each layer's activations X[layer] [T, K].
struct ProjMat {
  const uint16_t* w;
  int rows;
  int layer;
  int col_tile;
};

// part[layer][s][t][col]; ld_part = the column tiles of one layer * 128.
// Launches one grid per 256 tokens.
fm_status proj_gemm(const uint16_t* const* X, int n_layers, int T, int K, const ProjMat* mats, int n_mats,
                    int64_t ld_part, int num_sms, float* part, int* splits_out, unsigned int* status, bool pdl,
                    bool prefetch, cudaStream_t stream) {
  GemmParams gp = {};
  GemmMaps maps;
  int tiles = 0;
  for (int m = 0; m < n_mats; ++m) {
    gp.mat_tile0[m] = tiles;
    gp.mat_layer[m] = mats[m].layer;
    gp.mat_col_tile[m] = mats[m].col_tile;
    tiles += (mats[m].rows + kGM - 1) / kGM;
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)mats[m].rows};
    const uint64_t strides[1] = {(uint64_t)K * 2};
    const uint32_t box[2] = {(uint32_t)kGK, (uint32_t)kGM};
    fm_status st = make_tmap(&maps.w[m], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, mats[m].w, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != FM_OK) return st;
  }
  gp.mat_tile0[n_mats] = tiles;
  for (int m = n_mats; m < kGMaxMats; ++m) maps.w[m] = maps.w[0];
  const int kc = (K + kGKStage - 1) / kGKStage;
  const int splits = gemm_splits(tiles, kc, num_sms);
  *splits_out = splits;
  for (int t_base = 0; t_base < T; t_base += kGMaxTokens) {
    const int Tb = T - t_base < kGMaxTokens ? T - t_base : kGMaxTokens;
    const int tpad = (Tb + 15) / 16 * 16;
    for (int l = 0; l < kGMaxLayers; ++l) {
      // rows past T read as zeros (the copy's out-of-bounds fill)
      const uint64_t dims[2] = {(uint64_t)K, (uint64_t)T};
      const uint64_t strides[1] = {(uint64_t)K * 2};
      const uint32_t box[2] = {(uint32_t)kGK, (uint32_t)tpad};
      fm_status st = make_tmap(&maps.x[l], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, X[l < n_layers ? l : 0], dims,
                               strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
      if (st != FM_OK) return st;
    }
    gp.part = part;
    gp.status = status;
    gp.ld_part = ld_part;
    gp.t_rows = T;
    gp.t_base = t_base;
    gp.T = Tb;
    gp.tpad = tpad;
    gp.kc = kc;
    gp.n_mats = n_mats;
    gp.splits = splits;
    const int stage_bytes = kGAtoms * (kGAtomA + tpad * 128);
    int stages = (200 * 1024) / stage_bytes;
    if (stages > kGMaxStages) stages = kGMaxStages;
    gp.stages = stages;
    uint32_t cols = 32;
    while (cols < (uint32_t)tpad) cols <<= 1;
    gp.tmem_cols = cols;
    gp.prefetch_weights = prefetch ? 1 : 0;
    const int smem = 1024 + stages * stage_bytes;
    cudaError_t e = cudaFuncSetAttribute(proj_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "query chain: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    const unsigned grid = (unsigned)(tiles * splits);
    if (pdl) {
      e = launch_pdl(proj_gemm_kernel, dim3(grid), kGThreads, (size_t)smem, stream, maps, gp);
    } else {
      proj_gemm_kernel<<<grid, kGThreads, smem, stream>>>(maps, gp);
      e = cudaGetLastError();
    }
    if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "query chain: GEMM launch: %s", cudaGetErrorString(e));
  }
  return FM_OK;
}

// One CTA per (token t, layer l): a = sum of the splits of part[l, ., t, 0..r),
// RMSNorm with layer l's gain, rounded to bf16 into c[l, t]; w[t, l, h] =
// w_scale * sum of the splits of part[l, ., t, w_col0 + h].
// The splits are summed in order 0, 1, ...  A thread takes its elements two at
// a time with the partial loads of up to eight splits issued together, so the
// row's reduction costs a few memory round trips, not one per split.
constexpr int kNormThreads = 1024;
constexpr int kNormUnroll = 2;
constexpr int kNormSplitBatch = 8;
__global__ void __launch_bounds__(kNormThreads)
    rmsnorm_kernel(const float* __restrict__ part, int splits, int64_t ld, int64_t T, int r, LayerPtrs gains,
                   float eps, uint16_t* __restrict__ c_out, int n_h, int64_t w_col0, float w_scale,
                   float* __restrict__ w_out, const int64_t* __restrict__ pos, RopeFreqs rf,
                   float2* __restrict__ trig) {
  __shared__ float warp_ss[kNormThreads / 32];
  grid_dep_launch_dependents();
  grid_dep_wait();  // part is the previous kernel's output
  const int64_t t = blockIdx.x;
  const int layer = blockIdx.y, n_layers = gridDim.y;
  const int tid = threadIdx.x;
  if (layer == 0 && tid < kRopeDim / 2) {
    // the token's rotary (cos, sin) for the rotary kernel, once per token:
    // the angle pos * theta'_i is formed and reduced modulo 2 pi in fp64 (it
    // reaches 2^31 radians); sine and cosine of the reduced angle in fp32
    const double two_pi = 6.283185307179586476925286766559;
    const double inv_two_pi = 0.15915494309189533576888376337251;
    double a = (double)pos[t] * rf.f[tid];
    a -= two_pi * floor(a * inv_two_pi);
    float sn, cs;
    sincosf((float)a, &sn, &cs);
    trig[t * (kRopeDim / 2) + tid] = make_float2(cs, sn);
  }
  const int64_t split_stride = T * ld;
  const float* row = part + (int64_t)layer * splits * split_stride + t * ld;
  const uint16_t* g = gains.p[layer];
  uint16_t* out = c_out + (int64_t)layer * T * r;
  // a[j] = the sum over splits of column c0 + j * kNormThreads (0 where that is >= n)
  auto sums = [&](int64_t c0, int64_t n, float (&a)[kNormUnroll]) {
#pragma unroll
    for (int j = 0; j < kNormUnroll; ++j) a[j] = 0.f;
    for (int s0 = 0; s0 < splits; s0 += kNormSplitBatch) {
      float x[kNormSplitBatch][kNormUnroll];
#pragma unroll
      for (int u = 0; u < kNormSplitBatch; ++u)
#pragma unroll
        for (int j = 0; j < kNormUnroll; ++j) {
          const int64_t c = c0 + j * kNormThreads;
          x[u][j] = (s0 + u < splits && c < n) ? __ldg(row + (s0 + u) * split_stride + c) : 0.f;
        }
#pragma unroll
      for (int u = 0; u < kNormSplitBatch; ++u)
#pragma unroll
        for (int j = 0; j < kNormUnroll; ++j) a[j] += x[u][j];
    }
  };
  float ss = 0.f;
  for (int i0 = tid; i0 < r; i0 += kNormThreads * kNormUnroll) {
    float a[kNormUnroll];
    sums(i0, r, a);
#pragma unroll
    for (int j = 0; j < kNormUnroll; ++j) ss = fmaf(a[j], a[j], ss);
  }
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((tid & 31) == 0) warp_ss[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < kNormThreads / 32; ++i) tot += warp_ss[i];
  const float inv = rsqrtf(tot / (float)r + eps);
  for (int i0 = tid; i0 < r; i0 += kNormThreads * kNormUnroll) {
    float a[kNormUnroll];
    sums(i0, r, a);
#pragma unroll
    for (int j = 0; j < kNormUnroll; ++j) {
      const int i = i0 + j * kNormThreads;
      if (i < r) out[t * r + i] = f32_to_bf16_rne(a[j] * inv * __uint_as_float((uint32_t)g[i] << 16));
    }
  }
  for (int h0 = tid; h0 < n_h; h0 += kNormThreads * kNormUnroll) {
    float a[kNormUnroll];
    sums(w_col0 + h0, w_col0 + n_h, a);
#pragma unroll
    for (int j = 0; j < kNormUnroll; ++j) {
      const int h = h0 + j * kNormThreads;
      if (h < n_h) w_out[(t * n_layers + layer) * n_h + h] = w_scale * a[j];
    }
  }
}

// YaRN NTK-by-parts frequency of rotary pair i: theta_i = base^(-2i/64);
// pairs that turn fewer than beta_slow times over the original context take
// theta_i / factor, pairs that turn more than beta_fast times keep theta_i,
// and the ones between blend the two linearly in the number of turns.
RopeFreqs yarn_freqs(double base, double factor, double orig_len, double beta_fast, double beta_slow) {
  const double two_pi = 6.283185307179586476925286766559;
  RopeFreqs r;
  for (int i = 0; i < kRopeDim / 2; ++i) {
    const double theta = std::pow(base, -2.0 * (double)i / (double)kRopeDim);
    const double turns = orig_len * theta / two_pi;
    double gamma = (turns - beta_slow) / (beta_fast - beta_slow);
    gamma = gamma < 0.0 ? 0.0 : (gamma > 1.0 ? 1.0 : gamma);
    r.f[i] = (1.0 - gamma) * theta / factor + gamma * theta;
  }
  return r;
}

// u = the splits of part summed in order; part is [layers][splits][T * n_h * 128]
// (rows of one layer's split block: (token, head)).  q_out is [T, layers, n_h, 128].
__global__ void __launch_bounds__(256)
    rope_hadamard_kernel(const float* __restrict__ part, int splits, const float2* __restrict__ trig, int64_t T,
                         int n_layers, int n_h, uint16_t* __restrict__ q_out, float* __restrict__ q_out_f32) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = T * n_h;                                         // per layer
  const int64_t grow = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);    // (layer, token, head)
  grid_dep_launch_dependents();
  grid_dep_wait();  // part is the previous kernel's output
  if (grow >= rows * n_layers) return;
  const int64_t layer = grow / rows, prow = grow % rows;
  const int64_t t = prow / n_h, hh = prow % n_h;
  const int64_t row = (t * n_layers + layer) * n_h + hh;               // output row
  const float* lp = part + layer * splits * rows * kHeadDim;
  float4 in = *reinterpret_cast<const float4*>(lp + prow * kHeadDim + 4 * lane);
  for (int s = 1; s < splits; ++s) {
    const float4 x = *reinterpret_cast<const float4*>(lp + (s * rows + prow) * kHeadDim + 4 * lane);
    in.x += x.x;
    in.y += x.y;
    in.z += x.z;
    in.w += x.w;
  }
  float v[4] = {in.x, in.y, in.z, in.w};
  // rotary on entries 64..127 (lanes 16..31): pairs (2i, 2i+1), i = 2 lane - 32 + {0, 1},
  // with the token's (cos, sin) from the RMSNorm kernel; the rotation in fp32
  if (lane >= 16) {
    const float4 cs = *reinterpret_cast<const float4*>(trig + t * (kRopeDim / 2) + 2 * lane - 32);
    const float c[2] = {cs.x, cs.z}, sn[2] = {cs.y, cs.w};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float x0 = v[2 * k], x1 = v[2 * k + 1];
      v[2 * k] = x0 * c[k] - x1 * sn[k];
      v[2 * k + 1] = x0 * sn[k] + x1 * c[k];
    }
  }
  // Walsh-Hadamard butterflies: strides 1, 2 inside the lane, 4..64 across lanes
  {
    const float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
    v[0] = a0 + a2;
    v[1] = a1 + a3;
    v[2] = a0 - a2;
    v[3] = a1 - a3;
  }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float other = __shfl_xor_sync(0xffffffffu, v[j], m);
      v[j] = upper ? other - v[j] : v[j] + other;
    }
  }
  const float norm = 0.08838834764831845f;  // 1 / sqrt(128)
#pragma unroll
  for (int j = 0; j < 4; ++j) v[j] *= norm;
  uint2 packed;
  packed.x = (uint32_t)f32_to_bf16_rne(v[0]) | ((uint32_t)f32_to_bf16_rne(v[1]) << 16);
  packed.y = (uint32_t)f32_to_bf16_rne(v[2]) | ((uint32_t)f32_to_bf16_rne(v[3]) << 16);
  *reinterpret_cast<uint2*>(q_out + row * kHeadDim + 4 * lane) = packed;
  if (q_out_f32 != nullptr)
    *reinterpret_cast<float4*>(q_out_f32 + row * kHeadDim + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace: per layer, the K-split partials of [a | w] (tiles of wq_a then
// w_proj), the bf16 RMSNorm output, the K-split partials of u.
struct ChainWs {
  size_t part1, c, part2, trig, bytes;
};
ChainWs chain_ws(int L, int T, int r, int n_h) {
  const int nt1 = (r + kGM - 1) / kGM + (n_h + kGM - 1) / kGM;  // per layer
  const int nt2 = n_h;                                           // n_h * 128 rows per layer
  ChainWs w;
  w.part1 = 0;
  w.c = align256((size_t)L * gemm_splits_max(L * nt1) * T * nt1 * kGM * 4);
  w.part2 = w.c + align256((size_t)L * T * r * 2);
  w.trig = w.part2 + align256((size_t)L * gemm_splits_max(L * nt2) * T * nt2 * kGM * 4);
  w.bytes = w.trig + align256((size_t)T * (kRopeDim / 2) * 8);  // per token, (cos, sin) of the 32 rotary pairs
  return w;
}

fm_status run_chain(int L, const uint16_t* const* hidden, const uint16_t* const* wq_a, const uint16_t* const* q_norm,
                    const uint16_t* const* wq_b, const uint16_t* const* w_proj, const int64_t* pos, int T, int dim,
                    int r, int n_h, int head_dim, int rope_dim, double rope_base, double rope_factor,
                    double rope_orig_len, double rope_beta_fast, double rope_beta_slow, float eps, uint16_t* q_out,
                    float* q_out_f32, float* w_out, void* workspace, size_t workspace_bytes, cudaStream_t s,
                    const char* who) {
  if (L < 1 || L > kGMaxLayers)
    return set_error(FM_ERR_INVALID_ARG, "%s: L=%d (1..%d layers)", who, L, kGMaxLayers);
  if (head_dim != kHeadDim || rope_dim != kRopeDim)
    return set_error(FM_ERR_INVALID_ARG, "%s: head_dim=%d rope_dim=%d (need 128, 64)", who, head_dim, rope_dim);
  if (T < 0 || dim < 8 || r < 8 || n_h < 1 || dim % 8 != 0 || r % 8 != 0 || n_h > 1024)
    return set_error(FM_ERR_INVALID_ARG, "%s: bad sizes T=%d dim=%d r=%d n_h=%d (dim, r: multiples of 8)", who, T,
                     dim, r, n_h);
  if (!(rope_base > 1.0) || !(rope_factor >= 1.0) || !(rope_orig_len > 0.0) || !(rope_beta_fast > rope_beta_slow) ||
      !(eps >= 0.0f))
    return set_error(FM_ERR_INVALID_ARG, "%s: bad rotary or norm parameters", who);
  if (T == 0) return FM_OK;
  if (!hidden || !wq_a || !q_norm || !wq_b || !w_proj || !pos || !q_out || !w_out)
    return set_error(FM_ERR_INVALID_ARG, "%s: required pointer is NULL", who);
  for (int l = 0; l < L; ++l) {
    if (!hidden[l] || !wq_a[l] || !q_norm[l] || !wq_b[l] || !w_proj[l])
      return set_error(FM_ERR_INVALID_ARG, "%s: layer %d: required pointer is NULL", who, l);
    if (!aligned(hidden[l], 16) || !aligned(wq_a[l], 16) || !aligned(wq_b[l], 16) || !aligned(w_proj[l], 16) ||
        !aligned(q_norm[l], 2))
      return set_error(FM_ERR_INVALID_ARG, "%s: layer %d: misaligned pointer", who, l);
  }
  if (!aligned(pos, 8) || !aligned(q_out, 8) || !aligned(w_out, 4) || (q_out_f32 && !aligned(q_out_f32, 16)))
    return set_error(FM_ERR_INVALID_ARG, "%s: misaligned pointer", who);
  const ChainWs lay = chain_ws(L, T, r, n_h);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < lay.bytes)
    return set_error(FM_ERR_WORKSPACE, "%s: workspace needs %zu bytes, 256-byte aligned", who, lay.bytes);
  int sms = 0;
  fm_status st = check_device(&sms);
  if (st != FM_OK) return st;
  unsigned int* status = nullptr;
  if ((st = status_word(&status)) != FM_OK) return st;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  float* part1 = reinterpret_cast<float*>(base + lay.part1);
  uint16_t* c = reinterpret_cast<uint16_t*>(base + lay.c);
  float* part2 = reinterpret_cast<float*>(base + lay.part2);
  float2* trig = reinterpret_cast<float2*>(base + lay.trig);
  // [a | w] = h . [wq_a | w_proj]^T, every layer in one launch
  const int nt_a = (r + kGM - 1) / kGM;
  const int64_t ld1 = (int64_t)(nt_a + (n_h + kGM - 1) / kGM) * kGM;
  ProjMat mats[kGMaxMats];
  for (int l = 0; l < L; ++l) {
    mats[2 * l] = ProjMat{wq_a[l], r, l, 0};
    mats[2 * l + 1] = ProjMat{w_proj[l], n_h, l, nt_a};
  }
  int splits1 = 1, splits2 = 1;
  if ((st = proj_gemm(hidden, L, T, dim, mats, 2 * L, ld1, sms, part1, &splits1, status, true, false, s)) != FM_OK)
    return st;
  // RMSNorm of a, and the head weights w_proj . h scaled by head_dim^-1/2 n_h^-1/2
  LayerPtrs gains = {};
  for (int l = 0; l < L; ++l) gains.p[l] = q_norm[l];
  const float w_scale = (float)(1.0 / sqrt((double)head_dim) / sqrt((double)n_h));
  const RopeFreqs rf = yarn_freqs(rope_base, rope_factor, rope_orig_len, rope_beta_fast, rope_beta_slow);
  cudaError_t e = launch_pdl(rmsnorm_kernel, dim3((unsigned)T, (unsigned)L), kNormThreads, 0, s, (const float*)part1,
                             splits1, ld1, (int64_t)T, r, gains, eps, c, n_h, (int64_t)nt_a * kGM, w_scale, w_out,
                             pos, rf, trig);
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "%s: rmsnorm launch: %s", who, cudaGetErrorString(e));
  // u = c . wq_b^T, every layer in one launch (layer l's rows of c start at l * T)
  const uint16_t* c_l[kGMaxLayers];
  for (int l = 0; l < L; ++l) {
    c_l[l] = c + (int64_t)l * T * r;
    mats[l] = ProjMat{wq_b[l], n_h * kHeadDim, l, 0};
  }
  if ((st = proj_gemm(c_l, L, T, r, mats, L, (int64_t)n_h * kHeadDim, sms, part2, &splits2, status, true, true, s)) !=
      FM_OK)
    return st;
  const int64_t rows = (int64_t)L * T * n_h;
  e = launch_pdl(rope_hadamard_kernel, dim3((unsigned)((rows + 7) / 8)), 256, 0, s, (const float*)part2, splits2,
                 (const float2*)trig, (int64_t)T, L, n_h, q_out, q_out_f32);
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "%s: rope launch: %s", who, cudaGetErrorString(e));
  return FM_OK;
}

}  // namespace
}  // namespace fm

FM_API size_t fm_query_chain_workspace(int T, int r, int n_h) {
  if (T < 0 || r < 1 || n_h < 1) return 0;
  return fm::chain_ws(1, T, r, n_h).bytes;
}

FM_API size_t fm_query_chain_layers_workspace(int L, int T, int r, int n_h) {
  if (L < 1 || L > fm::kGMaxLayers || T < 0 || r < 1 || n_h < 1) return 0;
  return fm::chain_ws(L, T, r, n_h).bytes;
}

FM_API fm_status fm_query_chain(const uint16_t* hidden, const uint16_t* wq_a, const uint16_t* q_norm,
                                const uint16_t* wq_b, const uint16_t* w_proj, const int64_t* pos, int T, int dim,
                                int r, int n_h, int head_dim, int rope_dim, double rope_base, double rope_factor,
                                double rope_orig_len, double rope_beta_fast, double rope_beta_slow, float eps,
                                uint16_t* q_out, float* q_out_f32, float* w_out, void* workspace,
                                size_t workspace_bytes, fm_stream_t stream) {
  return fm::run_chain(1, &hidden, &wq_a, &q_norm, &wq_b, &w_proj, pos, T, dim, r, n_h, head_dim, rope_dim, rope_base,
                       rope_factor, rope_orig_len, rope_beta_fast, rope_beta_slow, eps, q_out, q_out_f32, w_out,
                       workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream), "fm_query_chain");
}

FM_API fm_status fm_query_chain_layers(int L, const uint16_t* const* hidden, const uint16_t* const* wq_a,
                                       const uint16_t* const* q_norm, const uint16_t* const* wq_b,
                                       const uint16_t* const* w_proj, const int64_t* pos, int T, int dim, int r,
                                       int n_h, int head_dim, int rope_dim, double rope_base, double rope_factor,
                                       double rope_orig_len, double rope_beta_fast, double rope_beta_slow, float eps,
                                       uint16_t* q_out, float* q_out_f32, float* w_out, void* workspace,
                                       size_t workspace_bytes, fm_stream_t stream) {
  return fm::run_chain(L, hidden, wq_a, q_norm, wq_b, w_proj, pos, T, dim, r, n_h, head_dim, rope_dim, rope_base,
                       rope_factor, rope_orig_len, rope_beta_fast, rope_beta_slow, eps, q_out, q_out_f32, w_out,
                       workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream), "fm_query_chain_layers");
}

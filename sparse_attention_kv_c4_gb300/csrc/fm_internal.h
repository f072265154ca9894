// fm_internal.h -- host-side declarations shared by the library's translation
// units (argument checking helpers, tensor-map encoding, kernel launchers).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/fm_index.h"

namespace fm {

// Record a message for fm_last_error() and return `st`.
fm_status set_error(fm_status st, const char* fmt, ...);

// Current device must be sm_103; fills the SM count.
fm_status check_device(int* num_sms);

// Device address of the status word on the current device.
fm_status status_word(unsigned int** ptr);

// cuTensorMapEncodeTiled through the runtime's driver entry point.
fm_status make_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                    const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                    CUtensorMapSwizzle swizzle);

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---- launchers (arguments already validated) -------------------------------
struct MemindexArgs {
  const uint16_t* q;
  const float* w;
  const uint16_t* keys;
  int64_t key_stride_b, key_stride_l;
  int B, L;
  int64_t S;
  float thr_logit;
  uint32_t* mask;
  float* maxsig;
  float* logits;
};
fm_status launch_memindex(const MemindexArgs& a, int num_sms, unsigned int* status, cudaStream_t stream);

// Exact top-k of each row, one CTA per row.  Candidate i of row r has id i;
// with page_ids, page_ids[r*page_ld + i/64]*64 + i%64; with page_ids,
// page_prefix [rows, page_ld+1] and page_mask [rows, page_ld] (a row compacted
// to its resident chunks), page_ids[r*page_ld + j]*64 + o for the page j whose
// prefix range holds i and the (i - prefix[j])-th set bit o of its mask.
size_t topk_workspace_bytes(int rows, int n);
fm_status launch_topk_rows(const float* scores, int64_t ld, const int32_t* n_valid, int rows, int n, int k,
                           const int32_t* page_ids, int64_t page_ld, const int32_t* page_prefix,
                           const unsigned long long* page_mask, int32_t* idx_out, float* score_out,
                           cudaStream_t stream);
// The same select (candidate i has id i) for rows that come with segment
// maxima: segmax[r*seg_ld + g] is, for the scores 32g .. 32g+31 of row r below
// its n_valid, the largest of their bit patterns read as signed integers.  Rows
// with at least 2k segments read only the segments that can hold a top-k score.
fm_status launch_topk_rows_segmax(const float* scores, int64_t ld, const int32_t* n_valid, const int32_t* segmax,
                                  int64_t seg_ld, int rows, int n, int k, int32_t* idx_out, float* score_out,
                                  cudaStream_t stream);

struct PagedArgs {
  const uint16_t* q;
  const float* w;
  const void* k_pool;        // E4M3 codes [P, 64, 128] or bf16 keys [P, 64, 128]
  int key_dtype;             // FM_DTYPE_FP8_E4M3 or FM_DTYPE_BF16
  const float* k_scale;
  int64_t P;
  const int32_t* page_phys;
  const int32_t* page_logical;
  const int32_t* n_res;
  int Q, R, k;
  const uint32_t* res_mask;  // [ceil(Q/mask_group), mask_ld] resident chunks, or null (every listed chunk)
  int64_t mask_ld;
  int mask_group;
  int id_mode;               // 0: logical chunk ids, 1: reserve cells phys*64 + o
  int32_t* idx_out;
  float* score_out;
  void* workspace;
};
size_t paged_workspace_bytes(int Q, int R);

struct PrefillArgs {
  const uint16_t* q;
  const float* w;
  const int64_t* pos;
  const uint16_t* keys;
  int T;
  int64_t S;
  int ratio, k;
  int32_t* idx_out;
  float* score_out;
  void* workspace;
};
size_t prefill_workspace_bytes(int T, int64_t S);
fm_status launch_prefill(const PrefillArgs& a, int num_sms, unsigned int* status, cudaStream_t stream);
// The dense scores Y [T, S] into `logits` (row stride S) for s below each
// token's causal limit; with fill_masked, -inf at every other s.  With segmax
// ([T, ceil(S / 32)]), also each token's segment maxima (launch_topk_rows_segmax).
fm_status launch_prefill_scores(const PrefillArgs& a, float* logits, int32_t* segmax, bool fill_masked, int num_sms,
                                unsigned int* status, cudaStream_t stream);
fm_status launch_paged(const PagedArgs& a, int num_sms, unsigned int* status, cudaStream_t stream);

}  // namespace fm

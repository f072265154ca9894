// fm_api.cu -- the C ABI of libfm_index.so: argument validation, device
// checks, tensor-map encoding, error reporting, dispatch to the launchers.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <cudaTypedefs.h>

#include "fm_common.cuh"
#include "fm_internal.h"

#define FM_API extern "C" __attribute__((visibility("default")))

// Device status word: OR of FM_DEVERR_* bits raised by kernels.
__device__ unsigned int g_fm_device_status;

namespace fm {

static thread_local char t_last_error[512] = "no error";

fm_status set_error(fm_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
  va_end(ap);
  return st;
}

fm_status check_device(int* num_sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  int major = 0, minor = 0, sms = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
  if (major != 10 || minor != 3)
    return set_error(FM_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a", dev, major,
                     minor);
  if (num_sms) *num_sms = sms;
  return FM_OK;
}

fm_status status_word(unsigned int** ptr) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_fm_device_status);
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "cudaGetSymbolAddress(status): %s", cudaGetErrorString(e));
  *ptr = static_cast<unsigned int*>(p);
  return FM_OK;
}

fm_status make_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
      return set_error(FM_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  uint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = encode(map, dtype, (cuuint32_t)rank, const_cast<void*>(base), (const cuuint64_t*)dims,
                      (const cuuint64_t*)strides_bytes, (const cuuint32_t*)box, (const cuuint32_t*)estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(FM_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  return FM_OK;
}

}  // namespace fm

using namespace fm;

FM_API int fm_version(void) { return 1 * 10000 + 1 * 100 + 0; }

FM_API const char* fm_last_error(void) { return t_last_error; }

FM_API fm_status fm_device_status(uint32_t* status_out, int reset, fm_stream_t stream) {
  if (status_out == nullptr) return set_error(FM_ERR_INVALID_ARG, "fm_device_status: status_out is NULL");
  unsigned int* dptr = nullptr;
  fm_status st = status_word(&dptr);
  if (st != FM_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, dptr, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && reset) e = cudaMemsetAsync(dptr, 0, sizeof(unsigned int), s);
  if (e == cudaSuccess && reset) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return set_error(FM_ERR_CUDA, "fm_device_status: %s", cudaGetErrorString(e));
  *status_out = v;
  return FM_OK;
}

FM_API fm_status fm_check_device_status(fm_stream_t stream) {
  uint32_t v = 0;
  const fm_status st = fm_device_status(&v, 1, stream);
  if (st != FM_OK) return st;
  if (v == 0) return FM_OK;
  const bool timeout = (v & FM_DEVERR_TIMEOUT) != 0;
  set_error(timeout ? FM_ERR_DEVICE_TIMEOUT : FM_ERR_DEVICE_BOUNDS,
            "device status 0x%x:%s%s%s", v, (v & FM_DEVERR_TIMEOUT) ? " a bounded wait ran out;" : "",
            (v & FM_DEVERR_PAGE_RANGE) ? " a page id was out of range;" : "",
            (v & FM_DEVERR_DUP_PAGE) ? " a logical page was repeated in a page table;" : "");
  return timeout ? FM_ERR_DEVICE_TIMEOUT : FM_ERR_DEVICE_BOUNDS;
}

FM_API fm_status fm_memindex_score_mask(const uint16_t* q, const float* w, const uint16_t* keys,
                                        int64_t key_stride_b, int64_t key_stride_l, int B, int L, int64_t S,
                                        int n_h, int d, float threshold, uint32_t* mask_out, float* maxsig_out,
                                        float* logits_out, fm_stream_t stream) {
  if (n_h != 64 || d != 128)
    return set_error(FM_ERR_INVALID_ARG, "fm_memindex_score_mask: n_h=%d d=%d (need 64, 128)", n_h, d);
  if (B < 0 || L < 1 || L > 4 || S < 0 || S >= (int64_t(1) << 31))
    return set_error(FM_ERR_INVALID_ARG, "fm_memindex_score_mask: bad sizes B=%d L=%d S=%lld", B, L, (long long)S);
  if (!(threshold > 0.0f && threshold < 1.0f))
    return set_error(FM_ERR_INVALID_ARG, "fm_memindex_score_mask: threshold %g not in (0, 1)", (double)threshold);
  if (B == 0 || S == 0) return FM_OK;
  if (!q || !w || !keys || !mask_out)
    return set_error(FM_ERR_INVALID_ARG, "fm_memindex_score_mask: q, w, keys and mask_out must be non-NULL");
  if (!aligned(q, 16) || !aligned(keys, 16) || !aligned(w, 16) || !aligned(mask_out, 4) ||
      (maxsig_out && !aligned(maxsig_out, 4)) || (logits_out && !aligned(logits_out, 4)))
    return set_error(FM_ERR_INVALID_ARG, "fm_memindex_score_mask: q/keys/w need 16-byte alignment");
  if (key_stride_l < S * d || key_stride_b < (int64_t)(L - 1) * key_stride_l + S * d || key_stride_l % 8 != 0 ||
      key_stride_b % 8 != 0)
    return set_error(FM_ERR_INVALID_ARG,
                     "fm_memindex_score_mask: key strides (b=%lld, l=%lld) must be multiples of 8 elements and "
                     "lay the [L, S, d] blocks out without overlap",
                     (long long)key_stride_b, (long long)key_stride_l);
  int sms = 0;
  fm_status st = check_device(&sms);
  if (st != FM_OK) return st;
  unsigned int* status = nullptr;
  st = status_word(&status);
  if (st != FM_OK) return st;

  MemindexArgs a;
  a.q = q;
  a.w = w;
  a.keys = keys;
  a.key_stride_b = key_stride_b;
  a.key_stride_l = key_stride_l;
  a.B = B;
  a.L = L;
  a.S = S;
  a.thr_logit = (float)log((double)threshold / (1.0 - (double)threshold));
  a.mask = mask_out;
  a.maxsig = maxsig_out;
  a.logits = logits_out;
  return launch_memindex(a, sms, status, reinterpret_cast<cudaStream_t>(stream));
}

FM_API size_t fm_topk_workspace(int rows, int64_t n) {
  if (rows <= 0 || n <= 0 || n >= (int64_t(1) << 31)) return 0;
  return topk_workspace_bytes(rows, (int)n);
}

FM_API fm_status fm_topk_select(const float* scores, int64_t ld, const int32_t* n_valid, int rows, int64_t n, int k,
                                int32_t* idx_out, float* score_out, void* workspace, size_t workspace_bytes,
                                fm_stream_t stream) {
  if (rows < 0 || n < 0 || n >= (int64_t(1) << 31) || k < 1 || k > 1024)
    return set_error(FM_ERR_INVALID_ARG, "fm_topk_select: bad sizes rows=%d n=%lld k=%d (1 <= k <= 1024)", rows,
                     (long long)n, k);
  if (rows == 0) return FM_OK;
  if (ld < n) return set_error(FM_ERR_INVALID_ARG, "fm_topk_select: ld=%lld < n=%lld", (long long)ld, (long long)n);
  if (!idx_out || (n > 0 && !scores))
    return set_error(FM_ERR_INVALID_ARG, "fm_topk_select: scores and idx_out must be non-NULL");
  if (!aligned(scores, 4) || !aligned(idx_out, 4) || (score_out && !aligned(score_out, 4)) ||
      (n_valid && !aligned(n_valid, 4)))
    return set_error(FM_ERR_INVALID_ARG, "fm_topk_select: pointers need 4-byte alignment");
  if (workspace != nullptr && !aligned(workspace, 256))
    return set_error(FM_ERR_WORKSPACE, "fm_topk_select: workspace must be 256-byte aligned");
  int sms = 0;
  fm_status st = check_device(&sms);
  if (st != FM_OK) return st;
  (void)workspace_bytes;  // the select needs no scratch (fm_topk_workspace is 0)
  return launch_topk_rows(scores, ld, n_valid, rows, (int)n, k, nullptr, 0, nullptr, nullptr, idx_out, score_out,
                          reinterpret_cast<cudaStream_t>(stream));
}

FM_API size_t fm_native_topk_paged_workspace(int Q, int R) {
  if (Q < 0 || R < 1 || R > FM_PAGED_MAX_R) return 0;
  return paged_workspace_bytes(Q, R);
}

FM_API fm_status fm_native_topk_paged_ex(const uint16_t* q, const float* w, const void* k_pool, int key_dtype,
                                         const float* k_scale, int64_t P, const int32_t* page_phys,
                                         const int32_t* page_logical, const int32_t* n_res, int Q, int R, int n_h,
                                         int d, int k, const uint32_t* res_mask, int64_t mask_ld, int mask_group,
                                         int id_mode, int32_t* idx_out, float* score_out, void* workspace,
                                         size_t workspace_bytes, fm_stream_t stream) {
  if (n_h != 64 || d != 128)
    return set_error(FM_ERR_INVALID_ARG, "fm_native_topk_paged: n_h=%d d=%d (need 64, 128)", n_h, d);
  if (Q < 0 || R < 1 || R > FM_PAGED_MAX_R || k < 1 || k > 1024 || P < 0 || P > (int64_t(1) << 26))
    return set_error(FM_ERR_INVALID_ARG, "fm_native_topk_paged: bad sizes Q=%d R=%d k=%d P=%lld", Q, R, k,
                     (long long)P);
  if (id_mode != 0 && id_mode != 1)
    return set_error(FM_ERR_INVALID_ARG, "fm_native_topk_paged: id_mode=%d (0 = chunk ids, 1 = reserve cells)",
                     id_mode);
  if (key_dtype != FM_DTYPE_FP8_E4M3 && key_dtype != FM_DTYPE_BF16)
    return set_error(FM_ERR_INVALID_ARG, "fm_native_topk_paged: key_dtype=%d (FM_DTYPE_FP8_E4M3 or FM_DTYPE_BF16)",
                     key_dtype);
  if (key_dtype == FM_DTYPE_BF16 && k_scale != nullptr)
    return set_error(FM_ERR_INVALID_ARG, "fm_native_topk_paged: a bf16 key pool takes no k_scale (pass NULL)");
  if (res_mask != nullptr && (mask_ld < 1 || mask_group < 1 || !aligned(res_mask, 4)))
    return set_error(FM_ERR_INVALID_ARG,
                     "fm_native_topk_paged: resident mask needs mask_ld >= 1, mask_group >= 1, 4-byte alignment");
  if (Q == 0) return FM_OK;
  if (!q || !w || !page_phys || !page_logical || !idx_out ||
      (P > 0 && (!k_pool || (key_dtype == FM_DTYPE_FP8_E4M3 && !k_scale))))
    return set_error(FM_ERR_INVALID_ARG, "fm_native_topk_paged: required pointer is NULL");
  if (!aligned(q, 16) || !aligned(w, 16) || (k_pool && !aligned(k_pool, 16)) || (k_scale && !aligned(k_scale, 16)) ||
      !aligned(page_phys, 4) || !aligned(page_logical, 4) || (n_res && !aligned(n_res, 4)) ||
      !aligned(idx_out, 4) || (score_out && !aligned(score_out, 4)))
    return set_error(FM_ERR_INVALID_ARG, "fm_native_topk_paged: q/w/k_pool/k_scale need 16-byte alignment");
  const size_t need = paged_workspace_bytes(Q, R);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need)
    return set_error(FM_ERR_WORKSPACE, "fm_native_topk_paged: workspace needs %zu bytes, 256-byte aligned", need);
  int sms = 0;
  fm_status st = check_device(&sms);
  if (st != FM_OK) return st;
  unsigned int* status = nullptr;
  st = status_word(&status);
  if (st != FM_OK) return st;
  PagedArgs a;
  a.q = q;
  a.w = w;
  a.k_pool = k_pool;
  a.key_dtype = key_dtype;
  a.k_scale = k_scale;
  a.P = P;
  a.page_phys = page_phys;
  a.page_logical = page_logical;
  a.n_res = n_res;
  a.Q = Q;
  a.R = R;
  a.k = k;
  a.res_mask = res_mask;
  a.mask_ld = mask_ld;
  a.mask_group = mask_group;
  a.id_mode = id_mode;
  a.idx_out = idx_out;
  a.score_out = score_out;
  a.workspace = workspace;
  return launch_paged(a, sms, status, reinterpret_cast<cudaStream_t>(stream));
}

FM_API fm_status fm_native_topk_paged(const uint16_t* q, const float* w, const void* k_pool, int key_dtype,
                                      const float* k_scale, int64_t P, const int32_t* page_phys,
                                      const int32_t* page_logical, const int32_t* n_res, int Q, int R, int n_h, int d,
                                      int k, int32_t* idx_out, float* score_out, void* workspace,
                                      size_t workspace_bytes, fm_stream_t stream) {
  return fm_native_topk_paged_ex(q, w, k_pool, key_dtype, k_scale, P, page_phys, page_logical, n_res, Q, R, n_h, d, k,
                                 nullptr, 0, 1, 0, idx_out, score_out, workspace, workspace_bytes, stream);
}

FM_API size_t fm_index_prefill_workspace(int T, int64_t S) {
  if (T < 0 || S < 0) return 0;
  return prefill_workspace_bytes(T, S);
}

FM_API fm_status fm_index_prefill_topk(const uint16_t* q, const float* w, const int64_t* pos, const uint16_t* keys,
                                       int T, int64_t S, int n_h, int d, int ratio, int k, int32_t* idx_out,
                                       float* score_out, void* workspace, size_t workspace_bytes,
                                       fm_stream_t stream) {
  if (n_h != 64 || d != 128)
    return set_error(FM_ERR_INVALID_ARG, "fm_index_prefill_topk: n_h=%d d=%d (need 64, 128)", n_h, d);
  if (T < 0 || S < 0 || S >= (int64_t(1) << 31) || ratio < 1 || k < 1 || k > 1024)
    return set_error(FM_ERR_INVALID_ARG, "fm_index_prefill_topk: bad sizes T=%d S=%lld ratio=%d k=%d", T,
                     (long long)S, ratio, k);
  if (T == 0) return FM_OK;
  if (!q || !w || !pos || !idx_out || (S > 0 && !keys))
    return set_error(FM_ERR_INVALID_ARG, "fm_index_prefill_topk: required pointer is NULL");
  if (!aligned(q, 16) || !aligned(w, 16) || !aligned(pos, 8) || (keys && !aligned(keys, 16)) ||
      !aligned(idx_out, 4) || (score_out && !aligned(score_out, 4)))
    return set_error(FM_ERR_INVALID_ARG, "fm_index_prefill_topk: q/w/keys need 16-byte alignment");
  const size_t need = prefill_workspace_bytes(T, S);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need)
    return set_error(FM_ERR_WORKSPACE, "fm_index_prefill_topk: workspace needs %zu bytes, 256-byte aligned", need);
  int sms = 0;
  fm_status st = check_device(&sms);
  if (st != FM_OK) return st;
  unsigned int* status = nullptr;
  st = status_word(&status);
  if (st != FM_OK) return st;
  PrefillArgs a;
  a.q = q;
  a.w = w;
  a.pos = pos;
  a.keys = keys;
  a.T = T;
  a.S = S;
  a.ratio = ratio;
  a.k = k;
  a.idx_out = idx_out;
  a.score_out = score_out;
  a.workspace = workspace;
  return launch_prefill(a, sms, status, reinterpret_cast<cudaStream_t>(stream));
}

FM_API fm_status fm_index_prefill_scores(const uint16_t* q, const float* w, const int64_t* pos, const uint16_t* keys,
                                         int T, int64_t S, int n_h, int d, int ratio, float* logits_out,
                                         fm_stream_t stream) {
  if (n_h != 64 || d != 128)
    return set_error(FM_ERR_INVALID_ARG, "fm_index_prefill_scores: n_h=%d d=%d (need 64, 128)", n_h, d);
  if (T < 0 || S < 0 || S >= (int64_t(1) << 31) || ratio < 1)
    return set_error(FM_ERR_INVALID_ARG, "fm_index_prefill_scores: bad sizes T=%d S=%lld ratio=%d", T, (long long)S,
                     ratio);
  if (T == 0 || S == 0) return FM_OK;
  if (!q || !w || !pos || !keys || !logits_out)
    return set_error(FM_ERR_INVALID_ARG, "fm_index_prefill_scores: required pointer is NULL");
  if (!aligned(q, 16) || !aligned(w, 16) || !aligned(pos, 8) || !aligned(keys, 16) || !aligned(logits_out, 4))
    return set_error(FM_ERR_INVALID_ARG, "fm_index_prefill_scores: q/w/keys need 16-byte alignment");
  int sms = 0;
  fm_status st = check_device(&sms);
  if (st != FM_OK) return st;
  unsigned int* status = nullptr;
  st = status_word(&status);
  if (st != FM_OK) return st;
  PrefillArgs a = {};
  a.q = q;
  a.w = w;
  a.pos = pos;
  a.keys = keys;
  a.T = T;
  a.S = S;
  a.ratio = ratio;
  return launch_prefill_scores(a, logits_out, nullptr, true, sms, status, reinterpret_cast<cudaStream_t>(stream));
}

// noalloc.cu -- native paged top-k for callers that cannot allocate device
// memory.
//
// fm_native_topk_paged needs a caller-provided device workspace.  Some callers
// have no way to obtain one: a serving engine that handed nearly all of HBM to
// its KV-cache pool when it started (so a further cudaMalloc fails or
// fragments that pool), a decode loop that must not stall on the implicit
// device synchronisation cudaMalloc/cudaFree may perform, or a plugin host that
// gives its kernels no allocator at all.  For them this file provides a variant
// whose scratch is a fixed array in the library's own device image.
//
// Properties of that scratch (also stated in include/fm_index.h):
//  - it is FM_NOALLOC_SCRATCH_BYTES (16 MiB) on every GPU that loads the
//    library, held until the process exits;
//  - every call resolves its device address with the calling thread's
//    current device (cudaGetSymbolAddress); the first call on a device also
//    loads the library's device image there, so make that first call before
//    any stream capture;
//  - every call shares it and it keeps the last call's contents: nothing in
//    it has to start at zero (each launch writes every byte it later reads),
//    but calls that overlap on the GPU -- on different streams, or from
//    different host threads -- race on it and must be serialised by the
//    caller.
#include "fm_common.cuh"
#include "fm_internal.h"

#define FM_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr size_t kScratchBytes = FM_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of g_noalloc_scratch on the current device.  It is looked up
// on every call rather than cached: after a cudaDeviceReset, or when the
// primary context is destroyed and created again, the library's device image
// is loaded anew and the array may sit at another address, so a cached
// pointer could send the kernels' scratch writes to unmapped memory.
fm_status scratch_for_current_device(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || p == nullptr)
    return fm::set_error(FM_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
  *out = p;
  return FM_OK;
}

}  // namespace

FM_API fm_status fm_native_topk_paged_noalloc(const uint16_t* q, const float* w, const uint8_t* k_pool,
                                              const float* k_scale, int64_t P, const int32_t* page_phys,
                                              const int32_t* page_logical, const int32_t* n_res, int Q, int R,
                                              int n_h, int d, int k, int32_t* idx_out, float* score_out,
                                              fm_stream_t stream) {
  if (n_h != 64 || d != 128)
    return fm::set_error(FM_ERR_INVALID_ARG, "fm_native_topk_paged_noalloc: n_h=%d d=%d (need 64, 128)", n_h, d);
  if (Q < 0 || R < 1 || R > FM_PAGED_MAX_R || k < 1 || k > 1024 || P < 0 || P > (int64_t(1) << 26))
    return fm::set_error(FM_ERR_INVALID_ARG, "fm_native_topk_paged_noalloc: bad sizes Q=%d R=%d k=%d P=%lld", Q, R,
                         k, (long long)P);
  if (Q == 0) return FM_OK;
  if (!q || !w || !page_phys || !page_logical || !idx_out || (P > 0 && (!k_pool || !k_scale)))
    return fm::set_error(FM_ERR_INVALID_ARG, "fm_native_topk_paged_noalloc: required pointer is NULL");
  if (!fm::aligned(q, 16) || !fm::aligned(w, 16) || (k_pool && !fm::aligned(k_pool, 16)) ||
      (k_scale && !fm::aligned(k_scale, 16)) || !fm::aligned(page_phys, 4) || !fm::aligned(page_logical, 4) ||
      (n_res && !fm::aligned(n_res, 4)) || !fm::aligned(idx_out, 4) || (score_out && !fm::aligned(score_out, 4)))
    return fm::set_error(FM_ERR_INVALID_ARG,
                         "fm_native_topk_paged_noalloc: q/w/k_pool/k_scale need 16-byte alignment");
  const size_t need = fm::paged_workspace_bytes(Q, R);
  if (need > kScratchBytes)
    return fm::set_error(FM_ERR_INVALID_ARG,
                         "fm_native_topk_paged_noalloc: Q=%d, R=%d needs %zu bytes of scratch, more than the "
                         "built-in %zu; split the queries over several calls or use fm_native_topk_paged",
                         Q, R, need, kScratchBytes);
  int sms = 0;
  fm_status st = fm::check_device(&sms);
  if (st != FM_OK) return st;
  unsigned int* status = nullptr;
  st = fm::status_word(&status);
  if (st != FM_OK) return st;
  void* scratch = nullptr;
  st = scratch_for_current_device(&scratch);
  if (st != FM_OK) return st;
  fm::PagedArgs a;
  a.q = q;
  a.w = w;
  a.k_pool = k_pool;
  a.key_dtype = FM_DTYPE_FP8_E4M3;
  a.k_scale = k_scale;
  a.P = P;
  a.page_phys = page_phys;
  a.page_logical = page_logical;
  a.n_res = n_res;
  a.Q = Q;
  a.R = R;
  a.k = k;
  a.res_mask = nullptr;
  a.mask_ld = 0;
  a.mask_group = 1;
  a.id_mode = 0;
  a.idx_out = idx_out;
  a.score_out = score_out;
  a.workspace = scratch;
  return fm::launch_paged(a, sms, status, reinterpret_cast<cudaStream_t>(stream));
}

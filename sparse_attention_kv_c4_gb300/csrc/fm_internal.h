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

}  // namespace fm

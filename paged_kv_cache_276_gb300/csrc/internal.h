// Host-side helpers shared by the C-ABI translation units.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "pkv.h"

namespace pkv {

void set_cuda_error(cudaError_t e);
int num_sms();

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Returns PKV_OK or PKV_ERR_CUDA after a launch, recording the CUDA error text.
inline int check_launch() {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_cuda_error(e);
    return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace pkv

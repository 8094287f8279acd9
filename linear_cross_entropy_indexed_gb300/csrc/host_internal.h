// Host helpers shared by the entry-point translation units (defined in flce_api.cu).
#pragma once

#include <cuda_runtime.h>

namespace flce {

// The current device is one the library runs on (sm_103): returns the flce_status every
// entry point would return for it (set-up on first use per device).
int check_device();
// Remembers e for flce_last_cuda_error() and returns FLCE_ERR_CUDA.
int record_cuda_error(cudaError_t e);

}  // namespace flce

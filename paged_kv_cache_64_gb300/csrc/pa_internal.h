// Host-side helpers shared by the translation units of the library.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "pa.h"

namespace pa {

// Device address of the current device's error word (a file-scope __device__
// int in pa_cache.cu), looked up once per device.  nullptr on failure.
int *error_word();

// Number of SMs of the current device (cached per device); 0 on failure.
int sm_count();

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per (kernel, device).
bool ensure_smem_attr(const void *kernel, int bytes);

inline cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace pa

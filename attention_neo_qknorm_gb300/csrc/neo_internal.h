// Host-side helpers shared by the translation units of libneo.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "neo.h"

namespace neo {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline neo_status launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? NEO_OK : NEO_ERR_CUDA;
}

// Attention translation unit: device error word and wait limit.
neo_status attention_error_read_clear(cudaStream_t stream, uint32_t* word);
neo_status attention_set_timeout(uint64_t ns);

// Elementwise translation unit: its own device error word and wait limit.
neo_status elementwise_error_read_clear(uint32_t* word);
neo_status elementwise_set_timeout(uint64_t ns);

}  // namespace neo

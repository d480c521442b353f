// Host-side helpers shared by the translation units of libneo.
#pragma once

#include <cstdint>
#include <mutex>
#include <utility>
#include <cuda_runtime.h>

#include "neo.h"

namespace neo {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Whether the byte ranges [a, a + an) and [b, b + bn) share a byte (a null
// pointer or an empty range overlaps nothing).
inline bool overlap(const void* a, int64_t an, const void* b, int64_t bn) {
    if (!a || !b || an <= 0 || bn <= 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + (uintptr_t)bn && y < x + (uintptr_t)an;
}

// Host state that is set up once per device (kernel attributes, sizes
// derived from occupancy): one slot per device ordinal, filled the first time
// the library is called with that device current.
constexpr int kMaxDevices = 64;

struct DeviceOnce {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    int value[2] = {0, 0};
};

// The current device's slot of `slots` (kMaxDevices of them), or nullptr.
inline DeviceOnce* device_slot(DeviceOnce* slots) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    return &slots[dev];
}

inline neo_status launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? NEO_OK : NEO_ERR_CUDA;
}

// Launches `kernel` on `stream` allowing it to start while the previous kernel
// of the stream finishes (programmatic stream serialization); the kernel waits
// (griddepcontrol.wait) before its first global memory access.
template <typename... Params, typename... Args>
inline neo_status launch_overlapped(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return NEO_ERR_CUDA;
    }
    return launch_status();
}

// Attention translation unit: device error word and wait limit.
neo_status attention_error_read_clear(cudaStream_t stream, uint32_t* word);
neo_status attention_set_timeout(uint64_t ns);

// Elementwise translation unit: its own device error word and wait limit.
neo_status elementwise_error_read_clear(uint32_t* word);
neo_status elementwise_set_timeout(uint64_t ns);

}  // namespace neo

// Status strings, the device error word and the wait limit of libneo.

#include <cmath>
#include <cstdint>

#include <cuda_runtime.h>

#include "neo.h"
#include "neo_internal.h"

extern "C" const char* neo_status_string(neo_status s) {
    switch (s) {
        case NEO_OK: return "NEO_OK";
        case NEO_ERR_INVALID_ARG: return "NEO_ERR_INVALID_ARG: an argument failed the host-side checks";
        case NEO_ERR_UNSUPPORTED: return "NEO_ERR_UNSUPPORTED: valid arguments that this build does not implement";
        case NEO_ERR_CUDA: return "NEO_ERR_CUDA: a CUDA call or kernel launch failed";
        case NEO_ERR_TIMEOUT: return "NEO_ERR_TIMEOUT: a pipeline wait inside a kernel ran out of time";
        case NEO_ERR_DEVICE: return "NEO_ERR_DEVICE: a kernel rejected its device-side inputs";
    }
    return "unknown neo_status";
}

extern "C" neo_status neo_get_device_error(cudaStream_t stream, uint32_t* word) {
    uint32_t a = 0, e = 0;
    neo_status st = neo::attention_error_read_clear(stream, &a);   // synchronises the stream
    if (st == NEO_ERR_CUDA) return st;
    if (neo::elementwise_error_read_clear(&e) != NEO_OK) return NEO_ERR_CUDA;
    const uint32_t all = a | e;
    if (word) *word = all;
    if (all & NEO_DEVERR_TIMEOUT) return NEO_ERR_TIMEOUT;
    return all ? NEO_ERR_DEVICE : NEO_OK;
}

extern "C" neo_status neo_set_wait_timeout_ns(uint64_t ns) {
    if (ns == 0) return NEO_ERR_INVALID_ARG;
    const neo_status st = neo::attention_set_timeout(ns);
    return st != NEO_OK ? st : neo::elementwise_set_timeout(ns);
}

extern "C" int neo_version(void) { return 100; }

extern "C" neo_status neo_time_schedule(float* t_out, int n_steps, float shift) {
    if (!t_out || n_steps < 1 || !(shift > 0.f) || !std::isfinite(shift)) return NEO_ERR_INVALID_ARG;
    const double s = shift;
    for (int k = 0; k <= n_steps; ++k) {
        const double t = (double)k / n_steps;
        double sigma = 1.0 - t;
        sigma = s * sigma / (1.0 + (s - 1.0) * sigma);
        t_out[k] = (float)(1.0 - sigma);
    }
    return NEO_OK;
}

extern "C" neo_status neo_noise_scale(int grid_h, int grid_w, int merge, float base_seq_len, float base_scale,
                                      int mode, float max_value, float* out) {
    if (!out || grid_h < 1 || grid_w < 1 || merge < 1 || !(base_seq_len > 0.f) || !std::isfinite(base_scale) ||
        !std::isfinite(max_value))
        return NEO_ERR_INVALID_ARG;
    double s = base_scale;
    if (mode == NEO_NOISE_RESOLUTION || mode == NEO_NOISE_DYNAMIC || mode == NEO_NOISE_DYNAMIC_SQRT) {
        s = std::sqrt((double)grid_h * grid_w / ((double)merge * merge) / base_seq_len) * base_scale;
        if (mode == NEO_NOISE_DYNAMIC_SQRT) s = std::sqrt(s);
    } else if (mode != NEO_NOISE_CONSTANT) {
        return NEO_ERR_INVALID_ARG;
    }
    *out = (float)std::fmin(s, (double)max_value);
    return NEO_OK;
}

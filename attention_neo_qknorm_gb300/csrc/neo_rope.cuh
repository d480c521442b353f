// Rotary-angle helpers shared by the norm/RoPE kernels and the attention
// prologue that folds the query norm/RoPE in: both must produce the same bits.
#pragma once

#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>

namespace neo {

// The frequency theta^(-2i/d) of each rotation pair of the three-axis RoPE as
// a fraction of a full turn, f / (2 pi), in 64-bit fixed point (units of
// 2^-64 turn). Pairs [0,32) temporal (d = 64), [32,48) height, [48,64) width
// (d = 32 each).
struct RopeFreqs {
    uint64_t turn[64];
};

// f / (2 pi) in [0, 1) as round-down(f / (2 pi) * 2^64), from the double
// value: the two 32-bit halves of the fraction are taken one after the other,
// so all 53 bits of the double survive.
inline uint64_t turn_fraction64(double f) {
    const double two_pi = 6.283185307179586476925286766559;
    double t = f / two_pi;
    t -= std::floor(t);
    const double a = std::ldexp(t, 32);
    const double hi = std::floor(a);
    const double lo = std::floor(std::ldexp(a - hi, 32));
    return ((uint64_t)hi << 32) | (uint64_t)lo;
}

inline RopeFreqs rope3_freqs(float theta_t, float theta_hw) {
    RopeFreqs fr;
    for (int i = 0; i < 32; ++i) fr.turn[i] = turn_fraction64(std::pow((double)theta_t, -2.0 * i / 64.0));
    for (int i = 0; i < 16; ++i) {
        const uint64_t f = turn_fraction64(std::pow((double)theta_hw, -2.0 * i / 32.0));
        fr.turn[32 + i] = f;
        fr.turn[48 + i] = f;
    }
    return fr;
}

// sin/cos of the angle pos * f. The integer product pos * (f / 2 pi) modulo
// one turn is exact in wrapping 64-bit arithmetic (pos is an integer, the
// frequency a 64-bit fraction of a turn), so there is no range reduction and
// no position limit: every int32 position, negative ones included, gets its
// angle to within the frequency's own rounding (2^-53 relative) times pos.
// The top 32 bits, read as a signed fraction of a turn in [-1/2, 1/2), become
// the fp32 angle in [-pi, pi) for the SFU's sin/cos.
__device__ __forceinline__ void rope_sincos(int32_t pos, uint64_t turn, float* sn, float* cs) {
    constexpr float kRadPerUnit = 1.4629180792671596e-09f;   // 2 pi / 2^32
    const uint64_t phase = (uint64_t)(int64_t)pos * turn;    // mod 2^64 = mod one turn
    const float r = (float)(int32_t)(uint32_t)(phase >> 32) * kRadPerUnit;
    __sincosf(r, sn, cs);
}

// sin/cos of pos * f for a small position and an fp32 frequency (the vision
// tower's 2-D RoPE: patch rows and columns, a few hundred at most): the fp32
// product is reduced modulo 2 pi by the two-constant Cody-Waite scheme
// (2 pi = C1 + C2, each fp32, folded in with fma) before the SFU's sin/cos.
__device__ __forceinline__ void rope_sincos_small(float pos, float f, float* sn, float* cs) {
    constexpr float kTwoPiHi = 6.28318548202514648f;        // fp32(2 pi)
    constexpr float kTwoPiLo = -1.7484556025237907e-07f;    // 2 pi - kTwoPiHi
    constexpr float kInvTwoPi = 0.15915494309189535f;
    const float a = pos * f;
    const float k = rintf(a * kInvTwoPi);
    float r = fmaf(-k, kTwoPiHi, a);
    r = fmaf(-k, kTwoPiLo, r);
    __sincosf(r, sn, cs);
}

}  // namespace neo

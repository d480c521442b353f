// Rotary-angle helpers shared by the norm/RoPE kernels and the attention
// prologue that folds the query norm/RoPE in: both must produce the same bits.
#pragma once

#include <cmath>
#include <cuda_runtime.h>

namespace neo {

// theta^(-2i/d) of each rotation pair of the three-axis RoPE, split as hi + lo:
// hi keeps 11 significant bits so that pos * hi is exact in fp32 for positions
// below 2^13. Pairs [0,32) temporal (d = 64), [32,48) height, [48,64) width
// (d = 32 each).
struct RopeFreqs {
    float hi[64];
    float lo[64];
};

// f as hi (11 significant bits) + lo, computed in double.
inline void split_freq(double f, float* hi, float* lo) {
    int e;
    const double m = std::frexp(f, &e);                       // f = m * 2^e, m in [0.5, 1)
    const double h = std::ldexp(std::floor(m * 2048.0) / 2048.0, e);
    *hi = (float)h;
    *lo = (float)(f - h);
}

inline RopeFreqs rope3_freqs(float theta_t, float theta_hw) {
    RopeFreqs fr;
    for (int i = 0; i < 32; ++i) split_freq(std::pow((double)theta_t, -2.0 * i / 64.0), &fr.hi[i], &fr.lo[i]);
    for (int i = 0; i < 16; ++i) {
        const double f = std::pow((double)theta_hw, -2.0 * i / 32.0);
        split_freq(f, &fr.hi[32 + i], &fr.lo[32 + i]);
        split_freq(f, &fr.hi[48 + i], &fr.lo[48 + i]);
    }
    return fr;
}

// sin/cos of pos * f with f = hi + lo: the exact product pos * hi is reduced
// modulo 2*pi by the two-constant Cody-Waite scheme (2*pi = C1 + C2, each
// fp32, products folded with fma), then the small product pos * lo is added
// and the SFU evaluates sin/cos on the reduced argument in [-pi, pi].
__device__ __forceinline__ void rope_sincos(float pos, float f_hi, float f_lo, float* sn, float* cs) {
    constexpr float kTwoPiHi = 6.28318548202514648f;        // fp32(2*pi)
    constexpr float kTwoPiLo = -1.7484556025237907e-07f;    // 2*pi - kTwoPiHi
    constexpr float kInvTwoPi = 0.15915494309189535f;
    const float a = pos * f_hi;
    const float k = rintf(a * kInvTwoPi);
    float r = fmaf(-k, kTwoPiHi, a);
    r = fmaf(-k, kTwoPiLo, r);
    r = fmaf(pos, f_lo, r);
    __sincosf(r, sn, cs);
}

}  // namespace neo

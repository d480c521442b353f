// HBM-bound kernels of the generation-pass hot path: position indexes,
// QK-norm on head halves + three-axis RoPE, and the x0 -> v Euler step.
//
// Sources (page title, section):
//   [U15] "SenseNova-U1.5 (NEO-unify) architecture"
//   [U1]  "SenseNova-U1: Unifying Multimodal Understanding and Generation with
//          NEO-unify Architecture"

#include <algorithm>
#include <cmath>
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "neo.h"
#include "neo_internal.h"

namespace {

int sm_count() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
    }
    return n;
}

// ---------------------------------------------------------------------------
// Position indexes ([U15] "Three rotary axes", last paragraph).
// ---------------------------------------------------------------------------
struct SegmentList {
    neo_pos_segment seg[NEO_MAX_SEGMENTS];
    int64_t start[NEO_MAX_SEGMENTS + 1];
    int n;
};

__global__ void positions_kernel(int32_t* __restrict__ idx, int64_t S, const SegmentList L) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < S;
         i += (int64_t)gridDim.x * blockDim.x) {
        int s = 0;
        while (s + 1 < L.n && i >= L.start[s + 1]) ++s;
        const neo_pos_segment g = L.seg[s];
        const int64_t local = i - L.start[s];
        int32_t t, r, c;
        if (g.kind == NEO_SEG_TEXT) {
            t = r = c = g.a + (int32_t)local;
        } else {
            t = g.a;
            r = (int32_t)(local / g.c);
            c = (int32_t)(local % g.c);
        }
        idx[i] = t;
        idx[S + i] = r;
        idx[2 * S + i] = c;
    }
}

// ---------------------------------------------------------------------------
// QK-norm on halves + three-axis RoPE ([U15] "Three rotary axes").
//
// A CTA owns kTokensPerCta consecutive tokens and every q and k head row of
// them. It first builds the (cos, sin) table of the tokens' 64 rotation pairs
// in shared memory (pairs [0,32) temporal, [32,48) height, [48,64) width;
// the angle only depends on the token, so each sincos is shared by all
// Hq + Hkv heads), then streams the rows. Each row of 128 values is handled
// by 16 lanes with 16-byte accesses (8 bf16 or 4 fp32 per lane: 16 or 32
// lanes per row). The half's sum of squares is reduced with shuffles; the
// rotation partner of a lane's values sits d/2 dims away, i.e. a fixed lane
// xor within the same half, so one shuffle per value brings it over.
// ---------------------------------------------------------------------------
struct RopeFreqs {
    float f[64];   // theta^(-2i/d) per pair, in table order
};

constexpr int kNormThreads = 256;
constexpr int kTokensPerCta = 8;
constexpr int kRowUnroll = 2;

template <typename T>
struct LaneIO;

template <>
struct LaneIO<__nv_bfloat16> {
    static constexpr int E = 8;
    static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&x)[8]) {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
            const float2 f = __bfloat1622float2(h);
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&y)[8]) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(y[2 * i], y[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};

template <>
struct LaneIO<float> {
    static constexpr int E = 4;
    static __device__ __forceinline__ void load(const float* p, float (&x)[4]) {
        const float4 u = *reinterpret_cast<const float4*>(p);
        x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
    }
    static __device__ __forceinline__ void store(float* p, const float (&y)[4]) {
        *reinterpret_cast<float4*>(p) = make_float4(y[0], y[1], y[2], y[3]);
    }
};

template <typename T>
__global__ void __launch_bounds__(kNormThreads)
qknorm_rope3_kernel(T* __restrict__ q, T* __restrict__ k, int64_t S, int Hq, int Hkv,
                    const int32_t* __restrict__ idx,
                    const float* __restrict__ wq_t, const float* __restrict__ wq_hw,
                    const float* __restrict__ wk_t, const float* __restrict__ wk_hw,
                    const RopeFreqs freqs, float eps) {
    constexpr int E = LaneIO<T>::E;          // values per lane
    constexpr int LPR = 128 / E;             // lanes per row
    constexpr int ROWS_PER_WARP = 32 / LPR;
    constexpr int WORKERS = kNormThreads / LPR;
    constexpr int HALF_LANES = 64 / E;       // lanes per normalised half

    __shared__ float2 cs[kTokensPerCta][64];
    __shared__ float wq[128];
    __shared__ float wk[128];

    const int64_t tok0 = (int64_t)blockIdx.x * kTokensPerCta;
    const int ntok = (int)(S - tok0 < kTokensPerCta ? S - tok0 : kTokensPerCta);

    for (int e = threadIdx.x; e < ntok * 64; e += kNormThreads) {
        const int t = e >> 6, pr = e & 63;
        const int axis = pr < 32 ? 0 : (pr < 48 ? 1 : 2);
        const float pos = (float)idx[axis * S + tok0 + t];
        float sn, cn;
        sincosf(pos * freqs.f[pr], &sn, &cn);
        cs[t][pr] = make_float2(cn, sn);
    }
    for (int e = threadIdx.x; e < 128; e += kNormThreads) {
        wq[e] = Hq > 0 ? (e < 64 ? wq_t[e] : wq_hw[e - 64]) : 0.f;
        wk[e] = Hkv > 0 ? (e < 64 ? wk_t[e] : wk_hw[e - 64]) : 0.f;
    }
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int sub = threadIdx.x % LPR;              // lane within the row
    const int e0 = sub * E;                          // first head dim of this lane
    const bool temporal = e0 < 64;
    const int slice_off = temporal ? 0 : (e0 < 96 ? 64 : 96);
    const int half_w = temporal ? 32 : 16;           // half the slice width
    const bool first = (e0 - slice_off) < half_w;    // lane holds the u side of its pairs
    const int pair0 = (temporal ? 0 : (e0 < 96 ? 32 : 48)) + (e0 - slice_off) % half_w;
    const int partner = lane ^ (half_w / E);

    const int H = Hq + Hkv;
    const int rows = ntok * H;
    const int warp_row0 = (threadIdx.x >> 5) * ROWS_PER_WARP;
    const int my_off = lane / LPR;

    for (int rb = warp_row0; rb < rows; rb += WORKERS * kRowUnroll) {
        float x[kRowUnroll][E];
        T* ptr[kRowUnroll];
        int tok[kRowUnroll];
        bool active[kRowUnroll];
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) {
            const int r = rb + u * WORKERS + my_off;
            active[u] = r < rows;
            const int t = active[u] ? r / H : 0;
            const int h = active[u] ? r % H : 0;
            tok[u] = t;
            ptr[u] = h < Hq ? q + ((tok0 + t) * Hq + h) * 128 + e0
                            : k + ((tok0 + t) * Hkv + (h - Hq)) * 128 + e0;
            if (active[u]) {
                LaneIO<T>::load(ptr[u], x[u]);
            } else {
#pragma unroll
                for (int j = 0; j < E; ++j) x[u][j] = 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) {
            const int r = rb + u * WORKERS + my_off;
            const float* w = (active[u] && (r % H) < Hq) ? wq : wk;
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < E; ++j) ss = fmaf(x[u][j], x[u][j], ss);
#pragma unroll
            for (int m = 1; m < HALF_LANES; m <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
            const float rs = rsqrtf(ss * (1.0f / 64.0f) + eps);
            float y[E], yp[E], o[E];
#pragma unroll
            for (int j = 0; j < E; ++j) y[j] = x[u][j] * rs * w[e0 + j];
#pragma unroll
            for (int j = 0; j < E; ++j) yp[j] = __shfl_sync(0xffffffffu, y[j], partner);
#pragma unroll
            for (int j = 0; j < E; ++j) {
                const float2 c = cs[tok[u]][pair0 + j];
                o[j] = first ? fmaf(y[j], c.x, -yp[j] * c.y) : fmaf(y[j], c.x, yp[j] * c.y);
            }
            if (active[u]) LaneIO<T>::store(ptr[u], o);
        }
    }
}

// ---------------------------------------------------------------------------
// x0 -> v and the Euler step ([U15] "Flow matching without a VAE").
// ---------------------------------------------------------------------------
constexpr int kEulerThreads = 256;
constexpr int kEulerUnroll = 4;

__global__ void __launch_bounds__(kEulerThreads)
flow_euler_kernel(float* __restrict__ z, const float* __restrict__ x0, int64_t n, float den,
                  float dt, float* __restrict__ v_out) {
    const int64_t n4 = n >> 2;
    const int64_t stride = (int64_t)gridDim.x * kEulerThreads;
    const int64_t tid = (int64_t)blockIdx.x * kEulerThreads + threadIdx.x;
    float4* z4 = reinterpret_cast<float4*>(z);
    const float4* x4 = reinterpret_cast<const float4*>(x0);
    float4* v4 = reinterpret_cast<float4*>(v_out);
    for (int64_t base = tid; base < n4; base += stride * kEulerUnroll) {
        float4 zz[kEulerUnroll], xx[kEulerUnroll];
#pragma unroll
        for (int u = 0; u < kEulerUnroll; ++u) {
            const int64_t i = base + u * stride;
            if (i < n4) {
                zz[u] = z4[i];
                xx[u] = __ldg(x4 + i);
            }
        }
#pragma unroll
        for (int u = 0; u < kEulerUnroll; ++u) {
            const int64_t i = base + u * stride;
            if (i < n4) {
                float4 v;
                v.x = (xx[u].x - zz[u].x) / den;
                v.y = (xx[u].y - zz[u].y) / den;
                v.z = (xx[u].z - zz[u].z) / den;
                v.w = (xx[u].w - zz[u].w) / den;
                float4 zn;
                zn.x = fmaf(dt, v.x, zz[u].x);
                zn.y = fmaf(dt, v.y, zz[u].y);
                zn.z = fmaf(dt, v.z, zz[u].z);
                zn.w = fmaf(dt, v.w, zz[u].w);
                z4[i] = zn;
                if (v_out) v4[i] = v;
            }
        }
    }
    for (int64_t i = (n4 << 2) + tid; i < n; i += stride) {
        const float v = (x0[i] - z[i]) / den;
        z[i] = fmaf(dt, v, z[i]);
        if (v_out) v_out[i] = v;
    }
}

}  // namespace

// ===========================================================================
// C ABI
// ===========================================================================
extern "C" neo_status neo_build_positions(int32_t* indexes, int64_t S, const neo_pos_segment* segs,
                                          int n_segs, cudaStream_t stream) {
    if (!indexes || !segs || S < 0 || n_segs < 1 || n_segs > NEO_MAX_SEGMENTS) return NEO_ERR_INVALID_ARG;
    SegmentList L{};
    L.n = n_segs;
    int64_t total = 0;
    for (int s = 0; s < n_segs; ++s) {
        const neo_pos_segment g = segs[s];
        int64_t count;
        if (g.kind == NEO_SEG_TEXT) {
            if (g.b < 0 || g.a < 0) return NEO_ERR_INVALID_ARG;
            count = g.b;
        } else if (g.kind == NEO_SEG_IMAGE) {
            if (g.a < 0 || g.b < 0 || g.c < 0 || (g.b > 0 && g.c == 0)) return NEO_ERR_INVALID_ARG;
            count = (int64_t)g.b * g.c;
        } else {
            return NEO_ERR_INVALID_ARG;
        }
        L.seg[s] = g;
        L.start[s] = total;
        total += count;
    }
    L.start[n_segs] = total;
    if (total != S) return NEO_ERR_INVALID_ARG;
    if (S == 0) return NEO_OK;
    const int threads = 256;
    const int64_t blocks = std::min<int64_t>((S + threads - 1) / threads, (int64_t)sm_count() * 8);
    positions_kernel<<<(unsigned)blocks, threads, 0, stream>>>(indexes, S, L);
    return neo::launch_status();
}

extern "C" neo_status neo_qknorm_rope3(void* q, void* k, neo_dtype dtype, int64_t S, int Hq, int Hkv,
                                       int D, const int32_t* indexes, const float* q_norm_w,
                                       const float* q_norm_hw_w, const float* k_norm_w,
                                       const float* k_norm_hw_w, float theta_t, float theta_hw,
                                       float eps, cudaStream_t stream) {
    if (D != 128 || S < 0 || Hq < 0 || Hkv < 0) return NEO_ERR_INVALID_ARG;
    if (dtype != NEO_BF16 && dtype != NEO_F32) return NEO_ERR_INVALID_ARG;
    if (Hq > 0 && (!q || !q_norm_w || !q_norm_hw_w || !neo::aligned16(q))) return NEO_ERR_INVALID_ARG;
    if (Hkv > 0 && (!k || !k_norm_w || !k_norm_hw_w || !neo::aligned16(k))) return NEO_ERR_INVALID_ARG;
    if (!(theta_t > 0.f) || !(theta_hw > 0.f) || !(eps >= 0.f) || !std::isfinite(theta_t) ||
        !std::isfinite(theta_hw) || !std::isfinite(eps))
        return NEO_ERR_INVALID_ARG;
    if (S == 0 || Hq + Hkv == 0) return NEO_OK;
    if (!indexes) return NEO_ERR_INVALID_ARG;

    // theta^(-2i/d) per pair, computed in double and rounded once to fp32.
    RopeFreqs fr;
    for (int i = 0; i < 32; ++i) fr.f[i] = (float)std::pow((double)theta_t, -2.0 * i / 64.0);
    for (int i = 0; i < 16; ++i) {
        const float f = (float)std::pow((double)theta_hw, -2.0 * i / 32.0);
        fr.f[32 + i] = f;
        fr.f[48 + i] = f;
    }
    const int64_t blocks = (S + kTokensPerCta - 1) / kTokensPerCta;
    if (blocks > 0x7fffffffLL) return NEO_ERR_INVALID_ARG;
    if (dtype == NEO_BF16) {
        qknorm_rope3_kernel<__nv_bfloat16><<<(unsigned)blocks, kNormThreads, 0, stream>>>(
            static_cast<__nv_bfloat16*>(q), static_cast<__nv_bfloat16*>(k), S, Hq, Hkv, indexes,
            q_norm_w, q_norm_hw_w, k_norm_w, k_norm_hw_w, fr, eps);
    } else {
        qknorm_rope3_kernel<float><<<(unsigned)blocks, kNormThreads, 0, stream>>>(
            static_cast<float*>(q), static_cast<float*>(k), S, Hq, Hkv, indexes, q_norm_w,
            q_norm_hw_w, k_norm_w, k_norm_hw_w, fr, eps);
    }
    return neo::launch_status();
}

extern "C" neo_status neo_flow_euler_step(float* z, const float* x0_hat, int64_t n, float t,
                                          float t_next, float t_eps, float* v_out,
                                          cudaStream_t stream) {
    if (n < 0 || !std::isfinite(t) || !std::isfinite(t_next) || !std::isfinite(t_eps))
        return NEO_ERR_INVALID_ARG;
    if (n == 0) return NEO_OK;
    if (!z || !x0_hat || !neo::aligned16(z) || !neo::aligned16(x0_hat)) return NEO_ERR_INVALID_ARG;
    if (v_out && !neo::aligned16(v_out)) return NEO_ERR_INVALID_ARG;
    const float den = std::fmax(1.0f - t, t_eps);
    if (!(den > 0.f)) return NEO_ERR_INVALID_ARG;
    const float dt = t_next - t;
    const int64_t n4 = (n + 3) / 4;
    const int64_t want = (n4 + kEulerThreads * kEulerUnroll - 1) / (kEulerThreads * kEulerUnroll);
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sm_count() * 8));
    flow_euler_kernel<<<(unsigned)blocks, kEulerThreads, 0, stream>>>(z, x0_hat, n, den, dt, v_out);
    return neo::launch_status();
}

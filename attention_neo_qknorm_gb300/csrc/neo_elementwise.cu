// HBM-bound kernels of the generation-pass hot path: position indexes,
// QK-norm on head halves + three-axis RoPE, and the x0 -> v Euler step.
//
// Sources (page title, section):
//   [U15] "SenseNova-U1.5 (NEO-unify) architecture"
//   [U1]  "SenseNova-U1: Unifying Multimodal Understanding and Generation with
//          NEO-unify Architecture"

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "neo.h"
#include "neo_internal.h"
#include "neo_rope.cuh"
#include "sm103_ptx.cuh"

namespace {

using neo::RopeFreqs;
using neo::rope_sincos;

// The current device's SM count (looked up once per device).
int sm_count() {
    static neo::DeviceOnce slots[neo::kMaxDevices];
    neo::DeviceOnce* s = neo::device_slot(slots);
    if (!s) return 152;
    std::call_once(s->once, [s] {
        int dev = 0, n = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 152;
        s->value[0] = n;
    });
    return s->value[0];
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
// One warp per token and tensor: it normalises and rotates the token's Hq
// query rows (or its Hkv key rows), so the (cos, sin) of the token's angles
// are computed once per lane and serve all of them. A row of 128 values is owned by a group
// of lanes in which every lane holds BOTH members of its rotation pairs: two
// 16-byte chunks at dims [a, a+E) and [a+d/2, a+d/2+E) of its slice (E = 8
// bf16 or 4 fp32), so the rotation needs no data exchange. Lanes [0, 32/E) of
// the group cover the temporal slice [0,64) (= the first normalised half), the
// others the height [64,96) and width [96,128) slices (= the second half); a
// half's sum of squares is a shuffle reduction inside that aligned lane group.
// With the norm weight w folded into the angle's (cos, sin), a pair (u, v) of
// a row with inverse RMS r becomes
//   u' = r * (u * w_u * cos - v * w_v * sin),  v' = r * (v * w_v * cos + u * w_u * sin),
// four products per lane and token kept in registers. The token's rows stream
// through a private ring of kNormDepth chunks of kNormChunkRows rows in shared
// memory, filled with cp.async: a lane copies exactly the bytes it later
// reads, so its own wait_group is the only synchronisation. The arithmetic
// runs on the packed fp32x2 datapath.
// ---------------------------------------------------------------------------
__device__ unsigned int g_elem_error = 0;
__device__ unsigned long long g_elem_wait_limit_ns = 1000000000ull;


constexpr int kNormWarps = 4;        // tokens per CTA, one per warp
constexpr int kNormChunkRows = 8;    // rows per ring slot
constexpr int kNormDepth = 3;        // ring slots per warp (24 rows in flight)


template <typename T>
struct Chunk;    // one 16-byte chunk of a row

template <>
struct Chunk<__nv_bfloat16> {
    static constexpr int E = 8;
    static __device__ __forceinline__ void unpack(uint4 u, float (&x)[8]) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        }
    }
    // Elements (2i, 2i+1) as one pair: a bf16 is the top half of an fp32.
    static __device__ __forceinline__ void unpack2(uint4 u, float2 (&x)[4]) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
    }
    static __device__ __forceinline__ uint4 pack2(const float2 (&y)[4]) {
        return make_uint4(sm103::pack_bf16x2(y[0].x, y[0].y), sm103::pack_bf16x2(y[1].x, y[1].y),
                          sm103::pack_bf16x2(y[2].x, y[2].y), sm103::pack_bf16x2(y[3].x, y[3].y));
    }
    static __device__ __forceinline__ uint4 pack(const float (&y)[8]) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(y[2 * i], y[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

template <>
struct Chunk<float> {
    static constexpr int E = 4;
    static __device__ __forceinline__ void unpack(uint4 u, float (&x)[4]) {
        x[0] = __uint_as_float(u.x); x[1] = __uint_as_float(u.y);
        x[2] = __uint_as_float(u.z); x[3] = __uint_as_float(u.w);
    }
    static __device__ __forceinline__ uint4 pack(const float (&y)[4]) {
        return make_uint4(__float_as_uint(y[0]), __float_as_uint(y[1]), __float_as_uint(y[2]), __float_as_uint(y[3]));
    }
    static __device__ __forceinline__ void unpack2(uint4 u, float2 (&x)[2]) {
        x[0] = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
        x[1] = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
    }
    static __device__ __forceinline__ uint4 pack2(const float2 (&y)[2]) {
        return make_uint4(__float_as_uint(y[0].x), __float_as_uint(y[0].y), __float_as_uint(y[1].x),
                          __float_as_uint(y[1].y));
    }
};

template <typename T>
__global__ void __launch_bounds__(kNormWarps * 32)
qknorm_rope3_kernel(T* __restrict__ q, T* __restrict__ k, int64_t S, int Hq, int Hkv,
                    const int32_t* __restrict__ idx,
                    const float* __restrict__ wq_t, const float* __restrict__ wq_hw,
                    const float* __restrict__ wk_t, const float* __restrict__ wk_hw,
                    const __grid_constant__ RopeFreqs freqs, float eps) {
    using sm103::ffma2;
    using sm103::fmul2;
    constexpr int E = Chunk<T>::E;
    constexpr int P = E / 2;                 // element pairs per chunk
    constexpr int LPR = 64 / E;              // lanes per row (8 bf16, 16 fp32)
    constexpr int HALF_LANES = 32 / E;       // lanes per normalised half
    constexpr int RPW = 32 / LPR;            // rows per warp instruction
    constexpr int ROW_BYTES = 128 * (int)sizeof(T);
    constexpr int CHUNK_BYTES = kNormChunkRows * ROW_BYTES;
    static_assert(kNormChunkRows % RPW == 0, "a ring slot holds whole row groups");

    extern __shared__ __align__(16) uint8_t ring_mem[];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int sub = lane % LPR;
    const int rslot = lane / LPR;
    // This lane's slice, first dims of its u and v chunks, first pair (table order).
    int dim_a, half_w, pair0, axis;
    if (sub < HALF_LANES) {
        dim_a = sub * E; half_w = 32; pair0 = sub * E; axis = 0;
    } else if (sub < HALF_LANES + HALF_LANES / 2) {
        const int m = sub - HALF_LANES;
        dim_a = 64 + m * E; half_w = 16; pair0 = 32 + m * E; axis = 1;
    } else {
        const int m = sub - HALF_LANES - HALF_LANES / 2;
        dim_a = 96 + m * E; half_w = 16; pair0 = 48 + m * E; axis = 2;
    }
    const int dim_b = dim_a + half_w;
    const int64_t tok = (int64_t)blockIdx.x * kNormWarps + warp;
    if (tok >= S) return;
    // blockIdx.y picks the tensor: the q rows and the k rows of a token are
    // handled by different CTAs, so that each CTA streams one contiguous region.
    const int which = Hq > 0 ? (int)blockIdx.y : 1;
    const int R = which ? Hkv : Hq;          // the token's rows of that tensor
    const int n_chunks = (R + kNormChunkRows - 1) / kNormChunkRows;
    uint8_t* ring = ring_mem + (size_t)warp * kNormDepth * CHUNK_BYTES;
    T* const rows = which ? k + tok * Hkv * 128 : q + tok * Hq * 128;
    auto row_ptr = [&](int r) -> T* { return rows + r * 128; };
    auto issue = [&](int c) {
        if (c < n_chunks) {
            const uint32_t slot = sm103::smem_addr(ring + (c % kNormDepth) * CHUNK_BYTES);
#pragma unroll
            for (int g = 0; g < kNormChunkRows / RPW; ++g) {
                const int rr = g * RPW + rslot;
                const int r = c * kNormChunkRows + rr;
                if (r < R) {
                    const T* src = row_ptr(r);
                    const uint32_t d = slot + (uint32_t)(rr * ROW_BYTES);
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d + dim_a * (uint32_t)sizeof(T)),
                                 "l"(src + dim_a) : "memory");
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d + dim_b * (uint32_t)sizeof(T)),
                                 "l"(src + dim_b) : "memory");
                }
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");   // possibly empty: keeps the group count uniform
    };
    // The attention launched after this kernel may start setting up its CTAs
    // now; it waits for this grid to complete before it reads q and k.
    sm103::griddep_launch_dependents();
#pragma unroll
    for (int c = 0; c < kNormDepth; ++c) issue(c);

    // The token's angles for this lane's pairs, and the weight-folded products
    // (w_u cos, -w_v sin) for u' and (w_v cos, w_u sin) for v', element pairs packed.
    const int32_t pos = __ldg(idx + axis * S + tok);
    float cs[E], sn[E];
#pragma unroll
    for (int j = 0; j < E; ++j) rope_sincos(pos, freqs.turn[pair0 + j], &sn[j], &cs[j]);
    float2 uc[P], vs[P], vc[P], us[P];
    auto fold = [&](int which) {
        // The lane's dims lie in one normalised half: the temporal weights for
        // [0,64), the height/width weights for [64,128). The weight loads come
        // after the ring's copies are in flight.
        const float* w = dim_a < 64 ? (which ? wk_t : wq_t) : (which ? wk_hw : wq_hw) - 64;
#pragma unroll
        for (int i = 0; i < P; ++i) {
            const float wu0 = __ldg(w + dim_a + 2 * i), wu1 = __ldg(w + dim_a + 2 * i + 1);
            const float wv0 = __ldg(w + dim_b + 2 * i), wv1 = __ldg(w + dim_b + 2 * i + 1);
            uc[i] = make_float2(wu0 * cs[2 * i], wu1 * cs[2 * i + 1]);
            vs[i] = make_float2(-wv0 * sn[2 * i], -wv1 * sn[2 * i + 1]);
            vc[i] = make_float2(wv0 * cs[2 * i], wv1 * cs[2 * i + 1]);
            us[i] = make_float2(wu0 * sn[2 * i], wu1 * sn[2 * i + 1]);
        }
    };
    fold(which);

    for (int c = 0; c < n_chunks; ++c) {
        asm volatile("cp.async.wait_group %0;" ::"n"(kNormDepth - 1) : "memory");
        const uint8_t* slot = ring + (c % kNormDepth) * CHUNK_BYTES;
#pragma unroll
        for (int g = 0; g < kNormChunkRows / RPW; ++g) {
            const int rr = g * RPW + rslot;
            const int r = c * kNormChunkRows + rr;
            const bool live = r < R;
            uint4 ua = make_uint4(0u, 0u, 0u, 0u), ub = ua;
            if (live) {
                ua = *reinterpret_cast<const uint4*>(slot + rr * ROW_BYTES + dim_a * (int)sizeof(T));
                ub = *reinterpret_cast<const uint4*>(slot + rr * ROW_BYTES + dim_b * (int)sizeof(T));
            }
            float2 xa[P], xb[P];
            Chunk<T>::unpack2(ua, xa);
            Chunk<T>::unpack2(ub, xb);
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < P; ++i) acc = ffma2(xa[i], xa[i], ffma2(xb[i], xb[i], acc));
            float ss = acc.x + acc.y;
#pragma unroll
            for (int m = 1; m < HALF_LANES; m <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
            const float rs = rsqrtf(ss * (1.0f / 64.0f) + eps);
            const float2 rs2 = make_float2(rs, rs);
            float2 ya[P], yb[P];
#pragma unroll
            for (int i = 0; i < P; ++i) {
                const float2 u = fmul2(xa[i], rs2), v = fmul2(xb[i], rs2);
                ya[i] = ffma2(u, uc[i], fmul2(v, vs[i]));
                yb[i] = ffma2(v, vc[i], fmul2(u, us[i]));
            }
            if (live) {
                T* dst = row_ptr(r);
                *reinterpret_cast<uint4*>(dst + dim_a) = Chunk<T>::pack2(ya);
                *reinterpret_cast<uint4*>(dst + dim_b) = Chunk<T>::pack2(yb);
            }
        }
        issue(c + kNormDepth);   // into the slot this lane just read
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
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

// ---------------------------------------------------------------------------
// Classifier-free guidance fused with the Euler step ([U1] §2.7). Every
// branch's velocity is v_X = (x0_X - z) / den and the guidance weights of a
// branch sum to one, so the guided velocity is v = (sum_X w_X x0_X - z) / den;
// the kernel reads the K x0 buffers the branch needs once, with z.
// ---------------------------------------------------------------------------
template <int K>
__global__ void __launch_bounds__(kEulerThreads)
flow_cfg_kernel(float* __restrict__ z, const float* __restrict__ xa, const float* __restrict__ xb,
                const float* __restrict__ xc, int64_t n, float wa, float wb, float wc, float den, float dt,
                float* __restrict__ v_out) {
    const int64_t n4 = n >> 2;
    const int64_t stride = (int64_t)gridDim.x * kEulerThreads;
    const int64_t tid = (int64_t)blockIdx.x * kEulerThreads + threadIdx.x;
    float4* z4 = reinterpret_cast<float4*>(z);
    const float4* a4 = reinterpret_cast<const float4*>(xa);
    const float4* b4 = reinterpret_cast<const float4*>(xb);
    const float4* c4 = reinterpret_cast<const float4*>(xc);
    float4* v4 = reinterpret_cast<float4*>(v_out);
    auto mix = [&](float a, float b, float c) {
        float x = wa * a;
        if (K > 1) x = fmaf(wb, b, x);
        if (K > 2) x = fmaf(wc, c, x);
        return x;
    };
    for (int64_t base = tid; base < n4; base += stride * 2) {
        float4 zz[2], aa[2], bb[2], cc[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t i = base + u * stride;
            if (i < n4) {
                zz[u] = z4[i];
                aa[u] = __ldg(a4 + i);
                if (K > 1) bb[u] = __ldg(b4 + i);
                if (K > 2) cc[u] = __ldg(c4 + i);
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t i = base + u * stride;
            if (i < n4) {
                float4 v;
                v.x = (mix(aa[u].x, bb[u].x, cc[u].x) - zz[u].x) / den;
                v.y = (mix(aa[u].y, bb[u].y, cc[u].y) - zz[u].y) / den;
                v.z = (mix(aa[u].z, bb[u].z, cc[u].z) - zz[u].z) / den;
                v.w = (mix(aa[u].w, bb[u].w, cc[u].w) - zz[u].w) / den;
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
        const float v = (mix(xa[i], K > 1 ? xb[i] : 0.f, K > 2 ? xc[i] : 0.f) - z[i]) / den;
        z[i] = fmaf(dt, v, z[i]);
        if (v_out) v_out[i] = v;
    }
}

// z_0 = sigma * eps ([U1] §2.3).
__global__ void __launch_bounds__(kEulerThreads)
scale_noise_kernel(float* z, const float* eps, int64_t n, float sigma) {
    const int64_t n4 = n >> 2;
    const int64_t stride = (int64_t)gridDim.x * kEulerThreads;
    const int64_t tid = (int64_t)blockIdx.x * kEulerThreads + threadIdx.x;
    for (int64_t i = tid; i < n4; i += stride) {
        float4 e = reinterpret_cast<const float4*>(eps)[i];
        e.x *= sigma; e.y *= sigma; e.z *= sigma; e.w *= sigma;
        reinterpret_cast<float4*>(z)[i] = e;
    }
    for (int64_t i = (n4 << 2) + tid; i < n; i += stride) z[i] = sigma * eps[i];
}

// ---------------------------------------------------------------------------
// Interleaved 2-D RoPE of the vision tower ([U15] §Vision tower): channels
// [0, C/2) turn with the patch column, [C/2, C) with the patch row, pairs
// (2i, 2i+1) share the angle pos * theta^(-2i/(C/2)).
//
// A thread owns one 16-byte chunk of channels (8 bf16 or 4 fp32: 4 or 2
// pairs) of a sequence of patches: the `lanes` threads of a token cover its
// chunks with consecutive addresses, a block holds `tpb` tokens, and the
// patches of one thread lie `stride` tokens apart. The chunk's frequencies
// are computed once; a patch's (row, column) advances by (stride / cols,
// stride % cols) with carries, so the loop divides nothing. kRopeU patches
// are in flight per thread.
// ---------------------------------------------------------------------------
template <typename T>
struct Chunk16;   // 16 bytes of channels as floats

template <>
struct Chunk16<__nv_bfloat16> {
    static constexpr int kVec = 8;
    static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&x)[8]) {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
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
struct Chunk16<float> {
    static constexpr int kVec = 4;
    static __device__ __forceinline__ void load(const float* p, float (&x)[4]) {
        const float4 u = *reinterpret_cast<const float4*>(p);
        x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
    }
    static __device__ __forceinline__ void store(float* p, const float (&y)[4]) {
        *reinterpret_cast<float4*>(p) = make_float4(y[0], y[1], y[2], y[3]);
    }
};

constexpr int kRopeThreads = 256;
constexpr int kRopeU = 2;

template <typename T>
__global__ void __launch_bounds__(kRopeThreads)
rope2d_interleaved_kernel(T* __restrict__ x, int64_t n_tokens, int rows, int cols, int C, int lanes, int tpb,
                          float log2_theta) {
    constexpr int kVec = Chunk16<T>::kVec;
    constexpr int kPairs = kVec / 2;
    const int chunks = C / kVec;
    const int d = C / 2;
    const int per_img = rows * cols;
    const int lane = (int)threadIdx.x % lanes;
    const int slot = (int)threadIdx.x / lanes;
    if (slot >= tpb) return;
    const int64_t stride = (int64_t)gridDim.x * tpb;            // tokens between a thread's patches
    const int smod = (int)(stride % per_img);
    const int dr = smod / cols, dc = smod % cols;
    const int64_t tok0 = (int64_t)blockIdx.x * tpb + slot;
    if (tok0 >= n_tokens) return;
    const int t0 = (int)(tok0 % per_img);
    for (int cc = lane; cc < chunks; cc += lanes) {
        const int ch = cc * kVec;
        float fh[kPairs];
        bool by_row[kPairs];
#pragma unroll
        for (int k = 0; k < kPairs; ++k) {
            const int c0 = ch + 2 * k;                           // first channel of the pair
            by_row[k] = c0 >= d;
            const int i = (c0 - (by_row[k] ? d : 0)) >> 1;
            fh[k] = exp2f(-2.0f * (float)i / (float)d * log2_theta);
        }
        int r = t0 / cols, c = t0 % cols;
        for (int64_t tok = tok0; tok < n_tokens; tok += (int64_t)kRopeU * stride) {
            float v[kRopeU][kVec];
#pragma unroll
            for (int u = 0; u < kRopeU; ++u) {
                const int64_t t = tok + (int64_t)u * stride;
                if (t < n_tokens) Chunk16<T>::load(x + t * C + ch, v[u]);
            }
#pragma unroll
            for (int u = 0; u < kRopeU; ++u) {
                const int64_t t = tok + (int64_t)u * stride;
                if (t < n_tokens) {
                    float o[kVec];
#pragma unroll
                    for (int k = 0; k < kPairs; ++k) {
                        float sn, cs;
                        neo::rope_sincos_small((float)(by_row[k] ? r : c), fh[k], &sn, &cs);
                        o[2 * k] = fmaf(v[u][2 * k], cs, -v[u][2 * k + 1] * sn);
                        o[2 * k + 1] = fmaf(v[u][2 * k + 1], cs, v[u][2 * k] * sn);
                    }
                    Chunk16<T>::store(x + t * C + ch, o);
                }
                // The next patch of this thread: (r, c) + (dr, dc) within its image.
                c += dc;
                if (c >= cols) {
                    c -= cols;
                    ++r;
                }
                r += dr;
                if (r >= rows) r -= rows;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Prefix-cache write ([U15] "Mixture of Transformers" item 1: the
// understanding pass writes a KV cache; [U1] section 4.4: the prefix cache in
// the [B, S, H, D] form the attention reads, here packed without padding).
// Sequence b's rows of the output are its old rows followed by the first n_b
// rows of its chunk. CTA (x, b) copies every gridDim.x-th row of sequence b
// in 16-byte units; b's output offset is cu_old[b] plus the chunk rows of the
// sequences before it, summed by the CTA (which also checks them).
// ---------------------------------------------------------------------------
constexpr int kCacheThreads = 128;

__global__ void __launch_bounds__(kCacheThreads)
write_prefix_cache_kernel(const uint4* __restrict__ k_old, const uint4* __restrict__ v_old,
                          const int32_t* __restrict__ cu_old, int64_t total_old, const uint4* __restrict__ k_new,
                          const uint4* __restrict__ v_new, const int32_t* __restrict__ n_new, int N, int row_u4,
                          uint4* __restrict__ k_out, uint4* __restrict__ v_out, int32_t* __restrict__ cu_out,
                          int64_t capacity, bool in_place) {
    __shared__ long long red_sum[kCacheThreads / 32];
    __shared__ int red_bad[kCacheThreads / 32];
    const int b = blockIdx.y;
    const int lo = cu_old[b], hi = cu_old[b + 1];
    const int n = n_new ? n_new[b] : N;
    long long before = 0;
    int bad = 0;
    for (int i = threadIdx.x; i < b; i += kCacheThreads) {
        const int ni = n_new ? n_new[i] : N;
        bad |= ni < 0 || ni > N;
        before += ni;
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        before += __shfl_xor_sync(0xffffffffu, before, m);
        bad |= __shfl_xor_sync(0xffffffffu, bad, m);
    }
    if ((threadIdx.x & 31) == 0) {
        red_sum[threadIdx.x >> 5] = before;
        red_bad[threadIdx.x >> 5] = bad;
    }
    __syncthreads();
    before = 0;
    bad = 0;
#pragma unroll
    for (int w = 0; w < kCacheThreads / 32; ++w) {
        before += red_sum[w];
        bad |= red_bad[w];
    }
    const int64_t base = (int64_t)lo + before;
    const int64_t old_rows = (int64_t)hi - lo;
    const int64_t rows = old_rows + n;
    if (bad || cu_old[0] != 0 || lo < 0 || hi < lo || hi > total_old || n < 0 || n > N || base + rows > capacity) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(&g_elem_error, NEO_DEVERR_BAD_PREFIX);
        return;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        cu_out[b + 1] = (int32_t)(base + rows);
        if (b == 0) cu_out[0] = 0;
    }
    for (int64_t r = in_place ? old_rows + blockIdx.x : blockIdx.x; r < rows; r += gridDim.x) {
        const bool old = r < old_rows;
        const int64_t src = old ? (int64_t)lo + r : ((int64_t)b * N + (r - old_rows));
        const uint4* ks = (old ? k_old : k_new) + src * row_u4;
        const uint4* vs = (old ? v_old : v_new) + src * row_u4;
        uint4* kd = k_out + (base + r) * row_u4;
        uint4* vd = v_out + (base + r) * row_u4;
        for (int c = threadIdx.x; c < row_u4; c += kCacheThreads) {
            kd[c] = ks[c];
            vd[c] = vs[c];
        }
    }
}

}  // namespace

namespace neo {

neo_status elementwise_error_read_clear(uint32_t* word) {
    unsigned int h = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&h, g_elem_error, sizeof(h)) != cudaSuccess) return NEO_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_elem_error, &zero, sizeof(zero)) != cudaSuccess) return NEO_ERR_CUDA;
    *word = h;
    return NEO_OK;
}

neo_status elementwise_set_timeout(uint64_t ns) {
    unsigned long long v = ns;
    return cudaMemcpyToSymbol(g_elem_wait_limit_ns, &v, sizeof(v)) == cudaSuccess ? NEO_OK : NEO_ERR_CUDA;
}

}  // namespace neo

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
    const int64_t esz = dtype == NEO_BF16 ? 2 : 4;
    if (Hq > 0 && Hkv > 0 && neo::overlap(q, S * Hq * 128 * esz, k, S * Hkv * 128 * esz)) return NEO_ERR_INVALID_ARG;

    const RopeFreqs fr = neo::rope3_freqs(theta_t, theta_hw);
    const int64_t blocks = (S + kNormWarps - 1) / kNormWarps;
    if (blocks > INT32_MAX) return NEO_ERR_UNSUPPORTED;
    const dim3 grid((unsigned)blocks, (Hq > 0 ? 1u : 0u) + (Hkv > 0 ? 1u : 0u));
    const size_t ring = (size_t)kNormWarps * kNormDepth * kNormChunkRows * 128 * (dtype == NEO_BF16 ? 2 : 4);
    static neo::DeviceOnce attr_slots[neo::kMaxDevices];
    neo::DeviceOnce* attr = neo::device_slot(attr_slots);
    if (!attr) return NEO_ERR_CUDA;
    std::call_once(attr->once, [attr] {
        const int bytes = 96 * 1024;
        attr->err = cudaFuncSetAttribute(qknorm_rope3_kernel<__nv_bfloat16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (attr->err == cudaSuccess)
            attr->err = cudaFuncSetAttribute(qknorm_rope3_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             bytes);
    });
    if (attr->err != cudaSuccess) return NEO_ERR_CUDA;
    if (dtype == NEO_BF16) {
        qknorm_rope3_kernel<__nv_bfloat16><<<grid, kNormWarps * 32, ring, stream>>>(
            static_cast<__nv_bfloat16*>(q), static_cast<__nv_bfloat16*>(k), S, Hq, Hkv, indexes, q_norm_w,
            q_norm_hw_w, k_norm_w, k_norm_hw_w, fr, eps);
    } else {
        qknorm_rope3_kernel<float><<<grid, kNormWarps * 32, ring, stream>>>(
            static_cast<float*>(q), static_cast<float*>(k), S, Hq, Hkv, indexes, q_norm_w, q_norm_hw_w,
            k_norm_w, k_norm_hw_w, fr, eps);
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
    // The kernel reads z and x0_hat once and writes z and v_out: no overlaps.
    const int64_t nb = n * 4;
    if (neo::overlap(z, nb, x0_hat, nb) || neo::overlap(v_out, nb, z, nb) || neo::overlap(v_out, nb, x0_hat, nb))
        return NEO_ERR_INVALID_ARG;
    const float den = std::fmax(1.0f - t, t_eps);
    if (!(den > 0.f)) return NEO_ERR_INVALID_ARG;
    const float dt = t_next - t;
    const int64_t n4 = (n + 3) / 4;
    const int64_t want = (n4 + kEulerThreads * kEulerUnroll - 1) / (kEulerThreads * kEulerUnroll);
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sm_count() * 8));
    flow_euler_kernel<<<(unsigned)blocks, kEulerThreads, 0, stream>>>(z, x0_hat, n, den, dt, v_out);
    return neo::launch_status();
}

extern "C" neo_status neo_flow_cfg_euler_step(float* z, const float* x0_cond, const float* x0_text_uncond,
                                              const float* x0_uncond, int64_t n, float t, float t_next,
                                              float t_eps, float cfg_scale, float img_cfg_scale,
                                              float cfg_interval_lo, float cfg_interval_hi, float* v_out,
                                              int32_t* branch_out, cudaStream_t stream) {
    if (n < 0 || !std::isfinite(t) || !std::isfinite(t_next) || !std::isfinite(t_eps) ||
        !std::isfinite(cfg_scale) || !std::isfinite(img_cfg_scale) || !std::isfinite(cfg_interval_lo) ||
        !std::isfinite(cfg_interval_hi))
        return NEO_ERR_INVALID_ARG;
    // Branch of the inference loop ([U1] section 2.7).
    const bool use_cfg = (t > cfg_interval_lo && t < cfg_interval_hi) || cfg_interval_lo == 0.0f;
    int branch;
    if (!use_cfg || (cfg_scale == 1.0f && img_cfg_scale == 1.0f)) branch = NEO_CFG_NONE;
    else if (img_cfg_scale == 1.0f) branch = NEO_CFG_TEXT;
    else if (cfg_scale == img_cfg_scale) branch = NEO_CFG_CLASSIC;
    else branch = NEO_CFG_DUAL;
    if (branch_out) *branch_out = branch;
    // Weights on (cond, text-uncond, uncond); each row sums to one.
    const float* xa = x0_cond;
    const float* xb = nullptr;
    const float* xc = nullptr;
    float wa = 1.f, wb = 0.f, wc = 0.f;
    int K = 1;
    if (branch == NEO_CFG_TEXT) {
        xb = x0_text_uncond; wa = cfg_scale; wb = 1.f - cfg_scale; K = 2;
    } else if (branch == NEO_CFG_CLASSIC) {
        xb = x0_uncond; wa = cfg_scale; wb = 1.f - cfg_scale; K = 2;
    } else if (branch == NEO_CFG_DUAL) {
        xb = x0_text_uncond; xc = x0_uncond;
        wa = cfg_scale; wb = img_cfg_scale - cfg_scale; wc = 1.f - img_cfg_scale; K = 3;
    }
    if (n == 0) return NEO_OK;
    if (!z || !xa || (K > 1 && !xb) || (K > 2 && !xc)) return NEO_ERR_INVALID_ARG;
    if (!neo::aligned16(z) || !neo::aligned16(xa) || (xb && !neo::aligned16(xb)) || (xc && !neo::aligned16(xc)) ||
        (v_out && !neo::aligned16(v_out)))
        return NEO_ERR_INVALID_ARG;
    // Predictions are only read and may share a buffer; z and v_out are
    // written, so neither may overlap anything the kernel reads, nor each other.
    {
        const int64_t nb = n * 4;
        const void* reads[3] = {xa, K > 1 ? xb : nullptr, K > 2 ? xc : nullptr};
        for (const void* r : reads)
            if (neo::overlap(z, nb, r, nb) || neo::overlap(v_out, nb, r, nb)) return NEO_ERR_INVALID_ARG;
        if (neo::overlap(v_out, nb, z, nb)) return NEO_ERR_INVALID_ARG;
    }
    const float den = std::fmax(1.0f - t, t_eps);
    if (!(den > 0.f)) return NEO_ERR_INVALID_ARG;
    const float dt = t_next - t;
    const int64_t n4 = (n + 3) / 4;
    const int64_t want = (n4 + kEulerThreads * 2 - 1) / (kEulerThreads * 2);
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sm_count() * 8));
    if (K == 1)
        flow_cfg_kernel<1><<<(unsigned)blocks, kEulerThreads, 0, stream>>>(z, xa, xa, xa, n, wa, wb, wc, den, dt, v_out);
    else if (K == 2)
        flow_cfg_kernel<2><<<(unsigned)blocks, kEulerThreads, 0, stream>>>(z, xa, xb, xb, n, wa, wb, wc, den, dt, v_out);
    else
        flow_cfg_kernel<3><<<(unsigned)blocks, kEulerThreads, 0, stream>>>(z, xa, xb, xc, n, wa, wb, wc, den, dt, v_out);
    return neo::launch_status();
}

extern "C" neo_status neo_scale_noise(float* z, const float* eps, int64_t n, float sigma, cudaStream_t stream) {
    if (n < 0 || !std::isfinite(sigma)) return NEO_ERR_INVALID_ARG;
    if (n == 0) return NEO_OK;
    if (!z || !eps || !neo::aligned16(z) || !neo::aligned16(eps)) return NEO_ERR_INVALID_ARG;
    const int64_t n4 = (n + 3) / 4;
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((n4 + kEulerThreads - 1) / kEulerThreads,
                                                                  (int64_t)sm_count() * 8));
    scale_noise_kernel<<<(unsigned)blocks, kEulerThreads, 0, stream>>>(z, eps, n, sigma);
    return neo::launch_status();
}

extern "C" neo_status neo_rope2d_interleaved(void* x, neo_dtype dtype, int64_t n_images, int rows, int cols, int C,
                                             float theta, cudaStream_t stream) {
    if (n_images < 0 || rows < 0 || cols < 0 || C < 4 || C % 4 != 0 || !(theta > 0.f) || !std::isfinite(theta))
        return NEO_ERR_INVALID_ARG;
    if (dtype != NEO_BF16 && dtype != NEO_F32) return NEO_ERR_INVALID_ARG;
    const int64_t n_tokens = n_images * rows * cols;
    if (n_tokens == 0) return NEO_OK;
    if (!x || !neo::aligned16(x) || (dtype == NEO_BF16 && C % 8 != 0)) return NEO_ERR_INVALID_ARG;
    const float log2_theta = (float)std::log2((double)theta);
    if ((int64_t)rows * cols > 0x7fffffffLL) return NEO_ERR_UNSUPPORTED;
    // Threads of a token: one per 16-byte chunk, at most a block's worth.
    const int chunks = C / (dtype == NEO_BF16 ? 8 : 4);
    const int lanes = std::min(chunks, kRopeThreads);
    const int tpb = kRopeThreads / lanes;                      // tokens a block holds
    // One resident wave of 4 blocks an SM (measured best at the 128 x 128 x 1024
    // patch grid against 2-16 blocks an SM and 1-8 patches in flight).
    const int64_t want = (n_tokens + (int64_t)tpb * kRopeU - 1) / ((int64_t)tpb * kRopeU);
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sm_count() * 4));
    if (dtype == NEO_BF16)
        rope2d_interleaved_kernel<__nv_bfloat16><<<(unsigned)blocks, lanes * tpb, 0, stream>>>(
            static_cast<__nv_bfloat16*>(x), n_tokens, rows, cols, C, lanes, tpb, log2_theta);
    else
        rope2d_interleaved_kernel<float><<<(unsigned)blocks, lanes * tpb, 0, stream>>>(
            static_cast<float*>(x), n_tokens, rows, cols, C, lanes, tpb, log2_theta);
    return neo::launch_status();
}

extern "C" neo_status neo_write_prefix_cache(const void* k_old, const void* v_old, const int32_t* cu_old,
                                             int64_t total_old, const void* k_new, const void* v_new,
                                             const int32_t* n_new, int B, int N, int Hkv, int D, neo_dtype dtype,
                                             void* k_out, void* v_out, int32_t* cu_out, int64_t capacity,
                                             cudaStream_t stream) {
    if (D != 128 || B < 1 || N < 0 || Hkv < 1 || total_old < 0 || capacity < 0) return NEO_ERR_INVALID_ARG;
    if (dtype != NEO_BF16 && dtype != NEO_F32) return NEO_ERR_INVALID_ARG;
    if (!cu_old || !cu_out || !k_out || !v_out) return NEO_ERR_INVALID_ARG;
    if (total_old > 0 && (!k_old || !v_old)) return NEO_ERR_INVALID_ARG;
    if (N > 0 && (!k_new || !v_new)) return NEO_ERR_INVALID_ARG;
    if (B > 65535 || capacity > 0x7fffffffLL || total_old > capacity) return NEO_ERR_UNSUPPORTED;
    const void* ptrs[6] = {k_old, v_old, k_new, v_new, k_out, v_out};
    for (const void* q : ptrs)
        if (q && !neo::aligned16(q)) return NEO_ERR_INVALID_ARG;
    const int64_t row = (int64_t)Hkv * D * (dtype == NEO_BF16 ? 2 : 4);   // bytes per cache row
    // The outputs may not overlap any input, except the in-place append of a
    // single sequence (k_out == k_old and v_out == v_old).
    const bool in_place = B == 1 && k_out == k_old && v_out == v_old && total_old > 0;
    using neo::overlap;
    const int64_t out_bytes = capacity * row, old_bytes = total_old * row, new_bytes = (int64_t)B * N * row;
    const void* outs[2] = {k_out, v_out};
    for (const void* o : outs) {
        if (!in_place && (overlap(o, out_bytes, k_old, old_bytes) || overlap(o, out_bytes, v_old, old_bytes)))
            return NEO_ERR_INVALID_ARG;
        if (overlap(o, out_bytes, k_new, new_bytes) || overlap(o, out_bytes, v_new, new_bytes)) return NEO_ERR_INVALID_ARG;
    }
    if (overlap(k_out, out_bytes, v_out, out_bytes)) return NEO_ERR_INVALID_ARG;
    if (in_place && (overlap(k_out, out_bytes, v_old, old_bytes) || overlap(v_out, out_bytes, k_old, old_bytes)))
        return NEO_ERR_INVALID_ARG;
    const int64_t want = ((int64_t)sm_count() * 8 + B - 1) / B;
    const unsigned gx = (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, 4096));
    write_prefix_cache_kernel<<<dim3(gx, (unsigned)B), kCacheThreads, 0, stream>>>(
        static_cast<const uint4*>(k_old), static_cast<const uint4*>(v_old), cu_old, total_old,
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), n_new, N, (int)(row / 16),
        static_cast<uint4*>(k_out), static_cast<uint4*>(v_out), cu_out, capacity, in_place);
    return neo::launch_status();
}

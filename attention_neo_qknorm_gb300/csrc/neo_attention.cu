// Generation-pass attention of NEO-unify on tcgen05 tensor cores.
//
// What it computes ("SenseNova-U1.5 (NEO-unify) architecture", sections
// "Mixture of Transformers" items 1-2 and "GQA fusion does not apply"): every
// noisy image token's query attends, without a mask, over the frozen prefix
// keys/values of its own sequence followed by the image tokens' own
// keys/values; query head h reads KV head h / (Hq/Hkv). The same kernel also
// applies the block-causal mask of the mixed prefill (section "Block-causal
// attention"): key j visible to query i iff T_j == T_i or j <= i.
//
// Two kernels share the roles below. gen_attention_persistent_kernel (the
// full mask, with or without the query norm folded in, and the block-causal
// mask of a single sequence) keeps one cluster per pair of SMs resident and
// walks it through a sequence of query-tile pairs, so one pair's epilogue
// overlaps the next pair's first tiles (its own comment, further down, gives
// the hand-over). gen_attention_kernel (the block-causal mask of several
// sequences, or of one with the folded query norm) runs one query tile per
// CTA.
//
// Kernel shape (one CTA per 128-row query tile; D = 128; 12 warps; clusters
// of two CTAs):
//   * A query tile packs the G = Hq/Hkv heads of one KV group for 128/G
//     consecutive tokens (row r = token * G + head-in-group), so each K/V tile
//     brought into shared memory serves the whole GQA group.
//   * Warp 0 (one lane) loads Q once and streams K tiles of 128 keys through
//     a three-stage TMA ring; warp 2 (one lane) streams the V tiles through a
//     two-stage ring (128-byte swizzle). The two CTAs of a cluster work on
//     neighbouring query tiles of the same sequence and KV head: each fetches
//     one 64-wide head-dim half of every K/V tile and multicasts it into both.
//     Prefix tiles come first (from the packed prefix, ceil(L_b/128) of
//     them), then the image tiles; keys past a segment's end are masked, so
//     ragged prefixes need no padding.
//   * Warp 1 (one lane) issues the tcgen05.mma batches of S = Q K^T (Q and K
//     K-major in shared memory, fp32 accumulator in TMEM, three buffers);
//     warp 3 (one lane) those of O += P V (P bf16 from TMEM, V MN-major in
//     shared memory, O accumulated in TMEM). Issuing a batch blocks while the
//     tensor pipe's queue is full, so two independent issuers keep it fed
//     while either one waits on a barrier.
//   * Warps 4..11 run the online softmax in fp32. Query row r is TMEM lane r.
//     Warps w and w + 4 share the lanes of sub-partition w & 3 and each owns
//     16 whole rows of it, loaded with the 16-lane tcgen05.ld shape: a thread
//     holds two rows (r, r + 8) and 32 of their 128 key columns, so a row's
//     maximum is reduced over four threads of one warp with two shuffles and
//     the two warps of a sub-partition never wait for each other within a
//     unit. Each thread keeps partial row sums until the end. exp2 runs on
//     the SFU; P_j goes to TMEM as bf16 (16x128b stores, whose layout is the
//     packed form of the 16x256b load's) over the rows' own first 64 columns
//     of the S buffer it came from, so S_j reuses a buffer only once PV_{j-3}
//     has read it and the softmax never waits for PV. O is rescaled only when
//     the running maximum grew by more than 2^8 (the final division uses the
//     same stale maximum, so the result is unchanged). The epilogue reads O
//     one row a thread, each warp a 64-wide half of the columns of all 32
//     rows (sums and maxima through shared memory), and writes O / l as bf16
//     through shared memory and a TMA store.
// TMEM: S0 [0,128) S1 [128,256) S2 [256,384) O [384,512).

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "neo.h"
#include "neo_internal.h"
#include "neo_rope.cuh"
#include "sm103_ptx.cuh"

using namespace sm103;

namespace {

__device__ unsigned int g_dev_error = 0;
__device__ unsigned long long g_wait_limit_ns = 1000000000ull;

constexpr int kThreads = 384;
constexpr int kCluster = 2;                  // CTAs per cluster sharing each K/V tile
constexpr uint16_t kClusterMask = (1u << kCluster) - 1u;
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kSBufs = 3;                   // S (and P, written over S) buffers in TMEM
constexpr uint32_t kHalfTile = 128u * 64u * 2u;   // 128 rows x 64 bf16 (one 128-byte swizzle span)
constexpr uint32_t kTile = 2u * kHalfTile;         // 128 rows x 128 bf16

constexpr uint32_t kSmQ = 0;
constexpr uint32_t kSmK = kSmQ + kTile;
constexpr uint32_t kSmV = kSmK + kKStages * kTile;
constexpr uint32_t kSmMax = kSmV + kVStages * kTile;   // float [128 rows]: the rows' running maxima
constexpr uint32_t kSmLsum = kSmMax + 128 * 4;         // float [128 rows]: the rows' sums
constexpr uint32_t kSmBar = kSmLsum + 128 * 4;

enum : int {
    BAR_Q_FULL = 0,
    BAR_K_FULL = 1,
    BAR_K_EMPTY = BAR_K_FULL + kKStages,
    BAR_V_FULL = BAR_K_EMPTY + kKStages,
    BAR_V_EMPTY = BAR_V_FULL + kVStages,
    BAR_S_FULL = BAR_V_EMPTY + kVStages,
    BAR_P_FULL = BAR_S_FULL + kSBufs,
    BAR_PV_DONE = BAR_P_FULL + kSBufs,
    BAR_DRAIN = BAR_PV_DONE + kSBufs,
    BAR_Q_READY = BAR_DRAIN + 1,   // folded query norm/RoPE done (one arrival per softmax thread)
    NUM_BARS = BAR_Q_READY + 1
};

constexpr uint32_t kSmTmemSlot = kSmBar + NUM_BARS * 8;
constexpr uint32_t kSmAbort = kSmTmemSlot + 4;
constexpr uint32_t kSmEpiSkip = kSmAbort + 4;   // written only by the softmax warps
// Block-causal mode: the queries' temporal-index range, the image tiles past
// the diagonal that are kept (bitmask, then compacted into a list), their
// count, and the [min, max] temporal index of each 64-key half of every image
// tile from the cluster's first query tile on.
constexpr int kMaxImgTiles = 1024;                 // image segment of at most 131072 tokens
constexpr uint32_t kSmTRange = kSmEpiSkip + 4;     // int [2]
constexpr uint32_t kSmNExtra = kSmTRange + 8;
constexpr uint32_t kSmTileBits = kSmNExtra + 4;    // uint32 [kMaxImgTiles / 32]
constexpr uint32_t kSmTileList = kSmTileBits + kMaxImgTiles / 8;   // uint16 [kMaxImgTiles]
constexpr uint32_t kSmTileT = (kSmTileList + kMaxImgTiles * 2 + 15u) & ~15u;   // int4 [kMaxImgTiles]: min0 max0 min1 max1
constexpr uint32_t kSmQnW = kSmTileT + kMaxImgTiles * 16;   // float [128]: folded query norm weights
constexpr uint32_t kSmUsed = kSmQnW + 128 * 4;
static_assert(kSmTileT % 16 == 0, "int4 entries need 16-byte alignment");
constexpr uint32_t kSmemBytes = kSmUsed + 1024;    // slack to align the base to 1024 bytes
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB of shared memory a CTA may use");

constexpr uint32_t kTmS0 = 0, kTmO = kSBufs * 128, kTmCols = 512;
constexpr int kSoftmaxThreads = 256;               // warps 4..11

constexpr uint32_t kIdescS = idesc_bf16_f32(kBlockM, kBlockN, 0, 0);   // Q, K both K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(kBlockM, 128, 0, 1);      // V is MN-major

constexpr float kRescaleThreshold = 8.0f;   // log2 units

struct AttnParams {
    const int32_t* cu_prefix;
    const int32_t* t_prefix;   // block-causal mode: temporal index of every packed prefix row
    const int32_t* t_img;      // block-causal mode: temporal index of every image token [B*N]
    int mask_mode;
    float* lse;
    int64_t total_prefix;
    int B, N, Hq, Hkv, G, tok_per_tile, max_prefix;
    float scale_log2;
    // Folded query norm + RoPE (null qn_idx: the queries arrive normalised).
    const int32_t* qn_idx;     // [3, B*N] positions of the image tokens
    const float* qn_w_t;       // [64] weights of dims [0,64)
    const float* qn_w_hw;      // [64] weights of dims [64,128)
    float qn_eps;
};

__device__ __forceinline__ uint32_t bar_addr(uint32_t sbase, int i) { return sbase + kSmBar + 8u * i; }

// Query norm on halves + three-axis RoPE of one 64-dim half of one Q row in
// shared memory ("Three rotary axes"), in place. The tile is 128-byte swizzled:
// 16-byte chunk c of row r sits at r * 128 + ((c ^ (r & 7)) << 4) of its half.
// Half 0 holds the temporal slice, rotation pairs (i, i+32) = chunks (c, c+4);
// half 1 the height slice, pairs (i, i+16) = chunks (0,2), (1,3), and the
// width slice, chunks (4,6), (5,7). The four chunk pairs are taken in the
// order, and with the arithmetic (fp32x2 sums of squares combined as
// (s0 + s1) + (s2 + s3), norm weights folded into cos/sin), of the standalone
// norm/RoPE kernel's bf16 path, so the normalised query has the same bits.
// The 32 (cos, sin) of one 64-dim half of a row, in the lane-partial order
// below (chunk pair s, element pair j -> index 8 s + j). They depend only on
// the token's positions, so they are computed while the Q tile is in flight.
template <int half>
__device__ __forceinline__ void qnorm_rope_angles(const int32_t pos[3], const neo::RopeFreqs& fr, float (&cs)[32],
                                                  float (&sn)[32]) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const int pair0 = half ? (s < 2 ? 32 + 8 * s : 48 + 8 * (s - 2)) : 8 * s;
        const int32_t p_s = pos[half ? (s < 2 ? 1 : 2) : 0];
#pragma unroll
        for (int j = 0; j < 8; ++j) neo::rope_sincos(p_s, fr.turn[pair0 + j], &sn[8 * s + j], &cs[8 * s + j]);
    }
}

// Query norm on halves + three-axis RoPE of one 64-dim half of one Q row in
// shared memory ("Three rotary axes"), in place. The tile is 128-byte swizzled:
// 16-byte chunk c of row r sits at r * 128 + ((c ^ (r & 7)) << 4) of its half.
// Half 0 holds the temporal slice, rotation pairs (i, i+32) = chunks (c, c+4);
// half 1 the height slice, pairs (i, i+16) = chunks (0,2), (1,3), and the
// width slice, chunks (4,6), (5,7). The four chunk pairs are taken in the
// order, and with the arithmetic (fp32x2 sums of squares combined as
// (s0 + s1) + (s2 + s3), norm weights folded into cos/sin), of the standalone
// norm/RoPE kernel's bf16 path, so the normalised query has the same bits.
// w: this half's 64 weights (shared memory).
template <int half>
__device__ __forceinline__ void qnorm_rope_q_half(uint8_t* half_tile, int row, const float (&cs)[32],
                                                  const float (&sn)[32], const float* w, float eps) {
    uint8_t* rowp = half_tile + row * 128;
    uint4 raw[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) raw[c] = *reinterpret_cast<const uint4*>(rowp + ((c ^ (row & 7)) << 4));
    auto unpack = [](uint4 u, float2 (&x)[4]) {
        const uint32_t v[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = make_float2(__uint_as_float(v[i] << 16), __uint_as_float(v[i] & 0xffff0000u));
    };
    // chunk pairs (a, b) of this half, in lane-partial order
    constexpr int pa[4] = {0, 1, half ? 4 : 2, half ? 5 : 3};
    constexpr int pb[4] = {half ? 2 : 4, half ? 3 : 5, 6, 7};
    float part[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        float2 xa[4], xb[4];
        unpack(raw[pa[s]], xa);
        unpack(raw[pb[s]], xb);
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc = ffma2(xa[i], xa[i], ffma2(xb[i], xb[i], acc));
        part[s] = acc.x + acc.y;
    }
    const float ss = (part[0] + part[1]) + (part[2] + part[3]);
    const float rs = rsqrtf(ss * (1.0f / 64.0f) + eps);
    const float2 rs2 = make_float2(rs, rs);
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const float4* wa4 = reinterpret_cast<const float4*>(w + 8 * pa[s]);
        const float4* wb4 = reinterpret_cast<const float4*>(w + 8 * pb[s]);
        const float4 wa_lo = wa4[0], wa_hi = wa4[1], wb_lo = wb4[0], wb_hi = wb4[1];
        const float wa[8] = {wa_lo.x, wa_lo.y, wa_lo.z, wa_lo.w, wa_hi.x, wa_hi.y, wa_hi.z, wa_hi.w};
        const float wb[8] = {wb_lo.x, wb_lo.y, wb_lo.z, wb_lo.w, wb_hi.x, wb_hi.y, wb_hi.z, wb_hi.w};
        float2 xa[4], xb[4];
        unpack(raw[pa[s]], xa);
        unpack(raw[pb[s]], xb);
        uint32_t oa[4], ob[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = 8 * s + 2 * i;
            const float2 uc = make_float2(wa[2 * i] * cs[e], wa[2 * i + 1] * cs[e + 1]);
            const float2 vs = make_float2(-wb[2 * i] * sn[e], -wb[2 * i + 1] * sn[e + 1]);
            const float2 vc = make_float2(wb[2 * i] * cs[e], wb[2 * i + 1] * cs[e + 1]);
            const float2 us = make_float2(wa[2 * i] * sn[e], wa[2 * i + 1] * sn[e + 1]);
            const float2 u = fmul2(xa[i], rs2), v = fmul2(xb[i], rs2);
            const float2 ya = ffma2(u, uc, fmul2(v, vs));
            const float2 yb = ffma2(v, vc, fmul2(u, us));
            oa[i] = pack_bf16x2(ya.x, ya.y);
            ob[i] = pack_bf16x2(yb.x, yb.y);
        }
        *reinterpret_cast<uint4*>(rowp + ((pa[s] ^ (row & 7)) << 4)) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
        *reinterpret_cast<uint4*>(rowp + ((pb[s] ^ (row & 7)) << 4)) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
    }
}

// As qnorm_rope_angles + qnorm_rope_q_half, with each chunk pair's eight
// (cos, sin) computed where they are used instead of all 32 up front, and the
// row's chunks read again from shared memory for the rotation instead of kept
// in registers: the same calls and operations on the same values (hence the
// same bits) in fewer registers.
template <int half>
__device__ __forceinline__ void qnorm_rope_q_half_lowreg(uint8_t* half_tile, int row, const int32_t pos[3],
                                                         const neo::RopeFreqs& fr, const float* w, float eps) {
    uint8_t* rowp = half_tile + row * 128;
    auto chunk = [&](int c) { return *reinterpret_cast<const uint4*>(rowp + ((c ^ (row & 7)) << 4)); };
    auto unpack = [](uint4 u, float2 (&x)[4]) {
        const uint32_t v[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = make_float2(__uint_as_float(v[i] << 16), __uint_as_float(v[i] & 0xffff0000u));
    };
    constexpr int pa[4] = {0, 1, half ? 4 : 2, half ? 5 : 3};
    constexpr int pb[4] = {half ? 2 : 4, half ? 3 : 5, 6, 7};
    float part[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        float2 xa[4], xb[4];
        unpack(chunk(pa[s]), xa);
        unpack(chunk(pb[s]), xb);
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc = ffma2(xa[i], xa[i], ffma2(xb[i], xb[i], acc));
        part[s] = acc.x + acc.y;
    }
    const float ss = (part[0] + part[1]) + (part[2] + part[3]);
    const float rs = rsqrtf(ss * (1.0f / 64.0f) + eps);
    const float2 rs2 = make_float2(rs, rs);
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const int pair0 = half ? (s < 2 ? 32 + 8 * s : 48 + 8 * (s - 2)) : 8 * s;
        const int32_t p_s = pos[half ? (s < 2 ? 1 : 2) : 0];
        float cs[8], sn[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) neo::rope_sincos(p_s, fr.turn[pair0 + j], &sn[j], &cs[j]);
        float2 xa[4], xb[4];
        unpack(chunk(pa[s]), xa);   // not yet written: chunk pairs are disjoint
        unpack(chunk(pb[s]), xb);
        uint32_t oa[4], ob[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 wa = *reinterpret_cast<const float2*>(w + 8 * pa[s] + 2 * i);
            const float2 wb = *reinterpret_cast<const float2*>(w + 8 * pb[s] + 2 * i);
            const int e = 2 * i;
            const float2 uc = make_float2(wa.x * cs[e], wa.y * cs[e + 1]);
            const float2 vs = make_float2(-wb.x * sn[e], -wb.y * sn[e + 1]);
            const float2 vc = make_float2(wb.x * cs[e], wb.y * cs[e + 1]);
            const float2 us = make_float2(wa.x * sn[e], wa.y * sn[e + 1]);
            const float2 u = fmul2(xa[i], rs2), v = fmul2(xb[i], rs2);
            const float2 ya = ffma2(u, uc, fmul2(v, vs));
            const float2 yb = ffma2(v, vc, fmul2(u, us));
            oa[i] = pack_bf16x2(ya.x, ya.y);
            ob[i] = pack_bf16x2(yb.x, yb.y);
        }
        *reinterpret_cast<uint4*>(rowp + ((pa[s] ^ (row & 7)) << 4)) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
        *reinterpret_cast<uint4*>(rowp + ((pb[s] ^ (row & 7)) << 4)) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
    }
}

// max of 32 values: three-input max tree (11, 4, 1).
__device__ __forceinline__ float max32(const float (&v)[32]) {
    float t[11];
#pragma unroll
    for (int i = 0; i < 10; ++i) t[i] = fmax3(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
    t[10] = fmaxf(v[30], v[31]);
    const float u0 = fmax3(t[0], t[1], t[2]), u1 = fmax3(t[3], t[4], t[5]), u2 = fmax3(t[6], t[7], t[8]);
    return fmaxf(fmax3(u0, u1, u2), fmaxf(t[9], t[10]));
}

// Block-causal mode: the keep bits of one 64-key half of key tile j for one query row
// (bit c: key key0 + c). Key j of [prefix ; image] is visible to query i iff
// T_j == T_i or j <= i ("Block-causal attention"). The row's 64 keys all at or
// before the row or all sharing its index -> nothing to hide beyond the
// segment end; the row's index outside the keys' range -> causal, a
// threshold; otherwise (a block boundary) key by key. i_row = L + the row's
// image token, t_row its temporal index; t_img: the sequence's image tokens.
__device__ __forceinline__ uint64_t bc_keep_half(const int32_t* t_img, const int4* tile_t, int j, int n_pre, int L,
                                                 int it, int half, int valid, int i_row, int t_row) {
    const int key0 = (j < n_pre ? j * kBlockN : L + it * kBlockN) + half * 64;
    uint64_t keep = valid >= 64 ? ~0ull : (valid <= 0 ? 0ull : (1ull << valid) - 1ull);
    if (j >= n_pre && key0 + 63 > i_row) {
        const int4 tr = tile_t[it];
        const int klo = half ? tr.z : tr.x, khi = half ? tr.w : tr.y;
        if (!(klo == t_row && khi == t_row)) {
            const int lim = i_row - key0 + 1;   // columns c < lim are at or before the row
            const uint64_t causal = lim >= 64 ? ~0ull : (lim <= 0 ? 0ull : (1ull << lim) - 1ull);
            if (t_row < klo || t_row > khi) {
                keep &= causal;
            } else {
                const int32_t* tk = t_img + (key0 - L);
                for (int c = max(lim, 0); c < min(valid, 64); ++c)
                    if (__ldg(tk + c) != t_row) keep &= ~(1ull << c);
            }
        }
    }
    return keep;
}

// Block-causal mode, off the tile loop's hot path, for the 16-lane softmax
// layout: the mask of key tile j for this thread's two rows
// (image tokens n_a, n_b), written into S in TMEM (hidden keys become -inf)
// before the softmax loads it; called by a whole warp. taddr: the S buffer
// at the warp's 16 lanes; jq: the thread's column group.
__device__ __noinline__ void bc_mask_s_cold16(uint32_t taddr, const int32_t* t_img, const int4* tile_t, int j,
                                              int n_pre, int L, int it, int tile_valid, int n_a, int n_b, int jq) {
    uint64_t keep[2][2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int n_row = r ? n_b : n_a;
        const int t_row = __ldg(t_img + n_row);
#pragma unroll
        for (int h = 0; h < 2; ++h)
            keep[r][h] = bc_keep_half(t_img, tile_t, j, n_pre, L, it, h, tile_valid - 64 * h, L + n_row, t_row);
    }
    if (!__any_sync(0xffffffffu, (keep[0][0] & keep[0][1] & keep[1][0] & keep[1][1]) != ~0ull)) return;
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t r[32];
        tmem_ld16x256b_x8(taddr + 64u * (uint32_t)h, r);
#pragma unroll
        for (int k = 0; k < 8; ++k)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (!((keep[e >> 1][h] >> (8 * k + 2 * jq + (e & 1))) & 1ull)) r[4 * k + e] = __float_as_uint(-INFINITY);
        tmem_st16x256b_x8(taddr + 64u * (uint32_t)h, r);
    }
    tmem_st_wait();
}

// kQNorm: the query norm + RoPE is folded into the prologue (a separate
// instantiation, so that the plain kernel's code is unchanged by it).
template <bool kBlockCausal, bool kQNorm>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 1)
gen_attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o,
                     const __grid_constant__ CUtensorMap tm_kimg,
                     const __grid_constant__ CUtensorMap tm_vimg,
                     const __grid_constant__ CUtensorMap tm_kpre,
                     const __grid_constant__ CUtensorMap tm_vpre, const __grid_constant__ neo::RopeFreqs qn_freqs,
                     const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_addr(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int qt = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_kpre);
        prefetch_tensormap(&tm_kimg);
        prefetch_tensormap(&tm_vpre);
        prefetch_tensormap(&tm_vimg);
        prefetch_tensormap(&tm_o);
    }

    // Prefix segment of this sequence; an inconsistent cu_prefix skips the CTA.
    const int lo = p.cu_prefix[b];
    const int hi = p.cu_prefix[b + 1];
    const int L = hi - lo;
    if (lo < 0 || L < 0 || (int64_t)hi > p.total_prefix || L > p.max_prefix) {
        if (threadIdx.x == 0) atomicOr(&g_dev_error, NEO_DEVERR_BAD_PREFIX);
        return;
    }
    const int n_pre = (L + kBlockN - 1) / kBlockN;
    const int n_img = (p.N + kBlockN - 1) / kBlockN;
    int n_tiles = n_pre + n_img;
    const int n0 = qt * p.tok_per_tile;

    // Block-causal mode ("Block-causal attention"): image key tile t is needed
    // by the cluster's queries [np0, np1) if it holds a key at or before the
    // last of them (j <= i), or a key whose temporal index lies within the
    // queries' [min, max] range (a superset of T_j == T_i). Tiles past the
    // diagonal that fail the second test are masked for every row and are
    // skipped by all roles; inside every tile kept the per-element mask still
    // decides. Both CTAs of a cluster derive the same list, so they keep
    // sharing one K/V stream.
    [[maybe_unused]] const int np0 = (qt & ~(kCluster - 1)) * p.tok_per_tile;
    [[maybe_unused]] const int np1 = min(p.N, np0 + kCluster * p.tok_per_tile);
    [[maybe_unused]] const int j_diag = (np1 - 1) / kBlockN;
    [[maybe_unused]] const uint16_t* tile_list = reinterpret_cast<const uint16_t*>(smem + kSmTileList);
    // Position u of the image part of the tile sequence -> image tile index.
    auto img_tile = [&](int u) -> int {
        if constexpr (kBlockCausal) return u <= j_diag ? u : (int)tile_list[u - j_diag - 1];
        else return u;
    };

    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmAbort);
    volatile int* epi_skip = reinterpret_cast<volatile int*>(smem + kSmEpiSkip);
    const BoundedWait wait{abort_flag, &g_dev_error, NEO_DEVERR_TIMEOUT, g_wait_limit_ns};

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        *epi_skip = 0;
        for (int i = 0; i < NUM_BARS; ++i) {
            uint32_t count = 1;
            if (i >= BAR_P_FULL && i < BAR_P_FULL + kSBufs)
                count = kSoftmaxThreads;
            if ((i >= BAR_K_EMPTY && i < BAR_K_EMPTY + kKStages) || (i >= BAR_V_EMPTY && i < BAR_V_EMPTY + kVStages))
                count = kCluster;                // released by the MMA of every CTA of the cluster
            if (i == BAR_DRAIN) count = 2;      // one commit from each MMA issuer
            if (i == BAR_Q_READY) count = kSoftmaxThreads;
            mbar_init(bar_addr(sb, i), count);
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(sb + kSmTmemSlot, kTmCols);
        tmem_relinquish();
    }
    if constexpr (kBlockCausal) {
        if (warp == 3) {
            int tmin = INT_MAX, tmax = INT_MIN;
            for (int n = np0 + lane; n < np1; n += 32) {
                const int t = __ldg(p.t_img + (int64_t)b * p.N + n);
                tmin = min(tmin, t);
                tmax = max(tmax, t);
            }
            tmin = __reduce_min_sync(0xffffffffu, tmin);
            tmax = __reduce_max_sync(0xffffffffu, tmax);
            if (lane == 0) {
                reinterpret_cast<int*>(smem + kSmTRange)[0] = tmin;
                reinterpret_cast<int*>(smem + kSmTRange)[1] = tmax;
            }
        } else if (warp >= 4) {
            for (int i = (int)threadIdx.x - 128; i < kMaxImgTiles / 32; i += kThreads - 128)
                reinterpret_cast<uint32_t*>(smem + kSmTileBits)[i] = 0u;
        }
    }
    tc_fence_before();
    __syncthreads();
    // No CTA may multicast into a peer before the peer's barriers exist.
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kSmTmemSlot);
    const uint32_t crank = cluster_ctarank();

    if constexpr (kBlockCausal) {
        // One warp per image tile from the one holding the cluster's first
        // query on: the temporal-index range of each 64-key half, and for tiles
        // past the diagonal whether any key's index lies in the queries' range.
        const int tmin = reinterpret_cast<const int*>(smem + kSmTRange)[0];
        const int tmax = reinterpret_cast<const int*>(smem + kSmTRange)[1];
        uint32_t* bits = reinterpret_cast<uint32_t*>(smem + kSmTileBits);
        int4* tile_t = reinterpret_cast<int4*>(smem + kSmTileT);
        for (int t = np0 / kBlockN + warp; t < n_img; t += kThreads / 32) {
            bool hit = false;
            int lo2[2] = {INT_MAX, INT_MAX}, hi2[2] = {INT_MIN, INT_MIN};
#pragma unroll
            for (int c = 0; c < kBlockN / 32; ++c) {
                const int key = t * kBlockN + c * 32 + lane;
                if (key < p.N) {
                    const int tk = __ldg(p.t_img + (int64_t)b * p.N + key);
                    hit |= tk >= tmin && tk <= tmax;
                    lo2[c >> 1] = min(lo2[c >> 1], tk);
                    hi2[c >> 1] = max(hi2[c >> 1], tk);
                }
            }
            const int4 range = make_int4(__reduce_min_sync(0xffffffffu, lo2[0]), __reduce_max_sync(0xffffffffu, hi2[0]),
                                         __reduce_min_sync(0xffffffffu, lo2[1]), __reduce_max_sync(0xffffffffu, hi2[1]));
            if (lane == 0) tile_t[t] = range;
            if (t > j_diag && __any_sync(0xffffffffu, hit) && lane == 0) atomicOr(bits + (t >> 5), 1u << (t & 31));
        }
        __syncthreads();
        // Compact the kept tiles, in ascending order, into the list.
        if (warp == 0) {
            uint16_t* list = reinterpret_cast<uint16_t*>(smem + kSmTileList);
            const int n_words = (n_img + 31) >> 5;
            int base = 0;
            for (int w0 = (j_diag + 1) >> 5; w0 < n_words; w0 += 32) {
                const int w = w0 + lane;
                uint32_t rem = w < n_words ? bits[w] : 0u;
                const int cnt = __popc(rem);
                int incl = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += v;
                }
                int pos = base + incl - cnt;
                while (rem) {
                    list[pos++] = (uint16_t)(w * 32 + __ffs(rem) - 1);
                    rem &= rem - 1;
                }
                base += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (lane == 0) *reinterpret_cast<int*>(smem + kSmNExtra) = base;
        }
        __syncthreads();
        n_tiles = n_pre + j_diag + 1 + *reinterpret_cast<const int*>(smem + kSmNExtra);
    }

    if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------ producers: K (warp 0) and V (warp 2)
        if (lane == 0) {
            const bool is_k = warp == 0;
            if (is_k) {
                const uint32_t sQ = sb + kSmQ;
                mbar_arrive_expect_tx(bar_addr(sb, BAR_Q_FULL), kTile);
                tma_load_4d(sQ, &tm_q, bar_addr(sb, BAR_Q_FULL), 0, kvh * p.G, n0, b);
                tma_load_4d(sQ + kHalfTile, &tm_q, bar_addr(sb, BAR_Q_FULL), 64, kvh * p.G, n0, b);
            }
            const int stages = is_k ? kKStages : kVStages;
            const int full0 = is_k ? BAR_K_FULL : BAR_V_FULL;
            const int empty0 = is_k ? BAR_K_EMPTY : BAR_V_EMPTY;
            const uint32_t ring = sb + (is_k ? kSmK : kSmV);
            const CUtensorMap* pre_map = is_k ? &tm_kpre : &tm_vpre;
            const CUtensorMap* img_map = is_k ? &tm_kimg : &tm_vimg;
            int issued = 0;
            for (int j = 0; j < n_tiles; ++j) {
                const int st = j % stages;
                const uint32_t ph = (uint32_t)(j / stages) & 1u;
                if (!wait(bar_addr(sb, empty0 + st), ph ^ 1u)) break;
                const uint32_t fb = bar_addr(sb, full0 + st);
                const uint32_t dst = ring + (uint32_t)st * kTile;
                // The tile's two 64-wide head-dim halves come from the two CTAs of
                // the cluster, each multicast into both; every CTA expects the full tile.
                mbar_arrive_expect_tx(fb, kTile);
                const uint32_t hdst = dst + crank * kHalfTile;
                const int d0 = 64 * (int)crank;
                if (j < n_pre) {
                    tma_load_3d_mc(hdst, pre_map, fb, d0, kvh, lo + j * kBlockN, kClusterMask);
                } else {
                    tma_load_4d_mc(hdst, img_map, fb, d0, kvh, img_tile(j - n_pre) * kBlockN, b, kClusterMask);
                }
                issued = j + 1;
            }
            if (*abort_flag) {
                // Let copies already in flight land before the CTA's shared memory goes away.
                if (is_k) wait(bar_addr(sb, BAR_Q_FULL), 0, false);
                for (int j = (issued > stages ? issued - stages : 0); j < issued; ++j)
                    wait(bar_addr(sb, full0 + j % stages), (uint32_t)(j / stages) & 1u, false);
            }
        }
        __syncwarp();
    } else if (warp == 1 || warp == 3) {
        // ------------------------------------------------------------ MMA issuers
        // Warp 1 issues S = Q K^T, warp 3 issues O += P V. Issuing a batch blocks
        // while the tensor pipe's queue is full, so a single issuing thread would
        // leave the pipe idle whenever it waits on a barrier or commits; two
        // independent issuers keep it fed. They write disjoint TMEM (S buffers vs
        // O) and each commits only the barriers of its own product.
        if (lane == 0) {
            bool ok = true;
            if (warp == 1) {
                const uint32_t sQ = sb + kSmQ;
                ok = wait(bar_addr(sb, kQNorm ? BAR_Q_READY : BAR_Q_FULL), 0);
                tc_fence_after();
                for (int j = 0; ok && j < n_tiles; ++j) {
                    const int st = j % kKStages;
                    if (!wait(bar_addr(sb, BAR_K_FULL + st), (uint32_t)(j / kKStages) & 1u)) break;
                    // S buffer j%3 holds P_{j-3} until PV_{j-3} has read it.
                    const int sbuf = j % kSBufs;
                    const uint32_t sph = (uint32_t)(j / kSBufs) & 1u;
                    if (j >= kSBufs && !wait(bar_addr(sb, BAR_PV_DONE + sbuf), sph ^ 1u)) break;
                    tc_fence_after();
                    const uint32_t sK = sb + kSmK + (uint32_t)st * kTile;
                    const uint32_t d = tmem + kTmS0 + (uint32_t)sbuf * 128u;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        // 16 head dims per step: 32 bytes into a Q row and a K row.
                        const uint32_t off = (uint32_t)(kk >> 2) * kHalfTile + (uint32_t)(kk & 3) * 32u;
                        mma_ss(d, smem_desc_sw128(sQ + off, 16, 1024), smem_desc_sw128(sK + off, 16, 1024), kIdescS,
                               kk > 0 ? 1u : 0u);
                    }
                    mma_commit(bar_addr(sb, BAR_S_FULL + sbuf));
                    mma_commit_mc(bar_addr(sb, BAR_K_EMPTY + st), kClusterMask);
                }
            } else {
                for (int j = 0; j < n_tiles; ++j) {
                    const int st = j % kVStages;
                    const int sbuf = j % kSBufs;
                    if (!wait(bar_addr(sb, BAR_P_FULL + sbuf), (uint32_t)(j / kSBufs) & 1u)) break;
                    if (!wait(bar_addr(sb, BAR_V_FULL + st), (uint32_t)(j / kVStages) & 1u)) break;
                    tc_fence_after();
                    const uint32_t sV = sb + kSmV + (uint32_t)st * kTile;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        // 16 keys per step: rows 16*kk.. of V (2048 bytes); the two
                        // 64-wide halves of the head dim are 16 KB apart.
                        mma_ts(tmem + kTmO, tmem + kTmS0 + (uint32_t)sbuf * 128u + (uint32_t)kk * 8u,
                               smem_desc_sw128(sV + (uint32_t)kk * 2048u, kHalfTile, 1024), kIdescPV,
                               (j > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(bar_addr(sb, BAR_PV_DONE + sbuf));
                    mma_commit_mc(bar_addr(sb, BAR_V_EMPTY + st), kClusterMask);
                }
            }
            // Drain: every MMA issued above completes before TMEM is released
            // (the barrier counts one commit from each issuer).
            mma_commit(bar_addr(sb, BAR_DRAIN));
            wait(bar_addr(sb, BAR_DRAIN), 0, false);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax + epilogue
        // Warps w and w + 4 share the TMEM lanes of quadrant w & 3 and each owns
        // 16 of its rows, read and written with the 16-lane shapes: thread
        // 4i + jq holds rows i and i + 8 of the 16, key columns 8k + 2jq and
        // 8k + 2jq + 1 of every group of eight. A row's maximum and sum stay
        // within one warp (four threads), so the two warps do not meet per tile.
        const int hw = (warp - 4) >> 2;
        const int quad = warp & 3;
        const int jq = lane & 3;
        const int row_a = quad * 32 + hw * 16 + (lane >> 2);   // and row_a + 8
        const uint32_t lane16 = tmem + ((uint32_t)(quad * 32 + hw * 16) << 16);
        // The epilogue reads O one row a thread (all 32 rows of the quadrant),
        // 64 of its columns a warp.
        const int half = hw;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        float* mx_s = reinterpret_cast<float*>(smem + kSmMax);    // the rows' maxima, [128]
        float* ls_s = reinterpret_cast<float*>(smem + kSmLsum);   // the rows' sums, [128]
        float m_a = -INFINITY, m_b = -INFINITY;   // running maxima of rows a and a + 8 (log2 units)
        float l_a = 0.f, l_b = 0.f;               // this thread's part of their sums
        bool failed = false;
        if constexpr (kQNorm) {
            // Folded query norm + RoPE: thread t normalises and rotates one
            // 64-dim half (t / 128) of Q row t % 128. The positions, weights and
            // angles do not depend on Q, so they are prepared while the tile is
            // in flight; the S issuer starts when all 256 threads have arrived.
            const int t = (int)threadIdx.x - 128;
            const int qrow = t & 127, qhalf = t >> 7;
            const int64_t S = (int64_t)p.B * p.N;
            float* w_s = reinterpret_cast<float*>(smem + kSmQnW);
            if (t < 128) w_s[t] = t < 64 ? __ldg(p.qn_w_t + t) : __ldg(p.qn_w_hw + (t - 64));
            const int64_t tok = (int64_t)b * p.N + min(n0 + qrow / p.G, p.N - 1);
            int32_t pos[3];
#pragma unroll
            for (int a = 0; a < 3; ++a) pos[a] = __ldg(p.qn_idx + a * S + tok);
            float cs[32], sn[32];
            if (qhalf == 0)   // warp-uniform
                qnorm_rope_angles<0>(pos, qn_freqs, cs, sn);
            else
                qnorm_rope_angles<1>(pos, qn_freqs, cs, sn);
            named_barrier_sync(1, kSoftmaxThreads);   // the weights are in shared memory
            if (wait(bar_addr(sb, BAR_Q_FULL), 0)) {
                if (qhalf == 0)
                    qnorm_rope_q_half<0>(smem + kSmQ, qrow, cs, sn, w_s, p.qn_eps);
                else
                    qnorm_rope_q_half<1>(smem + kSmQ + kHalfTile, qrow, cs, sn, w_s + 64, p.qn_eps);
                fence_proxy_async_smem();   // generic-proxy writes, read next by tcgen05.mma
                mbar_arrive(bar_addr(sb, BAR_Q_READY));
            } else {
                failed = true;
            }
        }
        // Block-causal mode: the rows' queries are image tokens n_a, n_b
        // (clamped for padding rows, whose output is never stored).
        const int n_a = min(n0 + row_a / p.G, p.N - 1);
        const int n_b = min(n0 + (row_a + 8) / p.G, p.N - 1);
        const int32_t* t_seq = kBlockCausal ? p.t_img + (int64_t)b * p.N : nullptr;
        // A failed (timed-out or aborted) wait sets `failed`; the loop then runs
        // on without touching TMEM or the pipeline barriers.
        for (int j = 0; j < n_tiles; ++j) {
            if (failed) continue;
            const int sbuf = j % kSBufs;
            const uint32_t scol = kTmS0 + (uint32_t)sbuf * 128u;
            if (!__all_sync(0xffffffffu, wait(bar_addr(sb, BAR_S_FULL + sbuf), (uint32_t)(j / kSBufs) & 1u))) {
                failed = true;
                continue;
            }
            const int it = j < n_pre ? 0 : img_tile(j - n_pre);   // image tile index
            const int tile_valid = j < n_pre ? min(kBlockN, L - j * kBlockN) : min(kBlockN, p.N - it * kBlockN);
            tc_fence_after();
            // Block-causal image tiles have their hidden keys written into S first
            // (out of line); prefix keys precede every query.
            if (kBlockCausal && j >= n_pre)   // warp-uniform
                bc_mask_s_cold16(lane16 + scol, t_seq, reinterpret_cast<const int4*>(smem + kSmTileT), j, n_pre, L, it,
                                 tile_valid, n_a, n_b, jq);
            float s[64];
            {
                uint32_t r[64];
                tmem_ld16x256b_x16(lane16 + scol, r);
#pragma unroll
                for (int i = 0; i < 64; ++i) s[i] = __uint_as_float(r[i]);
            }
            // Keys past the end of the prefix or image segment do not exist:
            // warp-uniform, so the per-element mask is a branch that full tiles
            // skip (the opaque statement keeps the compiler from turning it into
            // selects run on every tile).
            if (tile_valid < kBlockN) {
                asm volatile("");
#pragma unroll
                for (int k = 0; k < 16; ++k)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        s[4 * k + e] = 8 * k + 2 * jq + (e & 1) < tile_valid ? s[4 * k + e] : -INFINITY;
            }
            // Row maxima of the raw logits: this thread's 32 columns of each row,
            // then the row's four threads.
            float xa, xb;
            {
                float va[32], vb[32];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    va[2 * k] = s[4 * k];
                    va[2 * k + 1] = s[4 * k + 1];
                    vb[2 * k] = s[4 * k + 2];
                    vb[2 * k + 1] = s[4 * k + 3];
                }
                xa = max32(va);
                xb = max32(vb);
            }
            xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, 1));
            xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, 1));
            xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, 2));
            xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, 2));
            const float na = fmaxf(m_a, xa * p.scale_log2);
            const float nb = fmaxf(m_b, xb * p.scale_log2);
            const bool need_a = na > m_a + kRescaleThreshold;
            const bool need_b = nb > m_b + kRescaleThreshold;
            if (__any_sync(0xffffffffu, need_a || need_b)) {
                const float alpha_a = need_a ? ex2(m_a - na) : 1.0f;
                const float alpha_b = need_b ? ex2(m_b - nb) : 1.0f;
                if (need_a) m_a = na;
                if (need_b) m_b = nb;
                l_a *= alpha_a;
                l_b *= alpha_b;
                if (j > 0) {
                    if (!__all_sync(0xffffffffu, wait(bar_addr(sb, BAR_PV_DONE + (j - 1) % kSBufs),
                                                      (uint32_t)((j - 1) / kSBufs) & 1u))) {
                        failed = true;
                        continue;
                    }
                    tc_fence_after();
                    uint32_t r[32];
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const uint32_t ocol = lane16 + kTmO + (uint32_t)c * 64u;
                        tmem_ld16x256b_x8(ocol, r);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            r[i] = __float_as_uint(__uint_as_float(r[i]) * ((i & 2) ? alpha_b : alpha_a));
                        tmem_st16x256b_x8(ocol, r);
                    }
                    tmem_st_wait();
                }
            }
            // p = 2^(s*scale*log2e - m): one packed FMA per pair, ex2 on the SFU.
            // A hidden key's logit is -inf and stays -inf here (the scale is > 0
            // and m finite from the first tile on), so its p is 0. P_j goes over
            // the rows' own S columns [0, 64) in the 16x128b layout: register 2k
            // (row a) and 2k + 1 (row b) hold keys 8k + 2jq, 8k + 2jq + 1.
            const float2 cc = make_float2(p.scale_log2, p.scale_log2);
            const float2 nma = make_float2(-m_a, -m_a);
            const float2 nmb = make_float2(-m_b, -m_b);
            float2 acc_a[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            float2 acc_b[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            uint32_t pk[32];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float2 aa = ffma2(make_float2(s[4 * k], s[4 * k + 1]), cc, nma);
                const float2 ab = ffma2(make_float2(s[4 * k + 2], s[4 * k + 3]), cc, nmb);
                const float2 ea = make_float2(ex2(aa.x), ex2(aa.y));
                const float2 eb = make_float2(ex2(ab.x), ex2(ab.y));
                acc_a[k & 1] = fadd2(acc_a[k & 1], ea);
                acc_b[k & 1] = fadd2(acc_b[k & 1], eb);
                pk[2 * k] = pack_bf16x2(ea.x, ea.y);
                pk[2 * k + 1] = pack_bf16x2(eb.x, eb.y);
            }
            l_a += (acc_a[0].x + acc_a[0].y) + (acc_a[1].x + acc_a[1].y);
            l_b += (acc_b[0].x + acc_b[0].y) + (acc_b[1].x + acc_b[1].y);
            tmem_st16x128b_x16(lane16 + scol, pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar_addr(sb, BAR_P_FULL + sbuf));
        }
        bool ok = !failed;

        // Only these eight warps write epi_skip, and only before this barrier,
        // so after it every warp of the group takes the same branch.
        if (ok) {
            const int jl = n_tiles - 1;
            ok = __all_sync(0xffffffffu, wait(bar_addr(sb, BAR_PV_DONE + jl % kSBufs), (uint32_t)(jl / kSBufs) & 1u));
        }
        if (!ok) *epi_skip = 1;
        // Each row's sum over its four threads; the row's owner publishes it with
        // the row's maximum.
        l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
        l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
        if (jq == 0) {
            ls_s[row_a] = l_a;
            ls_s[row_a + 8] = l_b;
            mx_s[row_a] = m_a;
            mx_s[row_a + 8] = m_b;
        }
        named_barrier_sync(1, kSoftmaxThreads);
        if (!*epi_skip) {
            tc_fence_after();
            const float l_sum = ls_s[row];
            const float inv_l = 1.0f / l_sum;
            uint8_t* stage = smem + kSmQ + (uint32_t)half * kHalfTile;   // Q is no longer read
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t r[32];
                tmem_ld32(lane_base + kTmO + (uint32_t)half * 64u + (uint32_t)c * 32u, r);
#pragma unroll
                for (int qd = 0; qd < 4; ++qd) {
                    uint4 v;
                    v.x = pack_bf16x2(__uint_as_float(r[qd * 8 + 0]) * inv_l, __uint_as_float(r[qd * 8 + 1]) * inv_l);
                    v.y = pack_bf16x2(__uint_as_float(r[qd * 8 + 2]) * inv_l, __uint_as_float(r[qd * 8 + 3]) * inv_l);
                    v.z = pack_bf16x2(__uint_as_float(r[qd * 8 + 4]) * inv_l, __uint_as_float(r[qd * 8 + 5]) * inv_l);
                    v.w = pack_bf16x2(__uint_as_float(r[qd * 8 + 6]) * inv_l, __uint_as_float(r[qd * 8 + 7]) * inv_l);
                    const int chunk = c * 4 + qd;
                    const uint32_t off = (uint32_t)row * 128u + (uint32_t)((chunk ^ (row & 7)) << 4);
                    *reinterpret_cast<uint4*>(stage + off) = v;
                }
            }
            fence_proxy_async_smem();
            named_barrier_sync(1, kSoftmaxThreads);
            if (threadIdx.x == 4 * 32 && n0 < p.N) {
                tma_store_4d(&tm_o, sb + kSmQ, 0, kvh * p.G, n0, b);
                tma_store_4d(&tm_o, sb + kSmQ + kHalfTile, 64, kvh * p.G, n0, b);
                tma_store_commit_and_wait_read();
            }
            const int n = n0 + row / p.G;
            if (half == 0 && p.lse != nullptr && n < p.N) {
                const int h = kvh * p.G + row % p.G;
                p.lse[((int64_t)b * p.Hq + h) * p.N + n] = (mx_s[row] + log2f(l_sum)) * 0.69314718055994531f;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    // The peer may still multicast into this CTA's shared memory or arrive on its
    // barriers until it is done as well.
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmCols);
    }
}

// --------------------------------------------------------------------- persistent
// Persistent form of the full-mask kernel. A CTA's own work is 40 key tiles
// at 2048^2, and a trace of the one-tile-per-CTA kernel showed ~6.7k cycles
// before the first S and ~4k cycles of epilogue around ~56k cycles of tiles
// (whose steady state runs near the tensor pipe's peak). Here each cluster of
// two CTAs works through a sequence of units (a pair of neighbouring query
// tiles of one sequence and KV head: one tile per CTA) and every role streams
// straight from one unit into the next, so a unit's epilogue and the next
// unit's first tiles overlap:
//   * Q is double-buffered. The next unit's Q is loaded kQLead tiles before
//     the current unit's last K tile; a unit's Q buffer becomes the staging
//     buffer of its output once its last S has completed.
//   * The softmax threads' part of the epilogue is short: each row's sum is
//     combined over its four threads and published with the row's maximum in
//     shared memory (one barrier of the two warps of a sub-partition, the
//     only point where they meet), the LSE is written, then
//     O is read from TMEM (O_FREE: the next unit's first PV may overwrite it),
//     normalised and staged; each thread then arrives on STAGED and goes on
//     to the next unit. The Q/K producer lane issues the staged tile's TMA
//     store when it sees STAGED complete (polled between its K loads) and
//     waits for the store's shared-memory read only before it loads a later
//     unit's Q into that buffer.
//   * Every role decodes the unit after the one it is working on in advance,
//     so the prefix offsets' global loads are off the unit boundary.
//   * The S issuer holds a unit's second S until the previous unit's last PV
//     has completed, so that PV, which the epilogue waits for, is not queued
//     behind two S batches of the next unit.
//   * K and V rings and S buffers run on one tile counter across units. K has
//     two stages here to make room for the second Q.
// The softmax of a tile is the same as in gen_attention_kernel.
//
// Block-causal instantiation (kBC, one sequence: a prefill): the temporal-
// index range of every 64-key half of the image tiles is computed once per
// CTA into shared memory. A unit's key tiles are the prefix tiles, the image
// tiles up to the one holding its last query (the diagonal), and the later
// image tiles with a half whose range meets the unit's queries' range (a
// superset of the tiles holding a key with T_j == T_i); every role walks that
// sequence with the same cursor. Units are taken pair-major (unit U: KV head
// U % Hkv, query-tile pair U / Hkv), so that each cluster's share mixes
// early, cheap query tiles with late, expensive ones.
//
// Folded query norm instantiation (kQN, the full mask): a fourth warpgroup
// (warps 12-15) waits for each unit's raw Q tile, normalises its halves and
// rotates it in shared memory (the arithmetic of the standalone norm/RoPE
// kernel's bf16 path, hence the same bits) and arrives on Q_READY, which the
// S issuer waits for instead of Q_FULL. The next unit's Q is loaded
// kQLeadQN tiles ahead so that this work is hidden. setmaxnreg splits the
// 512 x 128 registers of the launch: 72 a thread for the roles, 168 for the
// softmax, 104 for the norm warpgroup (128 x 72 + 256 x 168 + 128 x 104 = 65536).
namespace pk {

constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr int kQLead = 4;                          // tiles ahead that the next Q is loaded
constexpr int kQLeadQN = 12;                       // ... with the folded query norm
constexpr int kThreadsQN = 512;                    // kQN: 16 warps
constexpr int kQnWarp0 = 12;                       // kQN: the norm warpgroup, warps 12..15
constexpr uint32_t kQnBar = 6;                     // its named barrier (2..5: the sub-partitions' epilogues)
constexpr int kRegsLaunchQN = 65536 / kThreadsQN;      // registers a thread at launch (__launch_bounds__)
constexpr int kRegsRolesQN = 72, kRegsSoftmaxQN = 168, kRegsNormQN = 104;
static_assert(128 * kRegsRolesQN + 256 * kRegsSoftmaxQN + 128 * kRegsNormQN <= kThreadsQN * kRegsLaunchQN,
              "register split above the launch's total");

constexpr uint32_t kSmQ0 = 0;                      // Q buffers 0 and 1 (also output staging)
constexpr uint32_t kSmK = 2 * kTile;
constexpr uint32_t kSmV = kSmK + kKStages * kTile;
constexpr uint32_t kSmRowStats = kSmV + kVStages * kTile;   // float [2 unit parity][sum, max][128 rows]
constexpr uint32_t kSmTileTP = kSmRowStats + 2 * 2 * 128 * 4;  // int4 [kMaxImgTiles] (kBC): min0 max0 min1 max1
constexpr int kMaxUnitsBC = 2048;                      // kBC: units a cluster may take (host-checked)
constexpr uint32_t kSmUnitTiles = kSmTileTP + kMaxImgTiles * 16;   // int [kMaxUnitsBC] (kBC): key tiles of unit k
constexpr uint32_t kSmQnWP = kSmUnitTiles + kMaxUnitsBC * 4;   // float [128] (kQN): the q norm weights
constexpr uint32_t kSmBar = kSmQnWP + 128 * 4;

enum : int {
    Q_FULL = 0,                                    // [2]
    STAGED = Q_FULL + 2,                           // [2] a unit's output is in its Q buffer
    K_FULL = STAGED + 2,
    K_EMPTY = K_FULL + kKStages,
    V_FULL = K_EMPTY + kKStages,
    V_EMPTY = V_FULL + kVStages,
    S_FULL = V_EMPTY + kVStages,
    P_FULL = S_FULL + kSBufs,
    PV_DONE = P_FULL + kSBufs,
    O_FREE = PV_DONE + kSBufs,
    DRAIN = O_FREE + 1,
    Q_READY = DRAIN + 1,                           // [2] kQN: the unit's Q is normalised and rotated
    NUM_BARS = Q_READY + 2
};

constexpr uint32_t kSmTmemSlot = kSmBar + NUM_BARS * 8;
constexpr uint32_t kSmAbort = kSmTmemSlot + 4;
constexpr uint32_t kSmUsed = kSmAbort + 4;
constexpr uint32_t kSmemBytes = kSmUsed + 1024;    // slack to align the base to 1024 bytes
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB of shared memory a CTA may use");

__device__ __forceinline__ uint32_t bar(uint32_t sbase, int i) { return sbase + kSmBar + 8u * i; }

// One unit of work: sequence b, KV head kvh, query tile qt (this CTA's of the pair).
struct Unit {
    int b, kvh, n0, lo, L, n_pre, n_tiles;
    bool ok;                                       // consistent prefix offsets
    int j_diag, tmin, tmax;                        // kBC: the diagonal image tile; the queries' T range
    int run;                                       // kBC: key tiles [0, run) are the prefix tiles and image
                                                   // tiles 0, 1, ..., every key visible to every row of this CTA
};

// kBC: the image tile after t (-1: the first) in a unit's key sequence.
__device__ __forceinline__ int bc_next(const int4* tile_t, const Unit& u, int t, int n_img) {
    if (t < u.j_diag) return t + 1;
    for (int x = t + 1; x < n_img; ++x) {
        const int4 r = tile_t[x];
        if ((r.x <= u.tmax && r.y >= u.tmin) || (r.z <= u.tmax && r.w >= u.tmin)) return x;
    }
    return n_img;
}

// The prefix offsets of unit U's sequence. Every role loads them a unit
// ahead: the loads are issued when a unit starts and their values are first
// used (finish_unit) when it ends, so that their latency is not spent at the
// unit boundary.
struct UnitLoad {
    int U, lo, hi;
};

__device__ __forceinline__ int ld_nc_s32(const int* ptr) {
    int v;
    asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(ptr));
    return v;
}

__device__ __forceinline__ UnitLoad load_unit(const AttnParams& p, int U, int pairs) {
    const int b = U / (p.Hkv * pairs);
    return UnitLoad{U, ld_nc_s32(p.cu_prefix + b), ld_nc_s32(p.cu_prefix + b + 1)};
}

// kBC: kWarp = all 32 lanes of the calling warp take part (the tile count is
// then a ballot over the tiles past the diagonal instead of a serial walk).
template <bool kBC, bool kWarp = false>
__device__ __forceinline__ Unit finish_unit(const AttnParams& p, const UnitLoad& l, int pairs, uint32_t crank,
                                            const uint8_t* smem) {
    Unit u;
    int pair;
    if constexpr (kBC) {
        u.b = 0;
        u.kvh = l.U % p.Hkv;
        pair = l.U / p.Hkv;
    } else {
        const int per_b = p.Hkv * pairs;
        u.b = l.U / per_b;
        const int r = l.U - u.b * per_b;
        u.kvh = r / pairs;
        pair = r - u.kvh * pairs;
    }
    u.n0 = (pair * kCluster + (int)crank) * p.tok_per_tile;
    u.lo = l.lo;
    const int hi = l.hi;
    u.L = hi - u.lo;
    u.ok = !(u.lo < 0 || u.L < 0 || (int64_t)hi > p.total_prefix || u.L > p.max_prefix);
    u.n_pre = (u.L + kBlockN - 1) / kBlockN;
    const int n_img = (p.N + kBlockN - 1) / kBlockN;
    u.n_tiles = u.ok ? u.n_pre + n_img : 0;
    u.j_diag = n_img - 1;
    u.tmin = INT_MIN;
    u.tmax = INT_MAX;
    u.run = u.n_tiles;
    if constexpr (kBC) {
        // The cluster's queries are image tokens [np0, np1): their T range from
        // the 64-key halves holding them (a superset for pairs of under 64 tokens).
        const int4* tile_t = reinterpret_cast<const int4*>(smem + kSmTileTP);
        const int np0 = pair * kCluster * p.tok_per_tile;
        const int np1 = min(p.N, np0 + kCluster * p.tok_per_tile);
        u.j_diag = (np1 - 1) / kBlockN;
        u.tmin = INT_MAX;
        u.tmax = INT_MIN;
        for (int h = np0 / 64; h <= (np1 - 1) / 64; ++h) {
            const int4 r = tile_t[h >> 1];
            u.tmin = min(u.tmin, (h & 1) ? r.z : r.x);
            u.tmax = max(u.tmax, (h & 1) ? r.w : r.y);
        }
        if constexpr (kWarp) {
            // All 32 lanes: count the image tiles of the unit's key sequence.
            const int lane = (int)(threadIdx.x & 31);
            int cnt = u.j_diag + 1;
            for (int t0 = u.j_diag + 1; t0 < n_img; t0 += 32) {
                bool kept = false;
                if (t0 + lane < n_img) {
                    const int4 r = tile_t[t0 + lane];
                    kept = (r.x <= u.tmax && r.y >= u.tmin) || (r.z <= u.tmax && r.w >= u.tmin);
                }
                cnt += __popc(__ballot_sync(0xffffffffu, kept));
            }
            u.n_tiles = u.ok ? u.n_pre + cnt : 0;
            u.run = 0;
        } else {
            // Counted once in the prologue (unit k of this cluster: U = cluster + k * clusters):
            // the image tiles of the key sequence (low 16 bits) and of the run (high 16 bits).
            const int ncl = (int)(gridDim.x / kCluster), cid = (int)(blockIdx.x / kCluster);
            const int packed = reinterpret_cast<const int*>(smem + kSmUnitTiles)[(l.U - cid) / ncl];
            u.n_tiles = u.ok ? u.n_pre + (packed & 0xffff) : 0;
            u.run = u.ok ? u.n_pre + (packed >> 16) : 0;
        }
    }
    return u;
}

template <bool kBC, bool kWarp = false>
__device__ __forceinline__ Unit decode(const AttnParams& p, int U, int pairs, uint32_t crank, const uint8_t* smem) {
    return finish_unit<kBC, kWarp>(p, load_unit(p, U, pairs), pairs, crank, smem);
}

// kBC, all 32 lanes: the number of image tiles at the head of unit u's key
// sequence (tiles 0, 1, ... with none skipped) whose every key is visible to
// every row of this CTA, so that the softmax takes them without the per-row
// classification. Query rows are image tokens [n0, n1] (i = L + n); key k of
// an image tile (j = L + k) is visible to all of them if k <= n0 (at or
// before every query), and a 64-key half is visible as a whole if its last
// existing key is, or if its keys and the queries share one temporal index.
// Prefix keys precede every query and are always visible. A CTA whose rows
// are all padding (n0 >= N) stores nothing: its run is the kept prefix.
__device__ __forceinline__ int bc_visible_run(const AttnParams& p, const Unit& u, const int4* tile_t, int n_img) {
    const int lane = (int)(threadIdx.x & 31);
    // The queries' temporal range, from the ranges of the 64-key halves that
    // hold them (a superset: at worst the run ends earlier than it could).
    const int n1 = min(p.N, u.n0 + p.tok_per_tile) - 1;
    int qlo = INT_MAX, qhi = INT_MIN;
    for (int h = u.n0 / 64; h <= n1 / 64; ++h) {
        const int4 r = tile_t[h >> 1];
        qlo = min(qlo, (h & 1) ? r.z : r.x);
        qhi = max(qhi, (h & 1) ? r.w : r.y);
    }
    const bool one_t = qlo == qhi;
    for (int t0 = 0; t0 < n_img; t0 += 32) {
        const int t = t0 + lane;
        bool good = false;
        if (t < n_img) {
            const int4 r = tile_t[t];
            const bool kept = t <= u.j_diag || (r.x <= u.tmax && r.y >= u.tmin) || (r.z <= u.tmax && r.w >= u.tmin);
            bool full = true;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int lo = h ? r.z : r.x, hi = h ? r.w : r.y;
                const int last = min(p.N - 1, t * kBlockN + 64 * h + 63);
                const bool empty = lo > hi;
                const bool before = last <= u.n0;
                const bool shared = one_t && lo == qlo && hi == qlo;
                full = full && (empty || before || shared || u.n0 >= p.N);
            }
            good = kept && full;
        }
        const uint32_t bad = __ballot_sync(0xffffffffu, !good);
        if (bad) return t0 + __ffs(bad) - 1;
    }
    return n_img;
}

// kBC, off the tile loop's hot path: the next kept image tile after t past
// the unit's diagonal (bc_next out of line, so that its walk takes no
// registers in the loop of the common case).
__device__ __noinline__ int bc_next_cold(const int4* tile_t, Unit u, int t, int n_img) {
    return bc_next(tile_t, u, t, n_img);
}



}  // namespace pk

template <bool kBC, bool kQN>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kQN ? pk::kThreadsQN : kThreads, 1)
gen_attention_persistent_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o,
                                const __grid_constant__ CUtensorMap tm_kimg,
                                const __grid_constant__ CUtensorMap tm_vimg,
                                const __grid_constant__ CUtensorMap tm_kpre,
                                const __grid_constant__ CUtensorMap tm_vpre, const AttnParams p, int n_units,
                                int pairs, const neo::RopeFreqs qn_freqs) {
    using pk::bar;
    using pk::decode;
    using pk::finish_unit;
    using pk::load_unit;
    using pk::UnitLoad;
    using pk::Unit;
    using pk::Q_FULL;
    using pk::STAGED;
    using pk::K_FULL;
    using pk::K_EMPTY;
    using pk::V_FULL;
    using pk::V_EMPTY;
    using pk::S_FULL;
    using pk::P_FULL;
    using pk::PV_DONE;
    using pk::O_FREE;
    using pk::DRAIN;
    using pk::kSmQ0;
    using pk::kQLead;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_addr(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cid = blockIdx.x / kCluster;             // cluster index
    const int ncl = gridDim.x / kCluster;

    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + pk::kSmAbort);
    const BoundedWait wait{abort_flag, &g_dev_error, NEO_DEVERR_TIMEOUT, g_wait_limit_ns};
    // The tensor maps into the TMA unit's descriptor cache, by the lanes that
    // issue the copies, while the barriers and TMEM are being set up.
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_kpre);
        prefetch_tensormap(&tm_kimg);
        prefetch_tensormap(&tm_o);
    } else if (threadIdx.x == 2 * 32) {
        prefetch_tensormap(&tm_vpre);
        prefetch_tensormap(&tm_vimg);
    }
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < pk::NUM_BARS; ++i) {
            uint32_t count = 1;
            if ((i >= P_FULL && i < P_FULL + kSBufs) || i == O_FREE || (i >= STAGED && i < STAGED + 2))
                count = kSoftmaxThreads;
            if (i >= pk::Q_READY && i < pk::Q_READY + 2) count = 128;   // the norm warpgroup
            if ((i >= K_EMPTY && i < K_EMPTY + pk::kKStages) || (i >= V_EMPTY && i < V_EMPTY + pk::kVStages))
                count = kCluster;                // released by the MMA of every CTA of the cluster
            if (i == DRAIN) count = 2;          // one commit from each MMA issuer
            mbar_init(bar(sb, i), count);
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(sb + pk::kSmTmemSlot, kTmCols);
        tmem_relinquish();
    }
    // Everything above touches only this CTA's own resources and may overlap the
    // previous kernel of the stream; global memory is read after this wait.
    griddep_wait();
    const UnitLoad first = cid < n_units ? pk::load_unit(p, cid, pairs) : UnitLoad{0, 0, 0};
    const int n_img = (p.N + kBlockN - 1) / kBlockN;
    if constexpr (kBC) {
        // One warp per image tile: the temporal-index range of each 64-key half
        // (empty halves past the last key: [INT_MAX, INT_MIN]).
        // Four tiles a warp at a time, all loads issued before any is used.
        int4* tile_t = reinterpret_cast<int4*>(smem + pk::kSmTileTP);
        constexpr int kW = kThreads / 32;
        for (int t0 = warp; t0 < n_img; t0 += 4 * kW) {
            int tk[4][kBlockN / 32];
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int c = 0; c < kBlockN / 32; ++c) {
                    const int key = (t0 + q * kW) * kBlockN + c * 32 + lane;
                    tk[q][c] = key < p.N ? __ldg(p.t_img + key) : INT_MIN;
                }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int t = t0 + q * kW;
                if (t >= n_img) break;   // warp-uniform
                int lo2[2] = {INT_MAX, INT_MAX}, hi2[2] = {INT_MIN, INT_MIN};
#pragma unroll
                for (int c = 0; c < kBlockN / 32; ++c)
                    if (t * kBlockN + c * 32 + lane < p.N) {
                        lo2[c >> 1] = min(lo2[c >> 1], tk[q][c]);
                        hi2[c >> 1] = max(hi2[c >> 1], tk[q][c]);
                    }
                const int4 range = make_int4(__reduce_min_sync(0xffffffffu, lo2[0]), __reduce_max_sync(0xffffffffu, hi2[0]),
                                             __reduce_min_sync(0xffffffffu, lo2[1]), __reduce_max_sync(0xffffffffu, hi2[1]));
                if (lane == 0) tile_t[t] = range;
            }
        }
        __syncthreads();
        // The image key tiles of each of this cluster's units, one warp a unit.
        int* unit_tiles = reinterpret_cast<int*>(smem + pk::kSmUnitTiles);
        // One sequence (the only case this kernel takes the block-causal mask
        // for): every unit's prefix offsets are the first unit's, already loaded.
        const uint32_t rank = cluster_ctarank();
        for (int k = warp; cid + k * ncl < n_units; k += kThreads / 32) {
            const Unit u = pk::finish_unit<true, true>(p, UnitLoad{cid + k * ncl, first.lo, first.hi}, pairs, rank, smem);
            const int run = u.ok ? pk::bc_visible_run(p, u, tile_t, n_img) : 0;
            if (lane == 0) unit_tiles[k] = (u.n_tiles - u.n_pre) | (run << 16);
        }
    }
    tc_fence_before();
    __syncthreads();
    // No CTA may multicast into a peer before the peer's barriers exist.
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + pk::kSmTmemSlot);
    const uint32_t crank = cluster_ctarank();
    if (threadIdx.x == 4 * 32) {
        // Report inconsistent prefix offsets once per CTA; such units are skipped by every role.
        // A softmax thread does it: its first wait (for S) is longer than these loads.
        for (int U = cid; U < n_units; U += ncl)
            if (!decode<kBC>(p, U, pairs, crank, smem).ok) {
                atomicOr(&g_dev_error, NEO_DEVERR_BAD_PREFIX);
                break;
            }
    }

    if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------ producers: Q, K and the output stores (warp 0), V (warp 2)
        if constexpr (kQN) setmaxnreg_to<pk::kRegsRolesQN, pk::kRegsLaunchQN>();
        if (lane == 0) {
            const bool is_k = warp == 0;
            const int stages = is_k ? pk::kKStages : pk::kVStages;
            const int full0 = is_k ? K_FULL : V_FULL;
            const int empty0 = is_k ? K_EMPTY : V_EMPTY;
            const uint32_t ring = sb + (is_k ? pk::kSmK : pk::kSmV);
            const CUtensorMap* pre_map = is_k ? &tm_kpre : &tm_vpre;
            const CUtensorMap* img_map = is_k ? &tm_kimg : &tm_vimg;
            bool ok = true;
            int gt = 0, uq = 0, q_issued = -1;
            // Output stores. st_next: the first non-empty unit whose output has not
            // been stored; qc0 / qc1: head, token and sequence coordinates of the
            // unit whose Q (and then output) is in buffer 0 / 1.
            int st_next = 0;
            int3 qc0 = make_int3(0, 0, 0), qc1 = make_int3(0, 0, 0);
            // The TMA store of unit st_next's output once the softmax threads have
            // staged it; without `block` only if they already have.
            auto store_next = [&](bool block) -> bool {
                const int buf = st_next & 1;
                const uint32_t sbar = bar(sb, STAGED + buf);
                const uint32_t par = (uint32_t)(st_next >> 1) & 1u;
                if (block ? !wait(sbar, par) : !mbar_test_wait(sbar, par)) return false;
                const int3 c = buf ? qc1 : qc0;
                if (c.y < p.N) {
                    const uint32_t sQ = sb + kSmQ0 + (uint32_t)buf * kTile;
                    tma_store_4d(&tm_o, sQ, 0, c.x, c.y, c.z);
                    tma_store_4d(&tm_o, sQ + kHalfTile, 64, c.x, c.y, c.z);
                    tma_store_commit();
                }
                ++st_next;
                return true;
            };
            // Q of the uq-th non-empty unit into buffer uq % 2, once the output of
            // the unit that used that buffer before has been stored and read.
            auto issue_q = [&](const Unit& u, int uqi) -> bool {
                const int buf = uqi & 1;
                if (uqi >= 2) {
                    while (st_next <= uqi - 2)
                        if (!store_next(true)) return false;
                    tma_store_wait_read();
                }
                const uint32_t sQ = sb + kSmQ0 + (uint32_t)buf * kTile;
                mbar_arrive_expect_tx(bar(sb, Q_FULL + buf), kTile);
                tma_load_4d(sQ, &tm_q, bar(sb, Q_FULL + buf), 0, u.kvh * p.G, u.n0, u.b);
                tma_load_4d(sQ + kHalfTile, &tm_q, bar(sb, Q_FULL + buf), 64, u.kvh * p.G, u.n0, u.b);
                (buf ? qc1 : qc0) = make_int3(u.kvh * p.G, u.n0, u.b);
                q_issued = uqi;
                return true;
            };
            Unit nxt = cid < n_units ? finish_unit<kBC>(p, first, pairs, crank, smem) : Unit{};
            for (int U = cid; ok && U < n_units; U += ncl) {
                const Unit u = nxt;
                const bool more = U + ncl < n_units;
                const UnitLoad ahead = more ? load_unit(p, U + ncl, pairs) : UnitLoad{0, 0, 0};
                if (u.n_tiles > 0) {
                    if (is_k && uq == 0) ok = issue_q(u, 0);
                    int it = -1;                   // image tile of key tile j
                    for (int j = 0; ok && j < u.n_tiles; ++j) {
                        if (j >= u.n_pre)
                            it = kBC && j >= u.run
                                     ? pk::bc_next(reinterpret_cast<const int4*>(smem + pk::kSmTileTP), u, it, n_img)
                                     : j - u.n_pre;
                        const int st = gt % stages;
                        if (!wait(bar(sb, empty0 + st), ((uint32_t)(gt / stages) & 1u) ^ 1u)) {
                            ok = false;
                            break;
                        }
                        const uint32_t fb = bar(sb, full0 + st);
                        const uint32_t dst = ring + (uint32_t)st * kTile;
                        mbar_arrive_expect_tx(fb, kTile);
                        const uint32_t hdst = dst + crank * kHalfTile;
                        const int d0 = 64 * (int)crank;
                        if (j < u.n_pre)
                            tma_load_3d_mc(hdst, pre_map, fb, d0, u.kvh, u.lo + j * kBlockN, kClusterMask);
                        else
                            tma_load_4d_mc(hdst, img_map, fb, d0, u.kvh, it * kBlockN, u.b, kClusterMask);
                        ++gt;
                        if (is_k && st_next < uq) store_next(false);
                        // The next unit's Q, kQLead tiles before this unit's last K tile.
                        // Its buffer holds the output of the unit before this one, whose
                        // epilogue needs none of this unit's loads.
                        if (is_k && more && j == max(0, u.n_tiles - (kQN ? pk::kQLeadQN : kQLead))) {
                            // The next non-empty unit (empty ones come only from bad prefix offsets).
                            Unit u2 = finish_unit<kBC>(p, ahead, pairs, crank, smem);
                            for (int U2 = U + 2 * ncl; u2.n_tiles == 0 && U2 < n_units; U2 += ncl)
                                u2 = decode<kBC>(p, U2, pairs, crank, smem);
                            if (u2.n_tiles > 0) ok = issue_q(u2, uq + 1);
                        }
                    }
                    ++uq;
                }
                if (more) nxt = finish_unit<kBC>(p, ahead, pairs, crank, smem);
            }
            if (is_k) {
                // The outputs of the last units; then every store has read its tile.
                while (ok && st_next < uq) ok = store_next(true);
                tma_store_wait_read();
            }
            if (*abort_flag) {
                // Let copies already in flight land before the CTA's shared memory goes away.
                if (is_k && q_issued >= 0) {
                    wait(bar(sb, Q_FULL + (q_issued & 1)), (uint32_t)(q_issued >> 1) & 1u, false);
                    if (q_issued >= 1)
                        wait(bar(sb, Q_FULL + ((q_issued - 1) & 1)), (uint32_t)((q_issued - 1) >> 1) & 1u, false);
                }
                for (int g = (gt > stages ? gt - stages : 0); g < gt; ++g)
                    wait(bar(sb, full0 + g % stages), (uint32_t)(g / stages) & 1u, false);
            }
        }
        __syncwarp();
    } else if (warp == 1 || warp == 3) {
        // ------------------------------------------------------------ MMA issuers
        if constexpr (kQN) setmaxnreg_to<pk::kRegsRolesQN, pk::kRegsLaunchQN>();
        if (lane == 0) {
            bool ok = true;
            int gt = 0, uq = 0;
            Unit nxt = cid < n_units ? finish_unit<kBC>(p, first, pairs, crank, smem) : Unit{};
            for (int U = cid; ok && U < n_units; U += ncl) {
                const Unit u = nxt;
                const bool more = U + ncl < n_units;
                const UnitLoad ahead = more ? load_unit(p, U + ncl, pairs) : UnitLoad{0, 0, 0};
                if (u.n_tiles > 0) {
                    if (warp == 1) {
                        const int buf = uq & 1;
                        const uint32_t sQ = sb + kSmQ0 + (uint32_t)buf * kTile;
                        if (!wait(bar(sb, (kQN ? pk::Q_READY : Q_FULL) + buf), (uint32_t)(uq >> 1) & 1u)) break;
                        tc_fence_after();
                        for (int j = 0; j < u.n_tiles; ++j, ++gt) {
                            const int st = gt % pk::kKStages;
                            if (!wait(bar(sb, K_FULL + st), (uint32_t)(gt / pk::kKStages) & 1u)) {
                                ok = false;
                                break;
                            }
                            // S buffer gt%3 holds P of tile gt-3 until that tile's PV has read it.
                            const int sbuf = gt % kSBufs;
                            if (gt >= kSBufs && !wait(bar(sb, PV_DONE + sbuf), ((uint32_t)(gt / kSBufs) & 1u) ^ 1u)) {
                                ok = false;
                                break;
                            }
                            // The previous unit's last PV (tile gt-2) goes ahead of this unit's second S.
                            if (j == 1 && uq > 0 &&
                                !wait(bar(sb, PV_DONE + (gt - 2) % kSBufs), (uint32_t)((gt - 2) / kSBufs) & 1u)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            const uint32_t sK = sb + pk::kSmK + (uint32_t)st * kTile;
                            const uint32_t d = tmem + kTmS0 + (uint32_t)sbuf * 128u;
    #pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                const uint32_t off = (uint32_t)(kk >> 2) * kHalfTile + (uint32_t)(kk & 3) * 32u;
                                mma_ss(d, smem_desc_sw128(sQ + off, 16, 1024), smem_desc_sw128(sK + off, 16, 1024),
                                       kIdescS, kk > 0 ? 1u : 0u);
                            }
                            mma_commit(bar(sb, S_FULL + sbuf));
                            mma_commit_mc(bar(sb, K_EMPTY + st), kClusterMask);
                        }
                    } else {
                        // The unit's first PV overwrites O: the previous unit's epilogue must have read it.
                        if (uq > 0 && !wait(bar(sb, O_FREE), (uint32_t)(uq - 1) & 1u)) break;
                        for (int j = 0; j < u.n_tiles; ++j, ++gt) {
                            const int st = gt % pk::kVStages;
                            const int sbuf = gt % kSBufs;
                            if (!wait(bar(sb, P_FULL + sbuf), (uint32_t)(gt / kSBufs) & 1u) ||
                                !wait(bar(sb, V_FULL + st), (uint32_t)(gt / pk::kVStages) & 1u)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            const uint32_t sV = sb + pk::kSmV + (uint32_t)st * kTile;
    #pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                mma_ts(tmem + kTmO, tmem + kTmS0 + (uint32_t)sbuf * 128u + (uint32_t)kk * 8u,
                                       smem_desc_sw128(sV + (uint32_t)kk * 2048u, kHalfTile, 1024), kIdescPV,
                                       (j > 0 || kk > 0) ? 1u : 0u);
                            }
                            mma_commit(bar(sb, PV_DONE + sbuf));
                            mma_commit_mc(bar(sb, V_EMPTY + st), kClusterMask);
                        }
                    }
                    ++uq;
                }
                if (more) nxt = finish_unit<kBC>(p, ahead, pairs, crank, smem);
            }
            // Drain: every MMA issued above completes before TMEM is released.
            mma_commit(bar(sb, DRAIN));
            wait(bar(sb, DRAIN), 0, false);
        }
        __syncwarp();
    } else if (warp < 12) {
        // ------------------------------------------------------------ softmax + epilogue
        if constexpr (kQN) setmaxnreg_to<pk::kRegsSoftmaxQN, pk::kRegsLaunchQN>();
        // Warps w and w + 4 share the TMEM lanes of quadrant w & 3 and each owns
        // 16 of its rows, read and written with the 16-lane shapes: thread
        // 4i + jq holds rows i and i + 8 of the 16, key columns 8k + 2jq and
        // 8k + 2jq + 1 of every group of eight. A row's maximum and sum stay
        // within one warp (four threads), so the two warps do not meet per tile.
        const int hw = (warp - 4) >> 2;
        const int quad = warp & 3;
        const int jq = lane & 3;
        const int row_a = quad * 32 + hw * 16 + (lane >> 2);   // and row_a + 8
        const uint32_t lane16 = tmem + ((uint32_t)(quad * 32 + hw * 16) << 16);
        // The epilogue reads O one row a thread (all 32 rows of the quadrant),
        // 64 of its columns a warp.
        const int row = quad * 32 + lane;
        const uint32_t pair_bar = 2u + (uint32_t)quad;   // the two warps sharing these TMEM lanes
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        float* rs_s = reinterpret_cast<float*>(smem + pk::kSmRowStats);   // [unit parity][sum, max][128 rows]
        const int4* tile_t = reinterpret_cast<const int4*>(smem + pk::kSmTileTP);
        bool failed = false;
        int gt = 0, uq = 0;
        int sbuf = 0;                              // gt % kSBufs
        uint32_t sphase = 0;                       // (gt / kSBufs) & 1
        // The epilogue of a unit. Both warps of a quadrant reach it after the
        // unit's tiles, failed or not, so that they meet at its barrier.
        struct Pending {
            int b, kvh, n0, buf, last_gt;
            float m_a, m_b, l_a, l_b;
        };
        auto epilogue = [&](const Pending& e) {
            // Each row's sum over its four threads; the row's owner publishes it with
            // the row's maximum. This parity's slot was last read two units ago,
            // before the barrier of the unit in between.
            float la = e.l_a, lb = e.l_b;
            la += __shfl_xor_sync(0xffffffffu, la, 1);
            lb += __shfl_xor_sync(0xffffffffu, lb, 1);
            la += __shfl_xor_sync(0xffffffffu, la, 2);
            lb += __shfl_xor_sync(0xffffffffu, lb, 2);
            float* slot = rs_s + e.buf * 256;
            if (jq == 0) {
                slot[row_a] = la;
                slot[row_a + 8] = lb;
                slot[128 + row_a] = e.m_a;
                slot[128 + row_a + 8] = e.m_b;
            }
            if (!named_barrier_and(pair_bar, 64, !failed)) {
                failed = true;
                return;
            }
            const float l_sum = slot[row];
            const int n = e.n0 + row / p.G;
            if (hw == 0 && p.lse != nullptr && n < p.N) {
                const int h = e.kvh * p.G + row % p.G;
                p.lse[((int64_t)e.b * p.Hq + h) * p.N + n] = (slot[128 + row] + log2f(l_sum)) * 0.69314718055994531f;
            }
            // A warp whose wait fails skips the arrivals below; the roles waiting on
            // them then see the abort flag, and its partner learns of the failure at
            // the next epilogue barrier.
            if (!__all_sync(0xffffffffu, wait(bar(sb, PV_DONE + e.last_gt % kSBufs),
                                              (uint32_t)(e.last_gt / kSBufs) & 1u))) {
                failed = true;
                return;
            }
            tc_fence_after();
            const float inv_l = 1.0f / l_sum;
            uint32_t r[2][32];
#pragma unroll
            for (int c = 0; c < 2; ++c) tmem_ld32(lane_base + kTmO + (uint32_t)hw * 64u + (uint32_t)c * 32u, r[c]);
            // O is read: the next unit's first PV may overwrite it.
            tc_fence_before();
            mbar_arrive(bar(sb, O_FREE));
            // The unit's Q buffer (its last S has completed) stages the output.
            uint8_t* stage = smem + kSmQ0 + (uint32_t)e.buf * kTile + (uint32_t)hw * kHalfTile;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
#pragma unroll
                for (int qd = 0; qd < 4; ++qd) {
                    uint4 v;
                    v.x = pack_bf16x2(__uint_as_float(r[c][qd * 8 + 0]) * inv_l, __uint_as_float(r[c][qd * 8 + 1]) * inv_l);
                    v.y = pack_bf16x2(__uint_as_float(r[c][qd * 8 + 2]) * inv_l, __uint_as_float(r[c][qd * 8 + 3]) * inv_l);
                    v.z = pack_bf16x2(__uint_as_float(r[c][qd * 8 + 4]) * inv_l, __uint_as_float(r[c][qd * 8 + 5]) * inv_l);
                    v.w = pack_bf16x2(__uint_as_float(r[c][qd * 8 + 6]) * inv_l, __uint_as_float(r[c][qd * 8 + 7]) * inv_l);
                    const int chunk = c * 4 + qd;
                    const uint32_t off = (uint32_t)row * 128u + (uint32_t)((chunk ^ (row & 7)) << 4);
                    *reinterpret_cast<uint4*>(stage + off) = v;
                }
            }
            // The TMA store that the producer lane issues reads these bytes.
            fence_proxy_async_smem();
            mbar_arrive(bar(sb, STAGED + e.buf));
        };
        Unit nxt = cid < n_units ? finish_unit<kBC>(p, first, pairs, crank, smem) : Unit{};
        for (int U = cid; U < n_units; U += ncl) {
            const Unit u = nxt;
            const bool more = U + ncl < n_units;
            const UnitLoad ahead = more ? load_unit(p, U + ncl, pairs) : UnitLoad{0, 0, 0};
            float m_a = -INFINITY, m_b = -INFINITY;   // running maxima of rows a and a + 8 (log2 units)
            float l_a = 0.f, l_b = 0.f;               // this thread's part of their sums
            if (u.n_tiles > 0) {
                // kBC: the rows' queries are image tokens n_a, n_b (clamped for
                // padding rows, whose output is never stored).
                const int n_a = min(u.n0 + row_a / p.G, p.N - 1);
                const int n_b = min(u.n0 + (row_a + 8) / p.G, p.N - 1);
                int it = -1;                       // image tile of key tile j
                // A failed wait sets `failed`: the loop then runs on without touching
                // TMEM or the pipeline barriers, to the unit's epilogue barrier.
                for (int j = 0; j < u.n_tiles;
                     ++j, ++gt, sphase ^= (sbuf == kSBufs - 1) ? 1u : 0u, sbuf = sbuf == kSBufs - 1 ? 0 : sbuf + 1) {
                    // Image tiles up to the diagonal and those of the run follow one
                    // another; only kept tiles past both are looked up.
                    if (j >= u.n_pre)
                        it = kBC && j >= u.run && j - u.n_pre > u.j_diag
                                 ? pk::bc_next_cold(tile_t, u, it, n_img)
                                 : j - u.n_pre;
                    if (failed) continue;
                    const uint32_t scol = kTmS0 + (uint32_t)sbuf * 128u;
                    if (!__all_sync(0xffffffffu, wait(bar(sb, S_FULL + sbuf), sphase))) {
                        failed = true;
                        continue;
                    }
                    const int tile_valid = j < u.n_pre ? min(kBlockN, u.L - j * kBlockN) : min(kBlockN, p.N - it * kBlockN);
                    tc_fence_after();
                    // A block-causal tile outside the unit's run has its hidden keys
                    // written into S first (out of line).
                    if (kBC && j >= u.run)   // warp-uniform
                        bc_mask_s_cold16(lane16 + scol, p.t_img, tile_t, j, u.n_pre, u.L, it, tile_valid, n_a, n_b, jq);
                    float s[64];
                    {
                        uint32_t r[64];
                        tmem_ld16x256b_x16(lane16 + scol, r);
    #pragma unroll
                        for (int i = 0; i < 64; ++i) s[i] = __uint_as_float(r[i]);
                    }
                    // Keys past the end of the prefix or image segment do not exist:
                    // warp-uniform, so the per-element mask is a branch that full tiles
                    // skip (the opaque statement keeps the compiler from turning it
                    // into selects run on every tile).
                    if (tile_valid < kBlockN) {
                        asm volatile("");
    #pragma unroll
                        for (int k = 0; k < 16; ++k)
    #pragma unroll
                            for (int e = 0; e < 4; ++e)
                                s[4 * k + e] = 8 * k + 2 * jq + (e & 1) < tile_valid ? s[4 * k + e] : -INFINITY;
                    }
                    // Row maxima of the raw logits: this thread's 32 columns of each row
                    // (three-input max trees), then the row's four threads.
                    float xa, xb;
                    {
                        float va[32], vb[32];
    #pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            va[2 * k] = s[4 * k];
                            va[2 * k + 1] = s[4 * k + 1];
                            vb[2 * k] = s[4 * k + 2];
                            vb[2 * k + 1] = s[4 * k + 3];
                        }
                        xa = max32(va);
                        xb = max32(vb);
                    }
                    xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, 1));
                    xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, 1));
                    xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, 2));
                    xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, 2));
                    const float na = fmaxf(m_a, xa * p.scale_log2);
                    const float nb = fmaxf(m_b, xb * p.scale_log2);
                    const bool need_a = na > m_a + kRescaleThreshold;
                    const bool need_b = nb > m_b + kRescaleThreshold;
                    if (__any_sync(0xffffffffu, need_a || need_b)) {
                        const float alpha_a = need_a ? ex2(m_a - na) : 1.0f;
                        const float alpha_b = need_b ? ex2(m_b - nb) : 1.0f;
                        if (need_a) m_a = na;
                        if (need_b) m_b = nb;
                        l_a *= alpha_a;
                        l_b *= alpha_b;
                        if (j > 0) {
                            const int pbuf = sbuf == 0 ? kSBufs - 1 : sbuf - 1;   // tile gt - 1
                            if (!__all_sync(0xffffffffu, wait(bar(sb, PV_DONE + pbuf), sbuf == 0 ? sphase ^ 1u : sphase))) {
                                failed = true;
                                continue;
                            }
                            tc_fence_after();
                            uint32_t r[32];
    #pragma unroll
                            for (int c = 0; c < 2; ++c) {
                                const uint32_t ocol = lane16 + kTmO + (uint32_t)c * 64u;
                                tmem_ld16x256b_x8(ocol, r);
    #pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    r[i] = __float_as_uint(__uint_as_float(r[i]) * ((i & 2) ? alpha_b : alpha_a));
                                tmem_st16x256b_x8(ocol, r);
                            }
                            tmem_st_wait();
                        }
                    }
                    // p = 2^(s*scale*log2e - m): a hidden key's -inf logit stays -inf
                    // (the scale is > 0 and m finite from the first tile on), so its p is 0.
                    // P_j goes over the rows' own S columns [0, 64) in the 16x128b layout:
                    // register 2k (row a) and 2k + 1 (row b) hold keys 8k + 2jq, 8k + 2jq + 1.
                    const float2 cc = make_float2(p.scale_log2, p.scale_log2);
                    const float2 nma = make_float2(-m_a, -m_a);
                    const float2 nmb = make_float2(-m_b, -m_b);
                    float2 acc_a[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                    float2 acc_b[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                    uint32_t pk[32];
    #pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const float2 aa = ffma2(make_float2(s[4 * k], s[4 * k + 1]), cc, nma);
                        const float2 ab = ffma2(make_float2(s[4 * k + 2], s[4 * k + 3]), cc, nmb);
                        const float2 ea = make_float2(ex2(aa.x), ex2(aa.y));
                        const float2 eb = make_float2(ex2(ab.x), ex2(ab.y));
                        acc_a[k & 1] = fadd2(acc_a[k & 1], ea);
                        acc_b[k & 1] = fadd2(acc_b[k & 1], eb);
                        pk[2 * k] = pack_bf16x2(ea.x, ea.y);
                        pk[2 * k + 1] = pack_bf16x2(eb.x, eb.y);
                    }
                    l_a += (acc_a[0].x + acc_a[0].y) + (acc_a[1].x + acc_a[1].y);
                    l_b += (acc_b[0].x + acc_b[0].y) + (acc_b[1].x + acc_b[1].y);
                    tmem_st16x128b_x16(lane16 + scol, pk);
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(bar(sb, P_FULL + sbuf));
                }
            }
            // Before the epilogue, whose wait for the last PV hides it.
            if (more) nxt = finish_unit<kBC>(p, ahead, pairs, crank, smem);
            if (u.n_tiles > 0) {
                epilogue(Pending{u.b, u.kvh, u.n0, uq & 1, gt - 1, m_a, m_b, l_a, l_b});
                ++uq;
            }
        }
    } else if constexpr (kQN) {
        // ------------------------------------------------------------ query norm + RoPE (warps 12..15)
        // Thread t normalises and rotates both 64-dim halves of Q row t of each
        // unit's tile in shared memory (128-byte swizzled, as the TMA wrote it).
        setmaxnreg_to<pk::kRegsNormQN, pk::kRegsLaunchQN>();
        const int t = (int)threadIdx.x - pk::kQnWarp0 * 32;
        float* w_s = reinterpret_cast<float*>(smem + pk::kSmQnWP);
        w_s[t] = t < 64 ? __ldg(p.qn_w_t + t) : __ldg(p.qn_w_hw + (t - 64));
        named_barrier_sync(pk::kQnBar, 128);           // the weights are in shared memory
        const int64_t S = (int64_t)p.B * p.N;
        bool ok = true;
        int uq = 0;
        Unit nxt = cid < n_units ? finish_unit<kBC>(p, first, pairs, crank, smem) : Unit{};
        for (int U = cid; ok && U < n_units; U += ncl) {
            const Unit u = nxt;
            const bool more = U + ncl < n_units;
            const UnitLoad ahead = more ? load_unit(p, U + ncl, pairs) : UnitLoad{0, 0, 0};
            if (u.n_tiles > 0) {
                const int buf = uq & 1;
                uint8_t* sQ = smem + kSmQ0 + (uint32_t)buf * kTile;
                const int64_t tok = (int64_t)u.b * p.N + min(u.n0 + t / p.G, p.N - 1);
                int32_t pos[3];
#pragma unroll
                for (int a = 0; a < 3; ++a) pos[a] = __ldg(p.qn_idx + a * S + tok);
                ok = __all_sync(0xffffffffu, wait(bar(sb, Q_FULL + buf), (uint32_t)(uq >> 1) & 1u));
                if (ok) {
                    qnorm_rope_q_half_lowreg<0>(sQ, t, pos, qn_freqs, w_s, p.qn_eps);
                    qnorm_rope_q_half_lowreg<1>(sQ + kHalfTile, t, pos, qn_freqs, w_s + 64, p.qn_eps);
                    fence_proxy_async_smem();       // generic-proxy writes, read next by tcgen05.mma
                    mbar_arrive(bar(sb, pk::Q_READY + buf));
                }
                ++uq;
            }
            if (more) nxt = finish_unit<kBC>(p, ahead, pairs, crank, smem);
        }
    }

    tc_fence_before();
    __syncthreads();
    // The peer may still multicast into this CTA's shared memory or arrive on its
    // barriers until it is done as well.
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmCols);
    }
}

// --------------------------------------------------------------------- wait self-test
// One thread waits, with the kernels' bounded wait, on an mbarrier that
// nothing arrives at. The wait gives up after the configured limit, raises the
// abort flag and records NEO_DEVERR_TIMEOUT, exactly as a stalled pipeline
// wait inside the attention kernels does; there are no copies, MMAs or TMEM
// to unwind, so the test leaves the context as it found it.
__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel() {
    __shared__ __align__(8) uint64_t barrier;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    const uint32_t b = smem_addr(&barrier);
    mbar_init(b, 1);
    fence_barrier_init();
    const BoundedWait wait{&abort_flag, &g_dev_error, NEO_DEVERR_TIMEOUT, g_wait_limit_ns};
    wait(b, 0);   // phase 0 never completes
}

// --------------------------------------------------------------------- host
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// bf16 tensor map with 128-byte swizzle; dims[0] is the contiguous head dim.
bool make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
              const uint32_t* box) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t d[5], s[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
    }
    for (int i = 0; i < rank - 1; ++i) s[i] = strides_bytes[i];
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), d, s, bx, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace neo {

neo_status attention_error_read_clear(cudaStream_t stream, uint32_t* word) {
    unsigned int h = 0, zero = 0;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return NEO_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&h, g_dev_error, sizeof(h)) != cudaSuccess) return NEO_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_dev_error, &zero, sizeof(zero)) != cudaSuccess) return NEO_ERR_CUDA;
    if (word) *word = h;
    if (h & NEO_DEVERR_TIMEOUT) return NEO_ERR_TIMEOUT;
    return h ? NEO_ERR_DEVICE : NEO_OK;
}

neo_status attention_set_timeout(uint64_t ns) {
    unsigned long long v = ns;
    return cudaMemcpyToSymbol(g_wait_limit_ns, &v, sizeof(v)) == cudaSuccess ? NEO_OK : NEO_ERR_CUDA;
}

}  // namespace neo

namespace {

neo_status launch_attention(const void* q_img, const void* k_prefix, const void* v_prefix, const void* k_img,
                            const void* v_img, neo_dtype dtype, const int32_t* cu_prefix, int64_t total_prefix,
                            int32_t max_prefix, int B, int N, int Hq, int Hkv, int D, neo_mask mask_mode,
                            const int32_t* t_prefix, const int32_t* t_img, const neo_qnorm_params* qn,
                            float scale, void* out, float* lse, cudaStream_t stream) {
    if (D != 128 || B < 1 || N < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return NEO_ERR_INVALID_ARG;
    const int G = Hq / Hkv;
    if (kBlockM % G != 0) return NEO_ERR_UNSUPPORTED;
    if (total_prefix < 0 || max_prefix < 0 || total_prefix > 0x7fffffffLL) return NEO_ERR_INVALID_ARG;
    if (!q_img || !k_img || !v_img || !out || !cu_prefix) return NEO_ERR_INVALID_ARG;
    if (total_prefix > 0 && (!k_prefix || !v_prefix)) return NEO_ERR_INVALID_ARG;
    if (!neo::aligned16(q_img) || !neo::aligned16(k_img) || !neo::aligned16(v_img) || !neo::aligned16(out) ||
        (total_prefix > 0 && (!neo::aligned16(k_prefix) || !neo::aligned16(v_prefix))))
        return NEO_ERR_INVALID_ARG;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return NEO_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || scale < 0.f) return NEO_ERR_INVALID_ARG;
    if (mask_mode != NEO_MASK_FULL && mask_mode != NEO_MASK_BLOCK_CAUSAL) return NEO_ERR_INVALID_ARG;
    if (mask_mode == NEO_MASK_BLOCK_CAUSAL && (!t_img || (total_prefix > 0 && !t_prefix))) return NEO_ERR_INVALID_ARG;
    if (mask_mode == NEO_MASK_BLOCK_CAUSAL && (N + kBlockN - 1) / kBlockN > kMaxImgTiles) return NEO_ERR_UNSUPPORTED;
    if (dtype != NEO_BF16) return NEO_ERR_UNSUPPORTED;
    if (B > 65535 || Hkv > 65535) return NEO_ERR_UNSUPPORTED;
    if (qn && (!qn->indexes || !qn->q_norm_w || !qn->q_norm_hw_w || !(qn->theta_t > 0.f) ||
               !(qn->theta_hw > 0.f) || !std::isfinite(qn->theta_t) || !std::isfinite(qn->theta_hw) ||
               !(qn->eps >= 0.f) || !std::isfinite(qn->eps)))
        return NEO_ERR_INVALID_ARG;

    const int tok_per_tile = kBlockM / G;
    const uint64_t row = 128 * 2;   // bytes per head row
    CUtensorMap tq, to, tki, tvi, tkp, tvp;
    {
        const uint64_t dims[4] = {128, (uint64_t)Hq, (uint64_t)N, (uint64_t)B};
        const uint64_t strides[3] = {row, row * Hq, row * Hq * N};
        const uint32_t box[4] = {64, (uint32_t)G, (uint32_t)tok_per_tile, 1};
        if (!make_map(&tq, q_img, 4, dims, strides, box) || !make_map(&to, out, 4, dims, strides, box))
            return NEO_ERR_CUDA;
    }
    {
        const uint64_t dims[4] = {128, (uint64_t)Hkv, (uint64_t)N, (uint64_t)B};
        const uint64_t strides[3] = {row, row * Hkv, row * Hkv * N};
        const uint32_t box[4] = {64, 1, (uint32_t)kBlockN, 1};
        if (!make_map(&tki, k_img, 4, dims, strides, box) || !make_map(&tvi, v_img, 4, dims, strides, box))
            return NEO_ERR_CUDA;
    }
    {
        // With no prefix rows at all the prefix maps are never read; point them at the image keys.
        const bool empty = total_prefix == 0;
        const uint64_t dims[3] = {128, (uint64_t)Hkv, empty ? 1 : (uint64_t)total_prefix};
        const uint64_t strides[2] = {row, row * Hkv};
        const uint32_t box[3] = {64, 1, (uint32_t)kBlockN};
        if (!make_map(&tkp, empty ? k_img : k_prefix, 3, dims, strides, box) ||
            !make_map(&tvp, empty ? v_img : v_prefix, 3, dims, strides, box))
            return NEO_ERR_CUDA;
    }

    static neo::DeviceOnce attr_slots[neo::kMaxDevices];
    neo::DeviceOnce* attr = neo::device_slot(attr_slots);
    if (!attr) return NEO_ERR_CUDA;
    std::call_once(attr->once, [attr] {
        // (the full mask without the folded norm runs in the persistent kernel)
        const void* kernels[2] = {(const void*)gen_attention_kernel<true, false>,
                                  (const void*)gen_attention_kernel<true, true>};
        for (const void* k : kernels)
            if (attr->err == cudaSuccess)
                attr->err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        const void* persistent[3] = {(const void*)gen_attention_persistent_kernel<false, false>,
                                     (const void*)gen_attention_persistent_kernel<true, false>,
                                     (const void*)gen_attention_persistent_kernel<false, true>};
        for (const void* k : persistent)
            if (attr->err == cudaSuccess)
                attr->err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pk::kSmemBytes);
    });
    if (attr->err != cudaSuccess) return NEO_ERR_CUDA;

    AttnParams prm;
    prm.cu_prefix = cu_prefix;
    prm.t_prefix = t_prefix;
    prm.t_img = t_img;
    prm.mask_mode = (int)mask_mode;
    prm.lse = lse;
    prm.total_prefix = total_prefix;
    prm.B = B;
    prm.N = N;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.G = G;
    prm.tok_per_tile = tok_per_tile;
    prm.max_prefix = max_prefix;
    // A zero scale becomes a tiny positive one: every logit times it is then
    // far below an ulp of the exponent (the same uniform softmax), and a hidden
    // key's -inf logit stays -inf instead of becoming NaN.
    prm.scale_log2 = std::max(scale * 1.4426950408889634f, 1e-30f);
    prm.qn_idx = qn ? qn->indexes : nullptr;
    prm.qn_w_t = qn ? qn->q_norm_w : nullptr;
    prm.qn_w_hw = qn ? qn->q_norm_hw_w : nullptr;
    prm.qn_eps = qn ? qn->eps : 0.f;
    const neo::RopeFreqs fr = qn ? neo::rope3_freqs(qn->theta_t, qn->theta_hw) : neo::RopeFreqs{};

    // Query tiles come in clusters of kCluster (a tile past the last token loads,
    // computes and stores nothing of its own but still shares the K/V stream).
    const int qtiles = (N + tok_per_tile - 1) / tok_per_tile;
    const bool bc = mask_mode == NEO_MASK_BLOCK_CAUSAL;
    if ((!qn && (!bc || B == 1)) || (qn && !bc)) {
        // Full mask (with or without the folded query norm), and the
        // block-causal mask of one sequence (a prefill): the persistent kernel,
        // one cluster per pair of SMs it can keep resident, each working through
        // its share of the units.
        // Clusters the device keeps resident, per variant (plain, folded norm),
        // found once per device after the attributes above are set.
        static neo::DeviceOnce occ_slots[neo::kMaxDevices];
        neo::DeviceOnce* occ = neo::device_slot(occ_slots);
        if (!occ) return NEO_ERR_CUDA;
        std::call_once(occ->once, [occ] {
            for (int v = 0; v < 2; ++v) {
                cudaLaunchConfig_t cfg = {};
                cudaLaunchAttribute attr;
                attr.id = cudaLaunchAttributeClusterDimension;
                attr.val.clusterDim.x = kCluster;
                attr.val.clusterDim.y = 1;
                attr.val.clusterDim.z = 1;
                cfg.gridDim = dim3(kCluster * 1024, 1, 1);
                cfg.blockDim = dim3(v ? pk::kThreadsQN : kThreads, 1, 1);
                cfg.dynamicSmemBytes = pk::kSmemBytes;
                cfg.attrs = &attr;
                cfg.numAttrs = 1;
                int& mc = occ->value[v];
                const void* k = v ? (const void*)gen_attention_persistent_kernel<false, true>
                                  : (const void*)gen_attention_persistent_kernel<false, false>;
                if (cudaOccupancyMaxActiveClusters(&mc, k, &cfg) != cudaSuccess) mc = 0;
                cudaGetLastError();
            }
        });
        const int max_clusters = occ->value[qn ? 1 : 0];
        if (max_clusters < 1) return NEO_ERR_CUDA;
        const int pairs = (qtiles + kCluster - 1) / kCluster;
        const int64_t n_units = (int64_t)B * Hkv * pairs;
        if (n_units > 0x7fffffffLL) return NEO_ERR_UNSUPPORTED;
        const int clusters = (int)std::min<int64_t>(n_units, max_clusters);
        // A one-sequence block-causal launch keeps one tile count per unit of a
        // cluster in shared memory (at most pk::kMaxUnitsBC of them); beyond that
        // it takes the one-tile-per-CTA kernel below.
        if (!bc || (n_units + clusters - 1) / clusters <= pk::kMaxUnitsBC) {
            auto kernel = qn ? gen_attention_persistent_kernel<false, true>
                             : (bc ? gen_attention_persistent_kernel<true, false> : gen_attention_persistent_kernel<false, false>);
            return neo::launch_overlapped(kernel, dim3((unsigned)(clusters * kCluster)),
                                          dim3(qn ? pk::kThreadsQN : kThreads), pk::kSmemBytes, stream, tq, to, tki,
                                          tvi, tkp, tvp, prm, (int)n_units, pairs, fr);
        }
    }
    // The block-causal mask of several sequences, with or without the folded
    // query norm, and of one sequence with it: one query tile per CTA (the
    // full mask always returned above).
    const dim3 grid((unsigned)((qtiles + kCluster - 1) / kCluster * kCluster), (unsigned)Hkv, (unsigned)B);
    auto kernel = qn ? gen_attention_kernel<true, true> : gen_attention_kernel<true, false>;
    kernel<<<grid, kThreads, kSmemBytes, stream>>>(tq, to, tki, tvi, tkp, tvp, fr, prm);
    return neo::launch_status();
}

}  // namespace

extern "C" neo_status neo_gen_attention(const void* q_img, const void* k_prefix, const void* v_prefix,
                                        const void* k_img, const void* v_img, neo_dtype dtype,
                                        const int32_t* cu_prefix, int64_t total_prefix, int32_t max_prefix,
                                        int B, int N, int Hq, int Hkv, int D, neo_mask mask_mode,
                                        const int32_t* t_prefix, const int32_t* t_img, float scale, void* out,
                                        float* lse, cudaStream_t stream) {
    return launch_attention(q_img, k_prefix, v_prefix, k_img, v_img, dtype, cu_prefix, total_prefix, max_prefix, B,
                            N, Hq, Hkv, D, mask_mode, t_prefix, t_img, nullptr, scale, out, lse, stream);
}

extern "C" neo_status neo_gen_attention_qnorm(const void* q_img_raw, const void* k_prefix, const void* v_prefix,
                                              const void* k_img, const void* v_img, neo_dtype dtype,
                                              const int32_t* cu_prefix, int64_t total_prefix, int32_t max_prefix,
                                              int B, int N, int Hq, int Hkv, int D, neo_mask mask_mode,
                                              const int32_t* t_prefix, const int32_t* t_img,
                                              const neo_qnorm_params* qnorm, float scale, void* out, float* lse,
                                              cudaStream_t stream) {
    if (!qnorm) return NEO_ERR_INVALID_ARG;
    return launch_attention(q_img_raw, k_prefix, v_prefix, k_img, v_img, dtype, cu_prefix, total_prefix, max_prefix,
                            B, N, Hq, Hkv, D, mask_mode, t_prefix, t_img, qnorm, scale, out, lse, stream);
}

extern "C" neo_status neo_selftest_bounded_wait(cudaStream_t stream) {
    bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>();
    return neo::launch_status();
}

/*
 * libneo: the generation-pass hot path of NEO-unify (SenseNova-U1.5) on one
 * GB300 GPU (sm_103a), as a plain C ABI.
 *
 * Sources of the operations (page title, section):
 *   [U15] "SenseNova-U1.5 (NEO-unify) architecture"
 *   [U1]  "SenseNova-U1: Unifying Multimodal Understanding and Generation
 *          with NEO-unify Architecture"
 *
 * Conventions shared by every entry point:
 *   - Every tensor argument is a DEVICE pointer owned by the caller; the
 *     library never frees, keeps or allocates caller memory. Layouts are
 *     row-major and contiguous, in the flash-attention [B, S, H, D] order
 *     ([U1] section 4.4, KV-cache reuse). Tensor pointers must be 16-byte aligned.
 *   - Work is enqueued on `stream` and runs asynchronously; no entry point
 *     synchronises the device except neo_get_device_error.
 *   - Arguments are checked on the host before anything is enqueued. A bad
 *     argument returns NEO_ERR_INVALID_ARG, a valid but unimplemented case
 *     NEO_ERR_UNSUPPORTED, a CUDA launch failure NEO_ERR_CUDA; nothing is
 *     enqueued in those cases. Device-side faults that a host check cannot
 *     see (an inconsistent cu_prefix array, a pipeline wait that ran out of
 *     time) are recorded in a device error word read by neo_get_device_error.
 *   - No C++ exception crosses this boundary.
 */
#ifndef NEO_H
#define NEO_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NEO_OK = 0,
    NEO_ERR_INVALID_ARG = 1,
    NEO_ERR_UNSUPPORTED = 2,
    NEO_ERR_CUDA = 3,
    NEO_ERR_TIMEOUT = 4,
    NEO_ERR_DEVICE = 5
} neo_status;

typedef enum { NEO_BF16 = 0, NEO_F32 = 1 } neo_dtype;

typedef enum { NEO_MASK_FULL = 0, NEO_MASK_BLOCK_CAUSAL = 1 } neo_mask;

/* Device error word bits (neo_get_device_error). */
#define NEO_DEVERR_TIMEOUT     0x1u  /* a pipeline wait exceeded its time limit */
#define NEO_DEVERR_BAD_PREFIX  0x2u  /* cu_prefix not ascending / beyond total_prefix / above max_prefix */

/* ------------------------------------------------------------------------
 * Position indexes (three rotary axes).
 * [U15] section "Three rotary axes", last paragraph: all tokens of one image
 * share one temporal index and their height/width indices tile the token
 * grid; each CFG branch derives the image's temporal index from its own
 * prompt length ([U15] section "Runtime / metadata status").
 *
 * A sequence is described as consecutive segments:
 *   kind NEO_SEG_TEXT : a = first position p0, b = count; token i -> (p0+i, p0+i, p0+i)
 *   kind NEO_SEG_IMAGE: a = temporal index T, b = rows, c = cols; token
 *                       r*cols + c (row-major) -> (T, r, c)
 * ------------------------------------------------------------------------ */
#define NEO_SEG_TEXT 0
#define NEO_SEG_IMAGE 1
#define NEO_MAX_SEGMENTS 64

typedef struct {
    int32_t kind;
    int32_t a;
    int32_t b;
    int32_t c;
} neo_pos_segment;

/* Writes indexes[3, S] (int32, device, row k = axis k) for the concatenation
 * of `n_segs` segments (host array, 1..NEO_MAX_SEGMENTS) whose token counts
 * sum to S. Returns NEO_ERR_INVALID_ARG if the counts do not sum to S, a
 * segment has a negative size or unknown kind, or indexes is NULL. */
neo_status neo_build_positions(int32_t* indexes, int64_t S,
                               const neo_pos_segment* segs, int n_segs,
                               cudaStream_t stream);

/* ------------------------------------------------------------------------
 * QK-norm on head halves, then three-axis RoPE, in place.
 * [U15] section "Three rotary axes": q_norm/k_norm (weight [64]) normalise
 * head dims [0:64), q_norm_hw/k_norm_hw dims [64:128); then dims [0:64)
 * rotate with base theta_t (rope_theta, 5e6) at position indexes[0],
 * [64:96) with base theta_hw (rope_theta_hw, 1e4) at indexes[1] and
 * [96:128) with theta_hw at indexes[2]. Each half is
 *   y = x / sqrt(mean(x^2) + eps) * w,
 * and each slice of width d at offset o pairs dims (o+i, o+i+d/2),
 * i < d/2, turning the pair by the angle p * theta^(-2i/d):
 *   (u, w) -> (u cos a - w sin a, w cos a + u sin a).
 *
 * q: [S, Hq, D] and k: [S, Hkv, D] of `dtype` (bf16 or fp32), overwritten
 * with the result; arithmetic in fp32, one rounding to `dtype` at the end.
 * Either tensor may be NULL with its head count 0 (e.g. keys only).
 * indexes: int32 [3, S]; any int32 position is valid: each angle is reduced
 * modulo 2 pi exactly (the frequency is held as a 64-bit fraction of a turn),
 * so the angle error does not grow with the position. Norm weights: fp32 [64]
 * each; the q weights may be NULL when Hq == 0 and the k weights when
 * Hkv == 0. D must be 128. q and k must not overlap.
 * ------------------------------------------------------------------------ */
neo_status neo_qknorm_rope3(void* q, void* k, neo_dtype dtype,
                            int64_t S, int Hq, int Hkv, int D,
                            const int32_t* indexes,
                            const float* q_norm_w, const float* q_norm_hw_w,
                            const float* k_norm_w, const float* k_norm_hw_w,
                            float theta_t, float theta_hw, float eps,
                            cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Generation-pass attention over the frozen prefix plus the image tokens.
 * [U15] section "Mixture of Transformers", items 1-2: the noisy image tokens
 * attend over the keys/values that the understanding pass wrote for the
 * prefix, together with their own keys/values, and the cache is not written
 * (update_cache=False). [U15] section "GQA fusion does not apply": the
 * generation pass is unmasked (mask_mode NEO_MASK_FULL). For each sequence b
 * and query head h, with KV head kv = h / (Hq/Hkv):
 *   out[b,n,h,:] = sum_j softmax_j(scale * <q[b,n,h,:], key_j>) * value_j
 * over the keys [k_prefix rows of b ; k_img[b,:,kv,:]] (and values alike).
 *
 * q_img: [B, N, Hq, D] bf16; k_img, v_img: [B, N, Hkv, D] bf16.
 * k_prefix, v_prefix: [total_prefix, Hkv, D] bf16, the prefixes of all
 *   sequences packed without padding; sequence b owns rows
 *   cu_prefix[b] .. cu_prefix[b+1]-1. NULL allowed when total_prefix == 0.
 * cu_prefix: int32 [B+1] on the device, cu_prefix[0] = 0, non-decreasing,
 *   cu_prefix[B] <= total_prefix, every length <= max_prefix (checked on
 *   the device: a violation sets NEO_DEVERR_BAD_PREFIX and the affected
 *   sequence's output is left unwritten). A length of 0 is allowed.
 * D must be 128; Hq must be a multiple of Hkv and 128 a multiple of Hq/Hkv.
 * mask_mode: NEO_MASK_FULL, or NEO_MASK_BLOCK_CAUSAL ([U15] section
 *   "Block-causal attention"): in the concatenated order [prefix_b ; image_b]
 *   key j is visible to query i (i = L_b + n) iff T_j == T_i or j <= i, with
 *   T the temporal index (indexes[0]) from t_prefix (device int32
 *   [total_prefix], may be NULL when total_prefix == 0) and t_img (device
 *   int32 [B*N]); both are ignored in NEO_MASK_FULL. A mixed prefill passes
 *   its tokens as the image segment with L_b = 0 (or a cached chunk as the
 *   prefix). Missing temporal indexes return NEO_ERR_INVALID_ARG; an image
 *   segment of more than 131072 tokens returns NEO_ERR_UNSUPPORTED. Key
 *   tiles that the mask hides from every query of a tile are skipped; any
 *   temporal indexes are allowed (no ordering is assumed).
 * scale: logit scale (1/sqrt(128) in the model), finite and >= 0.
 * out: [B, N, Hq, D] bf16. lse: optional fp32 [B, Hq, N] natural-log
 *   sum of exp(logits) per query row, or NULL.
 * ------------------------------------------------------------------------ */
neo_status neo_gen_attention(const void* q_img, const void* k_prefix,
                             const void* v_prefix, const void* k_img,
                             const void* v_img, neo_dtype dtype,
                             const int32_t* cu_prefix, int64_t total_prefix,
                             int32_t max_prefix, int B, int N, int Hq, int Hkv,
                             int D, neo_mask mask_mode,
                             const int32_t* t_prefix, const int32_t* t_img,
                             float scale, void* out, float* lse,
                             cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Generation attention with the query norm and RoPE folded in.
 * The same result as neo_qknorm_rope3 on the queries (steps a1 + a2, [U15]
 * section "Three rotary axes") followed by neo_gen_attention, in one launch:
 * each query tile is normalised on its halves and rotated in shared memory
 * right after it is loaded, so the normalised queries never go to memory.
 * The arithmetic is that of neo_qknorm_rope3's bf16 path, so the attention
 * sees the same query bits (the keys still go through neo_qknorm_rope3).
 *
 * q_img_raw: [B, N, Hq, D] bf16 queries before the norm (read only).
 * qnorm (host pointer, read during the call):
 *   indexes     device int32 [3, B*N]: positions of the image tokens, token
 *               b*N + n (as neo_build_positions writes them);
 *   q_norm_w, q_norm_hw_w  device fp32 [64] each: weights of dims [0,64)
 *               and [64,128);
 *   theta_t, theta_hw      rotary bases (5e6, 1e4), finite and > 0;
 *   eps         finite and >= 0 (1e-6).
 * Every other argument, the layouts and the errors are those of
 * neo_gen_attention; a NULL qnorm or a NULL member returns
 * NEO_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------ */
typedef struct {
    const int32_t* indexes;
    const float* q_norm_w;
    const float* q_norm_hw_w;
    float theta_t;
    float theta_hw;
    float eps;
} neo_qnorm_params;

neo_status neo_gen_attention_qnorm(const void* q_img_raw, const void* k_prefix,
                                   const void* v_prefix, const void* k_img,
                                   const void* v_img, neo_dtype dtype,
                                   const int32_t* cu_prefix, int64_t total_prefix,
                                   int32_t max_prefix, int B, int N, int Hq, int Hkv,
                                   int D, neo_mask mask_mode,
                                   const int32_t* t_prefix, const int32_t* t_img,
                                   const neo_qnorm_params* qnorm, float scale,
                                   void* out, float* lse, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Append a chunk of keys/values to the packed prefix cache.
 * [U15] section "Mixture of Transformers", item 1: the understanding pass
 * (a prefill, possibly in chunks) writes the keys/values of its tokens into
 * the KV cache that every generation pass then reads; [U1] section 4.4: the
 * prefix cache is laid out once in the [B, S, H, D] form the attention
 * reads, here packed without padding (the layout neo_gen_attention takes).
 * The keys are expected already normalised and rotated (neo_qknorm_rope3
 * with the prefill positions).
 *
 * k_old, v_old: [total_old, Hkv, D], sequence b owning rows cu_old[b] ..
 *   cu_old[b+1]-1 (cu_old: device int32 [B+1], cu_old[0] = 0). NULL allowed
 *   when total_old == 0.
 * k_new, v_new: [B, N, Hkv, D]; sequence b appends its first n_new[b] rows
 *   (n_new: device int32 [B], each in [0, N]; NULL means N for all).
 * k_out, v_out: [capacity, Hkv, D]: sequence b's old rows, then its new rows,
 *   packed in sequence order; cu_out: device int32 [B+1], written. The
 *   outputs may not overlap the inputs, except that a single sequence (B = 1)
 *   may append in place (k_out == k_old, v_out == v_old; its old rows are then
 *   left untouched). dtype: NEO_BF16 or NEO_F32; D must be 128; pointers
 *   16-byte aligned.
 * Host-side errors: NEO_ERR_INVALID_ARG (sizes, pointers, overlap),
 * NEO_ERR_UNSUPPORTED (B > 65535, capacity >= 2^31, total_old > capacity).
 * Device-side: cu_old not ascending or beyond total_old, an n_new outside
 * [0, N], or a result beyond capacity sets NEO_DEVERR_BAD_PREFIX and the
 * affected sequence is not written.
 * ------------------------------------------------------------------------ */
neo_status neo_write_prefix_cache(const void* k_old, const void* v_old,
                                  const int32_t* cu_old, int64_t total_old,
                                  const void* k_new, const void* v_new,
                                  const int32_t* n_new, int B, int N, int Hkv, int D,
                                  neo_dtype dtype, void* k_out, void* v_out,
                                  int32_t* cu_out, int64_t capacity,
                                  cudaStream_t stream);

/* ------------------------------------------------------------------------
 * x0 -> velocity conversion and one Euler step, in place.
 * [U15] section "Flow matching without a VAE": the pixel head predicts x0
 * and the sampler forms v = (x0 - z) / max(1 - t, t_eps), then
 * z = z + (t_next - t) * v; t_eps is 0.02 at inference ([U15] section
 * "Dead or misleading upstream details"). Elementwise, so patch and pixel
 * layouts give the same result.
 *
 * z: fp32 [n], updated in place; x0_hat: fp32 [n]; v_out: optional fp32 [n]
 * receiving v, or NULL. fp32 arithmetic with a correctly rounded division.
 * x0_hat and v_out must not overlap z or each other (the kernel reads and
 * writes them without re-reading): an overlap returns NEO_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------ */
neo_status neo_flow_euler_step(float* z, const float* x0_hat, int64_t n,
                               float t, float t_next, float t_eps,
                               float* v_out, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Classifier-free guidance fused with the Euler step.
 * [U1] section 2.7 (three-branch CFG of the inference loop): with the
 * conditional (c), text-unconditional (tu: images kept, text removed) and
 * unconditional (u) predictions, per-branch velocities
 * v_X = (x0_X - z) / max(1 - t, t_eps) and g = cfg_scale, g_img = img_cfg_scale:
 *   use_cfg = (lo < t < hi) || lo == 0        (cfg_interval = [lo, hi])
 *   NEO_CFG_NONE    (!use_cfg or g == g_img == 1): v = v_c
 *   NEO_CFG_TEXT    (g_img == 1):                  v = v_tu + g (v_c - v_tu)
 *   NEO_CFG_CLASSIC (g == g_img):                  v = v_u + g (v_c - v_u)
 *   NEO_CFG_DUAL    (otherwise):                   v = v_u + g (v_c - v_tu) + g_img (v_tu - v_u)
 * then z = z + (t_next - t) v. The branch is chosen on the host; only the
 * predictions it needs are read (the others may be NULL).
 *
 * z: fp32 [n] in place; x0_*: fp32 [n]; v_out: optional fp32 [n];
 * branch_out: optional HOST int32 receiving the branch taken.
 * Returns NEO_ERR_INVALID_ARG if a prediction the branch needs is NULL, or if
 * v_out overlaps z or a prediction the branch reads, or a prediction overlaps
 * z (predictions may share one buffer: they are only read).
 * ------------------------------------------------------------------------ */
#define NEO_CFG_NONE 0
#define NEO_CFG_TEXT 1
#define NEO_CFG_CLASSIC 2
#define NEO_CFG_DUAL 3

neo_status neo_flow_cfg_euler_step(float* z, const float* x0_cond,
                                   const float* x0_text_uncond,
                                   const float* x0_uncond, int64_t n, float t,
                                   float t_next, float t_eps, float cfg_scale,
                                   float img_cfg_scale, float cfg_interval_lo,
                                   float cfg_interval_hi, float* v_out,
                                   int32_t* branch_out, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Sampler pieces around the Euler step.
 *
 * neo_time_schedule: HOST computation of the shifted time grid
 * ([U15] section "Timestep schedule", "standard" branch). t_out (host,
 * n_steps + 1 floats) receives, for t_k = k / n_steps,
 *   sigma = 1 - t_k; sigma = shift*sigma / (1 + (shift-1)*sigma); t = 1 - sigma
 * (computed in double, rounded once). n_steps >= 1, shift > 0.
 *
 * neo_noise_scale: HOST computation of the resolution-dependent noise scale
 * ([U15] section "Timestep and noise-scale conditioning"; [U1] section 2.3):
 *   NEO_NOISE_RESOLUTION / NEO_NOISE_DYNAMIC:
 *       s = sqrt(grid_h * grid_w / merge^2 / base_seq_len) * base_scale
 *   NEO_NOISE_DYNAMIC_SQRT: sqrt of the above;  NEO_NOISE_CONSTANT: base_scale
 *   result = min(s, max_value) (16.0 in the export code) -> *out (host).
 * grid_h, grid_w count patches before the merge.
 *
 * neo_scale_noise: DEVICE z[i] = sigma * eps[i] for i < n (the initial sample
 * z_0 = sigma_R * eps; eps is the caller's standard-normal draw). z may alias
 * eps. fp32, 16-byte aligned.
 * ------------------------------------------------------------------------ */
#define NEO_NOISE_RESOLUTION 0
#define NEO_NOISE_DYNAMIC 1
#define NEO_NOISE_DYNAMIC_SQRT 2
#define NEO_NOISE_CONSTANT 3

neo_status neo_time_schedule(float* t_out, int n_steps, float shift);

neo_status neo_noise_scale(int grid_h, int grid_w, int merge, float base_seq_len,
                           float base_scale, int mode, float max_value,
                           float* out);

neo_status neo_scale_noise(float* z, const float* eps, int64_t n, float sigma,
                           cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Interleaved 2-D rotary embedding of the vision tower, in place.
 * [U15] section "Vision tower": on the patch features (C = 1024 channels in
 * the model), channels [0, C/2) turn with the patch's column index and
 * [C/2, C) with its row index; pairs (2i, 2i+1) share one angle (interleaved,
 * unlike the backbone's half split), base theta (1e4). Within a half of width
 * d = C/2, pair i turns by p * theta^(-2i/d):
 *   (u, w) -> (u cos a - w sin a, w cos a + u sin a).
 *
 * x: [n_images, rows * cols, C] of `dtype` (bf16 or fp32), patch
 * t = r * cols + c of each image; fp32 arithmetic, one rounding at the end.
 * C must be a multiple of 4 (of 8 for bf16).
 * ------------------------------------------------------------------------ */
neo_status neo_rope2d_interleaved(void* x, neo_dtype dtype, int64_t n_images,
                                  int rows, int cols, int C, float theta,
                                  cudaStream_t stream);

/* Human-readable name of a status code (static string). */
const char* neo_status_string(neo_status s);

/* Synchronises `stream`, then returns the current device's error word
 * accumulated by earlier launches on it in *word (NEO_DEVERR_* bits) and
 * clears it (each device has its own word). Returns
 * NEO_ERR_TIMEOUT if the timeout bit was set, NEO_ERR_DEVICE for any other
 * bit, NEO_OK if the word was zero, NEO_ERR_CUDA on a CUDA failure.
 * `word` may be NULL. */
neo_status neo_get_device_error(cudaStream_t stream, uint32_t* word);

/* Sets the time limit of every pipeline wait inside the kernels, in
 * nanoseconds (default 1e9), for the current device. Applies to launches
 * enqueued afterwards. Kernel attributes and occupancy-derived launch sizes
 * are set up once per device, the first time an entry point runs with that
 * device current. */
neo_status neo_set_wait_timeout_ns(uint64_t ns);

/* Self-test of the kernels' bounded waits: one thread waits on a barrier
 * that nothing arrives at; after the limit set by neo_set_wait_timeout_ns the
 * wait gives up and records NEO_DEVERR_TIMEOUT, which the next
 * neo_get_device_error returns as NEO_ERR_TIMEOUT. Nothing else is touched,
 * so the context stays usable. */
neo_status neo_selftest_bounded_wait(cudaStream_t stream);

/* ABI version of this header (major * 100 + minor). */
int neo_version(void);

#ifdef __cplusplus
}
#endif

#endif /* NEO_H */

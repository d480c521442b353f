"""fp64 CPU oracle of the NEO-unify generation-pass hot path.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the CPU legs of the
benchmark (its cpu_baseline and its reference arm) may import this module. The CUDA library never calls it and
it shares no code with the CUDA library.

Every function here is the plain definition of one step, written in float64
with NumPy. A library primitive (matmul, exp) may serve as one step; there is
no tiling, fusion or reordering beyond what the definition states. Inputs are
taken as exact real numbers: bf16 inputs are widened to float64 once and no
intermediate result is rounded.

Sources (cited by page title and section):
  [U15]  "SenseNova-U1.5 (NEO-unify) architecture" (ONNX Mobius design note)
  [U1]   "SenseNova-U1: Unifying Multimodal Understanding and Generation with
          NEO-unify Architecture" (paper walkthrough)

Readings where the pages are silent are marked READING and listed, with the
same labels, in the design notes of the repository.
"""

from __future__ import annotations

import numpy as np

# Slices of the 128-wide head and the rotary axis each one follows
# ([U15] §Three rotary axes, table): (offset, width, axis row of indexes[], base).
HEAD_DIM = 128
NORM_HALF = 64


def rope_slices(theta_t: float, theta_hw: float):
    """The three rotary slices of one 128-wide head ([U15] §Three rotary axes).

    [0:64) temporal/text axis, base rope_theta, position indexes[0];
    [64:96) image height, base rope_theta_hw, position indexes[1];
    [96:128) image width, base rope_theta_hw, position indexes[2].
    """
    return ((0, 64, 0, float(theta_t)),
            (64, 32, 1, float(theta_hw)),
            (96, 32, 2, float(theta_hw)))


# ---------------------------------------------------------------------------
# a0: position indexes
# ---------------------------------------------------------------------------
def positions(segments) -> np.ndarray:
    """Three-row position index ``indexes[3, S]`` for a token sequence.

    ``segments`` lists the sequence's parts in order:
      ("text", start, count): text tokens; token i gets (start+i, start+i, start+i)
          (every text token has its own temporal index, [U15] §Block-causal
          attention: "for a pure-text prompt every index is distinct";
          READING A0: its height/width indices equal the temporal one).
      ("image", t_index, rows, cols): one image of rows x cols tokens in
          row-major order; token r*cols + c gets (t_index, r, c). All tokens of
          one image share one temporal index and their height/width indices
          tile the token grid ([U15] §Three rotary axes, last paragraph;
          READING A7: row-major order, indices start at 0).
    """
    cols_out = []
    for seg in segments:
        kind = seg[0]
        if kind == "text":
            _, start, count = seg
            p = np.arange(start, start + count, dtype=np.int64)
            cols_out.append(np.stack([p, p, p]))
        elif kind == "image":
            _, t_index, rows, cols = seg
            r = np.repeat(np.arange(rows, dtype=np.int64), cols)
            c = np.tile(np.arange(cols, dtype=np.int64), rows)
            t = np.full(rows * cols, t_index, dtype=np.int64)
            cols_out.append(np.stack([t, r, c]))
        else:
            raise ValueError(f"unknown segment kind {kind!r}")
    if not cols_out:
        return np.zeros((3, 0), dtype=np.int64)
    return np.concatenate(cols_out, axis=1)


# ---------------------------------------------------------------------------
# a1: QK-norm applied to head halves
# ---------------------------------------------------------------------------
def qknorm_halves(x: np.ndarray, w_t: np.ndarray, w_hw: np.ndarray,
                  eps: float) -> np.ndarray:
    """RMS-normalise each half of every 128-wide head row separately.

    [U15] §Three rotary axes: the QK-norm acts on halves; ``q_norm``/``k_norm``
    (weight [64]) normalise dims [0:64) and ``q_norm_hw``/``k_norm_hw`` dims
    [64:128). READING A2: the Qwen3 RMSNorm form
    ``y = x / sqrt(mean(x^2) + eps) * w`` with a plain weight w.

    x: [..., 128] float64. Returns a new array of the same shape.
    """
    x = np.asarray(x, dtype=np.float64)
    assert x.shape[-1] == HEAD_DIM
    out = np.empty_like(x)
    for sl, w in ((slice(0, NORM_HALF), w_t), (slice(NORM_HALF, HEAD_DIM), w_hw)):
        h = x[..., sl]
        mean_sq = np.mean(h * h, axis=-1, keepdims=True)
        out[..., sl] = h / np.sqrt(mean_sq + eps) * np.asarray(w, np.float64)
    return out


# ---------------------------------------------------------------------------
# a2: three-axis rotary embedding
# ---------------------------------------------------------------------------
def rope3(y: np.ndarray, indexes: np.ndarray, theta_t: float,
          theta_hw: float) -> np.ndarray:
    """Apply the three-axis rotary embedding to rows of 128.

    [U15] §Three rotary axes (table) gives each slice's base and position
    source; §Vision tower says the language backbone pairs dimensions by the
    half-split convention. READING A1: the half split is taken within each
    slice: for a slice at offset o of width d with base theta, pair i < d/2
    joins dims (o+i, o+i+d/2) and turns by the angle p * theta^(-2i/d), with
    p that slice's position index:
        y'[o+i]       = u*cos(a) - w*sin(a)
        y'[o+i+d/2]   = w*cos(a) + u*sin(a),   (u, w) = (y[o+i], y[o+i+d/2]).

    y: [S, H, 128] float64; indexes: [3, S] integer. Returns a new array.
    """
    y = np.asarray(y, dtype=np.float64)
    idx = np.asarray(indexes, dtype=np.float64)
    S = y.shape[0]
    assert y.ndim == 3 and y.shape[-1] == HEAD_DIM and idx.shape == (3, S)
    out = y.copy()
    for off, width, axis, theta in rope_slices(theta_t, theta_hw):
        half = width // 2
        i = np.arange(half, dtype=np.float64)
        freq = theta ** (-2.0 * i / width)                 # [half]
        angle = idx[axis][:, None] * freq[None, :]         # [S, half]
        cos = np.cos(angle)[:, None, :]                    # [S, 1, half]
        sin = np.sin(angle)[:, None, :]
        u = y[:, :, off:off + half]
        w = y[:, :, off + half:off + width]
        out[:, :, off:off + half] = u * cos - w * sin
        out[:, :, off + half:off + width] = w * cos + u * sin
    return out


def qknorm_rope3(x, indexes, w_t, w_hw, theta_t=5e6, theta_hw=1e4, eps=1e-6):
    """QK-norm on halves, then the three-axis RoPE ([U15] §Three rotary axes:
    the norm acts "before the height/width split"; READING A3: norm first).

    x: [S, H, 128]; indexes: [3, S]. Returns float64 [S, H, 128].
    """
    return rope3(qknorm_halves(x, w_t, w_hw, eps), indexes, theta_t, theta_hw)


# ---------------------------------------------------------------------------
# a3: generation-pass attention over the frozen prefix plus the image tokens
# ---------------------------------------------------------------------------
MASK_FULL = 0
MASK_BLOCK_CAUSAL = 1


def gen_attention(q, k_prefix, v_prefix, k_img, v_img, cu_prefix, scale,
                  mask_mode=MASK_FULL, t_prefix=None, t_img=None, rows=None):
    """GQA attention of the image queries over [prefix keys ; image keys].

    [U15] §Mixture of Transformers, items 1-2: the generation pass reads the
    keys/values that the understanding pass wrote for the prefix and attends
    over them together with the image tokens' own keys/values, without writing
    the cache. §GQA fusion does not apply: the generation pass is unmasked
    (mask_mode 0). §Block-causal attention gives the mixed-prefill mask
    ``allowed(i, j) = (T_j == T_i) or (j <= i)`` over the concatenated order,
    mask_mode 1. READING A5: query head h reads KV head floor(h / (Hq/Hkv)).

    q: [B, N, Hq, D]; k_img, v_img: [B, N, Hkv, D]; k_prefix, v_prefix:
    [sum L_b, Hkv, D] packed by ``cu_prefix`` ([B+1], cu_prefix[0] = 0).
    For mask_mode 1, t_prefix [sum L_b] and t_img [B, N] are the temporal
    indices (indexes[0]) of the prefix and image tokens.
    rows: optional int array [R, 3] of (b, n, h) query rows to compute.

    Returns (out, lse): out [B, N, Hq, D] (or [R, D] when rows is given) and the
    natural-log sum of exp(logits) per query row, [B, Hq, N] (or [R]).
    """
    q = np.asarray(q, np.float64)
    k_prefix = np.asarray(k_prefix, np.float64)
    v_prefix = np.asarray(v_prefix, np.float64)
    k_img = np.asarray(k_img, np.float64)
    v_img = np.asarray(v_img, np.float64)
    cu = np.asarray(cu_prefix, np.int64)
    B, N, Hq, D = q.shape
    Hkv = k_img.shape[2]
    assert Hq % Hkv == 0
    group = Hq // Hkv

    if rows is None:
        sel = {(b, h): np.arange(N) for b in range(B) for h in range(Hq)}
    else:
        rows = np.asarray(rows, np.int64).reshape(-1, 3)
        sel = {}
        for r, (b, n, h) in enumerate(rows):
            sel.setdefault((int(b), int(h)), []).append((int(n), r))

    if rows is None:
        out = np.zeros((B, N, Hq, D))
        lse = np.zeros((B, Hq, N))
    else:
        out = np.zeros((len(rows), D))
        lse = np.zeros(len(rows))

    for (b, h), which in sel.items():
        kvh = h // group
        lo, hi = int(cu[b]), int(cu[b + 1])
        L = hi - lo
        keys = np.concatenate([k_prefix[lo:hi, kvh, :], k_img[b, :, kvh, :]], axis=0)
        vals = np.concatenate([v_prefix[lo:hi, kvh, :], v_img[b, :, kvh, :]], axis=0)
        if rows is None:
            n_idx = np.asarray(which)
        else:
            n_idx = np.asarray([n for n, _ in which])
        logits = scale * (q[b, n_idx, h, :] @ keys.T)          # [R_bh, L+N]
        if mask_mode == MASK_BLOCK_CAUSAL:
            t_keys = np.concatenate([np.asarray(t_prefix)[lo:hi],
                                     np.asarray(t_img)[b]]).astype(np.int64)
            i = L + n_idx                                      # query position
            j = np.arange(L + N)                               # key position
            allowed = (t_keys[None, :] == t_keys[i][:, None]) | (j[None, :] <= i[:, None])
            logits = np.where(allowed, logits, -np.inf)
        elif mask_mode != MASK_FULL:
            raise ValueError("mask_mode must be 0 or 1")
        m = np.max(logits, axis=1, keepdims=True)
        e = np.exp(logits - m)
        s = np.sum(e, axis=1, keepdims=True)
        o = (e @ vals) / s
        row_lse = (m + np.log(s))[:, 0]
        if rows is None:
            out[b, n_idx, h, :] = o
            lse[b, h, n_idx] = row_lse
        else:
            dst = np.asarray([r for _, r in which])
            out[dst] = o
            lse[dst] = row_lse
    return out, lse


# ---------------------------------------------------------------------------
# a4: x0 -> velocity conversion and the Euler step
# ---------------------------------------------------------------------------
def write_prefix_cache(k_old, v_old, cu_old, k_new, v_new, n_new):
    """Append a chunk of keys/values to a packed per-sequence prefix cache.

    [U15] §Mixture of Transformers, item 1: the understanding pass (a prefill,
    possibly in chunks) writes the keys/values of its tokens into a KV cache
    that the generation passes then read. [U1] §4.4 (KV-cache reuse): the
    prefix cache is laid out once in the [B, S, H, D] form the attention
    reads; here that form is packed without padding, sequence b owning rows
    cu[b] .. cu[b+1]-1.

    k_old, v_old: [cu_old[B], Hkv, D]; k_new, v_new: [B, N, Hkv, D], of which
    sequence b contributes its first n_new[b] rows (its chunk), in order,
    after its old rows. Returns (k_out, v_out, cu_out).
    """
    cu_old = np.asarray(cu_old, np.int64)
    B = len(cu_old) - 1
    ks, vs, cu = [], [], [0]
    for b in range(B):
        lo, hi = int(cu_old[b]), int(cu_old[b + 1])
        n = int(n_new[b])
        ks += [np.asarray(k_old)[lo:hi], np.asarray(k_new)[b, :n]]
        vs += [np.asarray(v_old)[lo:hi], np.asarray(v_new)[b, :n]]
        cu.append(cu[-1] + (hi - lo) + n)
    return np.concatenate(ks), np.concatenate(vs), np.asarray(cu, np.int64)


def flow_euler_step(z, x0_hat, t, t_next, t_eps=0.02):
    """One sampler step of the pixel-space rectified flow.

    [U15] §Flow matching without a VAE: the head predicts x0; the sampler forms
    ``v = (x0 - z) / max(1 - t, t_eps)`` and steps ``z = z + (t_next - t) * v``.
    [U15] §Dead or misleading upstream details: inference uses t_eps = 0.02.
    [U1] §2.7: the ODE is solved with Euler steps z_{t+dt} = z_t + dt * v.

    Returns (z_next, v) in float64.
    """
    z = np.asarray(z, np.float64)
    x0_hat = np.asarray(x0_hat, np.float64)
    v = (x0_hat - z) / max(1.0 - float(t), float(t_eps))
    return z + (float(t_next) - float(t)) * v, v


def flow_interpolant(x, noise, t, sigma):
    """Rectified-flow noisy sample z_t = t * x + (1 - t) * sigma * noise.

    [U1] §2.2 (formula lost in extraction). READING A10: the only linear
    interpolation consistent with the worked example printed there
    (t = 0.6, x = 1, noise = 0, sigma = 1 gives z_t = 0.6) and with the target
    velocity v* = (x - z_t) / (1 - t).
    """
    return t * np.asarray(x, np.float64) + (1.0 - t) * sigma * np.asarray(noise, np.float64)


def flow_target_velocity(x, z_t, t):
    """Training target v* = (x - z_t) / (1 - t) ([U1] §2.2)."""
    return (np.asarray(x, np.float64) - np.asarray(z_t, np.float64)) / (1.0 - t)


# ---------------------------------------------------------------------------
# NEXT: classifier-free guidance fused with the Euler step
# ---------------------------------------------------------------------------
CFG_NONE, CFG_TEXT, CFG_CLASSIC, CFG_DUAL = 0, 1, 2, 3


def cfg_branch(t, cfg_scale, img_cfg_scale, cfg_interval=(0.0, 1.0)):
    """Which of the four inference branches of [U1] §2.7 applies at time t.

    use_cfg = (interval[0] < t < interval[1]) or interval[0] == 0;
    no CFG (or both scales 1) -> 0; img_cfg_scale == 1 -> 1 (text CFG against
    the text-unconditional branch); cfg_scale == img_cfg_scale -> 2 (classic
    CFG against the fully unconditional branch); otherwise -> 3 (both).
    """
    lo, hi = cfg_interval
    use_cfg = (lo < t < hi) or lo == 0
    if not use_cfg or (cfg_scale == 1 and img_cfg_scale == 1):
        return CFG_NONE
    if img_cfg_scale == 1:
        return CFG_TEXT
    if cfg_scale == img_cfg_scale:
        return CFG_CLASSIC
    return CFG_DUAL


def flow_cfg_euler_step(z, x0_cond, x0_text_uncond, x0_uncond, t, t_next, cfg_scale, img_cfg_scale,
                        cfg_interval=(0.0, 1.0), t_eps=0.02):
    """Guided velocity and Euler step ([U1] §2.7, three-branch CFG; [U15]
    §Flow matching without a VAE for x0 -> v).

    Each branch's x0 prediction becomes a velocity v_X = (x0_X - z) / max(1 - t,
    t_eps); the branches combine as
      0: v = v_c
      1: v = v_tu + g (v_c - v_tu)
      2: v = v_u + g (v_c - v_u)
      3: v = v_u + g (v_c - v_tu) + g_img (v_tu - v_u)
    with g = cfg_scale, g_img = img_cfg_scale, c = conditional, tu = text
    unconditional (image kept), u = unconditional; then z += (t_next - t) v.
    Returns (z_next, v, branch).
    """
    z = np.asarray(z, np.float64)
    den = max(1.0 - float(t), float(t_eps))
    vel = lambda x0: (np.asarray(x0, np.float64) - z) / den
    g, gi = float(cfg_scale), float(img_cfg_scale)
    branch = cfg_branch(float(t), g, gi, cfg_interval)
    v_c = vel(x0_cond)
    if branch == CFG_NONE:
        v = v_c
    elif branch == CFG_TEXT:
        v_tu = vel(x0_text_uncond)
        v = v_tu + g * (v_c - v_tu)
    elif branch == CFG_CLASSIC:
        v_u = vel(x0_uncond)
        v = v_u + g * (v_c - v_u)
    else:
        v_tu, v_u = vel(x0_text_uncond), vel(x0_uncond)
        v = v_u + g * (v_c - v_tu) + gi * (v_tu - v_u)
    return z + (float(t_next) - float(t)) * v, v, branch


# ---------------------------------------------------------------------------
# NEXT: sampler pieces (time grid, resolution-dependent noise scale)
# ---------------------------------------------------------------------------
def time_schedule(n_steps, shift):
    """Shifted time grid of the sampler ([U15] §Timestep schedule, "standard"
    branch): every point of the uniform grid t_k = k / n_steps (READING A14:
    n_steps + 1 points from 0 to 1) is mapped by
        sigma = 1 - t;  sigma = shift * sigma / (1 + (shift - 1) * sigma);  t = 1 - sigma.
    """
    out = []
    for k in range(n_steps + 1):
        t = k / n_steps
        sigma = 1.0 - t
        sigma = shift * sigma / (1.0 + (shift - 1.0) * sigma)
        out.append(1.0 - sigma)
    return np.asarray(out, np.float64)


NOISE_RESOLUTION, NOISE_DYNAMIC, NOISE_DYNAMIC_SQRT, NOISE_CONSTANT = 0, 1, 2, 3


def noise_scale(grid_h, grid_w, merge, base_seq_len, base_scale, mode, max_value=16.0):
    """Resolution-dependent noise scale sigma_R ([U15] §Timestep and
    noise-scale conditioning; [U1] §2.3): in the resolution / dynamic modes
    sigma = sqrt(grid_h * grid_w / merge^2 / base_seq_len) * base_scale, the
    dynamic_sqrt mode takes one more square root of that, the constant mode
    keeps base_scale; the result is capped at max_value (16.0 in the export
    code; READING A9: the cap is a parameter). grid_h, grid_w count patches
    before the merge, so grid_h * grid_w / merge^2 is the token count N."""
    s = float(base_scale)
    if mode in (NOISE_RESOLUTION, NOISE_DYNAMIC, NOISE_DYNAMIC_SQRT):
        s = np.sqrt(grid_h * grid_w / merge ** 2 / float(base_seq_len)) * float(base_scale)
        if mode == NOISE_DYNAMIC_SQRT:
            s = np.sqrt(s)
    return float(min(s, float(max_value)))


def initial_noise(eps, sigma):
    """z_0 = sigma_R * eps ([U1] §2.3: the initial sample is the scaled
    standard normal draw)."""
    return float(sigma) * np.asarray(eps, np.float64)


# ---------------------------------------------------------------------------
# NEXT: interleaved 2-D rotary embedding of the vision tower
# ---------------------------------------------------------------------------
def rope2d_interleaved(x, rows, cols, theta=1e4):
    """Interleaved 2-D RoPE of the patch features ([U15] §Vision tower).

    x: [n_images, rows * cols, C] with patch t = r * cols + c. Channels
    [0, C/2) turn with the patch's column (x) index and [C/2, C) with its row
    (y) index; the rotation is interleaved: pair (2i, 2i+1) of a half shares
    one angle. READING A15: within a half of width d = C/2, pair i turns by
    p * theta^(-2i/d) (the standard RoPE frequencies over that half), with
        (u, w) -> (u cos a - w sin a, w cos a + u sin a),  (u, w) = (x[2i], x[2i+1]).
    Returns a new float64 array.
    """
    x = np.asarray(x, np.float64)
    n_img, T, C = x.shape
    assert T == rows * cols and C % 4 == 0
    d = C // 2
    r = np.repeat(np.arange(rows, dtype=np.float64), cols)
    c = np.tile(np.arange(cols, dtype=np.float64), rows)
    i = np.arange(d // 2, dtype=np.float64)
    freq = theta ** (-2.0 * i / d)
    out = x.copy()
    for off, pos in ((0, c), (d, r)):
        a = pos[:, None] * freq[None, :]                    # [T, d/2]
        cos, sin = np.cos(a)[None], np.sin(a)[None]
        u = x[:, :, off:off + d:2]
        w = x[:, :, off + 1:off + d:2]
        out[:, :, off:off + d:2] = u * cos - w * sin
        out[:, :, off + 1:off + d:2] = w * cos + u * sin
    return out

"""Pins of the fp64 oracle against facts fixed outside the oracle itself:
values printed on the pages, closed forms, invariants, special cases that
reduce to a library routine. No GPU."""

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def _rows(S, H, seed=0):
    return np.random.default_rng(seed).standard_normal((S, H, 128))


# ---------------------------------------------------------------- positions
def test_positions_image_grid_row_major_shared_temporal():
    idx = O.positions([("image", 77, 3, 5)])
    assert idx.shape == (3, 15)
    assert (idx[0] == 77).all()                       # one temporal index per image
    grid = {(int(r), int(c)) for r, c in zip(idx[1], idx[2])}
    assert grid == {(r, c) for r in range(3) for c in range(5)}   # tiles the grid
    assert idx[1, 7] == 1 and idx[2, 7] == 2           # token r*cols + c


def test_positions_text_then_image():
    idx = O.positions([("text", 0, 4), ("image", 4, 2, 2)])
    np.testing.assert_array_equal(idx[:, :4], np.array([[0, 1, 2, 3]] * 3))
    np.testing.assert_array_equal(idx[:, 4:], np.array([[4, 4, 4, 4], [0, 0, 1, 1], [0, 1, 0, 1]]))


# ---------------------------------------------------------------- QK-norm
def test_norm_matches_torch_rms_norm_per_half():
    """Library pin: torch's RMSNorm (x * rsqrt(mean x^2 + eps) * w) per half."""
    x = _rows(9, 3)
    w_t, w_hw = rng.uniform(0.5, 1.5, 64), rng.uniform(0.5, 1.5, 64)
    eps = 1e-6
    y = O.qknorm_halves(x, w_t, w_hw, eps)
    xt = torch.from_numpy(x)
    ref_t = F.rms_norm(xt[..., :64], (64,), weight=torch.from_numpy(w_t), eps=eps)
    ref_hw = F.rms_norm(xt[..., 64:], (64,), weight=torch.from_numpy(w_hw), eps=eps)
    np.testing.assert_allclose(y[..., :64], ref_t.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(y[..., 64:], ref_hw.numpy(), rtol=1e-12, atol=1e-13)


def test_norm_half_rms_equals_constant_weight():
    """Closed form: with w = c the normed half has RMS c * sqrt(ms / (ms + eps))."""
    x = _rows(5, 2, seed=3) * 3.0
    c_t, c_hw, eps = 0.7, 1.3, 1e-6
    y = O.qknorm_halves(x, np.full(64, c_t), np.full(64, c_hw), eps)
    for sl, c in ((slice(0, 64), c_t), (slice(64, 128), c_hw)):
        ms = np.mean(x[..., sl] ** 2, axis=-1)
        rms = np.sqrt(np.mean(y[..., sl] ** 2, axis=-1))
        np.testing.assert_allclose(rms, c * np.sqrt(ms / (ms + eps)), rtol=1e-13)
    y0 = O.qknorm_halves(x, np.full(64, c_t), np.full(64, c_hw), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y0[..., :64] ** 2, -1)), c_t, rtol=1e-13)


def test_norm_halves_are_independent_and_scale_invariant():
    x = _rows(4, 2, seed=5)
    w = np.ones(64)
    y = O.qknorm_halves(x, w, w, 0.0)
    x2 = x.copy()
    x2[..., 64:] *= 1000.0                             # rescale only the spatial half
    y2 = O.qknorm_halves(x2, w, w, 0.0)
    np.testing.assert_allclose(y2, y, rtol=1e-12, atol=1e-14)
    # weights act on their own half only
    yz = O.qknorm_halves(x, np.zeros(64), w, 1e-6)
    assert np.all(yz[..., :64] == 0) and np.all(yz[..., 64:] != 0)


# ---------------------------------------------------------------- RoPE
def _rot(y, idx, tt=5e6, thw=1e4):
    return O.rope3(y, idx, tt, thw)


def test_rope_identity_at_position_zero():
    y = _rows(6, 2, seed=7)
    np.testing.assert_array_equal(_rot(y, np.zeros((3, 6), np.int64)), y)


def test_rope_preserves_each_pair_norm():
    y = _rows(10, 3, seed=8)
    idx = rng.integers(0, 7000, size=(3, 10))
    r = _rot(y, idx)
    for off, width, _, _ in O.rope_slices(5e6, 1e4):
        h = width // 2
        n0 = y[..., off:off + h] ** 2 + y[..., off + h:off + width] ** 2
        n1 = r[..., off:off + h] ** 2 + r[..., off + h:off + width] ** 2
        np.testing.assert_allclose(n1, n0, rtol=1e-12)


def test_rope_relative_position_per_axis():
    """<R(p)q, R(p')k> per slice depends only on p - p', for each axis alone."""
    q = _rows(1, 1, seed=9)
    k = _rows(1, 1, seed=10)
    p_q = np.array([[1234], [17], [40]])
    p_k = np.array([[1000], [3], [61]])
    shift = np.array([[3333], [250], [7]])
    rq, rk = _rot(q, p_q), _rot(k, p_k)
    rq2, rk2 = _rot(q, p_q + shift), _rot(k, p_k + shift)
    for off, width, _, _ in O.rope_slices(5e6, 1e4):
        sl = slice(off, off + width)
        np.testing.assert_allclose(np.sum(rq[..., sl] * rk[..., sl]),
                                   np.sum(rq2[..., sl] * rk2[..., sl]), rtol=1e-10)


def test_rope_each_axis_moves_only_its_slice():
    y = _rows(3, 2, seed=11)
    base = np.zeros((3, 3), np.int64)
    for axis, (lo, hi) in enumerate(((0, 64), (64, 96), (96, 128))):
        idx = base.copy()
        idx[axis] = 5
        r = _rot(y, idx)
        changed = np.any(r != y, axis=(0, 1))
        assert changed[lo:hi].all()
        assert not changed[:lo].any() and not changed[hi:].any()


def test_rope_is_complex_rotation_with_geometric_frequencies():
    """Each pair (u, w) of a slice is the complex number u + i*w multiplied by
    exp(i * p * f_i); the frequencies start at 1 and fall geometrically by
    theta^(-2/width), reaching theta^(-1) one step past the last pair."""
    tt, thw = 5e6, 1e4
    for off, width, axis, theta in O.rope_slices(tt, thw):
        h = width // 2
        y = np.zeros((1, 1, 128))
        y[0, 0, off:off + h] = 1.0                       # u = 1, w = 0 on every pair
        idx = np.zeros((3, 1), np.int64)
        idx[axis] = 1                                    # position 1: angle = f_i
        r = _rot(y, idx, tt, thw)
        zc = r[0, 0, off:off + h] + 1j * r[0, 0, off + h:off + width]
        f = np.angle(zc)
        assert f[0] == pytest.approx(1.0, rel=1e-14)
        ratio = f[1:] / f[:-1]
        np.testing.assert_allclose(ratio, theta ** (-2.0 / width), rtol=1e-12)
        assert f[-1] * theta ** (-2.0 / width) == pytest.approx(1.0 / theta, rel=1e-12)
        # at a large position the rotation is exp(i * p * f) of an arbitrary pair
        p = 4096 if axis == 0 else 63
        u, w = 0.3, -1.7
        y2 = np.zeros((1, 1, 128))
        y2[0, 0, off:off + h] = u
        y2[0, 0, off + h:off + width] = w
        idx2 = np.zeros((3, 1), np.int64)
        idx2[axis] = p
        r2 = _rot(y2, idx2, tt, thw)
        expect = (u + 1j * w) * np.exp(1j * p * f)
        np.testing.assert_allclose(r2[0, 0, off:off + h], expect.real, atol=1e-9)
        np.testing.assert_allclose(r2[0, 0, off + h:off + width], expect.imag, atol=1e-9)


def test_rope_landmark_frequencies():
    """Height slice (width 32, base 1e4): pair 8 has frequency 1e4^(-1/2) = 0.01,
    so position 100 turns it by exactly one radian; temporal slice (width 64,
    base 5e6): pair 16 has frequency 5e6^(-1/2)."""
    y = np.zeros((1, 1, 128))
    y[0, 0, 64 + 8] = 1.0
    r = _rot(y, np.array([[0], [100], [0]]))
    assert r[0, 0, 64 + 8] == pytest.approx(math.cos(1.0), abs=1e-13)
    assert r[0, 0, 64 + 16 + 8] == pytest.approx(math.sin(1.0), abs=1e-13)
    y = np.zeros((1, 1, 128))
    y[0, 0, 16] = 1.0
    p = round(math.sqrt(5e6))
    r = _rot(y, np.array([[p], [0], [0]]))
    a = p / math.sqrt(5e6)
    assert r[0, 0, 16] == pytest.approx(math.cos(a), abs=1e-12)
    assert r[0, 0, 48] == pytest.approx(math.sin(a), abs=1e-12)


def test_rope_temporal_slice_cancels_between_tokens_of_one_image():
    """Image tokens share one temporal index, so their temporal-slice dot
    product equals the unrotated one."""
    y = _rows(6, 1, seed=12)
    idx = O.positions([("image", 1536, 2, 3)])
    r = O.qknorm_rope3(y, idx, np.ones(64), np.ones(64))
    n = O.qknorm_halves(y, np.ones(64), np.ones(64), 1e-6)
    np.testing.assert_allclose(r[:, 0, :64] @ r[:, 0, :64].T, n[:, 0, :64] @ n[:, 0, :64].T, rtol=1e-10)


# ---------------------------------------------------------------- attention
def _attn_case(B=2, Ls=(5, 0), N=7, Hq=4, Hkv=2, D=128, seed=20):
    g = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(Ls)]).astype(np.int64)
    q = g.standard_normal((B, N, Hq, D))
    kp = g.standard_normal((cu[-1], Hkv, D))
    vp = g.standard_normal((cu[-1], Hkv, D))
    ki = g.standard_normal((B, N, Hkv, D))
    vi = g.standard_normal((B, N, Hkv, D))
    return q, kp, vp, ki, vi, cu


def test_attention_matches_torch_sdpa_gqa():
    """Library pin: torch scaled_dot_product_attention in float64 over the
    concatenated keys, with each KV head repeated for its query-head group."""
    q, kp, vp, ki, vi, cu = _attn_case(B=3, Ls=(5, 0, 9), N=7, Hq=6, Hkv=2)
    scale = 1 / math.sqrt(128)
    out, lse = O.gen_attention(q, kp, vp, ki, vi, cu, scale)
    for b in range(3):
        K = np.concatenate([kp[cu[b]:cu[b + 1]], ki[b]], 0)     # [L+N, Hkv, D]
        V = np.concatenate([vp[cu[b]:cu[b + 1]], vi[b]], 0)
        Kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(3, dim=0)
        Vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(3, dim=0)
        Qt = torch.from_numpy(q[b]).permute(1, 0, 2)
        ref = F.scaled_dot_product_attention(Qt, Kt, Vt, scale=scale)
        np.testing.assert_allclose(out[b], ref.permute(1, 0, 2).numpy(), rtol=1e-11, atol=1e-12)
        ref_lse = torch.logsumexp(scale * Qt @ Kt.transpose(1, 2), dim=-1)
        np.testing.assert_allclose(lse[b], ref_lse.numpy(), rtol=1e-12)


def test_attention_single_key_returns_value():
    q, kp, vp, ki, vi, cu = _attn_case(B=1, Ls=(0,), N=1, Hq=4, Hkv=1)
    out, _ = O.gen_attention(q, kp, vp, ki, vi, cu, 0.3)
    for h in range(4):
        np.testing.assert_allclose(out[0, 0, h], vi[0, 0, 0], rtol=1e-14)


def test_attention_equal_keys_or_zero_scale_give_mean_value():
    q, kp, vp, ki, vi, cu = _attn_case(B=1, Ls=(6,), N=5, Hq=2, Hkv=1)
    mean_v = np.concatenate([vp[:, 0], vi[0, :, 0]]).mean(0)
    out, _ = O.gen_attention(q, kp, vp, ki, vi, cu, 0.0)
    np.testing.assert_allclose(out[0, :, 0], np.broadcast_to(mean_v, (5, 128)), rtol=1e-12)
    same_kp = np.broadcast_to(ki[0, 0], kp.shape).copy()
    same_ki = np.broadcast_to(ki[0, 0], ki.shape).copy()
    out, _ = O.gen_attention(q, same_kp, vp, same_ki, vi, cu, 0.5)
    np.testing.assert_allclose(out[0, :, 1], np.broadcast_to(mean_v, (5, 128)), rtol=1e-12)


def test_attention_prefix_permutation_and_common_key_shift():
    q, kp, vp, ki, vi, cu = _attn_case(B=2, Ls=(8, 3), N=4, Hq=4, Hkv=2, seed=21)
    out, _ = O.gen_attention(q, kp, vp, ki, vi, cu, 0.2)
    perm = np.concatenate([np.random.default_rng(0).permutation(8), 8 + np.arange(3)[::-1]])
    out_p, _ = O.gen_attention(q, kp[perm], vp[perm], ki, vi, cu, 0.2)
    np.testing.assert_allclose(out_p, out, rtol=1e-12)
    c = np.random.default_rng(1).standard_normal(128)     # same vector added to every key
    out_s, _ = O.gen_attention(q, kp + c, vp, ki + c, vi, cu, 0.2)
    np.testing.assert_allclose(out_s, out, rtol=1e-10, atol=1e-12)


def test_attention_gqa_equals_mha_with_repeated_kv():
    q, kp, vp, ki, vi, cu = _attn_case(B=2, Ls=(3, 6), N=5, Hq=8, Hkv=2, seed=22)
    out, _ = O.gen_attention(q, kp, vp, ki, vi, cu, 0.1)
    rep = lambda a: np.repeat(a, 4, axis=-2)
    out_m, _ = O.gen_attention(q, rep(kp), rep(vp), rep(ki), rep(vi), cu, 0.1)
    np.testing.assert_allclose(out_m, out, rtol=1e-13)


def test_block_causal_with_generation_positions_equals_full_mask():
    """Prefix keys precede every query and the image keys share the queries'
    temporal index, so the block-causal mask allows everything."""
    q, kp, vp, ki, vi, cu = _attn_case(B=2, Ls=(6, 4), N=9, Hq=4, Hkv=1, seed=23)
    t_pre = np.concatenate([np.arange(6), np.arange(4)])
    t_img = np.array([[6] * 9, [4] * 9])
    full, _ = O.gen_attention(q, kp, vp, ki, vi, cu, 0.15)
    bc, _ = O.gen_attention(q, kp, vp, ki, vi, cu, 0.15, mask_mode=1, t_prefix=t_pre, t_img=t_img)
    np.testing.assert_allclose(bc, full, rtol=1e-13)


def test_block_causal_with_distinct_indices_is_plain_causal():
    """With every temporal index distinct the block-causal mask degenerates to
    the plain causal mask (stated on the architecture page); pinned against
    torch's causal scaled_dot_product_attention."""
    q, kp, vp, ki, vi, cu = _attn_case(B=1, Ls=(0,), N=11, Hq=2, Hkv=1, seed=24)
    t_img = np.arange(11)[None, :]
    out, _ = O.gen_attention(q, kp, vp, ki, vi, cu, 0.25, mask_mode=1,
                             t_prefix=np.zeros(0, np.int64), t_img=t_img)
    Q = torch.from_numpy(q[0]).permute(1, 0, 2)
    K = torch.from_numpy(ki[0]).permute(1, 0, 2).expand(2, -1, -1)
    V = torch.from_numpy(vi[0]).permute(1, 0, 2).expand(2, -1, -1)
    ref = F.scaled_dot_product_attention(Q, K, V, is_causal=True, scale=0.25)
    np.testing.assert_allclose(out[0], ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-13)


def test_block_causal_visible_sets_with_temporal_indexes_out_of_order():
    """Hand-checked visible sets of the block-causal rule with temporal indexes
    that are not in order ("SenseNova-U1.5" §Block-causal attention: tokens
    that share a temporal index see each other both ways; across differing
    indexes ordinary causality holds). Prefix of two keys (T = 0, 1), image
    segment of four tokens (T = 4, 2, 4, 3), so over the concatenated order
    T = [0, 1, 4, 2, 4, 3]. With scale 0 every visible key gets the same
    weight, and one-hot values make the output the indicator of the visible
    set divided by its size. A rule of T_j <= T_i would let query 2 (T = 4)
    see keys 3 and 5 and hide key 2 from query 3 (T = 2)."""
    D = 128
    g = np.random.default_rng(31)
    q = g.standard_normal((1, 4, 1, D))
    kp, ki = g.standard_normal((2, 1, D)), g.standard_normal((1, 4, 1, D))
    eye = np.eye(D)
    vp = eye[:2].reshape(2, 1, D)
    vi = eye[2:6].reshape(1, 4, 1, D)
    out, _ = O.gen_attention(q, kp, vp, ki, vi, np.array([0, 2]), 0.0, mask_mode=O.MASK_BLOCK_CAUSAL,
                             t_prefix=np.array([0, 1]), t_img=np.array([[4, 2, 4, 3]]))
    visible = {0: [0, 1, 2, 4], 1: [0, 1, 2, 3], 2: [0, 1, 2, 3, 4], 3: [0, 1, 2, 3, 4, 5]}
    for n, keys in visible.items():
        want = np.zeros(D)
        want[keys] = 1.0 / len(keys)
        np.testing.assert_allclose(out[0, n, 0], want, rtol=0, atol=1e-15, err_msg=f"query {n}")


def test_attention_sampled_rows_match_full():
    q, kp, vp, ki, vi, cu = _attn_case(B=2, Ls=(7, 2), N=6, Hq=4, Hkv=2, seed=25)
    full, full_lse = O.gen_attention(q, kp, vp, ki, vi, cu, 0.3)
    rows = np.array([[1, 5, 3], [0, 0, 0], [1, 2, 1], [0, 4, 2]])
    part, part_lse = O.gen_attention(q, kp, vp, ki, vi, cu, 0.3, rows=rows)
    for r, (b, n, h) in enumerate(rows):
        np.testing.assert_allclose(part[r], full[b, n, h], rtol=1e-13, atol=1e-15)
        assert part_lse[r] == pytest.approx(full_lse[b, h, n], rel=1e-14)


# ---------------------------------------------------------------- flow step
def test_flow_worked_example_from_the_pages():
    g = json.load(open(os.path.join(GOLDEN, "flow_worked_example.json")))
    z_t = O.flow_interpolant(g["x"], g["eps"], g["t"], g["sigma_R"])
    assert float(z_t) == pytest.approx(g["z_t"], abs=1e-15)
    assert float(O.flow_target_velocity(g["x"], z_t, g["t"])) == pytest.approx(g["v"], rel=1e-14)
    z_next, v = O.flow_euler_step(z_t, g["x"], g["t"], g["t"] + 0.1)
    assert float(v) == pytest.approx(g["v"], rel=1e-14)
    assert float(z_next) == pytest.approx(0.7, abs=1e-15)


def test_flow_euler_lands_on_the_straight_path():
    """If x0_hat equals the clean x, one step from z_t lands on z_{t_next};
    ten steps of 0.1 from pure noise land on x."""
    g = np.random.default_rng(30)
    x, noise = g.standard_normal(1000), g.standard_normal(1000)
    for t, tn in ((0.0, 0.1), (0.35, 0.6), (0.8, 0.9)):
        z_next, _ = O.flow_euler_step(O.flow_interpolant(x, noise, t, 2.0), x, t, tn)
        np.testing.assert_allclose(z_next, O.flow_interpolant(x, noise, tn, 2.0), rtol=1e-12, atol=1e-13)
    z = O.flow_interpolant(x, noise, 0.0, 3.0)
    for k in range(10):
        z, _ = O.flow_euler_step(z, x, k / 10, (k + 1) / 10)
    np.testing.assert_allclose(z, x, atol=1e-12)


def test_flow_t_eps_clamp_and_elementwise_permutation():
    z, x = np.array([0.5, -2.0, 1.0]), np.array([1.5, 0.0, 1.0])
    _, v = O.flow_euler_step(z, x, 0.99, 1.0, t_eps=0.02)
    np.testing.assert_allclose(v, (x - z) / 0.02, rtol=1e-15)
    _, v = O.flow_euler_step(z, x, 0.5, 0.6, t_eps=0.02)
    np.testing.assert_allclose(v, (x - z) / 0.5, rtol=1e-15)
    g = np.random.default_rng(31)
    z, x = g.standard_normal(48), g.standard_normal(48)
    perm = g.permutation(48)
    a, _ = O.flow_euler_step(z, x, 0.2, 0.3)
    b, _ = O.flow_euler_step(z[perm], x[perm], 0.2, 0.3)
    np.testing.assert_array_equal(a[perm], b)


# ---------------------------------------------------------------- CFG + Euler
def _cfg_inputs(n=64, seed=40):
    g = np.random.default_rng(seed)
    return g.standard_normal(n), g.standard_normal(n), g.standard_normal(n), g.standard_normal(n)


def test_cfg_branch_selection_follows_the_pages():
    """Branches of the inference loop: no CFG, text CFG (img scale 1), classic
    (equal scales), dual; the interval gates CFG unless its start is 0."""
    assert O.cfg_branch(0.5, 4.0, 1.0) == O.CFG_TEXT          # the T2I default (4.0, 1.0)
    assert O.cfg_branch(0.5, 1.0, 1.0) == O.CFG_NONE
    assert O.cfg_branch(0.5, 3.0, 3.0) == O.CFG_CLASSIC
    assert O.cfg_branch(0.5, 4.0, 1.5) == O.CFG_DUAL
    assert O.cfg_branch(0.5, 4.0, 1.5, (0.6, 1.0)) == O.CFG_NONE
    assert O.cfg_branch(0.7, 4.0, 1.5, (0.6, 1.0)) == O.CFG_DUAL
    assert O.cfg_branch(0.6, 4.0, 1.5, (0.6, 1.0)) == O.CFG_NONE    # strict bounds
    assert O.cfg_branch(0.95, 4.0, 1.5, (0.0, 0.5)) == O.CFG_DUAL    # start 0: always on


def test_cfg_none_is_the_plain_euler_step():
    z, c, tu, u = _cfg_inputs()
    zc, vc, br = O.flow_cfg_euler_step(z, c, tu, u, 0.3, 0.4, 1.0, 1.0)
    ze, ve = O.flow_euler_step(z, c, 0.3, 0.4)
    assert br == O.CFG_NONE
    np.testing.assert_array_equal(zc, ze)
    np.testing.assert_array_equal(vc, ve)


def test_cfg_text_branch_is_an_affine_blend():
    """The page notes the text-CFG branch equals (1 - g) * v_tu + g * v_c."""
    z, c, tu, u = _cfg_inputs(seed=41)
    t, g = 0.45, 4.0
    _, v, _ = O.flow_cfg_euler_step(z, c, tu, u, t, t + 0.1, g, 1.0)
    _, vc = O.flow_euler_step(z, c, t, t + 0.1)
    _, vtu = O.flow_euler_step(z, tu, t, t + 0.1)
    np.testing.assert_allclose(v, (1 - g) * vtu + g * vc, rtol=1e-12, atol=1e-12)


def test_cfg_dual_reduces_to_the_two_scale_branches():
    """Eq. 6 with img scale 1 is the text branch; with equal scales it is the
    classic branch; guidance weights sum to one, so a common x0 gives the
    unguided step."""
    z, c, tu, u = _cfg_inputs(seed=42)
    t = 0.2
    den = 1 - t
    vc, vtu, vu = (c - z) / den, (tu - z) / den, (u - z) / den
    dual = lambda g, gi: vu + g * (vc - vtu) + gi * (vtu - vu)
    np.testing.assert_allclose(dual(3.0, 1.0), vtu + 3.0 * (vc - vtu), rtol=1e-12)
    np.testing.assert_allclose(dual(2.5, 2.5), vu + 2.5 * (vc - vu), rtol=1e-12)
    _, v, br = O.flow_cfg_euler_step(z, c, tu, u, t, t + 0.1, 3.0, 1.7)
    assert br == O.CFG_DUAL
    np.testing.assert_allclose(v, dual(3.0, 1.7), rtol=1e-12, atol=1e-12)
    zs, _, _ = O.flow_cfg_euler_step(z, c, c, c, t, t + 0.1, 3.0, 1.7)
    ze, _ = O.flow_euler_step(z, c, t, t + 0.1)
    np.testing.assert_allclose(zs, ze, rtol=1e-12, atol=1e-12)


def test_cfg_branches_on_a_hand_worked_example():
    """The four branch formulas of the inference loop ("SenseNova-U1" §2.7),
    worked by hand: z = 0, t = 0.5 (so each v_X = 2 x0_X), t_next = 0.6,
    x0 = 1 (cond), 0.5 (text-unconditional), 0 (unconditional) give
    v_c = 2, v_tu = 1, v_u = 0."""
    z, c, tu, u = (np.zeros(3), np.ones(3), np.full(3, 0.5), np.zeros(3))
    cases = [  # (g, g_img, branch, v)
        (1.0, 1.0, O.CFG_NONE, 2.0),      # v_c
        (4.0, 1.0, O.CFG_TEXT, 5.0),      # v_tu + 4 (v_c - v_tu) = 1 + 4
        (3.0, 3.0, O.CFG_CLASSIC, 6.0),   # v_u + 3 (v_c - v_u) = 0 + 6
        (4.0, 1.5, O.CFG_DUAL, 5.5),      # v_u + 4 (v_c - v_tu) + 1.5 (v_tu - v_u) = 4 + 1.5
    ]
    for g, gi, branch, v in cases:
        zn, vv, br = O.flow_cfg_euler_step(z, c, tu, u, 0.5, 0.6, g, gi)
        assert br == branch
        np.testing.assert_allclose(vv, v, rtol=1e-15)
        np.testing.assert_allclose(zn, 0.1 * v, rtol=1e-14)


def test_cfg_classic_is_cond_against_the_full_unconditional():
    """The classic branch is single-axis guidance of cond against the fully
    unconditional prediction, (1 - g) v_u + g v_c ("SenseNova-U1" §2.7); it
    reads no text-unconditional prediction (NaN there changes nothing), and
    the text branch reads no unconditional one. Velocities come from the
    plain Euler step of each prediction."""
    z, c, tu, u = _cfg_inputs(seed=43)
    t, g = 0.35, 3.0
    nan = np.full_like(z, np.nan)
    zn, v, br = O.flow_cfg_euler_step(z, c, nan, u, t, t + 0.1, g, g)
    assert br == O.CFG_CLASSIC
    _, vc = O.flow_euler_step(z, c, t, t + 0.1)
    _, vu = O.flow_euler_step(z, u, t, t + 0.1)
    np.testing.assert_allclose(v, (1 - g) * vu + g * vc, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(zn, z + 0.1 * v, rtol=1e-12, atol=1e-12)
    _, vt, br = O.flow_cfg_euler_step(z, c, tu, nan, t, t + 0.1, g, 1.0)
    assert br == O.CFG_TEXT and np.all(np.isfinite(vt))


def test_cfg_dual_meets_the_text_and_classic_branches():
    """The dual form is affine in img_cfg_scale with slope v_tu - v_u, and it
    equals the text branch at img scale 1 and the classic branch at equal
    scales ("SenseNova-U1" §2.7, Eq. 6 and its two reductions). Both sides are
    oracle calls: the dual branch just off each meeting point against the
    branch the loop takes at that point."""
    z, c, tu, u = _cfg_inputs(seed=44)
    t, g, d = 0.25, 3.0, 0.5
    _, vtu = O.flow_euler_step(z, tu, t, t + 0.1)
    _, vu = O.flow_euler_step(z, u, t, t + 0.1)
    _, v_text, b_text = O.flow_cfg_euler_step(z, c, tu, u, t, t + 0.1, g, 1.0)
    _, v_cls, b_cls = O.flow_cfg_euler_step(z, c, tu, u, t, t + 0.1, g, g)
    _, v_d1, b_d1 = O.flow_cfg_euler_step(z, c, tu, u, t, t + 0.1, g, 1.0 + d)
    _, v_d2, b_d2 = O.flow_cfg_euler_step(z, c, tu, u, t, t + 0.1, g, g + d)
    assert (b_text, b_cls, b_d1, b_d2) == (O.CFG_TEXT, O.CFG_CLASSIC, O.CFG_DUAL, O.CFG_DUAL)
    np.testing.assert_allclose(v_d1 - v_text, d * (vtu - vu), rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(v_d2 - v_cls, d * (vtu - vu), rtol=1e-11, atol=1e-11)


# ---------------------------------------------------------------- sampler pieces
def test_time_schedule_endpoints_identity_and_shift_map():
    for n in (10, 50):
        for shift in (1.0, 3.0, 0.5):
            t = O.time_schedule(n, shift)
            assert t.shape == (n + 1,)
            assert t[0] == pytest.approx(0.0, abs=1e-15) and t[-1] == pytest.approx(1.0, abs=1e-15)
            assert np.all(np.diff(t) > 0)
    np.testing.assert_allclose(O.time_schedule(50, 1.0), np.linspace(0, 1, 51), atol=1e-15)
    # shift s maps sigma = 1/2 to s/(1+s): with s = 3 the middle of the grid lands at t = 1/4
    assert O.time_schedule(10, 3.0)[5] == pytest.approx(0.25, abs=1e-15)
    # shift > 1 spends more steps at high noise (small t)
    assert np.all(O.time_schedule(50, 3.0)[1:-1] < np.linspace(0, 1, 51)[1:-1])


def test_noise_scale_closed_forms():
    # 2048^2: 128x128 patches, merge 2 -> 4096 tokens; base 64 tokens -> sqrt(64) = 8
    assert O.noise_scale(128, 128, 2, 64, 1.0, O.NOISE_RESOLUTION) == pytest.approx(8.0)
    assert O.noise_scale(128, 128, 2, 64, 1.0, O.NOISE_DYNAMIC) == pytest.approx(8.0)
    assert O.noise_scale(128, 128, 2, 64, 1.0, O.NOISE_DYNAMIC_SQRT) == pytest.approx(np.sqrt(8.0))
    assert O.noise_scale(64, 64, 2, 64, 1.0, O.NOISE_RESOLUTION) == pytest.approx(4.0)   # 1024^2
    assert O.noise_scale(128, 128, 2, 64, 3.0, O.NOISE_RESOLUTION) == pytest.approx(16.0)   # capped
    assert O.noise_scale(128, 128, 2, 64, 3.0, O.NOISE_RESOLUTION, max_value=8.0) == pytest.approx(8.0)
    assert O.noise_scale(128, 128, 2, 64, 0.7, O.NOISE_CONSTANT) == pytest.approx(0.7)
    # sigma grows as the square root of the token count
    r = O.noise_scale(96, 96, 2, 64, 1.0, O.NOISE_RESOLUTION) / O.noise_scale(48, 48, 2, 64, 1.0, O.NOISE_RESOLUTION)
    assert r == pytest.approx(2.0)


def test_initial_noise_scales_the_draw():
    e = np.random.default_rng(60).standard_normal(100)
    np.testing.assert_array_equal(O.initial_noise(e, 1.0), e)
    np.testing.assert_allclose(O.initial_noise(e, 8.0), 8.0 * e, rtol=1e-15)


# ---------------------------------------------------------------- interleaved 2-D RoPE
def test_rope2d_identity_at_origin_and_pair_norms():
    g = np.random.default_rng(80)
    x = g.standard_normal((2, 12, 16))                       # 3 x 4 grid, 16 channels
    y = O.rope2d_interleaved(x, 3, 4)
    np.testing.assert_array_equal(y[:, 0], x[:, 0])          # patch (0, 0)
    n0 = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    n1 = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    np.testing.assert_allclose(n1, n0, rtol=1e-12)


def test_rope2d_halves_follow_column_and_row():
    g = np.random.default_rng(81)
    x = np.broadcast_to(g.standard_normal(16), (1, 12, 16)).copy()
    y = O.rope2d_interleaved(x, 3, 4)
    # same column (c = 1), different rows: first half equal, second half differs
    np.testing.assert_allclose(y[0, 1, :8], y[0, 5, :8], rtol=1e-13)
    assert not np.allclose(y[0, 1, 8:], y[0, 5, 8:])
    # same row (r = 2), different columns: second half equal
    np.testing.assert_allclose(y[0, 8, 8:], y[0, 11, 8:], rtol=1e-13)
    assert not np.allclose(y[0, 8, :8], y[0, 11, :8])


def test_rope2d_interleaved_complex_closed_form():
    """Pair (2i, 2i+1) is the complex number x[2i] + i x[2i+1] times
    exp(i p f_i) with f_0 = 1 and a geometric ratio theta^(-2/d)."""
    C, theta = 16, 1e4
    d = C // 2
    x = np.zeros((1, 2, C))
    x[0, 1, 0:d:2] = 1.0                                     # patch (0, 1): column 1
    y = O.rope2d_interleaved(x, 1, 2, theta)
    f = np.angle(y[0, 1, 0:d:2] + 1j * y[0, 1, 1:d:2])
    assert f[0] == pytest.approx(1.0, rel=1e-14)
    np.testing.assert_allclose(f[1:] / f[:-1], theta ** (-2.0 / d), rtol=1e-12)
    assert np.all(y[0, 1, d:] == 0)                          # row index 0: second half untouched (zeros)


def test_rope2d_relative_position():
    g = np.random.default_rng(82)
    q, k = g.standard_normal(32), g.standard_normal(32)
    rows, cols = 6, 7
    xq = np.broadcast_to(q, (1, rows * cols, 32)).copy()
    xk = np.broadcast_to(k, (1, rows * cols, 32)).copy()
    yq, yk = O.rope2d_interleaved(xq, rows, cols), O.rope2d_interleaved(xk, rows, cols)
    dot = lambda a, b: float(np.sum(yq[0, a] * yk[0, b]))
    # (r, c) pairs with equal offsets give equal dot products
    assert dot(1 * cols + 2, 3 * cols + 5) == pytest.approx(dot(2 * cols + 1, 4 * cols + 4), rel=1e-10)


# ------------------------------------------------------------------ prefix cache
def _cache_case(rng, lens, N, n_new, Hkv=2, D=8):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    k_old = rng.standard_normal((int(cu[-1]), Hkv, D))
    v_old = rng.standard_normal((int(cu[-1]), Hkv, D))
    k_new = rng.standard_normal((len(lens), N, Hkv, D))
    v_new = rng.standard_normal((len(lens), N, Hkv, D))
    return k_old, v_old, cu, k_new, v_new, np.asarray(n_new)


def test_cache_empty_chunk_leaves_the_cache():
    rng = np.random.default_rng(0)
    k_old, v_old, cu, k_new, v_new, n = _cache_case(rng, (3, 0, 5), 4, (0, 0, 0))
    k, v, cu_out = O.write_prefix_cache(k_old, v_old, cu, k_new, v_new, n)
    assert np.array_equal(k, k_old) and np.array_equal(v, v_old) and np.array_equal(cu_out, cu)


def test_cache_from_empty_is_a_masked_gather():
    """Appending to empty caches packs the valid rows of the chunk: the same
    rows, in the same order, as boolean-mask indexing of the padded chunk."""
    rng = np.random.default_rng(1)
    k_old, v_old, cu, k_new, v_new, n = _cache_case(rng, (0, 0, 0), 6, (6, 2, 4))
    k, v, cu_out = O.write_prefix_cache(k_old, v_old, cu, k_new, v_new, n)
    mask = np.arange(6)[None, :] < n[:, None]
    assert np.array_equal(k, k_new[mask]) and np.array_equal(v, v_new[mask])
    assert list(cu_out) == [0, 6, 8, 12]


def test_cache_two_appends_equal_one_append_of_the_joined_chunk():
    rng = np.random.default_rng(2)
    k_old, v_old, cu, k1, v1, n1 = _cache_case(rng, (2, 7), 3, (3, 1))
    _, _, _, k2, v2, n2 = _cache_case(rng, (2, 7), 5, (2, 5))
    ka, va, cua = O.write_prefix_cache(*O.write_prefix_cache(k_old, v_old, cu, k1, v1, n1), k2, v2, n2)
    kj = np.zeros((2, 8) + k1.shape[2:])
    vj = np.zeros_like(kj)
    for b in range(2):
        kj[b, :n1[b] + n2[b]] = np.concatenate([k1[b, :n1[b]], k2[b, :n2[b]]])
        vj[b, :n1[b] + n2[b]] = np.concatenate([v1[b, :n1[b]], v2[b, :n2[b]]])
    kb, vb, cub = O.write_prefix_cache(k_old, v_old, cu, kj, vj, n1 + n2)
    assert np.array_equal(ka, kb) and np.array_equal(va, vb) and np.array_equal(cua, cub)


def test_chunked_block_causal_prefill_through_the_cache_equals_one_pass():
    """Block-causal prefill of a sequence in one pass equals: prefill the
    first chunk, write its keys/values to the cache, then prefill the second
    chunk against that cache (the image block straddles the boundary)."""
    rng = np.random.default_rng(3)
    T = np.array(list(range(5)) + [5] * 9 + list(range(6, 10)))   # 18 tokens
    S, Hq, Hkv, D = len(T), 4, 2, 16
    q = rng.standard_normal((1, S, Hq, D))
    k = rng.standard_normal((1, S, Hkv, D))
    v = rng.standard_normal((1, S, Hkv, D))
    empty = np.zeros((0, Hkv, D))
    full, _ = O.gen_attention(q, empty, empty, k, v, [0, 0], 0.3, mask_mode=1, t_prefix=T[:0], t_img=T[None])
    c = 8
    kc, vc, cu = O.write_prefix_cache(empty, empty, [0, 0], k[:, :c], v[:, :c], [c])
    second, _ = O.gen_attention(q[:, c:], kc, vc, k[:, c:], v[:, c:], cu, 0.3, mask_mode=1,
                                t_prefix=T[:c], t_img=T[None, c:])
    np.testing.assert_allclose(second, full[:, c:], rtol=1e-12, atol=1e-12)

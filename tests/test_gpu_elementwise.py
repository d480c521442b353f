"""GPU parity of the HBM-bound kernels against the fp64 oracle: position
indexes (exact), QK-norm halves + three-axis RoPE (bf16 and fp32), and the
x0 -> v Euler step (fp32)."""

import numpy as np
import pytest
import torch

import oracle as O
from attention_neo_qknorm_gb300 import neo, synth
from helpers import F32_TOL, assert_bf16_close, f64, image_segments, max_abs, prefix_segments, rel_frob

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_positions_exact(gpu_lib, name):
    w = synth.WORKLOADS[name]
    for segs, S in ((image_segments(w), w.B * w.N), (prefix_segments(w), w.total_prefix)):
        idx = torch.full((3, S), -7, dtype=torch.int32, device="cuda")
        neo.neo_build_positions(idx, segs)
        np.testing.assert_array_equal(idx.cpu().numpy(), O.positions(segs))


def _norm_rope_case(S, Hq, Hkv, dtype, segs, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(S, Hq, 128, generator=g).to(dtype)
    k = torch.randn(S, Hkv, 128, generator=g).to(dtype)
    ws = [torch.rand(64, generator=g) + 0.5 for _ in range(4)]
    idx = O.positions(segs)
    qd, kd = q.cuda(), k.cuda()
    idx_d = torch.from_numpy(idx.astype(np.int32)).cuda()
    neo.neo_qknorm_rope3(qd, kd, idx_d, *[t.cuda() for t in ws])
    rq = O.qknorm_rope3(f64(q), idx, f64(ws[0]), f64(ws[1]))
    rk = O.qknorm_rope3(f64(k), idx, f64(ws[2]), f64(ws[3]))
    return f64(qd), rq, f64(kd), rk


@pytest.mark.parametrize("segs,Hq,Hkv", [
    ([("text", 0, 37)], 4, 1),
    ([("text", 0, 512), ("image", 512, 32, 32)], 32, 8),
    ([("image", 1024, 64, 64)], 32, 8),
    ([("image", 6000, 3, 5)], 6, 2),
])
def test_qknorm_rope3_bf16(gpu_lib, segs, Hq, Hkv):
    S = O.positions(segs).shape[1]
    gq, rq, gk, rk = _norm_rope_case(S, Hq, Hkv, torch.bfloat16, segs, seed=S)
    assert_bf16_close(gq, rq, "q")
    assert_bf16_close(gk, rk, "k")


def test_qknorm_rope3_fp32(gpu_lib):
    segs = [("text", 0, 32), ("image", 32, 8, 8)]
    gq, rq, gk, rk = _norm_rope_case(96, 4, 1, torch.float32, segs, seed=3)
    # fp32 end to end: only the fp32 angle (|a| up to 95 rad here) and rsqrt limit the error.
    assert max_abs(gq, rq) < 2e-5 and max_abs(gk, rk) < 2e-5


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_qknorm_rope3_large_positions(gpu_lib, dtype):
    """Positions far beyond any prompt of the workloads: a long text prefix
    (2^14 .. 2^16), an image at temporal index 2^20, and arbitrary int32
    positions up to 2^30 on each axis. The angle is reduced exactly for every
    int32 position, so the error stays that of fp32 sin/cos and rounding."""
    g = np.random.default_rng(17)
    text = [("text", 1 << 14, 40), ("text", (1 << 16) - 20, 20), ("image", 1 << 20, 4, 6)]
    idx = O.positions(text)
    extra = g.integers(0, 1 << 30, size=(3, 16))
    idx = np.concatenate([idx, extra], axis=1)
    S = idx.shape[1]
    gen = torch.Generator().manual_seed(18)
    q = torch.randn(S, 4, 128, generator=gen).to(dtype)
    k = torch.randn(S, 2, 128, generator=gen).to(dtype)
    ws = [torch.rand(64, generator=gen) + 0.5 for _ in range(4)]
    qd, kd = q.cuda(), k.cuda()
    neo.neo_qknorm_rope3(qd, kd, torch.from_numpy(idx.astype(np.int32)).cuda(), *[t.cuda() for t in ws])
    rq = O.qknorm_rope3(f64(q), idx, f64(ws[0]), f64(ws[1]))
    rk = O.qknorm_rope3(f64(k), idx, f64(ws[2]), f64(ws[3]))
    if dtype == torch.bfloat16:
        assert_bf16_close(f64(qd), rq, "q")
        assert_bf16_close(f64(kd), rk, "k")
    else:
        assert max_abs(f64(qd), rq) < 2e-5 and max_abs(f64(kd), rk) < 2e-5


def test_qknorm_rope3_keys_only_and_queries_only(gpu_lib):
    segs = [("text", 0, 20)]
    g = torch.Generator().manual_seed(9)
    x = torch.randn(20, 2, 128, generator=g).to(torch.bfloat16)
    w1, w2 = torch.rand(64, generator=g) + 0.5, torch.rand(64, generator=g) + 0.5
    idx = torch.from_numpy(O.positions(segs).astype(np.int32)).cuda()
    ref = O.qknorm_rope3(f64(x), O.positions(segs), f64(w1), f64(w2))
    kd = x.cuda()
    neo.neo_qknorm_rope3(None, kd, idx, None, None, w1.cuda(), w2.cuda())
    assert_bf16_close(f64(kd), ref, "k only")
    qd = x.cuda()
    neo.neo_qknorm_rope3(qd, None, idx, w1.cuda(), w2.cuda(), None, None)
    assert_bf16_close(f64(qd), ref, "q only")


def _euler_check(z, x0, t, tn, with_v=True):
    zd, xd = z.cuda(), x0.cuda()
    vd = torch.empty_like(zd) if with_v else None
    neo.neo_flow_euler_step(zd, xd, t, tn, 0.02, vd)
    rz, rv = O.flow_euler_step(f64(z), f64(x0), np.float32(t), np.float32(tn), np.float32(0.02))
    assert max_abs(f64(zd), rz) <= F32_TOL * max(1.0, np.abs(rz).max())
    assert rel_frob(f64(zd), rz) <= F32_TOL
    if with_v:
        assert rel_frob(f64(vd), rv) <= F32_TOL
    return zd


@pytest.mark.parametrize("name", ["tiny_ref", "gen_2048"])
def test_euler_step_matches_oracle(gpu_lib, name):
    w = synth.WORKLOADS[name]
    z, (x0,) = synth.make_flow(w)
    _euler_check(z, x0, w.t_steps[0], w.t_steps[0] + w.dt)


def test_euler_ragged_tail_and_t_eps_clamp(gpu_lib):
    g = torch.Generator().manual_seed(11)
    for n in (1, 3, 4097, 1000003):
        z, x0 = torch.randn(n, generator=g), torch.randn(n, generator=g)
        _euler_check(z, x0, 0.99, 1.0)
        _euler_check(z, x0, 0.25, 0.35, with_v=False)


def test_euler_worked_example(gpu_lib):
    """t = 0.6, x0 = 1, z = 0.6: v = 1 and the step to 0.7 lands on 0.7."""
    z = torch.full((8,), 0.6, device="cuda")
    x0 = torch.ones(8, device="cuda")
    v = torch.empty(8, device="cuda")
    neo.neo_flow_euler_step(z, x0, 0.6, 0.7, 0.02, v)
    assert np.allclose(v.cpu().numpy(), 1.0, atol=1e-6) and np.allclose(z.cpu().numpy(), 0.7, atol=1e-6)


def test_euler_ten_steps_ragged_batch_lands_on_x0(gpu_lib):
    """Ragged CFG workload: ten steps t = 0 .. 0.9 with a fixed x0_hat land on
    x0_hat (straight-path closed form), at the full 4 x 4096 x 3072 size."""
    w = synth.WORKLOADS["ragged_cfg"]
    z, (x0,) = synth.make_flow(w)
    zd, xd = z.cuda(), x0.cuda()
    for t in w.t_steps:
        neo.neo_flow_euler_step(zd, xd, t, t + w.dt, 0.02)
    x = f64(x0)
    assert max_abs(f64(zd), x) <= F32_TOL * max(1.0, float(np.abs(x).max()))
    assert rel_frob(f64(zd), x) <= F32_TOL


def test_euler_ten_steps_against_oracle(gpu_lib):
    g = torch.Generator().manual_seed(12)
    n = 3 * 4096 + 5
    z = torch.randn(n, generator=g)
    xs = [torch.randn(n, generator=g) for _ in range(10)]
    zd = z.cuda()
    rz = f64(z)
    for k in range(10):
        t, tn = np.float32(k / 10), np.float32((k + 1) / 10)
        neo.neo_flow_euler_step(zd, xs[k].cuda(), float(t), float(tn), 0.02)
        rz, _ = O.flow_euler_step(rz, f64(xs[k]), t, tn, np.float32(0.02))
    assert rel_frob(f64(zd), rz) <= F32_TOL


@pytest.mark.parametrize("g,gi,interval,t", [
    (1.0, 1.0, (0.0, 1.0), 0.3),     # no guidance
    (4.0, 1.0, (0.0, 1.0), 0.3),     # text CFG, the T2I default scales
    (3.0, 3.0, (0.0, 1.0), 0.5),     # classic CFG
    (4.0, 1.5, (0.0, 1.0), 0.7),     # dual (Eq. 6)
    (4.0, 1.5, (0.6, 1.0), 0.5),     # outside the interval: unguided
    (4.0, 1.5, (0.6, 1.0), 0.95),    # inside, clamped by t_eps
])
def test_cfg_euler_matches_oracle(gpu_lib, g, gi, interval, t):
    gen = torch.Generator().manual_seed(50)
    n = 3 * 4096 + 7
    z, c, tu, u = (torch.randn(n, generator=gen) for _ in range(4))
    zd, vd = z.cuda(), torch.empty(n, device="cuda")
    branch = neo.neo_flow_cfg_euler_step(zd, c.cuda(), tu.cuda(), u.cuda(), t, t + 0.05, g, gi, interval,
                                         v_out=vd)
    f32 = np.float32
    rz, rv, rb = O.flow_cfg_euler_step(f64(z), f64(c), f64(tu), f64(u), f32(t), f32(t + 0.05), f32(g), f32(gi),
                                       (f32(interval[0]), f32(interval[1])), t_eps=f32(0.02))
    assert branch == rb
    for got, ref in ((f64(zd), rz), (f64(vd), rv)):
        assert rel_frob(got, ref) <= F32_TOL
        assert max_abs(got, ref) <= F32_TOL * max(1.0, float(np.abs(ref).max()))


def test_cfg_euler_reads_only_the_needed_predictions(gpu_lib):
    """The unguided branch needs no unconditional predictions (None is fine);
    a guided branch without them is rejected before anything runs."""
    z = torch.randn(1000, device="cuda")
    c = torch.randn(1000, device="cuda")
    ref = z.clone()
    neo.neo_flow_euler_step(ref, c, 0.4, 0.5)
    zz = z.clone()
    assert neo.neo_flow_cfg_euler_step(zz, c, None, None, 0.4, 0.5, 1.0, 1.0) == neo.NEO_CFG_NONE
    assert torch.equal(zz, ref)
    with pytest.raises(neo.NeoError) as e:
        neo.neo_flow_cfg_euler_step(z.clone(), c, None, None, 0.4, 0.5, 4.0, 1.0)
    assert e.value.status == neo.NEO_ERR_INVALID_ARG


def test_scale_noise_and_sampler_loop(gpu_lib):
    """Initial sample z_0 = sigma_R * eps, then the shifted schedule drives ten
    Euler steps with a fixed x0_hat; compared with the oracle step by step."""
    gen = torch.Generator().manual_seed(70)
    n = 4096 * 3 + 3
    eps, x0 = torch.randn(n, generator=gen), torch.randn(n, generator=gen)
    sigma = neo.neo_noise_scale(64, 64, 2, 64.0, 1.0)
    z = torch.empty(n, device="cuda")
    neo.neo_scale_noise(z, eps.cuda(), sigma)
    rz = O.initial_noise(f64(eps), np.float32(sigma))
    assert max_abs(f64(z), rz) <= 6e-8 * float(np.abs(rz).max())   # one fp32 rounding
    ts = neo.neo_time_schedule(10, 3.0)
    xd = x0.cuda()
    for k in range(10):
        neo.neo_flow_euler_step(z, xd, ts[k], ts[k + 1])
        rz, _ = O.flow_euler_step(rz, f64(x0), np.float32(ts[k]), np.float32(ts[k + 1]), np.float32(0.02))
    assert rel_frob(f64(z), rz) <= F32_TOL


@pytest.mark.parametrize("dtype,n_img,rows,cols,C", [
    (torch.bfloat16, 2, 5, 7, 1024),      # model width, ragged grid
    (torch.bfloat16, 1, 128, 128, 1024),  # the 2048^2 patch grid (before the 2x2 merge)
    (torch.float32, 3, 4, 6, 64),
    (torch.bfloat16, 3, 9, 5, 24),        # 8-channel chunks straddle the column/row halves
    (torch.bfloat16, 1, 3, 4, 4096),      # more 16-byte chunks per patch than threads per block
    (torch.bfloat16, 700, 3, 3, 8),       # one chunk per patch: many patches per block
    (torch.float32, 2, 7, 3, 12),         # fp32 chunks straddle the halves
    (torch.bfloat16, 2, 17, 9, 32),       # lines longer than one segment, ragged last segments
    (torch.float32, 1, 1, 19, 16),        # one row: every column line a single patch
])
def test_rope2d_interleaved_matches_oracle(gpu_lib, dtype, n_img, rows, cols, C):
    gen = torch.Generator().manual_seed(rows * cols + C)
    x = torch.randn(n_img, rows * cols, C, generator=gen).to(dtype)
    xd = x.cuda()
    neo.neo_rope2d_interleaved(xd, rows, cols)
    ref = O.rope2d_interleaved(f64(x), rows, cols)
    if dtype == torch.bfloat16:
        assert_bf16_close(f64(xd), ref, "rope2d bf16")
    else:
        assert max_abs(f64(xd), ref) < 2e-5


def test_cfg_euler_full_size_dual(gpu_lib):
    """The configuration the bench times beside the step: dual guidance on the
    2048^2 workload's 4096 x 3072 fp32 patches with three predictions."""
    w = synth.WORKLOADS["gen_2048"]
    z, xs = synth.make_flow(w, n_x0=3)
    zd, vd = z.cuda(), torch.empty_like(z, device="cuda")
    branch = neo.neo_flow_cfg_euler_step(zd, xs[0].cuda(), xs[1].cuda(), xs[2].cuda(), 0.5, 0.55, 4.0, 1.5,
                                         v_out=vd)
    f32 = np.float32
    rz, rv, rb = O.flow_cfg_euler_step(f64(z), f64(xs[0]), f64(xs[1]), f64(xs[2]), f32(0.5), f32(0.55), f32(4.0),
                                       f32(1.5), (f32(0.0), f32(1.0)), t_eps=f32(0.02))
    assert branch == rb == neo.NEO_CFG_DUAL
    for got, ref in ((f64(zd), rz), (f64(vd), rv)):
        assert rel_frob(got, ref) <= F32_TOL
        assert max_abs(got, ref) <= F32_TOL * max(1.0, float(np.abs(ref).max()))

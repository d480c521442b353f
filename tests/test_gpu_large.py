"""Maximum-size cases: inputs whose element counts or byte offsets pass 2^31,
and an attention with a long prefix and a long image segment. The GPU works
on the whole input; the oracle recomputes sampled outputs one by one."""

import numpy as np
import pytest
import torch

import oracle as O
from attention_neo_qknorm_gb300 import neo
from helpers import F32_TOL, SCALE, assert_bf16_close, f64

pytestmark = pytest.mark.gpu


def _sample(n, count, seed):
    """Sorted distinct indices in [0, n): the first and last few and a random spread."""
    rng = np.random.default_rng(seed)
    idx = np.concatenate([np.arange(4), n - 1 - np.arange(4), rng.integers(0, n, size=count)])
    return np.unique(idx)


def test_euler_step_beyond_2_pow_31_elements(gpu_lib):
    """z and x0_hat of 2^31 + 4099 fp32 elements (8.6 GB each): element
    indexes and byte offsets beyond 32 bits."""
    n = (1 << 31) + 4099
    g = torch.Generator(device="cuda").manual_seed(41)
    z = torch.randn(n, device="cuda", generator=g)
    x0 = torch.randn(n, device="cuda", generator=g)
    sel = torch.from_numpy(_sample(n, 4096, 42)).cuda()
    z_before, x_sel = f64(z[sel]), f64(x0[sel])
    t, tn = 0.35, 0.45
    neo.neo_flow_euler_step(z, x0, t, tn, 0.02)
    torch.cuda.synchronize()
    rz, _ = O.flow_euler_step(z_before, x_sel, np.float32(t), np.float32(tn), np.float32(0.02))
    got = f64(z[sel])
    assert np.max(np.abs(got - rz)) <= F32_TOL * max(1.0, float(np.abs(rz).max()))
    del z, x0


def test_qknorm_rope3_beyond_2_pow_31_elements(gpu_lib):
    """530 000 tokens of 32 query and 8 key heads (q: 2.17e9 bf16 elements,
    4.3 GB) at positions up to 2^20; sampled tokens against the oracle."""
    S, Hq, Hkv = 530_000, 32, 8
    g = torch.Generator(device="cuda").manual_seed(43)
    q = torch.randn(S, Hq, 128, device="cuda", generator=g).to(torch.bfloat16)
    k = torch.randn(S, Hkv, 128, device="cuda", generator=g).to(torch.bfloat16)
    idx = torch.randint(0, 1 << 20, (3, S), device="cuda", generator=g, dtype=torch.int32)
    ws = [torch.rand(64, device="cuda", generator=g) + 0.5 for _ in range(4)]
    toks = torch.from_numpy(_sample(S, 400, 44)).cuda()
    q_in, k_in = f64(q[toks]), f64(k[toks])
    neo.neo_qknorm_rope3(q, k, idx, *ws)
    torch.cuda.synchronize()
    pos = idx[:, toks].cpu().numpy()
    rq = O.qknorm_rope3(q_in, pos, f64(ws[0]), f64(ws[1]))
    rk = O.qknorm_rope3(k_in, pos, f64(ws[2]), f64(ws[3]))
    assert_bf16_close(f64(q[toks]), rq, "q, sampled tokens")
    assert_bf16_close(f64(k[toks]), rk, "k, sampled tokens")
    del q, k


def test_attention_long_prefix_and_image(gpu_lib):
    """One sequence with a 65 536-token prefix and 32 768 image tokens (98 304
    keys, 32 / 8 heads: 52.8 TFLOP), plus a second sequence with a ragged
    prefix; sampled query rows against the oracle, with their log-sum-exps."""
    Ls, N, Hq, Hkv = (65_536, 1_037), 32_768, 32, 8
    B = len(Ls)
    g = torch.Generator(device="cuda").manual_seed(45)
    bf = lambda *sh: torch.randn(*sh, device="cuda", generator=g).to(torch.bfloat16)
    q, k, v = bf(B, N, Hq, 128), bf(B, N, Hkv, 128), bf(B, N, Hkv, 128)
    kp, vp = bf(sum(Ls), Hkv, 128), bf(sum(Ls), Hkv, 128)
    cu = torch.tensor([0, Ls[0], Ls[0] + Ls[1]], dtype=torch.int32, device="cuda")
    out = torch.empty(B, N, Hq, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, Hq, N, dtype=torch.float32, device="cuda")
    neo.neo_gen_attention(q, kp, vp, k, v, cu, max(Ls), out, scale=SCALE, lse=lse)
    st, word = neo.neo_get_device_error()
    assert st == neo.NEO_OK, hex(word)
    rng = np.random.default_rng(46)
    rows = np.stack([rng.integers(0, B, 192), rng.integers(0, N, 192), rng.integers(0, Hq, 192)], axis=1)
    rows[:4] = [[0, N - 1, Hq - 1], [1, N - 1, 0], [0, 0, 0], [1, 0, Hq - 1]]
    # the oracle sees only the sampled queries (other rows zero) and every key of their sequences
    qs = np.zeros((B, N, Hq, 128))
    for b, n, h in rows:
        qs[b, n, h] = f64(q[b, n, h])
    ref, ref_lse = O.gen_attention(qs, f64(kp), f64(vp), f64(k), f64(v), np.array([0, Ls[0], sum(Ls)]), SCALE,
                                   rows=rows)
    got = np.stack([f64(out[b, n, h]) for b, n, h in rows])
    got_lse = np.array([float(lse[b, h, n]) for b, n, h in rows])
    assert_bf16_close(got, ref, "long prefix, sampled rows")
    np.testing.assert_allclose(got_lse, ref_lse, rtol=1e-3, atol=2e-2)

"""The attention with the query norm + RoPE folded into its prologue
(neo_gen_attention_qnorm) against the two-launch path (neo_qknorm_rope3 on the
queries, then neo_gen_attention): both use the same arithmetic, so the outputs
and log-sum-exps must agree bit for bit; the raw queries are left unchanged."""

import numpy as np
import pytest
import torch

import oracle as O
from attention_neo_qknorm_gb300 import neo, synth
from helpers import GpuLayer, assert_bf16_close, f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("prefix,grid,Hq,Hkv", [
    ((200, 77), (12, 11), 8, 2),       # ragged prefixes, N = 132 (padding rows in the last tile)
    ((0, 130), (13, 13), 8, 2),        # an empty prefix
    ((64,), (8, 8), 4, 1),             # G = 4, one sequence
    ((130,), (10, 10), 2, 2),          # G = 1
    ((70,), (9, 10), 4, 2),            # G = 2
    ((5, 129, 300), (5, 8), 16, 2),    # G = 8, three sequences
    ((1000,), (24, 16), 32, 8),        # production head counts
])
def test_fused_equals_two_launches(gpu_lib, prefix, grid, Hq, Hkv):
    w = synth.small_workload(prefix=prefix, grid=grid, Hq=Hq, Hkv=Hkv, B=len(prefix))
    inp = synth.make_inputs(w, seed=31 + Hq)
    a = GpuLayer(w, inp)
    b = GpuLayer(w, inp)
    q_raw = a.q.clone()
    a.norm_rope()
    a.attention()
    b.norm_rope_k()
    b.attention_qnorm()
    assert torch.equal(b.q, q_raw), "the raw queries must be left unchanged"
    assert torch.equal(a.k, b.k)
    assert torch.equal(a.out, b.out), "fused and two-launch outputs differ"
    assert torch.equal(a.lse, b.lse)


@pytest.mark.parametrize("case", range(8))
def test_fused_equals_two_launches_random_shapes(gpu_lib, case):
    """Seeded random prefixes, grids and group sizes."""
    rng = np.random.default_rng(3000 + case)
    Hkv = int(rng.choice([1, 2]))
    Hq = Hkv * int(rng.choice([1, 2, 4, 8]))
    prefix = tuple(int(x) for x in rng.integers(0, 300, size=int(rng.integers(1, 4))))
    grid = (int(rng.integers(1, 18)), int(rng.integers(1, 18)))
    w = synth.small_workload(prefix=prefix, grid=grid, Hq=Hq, Hkv=Hkv, B=len(prefix))
    inp = synth.make_inputs(w, seed=50 + case)
    a = GpuLayer(w, inp)
    b = GpuLayer(w, inp)
    a.norm_rope()
    a.attention()
    b.norm_rope_k()
    b.attention_qnorm()
    assert torch.equal(a.out, b.out), f"fused and two-launch outputs differ: {prefix} {grid} {Hq}/{Hkv}"
    assert torch.equal(a.lse, b.lse)


def test_fused_matches_oracle_with_distinct_positions(gpu_lib):
    """Positions that differ on all three axes per token (a prefix of text
    tokens as the query segment): the temporal angle is not constant."""
    S, Hq, Hkv = 300, 8, 2
    g = torch.Generator().manual_seed(3)
    bf = lambda *sh: torch.randn(*sh, generator=g).to(torch.bfloat16)
    q, k, v = bf(1, S, Hq, 128), bf(1, S, Hkv, 128), bf(1, S, Hkv, 128)
    ws = [torch.rand(64, generator=g) + 0.5 for _ in range(4)]
    segs = [("text", 0, 100), ("image", 100, 10, 10), ("text", 101, 100)]
    idx = torch.empty(3, S, dtype=torch.int32, device="cuda")
    neo.neo_build_positions(idx, segs)
    kd = k.cuda().reshape(S, Hkv, 128).contiguous()
    neo.neo_qknorm_rope3(None, kd, idx, None, None, ws[2].cuda(), ws[3].cuda())
    out = torch.empty(1, S, Hq, 128, dtype=torch.bfloat16, device="cuda")
    cu = torch.zeros(2, dtype=torch.int32, device="cuda")
    neo.neo_gen_attention_qnorm(q.cuda(), None, None, kd.view(1, S, Hkv, 128), v.cuda(), cu, 0, out,
                                idx, ws[0].cuda(), ws[1].cuda())
    pos = O.positions(segs)
    qo = O.qknorm_rope3(f64(q).reshape(S, Hq, 128), pos, f64(ws[0]), f64(ws[1])).reshape(1, S, Hq, 128)
    ko = O.qknorm_rope3(f64(k).reshape(S, Hkv, 128), pos, f64(ws[2]), f64(ws[3])).reshape(1, S, Hkv, 128)
    ref, _ = O.gen_attention(qo, np.zeros((0, Hkv, 128)), np.zeros((0, Hkv, 128)), ko, f64(v),
                             np.array([0, 0]), 128 ** -0.5)
    assert_bf16_close(f64(out), ref, "fused, distinct positions")


def test_fused_block_causal_equals_two_launches(gpu_lib):
    S, Hq, Hkv = 257, 8, 2
    g = torch.Generator().manual_seed(4)
    q = torch.randn(1, S, Hq, 128, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(1, S, Hkv, 128, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(1, S, Hkv, 128, generator=g).to(torch.bfloat16).cuda()
    ws = [(torch.rand(64, generator=g) + 0.5).cuda() for _ in range(2)]
    segs = [("text", 0, 60), ("image", 60, 12, 12), ("text", 61, 53)]
    idx = torch.empty(3, S, dtype=torch.int32, device="cuda")
    neo.neo_build_positions(idx, segs)
    T = idx[0].contiguous()
    cu = torch.zeros(2, dtype=torch.int32, device="cuda")
    fused = torch.empty_like(q)
    neo.neo_gen_attention_qnorm(q, None, None, k, v, cu, 0, fused, idx, ws[0], ws[1],
                                mask_mode=neo.NEO_MASK_BLOCK_CAUSAL, t_img=T)
    qn = q.clone().reshape(S, Hq, 128)
    neo.neo_qknorm_rope3(qn, None, idx, ws[0], ws[1], None, None)
    plain = torch.empty_like(q)
    neo.neo_gen_attention(qn.view(1, S, Hq, 128), None, None, k, v, cu, 0, plain,
                          mask_mode=neo.NEO_MASK_BLOCK_CAUSAL, t_img=T)
    assert torch.equal(fused, plain)


def test_fused_rejects_missing_parameters(gpu_lib):
    q = torch.zeros(1, 8, 4, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 8, 1, 128, dtype=torch.bfloat16, device="cuda")
    cu = torch.zeros(2, dtype=torch.int32, device="cuda")
    idx = torch.zeros(3, 8, dtype=torch.int32, device="cuda")
    w = torch.ones(64, device="cuda")
    for kw in (dict(theta_t=0.0), dict(theta_hw=float("nan")), dict(eps=-1.0)):
        with pytest.raises(neo.NeoError) as e:
            neo.neo_gen_attention_qnorm(q, None, None, k, k, cu, 0, q.clone(), idx, w, w, **kw)
        assert e.value.status == neo.NEO_ERR_INVALID_ARG


def test_fused_equals_two_launches_at_large_positions(gpu_lib):
    """Positions up to 2^30 on every axis: the folded prologue and the
    standalone kernel reduce the angles the same way, so the bits agree."""
    S, Hq, Hkv = 200, 8, 2
    g = torch.Generator().manual_seed(6)
    q = torch.randn(1, S, Hq, 128, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(1, S, Hkv, 128, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(1, S, Hkv, 128, generator=g).to(torch.bfloat16).cuda()
    ws = [(torch.rand(64, generator=g) + 0.5).cuda() for _ in range(2)]
    idx = torch.randint(0, 1 << 30, (3, S), generator=g, dtype=torch.int32).cuda()
    cu = torch.zeros(2, dtype=torch.int32, device="cuda")
    fused = torch.empty_like(q)
    neo.neo_gen_attention_qnorm(q, None, None, k, v, cu, 0, fused, idx, ws[0], ws[1])
    qn = q.clone().reshape(S, Hq, 128)
    neo.neo_qknorm_rope3(qn, None, idx, ws[0], ws[1], None, None)
    plain = torch.empty_like(q)
    neo.neo_gen_attention(qn.view(1, S, Hq, 128), None, None, k, v, cu, 0, plain)
    assert torch.equal(fused, plain)

"""The persistent full-mask attention kernel on shapes the workload suite does
not reach: one unit with a very long prefix, a batch of more than a thousand
short sequences with ragged and empty prefixes, and repeated launches (every
launch must give the same bits)."""

import numpy as np
import pytest
import torch

import oracle as O
from attention_neo_qknorm_gb300 import neo, synth
from helpers import GpuLayer, SCALE, assert_bf16_close, f64, oracle_layer

pytestmark = pytest.mark.gpu


def check_device_ok():
    st, word = neo.neo_get_device_error()
    assert word == 0, f"device error word {word:#x}"


def test_one_unit_with_a_long_prefix(gpu_lib):
    """A 20000-token prefix: one unit of 158 key tiles per KV head."""
    w = synth.small_workload(prefix=(20000,), grid=(8, 8), Hq=4, Hkv=1, B=1)
    inp = synth.make_inputs(w, seed=5)
    layer = GpuLayer(w, inp)
    layer.norm_rope()
    layer.attention()
    torch.cuda.synchronize()
    check_device_ok()
    ref, ref_lse = oracle_layer(w, inp)
    assert_bf16_close(f64(layer.out), ref, "long prefix vs oracle")
    np.testing.assert_allclose(f64(layer.lse), ref_lse, rtol=1e-3, atol=2e-2)


def test_repeated_launches_identical(gpu_lib):
    """Ten launches in a row give the same bits."""
    w = synth.small_workload(prefix=(1000, 300), grid=(24, 16), Hq=32, Hkv=8, B=2)
    inp = synth.make_inputs(w, seed=3)
    layer = GpuLayer(w, inp)
    layer.norm_rope()
    layer.attention()
    torch.cuda.synchronize()
    first, first_lse = layer.out.clone(), layer.lse.clone()
    for _ in range(9):
        layer.attention()
    torch.cuda.synchronize()
    check_device_ok()
    assert torch.equal(layer.out, first)
    assert torch.equal(layer.lse, first_lse)


def test_many_short_sequences(gpu_lib):
    """1100 sequences of 4 image tokens with prefixes of 0..39 tokens."""
    g = torch.Generator().manual_seed(17)
    B, N, Hq, Hkv, D = 1100, 4, 4, 1, 128
    lens = torch.randint(0, 40, (B,), generator=g)
    cu = torch.zeros(B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(lens, 0)
    total = int(cu[-1])
    q = torch.randn(B, N, Hq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, N, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, N, Hkv, D, generator=g).to(torch.bfloat16)
    kp = torch.randn(total, Hkv, D, generator=g).to(torch.bfloat16)
    vp = torch.randn(total, Hkv, D, generator=g).to(torch.bfloat16)
    dq, dk, dv, dkp, dvp, dcu = (t.cuda() for t in (q, k, v, kp, vp, cu))
    out = torch.empty(B, N, Hq, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, Hq, N, dtype=torch.float32, device="cuda")
    neo.neo_gen_attention(dq, dkp, dvp, dk, dv, dcu, int(lens.max()), out, scale=SCALE, lse=lse)
    torch.cuda.synchronize()
    check_device_ok()
    ref, ref_lse = O.gen_attention(f64(q), f64(kp), f64(vp), f64(k), f64(v), cu.numpy(), SCALE)
    assert_bf16_close(f64(out.cpu()), ref, "1100 sequences, every row")
    np.testing.assert_allclose(f64(lse.cpu()), ref_lse, rtol=1e-3, atol=2e-2)


@pytest.mark.parametrize("mode", ["full", "folded", "prefill"])
def test_norm_then_attention_back_to_back(gpu_lib, mode):
    """The attention is launched so that its CTAs may start while the QK-norm
    kernel before it drains; it must still read the normed q and k. Ten rounds
    over fresh raw inputs, norm and attention back to back in one stream, give
    the same bits as the same rounds with a device synchronisation between the
    two launches: the full mask, the query norm folded into the attention (the
    keys' norm before it), and a one-sequence block-causal prefill."""
    if mode == "prefill":
        w = synth.small_workload(prefix=(0,), grid=(30, 30), Hq=32, Hkv=8, B=1)
    else:
        w = synth.small_workload(prefix=(700, 300), grid=(24, 24), Hq=32, Hkv=8, B=2)
    layer = GpuLayer(w, synth.make_inputs(w, seed=41))
    g = torch.Generator(device="cuda").manual_seed(42)
    raws = [(torch.randn(layer.q.shape, device="cuda", generator=g).to(torch.bfloat16),
             torch.randn(layer.k.shape, device="cuda", generator=g).to(torch.bfloat16)) for _ in range(10)]
    # A prefill: text-like temporal indexes, runs of 40 tokens sharing one.
    t_img = (torch.arange(w.N, dtype=torch.int32, device="cuda") // 40).contiguous()

    def rounds(sync):
        outs = []
        for q_raw, k_raw in raws:
            layer.q.copy_(q_raw)
            layer.k.copy_(k_raw)
            if mode == "folded":
                layer.norm_rope_k()
            else:
                layer.norm_rope()
            if sync:
                torch.cuda.synchronize()
            if mode == "folded":
                layer.attention_qnorm()
            elif mode == "prefill":
                neo.neo_gen_attention(layer.q.view(1, w.N, w.Hq, w.D), None, None,
                                      layer.k.view(1, w.N, w.Hkv, w.D), layer.v, layer.cu, 0, layer.out,
                                      scale=SCALE, lse=layer.lse, mask_mode=neo.NEO_MASK_BLOCK_CAUSAL,
                                      t_img=t_img)
            else:
                layer.attention()
            outs.append((layer.out.clone(), layer.lse.clone()))
        torch.cuda.synchronize()
        return outs

    serial = rounds(True)
    overlapped = rounds(False)
    check_device_ok()
    for (a, la), (b, lb) in zip(serial, overlapped):
        assert torch.equal(a, b) and torch.equal(la, lb)
    # and the rounds differ from one another (the inputs changed)
    assert not torch.equal(serial[0][0], serial[1][0])

"""Steps captured in a CUDA graph and replayed give exactly the results of
the same libneo calls launched one by one: every entry point enqueues its
work on the given stream only, so a capture records all of it (including the
programmatic dependent launch from the norm into the attention)."""

import pytest
import torch

from attention_neo_qknorm_gb300 import neo, synth
from attention_neo_qknorm_gb300.pipeline import GenPassLayer

pytestmark = pytest.mark.gpu


def _capture(fn):
    """fn() captured once in a CUDA graph on a side stream; nothing runs yet."""
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=cap):
        fn()
    torch.cuda.current_stream().wait_stream(cap)
    return g


@pytest.mark.parametrize("name", ["small", "gen_2048"])
@pytest.mark.parametrize("fused", [False, True])
def test_replayed_steps_equal_eager_steps(gpu_lib, name, fused):
    w = synth.small_workload(t_steps=(0.2, 0.3, 0.4)) if name == "small" else synth.WORKLOADS[name]
    inp = synth.make_inputs(w, seed=11)
    z0, (x0,) = synth.make_flow(w, seed=11)
    ts = [0.2, 0.3, 0.4]

    def run(L):
        for t in ts:
            L.step(t, t + 0.1, fused=fused)
            if fused:
                L.attention_qnorm(lse=True)
            else:
                L.attention(lse=True)

    eager = GenPassLayer(w, inp, z=z0, x0=x0)
    run(eager)
    torch.cuda.synchronize()

    graphed = GenPassLayer(w, inp, z=z0, x0=x0)
    torch.cuda.synchronize()
    g = _capture(lambda: run(graphed))
    # the capture ran nothing: the buffers still hold the inputs
    assert not torch.equal(graphed.z, eager.z)
    g.replay()
    torch.cuda.synchronize()
    st, word = neo.neo_get_device_error()
    assert st == neo.NEO_OK, hex(word)
    for name_ in ("q", "k", "out", "lse", "z"):
        assert torch.equal(getattr(graphed, name_), getattr(eager, name_)), name_


def test_replayed_block_causal_prefill_equals_eager(gpu_lib):
    """The block-causal mode (per-token temporal indexes from the positions
    kernel, no prefix) under capture and replay."""
    segs = [("text", 0, 96), ("image", 96, 24, 20), ("text", 97, 130)]
    S, Hq, Hkv = 96 + 480 + 130, 8, 2
    dev = torch.device("cuda")
    idx = torch.empty(3, S, dtype=torch.int32, device=dev)
    neo.neo_build_positions(idx, segs)
    T = idx[0].contiguous()
    g = torch.Generator(device=dev).manual_seed(12)
    q, k, v = (torch.randn(1, S, h, 128, device=dev, generator=g).to(torch.bfloat16) for h in (Hq, Hkv, Hkv))
    cu = torch.zeros(2, dtype=torch.int32, device=dev)
    outs = [torch.empty_like(q) for _ in range(2)]
    lses = [torch.empty(1, Hq, S, dtype=torch.float32, device=dev) for _ in range(2)]

    def call(i):
        neo.neo_gen_attention(q, None, None, k, v, cu, 0, outs[i], scale=128 ** -0.5, lse=lses[i],
                              mask_mode=neo.NEO_MASK_BLOCK_CAUSAL, t_img=T)
    call(0)
    torch.cuda.synchronize()
    gr = _capture(lambda: call(1))
    gr.replay()
    gr.replay()
    torch.cuda.synchronize()
    st, word = neo.neo_get_device_error()
    assert st == neo.NEO_OK, hex(word)
    assert torch.equal(outs[1], outs[0])
    assert torch.equal(lses[1], lses[0])

"""The host-streamed step driver (copies overlapped with compute on two
request slots) gives exactly the results of running the same steps one after
another."""

import pytest
import torch

from attention_neo_qknorm_gb300 import synth
from attention_neo_qknorm_gb300.pipeline import GenPassLayer, StreamedSteps

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fused", [False, True])
def test_streamed_steps_equal_serial_steps(gpu_lib, fused):
    w = synth.small_workload(t_steps=(0.1, 0.2, 0.3, 0.4, 0.5))
    inp = synth.make_inputs(w, seed=3)
    z0, (x0,) = synth.make_flow(w, seed=3)

    def slot():
        return GenPassLayer(w, inp, z=z0, x0=x0)
    h_in = {name: getattr(slot(), name).cpu().pin_memory() for name in ("q", "k", "v", "x0")}
    steps = [(0.1 * s, 0.1 * s + 0.1) for s in range(6)]

    # serial reference: each step loads its inputs, runs, reads its results
    ref = [slot(), slot()]
    ref_out = [None, None]
    for s, (t, tn) in enumerate(steps):
        L = ref[s % 2]
        for name in ("q", "k", "v", "x0"):
            getattr(L, name).copy_(h_in[name])
        L.step(t, tn, fused=fused)
        ref_out[s % 2] = (L.out.cpu(), L.z.cpu())

    slots = [slot(), slot()]
    h_out = [{"out": torch.empty(S.out.shape, dtype=S.out.dtype).pin_memory(),
              "z": torch.empty(S.z.shape, dtype=S.z.dtype).pin_memory()} for S in slots]
    runner = StreamedSteps(slots, h_in, h_out, fused=fused)
    for s, (t, tn) in enumerate(steps):
        runner.step(s, t, tn)
    runner.finish()
    torch.cuda.synchronize()
    for i in range(2):
        assert torch.equal(h_out[i]["out"], ref_out[i][0])
        assert torch.equal(h_out[i]["z"], ref_out[i][1])

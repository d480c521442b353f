"""End-to-end parity of one generation-pass layer (positions -> QK-norm +
three-axis RoPE -> attention over prefix + image keys) on the five workloads,
in the launch configurations the benchmark times (query norm in place before
the attention, or folded into it), element by element over every output row
at full size; and each workload's Euler step on its whole z."""

import numpy as np
import pytest
import torch

import oracle as O
from attention_neo_qknorm_gb300 import neo, synth
from helpers import F32_TOL, GpuLayer, assert_bf16_close, f64, max_abs, oracle_layer, rel_frob

pytestmark = pytest.mark.gpu


def run_layer(layer, fused):
    """The step's norm + attention: queries normed in place before a plain
    attention, or (fused) keys normed in place and queries inside the attention."""
    if fused:
        layer.norm_rope_k()
        layer.attention_qnorm()
    else:
        layer.norm_rope()
        layer.attention()


@pytest.mark.parametrize("fused", [False, True])
def test_small_workload_full_compare(gpu_lib, fused):
    w = synth.small_workload()
    inp = synth.make_inputs(w, seed=77)
    layer = GpuLayer(w, inp)
    run_layer(layer, fused)
    ref, ref_lse = oracle_layer(w, inp)
    assert_bf16_close(f64(layer.out), ref, "small workload")
    np.testing.assert_allclose(f64(layer.lse), ref_lse, rtol=1e-3, atol=2e-2)


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_workload_layer_matches_oracle(gpu_lib, name):
    """Every output row and every log-sum-exp of the workload, both launch
    configurations, against one oracle computation of the whole layer."""
    w = synth.WORKLOADS[name]
    inp = synth.make_inputs(w)
    ref, ref_lse = oracle_layer(w, inp)
    for fused in (False, True):
        layer = GpuLayer(w, inp)
        run_layer(layer, fused)
        tag = f"{name} ({'folded query norm' if fused else 'norm then attention'}, all rows)"
        assert_bf16_close(f64(layer.out), ref, tag)
        np.testing.assert_allclose(f64(layer.lse), ref_lse, rtol=1e-3, atol=2e-2, err_msg=tag)
        del layer


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_workload_euler_step_matches_oracle(gpu_lib, name):
    """The workload's Euler step on its whole z (B*N x 3072 fp32), with the
    velocity written out, at its first flow time."""
    w = synth.WORKLOADS[name]
    z, (x0,) = synth.make_flow(w)
    t, tn = w.t_steps[0], w.t_steps[0] + w.dt
    zd, xd = z.cuda(), x0.cuda()
    vd = torch.empty_like(zd)
    neo.neo_flow_euler_step(zd, xd, t, tn, 0.02, vd)
    rz, rv = O.flow_euler_step(f64(z), f64(x0), np.float32(t), np.float32(tn), np.float32(0.02))
    assert max_abs(f64(zd), rz) <= F32_TOL * max(1.0, float(np.abs(rz).max()))
    assert rel_frob(f64(zd), rz) <= F32_TOL and rel_frob(f64(vd), rv) <= F32_TOL

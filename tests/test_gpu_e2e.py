"""End-to-end parity of one generation-pass layer (positions -> QK-norm +
three-axis RoPE -> attention over prefix + image keys) on the five workloads,
in the launch configurations the benchmark times (query norm in place before
the attention, or folded into it). Small workloads are compared
element by element; the full-size ones on sampled query rows that the oracle
computes one by one."""

import numpy as np
import pytest

from attention_neo_qknorm_gb300 import synth
from helpers import GpuLayer, assert_bf16_close, f64, oracle_layer, take_rows

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


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_workload_layer_matches_oracle(gpu_lib, name, fused):
    w = synth.WORKLOADS[name]
    inp = synth.make_inputs(w)
    layer = GpuLayer(w, inp)
    run_layer(layer, fused)
    if w.B * w.N * w.Hq <= 4096:
        ref, _ = oracle_layer(w, inp)
        assert_bf16_close(f64(layer.out), ref, name)
    else:
        rows = synth.random_rows(w, 384, seed=5)
        ref, _ = oracle_layer(w, inp, rows=rows)
        got = take_rows(f64(layer.out), rows)
        assert_bf16_close(got, ref, name + " (sampled rows)")

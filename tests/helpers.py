"""Shared test plumbing: the GPU layer pipeline through the C-ABI binding,
the oracle chain on the same seeded inputs, and the parity measures."""

from __future__ import annotations

import numpy as np
import torch

import oracle as O
from attention_neo_qknorm_gb300 import synth
from attention_neo_qknorm_gb300.pipeline import GenPassLayer, image_segments, prefix_segments  # noqa: F401

# Tolerances: bf16 inputs with fp32 accumulation, and the fp32 Euler step.
BF16_REL_FROB = 5e-3
BF16_MAX_ABS = 2e-2
F32_TOL = 1e-5
SCALE = 1.0 / np.sqrt(128.0)


def rel_frob(a, ref):
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(a - ref) / max(np.linalg.norm(ref), 1e-300))


def max_abs(a, ref):
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(ref, np.float64))))


def assert_bf16_close(a, ref, what=""):
    rf, ma = rel_frob(a, ref), max_abs(a, ref)
    assert rf <= BF16_REL_FROB and ma <= BF16_MAX_ABS, f"{what}: rel_frob={rf:.3e} max_abs={ma:.3e}"
    return rf, ma


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


GpuLayer = GenPassLayer


# ------------------------------------------------------------------ oracle side
def oracle_norm_rope(w, inp):
    idx = O.positions(image_segments(w))
    q = O.qknorm_rope3(f64(inp.q).reshape(w.B * w.N, w.Hq, w.D), idx, f64(inp.q_norm), f64(inp.q_norm_hw))
    k = O.qknorm_rope3(f64(inp.k).reshape(w.B * w.N, w.Hkv, w.D), idx, f64(inp.k_norm), f64(inp.k_norm_hw))
    return q.reshape(w.B, w.N, w.Hq, w.D), k.reshape(w.B, w.N, w.Hkv, w.D)


def oracle_prefix_keys(w, inp):
    if w.total_prefix == 0:
        return f64(inp.k_prefix_raw)
    idx = O.positions(prefix_segments(w))
    return O.qknorm_rope3(f64(inp.k_prefix_raw), idx, f64(inp.k_norm_und), f64(inp.k_norm_hw_und))


def oracle_layer(w, inp, rows=None):
    q, k = oracle_norm_rope(w, inp)
    kp = oracle_prefix_keys(w, inp)
    return O.gen_attention(q, kp, f64(inp.v_prefix), k, f64(inp.v), w.cu_prefix, SCALE, rows=rows)

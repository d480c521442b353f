"""Seeded synthetic workloads for the generation-pass hot path.

This module only draws random numbers and describes workload shapes. It holds
none of the method's arithmetic, so both the CUDA path and the CPU oracle can
be fed from it: every tensor it returns lives on the host, in the dtype the
hot path consumes, and both sides read the same values.

Workloads (one generation-pass layer; D = 128 head dim):
  tiny_ref     B=1, text prefix 32, 8x8 image tokens, 4 Q / 1 KV heads,
               values drawn fp32 then rounded to bf16, one Euler step
               t=0.6 -> 0.7
  gen_1024     B=1, text prefix 512, 32x32 image tokens, 32 Q / 8 KV heads
  gen_2048     B=1, text prefix 1024, 64x64 image tokens, 32 Q / 8 KV heads,
               Euler on 4096 x 3072 fp32 pixel patches
  edit_2048    B=2, prefix = 512 text tokens + a 32x32-token reference image at
               temporal index 512 (1536 cached keys), 64x64 gen tokens at 1536
  ragged_cfg   B=4, prefixes of 300/777/1500/2048 text tokens (packed, no
               padding), 64x64 gen tokens each, 10 flow steps t = 0 .. 0.9
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

HEAD_DIM = 128
PATCH_ELEMS = 32 * 32 * 3   # pixels per image token (32x32 RGB patch)


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    prefix_segments: tuple          # per sequence: tuple of position segments
    grid: tuple                     # (rows, cols) of image tokens per sequence
    Hq: int
    Hkv: int
    t_img: tuple                    # temporal index of each sequence's image tokens
    t_steps: tuple = (0.6,)         # flow times of the sampler steps
    dt: float = 0.1
    draw_fp32: bool = False         # values drawn in fp32 then rounded to bf16
    description: str = ""
    D: int = HEAD_DIM

    @property
    def N(self) -> int:
        return self.grid[0] * self.grid[1]

    @property
    def prefix_lens(self) -> tuple:
        out = []
        for segs in self.prefix_segments:
            n = 0
            for s in segs:
                n += s[2] if s[0] == "text" else s[2] * s[3]
            out.append(n)
        return tuple(out)

    @property
    def total_prefix(self) -> int:
        return sum(self.prefix_lens)

    @property
    def cu_prefix(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.prefix_lens)]).astype(np.int32)

    def image_segments(self, b: int) -> tuple:
        return (("image", self.t_img[b], self.grid[0], self.grid[1]),)

    @property
    def euler_elems(self) -> int:
        return self.B * self.N * PATCH_ELEMS

    def attention_flops(self) -> int:
        """4 * N * (L_b + N) * D * Hq summed over sequences (QK^T and PV)."""
        return sum(4 * self.N * (L + self.N) * self.D * self.Hq for L in self.prefix_lens)


def _text(n, start=0):
    return (("text", start, n),)


WORKLOADS = {
    "tiny_ref": Workload(
        name="tiny_ref", B=1, prefix_segments=(_text(32),), grid=(8, 8), Hq=4, Hkv=1,
        t_img=(32,), t_steps=(0.6,), dt=0.1, draw_fp32=True,
        description="B=1, text prefix 32, 8x8 gen tokens, 4 Q / 1 KV heads, one Euler step t=0.6 dt=0.1"),
    "gen_1024": Workload(
        name="gen_1024", B=1, prefix_segments=(_text(512),), grid=(32, 32), Hq=32, Hkv=8,
        t_img=(512,), description="1024^2 generation: B=1, text prefix 512, 32x32 gen tokens, 32 Q / 8 KV heads"),
    "gen_2048": Workload(
        name="gen_2048", B=1, prefix_segments=(_text(1024),), grid=(64, 64), Hq=32, Hkv=8,
        t_img=(1024,), description="2048^2 generation: B=1, text prefix 1024, 64x64 gen tokens, 32 Q / 8 KV heads, "
                                   "Euler on 4096x3072 fp32 patches"),
    "edit_2048": Workload(
        name="edit_2048", B=2,
        prefix_segments=((("text", 0, 512), ("image", 512, 32, 32)),) * 2,
        grid=(64, 64), Hq=32, Hkv=8, t_img=(1536, 1536),
        description="editing: B=2, prefix 512 text + 32x32 reference-image tokens at t=512 (1536 cached), "
                    "64x64 gen tokens at t=1536"),
    "ragged_cfg": Workload(
        name="ragged_cfg", B=4, prefix_segments=(_text(300), _text(777), _text(1500), _text(2048)),
        grid=(64, 64), Hq=32, Hkv=8, t_img=(300, 777, 1500, 2048),
        t_steps=tuple(k / 10 for k in range(10)), dt=0.1,
        description="ragged CFG batch: B=4, unpadded prefixes 300/777/1500/2048, 64x64 gen tokens each, "
                    "10 flow steps t=0..0.9"),
}

# Seeds are fixed per workload so that every run draws the same values.
SEEDS = {name: 1000 + i for i, name in enumerate(WORKLOADS)}


def small_workload(name="small", B=2, prefix=(200, 77), grid=(12, 11), Hq=8, Hkv=2,
                   t_steps=(0.3,)):
    """A parity-sized workload: several tiles, ragged tails, unequal prefixes."""
    return Workload(name=name, B=B, prefix_segments=tuple(_text(L) for L in prefix),
                    grid=grid, Hq=Hq, Hkv=Hkv, t_img=tuple(prefix), t_steps=t_steps,
                    description=f"parity case B={B} prefixes={prefix} grid={grid} {Hq}/{Hkv} heads")


@dataclass
class Inputs:
    """Host tensors of one workload. Raw q/k are the projections before the
    norm and the rotary embedding; k_prefix_raw likewise for the prefix keys
    that the understanding pass turns into the frozen cache."""
    q: torch.Tensor             # [B, N, Hq, D] bf16
    k: torch.Tensor             # [B, N, Hkv, D] bf16
    v: torch.Tensor             # [B, N, Hkv, D] bf16
    k_prefix_raw: torch.Tensor  # [sum L, Hkv, D] bf16
    v_prefix: torch.Tensor      # [sum L, Hkv, D] bf16
    q_norm: torch.Tensor        # [64] fp32 generation-branch weights
    q_norm_hw: torch.Tensor
    k_norm: torch.Tensor
    k_norm_hw: torch.Tensor
    k_norm_und: torch.Tensor    # [64] fp32 understanding-branch weights (prefix keys)
    k_norm_hw_und: torch.Tensor
    extra: dict = field(default_factory=dict)


def _normal_bf16(g, shape):
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def _weight(g):
    return torch.rand(64, generator=g, dtype=torch.float32) + 0.5   # U(0.5, 1.5)


def make_inputs(w: Workload, seed: int | None = None) -> Inputs:
    """Draw the attention-side inputs: Q/K/V ~ N(0,1) rounded to bf16 and norm
    weights ~ U(0.5, 1.5) in fp32."""
    g = torch.Generator().manual_seed(SEEDS.get(w.name, 7) if seed is None else seed)
    q = _normal_bf16(g, (w.B, w.N, w.Hq, w.D))
    k = _normal_bf16(g, (w.B, w.N, w.Hkv, w.D))
    v = _normal_bf16(g, (w.B, w.N, w.Hkv, w.D))
    kp = _normal_bf16(g, (w.total_prefix, w.Hkv, w.D))
    vp = _normal_bf16(g, (w.total_prefix, w.Hkv, w.D))
    ws = [_weight(g) for _ in range(6)]
    return Inputs(q, k, v, kp, vp, *ws)


def make_flow(w: Workload, seed: int | None = None, n_x0: int = 1):
    """Draw the sampler state z ~ N(0,1) and ``n_x0`` predicted clean images
    x0_hat ~ N(0,1), fp32 [B*N, 3072] (pixel patches)."""
    g = torch.Generator().manual_seed((SEEDS.get(w.name, 7) if seed is None else seed) + 500)
    z = torch.randn(w.B * w.N, PATCH_ELEMS, generator=g, dtype=torch.float32)
    x0 = [torch.randn(w.B * w.N, PATCH_ELEMS, generator=g, dtype=torch.float32) for _ in range(n_x0)]
    return z, x0

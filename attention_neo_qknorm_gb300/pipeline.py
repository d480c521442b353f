"""One generation-pass layer's hot path as a sequence of libneo calls.

Plumbing only: device buffers (torch) and the order of the C-ABI calls.
Every step runs in a libneo kernel.
"""

from __future__ import annotations

import torch

from . import neo, synth

SCALE = 128 ** -0.5


def image_segments(w: synth.Workload):
    return [s for b in range(w.B) for s in w.image_segments(b)]


def prefix_segments(w: synth.Workload):
    return [s for segs in w.prefix_segments for s in segs]


class GenPassLayer:
    """Device buffers of one workload and the hot-path step.

    The frozen prefix cache is produced on construction the way the
    understanding pass writes it: the raw prefix keys go through the QK-norm
    and the three-axis RoPE with the prefix positions and the understanding
    branch's norm weights; the prefix values are stored unchanged.
    """

    def __init__(self, w: synth.Workload, inp: synth.Inputs, device="cuda", z=None, x0=None):
        self.w = w
        d = device
        self.q = inp.q.to(d).reshape(w.B * w.N, w.Hq, w.D).contiguous()
        self.k = inp.k.to(d).reshape(w.B * w.N, w.Hkv, w.D).contiguous()
        self.v = inp.v.to(d).contiguous()
        self.k_prefix = inp.k_prefix_raw.to(d).contiguous()
        self.v_prefix = inp.v_prefix.to(d).contiguous()
        self.wts = [t.to(d) for t in (inp.q_norm, inp.q_norm_hw, inp.k_norm, inp.k_norm_hw,
                                      inp.k_norm_und, inp.k_norm_hw_und)]
        self.cu = torch.from_numpy(w.cu_prefix).to(d)
        self.idx_img = torch.empty(3, w.B * w.N, dtype=torch.int32, device=d)
        neo.neo_build_positions(self.idx_img, image_segments(w))
        self.out = torch.empty(w.B, w.N, w.Hq, w.D, dtype=torch.bfloat16, device=d)
        self.lse = torch.empty(w.B, w.Hq, w.N, dtype=torch.float32, device=d)
        self.max_prefix = max(w.prefix_lens) if w.prefix_lens else 0
        if w.total_prefix > 0:
            self.idx_pre = torch.empty(3, w.total_prefix, dtype=torch.int32, device=d)
            neo.neo_build_positions(self.idx_pre, prefix_segments(w))
            neo.neo_qknorm_rope3(None, self.k_prefix, self.idx_pre, None, None, self.wts[4], self.wts[5])
        self.z = z.to(d).contiguous() if z is not None else None
        self.x0 = x0.to(d).contiguous() if x0 is not None else None

    def norm_rope(self, stream=None):
        neo.neo_qknorm_rope3(self.q, self.k, self.idx_img, *self.wts[:4], stream=stream)

    def norm_rope_k(self, stream=None):
        """The keys only: the queries' norm + RoPE is folded into attention_qnorm."""
        neo.neo_qknorm_rope3(None, self.k, self.idx_img, None, None, *self.wts[2:4], stream=stream)

    def attention(self, lse=True, stream=None):
        w = self.w
        neo.neo_gen_attention(self.q.view(w.B, w.N, w.Hq, w.D), self.k_prefix, self.v_prefix,
                              self.k.view(w.B, w.N, w.Hkv, w.D), self.v, self.cu, self.max_prefix, self.out,
                              scale=SCALE, lse=self.lse if lse else None, stream=stream)

    def attention_qnorm(self, lse=True, stream=None):
        """Attention over the raw queries (self.q, left unchanged), normalised
        and rotated inside the attention kernel."""
        w = self.w
        neo.neo_gen_attention_qnorm(self.q.view(w.B, w.N, w.Hq, w.D), self.k_prefix, self.v_prefix,
                                    self.k.view(w.B, w.N, w.Hkv, w.D), self.v, self.cu, self.max_prefix, self.out,
                                    self.idx_img, self.wts[0], self.wts[1], scale=SCALE,
                                    lse=self.lse if lse else None, stream=stream)

    def euler(self, t, t_next, t_eps=0.02, stream=None):
        neo.neo_flow_euler_step(self.z, self.x0, t, t_next, t_eps, stream=stream)

    def step(self, t, t_next, stream=None, fused=False):
        """Queries and keys normed in place, then attention and the Euler step;
        fused: keys normed in place and the queries inside the attention
        (self.q stays raw)."""
        if fused:
            self.norm_rope_k(stream)
            self.attention_qnorm(lse=False, stream=stream)
        else:
            self.norm_rope(stream)
            self.attention(lse=False, stream=stream)
        self.euler(t, t_next, stream=stream)


class StreamedSteps:
    """Steps whose inputs arrive from pinned host memory and whose results go
    back to it, with the copies of one step overlapping the compute of its
    neighbours.

    Two request slots (each a GenPassLayer with its own device buffers) take
    turns; slot s % 2 runs step s. Three streams: host-to-device copies of a
    step's inputs (q, k, v, x0_hat), the step itself on the compute stream,
    and device-to-host copies of its results (the attention output and z).
    Events order every reuse of a buffer: a slot's inputs are overwritten only
    after its previous step has computed, its compute waits for its inputs and
    for the read-back of its previous results, and a read-back waits for the
    compute. Plumbing only: the step is the same sequence of libneo calls.
    """

    def __init__(self, slots, h_inputs, h_outputs, fused=False):
        """slots: two GenPassLayer; h_inputs: dict of pinned host tensors
        q, k, v, x0 (shaped like the slot's buffers); h_outputs: per slot, a
        dict of pinned host tensors out, z."""
        assert len(slots) == 2 and len(h_outputs) == 2
        self.slots, self.h_in, self.h_out, self.fused = slots, h_inputs, h_outputs, fused
        dev = slots[0].q.device
        self.s_in = torch.cuda.Stream(dev)
        self.s_out = torch.cuda.Stream(dev)
        self.computed = [torch.cuda.Event() for _ in range(2)]
        self.loaded = [torch.cuda.Event() for _ in range(2)]
        self.read = [torch.cuda.Event() for _ in range(2)]
        self.started = [False, False]

    def step(self, s, t, t_next):
        i = s % 2
        L = self.slots[i]
        comp = torch.cuda.current_stream(L.q.device)
        with torch.cuda.stream(self.s_in):
            if self.started[i]:
                self.s_in.wait_event(self.computed[i])
            for name in ("q", "k", "v", "x0"):
                getattr(L, name).copy_(self.h_in[name], non_blocking=True)
            self.loaded[i].record(self.s_in)
        comp.wait_event(self.loaded[i])
        if self.started[i]:
            comp.wait_event(self.read[i])
        L.step(t, t_next, fused=self.fused)
        self.computed[i].record(comp)
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_event(self.computed[i])
            self.h_out[i]["out"].copy_(L.out, non_blocking=True)
            self.h_out[i]["z"].copy_(L.z, non_blocking=True)
            self.read[i].record(self.s_out)
        self.started[i] = True

    def finish(self):
        """Make the compute stream wait for every copy still in flight."""
        comp = torch.cuda.current_stream(self.slots[0].q.device)
        comp.wait_stream(self.s_in)
        comp.wait_stream(self.s_out)

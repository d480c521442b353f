"""fp64 CPU oracle of the NEO-unify generation-pass hot path.

TEST INFRASTRUCTURE: imported only by tests/, by the smoke check in
__graft_entry__ and by the CPU-baseline leg of bench.py. The CUDA library and
its Python binding never import it; the two share no code.
"""

from .neo_oracle import (  # noqa: F401
    CFG_CLASSIC,
    CFG_DUAL,
    CFG_NONE,
    CFG_TEXT,
    HEAD_DIM,
    MASK_BLOCK_CAUSAL,
    MASK_FULL,
    NOISE_CONSTANT,
    NOISE_DYNAMIC,
    NOISE_DYNAMIC_SQRT,
    NOISE_RESOLUTION,
    cfg_branch,
    flow_cfg_euler_step,
    flow_euler_step,
    flow_interpolant,
    flow_target_velocity,
    gen_attention,
    initial_noise,
    noise_scale,
    positions,
    qknorm_halves,
    qknorm_rope3,
    rope2d_interleaved,
    rope3,
    rope_slices,
    time_schedule,
    write_prefix_cache,
)

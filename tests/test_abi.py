"""The C-ABI library builds, loads, exports every entry point declared in
include/neo.h, and rejects bad arguments on the host before touching a GPU.
No GPU: every call here returns before any CUDA API call."""

import ctypes
import os
import re

import pytest

from attention_neo_qknorm_gb300 import neo
from attention_neo_qknorm_gb300.build import INCLUDE, build

HEADER = os.path.join(INCLUDE, "neo.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return neo.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(neo_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for required in ("neo_qknorm_rope3", "neo_gen_attention", "neo_flow_euler_step"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names
    for name in names:
        assert hasattr(lib, name), f"libneo.so does not export {name}"
    assert set(neo.EXPORTS) <= set(names)


def test_status_strings_and_version(lib):
    assert neo.neo_version() == 100
    for st in range(6):
        assert lib.neo_status_string(st).decode().startswith("NEO_")


V = ctypes.c_void_p
FAKE = V(0x10000)          # aligned, never dereferenced: the checks fail first
FAKE2 = V(0x4000000)       # a second buffer that overlaps no other fake one at the sizes used here
FAKE3 = V(0x8000000)
MISALIGNED = V(0x10008)


def _attn(lib, **kw):
    a = dict(q=FAKE, kp=FAKE, vp=FAKE, ki=FAKE, vi=FAKE, dt=neo.NEO_BF16, cu=FAKE, total=10, maxp=10,
             B=1, N=64, Hq=32, Hkv=8, D=128, mask=0, tp=None, ti=None, scale=0.088, out=FAKE,
             lse=None, stream=None)
    a.update(kw)
    return lib.neo_gen_attention(a["q"], a["kp"], a["vp"], a["ki"], a["vi"], a["dt"], a["cu"], a["total"],
                                 a["maxp"], a["B"], a["N"], a["Hq"], a["Hkv"], a["D"], a["mask"], a["tp"],
                                 a["ti"], a["scale"], a["out"], a["lse"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(D=64), neo.NEO_ERR_INVALID_ARG),
    (dict(Hq=30, Hkv=8), neo.NEO_ERR_INVALID_ARG),
    (dict(N=0), neo.NEO_ERR_INVALID_ARG),
    (dict(B=0), neo.NEO_ERR_INVALID_ARG),
    (dict(q=None), neo.NEO_ERR_INVALID_ARG),
    (dict(out=None), neo.NEO_ERR_INVALID_ARG),
    (dict(cu=None), neo.NEO_ERR_INVALID_ARG),
    (dict(kp=None), neo.NEO_ERR_INVALID_ARG),
    (dict(q=MISALIGNED), neo.NEO_ERR_INVALID_ARG),
    (dict(vp=MISALIGNED), neo.NEO_ERR_INVALID_ARG),
    (dict(scale=-1.0), neo.NEO_ERR_INVALID_ARG),
    (dict(scale=float("nan")), neo.NEO_ERR_INVALID_ARG),
    (dict(total=-1), neo.NEO_ERR_INVALID_ARG),
    (dict(mask=7), neo.NEO_ERR_INVALID_ARG),
    (dict(mask=1), neo.NEO_ERR_INVALID_ARG),                       # block-causal without temporal indices
    (dict(mask=1, ti=FAKE), neo.NEO_ERR_INVALID_ARG),              # ... prefix rows need theirs too
    (dict(mask=1, ti=FAKE, tp=FAKE, N=1024 * 128 + 1), neo.NEO_ERR_UNSUPPORTED),   # image segment too long
    (dict(dt=neo.NEO_F32), neo.NEO_ERR_UNSUPPORTED),
    (dict(Hq=3, Hkv=1), neo.NEO_ERR_UNSUPPORTED),
])
def test_attention_rejects_bad_arguments(lib, kw, status):
    assert _attn(lib, **kw) == status


def test_qknorm_rope3_rejects_bad_arguments(lib):
    f = lib.neo_qknorm_rope3
    args = [FAKE, FAKE2, neo.NEO_BF16, 16, 4, 1, 128, FAKE, FAKE, FAKE, FAKE, FAKE, 5e6, 1e4, 1e-6, None]
    bad = {6: 64, 2: 9, 0: MISALIGNED, 8: None, 12: -1.0, 14: float("inf"), 3: -5}
    for pos, val in bad.items():
        a = list(args)
        a[pos] = val
        assert f(*a) == neo.NEO_ERR_INVALID_ARG, pos
    a = list(args)
    a[3] = 0                        # S == 0: nothing to do
    assert f(*a) == neo.NEO_OK
    a = list(args)
    a[7] = None                     # indexes missing
    assert f(*a) == neo.NEO_ERR_INVALID_ARG
    a = list(args)
    a[1] = V(0x10000 + 16 * 4 * 128 * 2 - 256)   # k starts inside q
    assert f(*a) == neo.NEO_ERR_INVALID_ARG


def test_euler_rejects_bad_arguments(lib):
    f = lib.neo_flow_euler_step
    assert f(FAKE, FAKE2, 0, 0.5, 0.6, 0.02, None, None) == neo.NEO_OK
    assert f(None, FAKE2, 8, 0.5, 0.6, 0.02, None, None) == neo.NEO_ERR_INVALID_ARG
    assert f(MISALIGNED, FAKE2, 8, 0.5, 0.6, 0.02, None, None) == neo.NEO_ERR_INVALID_ARG
    assert f(FAKE, FAKE2, 8, 1.0, 1.1, 0.0, None, None) == neo.NEO_ERR_INVALID_ARG   # max(1-t, t_eps) = 0
    assert f(FAKE, FAKE2, 8, float("nan"), 0.6, 0.02, None, None) == neo.NEO_ERR_INVALID_ARG


def test_euler_rejects_overlapping_buffers(lib):
    """z is read and written, x0_hat read, v_out written: any overlap between
    them would let one element's write change another's input."""
    f = lib.neo_flow_euler_step
    n = 1024
    assert f(FAKE, FAKE, n, 0.5, 0.6, 0.02, None, None) == neo.NEO_ERR_INVALID_ARG            # x0_hat is z
    assert f(FAKE, V(0x10000 + 4 * n - 16), n, 0.5, 0.6, 0.02, None, None) == neo.NEO_ERR_INVALID_ARG
    assert f(FAKE, FAKE2, n, 0.5, 0.6, 0.02, FAKE, None) == neo.NEO_ERR_INVALID_ARG          # v_out is z
    assert f(FAKE, FAKE2, n, 0.5, 0.6, 0.02, FAKE2, None) == neo.NEO_ERR_INVALID_ARG         # v_out is x0_hat
    fc = lib.neo_flow_cfg_euler_step
    # dual CFG: z overlapping a prediction, v_out overlapping z or a prediction
    assert fc(FAKE, FAKE, FAKE2, FAKE3, n, 0.5, 0.6, 0.02, 4.0, 1.5, 0.0, 1.0, None, None, None) == \
        neo.NEO_ERR_INVALID_ARG
    assert fc(FAKE, FAKE2, FAKE3, V(0xC000000), n, 0.5, 0.6, 0.02, 4.0, 1.5, 0.0, 1.0, FAKE3, None, None) == \
        neo.NEO_ERR_INVALID_ARG
    assert fc(FAKE, FAKE2, FAKE3, V(0xC000000), n, 0.5, 0.6, 0.02, 4.0, 1.5, 0.0, 1.0, FAKE, None, None) == \
        neo.NEO_ERR_INVALID_ARG


def test_positions_rejects_bad_segments(lib):
    Seg = neo.neo_pos_segment
    segs = (Seg * 2)(Seg(neo.NEO_SEG_TEXT, 0, 4, 0), Seg(neo.NEO_SEG_IMAGE, 4, 2, 3))
    f = lib.neo_build_positions
    assert f(FAKE, 9, segs, 2, None) == neo.NEO_ERR_INVALID_ARG      # counts sum to 10
    assert f(None, 10, segs, 2, None) == neo.NEO_ERR_INVALID_ARG
    assert f(FAKE, 10, segs, 0, None) == neo.NEO_ERR_INVALID_ARG
    bad = (Seg * 1)(Seg(5, 0, 1, 1))
    assert f(FAKE, 1, bad, 1, None) == neo.NEO_ERR_INVALID_ARG


def test_cfg_euler_rejects_missing_predictions(lib):
    f = lib.neo_flow_cfg_euler_step
    br = ctypes.c_int32(-1)
    # text CFG needs the text-unconditional prediction
    assert f(FAKE, FAKE, None, None, 8, 0.5, 0.6, 0.02, 4.0, 1.0, 0.0, 1.0, None, ctypes.byref(br), None) == \
        neo.NEO_ERR_INVALID_ARG
    assert br.value == neo.NEO_CFG_TEXT
    # dual CFG needs both
    assert f(FAKE, FAKE, FAKE, None, 8, 0.5, 0.6, 0.02, 4.0, 1.5, 0.0, 1.0, None, ctypes.byref(br), None) == \
        neo.NEO_ERR_INVALID_ARG
    assert br.value == neo.NEO_CFG_DUAL
    # n == 0: nothing to do, but the branch is still reported
    assert f(None, None, None, None, 0, 0.7, 0.8, 0.02, 3.0, 3.0, 0.6, 1.0, None, ctypes.byref(br), None) == neo.NEO_OK
    assert br.value == neo.NEO_CFG_CLASSIC
    assert f(FAKE, MISALIGNED, None, None, 8, 0.5, 0.6, 0.02, 1.0, 1.0, 0.0, 1.0, None, None, None) == \
        neo.NEO_ERR_INVALID_ARG


def test_sampler_host_functions_match_the_oracle(lib):
    """Host-side entry points: no GPU involved."""
    import numpy as np
    import oracle as O
    for n, shift in ((50, 3.0), (10, 1.0), (20, 0.5)):
        np.testing.assert_allclose(neo.neo_time_schedule(n, shift), O.time_schedule(n, shift), atol=1e-7)
    for args in ((128, 128, 2, 64, 1.0, 0), (128, 128, 2, 64, 1.0, 2), (64, 64, 2, 64, 3.0, 1), (128, 128, 2, 64, 3.0, 0),
                 (100, 60, 2, 64, 0.7, 3)):
        assert neo.neo_noise_scale(*args) == pytest.approx(O.noise_scale(*args), rel=1e-6)
    assert neo.neo_noise_scale(128, 128, 2, 64, 3.0, 0, max_value=8.0) == pytest.approx(8.0)
    with pytest.raises(neo.NeoError):
        neo.neo_time_schedule(0, 3.0)
    with pytest.raises(neo.NeoError):
        neo.neo_noise_scale(128, 128, 2, 64, 1.0, 9)
    assert lib.neo_scale_noise(None, None, 0, 2.0, None) == neo.NEO_OK
    assert lib.neo_scale_noise(MISALIGNED, FAKE, 8, 2.0, None) == neo.NEO_ERR_INVALID_ARG


def test_rope2d_rejects_bad_arguments(lib):
    f = lib.neo_rope2d_interleaved
    assert f(FAKE, neo.NEO_BF16, 1, 4, 4, 1022, 1e4, None) == neo.NEO_ERR_INVALID_ARG    # C % 4
    assert f(FAKE, neo.NEO_BF16, 1, 4, 4, 12, 1e4, None) == neo.NEO_ERR_INVALID_ARG      # bf16 needs C % 8
    assert f(FAKE, neo.NEO_BF16, 1, 4, 4, 16, -1.0, None) == neo.NEO_ERR_INVALID_ARG
    assert f(MISALIGNED, neo.NEO_F32, 1, 4, 4, 16, 1e4, None) == neo.NEO_ERR_INVALID_ARG
    assert f(None, neo.NEO_F32, 0, 4, 4, 16, 1e4, None) == neo.NEO_OK


def test_fused_attention_rejects_bad_qnorm(lib):
    f = lib.neo_gen_attention_qnorm
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, neo.NEO_BF16, FAKE, 10, 10, 1, 64, 32, 8, 128, 0, None, None]
    tail = [0.088, FAKE, None, None]
    assert f(*args, None, *tail) == neo.NEO_ERR_INVALID_ARG                 # no qnorm parameters
    good = dict(indexes=0x10000, q_norm_w=0x10000, q_norm_hw_w=0x10000, theta_t=5e6, theta_hw=1e4, eps=1e-6)
    for bad in (dict(indexes=None), dict(q_norm_w=None), dict(q_norm_hw_w=None), dict(theta_t=0.0),
                dict(theta_hw=float("inf")), dict(eps=-1e-6)):
        qn = neo.neo_qnorm_params(**dict(good, **bad))
        assert f(*args, ctypes.byref(qn), *tail) == neo.NEO_ERR_INVALID_ARG, bad
    qn = neo.neo_qnorm_params(**good)
    a = list(args)
    a[13] = 64                                                             # D != 128 is still rejected
    assert f(*a, ctypes.byref(qn), *tail) == neo.NEO_ERR_INVALID_ARG


def test_prefix_cache_write_rejects_bad_arguments(lib):
    f = lib.neo_write_prefix_cache
    A, Bp, C, Dp = V(0x100000), V(0x200000), V(0x300000), V(0x400000)   # disjoint, aligned, never dereferenced
    args = dict(k_old=A, v_old=Bp, cu_old=FAKE, total_old=10, k_new=C, v_new=Dp, n_new=None, B=2, N=4, Hkv=1, D=128,
                dt=neo.NEO_BF16, k_out=V(0x500000), v_out=V(0x600000), cu_out=FAKE, cap=64, stream=None)

    def call(**kw):
        a = dict(args, **kw)
        return f(*a.values())
    assert call(D=64) == neo.NEO_ERR_INVALID_ARG
    assert call(cu_old=None) == neo.NEO_ERR_INVALID_ARG
    assert call(k_old=None) == neo.NEO_ERR_INVALID_ARG             # old rows but no buffer
    assert call(k_new=MISALIGNED) == neo.NEO_ERR_INVALID_ARG
    assert call(k_out=V(0x100000 + 256)) == neo.NEO_ERR_INVALID_ARG  # output overlaps the old keys
    assert call(v_out=V(0x300000)) == neo.NEO_ERR_INVALID_ARG        # output overlaps the chunk
    assert call(dt=7) == neo.NEO_ERR_INVALID_ARG
    assert call(total_old=100) == neo.NEO_ERR_UNSUPPORTED             # more old rows than capacity
    assert call(k_out=A, v_out=Bp) == neo.NEO_ERR_INVALID_ARG          # in place only for one sequence

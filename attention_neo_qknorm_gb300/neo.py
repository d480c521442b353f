"""Python binding of libneo: argument marshalling over ctypes, nothing else.

Each function has the name and the argument order of the C entry point
declared in include/neo.h; tensors are torch CUDA tensors whose device
pointers are passed through, and the launch goes on torch's current stream
unless ``stream`` is given. A non-OK status raises NeoError. There is no
fallback: if libneo.so is missing the first call raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libneo.so")

NEO_OK, NEO_ERR_INVALID_ARG, NEO_ERR_UNSUPPORTED, NEO_ERR_CUDA, NEO_ERR_TIMEOUT, NEO_ERR_DEVICE = range(6)
NEO_BF16, NEO_F32 = 0, 1
NEO_MASK_FULL, NEO_MASK_BLOCK_CAUSAL = 0, 1
NEO_SEG_TEXT, NEO_SEG_IMAGE = 0, 1
NEO_DEVERR_TIMEOUT, NEO_DEVERR_BAD_PREFIX = 0x1, 0x2
NEO_CFG_NONE, NEO_CFG_TEXT, NEO_CFG_CLASSIC, NEO_CFG_DUAL = range(4)
NEO_NOISE_RESOLUTION, NEO_NOISE_DYNAMIC, NEO_NOISE_DYNAMIC_SQRT, NEO_NOISE_CONSTANT = range(4)

EXPORTS = ("neo_build_positions", "neo_qknorm_rope3", "neo_gen_attention", "neo_gen_attention_qnorm",
           "neo_write_prefix_cache", "neo_flow_euler_step",
           "neo_flow_cfg_euler_step", "neo_time_schedule", "neo_noise_scale", "neo_scale_noise",
           "neo_rope2d_interleaved",
           "neo_status_string", "neo_get_device_error", "neo_set_wait_timeout_ns", "neo_selftest_bounded_wait",
           "neo_version")


class NeoError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


class neo_pos_segment(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("a", ctypes.c_int32), ("b", ctypes.c_int32), ("c", ctypes.c_int32)]


class neo_qnorm_params(ctypes.Structure):
    _fields_ = [("indexes", ctypes.c_void_p), ("q_norm_w", ctypes.c_void_p), ("q_norm_hw_w", ctypes.c_void_p),
                ("theta_t", ctypes.c_float), ("theta_hw", ctypes.c_float), ("eps", ctypes.c_float)]


_lib = None
_vp, _i32, _i64, _f32, _u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_uint64


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libneo.so once and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise FileNotFoundError(f"libneo.so not found at {path}; build it with "
                                "attention_neo_qknorm_gb300.build.build()")
    lib = ctypes.CDLL(path)
    c_int = ctypes.c_int
    lib.neo_build_positions.argtypes = [_vp, _i64, ctypes.POINTER(neo_pos_segment), c_int, _vp]
    lib.neo_qknorm_rope3.argtypes = [_vp, _vp, c_int, _i64, c_int, c_int, c_int, _vp, _vp, _vp, _vp, _vp,
                                     _f32, _f32, _f32, _vp]
    lib.neo_gen_attention.argtypes = [_vp, _vp, _vp, _vp, _vp, c_int, _vp, _i64, _i32, c_int, c_int, c_int,
                                      c_int, c_int, c_int, _vp, _vp, _f32, _vp, _vp, _vp]
    lib.neo_gen_attention_qnorm.argtypes = [_vp, _vp, _vp, _vp, _vp, c_int, _vp, _i64, _i32, c_int, c_int, c_int,
                                            c_int, c_int, c_int, _vp, _vp, ctypes.POINTER(neo_qnorm_params), _f32,
                                            _vp, _vp, _vp]
    lib.neo_flow_euler_step.argtypes = [_vp, _vp, _i64, _f32, _f32, _f32, _vp, _vp]
    lib.neo_write_prefix_cache.argtypes = [_vp, _vp, _vp, _i64, _vp, _vp, _vp, c_int, c_int, c_int, c_int, c_int,
                                           _vp, _vp, _vp, _i64, _vp]
    lib.neo_flow_cfg_euler_step.argtypes = [_vp, _vp, _vp, _vp, _i64, _f32, _f32, _f32, _f32, _f32, _f32, _f32,
                                            _vp, ctypes.POINTER(ctypes.c_int32), _vp]
    lib.neo_time_schedule.argtypes = [_vp, c_int, _f32]
    lib.neo_noise_scale.argtypes = [c_int, c_int, c_int, _f32, _f32, c_int, _f32, ctypes.POINTER(ctypes.c_float)]
    lib.neo_scale_noise.argtypes = [_vp, _vp, _i64, _f32, _vp]
    lib.neo_rope2d_interleaved.argtypes = [_vp, c_int, _i64, c_int, c_int, c_int, _f32, _vp]
    lib.neo_status_string.argtypes = [c_int]
    lib.neo_status_string.restype = ctypes.c_char_p
    lib.neo_get_device_error.argtypes = [_vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.neo_set_wait_timeout_ns.argtypes = [_u64]
    lib.neo_selftest_bounded_wait.argtypes = [_vp]
    lib.neo_version.argtypes = []
    for name in ("neo_build_positions", "neo_qknorm_rope3", "neo_gen_attention", "neo_flow_euler_step",
                 "neo_flow_cfg_euler_step", "neo_time_schedule", "neo_noise_scale", "neo_scale_noise",
           "neo_rope2d_interleaved", "neo_get_device_error", "neo_set_wait_timeout_ns", "neo_version"):
        getattr(lib, name).restype = c_int
    _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load_library().neo_status_string(int(status)).decode()
    except FileNotFoundError:
        return f"status {status}"


def _check(status: int, what: str):
    if status != NEO_OK:
        raise NeoError(status, what)


def _stream(stream, t=None):
    if stream is None:
        dev = t.device if (t is not None and t.is_cuda) else None
        return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t, dtype=None, what="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{what} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


_DT = {torch.bfloat16: NEO_BF16, torch.float32: NEO_F32}


def neo_build_positions(indexes: torch.Tensor, segments, stream=None):
    """Fill ``indexes`` (int32 [3, S]) from a list of segments
    ("text", start, count) / ("image", t_index, rows, cols)."""
    segs = (neo_pos_segment * max(1, len(segments)))()
    for i, s in enumerate(segments):
        if s[0] == "text":
            segs[i] = neo_pos_segment(NEO_SEG_TEXT, int(s[1]), int(s[2]), 0)
        elif s[0] == "image":
            segs[i] = neo_pos_segment(NEO_SEG_IMAGE, int(s[1]), int(s[2]), int(s[3]))
        else:
            raise ValueError(f"unknown segment {s!r}")
    S = indexes.shape[1]
    _check(load_library().neo_build_positions(_ptr(indexes, torch.int32, "indexes"), S, segs, len(segments),
                                              _stream(stream, indexes)), "neo_build_positions")


def neo_qknorm_rope3(q, k, indexes, q_norm_w, q_norm_hw_w, k_norm_w, k_norm_hw_w,
                     theta_t=5e6, theta_hw=1e4, eps=1e-6, stream=None):
    """In place: q [S, Hq, 128] and k [S, Hkv, 128] (bf16 or fp32; either may be None)."""
    ref = q if q is not None else k
    dt = _DT.get(ref.dtype)
    if dt is None:
        raise ValueError("q/k must be bf16 or fp32")
    S = ref.shape[0]
    Hq = q.shape[1] if q is not None else 0
    Hkv = k.shape[1] if k is not None else 0
    D = ref.shape[2]
    for t, n in ((q, "q"), (k, "k")):
        if t is not None and (t.dim() != 3 or t.shape[0] != S or t.dtype != ref.dtype):
            raise ValueError(f"{n} must be [S, H, 128] of one dtype")
    _check(load_library().neo_qknorm_rope3(
        _ptr(q, what="q"), _ptr(k, what="k"), dt, S, Hq, Hkv, D, _ptr(indexes, torch.int32, "indexes"),
        _ptr(q_norm_w, torch.float32, "q_norm_w") if q is not None else None,
        _ptr(q_norm_hw_w, torch.float32, "q_norm_hw_w") if q is not None else None,
        _ptr(k_norm_w, torch.float32, "k_norm_w") if k is not None else None,
        _ptr(k_norm_hw_w, torch.float32, "k_norm_hw_w") if k is not None else None,
        float(theta_t), float(theta_hw), float(eps), _stream(stream, ref)), "neo_qknorm_rope3")


def neo_gen_attention(q_img, k_prefix, v_prefix, k_img, v_img, cu_prefix, max_prefix, out,
                      scale=128 ** -0.5, mask_mode=NEO_MASK_FULL, t_prefix=None, t_img=None, lse=None,
                      stream=None):
    """out [B, N, Hq, 128] bf16 <- attention of q_img over [prefix ; image] keys."""
    B, N, Hq, D = q_img.shape
    Hkv = k_img.shape[2]
    total_prefix = k_prefix.shape[0] if k_prefix is not None else 0
    dt = _DT.get(q_img.dtype)
    if dt is None:
        raise ValueError("q_img must be bf16")
    _check(load_library().neo_gen_attention(
        _ptr(q_img, what="q_img"), _ptr(k_prefix if total_prefix else None, what="k_prefix"),
        _ptr(v_prefix if total_prefix else None, what="v_prefix"), _ptr(k_img, what="k_img"),
        _ptr(v_img, what="v_img"), dt, _ptr(cu_prefix, torch.int32, "cu_prefix"), int(total_prefix),
        int(max_prefix), B, N, Hq, Hkv, D, int(mask_mode), _ptr(t_prefix, torch.int32, "t_prefix"),
        _ptr(t_img, torch.int32, "t_img"), float(scale), _ptr(out, what="out"),
        _ptr(lse, torch.float32, "lse"), _stream(stream, q_img)), "neo_gen_attention")


def neo_gen_attention_qnorm(q_img_raw, k_prefix, v_prefix, k_img, v_img, cu_prefix, max_prefix, out, indexes,
                            q_norm_w, q_norm_hw_w, theta_t=5e6, theta_hw=1e4, eps=1e-6, scale=128 ** -0.5,
                            mask_mode=NEO_MASK_FULL, t_prefix=None, t_img=None, lse=None, stream=None):
    """neo_gen_attention with the query norm + RoPE folded in: q_img_raw
    [B, N, Hq, 128] bf16 before the norm (left unchanged), indexes int32
    [3, B*N] positions of the image tokens, q norm weights fp32 [64] each."""
    B, N, Hq, D = q_img_raw.shape
    Hkv = k_img.shape[2]
    total_prefix = k_prefix.shape[0] if k_prefix is not None else 0
    dt = _DT.get(q_img_raw.dtype)
    if dt is None:
        raise ValueError("q_img_raw must be bf16")
    qn = neo_qnorm_params(_ptr(indexes, torch.int32, "indexes"), _ptr(q_norm_w, torch.float32, "q_norm_w"),
                          _ptr(q_norm_hw_w, torch.float32, "q_norm_hw_w"), float(theta_t), float(theta_hw),
                          float(eps))
    _check(load_library().neo_gen_attention_qnorm(
        _ptr(q_img_raw, what="q_img_raw"), _ptr(k_prefix if total_prefix else None, what="k_prefix"),
        _ptr(v_prefix if total_prefix else None, what="v_prefix"), _ptr(k_img, what="k_img"),
        _ptr(v_img, what="v_img"), dt, _ptr(cu_prefix, torch.int32, "cu_prefix"), int(total_prefix),
        int(max_prefix), B, N, Hq, Hkv, D, int(mask_mode), _ptr(t_prefix, torch.int32, "t_prefix"),
        _ptr(t_img, torch.int32, "t_img"), ctypes.byref(qn), float(scale), _ptr(out, what="out"),
        _ptr(lse, torch.float32, "lse"), _stream(stream, q_img_raw)), "neo_gen_attention_qnorm")


def neo_write_prefix_cache(k_old, v_old, cu_old, k_new, v_new, k_out, v_out, cu_out, n_new=None, stream=None):
    """Append each sequence's first n_new[b] rows of k_new/v_new [B, N, Hkv, 128]
    after its rows of the packed cache k_old/v_old [total_old, Hkv, 128]
    (cu_old int32 [B+1]) into k_out/v_out [capacity, Hkv, 128]; cu_out int32
    [B+1] receives the new offsets."""
    B, N, Hkv, D = k_new.shape
    total_old = k_old.shape[0] if k_old is not None else 0
    dt = _DT.get(k_new.dtype)
    if dt is None:
        raise ValueError("k_new must be bf16 or fp32")
    _check(load_library().neo_write_prefix_cache(
        _ptr(k_old if total_old else None, what="k_old"), _ptr(v_old if total_old else None, what="v_old"),
        _ptr(cu_old, torch.int32, "cu_old"), int(total_old), _ptr(k_new if N else None, what="k_new"),
        _ptr(v_new if N else None, what="v_new"), _ptr(n_new, torch.int32, "n_new"), B, N, Hkv, D, dt,
        _ptr(k_out, what="k_out"), _ptr(v_out, what="v_out"), _ptr(cu_out, torch.int32, "cu_out"),
        int(k_out.shape[0]), _stream(stream, k_new)), "neo_write_prefix_cache")


def neo_flow_euler_step(z, x0_hat, t, t_next, t_eps=0.02, v_out=None, stream=None):
    """In place: z <- z + (t_next - t) * (x0_hat - z) / max(1 - t, t_eps) (fp32)."""
    n = z.numel()
    if x0_hat.numel() != n or (v_out is not None and v_out.numel() != n):
        raise ValueError("z, x0_hat and v_out must have the same number of elements")
    _check(load_library().neo_flow_euler_step(
        _ptr(z, torch.float32, "z"), _ptr(x0_hat, torch.float32, "x0_hat"), n, float(t), float(t_next),
        float(t_eps), _ptr(v_out, torch.float32, "v_out"), _stream(stream, z)), "neo_flow_euler_step")


def neo_flow_cfg_euler_step(z, x0_cond, x0_text_uncond, x0_uncond, t, t_next, cfg_scale, img_cfg_scale,
                            cfg_interval=(0.0, 1.0), t_eps=0.02, v_out=None, stream=None) -> int:
    """In place: classifier-free-guided Euler step; returns the branch taken."""
    n = z.numel()
    for x in (x0_cond, x0_text_uncond, x0_uncond, v_out):
        if x is not None and x.numel() != n:
            raise ValueError("all buffers must have the same number of elements")
    branch = ctypes.c_int32(-1)
    _check(load_library().neo_flow_cfg_euler_step(
        _ptr(z, torch.float32, "z"), _ptr(x0_cond, torch.float32, "x0_cond"),
        _ptr(x0_text_uncond, torch.float32, "x0_text_uncond"), _ptr(x0_uncond, torch.float32, "x0_uncond"), n,
        float(t), float(t_next), float(t_eps), float(cfg_scale), float(img_cfg_scale), float(cfg_interval[0]),
        float(cfg_interval[1]), _ptr(v_out, torch.float32, "v_out"), ctypes.byref(branch), _stream(stream, z)),
        "neo_flow_cfg_euler_step")
    return branch.value


def neo_time_schedule(n_steps: int, shift: float) -> list:
    """Host: the shifted time grid, n_steps + 1 floats from 0 to 1."""
    out = (ctypes.c_float * (n_steps + 1))()
    _check(load_library().neo_time_schedule(ctypes.cast(out, ctypes.c_void_p), int(n_steps), float(shift)),
           "neo_time_schedule")
    return list(out)


def neo_noise_scale(grid_h, grid_w, merge=2, base_seq_len=64.0, base_scale=1.0, mode=NEO_NOISE_RESOLUTION,
                    max_value=16.0) -> float:
    """Host: the resolution-dependent noise scale sigma_R."""
    out = ctypes.c_float(0.0)
    _check(load_library().neo_noise_scale(int(grid_h), int(grid_w), int(merge), float(base_seq_len),
                                          float(base_scale), int(mode), float(max_value), ctypes.byref(out)),
           "neo_noise_scale")
    return out.value


def neo_scale_noise(z, eps, sigma, stream=None):
    """z <- sigma * eps (fp32, same number of elements; z may be eps)."""
    if z.numel() != eps.numel():
        raise ValueError("z and eps must have the same number of elements")
    _check(load_library().neo_scale_noise(_ptr(z, torch.float32, "z"), _ptr(eps, torch.float32, "eps"), z.numel(),
                                          float(sigma), _stream(stream, z)), "neo_scale_noise")


def neo_rope2d_interleaved(x, rows, cols, theta=1e4, stream=None):
    """In place: x [n_images, rows * cols, C] (bf16 or fp32)."""
    dt = _DT.get(x.dtype)
    if dt is None or x.dim() != 3 or x.shape[1] != rows * cols:
        raise ValueError("x must be [n_images, rows*cols, C] bf16 or fp32")
    _check(load_library().neo_rope2d_interleaved(_ptr(x, what="x"), dt, x.shape[0], int(rows), int(cols),
                                                 x.shape[2], float(theta), _stream(stream, x)),
           "neo_rope2d_interleaved")


def neo_get_device_error(stream=None) -> tuple[int, int]:
    """(status, word): synchronises the stream, reads and clears the device error word."""
    word = ctypes.c_uint32(0)
    st = load_library().neo_get_device_error(_stream(stream), ctypes.byref(word))
    return st, word.value


def neo_set_wait_timeout_ns(ns: int):
    _check(load_library().neo_set_wait_timeout_ns(int(ns)), "neo_set_wait_timeout_ns")


def neo_selftest_bounded_wait(stream=None):
    """Enqueue the bounded-wait self-test (a wait that runs out; see neo.h)."""
    _check(load_library().neo_selftest_bounded_wait(_stream(stream)), "neo_selftest_bounded_wait")


def neo_version() -> int:
    return load_library().neo_version()

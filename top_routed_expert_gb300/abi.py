"""ctypes binding of the C ABI in include/moe_gb300.h (argument marshalling only).

Every function here has the name of the C entry point it calls and takes
torch tensors that already live on the current CUDA device; it passes their
data pointers and the current torch stream straight to the library and turns
a non-OK status into MoEError.  No arithmetic of the layer happens here, and
there is no fallback: if libmoe_gb300.so is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from .build import LIB

MOE_F32, MOE_BF16, MOE_E4M3, MOE_NVFP4 = 0, 1, 2, 3
MOE_FLAG_SIMT_FFN = 0x1
MOE_FLAG_SIMT_ROUTER = 0x2
MOE_FLAG_BF16_EXPERT_OUT = 0x4
MOE_FLAG_ACT_E4M3 = 0x8
MOE_FLAG_ACT_NVFP4 = 0x10
MOE_FLAG_NVFP4_F16 = 0x20
MOE_FLAG_NO_OVERLAP = 0x40
MOE_FLAG_INJECT_TIMEOUT = 0x100
MOE_NOALLOC_MAX_PAIRS = 65536

STATUS = {
    0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
    4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_TIMEOUT", 6: "MOE_ERR_DEVICE_BOUNDS", 7: "MOE_ERR_ARCH",
    8: "MOE_ERR_DEVICE_NONFINITE",
}

# Every symbol include/moe_gb300.h declares.
EXPORTS = ("moe_abi_version", "moe_status_str", "moe_workspace_bytes", "moe_route", "moe_permute",
           "moe_permute_noalloc", "moe_expert_ffn", "moe_combine", "moe_layer_forward", "moe_launch_count",
           "moe_get_device_status", "moe_qk_norm_rope")


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


class moe_config_t(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d_model", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("d_ff_shared", ctypes.c_int32),
                ("x_dtype", ctypes.c_int32), ("w_dtype", ctypes.c_int32), ("y_dtype", ctypes.c_int32),
                ("flags", ctypes.c_uint32)]


class moe_qk_rope_config_t(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("n_pos", ctypes.c_int32), ("eps", ctypes.c_float)]


class moe_weights_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "w13", "w13_scale", "w13_gscale", "w2", "w2_scale", "w2_gscale",
        "s13", "s13_scale", "s13_gscale", "s2", "s2_scale", "s2_gscale")]


_lib: Optional[ctypes.CDLL] = None


def load(path: str = LIB) -> ctypes.CDLL:
    """Load libmoe_gb300.so (built by top_routed_expert_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m top_routed_expert_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    cfgp = ctypes.POINTER(moe_config_t)
    wp = ctypes.POINTER(moe_weights_t)
    sig = {
        "moe_abi_version": (i32, []),
        "moe_status_str": (ctypes.c_char_p, [i32]),
        "moe_workspace_bytes": (sz, [cfgp]),
        "moe_route": (i32, [cfgp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "moe_permute": (i32, [cfgp, vp, vp, vp, vp, vp, sz, vp]),
        "moe_permute_noalloc": (i32, [cfgp, vp, vp, vp, vp, vp]),
        "moe_expert_ffn": (i32, [cfgp, vp, vp, vp, vp, wp, vp, vp, vp, sz, vp]),
        "moe_combine": (i32, [cfgp, vp, vp, vp, vp, vp]),
        "moe_layer_forward": (i32, [cfgp, vp, vp, vp, wp, vp, vp, vp, vp, vp, sz, vp]),
        "moe_launch_count": (ctypes.c_uint64, []),
        "moe_get_device_status": (i32, [vp]),
        "moe_qk_norm_rope": (i32, [ctypes.POINTER(moe_qk_rope_config_t), vp, vp, vp, vp, vp, vp, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(code: int, where: str):
    if code != 0:
        raise MoEError(code, where)


def make_config(T, d_model, n_experts, top_k, d_ff, d_ff_shared, x_dtype=MOE_BF16, w_dtype=MOE_E4M3,
                y_dtype=MOE_F32, flags=0) -> moe_config_t:
    return moe_config_t(T, d_model, n_experts, top_k, d_ff, d_ff_shared, x_dtype, w_dtype, y_dtype, flags)


def make_weights(w13, w13_scale, w13_gscale, w2, w2_scale, w2_gscale,
                 s13, s13_scale, s13_gscale, s2, s2_scale, s2_gscale) -> moe_weights_t:
    vals = [w13, w13_scale, w13_gscale, w2, w2_scale, w2_gscale, s13, s13_scale, s13_gscale, s2, s2_scale,
            s2_gscale]
    return moe_weights_t(*[None if v is None else v.data_ptr() for v in vals])


def moe_abi_version() -> int:
    return load().moe_abi_version()


def moe_status_str(code: int) -> str:
    return load().moe_status_str(code).decode()


def moe_workspace_bytes(cfg: moe_config_t) -> int:
    return load().moe_workspace_bytes(ctypes.byref(cfg))


def moe_route(cfg, x, w_router, expert_bias, topk_ids, topk_w, ws=None, stream=None):
    _check(load().moe_route(ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(expert_bias), _ptr(topk_ids),
                            _ptr(topk_w), _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                            _stream(stream)), "moe_route")


def moe_permute(cfg, topk_ids, expert_offsets, sorted_pair, row_of, ws, stream=None):
    _check(load().moe_permute(ctypes.byref(cfg), _ptr(topk_ids), _ptr(expert_offsets), _ptr(sorted_pair),
                              _ptr(row_of), _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                              _stream(stream)), "moe_permute")


def moe_permute_noalloc(cfg, topk_ids, expert_offsets, sorted_pair, row_of, stream=None):
    """moe_permute without a workspace: its scratch is a fixed array inside the
    library (at most MOE_NOALLOC_MAX_PAIRS = 65536 pairs; calls that overlap on
    the GPU race on it)."""
    _check(load().moe_permute_noalloc(ctypes.byref(cfg), _ptr(topk_ids), _ptr(expert_offsets),
                                      _ptr(sorted_pair), _ptr(row_of), _stream(stream)), "moe_permute_noalloc")


def moe_expert_ffn(cfg, x, topk_w, expert_offsets, sorted_pair, weights: moe_weights_t, out_perm, shared_out, ws,
                   stream=None):
    _check(load().moe_expert_ffn(ctypes.byref(cfg), _ptr(x), _ptr(topk_w), _ptr(expert_offsets),
                                 _ptr(sorted_pair), ctypes.byref(weights), _ptr(out_perm), _ptr(shared_out),
                                 _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                 _stream(stream)), "moe_expert_ffn")


def moe_combine(cfg, out_perm, row_of, shared_out, y, stream=None):
    _check(load().moe_combine(ctypes.byref(cfg), _ptr(out_perm), _ptr(row_of), _ptr(shared_out), _ptr(y),
                              _stream(stream)), "moe_combine")


def moe_layer_forward(cfg, x, w_router, expert_bias, weights: moe_weights_t, y, topk_ids=None, topk_w=None,
                      expert_offsets=None, ws=None, stream=None):
    _check(load().moe_layer_forward(ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(expert_bias),
                                    ctypes.byref(weights), _ptr(y), _ptr(topk_ids), _ptr(topk_w),
                                    _ptr(expert_offsets), _ptr(ws),
                                    0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
           "moe_layer_forward")


def moe_qk_norm_rope(cfg, q, k, gamma_q, gamma_k, cos_sin, positions, stream=None):
    """Fused QK-norm + RoPE, in place on q [T, Hq, D] and k [T, Hkv, D] (bf16)."""
    _check(load().moe_qk_norm_rope(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(gamma_q), _ptr(gamma_k),
                                   _ptr(cos_sin), _ptr(positions), _stream(stream)), "moe_qk_norm_rope")


def moe_launch_count() -> int:
    return load().moe_launch_count()


def moe_get_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    return load().moe_get_device_status(_stream(stream))

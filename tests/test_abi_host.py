"""Host-side checks of the C ABI: the library builds and loads without a GPU,
exports every symbol the header declares, and rejects bad arguments
synchronously, before anything would be launched."""
import ctypes
import os
import re

import pytest

import top_routed_expert_gb300 as moe
from top_routed_expert_gb300 import abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    moe.build()
    return abi.load()


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", fn)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"\b(moe_[a-z_]+)\s*\(", src)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert set(declared) == set(abi.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name
    assert abi.moe_abi_version() == 2


def test_status_strings(lib):
    for code, name in abi.STATUS.items():
        assert abi.moe_status_str(code) == name


def cfg(**kw):
    base = dict(T=64, d_model=4096, n_experts=128, top_k=6, d_ff=1024, d_ff_shared=1024,
                x_dtype=abi.MOE_BF16, w_dtype=abi.MOE_E4M3, y_dtype=abi.MOE_F32, flags=0)
    base.update(kw)
    return abi.moe_config_t(**base)


@pytest.mark.parametrize("bad", [
    dict(T=-1), dict(d_model=100), dict(d_model=0), dict(d_model=32768), dict(n_experts=0),
    dict(n_experts=300), dict(top_k=0), dict(top_k=17), dict(n_experts=4, top_k=5), dict(d_ff=100),
    dict(d_ff_shared=0), dict(x_dtype=abi.MOE_E4M3), dict(w_dtype=abi.MOE_BF16), dict(y_dtype=abi.MOE_NVFP4),
    dict(flags=0x80), dict(flags=0x10),
    # 8-bit activations only on the FP8 tensor-core path
    dict(flags=abi.MOE_FLAG_ACT_E4M3, w_dtype=abi.MOE_NVFP4), dict(flags=abi.MOE_FLAG_ACT_E4M3, w_dtype=abi.MOE_F32),
    dict(flags=abi.MOE_FLAG_ACT_E4M3, x_dtype=abi.MOE_F32), dict(flags=abi.MOE_FLAG_ACT_E4M3 | abi.MOE_FLAG_SIMT_FFN),
    dict(flags=abi.MOE_FLAG_ACT_E4M3, d_ff=192),
])
def test_invalid_config_rejected(lib, bad):
    c = cfg(**bad)
    assert lib.moe_workspace_bytes(ctypes.byref(c)) == 0
    assert lib.moe_route(ctypes.byref(c), None, None, None, None, None, None, 0, None) == 1
    assert lib.moe_layer_forward(ctypes.byref(c), None, None, None, None, None, None, None, None, None, 0,
                                 None) == 1


def test_null_config_rejected(lib):
    assert lib.moe_workspace_bytes(None) == 0
    assert lib.moe_route(None, None, None, None, None, None, None, 0, None) == 1
    assert lib.moe_combine(None, None, None, None, None, None) == 1


def test_null_pointers_rejected(lib):
    c = cfg()
    fake = ctypes.c_void_p(0x10000)   # aligned, never dereferenced: validation fails first
    assert lib.moe_route(ctypes.byref(c), None, fake, None, fake, fake, None, 0, None) == 1
    assert lib.moe_combine(ctypes.byref(c), fake, None, fake, fake, None) == 1
    assert lib.moe_expert_ffn(ctypes.byref(c), fake, fake, fake, fake, None, fake, fake, fake, 1 << 40,
                              None) == 1


def test_misaligned_pointers_rejected(lib):
    c = cfg()
    ok = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10002)
    assert lib.moe_route(ctypes.byref(c), odd, ok, None, ok, ok, None, 0, None) == 1
    assert lib.moe_combine(ctypes.byref(c), ok, ok, ok, odd, None) == 1


def test_workspace_too_small(lib):
    c = cfg()
    fake = ctypes.c_void_p(0x10000)
    assert lib.moe_permute(ctypes.byref(c), fake, fake, fake, fake, None, 0, None) == 3
    assert lib.moe_permute(ctypes.byref(c), fake, fake, fake, fake, fake, 16, None) == 3
    w = abi.moe_weights_t(*([0x10000] * 12))
    need = lib.moe_workspace_bytes(ctypes.byref(c))
    assert need > 0
    assert lib.moe_layer_forward(ctypes.byref(c), fake, fake, None, ctypes.byref(w), fake, None, None, None,
                                 fake, need - 256, None) == 3


def test_missing_weight_scales_rejected(lib):
    c = cfg()
    fake = ctypes.c_void_p(0x10000)
    w = abi.moe_weights_t(0x10000, None, None, 0x10000, 0x10000, None, 0x10000, 0x10000, None, 0x10000,
                          0x10000, None)
    assert lib.moe_layer_forward(ctypes.byref(c), fake, fake, None, ctypes.byref(w), fake, None, None, None,
                                 fake, 1 << 40, None) == 1
    c4 = cfg(w_dtype=abi.MOE_NVFP4)   # NVFP4 also needs the global scales
    w4 = abi.moe_weights_t(*([0x10000, 0x10000, None] * 4))
    assert lib.moe_layer_forward(ctypes.byref(c4), fake, fake, None, ctypes.byref(w4), fake, None, None, None,
                                 fake, 1 << 40, None) == 1


def test_zero_tokens_is_a_noop(lib):
    c = cfg(T=0)
    assert lib.moe_route(ctypes.byref(c), None, None, None, None, None, None, 0, None) == 0
    assert lib.moe_combine(ctypes.byref(c), None, None, None, None, None) == 0
    assert lib.moe_layer_forward(ctypes.byref(c), None, None, None, None, None, None, None, None, None, 0,
                                 None) == 0


def test_workspace_grows_with_tokens(lib):
    a = lib.moe_workspace_bytes(ctypes.byref(cfg(T=64)))
    b = lib.moe_workspace_bytes(ctypes.byref(cfg(T=8192)))
    assert 0 < a < b
    assert a % 256 == 0 and b % 256 == 0


def test_no_cuda_device_reports_error(lib):
    # With no GPU, a call that passes validation reaches the device query
    # and reports a CUDA or architecture error instead of crashing.
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    c = cfg()
    fake = ctypes.c_void_p(0x10000)
    assert lib.moe_route(ctypes.byref(c), fake, fake, None, fake, fake, None, 0, None) in (4, 7)


def test_act_e4m3_flag_is_accepted(lib):
    assert lib.moe_workspace_bytes(ctypes.byref(cfg(flags=abi.MOE_FLAG_ACT_E4M3))) > 0


def test_test_hook_flag_is_accepted(lib):
    assert lib.moe_workspace_bytes(ctypes.byref(cfg(flags=abi.MOE_FLAG_INJECT_TIMEOUT))) > 0
    assert lib.moe_workspace_bytes(ctypes.byref(cfg(flags=abi.MOE_FLAG_BF16_EXPERT_OUT))) < \
        lib.moe_workspace_bytes(ctypes.byref(cfg()))


def test_noalloc_permute_rejects_bad_sizes_on_the_host(lib):
    # more than 256 experts is an invalid configuration for every entry point;
    # more pairs than the fixed scratch holds is unsupported; both are
    # answered before any CUDA call
    fake = ctypes.c_void_p(0x10000)
    big_e = cfg(T=64, n_experts=257, top_k=6)
    assert lib.moe_permute_noalloc(ctypes.byref(big_e), fake, fake, fake, fake, None) == 1
    too_many = cfg(T=abi.MOE_NOALLOC_MAX_PAIRS // 6 + 1, top_k=6)
    assert lib.moe_permute_noalloc(ctypes.byref(too_many), fake, fake, fake, fake, None) == 2


def test_act_nvfp4_flag_validation(lib):
    nv = dict(w_dtype=abi.MOE_NVFP4, d_ff=2048, d_ff_shared=2048, top_k=8)
    assert lib.moe_workspace_bytes(ctypes.byref(cfg(flags=abi.MOE_FLAG_ACT_NVFP4, **nv))) > 0
    assert lib.moe_workspace_bytes(ctypes.byref(cfg(flags=abi.MOE_FLAG_NVFP4_F16, **nv))) > 0
    for bad in (dict(flags=abi.MOE_FLAG_ACT_NVFP4),                                   # FP8 weights
                dict(flags=abi.MOE_FLAG_ACT_NVFP4, **dict(nv, d_ff=128)),             # width not a multiple of 256
                dict(flags=abi.MOE_FLAG_ACT_NVFP4, **dict(nv, d_model=8192)),         # wider than 4096
                dict(flags=abi.MOE_FLAG_ACT_NVFP4 | abi.MOE_FLAG_NVFP4_F16, **nv),
                dict(flags=abi.MOE_FLAG_ACT_NVFP4 | abi.MOE_FLAG_SIMT_FFN, **nv),
                dict(flags=abi.MOE_FLAG_ACT_NVFP4, x_dtype=abi.MOE_F32, **nv)):
        assert lib.moe_workspace_bytes(ctypes.byref(cfg(**bad))) == 0, bad


def test_qk_norm_rope_rejects_bad_arguments(lib):
    fake = ctypes.c_void_p(0x10000)
    good = dict(T=4, n_q_heads=2, n_kv_heads=1, head_dim=128, n_pos=8, eps=1e-6)
    for bad in (dict(head_dim=96), dict(head_dim=0), dict(T=-1), dict(n_kv_heads=0), dict(n_pos=0),
                dict(eps=0.0), dict(eps=float("nan"))):
        c = abi.moe_qk_rope_config_t(**dict(good, **bad))
        assert lib.moe_qk_norm_rope(ctypes.byref(c), fake, fake, fake, fake, fake, fake, None) == 1, bad
    c = abi.moe_qk_rope_config_t(**good)
    odd = ctypes.c_void_p(0x10008)
    assert lib.moe_qk_norm_rope(ctypes.byref(c), odd, fake, fake, fake, fake, fake, None) == 1   # misaligned
    assert lib.moe_qk_norm_rope(ctypes.byref(c), None, fake, fake, fake, fake, fake, None) == 1
    assert lib.moe_qk_norm_rope(None, fake, fake, fake, fake, fake, fake, None) == 1
    c0 = abi.moe_qk_rope_config_t(**dict(good, T=0))
    assert lib.moe_qk_norm_rope(ctypes.byref(c0), None, None, None, None, None, None, None) == 0

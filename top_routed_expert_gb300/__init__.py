"""GB300-native (sm_103a) forward pass of a Sarvam-style MoE FFN layer.

The layer runs in hand-written CUDA kernels behind the C ABI of
include/moe_gb300.h (libmoe_gb300.so); `abi` is its thin ctypes binding and
`layer.MoELayer` keeps weights and workspace resident on the device.
"""
from . import abi  # noqa: F401
from .abi import (MoEError, moe_combine, moe_expert_ffn, moe_get_device_status,  # noqa: F401
                  moe_layer_forward, moe_permute, moe_route, moe_status_str, moe_workspace_bytes)
from .build import build  # noqa: F401

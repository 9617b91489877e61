"""Failure detection on the GPU without faulting it: a bounded wait is made to
run out on purpose (a completion signal that is never sent), the call reports
MOE_ERR_DEVICE_TIMEOUT through the device status word, and the same context
then runs the layer correctly."""
import numpy as np
import pytest
import torch

import moe_synth
from top_routed_expert_gb300 import abi
from top_routed_expert_gb300.layer import MoELayer

from .gpu_util import check_output, check_routing, device_x

pytestmark = pytest.mark.gpu


def test_bounded_wait_timeout_is_reported_and_context_survives():
    inp = moe_synth.make_custom(T=64, d=256, E=16, k=4, f=256, fs=128, x_dtype="bf16", w_dtype="e4m3", seed=3)
    layer = MoELayer(inp, flags=abi.MOE_FLAG_INJECT_TIMEOUT)
    x = device_x(inp)
    layer.forward(x)
    assert abi.moe_get_device_status() == 5          # MOE_ERR_DEVICE_TIMEOUT
    assert abi.moe_get_device_status() == 0          # read and cleared
    layer.flags = 0
    y, ids, w, offs = layer.forward(x, routing=True)
    assert abi.moe_get_device_status() == 0
    ids_np = ids.cpu().numpy()
    check_routing(inp, ids_np, w.cpu().numpy(), offs.cpu().numpy())
    check_output(inp, y.cpu().numpy(), ids_np)

"""Device-resident MoE layer: holds the weights and workspace on the GPU and
calls moe_layer_forward.  Plumbing only -- every step of the layer runs in
the CUDA library.
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import abi

_WDT = {"f32": abi.MOE_F32, "e4m3": abi.MOE_E4M3, "nvfp4": abi.MOE_NVFP4}
_XDT = {"f32": abi.MOE_F32, "bf16": abi.MOE_BF16}

_WEIGHT_NAMES = ("w13", "w13_scale", "w13_gscale", "w2", "w2_scale", "w2_gscale",
                 "s13", "s13_scale", "s13_gscale", "s2", "s2_scale", "s2_gscale")


def _to_dev(a, device) -> Optional[torch.Tensor]:
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        return a.to(device).contiguous()
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(device)


class MoELayer:
    """One MoE FFN layer resident on a CUDA device.

    `src` is any object with the attributes of the stored formats (x is not
    needed): cfg (with T, d, E, k, f, fs, x_dtype, w_dtype), w_router, bias,
    w13, w13_scale, w13_gscale, w2, ..., s2_gscale -- e.g. the synthetic
    workloads of moe_synth.  T may be overridden per call of forward().
    """

    def __init__(self, src, device="cuda", y_dtype=abi.MOE_F32, flags=0):
        c = src.cfg
        self.device = torch.device(device)
        self.T, self.d, self.E, self.k, self.f, self.fs = c.T, c.d, c.E, c.k, c.f, c.fs
        self.x_dtype, self.w_dtype = _XDT[c.x_dtype], _WDT[c.w_dtype]
        self.y_dtype, self.flags = y_dtype, flags
        self.w_router = _to_dev(src.w_router, self.device)
        self.bias = _to_dev(src.bias, self.device)
        self.tensors = {n: _to_dev(getattr(src, n), self.device) for n in _WEIGHT_NAMES}
        self.weights = abi.make_weights(*[self.tensors[n] for n in _WEIGHT_NAMES])
        self._ws = None

    def config(self, T=None) -> abi.moe_config_t:
        return abi.make_config(self.T if T is None else T, self.d, self.E, self.k, self.f, self.fs,
                               self.x_dtype, self.w_dtype, self.y_dtype, self.flags)

    def workspace(self, T=None) -> torch.Tensor:
        n = abi.moe_workspace_bytes(self.config(T))
        if n == 0:
            raise abi.MoEError(1, "moe_workspace_bytes")
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.empty(n, dtype=torch.uint8, device=self.device)
        return self._ws

    def empty_y(self, T) -> torch.Tensor:
        dt = torch.float32 if self.y_dtype == abi.MOE_F32 else torch.bfloat16
        return torch.empty((T, self.d), dtype=dt, device=self.device)

    def forward(self, x: torch.Tensor, y: Optional[torch.Tensor] = None, routing: bool = False, stream=None):
        """y = layer(x) for x [T, d] on the device (bf16 bits as int16/bfloat16, or fp32)."""
        T = x.shape[0]
        cfg = self.config(T)
        ws = self.workspace(T)
        if y is None:
            y = self.empty_y(T)
        ids = w = offs = None
        if routing:
            ids = torch.empty((T, self.k), dtype=torch.int32, device=self.device)
            w = torch.empty((T, self.k), dtype=torch.float32, device=self.device)
            offs = torch.empty((self.E + 1,), dtype=torch.int32, device=self.device)
        abi.moe_layer_forward(cfg, x, self.w_router, self.bias, self.weights, y, ids, w, offs, ws, stream)
        if routing:
            return y, ids, w, offs
        return y

    def capture(self, x: torch.Tensor, y: Optional[torch.Tensor] = None, warmup: int = 2):
        """Record one layer pass over the device buffers x -> y as a CUDA graph.

        Returns (graph, y); graph.replay() re-runs the whole layer (all its
        kernels) on whatever x holds at replay time.  Kernel attributes and the
        workspace are set up by the warm-up passes, so nothing is created while
        capturing.
        """
        T = x.shape[0]
        if y is None:
            y = self.empty_y(T)
        self.workspace(T)
        side = torch.cuda.Stream(self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            for _ in range(warmup):
                self.forward(x, y, stream=side)
        torch.cuda.current_stream(self.device).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            self.forward(x, y, stream=side)
        return graph, y

    def forward_host(self, x_host: torch.Tensor, y_host: torch.Tensor, x_dev: torch.Tensor,
                     y_dev: torch.Tensor, stream=None):
        """End to end from host buffers: H2D copy of x, the layer, D2H copy of y.

        x_host / y_host should be pinned; x_dev / y_dev are reusable device
        staging buffers of the same shapes.  Asynchronous on the stream.
        """
        s = stream or torch.cuda.current_stream()
        with torch.cuda.stream(s):
            x_dev.copy_(x_host, non_blocking=True)
            self.forward(x_dev, y_dev, stream=s)
            y_host.copy_(y_dev, non_blocking=True)
        return y_host

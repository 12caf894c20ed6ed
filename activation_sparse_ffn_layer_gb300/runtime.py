"""Decode-step runner over the C ABI: layers resident in HBM, one workspace,
one stream, optionally replayed as a CUDA graph.

A decode step for a stack of L layers is, per layer l:
``y_l = pi_ffn_layer(x_l)`` and ``x_{l+1} = pi_rmsnorm_half(y_l)`` (the
normalisation between layers of the stacked workloads).  Only launches go
through here; all arithmetic is in ``libpi.so``.
"""
from __future__ import annotations

from typing import List, Optional

import torch

from . import binding as B


class DeviceLayer:
    """One layer's tensors on the GPU plus the C descriptors over them."""

    def __init__(self, w, batch: int = 1):
        self.w = w
        self.batch = batch
        self.desc = B.layer_desc(w, batch)
        self.ws = B.weights_struct(w)

    def with_batch(self, batch: int) -> "DeviceLayer":
        return DeviceLayer(self.w, batch)


class DecodeStack:
    """Runs decode steps of `batch` tokens through a list of layers."""

    def __init__(self, layers: List, batch: int = 1, tau: float = -0.05, eps: float = 1e-6,
                 device: Optional[torch.device] = None):
        if not layers:
            raise ValueError("no layers")
        self.layers = [l if isinstance(l, DeviceLayer) and l.batch == batch else
                       DeviceLayer(l.w if isinstance(l, DeviceLayer) else l, batch) for l in layers]
        self.batch, self.tau, self.eps = batch, float(tau), float(eps)
        w0 = self.layers[0].w
        self.d = w0.d
        dev = device or w0.b1.device
        ws = max(B.pi_workspace_bytes(l.desc) for l in self.layers)
        if ws == 0:
            raise ValueError("layer descriptor rejected by the library")
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
        self.x_in = torch.empty(batch, self.d, dtype=torch.float16, device=dev)
        self.x_bufs = [torch.empty(batch, self.d, dtype=torch.float16, device=dev) for _ in range(2)]
        self.y = torch.empty(batch, self.d, dtype=torch.float32, device=dev)
        self.graph: Optional[torch.cuda.CUDAGraph] = None
        self.launches_per_step = None

    def _run(self, x: torch.Tensor, y: torch.Tensor, xs_out: Optional[list] = None):
        cur = x
        for l, layer in enumerate(self.layers):
            B.pi_ffn_layer(layer.desc, cur, layer.ws, self.tau, self.workspace, y)
            if l + 1 < len(self.layers):
                nxt = self.x_bufs[l % 2]
                B.pi_rmsnorm_half(self.d, self.batch, y, self.eps, nxt)
                if xs_out is not None:
                    xs_out.append(nxt.clone())
                cur = nxt

    def step(self, x: torch.Tensor) -> torch.Tensor:
        """One decode step, eager launches; returns the last layer's y."""
        self._run(x, self.y)
        return self.y

    def step_trace(self, x: torch.Tensor):
        """Eager step that also returns every layer's input (for parity checks)."""
        xs = [x.clone()]
        ys = []
        cur = x
        for l, layer in enumerate(self.layers):
            y = torch.empty_like(self.y)
            B.pi_ffn_layer(layer.desc, cur, layer.ws, self.tau, self.workspace, y)
            ys.append(y)
            if l + 1 < len(self.layers):
                nxt = torch.empty_like(self.x_in)
                B.pi_rmsnorm_half(self.d, self.batch, y, self.eps, nxt)
                xs.append(nxt)
                cur = nxt
        return xs, ys

    def capture(self) -> None:
        """Record one step (reading self.x_in, writing self.y) as a CUDA graph."""
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self._run(self.x_in, self.y)          # warm-up outside the graph
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self._run(self.x_in, self.y)
        self.graph = g

    def replay(self) -> None:
        self.graph.replay()

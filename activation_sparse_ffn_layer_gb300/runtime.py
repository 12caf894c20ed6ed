"""Decode-step runner over the C ABI: layers resident in HBM, one zero-filled
workspace, one stream, optionally replayed as a CUDA graph.

A decode step through a stack of L layers is one ``pi_ffn_stack`` call (layer
l: predictor -> compaction -> FC1 -> FC2, then the normalisation that feeds
layer l+1).  Only launches go through here; all arithmetic is in ``libpi.so``.
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


class DecodeStack:
    """Runs decode steps of `batch` tokens through a list of layers."""

    def __init__(self, layers: List, batch: int = 1, tau: float = -0.05, eps: float = 1e-6):
        if not layers:
            raise ValueError("no layers")
        ws = [l.w if isinstance(l, DeviceLayer) else l for l in layers]
        self.layers = [DeviceLayer(w, batch) for w in ws]
        self.weights = ws
        self.batch, self.tau, self.eps = batch, float(tau), float(eps)
        w0 = ws[0]
        self.d = w0.d
        dev = w0.b1.device
        rmax = max(w.r for w in ws)
        self.desc = B.desc_of(w0.d, w0.F, rmax, batch, w0.int4, w0.gated)
        self.warr = B.weights_array(ws)
        self.ranks = B.ranks_array(ws)
        nbytes = B.pi_workspace_bytes(self.desc)
        if nbytes == 0:
            raise ValueError("layer descriptor rejected by the library")
        self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        self.x_in = torch.zeros(batch, self.d, dtype=torch.float16, device=dev)
        self.y = torch.zeros(batch, self.d, dtype=torch.float32, device=dev)
        self.graph: Optional[torch.cuda.CUDAGraph] = None

    def _run(self, x: torch.Tensor, y: torch.Tensor, x_trace: Optional[torch.Tensor] = None,
             layer_counts: Optional[torch.Tensor] = None):
        B.pi_ffn_stack(self.desc, self.warr, self.ranks, x, self.tau, self.eps, self.workspace, y, x_trace,
                       layer_counts)

    def step_counts(self, x: torch.Tensor) -> torch.Tensor:
        """One step that also returns, per layer, [predicted-active neurons,
        neurons with a non-zero FC1 output] (int32 [L, 2], on the device)."""
        cnt = torch.zeros(len(self.layers), 2, dtype=torch.int32, device=x.device)
        self._run(x, self.y, None, cnt)
        return cnt

    def step(self, x: torch.Tensor) -> torch.Tensor:
        """One decode step (eager launch); returns the last layer's y."""
        self._run(x, self.y)
        return self.y

    def step_trace(self, x: torch.Tensor):
        """One step that also returns every layer's input (for parity checks):
        (list of [B, d] fp16 inputs, last layer's y)."""
        L = len(self.layers)
        tr = torch.zeros(max(L - 1, 1), self.batch, self.d, dtype=torch.float16, device=x.device)
        y = torch.zeros_like(self.y)
        self._run(x, y, tr if L > 1 else None)
        return [x.clone()] + [tr[l] for l in range(L - 1)], y

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

    def launches_per_step(self) -> int:
        """Kernel launches of one step, as the library reports them."""
        per = [B.pi_launches_per_layer(l.desc) for l in self.layers]
        if all(n == 1 for n in per):
            return 1                                  # one persistent kernel for the whole stack
        return sum(per) + (len(self.layers) - 1)      # per-step kernels + normalisations

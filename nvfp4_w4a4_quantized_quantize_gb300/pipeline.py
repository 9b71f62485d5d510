"""Host-to-host streaming of MoE expert-layer forwards.

A serving loop holds a batch's tokens, routing ids and routing weights in host memory and wants
the layer output back in host memory.  `HostPipeline` runs a sequence of such batches with the
copies of neighbouring batches overlapping the current batch's kernels: two device buffer sets,
one stream for host-to-device copies, one for the layer (a CUDA graph per buffer set), one for
device-to-host copies, ordered by events.  Every batch's inputs are copied up and every output
is copied back; only their overlap with the kernels of the batch in between is gained.
"""
from __future__ import annotations

import torch

from .layers import MoERacLayer


class HostPipeline:
    def __init__(self, layer: MoERacLayer, tokens: int, use_graph: bool = True):
        dev = layer.grp_off.device
        H, topk = layer.H, layer.topk
        self.layer = layer
        self.T = tokens
        self.sets = [dict(x=torch.empty(tokens, H, dtype=torch.bfloat16, device=dev),
                          ids=torch.zeros(tokens, topk, dtype=torch.int32, device=dev),
                          tw=torch.zeros(tokens, topk, dtype=torch.float32, device=dev),
                          out=torch.empty(tokens, H, dtype=torch.bfloat16, device=dev)) for _ in range(2)]
        self.s_in = torch.cuda.Stream(device=dev)
        self.s_comp = torch.cuda.Stream(device=dev)
        self.s_out = torch.cuda.Stream(device=dev)
        self.in_ready = [torch.cuda.Event() for _ in range(2)]
        self.comp_done = [torch.cuda.Event() for _ in range(2)]
        self.out_done = [torch.cuda.Event() for _ in range(2)]
        self.graphs = [None, None]
        if use_graph:
            for b, S in enumerate(self.sets):
                with torch.cuda.stream(self.s_comp):
                    layer.forward(S["x"], S["ids"], S["tw"], S["out"])  # warm on the capture stream
                self.s_comp.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=self.s_comp):
                    layer.forward(S["x"], S["ids"], S["tw"], S["out"])
                self.graphs[b] = g

    def _forward(self, b: int):
        if self.graphs[b] is not None:
            self.graphs[b].replay()
        else:
            S = self.sets[b]
            self.layer.forward(S["x"], S["ids"], S["tw"], S["out"])

    def run(self, x_h: torch.Tensor, ids_h: torch.Tensor, tw_h: torch.Tensor, out_h: torch.Tensor,
            steps: int) -> float:
        """`steps` batches from pinned host tensors (the same ones every step); returns the
        milliseconds from the first host-to-device copy to the end of the last device-to-host
        copy, measured with CUDA events."""
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(self.s_in)
        for i in range(steps):
            b = i % 2
            S = self.sets[b]
            if i >= 2:
                self.s_in.wait_event(self.comp_done[b])   # the forward of step i-2 has read set b
            with torch.cuda.stream(self.s_in):
                S["x"].copy_(x_h, non_blocking=True)
                S["ids"].copy_(ids_h, non_blocking=True)
                S["tw"].copy_(tw_h, non_blocking=True)
            self.in_ready[b].record(self.s_in)
            self.s_comp.wait_event(self.in_ready[b])
            if i >= 2:
                self.s_comp.wait_event(self.out_done[b])  # the output of step i-2 is on the host
            with torch.cuda.stream(self.s_comp):
                self._forward(b)
            self.comp_done[b].record(self.s_comp)
            self.s_out.wait_event(self.comp_done[b])
            with torch.cuda.stream(self.s_out):
                out_h.copy_(S["out"], non_blocking=True)
            self.out_done[b].record(self.s_out)
        end.record(self.s_out)
        end.synchronize()
        return start.elapsed_time(end)

    def last_output(self, steps: int) -> torch.Tensor:
        return self.sets[(steps - 1) % 2]["out"]

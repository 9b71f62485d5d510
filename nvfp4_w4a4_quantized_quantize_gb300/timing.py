"""Device timing of a launch sequence: CUDA-graph replays with CUDA events on the replaying
stream, the L2 cache flushed (a write larger than L2) before every replay, outside the events."""
from __future__ import annotations

import statistics

import torch


def time_graph_replays(fn, flush: torch.Tensor, steps: int, warmup: int) -> float:
    """Median milliseconds of one replay of a graph captured around fn()."""
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            fn()
    torch.cuda.current_stream().wait_stream(cap)
    times = []
    for i in range(warmup + steps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        b.synchronize()
        if i >= warmup:
            times.append(a.elapsed_time(b))
    return statistics.median(times)

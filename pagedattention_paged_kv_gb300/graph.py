"""A step of fixed shapes captured once as a CUDA graph and replayed.

A serving loop that runs the same batch shape every iteration (for example 128 decode
rows) spends more host time enqueueing the KV write and the attention launches than the
GPU spends on small steps.  CapturedStep records one call of `fn` -- which must take
its inputs from static device or pinned host buffers and make only stream-ordered
calls (copies, this package's kernels) -- and replays the whole launch sequence with
one call.  The kernels' programmatic-dependent-launch edges are kept in the graph.
"""
from __future__ import annotations


class CapturedStep:
    def __init__(self, fn, warmup: int = 2, stream=None):
        """`stream`: the (non-default) stream to capture and replay on; a new one if None."""
        import torch
        self.torch = torch
        self.stream = stream if stream is not None else torch.cuda.Stream()
        self.stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(self.stream):
            for _ in range(warmup):  # first calls set up per-device state outside capture
                fn()
        torch.cuda.current_stream().wait_stream(self.stream)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream, capture_error_mode="thread_local"):
            fn()

    def replay(self) -> None:
        """Enqueues the captured step on the capture stream (torch replays a graph on the
        current stream, so the capture stream is made current around it)."""
        with self.torch.cuda.stream(self.stream):
            self.graph.replay()

    def synchronize(self) -> None:
        self.stream.synchronize()

"""CUDA-graph shape buckets for fixed sequences of h3fp4 calls.

A transformer block runs the same projections with the same shapes step after
step ("H3 Runtime Current State", "Owned Performance Kernels": CUDA graph capture
and shape buckets).  ``GraphBuckets`` records the calls a caller issues for one
bucket key (for example the token count) into a CUDA graph and replays it on
later uses, so that the host issues one graph launch instead of every kernel
launch and memset of the sequence.

The h3fp4 calls are asynchronous, allocate nothing and never synchronise, so
they can be captured as they are.  Their one-time per-device setup (kernel
attributes, occupancy queries) happens in the eager warm-up run that precedes
each capture.  Buffers touched by a captured sequence must stay allocated and
at the same addresses while its graph is in use; new inputs are written into
them before a replay.  Nothing here computes: the graphs replay the library's
kernels.
"""
from typing import Callable, Dict, Hashable

import torch


class GraphBuckets:
    """One CUDA graph per bucket key of the call sequence ``issue(key)``."""

    def __init__(self, issue: Callable[[Hashable], None], warmup: int = 1):
        self._issue = issue
        self._warmup = warmup
        self._graphs: Dict[Hashable, torch.cuda.CUDAGraph] = {}

    def __len__(self) -> int:
        return len(self._graphs)

    def __contains__(self, key) -> bool:
        return key in self._graphs

    def capture(self, key: Hashable) -> torch.cuda.CUDAGraph:
        """Warm up eagerly on a side stream, then record ``issue(key)``."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(self._warmup):
                self._issue(key)
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self._issue(key)
        self._graphs[key] = g
        return g

    def run(self, key: Hashable) -> None:
        """Replay the graph of ``key`` on the current stream, capturing it first if new."""
        g = self._graphs.get(key)
        if g is None:
            g = self.capture(key)
        g.replay()

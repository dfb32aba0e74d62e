"""Rounds replayed from a CUDA graph.

A round's launches depend only on device data (the realignment reads the
n_emit that verification wrote; positions and mask read the new paddings),
so a serving loop whose buffers stay put -- the KV caches, positions, mask,
workspace, and input / output blocks -- can capture one round once and
replay it every step: one graph launch instead of a host call per kernel.
The library's programmatic launches become programmatic graph edges.

Typical use: two graphs, one per parity of double-buffered length / padding
blocks (a round reads one block and writes the other).
"""
from __future__ import annotations

import torch


class RoundGraph:
    """Capture `enqueue()` -- the library calls of one round plus any
    copies around them, all on the current stream -- into a CUDA graph."""

    def __init__(self, enqueue, device=None):
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
            with torch.cuda.graph(self.graph):
                enqueue()

    def replay(self):
        """Launch the captured round on the current stream."""
        self.graph.replay()

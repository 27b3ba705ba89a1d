"""One CUDA graph per draft-length tier of a verification step.

Each tier's step (verify attention, the linear layers at GEMM-M = B(1+D),
acceptance) is captured once on a side stream after a few warm-up runs;
a round then costs one graph launch, and switching tiers costs nothing
but launching another graph.  The step functions must use buffers that
stay put between rounds (graph replay reuses the captured addresses).
"""
from __future__ import annotations


class TierGraphs:
    def __init__(self, step_for_tier, tiers, warmup=2):
        """step_for_tier(D) enqueues one verification step of draft length D
        on the current stream."""
        import torch
        self.graphs = {}
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for D in tiers:
                for _ in range(warmup):
                    step_for_tier(D)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        for D in tiers:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                step_for_tier(D)
            self.graphs[D] = g
        torch.cuda.synchronize()

    def replay(self, D):
        self.graphs[D].replay()

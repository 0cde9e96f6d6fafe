"""The five synthetic decode workloads, named by what they are.

Each stands in for the GLM-5.2 MTP3 serving traces the FlashOffloading paper
measures on ("FlashOffloading ... What does it mean?", decode paragraphs and
Table 1), which are not available: keys and main rows are N(0,1) bf16, the
indexer query is a seeded random walk q <- a*q + sqrt(1-a^2)*N(0,I) per
(request, layer), and n_new tokens are appended each step.
"""
from dataclasses import dataclass, replace
from typing import Tuple


@dataclass(frozen=True)
class Workload:
    name: str
    n_requests: int
    n_layers: int
    context: int          # L0: tokens cached before step 0
    n_pos: int            # P: query positions per step (4 = MTP3)
    n_new: int            # tokens appended per step
    topk: int
    hot_capacity: int
    steps: int
    drift: float          # a in q <- a q + sqrt(1-a^2) eps
    seed: int
    idx_dim: int = 128
    row_elems: int = 576

    @property
    def n_units(self):
        return self.n_requests * self.n_layers

    def units_rl(self):
        """(request, layer) of unit u = request * n_layers + layer."""
        return [(r, l) for r in range(self.n_requests) for l in range(self.n_layers)]

    def max_tokens(self, steps=None):
        s = self.steps if steps is None else steps
        return self.context + s * self.n_new


WORKLOADS = {
    # 1 request x 1 layer, 4096 context, top-256 of a 512-slot shelf, no MTP
    "single_4k": Workload("single_4k", 1, 1, 4096, 1, 1, 256, 512, 20, 0.9, 1001),
    # 16 requests x 8 layers, 32768 context, MTP3, top-2048, 4096 slots
    "batch16x8_32k_mtp3": Workload("batch16x8_32k_mtp3", 16, 8, 32768, 4, 4, 2048, 4096, 50,
                                   0.9, 1002),
    # 32 requests x 16 layers, 65536 context, top-2048 of 16384 slots (1/4), drift 0.95
    "batch32x16_64k": Workload("batch32x16_64k", 32, 16, 65536, 1, 1, 2048, 16384, 50, 0.95,
                               1003),
    # 1 request x 8 layers, 1,048,576 context, MTP3, 131072 slots
    "long_1m_mtp3": Workload("long_1m_mtp3", 1, 8, 1048576, 4, 4, 2048, 131072, 20, 0.9, 1004),
    # 64 requests x 4 layers, 16384 context, MTP3, top-1024 of 2048 slots, drift swept
    "sweep64x4_16k_mtp3": Workload("sweep64x4_16k_mtp3", 64, 4, 16384, 4, 4, 1024, 2048, 30,
                                   0.9, 1005),
}

SWEEP_DRIFTS: Tuple[float, ...] = (0.0, 0.5, 0.9, 0.99, 1.0)


def reduced(w: Workload, n_requests=None, n_layers=None, context=None, topk=None,
            hot_capacity=None, steps=None, drift=None):
    """A smaller copy of a workload with the same structure (P, n_new, ratios)."""
    kw = {}
    for k, v in (("n_requests", n_requests), ("n_layers", n_layers), ("context", context),
                 ("topk", topk), ("hot_capacity", hot_capacity), ("steps", steps),
                 ("drift", drift)):
        if v is not None:
            kw[k] = v
    return replace(w, name=w.name + "_reduced", **kw)

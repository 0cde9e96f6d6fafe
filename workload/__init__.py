"""Seeded synthetic inputs for the sparse-decode KV offload workloads.

Holds no arithmetic of the offload method: it only produces bf16 numbers from
(seed, kind, request, layer, sub, index) so that the CPU oracle and the CUDA
path can be fed identical inputs.
"""
from .gen import (  # noqa: F401
    KIND_KEYS, KIND_ROWS, KIND_QINIT, KIND_QNOISE, KIND_ATTN_Q, build, lib, normal_bf16, normal_f64,
    token_rows, token_rows_into, query_walk, unit_queries, attention_queries, bf16_to_f32,
    f32_to_bf16_np,
)
from .configs import SWEEP_DRIFTS, WORKLOADS, Workload, reduced  # noqa: F401

"""Seeded synthetic inputs for the table-batched embedding workloads.

This package only draws inputs (table shapes, bag lengths, ids, weights, per-sample weights,
upstream gradients).  It holds none of the forward/backward arithmetic, and it serves both
the CPU oracle and the CUDA library, which share nothing else.
"""
from .configs import CONFIGS, TBEConfig, get_config  # noqa: F401
from .gen import (  # noqa: F401
    Batch,
    grad_out_rows,
    grad_out_tensor,
    make_batch,
    psw_values,
    weight_rows,
    weights_tensor,
)

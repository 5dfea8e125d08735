"""Inputs of the worked examples printed in "Table-Batched Embeddings in Triton: Gather,
Pool, and Run-Length Backward", regenerated from the chapter's description of how they are
drawn (torch's CPU generator is the only source of randomness).  The printed results they
produce are stored, with their citations, under tests/golden/.
"""
from __future__ import annotations

import numpy as np
import torch


def adagrad_trap_inputs():
    """Section 5, "The trap: one optimizer step per row, not per lookup": with the global
    generator seeded 0, a D=4 row w0 ~ randn(4) and then five gradients ~ randn(4) that five
    bags of one batch send to that same row; lr = 0.1, eps = 1e-8."""
    torch.manual_seed(0)
    D = 4
    w0 = torch.randn(D)
    grads = [torch.randn(D) for _ in range(5)]
    return (w0.numpy().astype(np.float32), torch.stack(grads).numpy().astype(np.float32),
            0.1, 1e-8)


def skewed_batch(seed: int = 1, T: int = 3, E: int = 50, B: int = 16, D: int = 24, max_L: int = 12):
    """Section 2 batch generator: one torch.Generator seeded `seed` draws, in order,
      1. the packed fp32 tables W ~ 0.1 * randn(T*E, D),
      2. a length per (table, bag), table-major, uniform in {0, ..., max_L},
      3. one uniform u per lookup, mapped to an exponentially skewed id
         min(E - 1, floor(-log1p(-u) / 0.15)).
    Section 3 runs it with T=3, E=50, B=16, D=24, max_L=12 and seed 1."""
    g = torch.Generator().manual_seed(seed)
    W = torch.randn(T * E, D, generator=g) * 0.1
    lengths = torch.randint(0, max_L + 1, (T * B,), generator=g)
    offsets = torch.zeros(T * B + 1, dtype=torch.int64)
    offsets[1:] = torch.cumsum(lengths, 0)
    u = torch.rand(int(offsets[-1]), generator=g)
    ids = torch.clamp(torch.floor(-torch.log1p(-u) / 0.15).to(torch.int64), max=E - 1)
    return dict(T=T, E=E, B=B, D=D, W=W.numpy().astype(np.float32),
                lengths=lengths.numpy().astype(np.int64), offsets=offsets.numpy(),
                indices=ids.numpy().astype(np.int64))


def skewed_batch_grad(B: int = 16, width: int = 72, seed: int = 2) -> np.ndarray:
    """Section 3 threshold sweep: upstream gradient randn(B, T*D) from a generator seeded 2."""
    g = torch.Generator().manual_seed(seed)
    return torch.randn(B, width, generator=g).numpy().astype(np.float32)

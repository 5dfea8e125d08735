"""GB300 (sm_103a) table-batched embedding: forward pooled gather and backward with one
optimizer update per touched row, as a C-ABI CUDA library (include/tbe.h) with a thin
ctypes binding.  Nothing here computes on the CPU; the library must be built
(``bwd_tbe_fwd_gb300.build.build()``) and a CUDA device must be present to run it."""
from .tbe import (  # noqa: F401
    BWD_STAGES,
    EXPORTED,
    FWD_STAGES,
    STAT_NAMES,
    TBE_NUM_STATS,
    TableBatchedEmbedding,
    TBEError,
    TBEOptions,
    load,
    tbe_backward_metadata,
    tbe_backward_update,
    tbe_bounds_check,
    tbe_forward,
)

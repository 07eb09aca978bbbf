"""ReLU activation-sparse feedforward layer for GB300 (sm_103a).

The computation runs in ``libtwell.so`` (CUDA kernels behind the C ABI of
``include/twell.h``); this package only marshals torch tensors into it.
"""
from ._lib import TwellError, lib_path, load  # noqa: F401
from .ops import (  # noqa: F401
    HybridFFN,
    HybridScratch,
    TwELL,
    Hybrid,
    TwellFFN,
    TwellSparseFFN,
    dense_gemm,
    fma_probe,
    gate_relu_dense,
    hybrid_neuron_counts,
    hybrid_pack,
    hybrid_unpack,
    l2_gather_probe,
    new_status,
    raise_if_device_error,
    reinit_dead_rows,
    twell_ffn_fwd,
    twell_gate_pack,
    twell_pack,
    twell_unpack,
)

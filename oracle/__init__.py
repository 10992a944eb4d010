"""CPU oracle of the mHC layer boundary: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s ``cpu_baseline``
leg / ``--impl reference`` arm may import this package. The CUDA product path
never imports it and shares no code with it; the product fails loudly when its
CUDA library is missing instead of falling back here.

The arithmetic lives in ``mhc_oracle.c`` (plain single-threaded C, compiled
with ``-ffp-contract=off``); this module only builds it and marshals numpy
arrays through ctypes. bf16 tensors travel as ``numpy.uint16`` bit patterns.
"""
from .oracle import (  # noqa: F401
    OracleParams,
    build_oracle,
    boundary,
    coefficients,
    f32_to_bf16,
    post,
    pre_split_k,
    sigmoid,
    sinkhorn,
    tf32_round,
    tf32_split,
    weight_tiles,
    MODE_PRE_ONLY,
    MODE_FUSED_UNSHIFTED,
    MODE_FUSED_SHIFTED,
)

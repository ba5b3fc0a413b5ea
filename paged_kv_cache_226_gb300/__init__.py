"""Paged decode attention for GB300 (sm_103a).

The compute path is ``libpa.so`` (CUDA kernels behind the C ABI in
``include/pa.h``); ``lib`` is its Python binding and ``inputs`` the host-side
block allocator and seeded workload builder.
"""
from . import inputs  # noqa: F401
from .lib import (  # noqa: F401
    DEFAULT_PARTITION, PaError, copy_blocks, decode, decode_split, decode_step,
    decode_step_balanced, load, prefill,
    num_partitions,
    paged_attention,
    StepPlan, InputStaging, read_device_errors, reduce, reshape_and_cache, split_workspace,
)

"""KDA (Kimi Delta Attention) chunked prefill forward for NVIDIA GB300.

The computation lives in hand-written sm_103a CUDA kernels behind a C ABI
(``include/kda.h``, built into ``libkda.so`` by ``build.py``). This package
holds the ctypes binding (``_lib``), the build script and the seeded input
generators (``inputs``).
"""
from ._lib import (KDA_DEBUG_SPLIT_COLUMNS, KDA_DEBUG_WHOLE_COLUMNS, KDA_DEBUG_WITHHOLD_READY, KDA_DEBUG_WY_CONSUMER,
                   KDA_DEBUG_WY_PRODUCER, KDA_ERR_BAD_SEQLENS, KDA_ERR_BOUNDS, KDA_ERR_CUDA, KDA_ERR_GATE_RANGE,
                   KDA_ERR_INVALID_ARG, KDA_ERR_SCRATCH_TOO_SMALL, KDA_ERR_TIMEOUT, KDA_ERR_UNSUPPORTED,
                   KDA_ERR_VALUE_RANGE, KDA_OK, KdaError, chunk_fwd, decode_fwd, kda_decode_fwd,
                   chunk_fwd_launches, chunk_fwd_plan, chunk_fwd_split, host_buffer_size, kda_chunk_fwd, kda_chunk_fwd_host,
                   kda_chunk_fwd_split, library_path,
                   load_library, split_plan, split_workspace_size, status_string, version, workspace_for,
                   workspace_size)

__all__ = [
    "KDA_OK", "KDA_ERR_INVALID_ARG", "KDA_ERR_UNSUPPORTED", "KDA_ERR_CUDA", "KDA_ERR_GATE_RANGE",
    "KDA_ERR_BAD_SEQLENS", "KDA_ERR_TIMEOUT", "KDA_ERR_VALUE_RANGE", "KDA_ERR_SCRATCH_TOO_SMALL", "KDA_ERR_BOUNDS",
    "KDA_DEBUG_WITHHOLD_READY", "KDA_DEBUG_WY_PRODUCER", "KDA_DEBUG_WY_CONSUMER", "KDA_DEBUG_SPLIT_COLUMNS",
    "KDA_DEBUG_WHOLE_COLUMNS", "KdaError", "decode_fwd", "kda_decode_fwd", "chunk_fwd", "chunk_fwd_launches", "chunk_fwd_plan",
    "kda_chunk_fwd", "library_path", "load_library", "status_string", "version", "workspace_for",
    "workspace_size", "chunk_fwd_split", "kda_chunk_fwd_split", "split_plan", "split_workspace_size",
    "kda_chunk_fwd_host", "host_buffer_size",
]

"""Paged relative-bias (Inkling-family) attention for GB300 (sm_103a).

The compute lives in the CUDA library ``lib/librelattn.so`` behind the C ABI
of ``include/relattn.h``; this package is its thin Python binding.
"""

from .relattn import (  # noqa: F401
    DEV_BAD_BLOCK_ID,
    DEV_BAD_LENGTH,
    DEV_WAIT_TIMEOUT,
    RelattnError,
    clear_status,
    new_workspace,
    read_status,
    relattn_decode,
    relattn_prefill,
    workspace_size,
)

"""Paged KV-cache decode + append attention for GB300 (sm_103a).

The product is the C-ABI library ``libpkv.so`` (``include/pkv.h``); this
package holds its CUDA sources (``csrc/``), the build step, the thin ctypes
binding (``api``) and the seeded synthetic workload generators
(``workloads``).
"""
from .api import (  # noqa: F401
    HND,
    DecodeStep,
    NHD,
    PagePool,
    PkvError,
    cache_desc,
    decode_workspace,
    default_decode_max_qlen,
    mixed_workspace,
    pkv_append,
    pkv_decode_bucket,
    pkv_decode_attn,
    pkv_decode_workspace_size,
    pkv_mixed_attn,
    pkv_mixed_workspace_size,
    pkv_pool_bytes,
    pkv_prefill_attn,
    pkv_prefill_workspace_size,
    prefill_workspace,
    pkv_validate_host,
)

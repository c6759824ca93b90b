"""Public Python entry points (same names as the C ABI, minus the prefix)."""
from ._lib import (BF16, DEV_BAD_BLOCK, DEV_BAD_LEN, DEV_BAD_SLOT, DEV_TIMEOUT, FP16,
                   PARTITION_STREAM, PATH_SIMT, PATH_TC, PATH_TC_CLUSTER, PATH_TC_STREAM, PkdError,
                   decode_plan, decode_workspace_bytes, gather_cached_kv, paged_decode_attention,
                   paged_prefill_attention, reshape_and_cache, version)

__all__ = ["BF16", "DEV_BAD_BLOCK", "DEV_BAD_LEN", "DEV_BAD_SLOT", "DEV_TIMEOUT", "FP16",
           "PARTITION_STREAM", "PATH_SIMT", "PATH_TC", "PATH_TC_CLUSTER", "PATH_TC_STREAM",
           "PkdError", "decode_plan", "decode_workspace_bytes", "gather_cached_kv",
           "paged_decode_attention", "paged_prefill_attention", "reshape_and_cache",
           "version"]

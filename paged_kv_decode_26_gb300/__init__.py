"""GB300-native paged-KV decode attention.

C ABI: include/pagedkv.h, implemented by libpagedkv.so (CUDA, sm_103a).
This package holds the CUDA sources (csrc/), the in-tree build, a thin torch
binding with the same entry-point names, and the seeded workload generator.
"""
from .api import (BlockManager, DecodeBatch, DeviceBlockManager, HostStep,
                  alloc_decode_workspace,
                  decode_launch_shape, decode_split_tokens,
                  decode_workspace_bytes, device_errors, get_tuning, kv_append, paged_attn_decode,
                  paged_attn_decode_append, paged_attn_decode_append_host,
                  paged_attn_multi_query,
                  reset_tuning, set_tuning, swap_blocks, swap_blocks_kv)
from ._lib import PagedKVError, lib

__all__ = ["paged_attn_decode", "paged_attn_decode_append", "paged_attn_decode_append_host",
           "paged_attn_multi_query", "kv_append", "swap_blocks", "swap_blocks_kv", "decode_workspace_bytes",
           "decode_split_tokens", "decode_launch_shape", "alloc_decode_workspace", "device_errors", "BlockManager", "DeviceBlockManager",
           "DecodeBatch", "HostStep", "PagedKVError", "lib", "set_tuning", "get_tuning", "reset_tuning"]

"""paged_kv_decode_slot_gb300 -- libpagedkv: decode-step attention over a paged KV cache on GB300.

The compute path is the C-ABI library ``libpagedkv.so`` (hand-written sm_103a CUDA, declared
in ``include/pkv.h``); ``binding`` exposes its entry points under the same names with torch
tensors as arguments (PyTorch supplies device memory and streams only).  ``inputs`` draws
seeded synthetic workloads.
"""
from .binding import (BLOCK_SIZE, PKV_ERR_ALIGN, PKV_ERR_CUDA, PKV_ERR_NULL, PKV_ERR_RANGE,  # noqa: F401
                      PKV_ERR_SHAPE, PKV_ERR_UNSUPPORTED, PKV_ERR_WORKSPACE, PKV_FLAG_BLOCK_RANGE,
                      PKV_FLAG_CTX_RANGE, PKV_FLAG_OUT_RANGE, PKV_FLAG_SLOT_RANGE, PKV_FLAG_TIMEOUT,
                      PKV_OK, CacheDesc, PkvError, cache_desc, check, library, max_partitions_for,
                      pkv_append, pkv_decode_attn, pkv_decode_attn_partitions,
                      pkv_decode_attn_splitk, pkv_gather, pkv_kv_bytes, pkv_last_error,
                      pkv_lse_merge, pkv_read_err_flag, pkv_slot_mapping,
                      pkv_splitk_workspace_bytes, pkv_status_string)

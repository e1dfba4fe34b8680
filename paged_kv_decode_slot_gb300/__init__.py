"""paged_kv_decode_slot_gb300 -- libpagedkv: decode-step attention over a paged KV cache on GB300.

The compute path is the C-ABI library ``libpagedkv.so`` (hand-written sm_103a CUDA, declared
in ``include/pkv.h``); ``binding`` exposes its entry points under the same names with torch
tensors as arguments (PyTorch supplies device memory and streams only).  ``inputs`` draws
seeded synthetic workloads; ``step`` runs a whole decode step.

The binding is loaded on first use of one of its names, so that ``build`` can be imported
before the library exists; using any entry point without the built library raises
ImportError (there is no fallback path).
"""


def __getattr__(name):
    if name.startswith(("pkv_", "PKV_")) or name in ("BLOCK_SIZE", "CacheDesc", "PkvError", "cache_desc",
                                                    "check", "library", "max_partitions_for", "tapered_partitions_for", "IN_KERNEL_MERGE_WEIGHTS",
                                                    "split_attention_launches", "multi_attention_launches"):
        from . import binding
        return getattr(binding, name)
    raise AttributeError(f"module {__name__!r} has no attribute {name!r}")

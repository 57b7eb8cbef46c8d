"""Paged-KV attention step for GB300 (sm_103a): Python binding of ``libpkv.so``.

The binding only marshals arguments (device pointers, sizes, strides, the
current CUDA stream) into the C ABI of ``include/pkv.h``; every step of the
computation runs in the library's CUDA kernels.  There is no CPU fallback: if
the library is missing or no sm_103 device is present, the calls raise.

    pkv_write(k, v, key_cache, value_cache, slot_mapping)
    pkv_attention(q, key_cache, value_cache, query_start_loc, seq_lens,
                  block_table, num_reqs, scale, out)
    pkv_write_int8 / pkv_attention_int8: the same over int8 caches with one
                  scale per cache (decode-path requests)
    pkv_plan / pkv_attention_planned: one step plan, then one call per layer

Tensors: bf16 q/k/v/out/caches (k, v, q, out may be row-strided views, e.g.
column slices of a fused qkv), int64 slot_mapping, int32 query_start_loc /
seq_lens / block_table.  Both calls enqueue on ``stream`` (default: torch's
current stream) and return immediately.
"""
from ._binding import (DEV_ERR_BITS, TRACE_KINDS, PkvError, library_path, load,
                       pkv_attention, pkv_attention_int8, pkv_attention_noalloc,
                       pkv_attention_planned, pkv_get_error, pkv_plan,
                       pkv_launch_count, pkv_num_sms, pkv_prepare_step,
                       pkv_reserve_workspace, pkv_trace_enable, pkv_trace_read,
                       pkv_workspace_size, pkv_write, pkv_write_int8)

__all__ = ["pkv_write", "pkv_attention", "pkv_attention_noalloc", "pkv_prepare_step",
           "pkv_write_int8", "pkv_attention_int8", "pkv_plan", "pkv_attention_planned",
           "pkv_get_error",
           "pkv_reserve_workspace", "pkv_workspace_size",
           "pkv_num_sms", "pkv_trace_enable", "pkv_trace_read", "pkv_launch_count",
           "PkvError", "DEV_ERR_BITS", "TRACE_KINDS", "load", "library_path"]

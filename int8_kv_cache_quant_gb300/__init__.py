"""INT8-KV-cache attention for GB300: Python binding of the libkvq C ABI.

The compute path is libkvq.so (hand-written CUDA for sm_103a, built by
``int8_kv_cache_quant_gb300.build.build()``); this package only marshals torch tensors.
"""
from . import kvq  # noqa: F401
from .kvq import (KVCache, KvqError, kvq_attn_decode_int8kv, kvq_attn_decode_int8kv_noalloc,  # noqa: F401
                  kvq_attn_prefill_first_bf16, kvq_attn_prefill_int8, kvq_attn_prefill_int8_qcodes, kvq_rope_quant_write,
                  kvq_attn_sparse_int8kv, kvq_attn_verify_int8kv, kvq_debug_fault_inject, kvq_debug_prefill_q_codes,
                  kvq_debug_stream_floor,
                  kvq_debug_prefill_qk_int32,
                  kvq_decode_auto_split_rows, kvq_decode_step_int8kv, kvq_decode_workspace_bytes, kvq_device_status,
                  kvq_prefill_split_tiles, kvq_device_accessible,
                  kvq_prefill_first_workspace_bytes, kvq_prefill_workspace_bytes, kvq_sparse_workspace_bytes, kvq_verify_workspace_bytes,
                  kvq_quant_write, kvq_version, lib)

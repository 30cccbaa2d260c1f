"""Asymmetric low-bit KV cache (per-channel keys, per-token values, fp16 window)
with split-K decode attention, as a CUDA library for GB300 (sm_103a).

The compute lives in ``_lib/libkvq.so`` (C ABI: ``include/kvq.h``); ``kvq``
is its Python binding.
"""
from .kvq import (KVCache, KVQError, kvq_append, kvq_config, kvq_create, kvq_decode_attention, kvq_decode_step,
                  kvq_destroy,
                  kvq_export_unit, kvq_get_splits, kvq_get_state, kvq_launch_count, kvq_page_layout,
                  kvq_prefill_quantize, kvq_reset, kvq_set_codebooks, kvq_set_splits, kvq_sync_status, lib, make_config, status_string)

__all__ = ["KVCache", "KVQError", "kvq_append", "kvq_config", "kvq_create", "kvq_decode_attention", "kvq_decode_step",
           "kvq_destroy",
           "kvq_export_unit", "kvq_get_splits", "kvq_get_state", "kvq_launch_count", "kvq_page_layout",
           "kvq_prefill_quantize",
           "kvq_reset", "kvq_set_codebooks", "kvq_set_splits", "kvq_sync_status", "lib", "make_config",
           "status_string"]

"""GB300-native (sm_103a) low-bit dual-path MLA KV cache: fused writer and decode attention.

The compute path is the CUDA library libmla_qcache.so (C ABI in include/mla_qcache.h);
``binding`` marshals torch tensors into it and ``cache.QuantizedMLACache`` owns the device
buffers (pool, BF16 sink/recent buffers, workspace) of one layer.
"""
from .binding import (DEV_BAD_PAGE, mla_qcache_absorb_query, mla_qcache_decode_attn_pending, mla_qcache_decode_attn_multi, mla_qcache_up_project, DEV_NONFINITE, DEV_RANGE, DEV_ROWS, DEV_SEQ_OVERFLOW, DEV_TIMEOUT, EXPORTS,
                      Config, QCacheError, bf16_workspace_bytes, decode_plan, decode_launches, lib, selftest_wait_timeout, make_config, mla_qcache_advance,
                      mla_qcache_decode_attn, mla_qcache_decode_attn_bf16, mla_qcache_row_transform,
                      mla_qcache_write, mla_qcache_write_advance, mla_qcache_write_transformed, page_bytes, strerror, workspace_bytes)
from .cache import QuantizedMLACache

__all__ = ["Config", "QCacheError", "QuantizedMLACache", "lib", "make_config", "mla_qcache_advance", "mla_qcache_decode_attn",
           "mla_qcache_decode_attn_pending",
           "mla_qcache_write", "mla_qcache_write_advance", "mla_qcache_decode_attn_bf16", "bf16_workspace_bytes",
           "mla_qcache_write_transformed", "mla_qcache_row_transform",
           "mla_qcache_absorb_query", "mla_qcache_up_project", "mla_qcache_decode_attn_multi", "decode_plan", "decode_launches",
           "selftest_wait_timeout",
           "page_bytes", "strerror", "workspace_bytes", "EXPORTS", "DEV_BAD_PAGE",
           "DEV_NONFINITE", "DEV_RANGE", "DEV_ROWS", "DEV_SEQ_OVERFLOW", "DEV_TIMEOUT"]

"""GB300-native quantized KV cache (KIVI-style asymmetric quantizer) with a
split-K GQA decode attention, exposed through the C ABI of include/kvq.h."""

from .binding import (EXPORTED, KVQ_BF16, KVQ_FP32, KVQCache, KVQError, compare, kvq_append,  # noqa: F401
                      kvq_bytes, kvq_compare, kvq_create, kvq_create_paged, kvq_dense_decode_attention,
                      kvq_create_segmented, kvq_decode_step, kvq_pool_state, kvq_release, kvq_required_bytes_paged,
                      kvq_required_bytes_segmented, kvq_restore, kvq_decode_attention, kvq_decode_attention_ex,
                      kvq_decode_attention_noalloc, kvq_destroy,
                      kvq_device_status, kvq_export_pages, kvq_export_unit, kvq_kernel_launches, kvq_ledger, kvq_page_bytes,
                      kvq_required_bytes, kvq_seq_state, load_library, make_config)

"""GB300-native closed-form cross-model KV-cache transfer.

The computation lives in libkvb.so (CUDA for sm_103a, C ABI in include/kvb.h);
this package is its thin Python binding plus the in-tree build script.
"""
from ._binding import (  # noqa: F401
    KVB_BF16,
    KVB_F32,
    Ctx,
    KvbError,
    SIGNATURES,
    Stats,
    kvb_attention_cosine,
    kvb_ctx_check,
    kvb_ctx_create,
    kvb_ctx_destroy,
    kvb_ctx_reserve,
    kvb_layer_select,
    kvb_map_apply,
    kvb_map_apply_noalloc,
    kvb_model_spec,
    kvb_profile_enable,
    kvb_profile_read,
    kvb_ridge_solve,
    kvb_stats_accumulate,
    kvb_stats_count,
    kvb_stats_create,
    kvb_stats_create_block,
    kvb_stats_destroy,
    kvb_stats_export,
    kvb_stats_import,
    kvb_stats_reset,
    kvb_version,
    load_library,
)

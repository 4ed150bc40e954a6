// Calibration statistics, selection and ridge solve: entry points.
#include "kvb_host.h"

using namespace kvb;

struct kvb_stats {
    kvb_ctx* ctx = nullptr;
};

extern "C" {

kvb_status kvb_stats_create(kvb_ctx* ctx, kvb_dtype, int64_t, kvb_stats** out) {
    g_last_error.clear();
    if (out) *out = nullptr;
    if (!ctx || !out) return fail(KVB_ERR_INVALID_ARG, "NULL argument");
    return fail(KVB_ERR_UNSUPPORTED, "statistics path not built yet");
}

kvb_status kvb_stats_destroy(kvb_stats* st) {
    delete st;
    return KVB_OK;
}

kvb_status kvb_stats_reset(kvb_stats*, void*) { return fail(KVB_ERR_UNSUPPORTED, "statistics path not built yet"); }

kvb_status kvb_stats_accumulate(kvb_ctx*, kvb_stats*, const void*, const void*, const void*, const void*,
                                const int32_t*, int64_t, int32_t, void*) {
    return fail(KVB_ERR_UNSUPPORTED, "statistics path not built yet");
}

kvb_status kvb_stats_count(kvb_stats*, int64_t*, void*) {
    return fail(KVB_ERR_UNSUPPORTED, "statistics path not built yet");
}

kvb_status kvb_layer_select(kvb_ctx*, kvb_stats*, double, int32_t*, int32_t*, float*, void*) {
    return fail(KVB_ERR_UNSUPPORTED, "statistics path not built yet");
}

kvb_status kvb_ridge_solve(kvb_ctx*, kvb_stats*, const int32_t*, const int32_t*, double, kvb_dtype, void*, void*,
                           float*, float*, void*) {
    return fail(KVB_ERR_UNSUPPORTED, "statistics path not built yet");
}

}  // extern "C"

// Host-side state of a libkvb context and the helpers every entry point uses.
#pragma once

#include <initializer_list>
#include <string>
#include <vector>

#include "kvb_internal.h"

struct kvb_ctx {
    kvb_model_spec src{}, tgt{};
    int L_s = 0, L_t = 0, H = 0, d = 0, k = 0;
    int max_pos = 0;
    int device = 0;
    int num_sms = 0;
    uint64_t timeout_ns = 0;
    float2* tab_s = nullptr;   // source RoPE cos/sin [max_pos][d/2]
    float2* tab_t = nullptr;   // target RoPE cos/sin [max_pos][d/2]
    void* scratch = nullptr;   // stripped source keys for the tensor-core path
    size_t scratch_bytes = 0;
    int* err_dev = nullptr;    // error word written by kernels
    int* strip_ctr = nullptr;  // [4]: next / finished chunk of the strip fused into the map kernel, next map tile
    int* err_mirror = nullptr; // pinned host copy, refreshed after each call
    // kernel timing (kvb_profile_enable / kvb_profile_read)
    struct ProfRec {
        const char* name;
        cudaEvent_t start, end;
    };
    bool profiling = false;
    std::vector<ProfRec> prof;
    std::vector<cudaEvent_t> event_pool;
};

namespace kvb {

extern thread_local std::string g_last_error;

kvb_status fail(kvb_status s, const std::string& msg);
kvb_status cuda_fail(cudaError_t e, const char* what);
bool aligned16(const void* p);
kvb_status check_device_ptrs(std::initializer_list<const void*> ptrs, const char* what);
// Rows [t_begin, t_end) of a [L_tgt][k] selection (t_end < 0: all rows).
kvb_status check_selection(const kvb_ctx* c, const int32_t* sel, const char* name, SelTable* tab, int kv,
                           int t_begin = 0, int t_end = -1);
kvb_status take_device_error(kvb_ctx* c);
void mirror_device_error(kvb_ctx* c, cudaStream_t s);
DevErr dev_err(const kvb_ctx* c);

// Bracket one launch with events when profiling is on (no-op otherwise).
struct ProfScope {
    kvb_ctx* c;
    cudaStream_t s;
    int idx = -1;
    ProfScope(kvb_ctx* ctx, cudaStream_t stream, const char* name);
    ~ProfScope();
};

}  // namespace kvb

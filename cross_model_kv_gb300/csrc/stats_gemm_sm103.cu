// Statistics GEMM on the tensor cores (placeholder until the tcgen05 kernel lands).
#include "stats_internal.h"

namespace kvb {

struct StatsGemmPlan {
    int* tiles = nullptr;
    int n_tiles = 0;
};

bool stats_gemm_tc_supported(const StatsJob*, int) { return false; }
cudaError_t stats_gemm_tc_plan(const StatsJob*, int, StatsGemmPlan** plan) {
    *plan = nullptr;
    return cudaErrorNotSupported;
}
void stats_gemm_tc_free(StatsGemmPlan* plan) { delete plan; }
cudaError_t launch_stats_gemm_tc(StatsGemmPlan*, const StatsJob*, int, int64_t, const float*, const int*, DevErr,
                                 int, cudaStream_t, std::string* why) {
    if (why) *why = "not available";
    return cudaErrorNotSupported;
}

}  // namespace kvb

// Internal declarations of the fit kernels (gather, R^2, top-k, W and b output).
#pragma once

#include "stats_internal.h"

namespace kvb {

constexpr int MAX_SYS = 64;  // systems solved together in one batch (every target layer of a 64-layer model)

// Feature blocks of each system: system b uses source layers layer[b][0..k) (each
// q = H*d features wide) and target columns col0[b] .. col0[b] + m.
struct SysLayers {
    int layer[MAX_SYS][MAX_K];
    int64_t col0[MAX_SYS];
};

// Where system b writes its solution: W [q][n] (output-major) and bias [q].
struct SysOut {
    void* W[MAX_SYS];
    float* bias[MAX_SYS];
};

cudaError_t launch_gather_system(const float* M, int64_t ldm, const SysLayers& L, int q, int64_t n, float lambda,
                                 float* G, int64_t strideG, float* D, int batch, cudaStream_t s);
cudaError_t launch_gather_rhs(const float* C, int64_t ldc, const SysLayers& L, int q, int64_t n, int64_t m,
                              const float* D, float* R, int64_t strideR, int batch, cudaStream_t s);
cudaError_t launch_sse(const float* C, int64_t ldc, const SysLayers& L, int q, int64_t n, int64_t m, const float* D,
                       const float* Wsc, int64_t strideW, const float* syy, float lambda, float* sse, int batch,
                       cudaStream_t s);
cudaError_t launch_r2_head(const float* sse, int64_t m, const float* syy, int L_t, int H, int d,
                           const SysLayers& L, float* r2, int L_s, int batch, cudaStream_t s);
cudaError_t launch_topk(const float* r2, int rows, int L_s, int k, int* sel, cudaStream_t s);
cudaError_t launch_write_w(kvb_dtype dt, const float* Wsc, int64_t strideW, const float* D, int64_t n, int64_t m,
                           const SysOut& O, int batch, cudaStream_t s);
cudaError_t launch_bias(const float* Wsc, int64_t strideW, const float* D, int64_t n, int64_t m, const SysLayers& L,
                        int q, const float* xbar, const float* ybar, const SysOut& O, int batch, cudaStream_t s);

}  // namespace kvb

// Kernels of the fit that sit around the dense solves: gathering Jacobi-scaled
// systems out of the full-source statistics, the single-source R^2 closed
// form, top-k selection, and writing W and b.
//
// "KVBridge" README, "What ships": head-averaged single-source R^2, then top-k;
// "Loading": W = (X^T X + lambda I)^-1 X^T Y, b = Ybar - Xbar W on centered data.
// With the centered Gram M, cross C and S_yy of one (source, target) pair and
// the ridge solution W, the in-sample residual per target column is
//   SSE = S_yy - diag(C^T W) - lambda diag(W^T W)
// (expand |Yc - Xc W|^2 and use (M + lambda I) W = C).
#include "fit_internal.h"

namespace kvb {

namespace {

__device__ __forceinline__ int64_t feat_index(const SysLayers& L, int b, int64_t i, int q) {
    return static_cast<int64_t>(L.layer[b][i / q]) * q + (i % q);
}

__device__ __forceinline__ float gram_at(const float* M, int64_t ld, int64_t i, int64_t j) {
    return i >= j ? M[i * ld + j] : M[j * ld + i];  // lower triangle is the stored half
}

// D[b][i] = 1 / sqrt(M_ii + lambda);  G[b][i][j] = D_i D_j (M[f(i)][f(j)] + lambda [i == j]).
__global__ void gather_system_kernel(const float* __restrict__ M, int64_t ldm, SysLayers L, int q, int64_t n,
                                     float lambda, float* __restrict__ G, int64_t strideG,
                                     float* __restrict__ D) {
    const int b = blockIdx.z;
    const int64_t i = blockIdx.y * static_cast<int64_t>(blockDim.y) + threadIdx.y;
    const int64_t j = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (i >= n || j >= n) return;
    const int64_t fi = feat_index(L, b, i, q), fj = feat_index(L, b, j, q);
    const float di = rsqrtf(M[fi * ldm + fi] + lambda);
    const float dj = rsqrtf(M[fj * ldm + fj] + lambda);
    float v = gram_at(M, ldm, fi, fj) + (i == j ? lambda : 0.f);
    G[b * strideG + i * n + j] = di * v * dj;
    if (j == 0) D[b * n + i] = di;
}

// D[b][i] = 1 / sqrt(M_ii + lambda), once per system, for the tiled gather below.
__global__ void jacobi_scale_kernel(const float* __restrict__ M, int64_t ldm, SysLayers L, int q, int64_t n,
                                    float lambda, float* __restrict__ D) {
    const int b = blockIdx.y;
    const int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (i >= n) return;
    const int64_t fi = feat_index(L, b, i, q);
    D[b * n + i] = rsqrtf(M[fi * (ldm + 1)] + lambda);
}

// Same values as gather_system_kernel from 32 x 32 tiles of G (q a multiple of
// 32, so a tile's rows, and its columns, are 32 consecutive features of one
// layer), GS_TILES tiles of one tile row per block, with the scales D computed
// beforehand.  A tile whose row and column features do not overlap lies wholly
// in the stored lower triangle or wholly above it: it is read as 32 coalesced
// rows of M, either directly or transposed through shared memory.  Tiles whose
// feature ranges overlap take the element-wise path.
constexpr int GS_TILES = 8;

__global__ void __launch_bounds__(256) gather_system_tiled_kernel(const float* __restrict__ M, int64_t ldm,
                                                                  SysLayers L, int q, int64_t n, float lambda,
                                                                  float* __restrict__ G, int64_t strideG,
                                                                  const float* __restrict__ D) {
    __shared__ float tile[32][33];
    __shared__ float di_s[32], dj_s[32];
    const int b = blockIdx.z;
    const int64_t i0 = static_cast<int64_t>(blockIdx.y) * 32;
    const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8
    const int64_t fi0 = feat_index(L, b, i0, q);
    if (ty == 0) di_s[tx] = i0 + tx < n ? D[b * n + i0 + tx] : 0.f;
#pragma unroll 1
    for (int t = 0; t < GS_TILES; ++t) {
        const int64_t j0 = (static_cast<int64_t>(blockIdx.x) * GS_TILES + t) * 32;
        if (j0 >= n) break;  // uniform over the block
        const int64_t fj0 = feat_index(L, b, j0, q);
        __syncthreads();  // the previous tile is stored (and di_s is visible)
        if (ty == 1) dj_s[tx] = j0 + tx < n ? D[b * n + j0 + tx] : 0.f;
        const bool lower = fi0 >= fj0 + 32, upper = fj0 >= fi0 + 32;
        if (lower || upper) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int r = ty + 8 * k;
                // lower: row fi0 + r of M, columns fj0 ..; upper: row fj0 + r, columns fi0 ..
                const bool in = lower ? (i0 + r < n && j0 + tx < n) : (j0 + r < n && i0 + tx < n);
                tile[r][tx] = in ? (lower ? M[(fi0 + r) * ldm + fj0 + tx] : M[(fj0 + r) * ldm + fi0 + tx]) : 0.f;
            }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int r = ty + 8 * k;
            const int64_t i = i0 + r, j = j0 + tx;
            if (i >= n || j >= n) continue;
            float v;
            if (lower)
                v = tile[r][tx];
            else if (upper)
                v = tile[tx][r];
            else
                v = gram_at(M, ldm, fi0 + r, fj0 + tx) + (i == j ? lambda : 0.f);
            G[b * strideG + i * n + j] = di_s[r] * v * dj_s[tx];
        }
    }
}

// R[b][i][c] = D_i C[f(i)][col0_b + c] for c < m.
__global__ void gather_rhs_kernel(const float* __restrict__ C, int64_t ldc_stats, SysLayers L, int q, int64_t n,
                                  int64_t m, const float* __restrict__ D, float* __restrict__ R, int64_t strideR) {
    const int b = blockIdx.z;
    const int64_t i = blockIdx.y;
    const int64_t fi = feat_index(L, b, i, q);
    const float di = D[b * n + i];
    const float* src = C + fi * ldc_stats + L.col0[b];
    float* dst = R + b * strideR + i * m;
    for (int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; c < m;
         c += static_cast<int64_t>(gridDim.x) * blockDim.x)
        dst[c] = di * src[c];
}

// SSE[b][c] = S_yy[c] - sum_i C_ic W_ic - lambda sum_i W_ic^2, with the scaled
// solution W'_ic = W_ic / D_i and C_ic = C'_ic / D_i.
__global__ void sse_kernel(const float* __restrict__ C, int64_t ldc_stats, SysLayers L, int q, int64_t n,
                           int64_t m, const float* __restrict__ D, const float* __restrict__ Wsc, int64_t strideW,
                           const float* __restrict__ syy, float lambda, float* __restrict__ sse) {
    const int b = blockIdx.y;
    const int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (c >= m) return;
    float q1 = 0.f, q2 = 0.f;
    for (int64_t i = 0; i < n; ++i) {
        const float di = D[b * n + i];
        const float w = Wsc[b * strideW + i * m + c] * di;          // W_ic
        const float cc = C[feat_index(L, b, i, q) * ldc_stats + L.col0[b] + c];  // C_ic
        q1 = fmaf(cc, w, q1);
        q2 = fmaf(w, w, q2);
    }
    sse[static_cast<int64_t>(b) * m + c] = syy[L.col0[b] + c] - q1 - lambda * q2;
}

// R2[t][s_b] = mean over heads of 1 - sum SSE / sum S_yy over the head's d columns.
__global__ void r2_head_kernel(const float* __restrict__ sse, int64_t m, const float* __restrict__ syy, int L_t,
                               int H, int d, SysLayers L, float* __restrict__ r2, int L_s) {
    const int b = blockIdx.y;
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= L_t) return;
    float acc = 0.f;
    for (int h = 0; h < H; ++h) {
        float e = 0.f, tot = 0.f;
        const int64_t c0 = (static_cast<int64_t>(t) * H + h) * d;
        for (int c = 0; c < d; ++c) {
            e += sse[static_cast<int64_t>(b) * m + c0 + c];
            tot += syy[c0 + c];
        }
        acc += tot > 0.f ? 1.f - e / tot : 0.f;
    }
    r2[static_cast<int64_t>(t) * L_s + L.layer[b][0]] = acc / static_cast<float>(H);
}

// Per (kv, t) row of R2[kv][t][:]: the k best sources by (R2 desc, index asc), ascending.
__global__ void topk_kernel(const float* __restrict__ r2, int rows, int L_s, int k, int* __restrict__ sel) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= rows) return;
    const float* v = r2 + static_cast<int64_t>(r) * L_s;
    uint32_t taken[8] = {0, 0, 0, 0, 0, 0, 0, 0};  // up to 256 sources
    int out[MAX_K];
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int s = 0; s < L_s; ++s) {
            if (taken[s >> 5] & (1u << (s & 31))) continue;
            if (best < 0 || v[s] > v[best]) best = s;  // strict: ties keep the lower index
        }
        taken[best >> 5] |= 1u << (best & 31);
        out[j] = best;
    }
    for (int a = 1; a < k; ++a)  // ascending
        for (int b2 = a; b2 > 0 && out[b2 - 1] > out[b2]; --b2) {
            const int t2 = out[b2];
            out[b2] = out[b2 - 1];
            out[b2 - 1] = t2;
        }
    for (int j = 0; j < k; ++j) sel[static_cast<int64_t>(r) * k + j] = out[j];
}

// Output W[t][c][i] = D_i W'[i][c] (transposed, to the output-major layout).
template <typename To>
__global__ void write_w_kernel(const float* __restrict__ Wsc, int64_t strideW, const float* __restrict__ D,
                               int64_t n, int64_t m, SysOut O) {
    __shared__ float tile[32][33];
    const int b = blockIdx.z;
    const int64_t i0 = static_cast<int64_t>(blockIdx.y) * 32, c0 = static_cast<int64_t>(blockIdx.x) * 32;
    for (int r = threadIdx.y; r < 32; r += blockDim.y) {
        const int64_t i = i0 + r, c = c0 + threadIdx.x;
        tile[r][threadIdx.x] = (i < n && c < m) ? Wsc[b * strideW + i * m + c] * D[b * n + i] : 0.f;
    }
    __syncthreads();
    To* W = static_cast<To*>(O.W[b]);
    for (int r = threadIdx.y; r < 32; r += blockDim.y) {
        const int64_t c = c0 + r, i = i0 + threadIdx.x;
        if (c < m && i < n) {
            const float v = tile[threadIdx.x][r];
            if constexpr (sizeof(To) == 4)
                W[c * n + i] = v;
            else
                W[c * n + i] = __float2bfloat16_rn(v);
        }
    }
}

// b[c] = ybar[c] - sum_i xbar[f(i)] W_ic.
__global__ void bias_kernel(const float* __restrict__ Wsc, int64_t strideW, const float* __restrict__ D, int64_t n,
                            int64_t m, SysLayers L, int q, const float* __restrict__ xbar,
                            const float* __restrict__ ybar, SysOut O) {
    const int b = blockIdx.y;
    const int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (c >= m) return;
    float acc = 0.f;
    for (int64_t i = 0; i < n; ++i)
        acc = fmaf(xbar[feat_index(L, b, i, q)], Wsc[b * strideW + i * m + c] * D[b * n + i], acc);
    O.bias[b][c] = ybar[L.col0[b] + c] - acc;
}

}  // namespace

cudaError_t launch_gather_system(const float* M, int64_t ldm, const SysLayers& L, int q, int64_t n, float lambda,
                                 float* G, int64_t strideG, float* D, int batch, cudaStream_t s) {
    dim3 blk(32, 8);
    if (q % 32 == 0) {
        jacobi_scale_kernel<<<dim3(static_cast<unsigned>((n + 255) / 256), batch), 256, 0, s>>>(M, ldm, L, q, n,
                                                                                                 lambda, D);
        const int64_t tiles = (n + 31) / 32;
        dim3 grid(static_cast<unsigned>((tiles + GS_TILES - 1) / GS_TILES), static_cast<unsigned>(tiles), batch);
        gather_system_tiled_kernel<<<grid, blk, 0, s>>>(M, ldm, L, q, n, lambda, G, strideG, D);
        return cudaGetLastError();
    }
    dim3 grid(static_cast<unsigned>((n + 31) / 32), static_cast<unsigned>((n + 7) / 8), batch);
    gather_system_kernel<<<grid, blk, 0, s>>>(M, ldm, L, q, n, lambda, G, strideG, D);
    return cudaGetLastError();
}

cudaError_t launch_gather_rhs(const float* C, int64_t ldc, const SysLayers& L, int q, int64_t n, int64_t m,
                              const float* D, float* R, int64_t strideR, int batch, cudaStream_t s) {
    dim3 grid(static_cast<unsigned>(m >= 256 * 8 ? 8 : (m + 255) / 256), static_cast<unsigned>(n), batch);
    gather_rhs_kernel<<<grid, 256, 0, s>>>(C, ldc, L, q, n, m, D, R, strideR);
    return cudaGetLastError();
}

cudaError_t launch_sse(const float* C, int64_t ldc, const SysLayers& L, int q, int64_t n, int64_t m, const float* D,
                       const float* Wsc, int64_t strideW, const float* syy, float lambda, float* sse, int batch,
                       cudaStream_t s) {
    dim3 grid(static_cast<unsigned>((m + 255) / 256), batch);
    sse_kernel<<<grid, 256, 0, s>>>(C, ldc, L, q, n, m, D, Wsc, strideW, syy, lambda, sse);
    return cudaGetLastError();
}

cudaError_t launch_r2_head(const float* sse, int64_t m, const float* syy, int L_t, int H, int d,
                           const SysLayers& L, float* r2, int L_s, int batch, cudaStream_t s) {
    dim3 grid(static_cast<unsigned>((L_t + 63) / 64), batch);
    r2_head_kernel<<<grid, 64, 0, s>>>(sse, m, syy, L_t, H, d, L, r2, L_s);
    return cudaGetLastError();
}

cudaError_t launch_topk(const float* r2, int rows, int L_s, int k, int* sel, cudaStream_t s) {
    topk_kernel<<<(rows + 63) / 64, 64, 0, s>>>(r2, rows, L_s, k, sel);
    return cudaGetLastError();
}

cudaError_t launch_write_w(kvb_dtype dt, const float* Wsc, int64_t strideW, const float* D, int64_t n, int64_t m,
                           const SysOut& O, int batch, cudaStream_t s) {
    dim3 blk(32, 8);
    dim3 grid(static_cast<unsigned>((m + 31) / 32), static_cast<unsigned>((n + 31) / 32), batch);
    if (dt == KVB_F32)
        write_w_kernel<float><<<grid, blk, 0, s>>>(Wsc, strideW, D, n, m, O);
    else
        write_w_kernel<__nv_bfloat16><<<grid, blk, 0, s>>>(Wsc, strideW, D, n, m, O);
    return cudaGetLastError();
}

cudaError_t launch_bias(const float* Wsc, int64_t strideW, const float* D, int64_t n, int64_t m, const SysLayers& L,
                        int q, const float* xbar, const float* ybar, const SysOut& O, int batch, cudaStream_t s) {
    dim3 grid(static_cast<unsigned>((m + 127) / 128), batch);
    bias_kernel<<<grid, 128, 0, s>>>(Wsc, strideW, D, n, m, L, q, xbar, ybar, O);
    return cudaGetLastError();
}

}  // namespace kvb

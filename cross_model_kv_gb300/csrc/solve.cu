// Batched float32 dense linear algebra on the CUDA cores: GEMM, blocked
// Cholesky and the two triangular solves.  Used by the single-source R^2
// fits and by the ridge solve W = (M + lambda I)^-1 C ("KVBridge" README,
// "Loading"), on Jacobi-scaled systems.
#include "stats_internal.h"

namespace kvb {

namespace {

constexpr int GB = 128;  // tile M and N
constexpr int GK = 8;    // tile K
constexpr int NB = 64;   // Cholesky panel width

// 128x128x8 tiles, 256 threads, 8x8 outputs per thread (two 4x4 quadrants
// 64 apart so shared-memory reads stay conflict-free).
__global__ void __launch_bounds__(256) gemm_f32_kernel(const GemmArgs g) {
    __shared__ float As[GK][GB];
    __shared__ float Bs[GK][GB];
    const int b = blockIdx.z;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * GB;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * GB;
    if (g.lower && n0 > m0 + GB - 1) return;
    const float* A = g.A + b * g.strideA;
    const float* B = g.B + b * g.strideB;
    float* C = g.C + b * g.strideC;
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const bool a_kfast = g.sak == 1;
    const bool b_nfast = g.sbn == 1;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    for (int64_t k0 = 0; k0 < g.K; k0 += GK) {
#pragma unroll
        for (int q = 0; q < (GB * GK) / 256; ++q) {
            const int e = tid + q * 256;
            int mm, kk;
            if (a_kfast) {
                kk = e % GK;
                mm = e / GK;
            } else {
                mm = e % GB;
                kk = e / GB;
            }
            const int64_t gm = m0 + mm, gk = k0 + kk;
            As[kk][mm] = (gm < g.M && gk < g.K) ? A[gm * g.sam + gk * g.sak] : 0.f;
            int nn, kb;
            if (b_nfast) {
                nn = e % GB;
                kb = e / GB;
            } else {
                kb = e % GK;
                nn = e / GK;
            }
            const int64_t gn = n0 + nn, gk2 = k0 + kb;
            Bs[kb][nn] = (gn < g.N && gk2 < g.K) ? B[gk2 * g.sbk + gn * g.sbn] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < GK; ++kk) {
            float a[8], bb[8];
            const float4 a0 = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[kk][ty * 4 + 64]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4 + 64]);
            a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
            a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
            bb[0] = b0.x; bb[1] = b0.y; bb[2] = b0.z; bb[3] = b0.w;
            bb[4] = b1.x; bb[5] = b1.y; bb[6] = b1.z; bb[7] = b1.w;
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t gm = m0 + ty * 4 + (i & 3) + (i >> 2) * 64;
        if (gm >= g.M) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int64_t gn = n0 + tx * 4 + (j & 3) + (j >> 2) * 64;
            if (gn >= g.N) continue;
            float* p = C + gm * g.ldc + gn;
            *p = g.alpha * acc[i][j] + (g.beta == 0.f ? 0.f : g.beta * *p);
        }
    }
}

// Cholesky of the nb x nb diagonal block at (k0, k0), in shared memory.  One CTA per system.
__global__ void __launch_bounds__(256) potrf_diag_kernel(float* G, int64_t ldg, int64_t strideG, int64_t k0,
                                                         int nb, int* numeric_flag) {
    __shared__ float a[NB][NB + 1];
    float* Gb = G + blockIdx.x * strideG + k0 * ldg + k0;
    for (int e = threadIdx.x; e < nb * nb; e += blockDim.x) {
        const int i = e / nb, j = e % nb;
        a[i][j] = Gb[i * ldg + j];
    }
    __syncthreads();
    for (int j = 0; j < nb; ++j) {
        if (threadIdx.x == 0) {
            float v = a[j][j];
            if (!(v > 0.f)) {  // not positive definite (or NaN): record, keep going with a tiny pivot
                if (numeric_flag) atomicExch(numeric_flag, 1);
                v = 1e-30f;
            }
            a[j][j] = sqrtf(v);
        }
        __syncthreads();
        const float piv = a[j][j];
        for (int i = j + 1 + threadIdx.x; i < nb; i += blockDim.x) a[i][j] /= piv;
        __syncthreads();
        // trailing update of the lower triangle
        const int rem = nb - j - 1;
        for (int e = threadIdx.x; e < rem * rem; e += blockDim.x) {
            const int i = j + 1 + e / rem, c = j + 1 + e % rem;
            if (c <= i) a[i][c] = fmaf(-a[i][j], a[c][j], a[i][c]);
        }
        __syncthreads();
    }
    for (int e = threadIdx.x; e < nb * nb; e += blockDim.x) {
        const int i = e / nb, j = e % nb;
        Gb[i * ldg + j] = j <= i ? a[i][j] : 0.f;
    }
}

// Panel below the diagonal block: P <- P L_kk^-T (rows independent).  Thread per row.
__global__ void trsm_panel_kernel(float* G, int64_t ldg, int64_t strideG, int64_t k0, int nb, int64_t rows) {
    __shared__ float L[NB][NB + 1];
    float* Gs = G + blockIdx.y * strideG;
    for (int e = threadIdx.x; e < nb * nb; e += blockDim.x) {
        const int i = e / nb, j = e % nb;
        L[i][j] = Gs[(k0 + i) * ldg + k0 + j];
    }
    __syncthreads();
    const int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (r >= rows) return;
    float* row = Gs + (k0 + nb + r) * ldg + k0;
    float x[NB];
#pragma unroll 4
    for (int j = 0; j < nb; ++j) {
        float v = row[j];
        for (int k = 0; k < j; ++k) v = fmaf(-x[k], L[j][k], v);
        x[j] = v / L[j][j];
    }
    for (int j = 0; j < nb; ++j) row[j] = x[j];
}

// Block row k0..k0+nb of C: forward (L_kk Y = C_k) or backward (L_kk^T X = Y_k).
// Thread per right-hand-side column.
__global__ void trsm_rhs_kernel(const float* L, int64_t ldg, int64_t strideG, int64_t k0, int nb, float* C,
                                int64_t ldc, int64_t strideC, int64_t m, int backward) {
    __shared__ float Ls[NB][NB + 1];
    const float* Lb = L + blockIdx.y * strideG;
    for (int e = threadIdx.x; e < nb * nb; e += blockDim.x) {
        const int i = e / nb, j = e % nb;
        Ls[i][j] = Lb[(k0 + i) * ldg + k0 + j];
    }
    __syncthreads();
    const int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (c >= m) return;
    float* col = C + blockIdx.y * strideC + k0 * ldc + c;
    float y[NB];
    for (int i = 0; i < nb; ++i) y[i] = col[i * ldc];
    if (!backward) {
        for (int i = 0; i < nb; ++i) {
            float v = y[i];
            for (int k = 0; k < i; ++k) v = fmaf(-Ls[i][k], y[k], v);
            y[i] = v / Ls[i][i];
        }
    } else {
        for (int i = nb - 1; i >= 0; --i) {
            float v = y[i];
            for (int k = i + 1; k < nb; ++k) v = fmaf(-Ls[k][i], y[k], v);
            y[i] = v / Ls[i][i];
        }
    }
    for (int i = 0; i < nb; ++i) col[i * ldc] = y[i];
}

}  // namespace

cudaError_t launch_gemm_f32(const GemmArgs& g, cudaStream_t s) {
    if (g.M <= 0 || g.N <= 0 || g.batch <= 0) return cudaSuccess;
    dim3 grid(static_cast<unsigned>((g.N + GB - 1) / GB), static_cast<unsigned>((g.M + GB - 1) / GB), g.batch);
    gemm_f32_kernel<<<grid, 256, 0, s>>>(g);
    return cudaGetLastError();
}

cudaError_t chol_factor_batched(float* G, int64_t ldg, int64_t strideG, int64_t n, int batch, int* numeric_flag,
                                cudaStream_t s) {
    for (int64_t k0 = 0; k0 < n; k0 += NB) {
        const int nb = static_cast<int>(n - k0 < NB ? n - k0 : NB);
        potrf_diag_kernel<<<batch, 256, 0, s>>>(G, ldg, strideG, k0, nb, numeric_flag);
        const int64_t rem = n - k0 - nb;
        if (rem <= 0) continue;
        dim3 tg(static_cast<unsigned>((rem + 127) / 128), batch);
        trsm_panel_kernel<<<tg, 128, 0, s>>>(G, ldg, strideG, k0, nb, rem);
        GemmArgs g{};
        g.A = G + (k0 + nb) * ldg + k0;  // P: rem x nb
        g.B = G + (k0 + nb) * ldg + k0;  // P^T: B(k, n) = P[n][k]
        g.C = G + (k0 + nb) * ldg + (k0 + nb);
        g.sam = ldg;
        g.sak = 1;
        g.sbk = 1;
        g.sbn = ldg;
        g.ldc = ldg;
        g.strideA = g.strideB = g.strideC = strideG;
        g.M = g.N = rem;
        g.K = nb;
        g.alpha = -1.f;
        g.beta = 1.f;
        g.batch = batch;
        g.lower = 1;
        cudaError_t e = launch_gemm_f32(g, s);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t chol_solve_batched(const float* L, int64_t ldg, int64_t strideG, int64_t n, float* C, int64_t ldc,
                               int64_t strideC, int64_t m, int batch, cudaStream_t s) {
    dim3 tg(static_cast<unsigned>((m + 127) / 128), batch);
    // forward: L Y = C
    for (int64_t k0 = 0; k0 < n; k0 += NB) {
        const int nb = static_cast<int>(n - k0 < NB ? n - k0 : NB);
        trsm_rhs_kernel<<<tg, 128, 0, s>>>(L, ldg, strideG, k0, nb, C, ldc, strideC, m, 0);
        const int64_t rem = n - k0 - nb;
        if (rem <= 0) continue;
        GemmArgs g{};
        g.A = L + (k0 + nb) * ldg + k0;
        g.B = C + k0 * ldc;
        g.C = C + (k0 + nb) * ldc;
        g.sam = ldg;
        g.sak = 1;
        g.sbk = ldc;
        g.sbn = 1;
        g.ldc = ldc;
        g.strideA = strideG;
        g.strideB = g.strideC = strideC;
        g.M = rem;
        g.N = m;
        g.K = nb;
        g.alpha = -1.f;
        g.beta = 1.f;
        g.batch = batch;
        cudaError_t e = launch_gemm_f32(g, s);
        if (e != cudaSuccess) return e;
    }
    // backward: L^T X = Y
    const int64_t last = ((n - 1) / NB) * NB;
    for (int64_t k0 = last; k0 >= 0; k0 -= NB) {
        const int nb = static_cast<int>(n - k0 < NB ? n - k0 : NB);
        trsm_rhs_kernel<<<tg, 128, 0, s>>>(L, ldg, strideG, k0, nb, C, ldc, strideC, m, 1);
        if (k0 == 0) break;
        GemmArgs g{};
        g.A = L + k0 * ldg;  // A(i, kk) = L[k0 + kk][i]
        g.B = C + k0 * ldc;
        g.C = C;
        g.sam = 1;
        g.sak = ldg;
        g.sbk = ldc;
        g.sbn = 1;
        g.ldc = ldc;
        g.strideA = strideG;
        g.strideB = g.strideC = strideC;
        g.M = k0;
        g.N = m;
        g.K = nb;
        g.alpha = -1.f;
        g.beta = 1.f;
        g.batch = batch;
        cudaError_t e = launch_gemm_f32(g, s);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace kvb

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

// Vectorised, double-buffered variant for K % 16 == 0, M and N % 4 == 0 and
// 16-byte aligned operands: 16-byte global loads along the contiguous index of
// A (K or M) and of B (N or K), the next K-slice fetched into registers while
// the current one is multiplied out of shared memory.
template <bool A_KCONTIG, bool B_NCONTIG>
__global__ void __launch_bounds__(256, 2) gemm_f32_vec_kernel(const GemmArgs g) {
    constexpr int BKV = 16;
    __shared__ __align__(16) float As[2][BKV][GB + 4];
    __shared__ __align__(16) float Bs[2][BKV][GB + 4];
    const int b = blockIdx.z;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * GB;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * GB;
    if (g.lower && n0 > m0 + GB - 1) return;
    const float* A = g.A + b * g.strideA;
    const float* B = g.B + b * g.strideB;
    float* C = g.C + b * g.strideC;
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 ra[2], rb[2];

    auto load = [&](int64_t k0) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int e = tid + i * 256;
            if (A_KCONTIG) {
                const int64_t gm = m0 + (e >> 2), gk = k0 + (e & 3) * 4;
                ra[i] = (gm < g.M && gk < g.K) ? __ldg(reinterpret_cast<const float4*>(A + gm * g.sam + gk)) : zero;
            } else {
                const int64_t gk = k0 + (e >> 5), gm = m0 + (e & 31) * 4;
                ra[i] = (gm < g.M && gk < g.K) ? __ldg(reinterpret_cast<const float4*>(A + gk * g.sak + gm)) : zero;
            }
            if (B_NCONTIG) {
                const int64_t gk = k0 + (e >> 5), gn = n0 + (e & 31) * 4;
                rb[i] = (gn < g.N && gk < g.K) ? __ldg(reinterpret_cast<const float4*>(B + gk * g.sbk + gn)) : zero;
            } else {
                const int64_t gn = n0 + (e >> 2), gk = k0 + (e & 3) * 4;
                rb[i] = (gn < g.N && gk < g.K) ? __ldg(reinterpret_cast<const float4*>(B + gn * g.sbn + gk)) : zero;
            }
        }
    };
    auto store = [&](int buf) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int e = tid + i * 256;
            if (A_KCONTIG) {
                const int mm = e >> 2, kk = (e & 3) * 4;
                As[buf][kk + 0][mm] = ra[i].x;
                As[buf][kk + 1][mm] = ra[i].y;
                As[buf][kk + 2][mm] = ra[i].z;
                As[buf][kk + 3][mm] = ra[i].w;
            } else {
                *reinterpret_cast<float4*>(&As[buf][e >> 5][(e & 31) * 4]) = ra[i];
            }
            if (B_NCONTIG) {
                *reinterpret_cast<float4*>(&Bs[buf][e >> 5][(e & 31) * 4]) = rb[i];
            } else {
                const int nn = e >> 2, kk = (e & 3) * 4;
                Bs[buf][kk + 0][nn] = rb[i].x;
                Bs[buf][kk + 1][nn] = rb[i].y;
                Bs[buf][kk + 2][nn] = rb[i].z;
                Bs[buf][kk + 3][nn] = rb[i].w;
            }
        }
    };

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    load(0);
    store(0);
    __syncthreads();
    int buf = 0;
    for (int64_t k0 = 0; k0 < g.K; k0 += BKV) {
        const bool more = k0 + BKV < g.K;
        if (more) load(k0 + BKV);
#pragma unroll
        for (int kk = 0; kk < BKV; ++kk) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4 + 64]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4 + 64]);
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
        }
        if (more) store(buf ^ 1);
        __syncthreads();
        buf ^= 1;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t gm = m0 + ty * 4 + (i & 3) + (i >> 2) * 64;
        if (gm >= g.M) continue;
#pragma unroll
        for (int jh = 0; jh < 2; ++jh) {
            const int64_t gn = n0 + tx * 4 + jh * 64;
            if (gn >= g.N) continue;
            float4* p = reinterpret_cast<float4*>(C + gm * g.ldc + gn);
            float4 v = make_float4(g.alpha * acc[i][4 * jh + 0], g.alpha * acc[i][4 * jh + 1],
                                   g.alpha * acc[i][4 * jh + 2], g.alpha * acc[i][4 * jh + 3]);
            if (g.beta != 0.f) {
                const float4 o = *p;
                v.x = fmaf(g.beta, o.x, v.x);
                v.y = fmaf(g.beta, o.y, v.y);
                v.z = fmaf(g.beta, o.z, v.z);
                v.w = fmaf(g.beta, o.w, v.w);
            }
            *p = v;
        }
    }
}

// Cholesky of the nb x nb diagonal block at (k0, k0), in shared memory.  One CTA per system.
__global__ void __launch_bounds__(256) potrf_diag_kernel(float* G, int64_t ldg, int64_t strideG, int64_t k0,
                                                         int nb, int* numeric_flag, float* Linv, int64_t strideL) {
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
    // Inverse of the lower-triangular factor, column j by forward substitution
    // (one thread per column), stored as a dense NB x NB block.
    float* Li = Linv + blockIdx.x * strideL + k0 * NB;
    if (threadIdx.x < NB) {
        const int j = threadIdx.x;
        float x[NB];
        for (int i = 0; i < NB; ++i) {
            float v = 0.f;
            if (i < nb && i >= j) {
                v = i == j ? 1.f : 0.f;
                for (int k = j; k < i; ++k) v = fmaf(-a[i][k], x[k], v);
                v /= a[i][i];
            }
            x[i] = v;
        }
        for (int i = 0; i < NB; ++i) Li[i * NB + j] = x[i];
    }
}

// In place, X <- A X for one block of nb <= 64 right-hand-side rows (row stride
// ldc) and the inverse of its diagonal block, A(i, k) = Lb[i * NB + k], or that
// inverse transposed, A(i, k) = Lb[k * NB + i]: the triangular solves' diagonal
// steps.  One CTA per 256 columns of one system holds the 64 x 64 block and its
// 64 x 256 slab of X in shared memory (the slab is read whole before any of it is
// written back); each thread owns 8 rows x 8 columns (columns 4c..4c+3 and
// 128+4c..128+4c+3, so that a quarter warp's 16-byte reads cover all banks).
constexpr int DA_COLS = 256;
constexpr int DA_LDA = NB + 4;  // padded row of the block in shared memory (16-byte aligned)
constexpr int DA_SMEM = (NB * DA_LDA + NB * DA_COLS) * 4;

__global__ void __launch_bounds__(256, 2) diag_apply_kernel(const float* __restrict__ Linv, int64_t strideL,
                                                           float* __restrict__ C, int64_t ldc, int64_t strideC,
                                                           int nb, int64_t m, int transpose) {
    extern __shared__ __align__(16) float dsm[];
    float* sa = dsm;              // sa[k * DA_LDA + i] = A(i, k)
    float* sx = dsm + NB * DA_LDA;  // sx[k * DA_COLS + c] = X(k, c0 + c)
    const int b = blockIdx.y;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * DA_COLS;
    const float* Lb = Linv + b * strideL;
    float* X = C + b * strideC;
    for (int e = threadIdx.x; e < NB * NB; e += blockDim.x) {
        const int r = e / NB, q = e - r * NB;  // Lb element (r, q), read in order
        const float v = (r < nb && q < nb) ? Lb[r * NB + q] : 0.f;
        if (transpose)
            sa[r * DA_LDA + q] = v;  // A(q, r) = Lb[r * NB + q]
        else
            sa[q * DA_LDA + r] = v;  // A(r, q) = Lb[r * NB + q]
    }
    for (int e = threadIdx.x; e < NB * (DA_COLS / 4); e += blockDim.x) {
        const int k = e / (DA_COLS / 4), c = 4 * (e - k * (DA_COLS / 4));
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < nb && c0 + c < m) v = *reinterpret_cast<const float4*>(X + k * ldc + c0 + c);
        *reinterpret_cast<float4*>(sx + k * DA_COLS + c) = v;
    }
    __syncthreads();
    const int r0 = 8 * (threadIdx.x >> 5);
    const int cx = 4 * (threadIdx.x & 31);
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
#pragma unroll 4
    for (int k = 0; k < nb; ++k) {
        const float4 a0 = *reinterpret_cast<const float4*>(sa + k * DA_LDA + r0);
        const float4 a1 = *reinterpret_cast<const float4*>(sa + k * DA_LDA + r0 + 4);
        const float4 x0 = *reinterpret_cast<const float4*>(sx + k * DA_COLS + cx);
        const float4 x1 = *reinterpret_cast<const float4*>(sx + k * DA_COLS + 128 + cx);
        const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], xv[j], acc[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = r0 + i;
        if (r >= nb) break;
        float* row = X + r * ldc + c0;
        if (c0 + cx < m) *reinterpret_cast<float4*>(row + cx) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        if (c0 + 128 + cx < m)
            *reinterpret_cast<float4*>(row + 128 + cx) = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
    }
}

}  // namespace

cudaError_t launch_gemm_f32(const GemmArgs& g, cudaStream_t s) {
    if (g.M <= 0 || g.N <= 0 || g.batch <= 0) return cudaSuccess;
    dim3 grid(static_cast<unsigned>((g.N + GB - 1) / GB), static_cast<unsigned>((g.M + GB - 1) / GB), g.batch);
    auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const bool a_k = g.sak == 1, a_m = g.sam == 1, b_n = g.sbn == 1, b_k = g.sbk == 1;
    const int64_t sa = a_k ? g.sam : g.sak, sb = b_n ? g.sbk : g.sbn;
    const bool vec = g.K % 16 == 0 && g.M % 4 == 0 && g.N % 4 == 0 && (a_k || a_m) && (b_n || b_k) && sa % 4 == 0 &&
                     sb % 4 == 0 && g.ldc % 4 == 0 && g.strideA % 4 == 0 && g.strideB % 4 == 0 &&
                     g.strideC % 4 == 0 && al16(g.A) && al16(g.B) && al16(g.C);
    if (!vec) {
        gemm_f32_kernel<<<grid, 256, 0, s>>>(g);
    } else if (a_k && b_n) {
        gemm_f32_vec_kernel<true, true><<<grid, 256, 0, s>>>(g);
    } else if (a_k) {
        gemm_f32_vec_kernel<true, false><<<grid, 256, 0, s>>>(g);
    } else if (b_n) {
        gemm_f32_vec_kernel<false, true><<<grid, 256, 0, s>>>(g);
    } else {
        gemm_f32_vec_kernel<false, false><<<grid, 256, 0, s>>>(g);
    }
    return cudaGetLastError();
}

namespace {

// C[b] = alpha * A[b] B[b]^T + beta * C[b] over a batch of systems, A (M x K)
// and B (N x K) fp32 with element (r, k) at src[r * s_row + k * s_k]: on the
// tensor cores when the update is large, otherwise on the CUDA cores.
cudaError_t update(const TcSolve* tc, const float* A, int64_t a_row, int64_t a_k, int64_t strideA, int64_t M,
                   const float* B, int64_t b_row, int64_t b_k, int64_t strideB, int64_t N, int K, float* C,
                   int64_t ldc, int64_t strideC, float alpha, float beta, bool lower, int batch, cudaStream_t s) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    if (tc_update_supported(tc, M, N, K, C, ldc)) {
        const TcOperand a{A, M, a_row, a_k, strideA};
        if (A == B && a_row == b_row && a_k == b_k && M == N)
            return launch_tc_update(*tc, a, nullptr, K, C, ldc, strideC, alpha, beta, lower, batch, s, nullptr);
        const TcOperand b{B, N, b_row, b_k, strideB};
        return launch_tc_update(*tc, a, &b, K, C, ldc, strideC, alpha, beta, lower, batch, s, nullptr);
    }
    GemmArgs g{};
    g.A = A;
    g.sam = a_row;
    g.sak = a_k;
    g.B = B;  // B(k, n) = B[n * b_row + k * b_k]
    g.sbk = b_k;
    g.sbn = b_row;
    g.C = C;
    g.ldc = ldc;
    g.strideA = strideA;
    g.strideB = strideB;
    g.strideC = strideC;
    g.M = M;
    g.N = N;
    g.K = K;
    g.alpha = alpha;
    g.beta = beta;
    g.batch = batch;
    g.lower = lower ? 1 : 0;
    return launch_gemm_f32(g, s);
}

}  // namespace

// Right-looking blocked Cholesky with super-panels of NSUB 64-wide steps: each
// step's columns are first brought up to date with the earlier steps of the
// same super-panel (left-looking inside it), factored and inverted on the
// diagonal and multiplied into the panel below; the trailing matrix then takes
// one rank-(NSUB * 64) update, so it is read and written once per super-panel.
constexpr int NSUB = 4;
constexpr int SP = NSUB * NB;

cudaError_t chol_factor_batched(float* G, int64_t ldg, int64_t strideG, int64_t n, int batch, int* numeric_flag,
                                float* Linv, int64_t strideL, const TcSolve* tc, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    for (int64_t k0 = 0; k0 < n; k0 += SP) {
        for (int i = 0; i < NSUB; ++i) {
            const int64_t j0 = k0 + static_cast<int64_t>(i) * NB;  // first column of this step
            if (j0 >= n) break;
            const int nb = static_cast<int>(n - j0 < NB ? n - j0 : NB);
            if (i > 0) {  // columns j0.. of rows j0.. minus the earlier steps of this super-panel
                const float* Pp = G + j0 * ldg + k0;  // (n - j0) x (j0 - k0)
                e = update(tc, Pp, ldg, 1, strideG, n - j0, Pp, ldg, 1, strideG, nb, static_cast<int>(j0 - k0),
                           G + j0 * ldg + j0, ldg, strideG, -1.f, 1.f, false, batch, s);
                if (e != cudaSuccess) return e;
            }
            potrf_diag_kernel<<<batch, 256, 0, s>>>(G, ldg, strideG, j0, nb, numeric_flag, Linv, strideL);
            const int64_t rem = n - j0 - nb;
            if (rem <= 0) break;
            // panel below the diagonal block: P <- P L_jj^-T (rows independent, in place);
            // B(k, n) = Linv[n][k]
            e = update(nullptr, G + (j0 + nb) * ldg + j0, ldg, 1, strideG, rem, Linv + j0 * NB, NB, 1, strideL, nb,
                       nb, G + (j0 + nb) * ldg + j0, ldg, strideG, 1.f, 0.f, false, batch, s);
            if (e != cudaSuccess) return e;
        }
        const int64_t t0 = k0 + SP;  // trailing matrix of the super-panel
        if (t0 >= n) break;
        const float* P = G + t0 * ldg + k0;  // (n - t0) x SP
        e = update(tc, P, ldg, 1, strideG, n - t0, P, ldg, 1, strideG, n - t0, SP, G + t0 * ldg + t0, ldg, strideG,
                   -1.f, 1.f, true, batch, s);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t chol_solve_batched(const float* L, int64_t ldg, int64_t strideG, int64_t n, const float* Linv,
                               int64_t strideL, float* C, int64_t ldc, int64_t strideC, int64_t m, int batch,
                               const TcSolve* tc, cudaStream_t s) {
    // Block row j of C times the inverse diagonal block (or its transpose), in place:
    // every output column depends only on the same column of the block row.
    auto diag = [&](int64_t j0, int nb, bool transpose) {
        const bool vec = m % 4 == 0 && ldc % 4 == 0 && strideC % 4 == 0 && strideL % 4 == 0 &&
                         (reinterpret_cast<uintptr_t>(C) & 15u) == 0 && (reinterpret_cast<uintptr_t>(Linv) & 15u) == 0;
        if (vec) {
            const cudaError_t ea =
                cudaFuncSetAttribute(diag_apply_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, DA_SMEM);
            if (ea != cudaSuccess) return ea;
            dim3 grid(static_cast<unsigned>((m + DA_COLS - 1) / DA_COLS), static_cast<unsigned>(batch));
            diag_apply_kernel<<<grid, 256, DA_SMEM, s>>>(Linv + j0 * NB, strideL, C + j0 * ldc, ldc, strideC, nb, m,
                                                         transpose ? 1 : 0);
            return cudaGetLastError();
        }
        GemmArgs t{};
        t.A = Linv + j0 * NB;
        t.B = C + j0 * ldc;
        t.C = C + j0 * ldc;
        t.sam = transpose ? 1 : NB;
        t.sak = transpose ? NB : 1;
        t.sbk = ldc;
        t.sbn = 1;
        t.ldc = ldc;
        t.strideA = strideL;
        t.strideB = t.strideC = strideC;
        t.M = nb;
        t.N = m;
        t.K = nb;
        t.alpha = 1.f;
        t.beta = 0.f;
        t.batch = batch;
        return launch_gemm_f32(t, s);
    };
    cudaError_t e;
    // With many right-hand sides the updates read the super-block's rows of C as
    // their B operand on the tensor cores; each 64-row block is then split into
    // its bf16 parts once, right after its diagonal step (the rows are final for
    // the rest of the pass), into a cache after the A operand's part of the update
    // workspace, and every update reads the cache from the block's column on.
    const bool cached = tc && tc->ws && tc_update_supported(tc, NB, m, SP, C, ldc) &&
                        tc->ws_bytes >= tc_update_ws_bytes(n, m, batch);
    TcPreSplit cache{};
    if (cached) {
        cache.ld = SP;
        cache.part = static_cast<int64_t>(batch) * m * SP;
        cache.base = tc->ws + 3 * static_cast<int64_t>(batch) * n * SP;  // past the A parts (rows <= n, K <= SP)
    }
    auto split_rows = [&](int64_t k0, int64_t j0, int nb) {  // rows j0 .. j0+nb of C into cache columns j0 - k0 ..
        TcPreSplit d = cache;
        d.base += j0 - k0;
        return tc_split_into(TcOperand{C + j0 * ldc, m, 1, ldc, strideC}, nb, batch, d, s);
    };
    // C rows (Cd) -= A (M x K) times the K cached rows from cache column col0 on
    auto update_rhs = [&](const float* A, int64_t a_row, int64_t a_k, int64_t M, int64_t col0, int64_t row0, int K,
                          float* Cd) {
        if (cached && tc_update_supported(tc, M, m, K, Cd, ldc)) {
            TcPreSplit b = cache;
            b.base += col0;
            const TcOperand ao{A, M, a_row, a_k, strideG};
            const TcOperand bo{C + row0 * ldc, m, 1, ldc, strideC};
            return launch_tc_update(*tc, ao, &bo, K, Cd, ldc, strideC, -1.f, 1.f, false, batch, s, nullptr, &b);
        }
        return update(tc, A, a_row, a_k, strideG, M, C + row0 * ldc, 1, ldc, strideC, m, K, Cd, ldc, strideC, -1.f,
                      1.f, false, batch, s);
    };
    // forward, L Y = C, one super-block of rows at a time: each 64-row step takes
    // the earlier steps of its super-block, then its inverse diagonal block; then
    // one rank-(NSUB * 64) update of every row below.  B(k, n) = C[k][n]: row
    // stride 1, k stride ldc.
    for (int64_t k0 = 0; k0 < n; k0 += SP) {
        const int64_t kend = k0 + SP < n ? k0 + SP : n;
        for (int64_t j0 = k0; j0 < kend; j0 += NB) {
            const int nb = static_cast<int>(kend - j0 < NB ? kend - j0 : NB);
            if (j0 > k0) {
                e = update_rhs(L + j0 * ldg + k0, ldg, 1, nb, 0, k0, static_cast<int>(j0 - k0), C + j0 * ldc);
                if (e != cudaSuccess) return e;
            }
            if ((e = diag(j0, nb, false)) != cudaSuccess) return e;
            if (cached && (e = split_rows(k0, j0, nb)) != cudaSuccess) return e;
        }
        if (kend >= n) break;
        e = update_rhs(L + kend * ldg + k0, ldg, 1, n - kend, 0, k0, static_cast<int>(kend - k0), C + kend * ldc);
        if (e != cudaSuccess) return e;
    }
    // backward, L^T X = Y, last super-block first; inside it the last step first,
    // each step taking the later steps of the super-block; then one rank-(NSUB * 64)
    // update of every row above.  A(i, kk) = L[row0 + kk][col0 + i]: row stride 1,
    // k stride ldg.
    const int64_t last = ((n - 1) / SP) * SP;
    for (int64_t k0 = last; k0 >= 0; k0 -= SP) {
        const int64_t kend = k0 + SP < n ? k0 + SP : n;
        for (int64_t j0 = k0 + ((kend - 1 - k0) / NB) * NB; j0 >= k0; j0 -= NB) {
            const int nb = static_cast<int>(kend - j0 < NB ? kend - j0 : NB);
            if (j0 + nb < kend) {
                e = update_rhs(L + (j0 + nb) * ldg + j0, 1, ldg, nb, j0 + nb - k0, j0 + nb,
                               static_cast<int>(kend - j0 - nb), C + j0 * ldc);
                if (e != cudaSuccess) return e;
            }
            if ((e = diag(j0, nb, true)) != cudaSuccess) return e;
            if (cached && (e = split_rows(k0, j0, nb)) != cudaSuccess) return e;
        }
        if (k0 == 0) break;
        e = update_rhs(L + k0 * ldg, 1, ldg, k0, 0, k0, static_cast<int>(kend - k0), C);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace kvb

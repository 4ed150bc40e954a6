// Calibration statistics: stride gather, RoPE strip, batch means, centering,
// Chan merge coefficients, and the CUDA-core statistics GEMM.
//
// "KVBridge" README, "Loading": only centered sufficient statistics are kept,
// merged batch by batch with Chan/Welford updates:
//   n = n_a + n_b,  delta = mean_b - mean_a,  f = n_a n_b / n,
//   M <- M + M_b + f delta_x delta_x^T,  C <- C + C_b + f delta_x delta_y^T,
//   S_yy <- S_yy + S_yy,b + f delta_y^2,  mean <- mean_a + delta n_b / n.
// "Cross-Model KV Transfer" (VeloxQuant-MLX), "Configuration": deterministic
// token stride 4 (positions that are multiples of the stride are kept).
// Keys are stripped of RoPE with their own model's theta before any statistic.
#include "kvb_internal.h"
#include "stats_internal.h"

namespace kvb {

namespace {

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) {
    return v;
}
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}

// Retained token indices of one batch, in order; count -> *nb.  One CTA.
__global__ void __launch_bounds__(1024) select_rows_kernel(const int* __restrict__ pos, int64_t T, int stride,
                                                           int max_pos, int* __restrict__ rows,
                                                           int* __restrict__ nb, DevErr err) {
    __shared__ int warp_sums[32];
    __shared__ int base;
    if (threadIdx.x == 0) base = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int64_t c0 = 0; c0 < T; c0 += blockDim.x) {
        const int64_t i = c0 + threadIdx.x;
        int keep = 0;
        if (i < T) {
            const int p = pos[i];
            if (p < 0 || p >= max_pos) {
                dev_err_set(err, DEV_ERR_BAD_POS);
            } else {
                keep = (p % stride) == 0;
            }
        }
        const unsigned m = __ballot_sync(0xffffffffu, keep);
        const int before = __popc(m & ((1u << lane) - 1u));
        if (lane == 0) warp_sums[wid] = __popc(m);
        __syncthreads();
        if (wid == 0) {
            int v = lane < static_cast<int>(blockDim.x >> 5) ? warp_sums[lane] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            warp_sums[lane] = incl - v;  // exclusive
        }
        __syncthreads();
        if (keep) rows[base + warp_sums[wid] + before] = static_cast<int>(i);
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) base += warp_sums[wid] + before + keep;
        __syncthreads();
    }
    if (threadIdx.x == 0) *nb = base;
}

// Value of feature column e of one stored row, RoPE-stripped for keys.
template <typename T>
__device__ __forceinline__ float feature_value(const T* row, int e, int half, bool strip, const float2* tab_row) {
    const float x = to_f<T>(row[e]);
    if (!strip) return x;
    const int i = e < half ? e : e - half;
    const float2 cs = __ldg(tab_row + i);
    const float partner = to_f<T>(row[e < half ? e + half : e - half]);
    return e < half ? fmaf(x, cs.x, partner * cs.y) : fmaf(x, cs.x, -(partner * cs.y));
}

// Column means over the retained rows; one CTA per (layer, head) slab.
template <typename T>
__global__ void __launch_bounds__(256) colmean_kernel(const T* __restrict__ cache, int64_t T_len, int d,
                                                      const int* __restrict__ rows, const int* __restrict__ nb,
                                                      const int* __restrict__ pos, const float2* __restrict__ tab,
                                                      bool strip, float* __restrict__ mean) {
    __shared__ float part[256];
    const int slab = blockIdx.x;
    const int groups = blockDim.x / d;
    const int e = threadIdx.x % d;
    const int g = threadIdx.x / d;
    const int n = *nb;
    const int half = d >> 1;
    float s = 0.f;
    if (g < groups) {
        const T* base = cache + static_cast<int64_t>(slab) * T_len * d;
        for (int r = g; r < n; r += groups) {
            const int tok = rows[r];
            s += feature_value<T>(base + static_cast<int64_t>(tok) * d, e, half, strip,
                                  tab + static_cast<int64_t>(pos[tok]) * half);
        }
    }
    part[threadIdx.x] = s;
    __syncthreads();
    if (threadIdx.x < d) {
        float t = 0.f;
        for (int q = 0; q < groups; ++q) t += part[q * d + threadIdx.x];
        mean[static_cast<int64_t>(slab) * d + threadIdx.x] = n > 0 ? t / static_cast<float>(n) : 0.f;
    }
}

// Centered, transposed compaction: v = value(row r, f) - batch mean[f] for
// r < n_b, zero for n_b <= r < round_up(n_b, 64), stored at [f][r].  With
// out_lo == nullptr v is stored as float32; otherwise as the bf16 pair
// hi = bf16(v), lo = bf16(v - hi) (hi + lo carries ~16 significant bits), the
// operand form of the tensor-core statistics GEMM.  Grid (slab, 64-row chunk).
template <typename T>
__global__ void __launch_bounds__(256) center_transpose_kernel(const T* __restrict__ cache, int64_t T_len, int d,
                                                               const int* __restrict__ rows,
                                                               const int* __restrict__ nb,
                                                               const int* __restrict__ pos,
                                                               const float2* __restrict__ tab, bool strip,
                                                               const float* __restrict__ mean,
                                                               void* __restrict__ out, void* __restrict__ out_lo,
                                                               int64_t ld) {
    extern __shared__ float tile[];  // [64][d + 1]
    const int slab = blockIdx.x;
    const int r0 = blockIdx.y * 64;
    const int n = *nb;
    const int npad = (n + 63) & ~63;
    if (r0 >= npad) return;
    const int half = d >> 1;
    const int ldt = d + 1;
    const T* base = cache + static_cast<int64_t>(slab) * T_len * d;
    const float* mu = mean + static_cast<int64_t>(slab) * d;
    for (int i = threadIdx.x; i < 64 * d; i += blockDim.x) {
        const int rr = i / d;
        const int e = i - rr * d;
        const int r = r0 + rr;
        float v = 0.f;
        if (r < n) {
            const int tok = rows[r];
            v = feature_value<T>(base + static_cast<int64_t>(tok) * d, e, half, strip,
                                 tab + static_cast<int64_t>(pos[tok]) * half) -
                mu[e];
        }
        tile[rr * ldt + e] = v;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 64 * d; i += blockDim.x) {
        const int e = i / 64;
        const int rr = i - e * 64;
        const int64_t o = (static_cast<int64_t>(slab) * d + e) * ld + r0 + rr;
        const float v = tile[rr * ldt + e];
        if (out_lo == nullptr) {
            static_cast<float*>(out)[o] = v;
        } else {
            const __nv_bfloat16 hi = __float2bfloat16_rn(v);
            static_cast<__nv_bfloat16*>(out)[o] = hi;
            static_cast<__nv_bfloat16*>(out_lo)[o] = __float2bfloat16_rn(v - __bfloat162float(hi));
        }
    }
}

// ---------------------------------------------------------------------------
// Vectorised gather for bf16 caches with head_dim % 16 == 0: each lane owns 8
// contiguous dims of a row (one 16-byte load); the RoPE partner dims of the
// same row sit in lane ^ (d/16), fetched with a shuffle.  Each thread handles
// R rows per step with all their loads issued before any use, so R row loads,
// position loads and table loads are in flight at once.  Loops are
// warp-uniform so the shuffles always see the whole warp.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void unpack8(const uint4& v, float (&x)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(h[q]);
        x[2 * q] = f.x;
        x[2 * q + 1] = f.y;
    }
}

// Stripped (keys) or raw (values) features of 8 dims of R kept rows.
template <int R>
__device__ __forceinline__ void load_rows8(const __nv_bfloat16* __restrict__ slab_base, const bool (&valid)[R],
                                           const int (&tok)[R], int d, int sub, int pl,
                                           const int* __restrict__ pos, const float2* __restrict__ tab, bool strip,
                                           float (&y)[R][8]) {
    uint4 raw[R];
#pragma unroll
    for (int u = 0; u < R; ++u)
        raw[u] = valid[u] ? __ldg(reinterpret_cast<const uint4*>(slab_base + static_cast<int64_t>(tok[u]) * d + sub * 8))
                          : make_uint4(0, 0, 0, 0);
    if (!strip) {
#pragma unroll
        for (int u = 0; u < R; ++u) unpack8(raw[u], y[u]);
        return;
    }
    const int half = d >> 1;
    const bool lo = sub < pl;
    const int i0 = lo ? sub * 8 : sub * 8 - half;
    float4 cs[R][4];
#pragma unroll
    for (int u = 0; u < R; ++u) {
        const int p = valid[u] ? __ldg(pos + tok[u]) : 0;
        const float4* t4 = reinterpret_cast<const float4*>(tab + static_cast<int64_t>(p) * half + i0);
#pragma unroll
        for (int q = 0; q < 4; ++q) cs[u][q] = __ldg(t4 + q);
    }
#pragma unroll
    for (int u = 0; u < R; ++u) {
        uint4 pr;
        pr.x = __shfl_xor_sync(0xffffffffu, raw[u].x, pl);
        pr.y = __shfl_xor_sync(0xffffffffu, raw[u].y, pl);
        pr.z = __shfl_xor_sync(0xffffffffu, raw[u].z, pl);
        pr.w = __shfl_xor_sync(0xffffffffu, raw[u].w, pl);
        float x[8], p[8];
        unpack8(raw[u], x);
        unpack8(pr, p);
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // cs = (c, s) of two consecutive pairs
            const float s0 = lo ? cs[u][q].y : -cs[u][q].y, s1 = lo ? cs[u][q].w : -cs[u][q].w;
            y[u][2 * q] = fmaf(x[2 * q], cs[u][q].x, p[2 * q] * s0);
            y[u][2 * q + 1] = fmaf(x[2 * q + 1], cs[u][q].z, p[2 * q + 1] * s1);
        }
    }
}

constexpr int kRowsPerStep = 4;

// Partial column sums: part[split][slab*d + e] over the split's share of kept rows.
__global__ void __launch_bounds__(256) colsum_vec_kernel(const __nv_bfloat16* __restrict__ cache, int64_t T_len,
                                                         int d, const int* __restrict__ rows,
                                                         const int* __restrict__ nb, const int* __restrict__ pos,
                                                         const float2* __restrict__ tab, bool strip,
                                                         float* __restrict__ part, int64_t F) {
    __shared__ float red[256 * 8];
    const int slab = blockIdx.x, split = blockIdx.y, S = gridDim.y;
    const int lpr = d >> 3;           // lanes per row
    const int rpi = 256 / lpr;        // rows per row-slot sweep
    const int sub = threadIdx.x % lpr;
    const int rr = threadIdx.x / lpr;
    const int pl = d >> 4;
    const int n = *nb;
    const int chunk = (n + S - 1) / S;
    const int r0 = split * chunk, r1 = min(n, r0 + chunk);
    const __nv_bfloat16* base = cache + static_cast<int64_t>(slab) * T_len * d;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int b = r0; b < r1; b += rpi * kRowsPerStep) {
        bool valid[kRowsPerStep];
        int tok[kRowsPerStep];
#pragma unroll
        for (int u = 0; u < kRowsPerStep; ++u) {
            const int r = b + u * rpi + rr;
            valid[u] = r < r1;
            tok[u] = valid[u] ? __ldg(rows + r) : 0;
        }
        float y[kRowsPerStep][8];
        load_rows8<kRowsPerStep>(base, valid, tok, d, sub, pl, pos, tab, strip, y);
#pragma unroll
        for (int u = 0; u < kRowsPerStep; ++u)
            if (valid[u]) {
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] += y[u][i];
            }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) red[rr * d + sub * 8 + i] = acc[i];
    __syncthreads();
    for (int e = threadIdx.x; e < d; e += blockDim.x) {
        float s = 0.f;
        for (int q = 0; q < rpi; ++q) s += red[q * d + e];
        part[static_cast<int64_t>(split) * F + static_cast<int64_t>(slab) * d + e] = s;
    }
}

__global__ void mean_finalize_kernel(const float* __restrict__ part, int S, int64_t F, const int* __restrict__ nb,
                                     float* __restrict__ mean) {
    const int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (c >= F) return;
    const int n = *nb;
    float s = 0.f;
    for (int q = 0; q < S; ++q) s += part[q * F + c];
    mean[c] = n > 0 ? s / static_cast<float>(n) : 0.f;
}

// Centered, transposed compaction of 64 kept rows of one slab (see
// center_transpose_kernel), vectorised.  tile[e][r] in shared memory.
__global__ void __launch_bounds__(256) center_vec_kernel(const __nv_bfloat16* __restrict__ cache, int64_t T_len,
                                                         int d, const int* __restrict__ rows,
                                                         const int* __restrict__ nb, const int* __restrict__ pos,
                                                         const float2* __restrict__ tab, bool strip,
                                                         const float* __restrict__ mean, void* __restrict__ out,
                                                         void* __restrict__ out_lo, int64_t ld) {
    extern __shared__ float tile[];  // [d][65]
    const int slab = blockIdx.x;
    const int r0 = blockIdx.y * 64;
    const int n = *nb;
    if (r0 >= ((n + 63) & ~63)) return;
    const int lpr = d >> 3, rpi = 256 / lpr;
    const int sub = threadIdx.x % lpr, rq = threadIdx.x / lpr;
    const int pl = d >> 4;
    const __nv_bfloat16* base = cache + static_cast<int64_t>(slab) * T_len * d;
    float mu[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mu[i] = mean[static_cast<int64_t>(slab) * d + sub * 8 + i];
    for (int b = 0; b < 64; b += rpi * kRowsPerStep) {
        bool valid[kRowsPerStep];
        int tok[kRowsPerStep];
#pragma unroll
        for (int u = 0; u < kRowsPerStep; ++u) {
            const int rr = b + u * rpi + rq;
            valid[u] = rr < 64 && r0 + rr < n;
            tok[u] = valid[u] ? __ldg(rows + r0 + rr) : 0;
        }
        float y[kRowsPerStep][8];
        load_rows8<kRowsPerStep>(base, valid, tok, d, sub, pl, pos, tab, strip, y);
#pragma unroll
        for (int u = 0; u < kRowsPerStep; ++u) {
            const int rr = b + u * rpi + rq;
            if (rr < 64) {
#pragma unroll
                for (int i = 0; i < 8; ++i) tile[(sub * 8 + i) * 65 + rr] = valid[u] ? y[u][i] - mu[i] : 0.f;
            }
        }
    }
    __syncthreads();
    const int64_t row0 = static_cast<int64_t>(slab) * d;
    if (out_lo == nullptr) {
        for (int idx = threadIdx.x; idx < d * 16; idx += blockDim.x) {
            const int e = idx >> 4, q = idx & 15;
            const float* t = tile + e * 65 + 4 * q;
            *reinterpret_cast<float4*>(static_cast<float*>(out) + (row0 + e) * ld + r0 + 4 * q) =
                make_float4(t[0], t[1], t[2], t[3]);
        }
    } else {
        for (int idx = threadIdx.x; idx < d * 8; idx += blockDim.x) {
            const int e = idx >> 3, q = idx & 7;
            const float* t = tile + e * 65 + 8 * q;
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __nv_bfloat16 h0 = __float2bfloat16_rn(t[2 * j]), h1 = __float2bfloat16_rn(t[2 * j + 1]);
                const float l0 = t[2 * j] - __bfloat162float(h0), l1 = t[2 * j + 1] - __bfloat162float(h1);
                __nv_bfloat162 hh(h0, h1);
                hi[j] = *reinterpret_cast<uint32_t*>(&hh);
                lo[j] = pack_bf16x2(l0, l1);
            }
            const int64_t o = (row0 + e) * ld + r0 + 8 * q;
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out_lo) + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
    }
}

// delta = batch mean - running mean (before the merge); running mean updated;
// f = n_a n_b / (n_a + n_b).  Thread per column over the four mean vectors.
__global__ void chan_prepare_kernel(MeanSet ms, const long long* __restrict__ n_dev, const int* __restrict__ nb,
                                    float* __restrict__ f_out) {
    const long long na = *n_dev;
    const int n_b = *nb;
    const double n = static_cast<double>(na) + n_b;
    const float wb = n > 0 ? static_cast<float>(n_b / n) : 0.f;
    if (blockIdx.x == 0 && threadIdx.x == 0) *f_out = n > 0 ? static_cast<float>(static_cast<double>(na) * n_b / n) : 0.f;
    for (int m = 0; m < 4; ++m) {
        for (int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; c < ms.len[m];
             c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
            const float dl = n_b > 0 ? ms.bmean[m][c] - ms.mean[m][c] : 0.f;
            ms.delta[m][c] = dl;
            ms.mean[m][c] += dl * wb;
        }
    }
}

__global__ void chan_finish_kernel(long long* __restrict__ n_dev, const int* __restrict__ nb) {
    *n_dev += *nb;
}

// S_yy[j] += sum_r Y[j][r]^2 + f delta_y[j]^2.  One warp per target column.
// Y is float32, or a (hi, lo) bf16 pair when lo != nullptr.
__global__ void syy_kernel(const void* __restrict__ Y, const void* __restrict__ Ylo, int64_t ld, int64_t rows_n,
                           const int* __restrict__ nb, const float* __restrict__ dy, const float* __restrict__ f,
                           float* __restrict__ syy) {
    const int64_t j = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (j >= rows_n) return;
    const int n = *nb;
    float s = 0.f;
    for (int r = lane; r < n; r += 32) {
        float v;
        if (Ylo == nullptr)
            v = static_cast<const float*>(Y)[j * ld + r];
        else
            v = __bfloat162float(static_cast<const __nv_bfloat16*>(Y)[j * ld + r]) +
                __bfloat162float(static_cast<const __nv_bfloat16*>(Ylo)[j * ld + r]);
        s = fmaf(v, v, s);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) syy[j] += s + (*f) * dy[j] * dy[j];
}

// out[i][j] += sum_r A[i][r] B[j][r] + f da[i] db[j] over K = round_up(n_b, 64)
// (padding columns are zero).  64x64 tile, 256 threads, 4x4 per thread.
// With lower != 0, tiles entirely above the diagonal are skipped.
__global__ void __launch_bounds__(256) stats_gemm_simt_kernel(const float* __restrict__ A, const float* __restrict__ B,
                                                              int64_t ld, int64_t Ma, int64_t Nb, int lower,
                                                              const float* __restrict__ da,
                                                              const float* __restrict__ db,
                                                              const float* __restrict__ f,
                                                              const int* __restrict__ nb, float* __restrict__ out,
                                                              int64_t ldo) {
    constexpr int BT = 64, BKK = 16;
    __shared__ float As[BKK][BT + 4];
    __shared__ float Bs[BKK][BT + 4];
    const int64_t i0 = static_cast<int64_t>(blockIdx.y) * BT;
    const int64_t j0 = static_cast<int64_t>(blockIdx.x) * BT;
    if (lower && j0 > i0 + BT - 1) return;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    const int K = (*nb + 63) & ~63;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += BKK) {
        for (int q = threadIdx.x; q < BT * BKK; q += 256) {
            const int r = q / BKK, kk = q % BKK;
            As[kk][r] = (i0 + r < Ma) ? A[(i0 + r) * ld + k0 + kk] : 0.f;
            Bs[kk][r] = (j0 + r < Nb) ? B[(j0 + r) * ld + k0 + kk] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BKK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) a[x] = As[kk][ty * 4 + x];
#pragma unroll
            for (int y = 0; y < 4; ++y) b[y] = Bs[kk][tx * 4 + y];
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(a[x], b[y], acc[x][y]);
        }
        __syncthreads();
    }
    const float ff = *f;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        const int64_t i = i0 + ty * 4 + x;
        if (i >= Ma) continue;
        const float fa = ff * da[i];
#pragma unroll
        for (int y = 0; y < 4; ++y) {
            const int64_t j = j0 + tx * 4 + y;
            if (j >= Nb) continue;
            out[i * ldo + j] += acc[x][y] + fa * db[j];
        }
    }
}

// dst[i][j] = src[max(i,j)][min(i,j)]: the full symmetric Gram from its lower triangle.
__global__ void symmetrize_kernel(const float* __restrict__ src, float* __restrict__ dst, int64_t n) {
    const int64_t i = blockIdx.y * static_cast<int64_t>(blockDim.y) + threadIdx.y;
    const int64_t j = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (i >= n || j >= n) return;
    dst[i * n + j] = i >= j ? src[i * n + j] : src[j * n + i];
}

}  // namespace

cudaError_t launch_symmetrize(const float* src, float* dst, int64_t n, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    dim3 blk(32, 8);
    dim3 grid(static_cast<unsigned>((n + 31) / 32), static_cast<unsigned>((n + 7) / 8));
    symmetrize_kernel<<<grid, blk, 0, s>>>(src, dst, n);
    return cudaGetLastError();
}

cudaError_t launch_select_rows(const int* pos, int64_t T, int stride, int max_pos, int* rows, int* nb, DevErr err,
                               cudaStream_t s) {
    select_rows_kernel<<<1, 1024, 0, s>>>(pos, T, stride, max_pos, rows, nb, err);
    return cudaGetLastError();
}

constexpr int kMeanSplits = 8;

bool gather_vec_ok(kvb_dtype dt, int d) { return dt == KVB_BF16 && d % 16 == 0 && d <= 256; }

cudaError_t launch_colmean(kvb_dtype dt, const void* cache, int64_t n_slabs, int64_t T, int d, const int* rows,
                           const int* nb, const int* pos, const float2* tab, bool strip, float* mean, float* part,
                           cudaStream_t s) {
    if (n_slabs == 0) return cudaSuccess;
    if (gather_vec_ok(dt, d) && part != nullptr) {
        const int64_t F = n_slabs * d;
        colsum_vec_kernel<<<dim3(static_cast<unsigned>(n_slabs), kMeanSplits), 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(cache), T, d, rows, nb, pos, tab, strip, part, F);
        mean_finalize_kernel<<<static_cast<unsigned>((F + 255) / 256), 256, 0, s>>>(part, kMeanSplits, F, nb, mean);
    } else if (dt == KVB_F32) {
        colmean_kernel<float><<<static_cast<unsigned>(n_slabs), 256, 0, s>>>(
            static_cast<const float*>(cache), T, d, rows, nb, pos, tab, strip, mean);
    } else {
        colmean_kernel<__nv_bfloat16><<<static_cast<unsigned>(n_slabs), 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(cache), T, d, rows, nb, pos, tab, strip, mean);
    }
    return cudaGetLastError();
}

cudaError_t launch_center_transpose(kvb_dtype dt, const void* cache, int64_t n_slabs, int64_t T, int d,
                                    const int* rows, const int* nb, const int* pos, const float2* tab, bool strip,
                                    const float* mean, void* out, void* out_lo, int64_t ld, cudaStream_t s) {
    if (n_slabs == 0) return cudaSuccess;
    dim3 grid(static_cast<unsigned>(n_slabs), static_cast<unsigned>((T + 63) / 64));
    if (gather_vec_ok(dt, d)) {
        const size_t vsmem = static_cast<size_t>(d) * 65 * sizeof(float);
        cudaFuncSetAttribute(center_vec_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 80 * 1024);
        center_vec_kernel<<<grid, 256, vsmem, s>>>(static_cast<const __nv_bfloat16*>(cache), T, d, rows, nb, pos, tab,
                                                   strip, mean, out, out_lo, ld);
        return cudaGetLastError();
    }
    const size_t smem = 64 * (d + 1) * sizeof(float);
    if (dt == KVB_F32) {
        cudaFuncSetAttribute(center_transpose_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, 80 * 1024);
        center_transpose_kernel<float><<<grid, 256, smem, s>>>(static_cast<const float*>(cache), T, d, rows, nb, pos,
                                                               tab, strip, mean, out, out_lo, ld);
    } else {
        cudaFuncSetAttribute(center_transpose_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             80 * 1024);
        center_transpose_kernel<__nv_bfloat16><<<grid, 256, smem, s>>>(static_cast<const __nv_bfloat16*>(cache), T, d,
                                                                       rows, nb, pos, tab, strip, mean, out, out_lo,
                                                                       ld);
    }
    return cudaGetLastError();
}

cudaError_t launch_chan_prepare(const MeanSet& ms, const long long* n_dev, const int* nb, float* f,
                                cudaStream_t s) {
    chan_prepare_kernel<<<256, 256, 0, s>>>(ms, n_dev, nb, f);
    return cudaGetLastError();
}

cudaError_t launch_chan_finish(long long* n_dev, const int* nb, cudaStream_t s) {
    chan_finish_kernel<<<1, 1, 0, s>>>(n_dev, nb);
    return cudaGetLastError();
}

cudaError_t launch_syy(const void* Y, const void* Ylo, int64_t ld, int64_t rows_n, const int* nb, const float* dy,
                       const float* f, float* syy, cudaStream_t s) {
    const int64_t threads = rows_n * 32;
    const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
    if (blocks == 0) return cudaSuccess;
    syy_kernel<<<blocks, 256, 0, s>>>(Y, Ylo, ld, rows_n, nb, dy, f, syy);
    return cudaGetLastError();
}

cudaError_t launch_stats_gemm_simt(const float* A, const float* B, int64_t ld, int64_t Ma, int64_t Nb, bool lower,
                                   const float* da, const float* db, const float* f, const int* nb, float* out,
                                   int64_t ldo, cudaStream_t s) {
    dim3 grid(static_cast<unsigned>((Nb + 63) / 64), static_cast<unsigned>((Ma + 63) / 64));
    if (grid.x == 0 || grid.y == 0) return cudaSuccess;
    stats_gemm_simt_kernel<<<grid, 256, 0, s>>>(A, B, ld, Ma, Nb, lower ? 1 : 0, da, db, f, nb, out, ldo);
    return cudaGetLastError();
}

}  // namespace kvb

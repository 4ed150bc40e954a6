// Calibration statistics: stride gather, RoPE strip, shifted centering, Chan
// merge coefficients, and the CUDA-core statistics GEMM.
//
// "KVBridge" README, "Loading": only centered sufficient statistics are kept,
// merged batch by batch with Chan/Welford updates.  With a per-column shift s
// (any value known before the pass) and z = x - s over the n_b kept rows of a
// batch, zbar = mean(z), the batch mean is s + zbar and
//   n = n_a + n_b,  delta = (s + zbar) - mean_a,  f = n_a n_b / n,
//   M <- M + Z^T Z - n_b zbar zbar^T + f delta delta^T        (same for C, S_yy)
//   mean <- mean_a + delta n_b / n.
// Z^T Z - n_b zbar zbar^T is the batch's centered Gram exactly; with s near the
// batch mean (the running mean, or the batch's first kept row for the first
// batch) the subtraction is tiny, so no cancellation from large raw moments.
// The generic path centers on the batch mean itself (s = batch mean, zbar = 0).
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

// ---------------------------------------------------------------------------
// Generic path (any even head_dim, fp32 or bf16 caches): two passes, the
// batch means first, then centering on them.
// ---------------------------------------------------------------------------

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

// Centered, transposed compaction: z = value(row r, f) - mean[f] for r < n_b,
// zero for n_b <= r < round_up(n_b, 64), stored at [f][r].  With out_lo ==
// nullptr z is stored as float32; otherwise as the bf16 pair hi = bf16(z),
// lo = bf16(z - hi) (hi + lo carries ~16 significant bits), the operand form
// of the tensor-core statistics GEMM.  Grid (slab, 64-row chunk).
template <typename T>
__global__ void __launch_bounds__(256) center_transpose_kernel(const T* __restrict__ cache, int64_t T_len, int d,
                                                               const int* __restrict__ rows,
                                                               const int* __restrict__ nb,
                                                               const int* __restrict__ pos,
                                                               const float2* __restrict__ tab, bool strip,
                                                               const float* __restrict__ mean,
                                                               void* __restrict__ out, void* __restrict__ out_lo,
                                                               void* __restrict__ out_3, int64_t ld) {
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
        } else if (out_3 == nullptr) {
            const __nv_bfloat16 hi = __float2bfloat16_rn(v);
            static_cast<__nv_bfloat16*>(out)[o] = hi;
            static_cast<__nv_bfloat16*>(out_lo)[o] = __float2bfloat16_rn(v - __bfloat162float(hi));
        } else {  // three parts: x1 = bf16(v), x2 = bf16(v - x1), x3 = bf16(v - x1 - x2)
            const __nv_bfloat16 x1 = __float2bfloat16_rn(v);
            const float e1 = v - __bfloat162float(x1);
            const __nv_bfloat16 x2 = __float2bfloat16_rn(e1);
            static_cast<__nv_bfloat16*>(out)[o] = x1;
            static_cast<__nv_bfloat16*>(out_lo)[o] = x2;
            static_cast<__nv_bfloat16*>(out_3)[o] = __float2bfloat16_rn(e1 - __bfloat162float(x2));
        }
    }
}

// ---------------------------------------------------------------------------
// Single-pass path for bf16 caches with head_dim % 16 == 0.  Each lane owns 8
// RoPE pairs of a row: 8 dims of the low half and the 8 partner dims of the
// high half (two 16-byte loads, one 64-byte cos/sin load), the layout of the
// strip pass.  The shift s is known before the pass: the running mean, or for
// the first batch the first kept row of the batch.  One read of every kept row.
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

constexpr int kChunk = 128;  // kept rows per CTA of the single-pass gather

// Grid (chunk group, slab), 256 threads; a CTA takes chunks blockIdx.x,
// blockIdx.x + gridDim.x, ... of its slab (the host sizes gridDim.x from
// T / stride, so few CTAs find no kept rows).  Each thread owns R rows of its
// lane column (R = 128 / rows-per-sweep) and issues all their loads before any use.
// Writes z = feature - s transposed ([f][r], float32 or bf16 hi/lo), the
// chunk's column sums of z to part[chunk][slab*d + e], and (chunk 0) the shift.
template <int R>
__global__ void __launch_bounds__(256, (R <= 4 ? 2 : 1)) gather_shift_kernel(const __nv_bfloat16* __restrict__ cache, int64_t T_len,
                                                           int d, const int* __restrict__ rows,
                                                           const int* __restrict__ nb,
                                                           const long long* __restrict__ n_seen,
                                                           const int* __restrict__ pos,
                                                           const float2* __restrict__ tab, bool strip,
                                                           const float* __restrict__ mean_a,
                                                           float* __restrict__ shift_out, float* __restrict__ part,
                                                           int64_t F, void* __restrict__ out,
                                                           void* __restrict__ out_lo, int64_t ld) {
    extern __shared__ float tile[];  // [d][kChunk + 1] then [8 warps][d] partial sums
    constexpr int LT = kChunk + 1;
    const int slab = blockIdx.y;  // chunks of one slab run side by side: contiguous reads and writes
    const int n = *nb;
    if (static_cast<int>(blockIdx.x) * kChunk >= n) return;
    const int half = d >> 1;
    const int lpr = d >> 4;          // lanes per row (8 pairs each)
    const int rps = 256 / lpr;       // rows per sweep
    const int l = threadIdx.x % lpr;
    const int rq = threadIdx.x / lpr;
    const __nv_bfloat16* base = cache + static_cast<int64_t>(slab) * T_len * d;
    const int64_t f0 = static_cast<int64_t>(slab) * d;

    float slo[8], shi[8];  // shift: the running mean (on the first batch, the batch mean)
    (void)n_seen;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        slo[i] = mean_a[f0 + 8 * l + i];
        shi[i] = mean_a[f0 + half + 8 * l + i];
    }
    if (blockIdx.x == 0 && rq == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            shift_out[f0 + 8 * l + i] = slo[i];
            shift_out[f0 + half + 8 * l + i] = shi[i];
        }
    }

#pragma unroll 1
    for (int chunk = blockIdx.x; chunk * kChunk < n; chunk += gridDim.x) {
    const int r0 = chunk * kChunk;
    // issue every load of this thread's rows first
    uint4 ra[R], rb[R];
    float4 cs[R][4];
    bool valid[R];
#pragma unroll
    for (int u = 0; u < R; ++u) {
        const int rr = rq + u * rps;
        const int r = r0 + rr;
        valid[u] = rr < kChunk && r < n;
        const int tok = valid[u] ? __ldg(rows + r) : 0;
        const __nv_bfloat16* row = base + static_cast<int64_t>(tok) * d;
        ra[u] = valid[u] ? __ldg(reinterpret_cast<const uint4*>(row + 8 * l)) : make_uint4(0, 0, 0, 0);
        rb[u] = valid[u] ? __ldg(reinterpret_cast<const uint4*>(row + half + 8 * l)) : make_uint4(0, 0, 0, 0);
        if (strip) {
            const int p = valid[u] ? __ldg(pos + tok) : 0;
            const float4* t4 = reinterpret_cast<const float4*>(tab + static_cast<int64_t>(p) * half + 8 * l);
#pragma unroll
            for (int q = 0; q < 4; ++q) cs[u][q] = __ldg(t4 + q);
        }
    }

    float alo[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, ahi[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < R; ++u) {
        const int rr = rq + u * rps;
        if (rr >= kChunk) continue;
        float x[8], y[8], zl[8], zh[8];
        unpack8(ra[u], x);
        unpack8(rb[u], y);
        if (strip) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                zl[2 * q] = fmaf(x[2 * q], cs[u][q].x, y[2 * q] * cs[u][q].y);
                zh[2 * q] = fmaf(y[2 * q], cs[u][q].x, -(x[2 * q] * cs[u][q].y));
                zl[2 * q + 1] = fmaf(x[2 * q + 1], cs[u][q].z, y[2 * q + 1] * cs[u][q].w);
                zh[2 * q + 1] = fmaf(y[2 * q + 1], cs[u][q].z, -(x[2 * q + 1] * cs[u][q].w));
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                zl[i] = x[i];
                zh[i] = y[i];
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            zl[i] = valid[u] ? zl[i] - slo[i] : 0.f;
            zh[i] = valid[u] ? zh[i] - shi[i] : 0.f;
            alo[i] += zl[i];
            ahi[i] += zh[i];
            tile[(8 * l + i) * LT + rr] = zl[i];
            tile[(half + 8 * l + i) * LT + rr] = zh[i];
        }
    }
    // column sums: across the warp's rows by shuffles, then across the 8 warps
    float* red = tile + d * LT;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        for (int o = lpr; o < 32; o <<= 1) {
            alo[i] += __shfl_xor_sync(0xffffffffu, alo[i], o);
            ahi[i] += __shfl_xor_sync(0xffffffffu, ahi[i], o);
        }
    }
    const int wq = threadIdx.x >> 5;
    if ((threadIdx.x & 31) < lpr) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            red[wq * d + 8 * l + i] = alo[i];
            red[wq * d + half + 8 * l + i] = ahi[i];
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < d; e += blockDim.x) {
        float s = 0.f;
        for (int q = 0; q < 8; ++q) s += red[q * d + e];
        part[static_cast<int64_t>(chunk) * F + f0 + e] = s;
    }
    if (out_lo == nullptr) {
        for (int idx = threadIdx.x; idx < d * (kChunk / 4); idx += blockDim.x) {
            const int e = idx / (kChunk / 4), q = idx % (kChunk / 4);
            const float* t = tile + e * LT + 4 * q;
            *reinterpret_cast<float4*>(static_cast<float*>(out) + (f0 + e) * ld + r0 + 4 * q) =
                make_float4(t[0], t[1], t[2], t[3]);
        }
    } else {
        for (int idx = threadIdx.x; idx < d * (kChunk / 8); idx += blockDim.x) {
            const int e = idx / (kChunk / 8), q = idx % (kChunk / 8);
            const float* t = tile + e * LT + 8 * q;
            uint32_t h[4], lw[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __nv_bfloat16 h0 = __float2bfloat16_rn(t[2 * j]), h1 = __float2bfloat16_rn(t[2 * j + 1]);
                const float l0 = t[2 * j] - __bfloat162float(h0), l1 = t[2 * j + 1] - __bfloat162float(h1);
                __nv_bfloat162 hh(h0, h1);
                h[j] = *reinterpret_cast<uint32_t*>(&hh);
                lw[j] = pack_bf16x2(l0, l1);
            }
            const int64_t o = (f0 + e) * ld + r0 + 8 * q;
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + o) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out_lo) + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
    }
    __syncthreads();  // the tile and the sums are reused by the next chunk
    }
}

// Streaming variant of the single-pass gather (head_dim 64 or 128).  One CTA
// per SM; the (128-row chunk, slab) work items are split into one contiguous
// range per CTA, so a CTA walks a run of slabs of one chunk (or two).  Per chunk the kept-row indices, positions and (for
// keys) the chunk's RoPE table rows are staged in shared memory once; per
// slab the raw rows are copied in with cp.async, kStages - 1 slabs ahead of
// the one being processed.  Thread (pair i, row group q) strips pair
// (i, i + d/2) of rows 16q .. 16q + 15 straight from shared memory, keeps its
// centered values in registers, writes them as bf16 (hi, lo) runs of its
// observations into the feature-major outputs and sums them per column: no
// transpose through shared memory.
constexpr int kStages = 4;

__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}


// Threads of the streaming gather: every thread keeps 16 rows of one RoPE pair.
__host__ __device__ constexpr int stream_threads(int d) { return kChunk * (d / 2) / 16; }

size_t gather_stream_smem(int d) {
    return static_cast<size_t>(kStages) * kChunk * d * 2   // raw rows
           + static_cast<size_t>(kStages) * d * 4          // running means of the staged slabs
           + static_cast<size_t>(kChunk) * (d / 2) * 8     // RoPE table rows of the chunk
           + 2 * static_cast<size_t>(stream_threads(d) / (d / 2)) * d * 4  // per-row-group column sums, two slabs
           + 2 * kChunk * 4;                               // row indices, positions
}

template <int D>
__global__ void __launch_bounds__(stream_threads(D), 1) gather_stream_kernel(const __nv_bfloat16* __restrict__ cache, int64_t T_len,
                                                               const int* __restrict__ rows,
                                                               const int* __restrict__ nb,
                                                               const long long* __restrict__ n_seen,
                                                               const int* __restrict__ pos,
                                                               const float2* __restrict__ tab, bool strip,
                                                               const float* __restrict__ mean_a,
                                                               float* __restrict__ shift_out, float* __restrict__ part,
                                                               int64_t F, __nv_bfloat16* __restrict__ out,
                                                               __nv_bfloat16* __restrict__ out_lo, int64_t ld,
                                                               int n_slabs) {
    constexpr int HALF = D / 2;
    constexpr int QN = stream_threads(D) / HALF;  // row groups
    constexpr int ROWS = kChunk / QN;             // rows per thread (16)
    static_assert(ROWS % 16 == 0, "whole 32-byte output runs per thread");
    constexpr int PIECES = kChunk * (D / 8);
    extern __shared__ __align__(16) uint8_t gsm[];
    __nv_bfloat16* stg = reinterpret_cast<__nv_bfloat16*>(gsm);
    float* smean = reinterpret_cast<float*>(gsm + static_cast<size_t>(kStages) * kChunk * D * 2);
    float2* stab = reinterpret_cast<float2*>(smean + kStages * D);
    float* red = reinterpret_cast<float*>(stab + kChunk * HALF);
    int* srow = reinterpret_cast<int*>(red + 2 * QN * D);
    int* spos = srow + kChunk;
    const int n = *nb;
    const int i = threadIdx.x % HALF;  // RoPE pair (i, i + D/2)
    const int q = threadIdx.x / HALF;  // rows q*ROWS .. q*ROWS + ROWS - 1 of the chunk
    (void)n_seen;  // shift: the running mean (on the first batch, the batch mean)

    // work items (chunk, slab) in chunk-major order; CTA b takes one contiguous
    // range of them, i.e. runs of slabs within one or two chunks
    const int nchunks = (n + kChunk - 1) / kChunk;
    const int64_t items = static_cast<int64_t>(nchunks) * n_slabs;
    const int64_t per = (items + gridDim.x - 1) / gridDim.x;
    int64_t it0 = blockIdx.x * per;
    const int64_t it1 = it0 + per < items ? it0 + per : items;
#pragma unroll 1
    while (it0 < it1) {
        const int chunk = static_cast<int>(it0 / n_slabs);
        const int s_begin = static_cast<int>(it0 % n_slabs);
        const int mine = static_cast<int>(n_slabs - s_begin < it1 - it0 ? n_slabs - s_begin : it1 - it0);
        it0 += mine;
        const int r0 = chunk * kChunk;
        __syncthreads();  // the previous chunk is done with srow / spos / stab
        for (int t = threadIdx.x; t < kChunk; t += blockDim.x) {
            const int r = r0 + t;
            const int tok = r < n ? __ldg(rows + r) : -1;
            srow[t] = tok;
            spos[t] = tok >= 0 ? __ldg(pos + tok) : 0;
        }
        __syncthreads();
        if (strip) {  // the chunk's table rows ride in the first copy group
            for (int pc = threadIdx.x; pc < kChunk * (HALF / 2); pc += blockDim.x) {
                const int rr = pc / (HALF / 2), c2 = (pc % (HALF / 2)) * 2;
                cp_async16(stab + rr * HALF + c2, tab + static_cast<int64_t>(spos[rr]) * HALF + c2, 16);
            }
        }
        auto issue = [&](int j) {  // raw rows (and running means) of this CTA's j-th slab into stage j % kStages
            const int slab = s_begin + j;
            const __nv_bfloat16* base = cache + static_cast<int64_t>(slab) * T_len * D;
            __nv_bfloat16* dst = stg + static_cast<size_t>(j % kStages) * kChunk * D;
            if (threadIdx.x < D / 4)
                cp_async16(smean + (j % kStages) * D + 4 * threadIdx.x, mean_a + static_cast<int64_t>(slab) * D +
                           4 * threadIdx.x, 16);
            for (int pc = threadIdx.x; pc < PIECES; pc += blockDim.x) {
                const int rr = pc / (D / 8), c8 = (pc % (D / 8)) * 8;
                const int tok = srow[rr];
                cp_async16(dst + rr * D + c8, tok >= 0 ? base + static_cast<int64_t>(tok) * D + c8 : cache,
                           tok >= 0 ? 16 : 0);
            }
        };
#pragma unroll
        for (int j = 0; j < kStages - 1; ++j) {
            if (j < mine) issue(j);
            cp_async_commit();
        }
        // column sums of slab j-1 (staged in red[(j-1) & 1]) written by the first D threads
        auto flush_sums = [&](int jj) {
            const int64_t fp = static_cast<int64_t>(s_begin + jj) * D;
            const float* rs = red + (jj & 1) * QN * D;
            for (int e = threadIdx.x; e < D; e += blockDim.x) {
                float sm = 0.f;
#pragma unroll
                for (int g = 0; g < QN; ++g) sm += rs[g * D + e];
                part[static_cast<int64_t>(chunk) * F + fp + e] = sm;
            }
        };
#pragma unroll 1
        for (int j = 0; j < mine; ++j) {
            cp_async_wait<kStages - 2>();
            // every thread's copies of slab j (and the table) have landed, and every
            // thread is done with slab j - 1: its stage can be refilled
            __syncthreads();
            if (j > 0) flush_sums(j - 1);
            if (j + kStages - 1 < mine) issue(j + kStages - 1);
            cp_async_commit();

            const int slab = s_begin + j;
            const int64_t f0 = static_cast<int64_t>(slab) * D;
            const __nv_bfloat16* raw = stg + static_cast<size_t>(j % kStages) * kChunk * D;
            const float sl = smean[(j % kStages) * D + i];  // shift of features i and i + D/2
            const float sh = smean[(j % kStages) * D + HALF + i];
            if (chunk == 0 && q == 0) {
                shift_out[f0 + i] = sl;
                shift_out[f0 + HALF + i] = sh;
            }
            float zl[ROWS], zh[ROWS];
            float al = 0.f, ah = 0.f;
#pragma unroll
            for (int u = 0; u < ROWS; ++u) {
                const int rr = q * ROWS + u;
                const float x = __bfloat162float(raw[rr * D + i]);
                const float y = __bfloat162float(raw[rr * D + HALF + i]);
                float a = x, b = y;
                if (strip) {
                    const float2 cs = stab[rr * HALF + i];
                    a = fmaf(x, cs.x, y * cs.y);
                    b = fmaf(y, cs.x, -(x * cs.y));
                }
                const bool valid = srow[rr] >= 0;
                zl[u] = valid ? a - sl : 0.f;
                zh[u] = valid ? b - sh : 0.f;
                al += zl[u];
                ah += zh[u];
            }
            // feature-major outputs: ROWS consecutive observations per feature
            const int64_t ol = (f0 + i) * ld + r0 + q * ROWS;
            const int64_t oh = (f0 + HALF + i) * ld + r0 + q * ROWS;
            // 16 observations (32 bytes, one sector) per store
#pragma unroll
            for (int v = 0; v < ROWS / 16; ++v) {
                uint32_t hl[8], ll[8], hh[8], lh[8];
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    const int u = 16 * v + 2 * w;
                    const __nv_bfloat162 b0 = __floats2bfloat162_rn(zl[u], zl[u + 1]);
                    const float2 f0v = __bfloat1622float2(b0);
                    hl[w] = *reinterpret_cast<const uint32_t*>(&b0);
                    ll[w] = pack_bf16x2(zl[u] - f0v.x, zl[u + 1] - f0v.y);
                    const __nv_bfloat162 b1 = __floats2bfloat162_rn(zh[u], zh[u + 1]);
                    const float2 f1v = __bfloat1622float2(b1);
                    hh[w] = *reinterpret_cast<const uint32_t*>(&b1);
                    lh[w] = pack_bf16x2(zh[u] - f1v.x, zh[u + 1] - f1v.y);
                }
                st_global_v8(out + ol + 16 * v, hl);
                st_global_v8(out_lo + ol + 16 * v, ll);
                st_global_v8(out + oh + 16 * v, hh);
                st_global_v8(out_lo + oh + 16 * v, lh);
            }
            red[(j & 1) * QN * D + q * D + i] = al;
            red[(j & 1) * QN * D + q * D + HALF + i] = ah;
        }
        cp_async_wait<0>();
        __syncthreads();
        if (mine > 0) flush_sums(mine - 1);
    }
}

// First batch of a fit (nothing merged yet): the column means of the batch's
// first 128 kept rows (keys stripped) become the running means before the
// single-pass gather, which shifts every value by the running mean.  Later
// batches return at once.  A shift near the batch mean (within ~sigma / 11
// here) keeps every centered sum near its final size; a shift far from it (one
// row, say) leaves sums of order n * shift^2 that cancel in the merge and cost
// the fp32 accumulation its precision.  Grid (slab, matrix), 256 threads:
// thread (pair i, row group g) sums rows g, g + G, ... of its slab.
constexpr int kFirstRows = 128;

__global__ void __launch_bounds__(256) first_mean_kernel(FirstMeanArgs a) {
    if (*a.n_seen != 0) return;
    const int n = *a.nb < kFirstRows ? *a.nb : kFirstRows;
    const int m = blockIdx.y;
    const int64_t slab = blockIdx.x;
    if (n == 0 || slab >= a.n_slabs[m]) return;
    const int half = a.d >> 1;
    const int G = 256 / half;
    const int i = threadIdx.x % half, g = threadIdx.x / half;
    const __nv_bfloat16* base = a.cache[m] + slab * a.T * a.d;
    const float2* tab = a.tab[m];
    float sa = 0.f, sb = 0.f;
    if (g < G) {
        for (int r = g; r < n; r += G) {
            const int tok = __ldg(a.rows + r);
            const __nv_bfloat16* row = base + static_cast<int64_t>(tok) * a.d;
            const float x = __bfloat162float(row[i]), y = __bfloat162float(row[half + i]);
            if (tab) {
                const float2 cs = __ldg(tab + static_cast<int64_t>(__ldg(a.pos + tok)) * half + i);
                sa += fmaf(x, cs.x, y * cs.y);
                sb += fmaf(y, cs.x, -(x * cs.y));
            } else {
                sa += x;
                sb += y;
            }
        }
    }
    __shared__ float red[2][256];
    red[0][threadIdx.x] = sa;
    red[1][threadIdx.x] = sb;
    __syncthreads();
    if (threadIdx.x < half) {
        float ta = 0.f, tb = 0.f;
        for (int k = 0; k < G; ++k) {
            ta += red[0][k * half + threadIdx.x];
            tb += red[1][k * half + threadIdx.x];
        }
        a.mean[m][slab * a.d + threadIdx.x] = ta / static_cast<float>(n);
        a.mean[m][slab * a.d + half + threadIdx.x] = tb / static_cast<float>(n);
    }
}

// zsum[c] = sum over the batch's chunks of part[chunk][c].
__global__ void zsum_kernel(const float* __restrict__ part, int64_t F, const int* __restrict__ nb,
                            float* __restrict__ zsum) {
    const int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (c >= F) return;
    const int chunks = (*nb + kChunk - 1) / kChunk;
    float s = 0.f;
    for (int q = 0; q < chunks; ++q) s += part[q * F + c];
    zsum[c] = s;
}

// Per column of the four matrices: zbar, delta against the running mean, the
// running-mean update; coef = {f = n_a n_b / n, g = n_b}.
__global__ void chan_prepare_kernel(MeanSet ms, const long long* __restrict__ n_dev, const int* __restrict__ nb,
                                    float* __restrict__ coef) {
    const long long na = *n_dev;
    const int n_b = *nb;
    const double n = static_cast<double>(na) + n_b;
    const float wb = n > 0 ? static_cast<float>(n_b / n) : 0.f;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        coef[0] = n > 0 ? static_cast<float>(static_cast<double>(na) * n_b / n) : 0.f;
        coef[1] = static_cast<float>(n_b);
    }
    const float f = n > 0 ? static_cast<float>(static_cast<double>(na) * n_b / n) : 0.f;
    const int chunks = (n_b + kChunk - 1) / kChunk;
    for (int m = 0; m < 4; ++m) {
        for (int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; c < ms.len[m];
             c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
            float zbar = 0.f, xb;
            if (ms.part) {
                float zs = 0.f;
                for (int k = 0; k < chunks; ++k) zs += ms.part[k * ms.Fall + ms.foff[m] + c];
                zbar = n_b > 0 ? zs / static_cast<float>(n_b) : 0.f;
                xb = ms.shift[m][c] + zbar;
            } else if (ms.zsum[m]) {
                zbar = n_b > 0 ? ms.zsum[m][c] / static_cast<float>(n_b) : 0.f;
                xb = ms.shift[m][c] + zbar;
            } else {
                xb = ms.bmean[m][c];
            }
            const float dl = n_b > 0 ? xb - ms.mean[m][c] : 0.f;
            ms.delta[m][c] = dl;
            ms.zbar[m][c] = zbar;
            ms.mean[m][c] += dl * wb;
            if (ms.part && m >= 2) {  // S_yy += sum z^2 - g zbar^2 + f delta^2
                float sq = 0.f;
                for (int k = 0; k < chunks; ++k) sq += ms.part_sq[k * ms.Fsq + ms.qoff[m] + c];
                ms.syy[m - 2][c] += sq - static_cast<float>(n_b) * zbar * zbar + f * dl * dl;
            }
        }
    }
}

__global__ void chan_finish_kernel(long long* __restrict__ n_dev, const int* __restrict__ nb) {
    *n_dev += *nb;
}

// S_yy[j] += sum_r Z[j][r]^2 - g zbar_j^2 + f delta_j^2.  One warp per column.
// Z is float32, or a (hi, lo) bf16 pair when lo != nullptr.
__global__ void syy_kernel(const void* __restrict__ Y, const void* __restrict__ Ylo, const void* __restrict__ Y3,
                           int64_t ld, int64_t rows_n,
                           const int* __restrict__ nb, const float* __restrict__ dy, const float* __restrict__ zy,
                           const float* __restrict__ coef, float* __restrict__ syy) {
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
                __bfloat162float(static_cast<const __nv_bfloat16*>(Ylo)[j * ld + r]) +
                (Y3 ? __bfloat162float(static_cast<const __nv_bfloat16*>(Y3)[j * ld + r]) : 0.f);
        s = fmaf(v, v, s);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) syy[j] += s - coef[1] * zy[j] * zy[j] + coef[0] * dy[j] * dy[j];
}

// out[i][j] += sum_r A[i][r] B[j][r] - g za_i zb_j + f da_i db_j over
// K = round_up(n_b, 64) (padding columns are zero).  64x64 tiles, 256 threads,
// 4x4 per thread.  With lower != 0, tiles entirely above the diagonal are skipped.
__global__ void __launch_bounds__(256) stats_gemm_simt_kernel(const float* __restrict__ A, const float* __restrict__ B,
                                                              int64_t ld, int64_t Ma, int64_t Nb, int lower,
                                                              const float* __restrict__ da,
                                                              const float* __restrict__ db,
                                                              const float* __restrict__ za,
                                                              const float* __restrict__ zb,
                                                              const float* __restrict__ coef,
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
    const float ff = coef[0], gg = coef[1];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        const int64_t i = i0 + ty * 4 + x;
        if (i >= Ma) continue;
        const float fa = ff * da[i], ga = gg * za[i];
#pragma unroll
        for (int y = 0; y < 4; ++y) {
            const int64_t j = j0 + tx * 4 + y;
            if (j >= Nb) continue;
            out[i * ldo + j] += acc[x][y] - ga * zb[j] + fa * db[j];
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

bool gather_single_pass_ok(kvb_dtype dt, int d) { return dt == KVB_BF16 && d % 16 == 0 && d <= 256; }

cudaError_t launch_gather(const GatherArgs& g, cudaStream_t s) {
    if (g.n_slabs == 0) return cudaSuccess;
    const int64_t F = g.n_slabs * g.d;
    dim3 grid(static_cast<unsigned>(g.n_slabs), static_cast<unsigned>((g.T + 63) / 64));
    if (gather_single_pass_ok(g.dt, g.d)) {
        const int rps = 256 / (g.d >> 4);
        const int R = rps >= kChunk ? 1 : kChunk / rps;
        if (g.out_lo != nullptr && (g.d == 64 || g.d == 128) && g.num_sms > 0) {
            dim3 sgrid(static_cast<unsigned>(g.num_sms));  // one CTA per SM, work split in-kernel
            const size_t smem = gather_stream_smem(g.d);
            const __nv_bfloat16* c16 = static_cast<const __nv_bfloat16*>(g.cache);
            __nv_bfloat16* o16 = static_cast<__nv_bfloat16*>(g.out);
            __nv_bfloat16* l16 = static_cast<__nv_bfloat16*>(g.out_lo);
#define KVB_STREAM(DD)                                                                                             \
    do {                                                                                                           \
        cudaError_t e = cudaFuncSetAttribute(gather_stream_kernel<DD>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                             static_cast<int>(smem));                                              \
        if (e != cudaSuccess) return e;                                                                            \
        gather_stream_kernel<DD><<<sgrid, stream_threads(DD), smem, s>>>(c16, g.T, g.rows, g.nb, g.n_seen, g.pos, g.tab, g.strip, \
                                                          g.mean_a, g.shift, g.part, F, o16, l16, g.ld,            \
                                                          static_cast<int>(g.n_slabs));                            \
    } while (0)
            switch (g.d) {
                case 64: KVB_STREAM(64); break;
                default: KVB_STREAM(128); break;
            }
#undef KVB_STREAM
            zsum_kernel<<<static_cast<unsigned>((F + 255) / 256), 256, 0, s>>>(g.part, F, g.nb, g.zsum);
            return cudaGetLastError();
        }
        const size_t smem = (static_cast<size_t>(g.d) * (kChunk + 1) + 8 * static_cast<size_t>(g.d)) * sizeof(float);
        // kept rows are about T / stride; a CTA loops if there are more
        const int64_t n_guess = (g.T + g.stride - 1) / g.stride;
        dim3 cgrid(static_cast<unsigned>((n_guess + kChunk - 1) / kChunk), static_cast<unsigned>(g.n_slabs));
        const __nv_bfloat16* c16 = static_cast<const __nv_bfloat16*>(g.cache);
#define KVB_GATHER(RR)                                                                                          \
    do {                                                                                                        \
        cudaError_t e = cudaFuncSetAttribute(gather_shift_kernel<RR>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                             200 * 1024);                                                       \
        if (e != cudaSuccess) return e;                                                                         \
        gather_shift_kernel<RR><<<cgrid, 256, smem, s>>>(c16, g.T, g.d, g.rows, g.nb, g.n_seen, g.pos, g.tab,   \
                                                         g.strip, g.mean_a, g.shift, g.part, F, g.out, g.out_lo, \
                                                         g.ld);                                                 \
    } while (0)
        switch (R) {
            case 1: KVB_GATHER(1); break;
            case 2: KVB_GATHER(2); break;
            case 4: KVB_GATHER(4); break;
            default: KVB_GATHER(8); break;
        }
#undef KVB_GATHER
        zsum_kernel<<<static_cast<unsigned>((F + 255) / 256), 256, 0, s>>>(g.part, F, g.nb, g.zsum);
        return cudaGetLastError();
    }
    // generic two-pass path: batch means, then centering on them (zbar = 0)
    if (g.dt == KVB_F32)
        colmean_kernel<float><<<static_cast<unsigned>(g.n_slabs), 256, 0, s>>>(
            static_cast<const float*>(g.cache), g.T, g.d, g.rows, g.nb, g.pos, g.tab, g.strip, g.bmean);
    else
        colmean_kernel<__nv_bfloat16><<<static_cast<unsigned>(g.n_slabs), 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(g.cache), g.T, g.d, g.rows, g.nb, g.pos, g.tab, g.strip, g.bmean);
    const size_t smem = 64 * (g.d + 1) * sizeof(float);
    if (g.dt == KVB_F32) {
        cudaFuncSetAttribute(center_transpose_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, 80 * 1024);
        center_transpose_kernel<float><<<grid, 256, smem, s>>>(static_cast<const float*>(g.cache), g.T, g.d, g.rows,
                                                               g.nb, g.pos, g.tab, g.strip, g.bmean, g.out, g.out_lo,
                                                               g.out_3, g.ld);
    } else {
        cudaFuncSetAttribute(center_transpose_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             80 * 1024);
        center_transpose_kernel<__nv_bfloat16><<<grid, 256, smem, s>>>(
            static_cast<const __nv_bfloat16*>(g.cache), g.T, g.d, g.rows, g.nb, g.pos, g.tab, g.strip, g.bmean, g.out,
            g.out_lo, g.out_3, g.ld);
    }
    return cudaGetLastError();
}

cudaError_t launch_first_mean(const FirstMeanArgs& a, cudaStream_t s) {
    int64_t most = 0;
    for (int m = 0; m < 4; ++m) most = a.n_slabs[m] > most ? a.n_slabs[m] : most;
    if (most == 0) return cudaSuccess;
    first_mean_kernel<<<dim3(static_cast<unsigned>(most), 4), 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_chan_prepare(const MeanSet& ms, const long long* n_dev, const int* nb, float* coef,
                                cudaStream_t s) {
    chan_prepare_kernel<<<256, 256, 0, s>>>(ms, n_dev, nb, coef);
    return cudaGetLastError();
}

cudaError_t launch_chan_finish(long long* n_dev, const int* nb, cudaStream_t s) {
    chan_finish_kernel<<<1, 1, 0, s>>>(n_dev, nb);
    return cudaGetLastError();
}

cudaError_t launch_syy(const void* Y, const void* Ylo, const void* Y3, int64_t ld, int64_t rows_n, const int* nb, const float* dy,
                       const float* zy, const float* coef, float* syy, cudaStream_t s) {
    const int64_t threads = rows_n * 32;
    const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
    if (blocks == 0) return cudaSuccess;
    syy_kernel<<<blocks, 256, 0, s>>>(Y, Ylo, Y3, ld, rows_n, nb, dy, zy, coef, syy);
    return cudaGetLastError();
}

cudaError_t launch_stats_gemm_simt(const float* A, const float* B, int64_t ld, int64_t Ma, int64_t Nb, bool lower,
                                   const float* da, const float* db, const float* za, const float* zb,
                                   const float* coef, const int* nb, float* out, int64_t ldo, cudaStream_t s) {
    dim3 grid(static_cast<unsigned>((Nb + 63) / 64), static_cast<unsigned>((Ma + 63) / 64));
    if (grid.x == 0 || grid.y == 0) return cudaSuccess;
    stats_gemm_simt_kernel<<<grid, 256, 0, s>>>(A, B, ld, Ma, Nb, lower ? 1 : 0, da, db, za, zb, coef, nb, out, ldo);
    return cudaGetLastError();
}

}  // namespace kvb

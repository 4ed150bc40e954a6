// RoPE tables and the HBM-bound strip pass over bf16 source keys.
//
// "Cross-Model KV Transfer" (VeloxQuant-MLX), "The mapping": keys are
// un-rotated with the source model's RoPE before the map and re-rotated with
// the target's after it.  Rotate-half pairs (i, i + d/2) with frequency
// theta^(-2i/d); angles are reduced in float64 ("KVBridge", "What ships":
// exact inverse/forward RoPE), stored as float32 cos/sin.
#include "kvb_internal.h"

namespace kvb {

__global__ void rope_table_kernel(float2* __restrict__ tab, int max_pos, int half, double theta) {
    const int64_t n = static_cast<int64_t>(max_pos) * half;
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < n;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int p = static_cast<int>(g / half);
        const int i = static_cast<int>(g - static_cast<int64_t>(p) * half);
        const double w = pow(theta, -static_cast<double>(i) / static_cast<double>(half));
        double s, c;
        sincos(static_cast<double>(p) * w, &s, &c);
        tab[g] = make_float2(static_cast<float>(c), static_cast<float>(s));
    }
}

cudaError_t launch_rope_table(float2* tab, int max_pos, int d, double theta, cudaStream_t s) {
    const int half = d / 2;
    const int64_t n = static_cast<int64_t>(max_pos) * half;
    const int threads = 256;
    const int blocks = static_cast<int>((n + threads - 1) / threads < 65535 ? (n + threads - 1) / threads : 65535);
    rope_table_kernel<<<blocks, threads, 0, s>>>(tab, max_pos, half, theta);
    return cudaGetLastError();
}

// Each thread owns 8 pairs: 8 consecutive elements of the low half and the
// matching 8 of the high half (two 16-byte loads, two 16-byte stores).
// Strip = rotation by -angle: lo' = lo*c + hi*s, hi' = hi*c - lo*s.
__global__ void __launch_bounds__(256) strip_bf16_vec_kernel(const __nv_bfloat16* __restrict__ in,
                                                             __nv_bfloat16* __restrict__ out,
                                                             const int* __restrict__ pos,
                                                             const float2* __restrict__ tab, int64_t rows,
                                                             int64_t T, int d, int max_pos, DevErr err) {
    const int half = d >> 1;
    const int cpr = half >> 3;  // 8-pair chunks per row
    const int64_t n = rows * cpr;
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < n;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t row = g / cpr;
        const int c = static_cast<int>(g - row * cpr);
        const int64_t tok = row % T;
        const int e0 = c * 8;
        const __nv_bfloat16* src = in + row * d + e0;
        __nv_bfloat16* dst = out + row * d + e0;
        if (!KVB_IN_BOUNDS(err, row * d + e0, 8, rows * d) || !KVB_IN_BOUNDS(err, row * d + e0 + half, 8, rows * d) ||
            !KVB_IN_BOUNDS(err, tok, 1, T))
            continue;
        const int p = __ldg(pos + tok);
        if (p < 0 || p >= max_pos) {
            dev_err_set(err, DEV_ERR_BAD_POS);
            const uint4 z = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(dst) = z;
            *reinterpret_cast<uint4*>(dst + half) = z;
            continue;
        }
        if (!KVB_IN_BOUNDS(err, static_cast<int64_t>(p) * half + e0, 8, static_cast<int64_t>(max_pos) * half)) continue;
        const uint4 vlo = __ldcs(reinterpret_cast<const uint4*>(src));
        const uint4 vhi = __ldcs(reinterpret_cast<const uint4*>(src + half));
        const float4* tp = reinterpret_cast<const float4*>(tab + static_cast<int64_t>(p) * half + e0);
        float cs[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 t4 = __ldg(tp + q);
            cs[4 * q + 0] = t4.x;
            cs[4 * q + 1] = t4.y;
            cs[4 * q + 2] = t4.z;
            cs[4 * q + 3] = t4.w;
        }
        const __nv_bfloat162* lo2 = reinterpret_cast<const __nv_bfloat162*>(&vlo);
        const __nv_bfloat162* hi2 = reinterpret_cast<const __nv_bfloat162*>(&vhi);
        uint32_t olo[4], ohi[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 l = __bfloat1622float2(lo2[q]);
            const float2 h = __bfloat1622float2(hi2[q]);
            const float c0 = cs[4 * q + 0], s0 = cs[4 * q + 1];
            const float c1 = cs[4 * q + 2], s1 = cs[4 * q + 3];
            const float l0 = fmaf(l.x, c0, h.x * s0);
            const float h0 = fmaf(h.x, c0, -(l.x * s0));
            const float l1 = fmaf(l.y, c1, h.y * s1);
            const float h1 = fmaf(h.y, c1, -(l.y * s1));
            olo[q] = pack_bf16x2(l0, l1);
            ohi[q] = pack_bf16x2(h0, h1);
        }
        __stcs(reinterpret_cast<uint4*>(dst), make_uint4(olo[0], olo[1], olo[2], olo[3]));
        __stcs(reinterpret_cast<uint4*>(dst + half), make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]));
    }
}

// Scalar variant for head dims that are not a multiple of 16.
__global__ void strip_bf16_scalar_kernel(const __nv_bfloat16* __restrict__ in, __nv_bfloat16* __restrict__ out,
                                         const int* __restrict__ pos, const float2* __restrict__ tab,
                                         int64_t rows, int64_t T, int d, int max_pos, DevErr err) {
    const int half = d >> 1;
    const int64_t n = rows * half;
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < n;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t row = g / half;
        const int i = static_cast<int>(g - row * half);
        const int p = __ldg(pos + (row % T));
        const int64_t base = row * d;
        if (p < 0 || p >= max_pos) {
            dev_err_set(err, DEV_ERR_BAD_POS);
            out[base + i] = __float2bfloat16_rn(0.f);
            out[base + i + half] = __float2bfloat16_rn(0.f);
            continue;
        }
        const float2 cs = __ldg(tab + static_cast<int64_t>(p) * half + i);
        const float l = __bfloat162float(in[base + i]);
        const float h = __bfloat162float(in[base + i + half]);
        out[base + i] = __float2bfloat16_rn(fmaf(l, cs.x, h * cs.y));
        out[base + i + half] = __float2bfloat16_rn(fmaf(h, cs.x, -(l * cs.y)));
    }
}

cudaError_t launch_strip_bf16(const __nv_bfloat16* in, __nv_bfloat16* out, const int* pos, const float2* tab,
                              int64_t LH, int64_t T, int d, int max_pos, DevErr err, int num_sms,
                              cudaStream_t s) {
    const int64_t rows = LH * T;
    if (rows == 0) return cudaSuccess;
    const int threads = 256;
    const int blocks = num_sms * 8;  // persistent grid-stride: 8 resident CTAs per SM
    if (d % 16 == 0) {
        strip_bf16_vec_kernel<<<blocks, threads, 0, s>>>(in, out, pos, tab, rows, T, d, max_pos, err);
    } else {
        strip_bf16_scalar_kernel<<<blocks, threads, 0, s>>>(in, out, pos, tab, rows, T, d, max_pos, err);
    }
    return cudaGetLastError();
}

// ------------------------------------------------------------------------
// fp32 caches on the tensor cores: every fp32 operand x is carried as two
// bf16 values, hi = bf16(x) and lo = bf16(x - hi) (x - hi is exact in fp32),
// and the map accumulates hi*hi + hi*lo + lo*hi in fp32; the dropped lo*lo
// term is below 2^-16 of each product.

__device__ __forceinline__ void split8(const float* x, uint4& hi, uint4& lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(x[2 * q], x[2 * q + 1]);
        const float2 bf = __bfloat1622float2(b);
        h[q] = pack_bf16x2(bf.x, bf.y);
        l[q] = pack_bf16x2(x[2 * q] - bf.x, x[2 * q + 1] - bf.y);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// Strip source RoPE from fp32 keys [rows][d] (rows = LH*T) and split the
// result into bf16 hi / lo copies of the same layout.  Each thread owns 8
// pairs, as in the bf16 strip pass.
__global__ void __launch_bounds__(256) strip_split_f32_kernel(const float* __restrict__ in,
                                                              __nv_bfloat16* __restrict__ out_hi,
                                                              __nv_bfloat16* __restrict__ out_lo,
                                                              const int* __restrict__ pos,
                                                              const float2* __restrict__ tab, int64_t rows,
                                                              int64_t T, int d, int max_pos, DevErr err) {
    const int half = d >> 1;
    const int cpr = half >> 3;
    const int64_t n = rows * cpr;
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < n;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t row = g / cpr;
        const int e0 = static_cast<int>(g - row * cpr) * 8;
        const int64_t o = row * d + e0;
        const int p = __ldg(pos + row % T);
        float xl[8], xh[8];
        if (p < 0 || p >= max_pos) {
            dev_err_set(err, DEV_ERR_BAD_POS);
#pragma unroll
            for (int i = 0; i < 8; ++i) xl[i] = xh[i] = 0.f;
        } else {
            const float4* src = reinterpret_cast<const float4*>(in + o);
            const float4* srch = reinterpret_cast<const float4*>(in + o + half);
            const float4 a0 = __ldcs(src), a1 = __ldcs(src + 1), b0 = __ldcs(srch), b1 = __ldcs(srch + 1);
            const float l[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float h[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
            const float4* tp = reinterpret_cast<const float4*>(tab + static_cast<int64_t>(p) * half + e0);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 cs = __ldg(tp + q);  // (c, s) of pairs 2q and 2q+1
                xl[2 * q] = fmaf(l[2 * q], cs.x, h[2 * q] * cs.y);
                xh[2 * q] = fmaf(h[2 * q], cs.x, -(l[2 * q] * cs.y));
                xl[2 * q + 1] = fmaf(l[2 * q + 1], cs.z, h[2 * q + 1] * cs.w);
                xh[2 * q + 1] = fmaf(h[2 * q + 1], cs.z, -(l[2 * q + 1] * cs.w));
            }
        }
        uint4 hi, lo;
        split8(xl, hi, lo);
        __stcs(reinterpret_cast<uint4*>(out_hi + o), hi);
        __stcs(reinterpret_cast<uint4*>(out_lo + o), lo);
        split8(xh, hi, lo);
        __stcs(reinterpret_cast<uint4*>(out_hi + o + half), hi);
        __stcs(reinterpret_cast<uint4*>(out_lo + o + half), lo);
    }
}

// Split n fp32 values (n % 8 == 0, 16-byte aligned) into bf16 hi / lo.
__global__ void __launch_bounds__(256) split_f32_kernel(const float* __restrict__ in,
                                                        __nv_bfloat16* __restrict__ out_hi,
                                                        __nv_bfloat16* __restrict__ out_lo, int64_t n8) {
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < n8;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float4* src = reinterpret_cast<const float4*>(in) + 2 * g;
        const float4 a = __ldcs(src), b = __ldcs(src + 1);
        const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint4 hi, lo;
        split8(x, hi, lo);
        __stcs(reinterpret_cast<uint4*>(out_hi) + g, hi);
        __stcs(reinterpret_cast<uint4*>(out_lo) + g, lo);
    }
}

cudaError_t launch_strip_split_f32(const float* in, __nv_bfloat16* hi, __nv_bfloat16* lo, const int* pos,
                                   const float2* tab, int64_t LH, int64_t T, int d, int max_pos, DevErr err,
                                   int num_sms, cudaStream_t s) {
    if (LH * T == 0) return cudaSuccess;
    strip_split_f32_kernel<<<num_sms * 8, 256, 0, s>>>(in, hi, lo, pos, tab, LH * T, T, d, max_pos, err);
    return cudaGetLastError();
}

cudaError_t launch_split_f32(const float* in, __nv_bfloat16* hi, __nv_bfloat16* lo, int64_t n, int num_sms,
                             cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    split_f32_kernel<<<num_sms * 8, 256, 0, s>>>(in, hi, lo, n / 8);
    return cudaGetLastError();
}

}  // namespace kvb

// Mapper apply on the CUDA cores, for float32 caches and for shapes the
// tensor-core kernel does not tile (head_dim != 128).
//
// Same computation as the tensor-core path ("Cross-Model KV Transfer"
// (VeloxQuant-MLX), "The mapping"): the source-RoPE strip is fused into the
// operand load (keys only), the bias and the target RoPE into the epilogue.
// One CTA computes BM tokens x one whole head (d outputs) of one target layer,
// so each thread holds both members of its RoPE pairs (e, e + d/2).
#include "kvb_internal.h"

namespace kvb {

namespace {

constexpr int BK = 16;
constexpr int TM = 4;  // tokens per thread
constexpr int TC = 4;  // pairs per thread (4 low-half columns + their 4 partners)

template <typename T>
__device__ __forceinline__ float ld_as_float(const T* p);
template <>
__device__ __forceinline__ float ld_as_float<float>(const float* p) {
    return __ldg(p);
}
template <>
__device__ __forceinline__ float ld_as_float<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}

template <typename T>
__device__ __forceinline__ void store4(T* dst, const float* v);
template <>
__device__ __forceinline__ void store4<float>(float* dst, const float* v) {
    *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* dst, const float* v) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
}

struct SimtParams {
    int L_s, L_t, H, d, k, max_pos;
    int64_t T;
    int CG, TG, BM;
    const void* src[2];
    const void* w[2];
    const float* bias[2];
    void* out[2];
    const int* pos;
    const float2* tab_s;
    const float2* tab_t;
    DevErr err;
    SelTable sel;
};

template <typename T>
__global__ void map_simt_kernel(const __grid_constant__ SimtParams P) {
    extern __shared__ float sm[];
    const int BM = P.BM, d = P.d, half = d >> 1;
    float* As = sm;            // [BK][BM]
    float* Ws = sm + BK * BM;  // [BK][d]
    __shared__ int spos[1024];

    const int m = blockIdx.x;
    const int h = blockIdx.y;
    const int kv = blockIdx.z / P.L_t;
    const int t = blockIdx.z - kv * P.L_t;
    const int q = P.H * d;
    const int p = P.k * q;
    const int64_t tok0 = static_cast<int64_t>(m) * BM;
    const int nthreads = P.CG * P.TG;
    const int tid = threadIdx.x;
    const int cg = tid % P.CG;
    const int tg = tid / P.CG;

    const T* src = static_cast<const T*>(P.src[kv]);
    const T* w = static_cast<const T*>(P.w[kv]) + (static_cast<int64_t>(t) * q + static_cast<int64_t>(h) * d) * p;

    for (int i = tid; i < BM; i += nthreads) {
        const int64_t tok = tok0 + i;
        int pp = -1;
        if (tok < P.T) {
            pp = __ldg(P.pos + tok);
            if (pp < 0 || pp >= P.max_pos) {
                dev_err_set(P.err, DEV_ERR_BAD_POS);
                pp = -2;
            }
        }
        spos[i] = pp;
    }
    __syncthreads();

    float acc[TM][2 * TC];
#pragma unroll
    for (int a = 0; a < TM; ++a)
#pragma unroll
        for (int b = 0; b < 2 * TC; ++b) acc[a][b] = 0.f;

    for (int f0 = 0; f0 < p; f0 += BK) {
        // A: BM tokens x BK features, gathered (and stripped for keys)
        for (int i = tid; i < BM * BK; i += nthreads) {
            const int kk = i % BK;
            const int tl = i / BK;
            const int f = f0 + kk;
            float v = 0.f;
            const int pp = spos[tl];
            if (f < p && pp >= 0) {
                const int j = f / q;
                const int r = f - j * q;
                const int hh = r / d;
                const int e = r - hh * d;
                const int layer = P.sel.s[kv][t][j];
                const T* row = src + ((static_cast<int64_t>(layer) * P.H + hh) * P.T + tok0 + tl) * d;
                v = ld_as_float<T>(row + e);
                if (kv == 0) {
                    const int i2 = e < half ? e : e - half;
                    const float2 cs = __ldg(P.tab_s + static_cast<int64_t>(pp) * half + i2);
                    const float partner = ld_as_float<T>(row + (e < half ? e + half : e - half));
                    v = e < half ? fmaf(v, cs.x, partner * cs.y) : fmaf(v, cs.x, -(partner * cs.y));
                }
            }
            As[kk * BM + tl] = v;
        }
        // W: this head's d output rows x BK features
        for (int i = tid; i < d * BK; i += nthreads) {
            const int kk = i % BK;
            const int e = i / BK;
            const int f = f0 + kk;
            Ws[kk * d + e] = f < p ? ld_as_float<T>(w + static_cast<int64_t>(e) * p + f) : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int kk = 0; kk < BK; ++kk) {
            float a[TM], b[2 * TC];
#pragma unroll
            for (int x = 0; x < TM; ++x) a[x] = As[kk * BM + tg * TM + x];
#pragma unroll
            for (int y = 0; y < TC; ++y) {
                b[y] = Ws[kk * d + cg * TC + y];
                b[TC + y] = Ws[kk * d + half + cg * TC + y];
            }
#pragma unroll
            for (int x = 0; x < TM; ++x)
#pragma unroll
                for (int y = 0; y < 2 * TC; ++y) acc[x][y] = fmaf(a[x], b[y], acc[x][y]);
        }
        __syncthreads();
    }

    // Epilogue: bias, target RoPE for keys, store into [t][h][token][e].
    const float* bias = P.bias[kv] + static_cast<int64_t>(t) * q + static_cast<int64_t>(h) * d;
    float bl[TC], bh[TC];
#pragma unroll
    for (int y = 0; y < TC; ++y) {
        bl[y] = __ldg(bias + cg * TC + y);
        bh[y] = __ldg(bias + half + cg * TC + y);
    }
    T* out = static_cast<T*>(P.out[kv]) + (static_cast<int64_t>(t) * P.H + h) * P.T * d;
#pragma unroll
    for (int x = 0; x < TM; ++x) {
        const int tl = tg * TM + x;
        const int64_t tok = tok0 + tl;
        if (tok >= P.T) continue;
        const int pp = spos[tl];
        float lo[TC], hi[TC];
#pragma unroll
        for (int y = 0; y < TC; ++y) {
            lo[y] = acc[x][y] + bl[y];
            hi[y] = acc[x][TC + y] + bh[y];
        }
        if (pp < 0) {
#pragma unroll
            for (int y = 0; y < TC; ++y) lo[y] = hi[y] = 0.f;
        } else if (kv == 0) {
#pragma unroll
            for (int y = 0; y < TC; ++y) {
                const float2 cs = __ldg(P.tab_t + static_cast<int64_t>(pp) * half + cg * TC + y);
                const float l = lo[y], hv = hi[y];
                lo[y] = fmaf(l, cs.x, -(hv * cs.y));
                hi[y] = fmaf(hv, cs.x, l * cs.y);
            }
        }
        store4<T>(out + tok * d + cg * TC, lo);
        store4<T>(out + tok * d + half + cg * TC, hi);
    }
}

}  // namespace

cudaError_t launch_map_simt(const MapSimtArgs& a, cudaStream_t s) {
    const Shape& sh = a.sh;
    SimtParams P{};
    P.L_s = sh.L_s;
    P.L_t = sh.L_t;
    P.H = sh.H;
    P.d = sh.d;
    P.k = sh.k;
    P.max_pos = sh.max_pos;
    P.T = sh.T;
    P.CG = (sh.d / 2) / TC;
    P.TG = 256 / P.CG < 1 ? 1 : 256 / P.CG;
    P.BM = P.TG * TM;
    if (P.BM > 1024) return cudaErrorInvalidValue;
    for (int kv = 0; kv < 2; ++kv) {
        P.src[kv] = a.src[kv];
        P.w[kv] = a.w[kv];
        P.bias[kv] = a.bias[kv];
        P.out[kv] = a.out[kv];
    }
    P.pos = a.pos;
    P.tab_s = a.tab_s;
    P.tab_t = a.tab_t;
    P.err = a.err;
    P.sel = a.sel;
    const int64_t num_m = (sh.T + P.BM - 1) / P.BM;
    if (num_m > 0x7fffffffLL || sh.H > 65535 || 2 * sh.L_t > 65535) return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>(num_m), sh.H, 2 * sh.L_t);
    const int threads = P.CG * P.TG;
    const size_t smem = static_cast<size_t>(BK) * (P.BM + sh.d) * sizeof(float);
    if (a.dtype == KVB_F32) {
        cudaFuncSetAttribute(map_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
        map_simt_kernel<float><<<grid, threads, smem, s>>>(P);
    } else {
        cudaFuncSetAttribute(map_simt_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             96 * 1024);
        map_simt_kernel<__nv_bfloat16><<<grid, threads, smem, s>>>(P);
    }
    return cudaGetLastError();
}

}  // namespace kvb

// Attention-output cosine between two caches of the same target layer.
//
// "KVBridge" README, "Real-model T2 evidence" (attention-output cosine mean /
// minimum as a gate) and "Cross-Model KV Transfer" (VeloxQuant-MLX), "The
// honesty crux" item 6 (attention-output cosine, not R^2, predicts downstream
// retention): for target queries q, o = softmax(q K^T / sqrt(d)) V with the
// mapped cache and with the reference cache, compared by cosine.
//
// One CTA per (target layer, KV head, group of up to 64 query rows); the
// rows are the (query head of the group, query) pairs that share the KV head
// (query head hq reads KV head hq / (H_q / H)).  Keys stream through shared
// memory 32 at a time with an online softmax; the first cache's outputs stay
// in registers while the second cache streams, then each row's cosine is
// written.  Four threads per row, each scoring every fourth key and owning a
// quarter of the output dims.  Causal by position: key j is attended by
// query i iff kv_pos[j] <= q_pos[i].  fp32 arithmetic on CUDA cores: the
// diagnostic runs on a few held-out sequences, not on the transfer path.
#include <climits>

#include "kvb_host.h"

namespace kvb {

namespace {

constexpr int KT = 32;    // keys per shared-memory tile
constexpr int TPR = 4;    // threads per query row
constexpr int NT = 256;   // threads per CTA
constexpr int RMAX = NT / TPR;  // query rows per CTA

struct AttnParams {
    const void* q;      // [L][Hq][Tq][D]
    const void* k[2];   // [L][H][T][D]
    const void* v[2];
    const int* q_pos;   // [Tq]
    const int* kv_pos;  // [T]
    float* cos_out;     // [L][Hq][Tq]
    int L, H, Hq, Tq;
    int64_t T;
    float scale;
};

// Eight consecutive elements (16 bytes of bf16, two 16-byte words of fp32) to fp32.
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float* o) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        o[2 * i] = __uint_as_float(w[i] << 16);
        o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void load8(const float* p, float* o) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}
__device__ __forceinline__ void store8(float* s, const float* v) {
    reinterpret_cast<float4*>(s)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(s)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// Shared-memory layout (floats): q [RMAX][D+4] | k [KT][D+4] | v [KT][D] | p [RMAX][KT+1].
// The +4 keeps rows float4-aligned while shifting consecutive rows by four banks.
template <int D>
constexpr size_t attn_smem_bytes() {
    return (static_cast<size_t>(RMAX) * (D + 4) + KT * (D + 4) + KT * D + RMAX * (KT + 1)) * sizeof(float);
}

template <typename T, int D>
__global__ void __launch_bounds__(NT, 2) attn_cosine_kernel(const __grid_constant__ AttnParams P) {
    constexpr int QLD = D + 4;
    constexpr int DQ = D / TPR;   // output dims per thread
    constexpr int KQ = KT / TPR;  // keys per thread per tile
    extern __shared__ float4 sm4[];
    float* qs = reinterpret_cast<float*>(sm4);
    float* ks = qs + RMAX * QLD;
    float* vs = ks + KT * QLD;
    float* ps = vs + KT * D;
    __shared__ int qpos_s[RMAX];
    __shared__ int kpos_s[KT];

    const int g = P.Hq / P.H;
    const int rows = g * P.Tq;
    const int r0 = blockIdx.x * RMAX;
    const int l = blockIdx.y / P.H;
    const int kh = blockIdx.y % P.H;
    const int tid = threadIdx.x;
    const int r = tid / TPR;    // local row
    const int qd = tid % TPR;   // quarter: keys qd, qd+4, ...; float4 columns qd, qd+4, ...
    const bool row_ok = r0 + r < rows;

    // the CTA's query rows: row gr is (query head kh*g + gr / Tq, query gr % Tq)
    const T* qbase = static_cast<const T*>(P.q);
    for (int e = tid; e < RMAX * (D / 8); e += NT) {
        const int rr = e / (D / 8), c8 = (e % (D / 8)) * 8;
        const int grr = r0 + rr;
        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (grr < rows) {
            const int hh = kh * g + grr / P.Tq, ii = grr % P.Tq;
            load8(qbase + ((static_cast<int64_t>(l) * P.Hq + hh) * P.Tq + ii) * D + c8, v);
        }
        store8(qs + rr * QLD + c8, v);
    }
    __shared__ int qpos_max;
    if (tid == 0) qpos_max = INT_MIN;
    __syncthreads();
    for (int e = tid; e < RMAX; e += NT) {
        const int grr = r0 + e;
        qpos_s[e] = grr < rows ? P.q_pos[grr % P.Tq] : -1;
        if (grr < rows) atomicMax(&qpos_max, qpos_s[e]);
    }
    __syncthreads();
    const int my_qpos = qpos_s[r];
    const int cta_qpos = qpos_max;

    float oa[DQ];
    float na = 0.f, nb = 0.f, dot = 0.f;
#pragma unroll 1
    for (int which = 0; which < 2; ++which) {
        const int64_t head = (static_cast<int64_t>(l) * P.H + kh) * P.T * D;
        const T* K = static_cast<const T*>(P.k[which]) + head;
        const T* V = static_cast<const T*>(P.v[which]) + head;
        float acc[DQ];
#pragma unroll
        for (int c = 0; c < DQ; ++c) acc[c] = 0.f;
        float m = -INFINITY, lsum = 0.f;
#pragma unroll 1
        for (int64_t j0 = 0; j0 < P.T; j0 += KT) {
            // skip a tile none of whose keys any row of the CTA may see (the
            // upper triangle of causal attention); the barrier also retires
            // the previous tile's k, v and p
            const bool seen = tid < KT && j0 + tid < P.T && P.kv_pos[j0 + tid] <= cta_qpos;
            if (!__syncthreads_or(seen)) continue;
            for (int e = tid; e < KT * (D / 8); e += NT) {
                const int jj = e / (D / 8), c8 = (e % (D / 8)) * 8;
                float kv8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                float vv8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                if (j0 + jj < P.T) {
                    load8(K + (j0 + jj) * D + c8, kv8);
                    load8(V + (j0 + jj) * D + c8, vv8);
                }
                store8(ks + jj * QLD + c8, kv8);
                store8(vs + jj * D + c8, vv8);
            }
            for (int e = tid; e < KT; e += NT) kpos_s[e] = j0 + e < P.T ? P.kv_pos[j0 + e] : 0;
            __syncthreads();

            // scores of keys qd, qd + 4, ... of the tile
            float s[KQ];
            float tmax = -INFINITY;
            const float4* qr = reinterpret_cast<const float4*>(qs + r * QLD);
#pragma unroll
            for (int jj = 0; jj < KQ; ++jj) {
                const int j = jj * TPR + qd;
                const float4* kr = reinterpret_cast<const float4*>(ks + j * QLD);
                float a0 = 0.f, a1 = 0.f;
#pragma unroll 8
                for (int c = 0; c < D / 4; ++c) {
                    const float4 x = qr[c], y = kr[c];
                    a0 = fmaf(x.x, y.x, a0);
                    a1 = fmaf(x.y, y.y, a1);
                    a0 = fmaf(x.z, y.z, a0);
                    a1 = fmaf(x.w, y.w, a1);
                }
                const bool ok = row_ok && j0 + j < P.T && kpos_s[j] <= my_qpos;
                s[jj] = ok ? (a0 + a1) * P.scale : -INFINITY;
                tmax = fmaxf(tmax, s[jj]);
            }
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
            // online softmax: rescale what was accumulated to the new running max
            const float mnew = fmaxf(m, tmax);
            const float alpha = mnew == -INFINITY ? 1.f : __expf(m - mnew);
            float psum = 0.f;
#pragma unroll
            for (int jj = 0; jj < KQ; ++jj) {
                const float p = s[jj] == -INFINITY ? 0.f : __expf(s[jj] - mnew);
                ps[r * (KT + 1) + jj * TPR + qd] = p;
                psum += p;
            }
            psum += __shfl_xor_sync(0xffffffffu, psum, 1);
            psum += __shfl_xor_sync(0xffffffffu, psum, 2);
            lsum = lsum * alpha + psum;
            m = mnew;
            __syncwarp();  // the row's four threads are in one warp
#pragma unroll
            for (int c = 0; c < DQ; ++c) acc[c] *= alpha;
#pragma unroll 4
            for (int j = 0; j < KT; ++j) {
                const float p = ps[r * (KT + 1) + j];
                const float4* vr = reinterpret_cast<const float4*>(vs + j * D);
#pragma unroll
                for (int c = 0; c < DQ / 4; ++c) {
                    const float4 y = vr[c * TPR + qd];
                    acc[4 * c] = fmaf(p, y.x, acc[4 * c]);
                    acc[4 * c + 1] = fmaf(p, y.y, acc[4 * c + 1]);
                    acc[4 * c + 2] = fmaf(p, y.z, acc[4 * c + 2]);
                    acc[4 * c + 3] = fmaf(p, y.w, acc[4 * c + 3]);
                }
            }
        }
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        if (which == 0) {
#pragma unroll
            for (int c = 0; c < DQ; ++c) {
                oa[c] = acc[c] * inv;
                na = fmaf(oa[c], oa[c], na);
            }
        } else {
#pragma unroll
            for (int c = 0; c < DQ; ++c) {
                const float ob = acc[c] * inv;
                dot = fmaf(oa[c], ob, dot);
                nb = fmaf(ob, ob, nb);
            }
        }
    }
#pragma unroll
    for (int o = 1; o < TPR; o <<= 1) {
        dot += __shfl_xor_sync(0xffffffffu, dot, o);
        na += __shfl_xor_sync(0xffffffffu, na, o);
        nb += __shfl_xor_sync(0xffffffffu, nb, o);
    }
    if (row_ok && qd == 0) {
        const int gr = r0 + r;
        const int hq = kh * g + gr / P.Tq, qi = gr % P.Tq;
        const float den = sqrtf(na) * sqrtf(nb);
        P.cos_out[(static_cast<int64_t>(l) * P.Hq + hq) * P.Tq + qi] = den > 0.f ? dot / den : 0.f;
    }
}

template <typename T, int D>
cudaError_t launch_attn(const AttnParams& P, cudaStream_t s) {
    constexpr size_t smem = attn_smem_bytes<D>();
    cudaError_t e = cudaFuncSetAttribute(attn_cosine_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int64_t rows = static_cast<int64_t>(P.Hq / P.H) * P.Tq;
    dim3 grid(static_cast<unsigned>((rows + RMAX - 1) / RMAX), static_cast<unsigned>(P.L * P.H));
    attn_cosine_kernel<T, D><<<grid, NT, smem, s>>>(P);
    return cudaGetLastError();
}

}  // namespace
}  // namespace kvb

using namespace kvb;

extern "C" kvb_status kvb_attention_cosine(kvb_ctx* c, kvb_dtype dtype, const void* q, int32_t n_q_heads,
                                           const int32_t* q_pos, int64_t Tq, const void* k_a, const void* v_a,
                                           const void* k_b, const void* v_b, const int32_t* kv_pos, int64_t T,
                                           float* cos_out, void* stream) {
    g_last_error.clear();
    if (!c) return fail(KVB_ERR_INVALID_ARG, "ctx is NULL");
    if (dtype != KVB_F32 && dtype != KVB_BF16) return fail(KVB_ERR_UNSUPPORTED, "dtype must be KVB_F32 or KVB_BF16");
    if (n_q_heads < c->H || n_q_heads % c->H)
        return fail(KVB_ERR_INVALID_ARG, "n_q_heads must be a positive multiple of the KV heads");
    if (Tq < 0 || T < 0 || Tq > 0x7fffffffLL) return fail(KVB_ERR_INVALID_ARG, "negative size");
    const int d = c->d;
    if (d != 16 && d != 32 && d != 64 && d != 128)
        return fail(KVB_ERR_UNSUPPORTED, "kvb_attention_cosine supports head_dim 16, 32, 64 or 128");
    if (Tq == 0) return KVB_OK;
    kvb_status st;
    if ((st = check_device_ptrs({q, q_pos, cos_out}, "kvb_attention_cosine")) != KVB_OK) return st;
    if (T > 0 && (st = check_device_ptrs({k_a, v_a, k_b, v_b, kv_pos}, "kvb_attention_cosine")) != KVB_OK)
        return st;
    const int64_t rows = static_cast<int64_t>(n_q_heads / c->H) * Tq;
    if ((rows + RMAX - 1) / RMAX > 0x7fffffffLL || static_cast<int64_t>(c->L_t) * c->H > 65535)
        return fail(KVB_ERR_UNSUPPORTED, "too many query rows or layers");
    AttnParams P{};
    P.q = q;
    P.k[0] = k_a;
    P.v[0] = v_a;
    P.k[1] = k_b;
    P.v[1] = v_b;
    P.q_pos = q_pos;
    P.kv_pos = kv_pos;
    P.cos_out = cos_out;
    P.L = c->L_t;
    P.H = c->H;
    P.Hq = n_q_heads;
    P.Tq = static_cast<int>(Tq);
    P.T = T;
    P.scale = 1.f / sqrtf(static_cast<float>(d));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    ProfScope ps(c, s, "attention_cosine");
    const bool bf = dtype == KVB_BF16;
    switch (d) {
        case 16: e = bf ? launch_attn<__nv_bfloat16, 16>(P, s) : launch_attn<float, 16>(P, s); break;
        case 32: e = bf ? launch_attn<__nv_bfloat16, 32>(P, s) : launch_attn<float, 32>(P, s); break;
        case 64: e = bf ? launch_attn<__nv_bfloat16, 64>(P, s) : launch_attn<float, 64>(P, s); break;
        default: e = bf ? launch_attn<__nv_bfloat16, 128>(P, s) : launch_attn<float, 128>(P, s); break;
    }
    if (e != cudaSuccess) return cuda_fail(e, "attention cosine launch");
    return KVB_OK;
}

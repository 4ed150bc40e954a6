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
// written.  Eight threads share two query rows: each scores every eighth key
// of the tile for both rows and owns every eighth float4 column of both
// outputs (a 2 x 4 register tile per step).  Causal by position: key j is attended by
// query i iff kv_pos[j] <= q_pos[i].  fp32 arithmetic on CUDA cores: the
// diagnostic runs on a few held-out sequences, not on the transfer path.
#include <climits>

#include "kvb_host.h"

namespace kvb {

namespace {

constexpr int KT = 32;          // keys per shared-memory tile
constexpr int NT = 256;         // threads per CTA
constexpr int GRP = 8;          // threads per group; a group owns two query rows
constexpr int RMAX = 2 * NT / GRP;  // query rows per CTA (64)

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
// Store eight floats as two float4.  Thread i of an eight-thread phase writes
// its halves in the order given by bit 2 of i, so that each phase touches
// eight distinct 16-byte bank groups.
__device__ __forceinline__ void store8(float* s, const float* v, int lane) {
    const int h = (lane >> 2) & 1;
    float4* d = reinterpret_cast<float4*>(s);
    const float4 lo = make_float4(v[0], v[1], v[2], v[3]);
    const float4 hi = make_float4(v[4], v[5], v[6], v[7]);
    d[h] = h ? hi : lo;
    d[h ^ 1] = h ? lo : hi;
}

// Shared-memory layout (floats): q [RMAX][D+4] | k [KT][D+4] | v [KT][D] | p [RMAX][KT+4].
// The +4 keeps rows float4-aligned while shifting consecutive rows by four banks.
template <int D>
constexpr size_t attn_smem_bytes() {
    return (static_cast<size_t>(RMAX) * (D + 4) + KT * (D + 4) + KT * D + RMAX * (KT + 4)) * sizeof(float);
}

template <typename T, int D>
__global__ void __launch_bounds__(NT, 2) attn_cosine_kernel(const __grid_constant__ AttnParams P) {
    constexpr int QLD = D + 4;
    constexpr int PLD = KT + 4;
    constexpr int DC = D / 4;                     // float4 columns of a row
    constexpr int CPT = (DC + GRP - 1) / GRP;     // float4 columns per thread (ragged for D = 16)
    constexpr int KPT = KT / GRP;                 // keys per thread per tile
    extern __shared__ float4 sm4[];
    float* qs = reinterpret_cast<float*>(sm4);
    float* ks = qs + RMAX * QLD;
    float* vs = ks + KT * QLD;
    float* ps = vs + KT * D;
    __shared__ int qpos_s[RMAX];
    __shared__ int kpos_s[KT];
    __shared__ int qpos_max;

    const int g = P.Hq / P.H;
    const int rows = g * P.Tq;
    const int r0 = blockIdx.x * RMAX;
    const int l = blockIdx.y / P.H;
    const int kh = blockIdx.y % P.H;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int grp = tid / GRP;     // rows 2 grp, 2 grp + 1
    const int t = tid % GRP;       // keys t, t + 8, ...; float4 columns t, t + 8, ...
    const int ra = 2 * grp;

    // the CTA's query rows: row gr is (query head kh*g + gr / Tq, query gr % Tq)
    if (tid == 0) qpos_max = INT_MIN;
    const T* qbase = static_cast<const T*>(P.q);
    for (int e = tid; e < RMAX * (D / 8); e += NT) {
        const int rr = e / (D / 8), c8 = (e % (D / 8)) * 8;
        const int grr = r0 + rr;
        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (grr < rows) {
            const int hh = kh * g + grr / P.Tq, ii = grr % P.Tq;
            load8(qbase + ((static_cast<int64_t>(l) * P.Hq + hh) * P.Tq + ii) * D + c8, v);
        }
        store8(qs + rr * QLD + c8, v, lane);
    }
    __syncthreads();
    for (int e = tid; e < RMAX; e += NT) {
        const int grr = r0 + e;
        qpos_s[e] = grr < rows ? P.q_pos[grr % P.Tq] : INT_MIN;
        if (grr < rows) atomicMax(&qpos_max, qpos_s[e]);
    }
    __syncthreads();
    const int qpos0 = qpos_s[ra], qpos1 = qpos_s[ra + 1];
    const int cta_qpos = qpos_max;

    float oa[2][4 * CPT];
    float na[2] = {0.f, 0.f}, nb[2] = {0.f, 0.f}, dot[2] = {0.f, 0.f};
#pragma unroll 1
    for (int which = 0; which < 2; ++which) {
        const int64_t head = (static_cast<int64_t>(l) * P.H + kh) * P.T * D;
        const T* K = static_cast<const T*>(P.k[which]) + head;
        const T* V = static_cast<const T*>(P.v[which]) + head;
        float acc[2][4 * CPT];
#pragma unroll
        for (int c = 0; c < 4 * CPT; ++c) acc[0][c] = acc[1][c] = 0.f;
        float m[2] = {-INFINITY, -INFINITY}, lsum[2] = {0.f, 0.f};
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
                store8(ks + jj * QLD + c8, kv8, lane);
                store8(vs + jj * D + c8, vv8, lane);
            }
            if (tid < KT) kpos_s[tid] = j0 + tid < P.T ? P.kv_pos[j0 + tid] : 0;
            __syncthreads();

            // scores: 2 rows x KPT keys per thread, one float4 of q and k per step
            float s[2][KPT];
#pragma unroll
            for (int i = 0; i < KPT; ++i) s[0][i] = s[1][i] = 0.f;
            const float4* q0 = reinterpret_cast<const float4*>(qs + ra * QLD);
            const float4* q1 = reinterpret_cast<const float4*>(qs + (ra + 1) * QLD);
#pragma unroll 1
            for (int c = 0; c < DC; ++c) {
                const float4 x0 = q0[c], x1 = q1[c];
#pragma unroll
                for (int i = 0; i < KPT; ++i) {
                    const float4 y = reinterpret_cast<const float4*>(ks + (t + GRP * i) * QLD)[c];
                    s[0][i] = fmaf(x0.x, y.x, fmaf(x0.y, y.y, fmaf(x0.z, y.z, fmaf(x0.w, y.w, s[0][i]))));
                    s[1][i] = fmaf(x1.x, y.x, fmaf(x1.y, y.y, fmaf(x1.z, y.z, fmaf(x1.w, y.w, s[1][i]))));
                }
            }
            float alpha[2];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int qp = rr ? qpos1 : qpos0;
                float tmax = -INFINITY;
#pragma unroll
                for (int i = 0; i < KPT; ++i) {
                    const int j = t + GRP * i;
                    const bool ok = j0 + j < P.T && kpos_s[j] <= qp;
                    s[rr][i] = ok ? s[rr][i] * P.scale : -INFINITY;
                    tmax = fmaxf(tmax, s[rr][i]);
                }
#pragma unroll
                for (int o = 1; o < GRP; o <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
                // online softmax: rescale what was accumulated to the new running max
                const float mnew = fmaxf(m[rr], tmax);
                alpha[rr] = mnew == -INFINITY ? 1.f : __expf(m[rr] - mnew);
                float psum = 0.f;
#pragma unroll
                for (int i = 0; i < KPT; ++i) {
                    const float p = s[rr][i] == -INFINITY ? 0.f : __expf(s[rr][i] - mnew);
                    ps[(ra + rr) * PLD + t + GRP * i] = p;
                    psum += p;
                }
#pragma unroll
                for (int o = 1; o < GRP; o <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
                lsum[rr] = lsum[rr] * alpha[rr] + psum;
                m[rr] = mnew;
            }
            __syncwarp();  // a group's eight threads are in one warp
#pragma unroll
            for (int c = 0; c < 4 * CPT; ++c) {
                acc[0][c] *= alpha[0];
                acc[1][c] *= alpha[1];
            }
            // weighted values: 2 rows x CPT float4 columns per thread
#pragma unroll 4
            for (int j = 0; j < KT; ++j) {
                const float p0 = ps[ra * PLD + j], p1 = ps[(ra + 1) * PLD + j];
                const float4* vr = reinterpret_cast<const float4*>(vs + j * D);
#pragma unroll
                for (int c = 0; c < CPT; ++c) {
                    if (t + GRP * c < DC) {
                        const float4 y = vr[t + GRP * c];
                        acc[0][4 * c] = fmaf(p0, y.x, acc[0][4 * c]);
                        acc[0][4 * c + 1] = fmaf(p0, y.y, acc[0][4 * c + 1]);
                        acc[0][4 * c + 2] = fmaf(p0, y.z, acc[0][4 * c + 2]);
                        acc[0][4 * c + 3] = fmaf(p0, y.w, acc[0][4 * c + 3]);
                        acc[1][4 * c] = fmaf(p1, y.x, acc[1][4 * c]);
                        acc[1][4 * c + 1] = fmaf(p1, y.y, acc[1][4 * c + 1]);
                        acc[1][4 * c + 2] = fmaf(p1, y.z, acc[1][4 * c + 2]);
                        acc[1][4 * c + 3] = fmaf(p1, y.w, acc[1][4 * c + 3]);
                    }
                }
            }
        }
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const float inv = lsum[rr] > 0.f ? 1.f / lsum[rr] : 0.f;
#pragma unroll
            for (int c = 0; c < 4 * CPT; ++c) {
                const float o = acc[rr][c] * inv;  // columns a thread does not own stay 0
                if (which == 0) {
                    oa[rr][c] = o;
                    na[rr] = fmaf(o, o, na[rr]);
                } else {
                    dot[rr] = fmaf(oa[rr][c], o, dot[rr]);
                    nb[rr] = fmaf(o, o, nb[rr]);
                }
            }
        }
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
#pragma unroll
        for (int o = 1; o < GRP; o <<= 1) {
            dot[rr] += __shfl_xor_sync(0xffffffffu, dot[rr], o);
            na[rr] += __shfl_xor_sync(0xffffffffu, na[rr], o);
            nb[rr] += __shfl_xor_sync(0xffffffffu, nb[rr], o);
        }
        const int gr = r0 + ra + rr;
        if (t == 0 && gr < rows) {
            const int hq = kh * g + gr / P.Tq, qi = gr % P.Tq;
            const float den = sqrtf(na[rr]) * sqrtf(nb[rr]);
            P.cos_out[(static_cast<int64_t>(l) * P.Hq + hq) * P.Tq + qi] = den > 0.f ? dot[rr] / den : 0.f;
        }
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
    if (attn_tc_supported(dtype, d, T, static_cast<int64_t>(c->L_t) * n_q_heads * Tq)) {
        std::string why;
        {
            ProfScope ps(c, s, "attention_cosine_tcgen05");
            e = launch_attn_cosine_tc(q, q_pos, k_a, v_a, k_b, v_b, kv_pos, cos_out, c->L_t, c->H, n_q_heads,
                                      static_cast<int>(Tq), T, dev_err(c), s, &why);
        }
        if (e != cudaSuccess) {
            if (!why.empty()) return fail(KVB_ERR_CUDA, "attention cosine launch: " + why);
            return cuda_fail(e, "attention cosine launch");
        }
        mirror_device_error(c, s);
        return KVB_OK;
    }
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

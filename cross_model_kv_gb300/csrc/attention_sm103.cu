// Attention-output cosine on the 5th-generation tensor cores (bf16 caches,
// head_dim 128).
//
// Same quantity as the CUDA-core kernel in attention.cu ("KVBridge" README,
// "Real-model T2 evidence"; "Cross-Model KV Transfer", "The honesty crux"
// item 6): per target layer, query head and query, the cosine between
// softmax(q K^T / sqrt(d)) V computed with cache a and with cache b; query head
// hq reads KV head hq / (Hq / H); key j is visible to query i iff
// kv_pos[j] <= q_pos[i].
//
// One CTA per (layer, KV head, 128 query rows of the head's query group), one
// CTA per SM (all 512 TMEM columns).  For each cache and each 128-key tile
// that some row of the CTA may see:
//   warp 0      TMA: the key tile (two 64-wide swizzled boxes) and the value
//               tile (one plain box) into shared memory;
//   warp 1      tcgen05.mma: S = Q K^T into TMEM (M 128, N 128, K 128), then,
//               once the probabilities are written, O_t = P_hi V + P_lo V;
//   warps 2..5  one query row per thread: S from TMEM, mask, running max and
//               sum (online softmax, base-2 exponentials), P as a bf16 pair
//               (hi, lo: ~16 significant bits) into shared memory in the
//               operand layout, the value tile transposed into the operand
//               layout; then O = alpha O + O_t in TMEM.
// The cosine of the two outputs is taken at the end straight from TMEM; the
// softmax denominators cancel in it.  Every wait is bounded (DevErr); the
// softmax warps agree on a failed wait across the warp before leaving, so
// the warp-wide TMEM instructions are never divergent.
#include <climits>
#include <string>

#include "kvb_host.h"

namespace kvb {

namespace {

constexpr int TR = 128;                 // query rows per CTA (MMA M)
constexpr int TK = 128;                 // keys per tile
constexpr int HD = 128;                 // head dim
constexpr int ATOM = 128 * 128;         // bytes of a 128-row x 64-element bf16 swizzle block
constexpr int TILE = 2 * ATOM;          // 128 x 128 bf16
constexpr int NUM_THREADS = 192;
constexpr int MAX_FLAG_TILES = 1024;
constexpr int SMEM_BYTES = 6 * TILE + 1024 + 256 + MAX_FLAG_TILES + 4 * TK * 4;
constexpr uint64_t DRAIN_NS = 200ull * 1000 * 1000;
constexpr uint32_t COL_S = 0, COL_OT = 128, COL_O = 256;  // O of cache x at COL_O + 128 x

struct Params {
    const __nv_bfloat16* q;  // [L][Hq][Tq][128]
    const int* q_pos;
    const int* kv_pos;
    float* cos_out;  // [L][Hq][Tq]
    int L, H, Hq, Tq, T;
    float scale_log2;  // log2(e) / sqrt(d)
    DevErr err;
};

struct Maps {
    CUtensorMap k[2], v[2];
};

// Byte offset of 16-byte chunk c (0..15) of row r in a 128 x 128 bf16
// K-major tile with the 128-byte swizzle (two 64-element blocks).
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
    return static_cast<uint32_t>((c >> 3) * ATOM + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint64_t desc_k(const uint8_t* tile, int kk) {  // 16-wide K step kk of 8
    return sdesc_k_sw128(smem_u32(tile) + (kk >> 2) * ATOM + (kk & 3) * 32);
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_cosine_tc_kernel(const __grid_constant__ Maps Mp, const __grid_constant__ Params P) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sQ = smem;
    uint8_t* sK = sQ + TILE;
    uint8_t* sV = sK + TILE;   // plain [key][d]
    uint8_t* sVt = sV + TILE;  // [d][key], operand layout
    uint8_t* sPh = sVt + TILE;
    uint8_t* sPl = sPh + TILE;
    uint64_t* bar = reinterpret_cast<uint64_t*>(sPl + TILE);
    uint64_t* kv_full = bar;
    uint64_t* kv_empty = bar + 1;
    uint64_t* s_full = bar + 2;
    uint64_t* p_full = bar + 3;
    uint64_t* o_full = bar + 4;
    uint64_t* drain = bar + 5;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 6);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* qmax_s = reinterpret_cast<int*>(tmem_slot + 2);
    uint8_t* flags = reinterpret_cast<uint8_t*>(bar) + 256;
    int* wpos = reinterpret_cast<int*>(flags + MAX_FLAG_TILES);  // per softmax warp: the tile's key positions

    const int g = P.Hq / P.H;
    const int rows = g * P.Tq;
    const int r0 = blockIdx.x * TR;
    const int l = blockIdx.y / P.H;
    const int kh = blockIdx.y % P.H;
    const int slab = l * P.H + kh;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ntiles = (P.T + TK - 1) / TK;
    const bool use_flags = ntiles <= MAX_FLAG_TILES;

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        mbar_init(kv_empty, 128);
        mbar_init(s_full, 1);
        mbar_init(p_full, 128);
        mbar_init(o_full, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        *qmax_s = INT_MIN;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    __syncthreads();

    // query rows into shared memory (operand layout) and the CTA's largest position
    const int row = 32 * (warp & 3) + lane;  // softmax warps: TMEM lane = tile row
    const int grow = r0 + row;
    const bool valid = warp >= 2 && grow < rows;
    const int qp = valid ? __ldg(P.q_pos + grow % P.Tq) : INT_MIN;
    if (warp >= 2) {
        if (valid) atomicMax(qmax_s, qp);
        const uint4* src = valid ? reinterpret_cast<const uint4*>(
                                       P.q + ((static_cast<int64_t>(l) * P.Hq + kh * g + grow / P.Tq) * P.Tq +
                                              grow % P.Tq) * HD)
                                 : nullptr;
#pragma unroll 4
        for (int c = 0; c < 16; ++c) {
            const uint4 v = valid ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(sQ + sw_off(row, c)) = v;
        }
        fence_proxy_async_smem();
    }
    __syncthreads();
    // tiles that no row of the CTA can see are skipped by every role alike
    if (use_flags) {
        const int qmax = *qmax_s;
        for (int t = warp; t < ntiles; t += NUM_THREADS / 32) {
            const int j = t * TK + 4 * lane;
            bool any = false;
            if (j < P.T) {
                if (j + 3 < P.T && (reinterpret_cast<uintptr_t>(P.kv_pos + j) & 15u) == 0) {
                    const int4 p4 = __ldg(reinterpret_cast<const int4*>(P.kv_pos + j));
                    any = p4.x <= qmax || p4.y <= qmax || p4.z <= qmax || p4.w <= qmax;
                } else {
                    for (int u = 0; u < 4 && j + u < P.T; ++u) any |= __ldg(P.kv_pos + j + u) <= qmax;
                }
            }
            any = __any_sync(0xffffffffu, any);
            if (lane == 0) flags[t] = any ? 1 : 0;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    auto live = [&](int t) { return !use_flags || flags[t] != 0; };

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------- producer
            int it = 0, last = -1;
            bool ok = true;
            for (int x = 0; x < 2 && ok; ++x) {
                for (int t = 0; t < ntiles; ++t) {
                    if (!live(t)) continue;
                    if (!mbar_wait(kv_empty, (it & 1) ^ 1u, P.err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(kv_full, 2 * TILE);
                    tma_load_3d(sK, &Mp.k[x], kv_full, 0, t * TK, slab);
                    tma_load_3d(sK + ATOM, &Mp.k[x], kv_full, 64, t * TK, slab);
                    tma_load_3d(sV, &Mp.v[x], kv_full, 0, t * TK, slab);
                    last = it++;
                }
            }
            if (last >= 0) mbar_wait_drain(kv_full, static_cast<uint32_t>(last & 1), DRAIN_NS);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------- MMA issuer
            constexpr uint32_t idesc = idesc_bf16_f32(TR, TK);
            int it = 0;
            bool ok = true;
            for (int x = 0; x < 2 && ok; ++x) {
                for (int t = 0; t < ntiles; ++t) {
                    if (!live(t)) continue;
                    if (!mbar_wait(kv_full, it & 1, P.err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk)
                        umma_bf16(tmem_base + COL_S, desc_k(sQ, kk), desc_k(sK, kk), idesc, kk != 0);
                    umma_commit(s_full);
                    if (!mbar_wait(p_full, it & 1, P.err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < TK / 16; ++kk)
                        umma_bf16(tmem_base + COL_OT, desc_k(sPh, kk), desc_k(sVt, kk), idesc, kk != 0);
#pragma unroll
                    for (int kk = 0; kk < TK / 16; ++kk)
                        umma_bf16(tmem_base + COL_OT, desc_k(sPl, kk), desc_k(sVt, kk), idesc, 1);
                    umma_commit(o_full);
                    ++it;
                }
            }
            umma_commit(drain);  // every MMA issued here completes before TMEM is released
            mbar_wait_drain(drain, 0, DRAIN_NS);
        }
    } else {
        // ----------------------------------------------------------- softmax
        const uint32_t tl = tmem_base + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
        auto wait_all = [&](uint64_t* b, uint32_t parity) {  // warp-uniform outcome
            const bool got = mbar_wait(b, parity, P.err, abort_flag);
            return __all_sync(0xffffffffu, got);
        };
        int it = 0, done = 0;
        bool ok = true;
        for (int x = 0; x < 2 && ok; ++x) {
            float m = -INFINITY;
            bool first = true;
            for (int t = 0; t < ntiles; ++t) {
                if (!live(t)) continue;
                const int j0 = t * TK;
                // the value tile, transposed into the operand layout while the MMA computes S:
                // this thread's row is dim `row`
                if (!wait_all(kv_full, it & 1)) {
                    ok = false;
                    break;
                }
                const __nv_bfloat16* vcol = reinterpret_cast<const __nv_bfloat16*>(sV) + row;
#pragma unroll 2
                for (int c = 0; c < TK / 8; ++c) {
                    uint32_t w4[4];
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const uint32_t a = __bfloat16_as_ushort(vcol[(8 * c + 2 * w) * HD]);
                        const uint32_t b = __bfloat16_as_ushort(vcol[(8 * c + 2 * w + 1) * HD]);
                        w4[w] = a | (b << 16);
                    }
                    *reinterpret_cast<uint4*>(sVt + sw_off(row, c)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
                // the tile's key positions, staged per warp (INT_MAX past the end)
                int* kpos = wpos + (warp - 2) * TK;
                {
                    const int j = j0 + 4 * lane;
                    int4 p4 = make_int4(INT_MAX, INT_MAX, INT_MAX, INT_MAX);
                    if (j + 3 < P.T) {
                        p4 = __ldg(reinterpret_cast<const int4*>(P.kv_pos + j));
                    } else {
                        if (j < P.T) p4.x = __ldg(P.kv_pos + j);
                        if (j + 1 < P.T) p4.y = __ldg(P.kv_pos + j + 1);
                        if (j + 2 < P.T) p4.z = __ldg(P.kv_pos + j + 2);
                    }
                    __syncwarp();  // the warp is done with the previous tile's positions
                    reinterpret_cast<int4*>(kpos)[lane] = p4;
                    __syncwarp();
                }
                if (!wait_all(s_full, it & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // the whole score row, masked and scaled to base 2
                uint32_t sv[TK / 16][16];
#pragma unroll
                for (int c = 0; c < TK / 16; ++c) tmem_ld16(tl + COL_S + 16 * c, sv[c]);
                tmem_ld_wait();
                float mt = -INFINITY;
#pragma unroll
                for (int c = 0; c < TK / 16; ++c) {
#pragma unroll
                    for (int u = 0; u < 16; u += 4) {
                        const int4 p4 = reinterpret_cast<const int4*>(kpos)[(16 * c + u) >> 2];
                        const int pa[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            // positions past the end are INT_MAX; a query at INT_MAX is
                            // excluded from them by the index test
                            const bool vis = valid && pa[w] <= qp && j0 + 16 * c + u + w < P.T;
                            const float v = vis ? __uint_as_float(sv[c][u + w]) * P.scale_log2 : -INFINITY;
                            sv[c][u + w] = __float_as_uint(v);
                            mt = fmaxf(mt, v);
                        }
                    }
                }
                const float m_new = fmaxf(m, mt);
                const float alpha = m_new == -INFINITY ? 1.f : exp2f(m - m_new);
                // probabilities as bf16 (hi, lo) in the operand layout
#pragma unroll
                for (int c = 0; c < TK / 16; ++c) {
                    float p[16];
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const float v = __uint_as_float(sv[c][u]);
                        p[u] = v == -INFINITY ? 0.f : exp2f(v - m_new);
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t hi[4], lo[4];
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            const float a = p[8 * h + 2 * w], b = p[8 * h + 2 * w + 1];
                            const __nv_bfloat162 bh = __floats2bfloat162_rn(a, b);
                            const float2 bf = __bfloat1622float2(bh);
                            hi[w] = *reinterpret_cast<const uint32_t*>(&bh);
                            lo[w] = pack_bf16x2(a - bf.x, b - bf.y);
                        }
                        const uint32_t off = sw_off(row, 2 * c + h);
                        *reinterpret_cast<uint4*>(sPh + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        *reinterpret_cast<uint4*>(sPl + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    }
                }
                m = m_new;
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(p_full);
                mbar_arrive(kv_empty);  // key tile consumed by S, value tile transposed
                if (!wait_all(o_full, it & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // O = alpha O + O_t (O = O_t on the cache's first tile)
                const uint32_t co = COL_O + 128u * x;
#pragma unroll 1
                for (int c0 = 0; c0 < HD; c0 += 16) {
                    uint32_t ot[16], oo[16];
                    tmem_ld16(tl + COL_OT + c0, ot);
                    if (!first) tmem_ld16(tl + co + c0, oo);
                    tmem_ld_wait();
#pragma unroll
                    for (int u = 0; u < 16; ++u)
                        oo[u] = first ? ot[u]
                                      : __float_as_uint(fmaf(alpha, __uint_as_float(oo[u]), __uint_as_float(ot[u])));
                    tmem_st16(tl + co + c0, oo);
                }
                tmem_st_wait();
                tc_fence_before();
                first = false;
                ++it;
                if (x == 0) ++done;
            }
        }
        if (ok) {
            float dot = 0.f, na = 0.f, nb = 0.f;
            if (done > 0) {
                tc_fence_after();
#pragma unroll 1
                for (int c0 = 0; c0 < HD; c0 += 16) {
                    uint32_t oa[16], ob[16];
                    tmem_ld16(tl + COL_O + c0, oa);
                    tmem_ld16(tl + COL_O + 128 + c0, ob);
                    tmem_ld_wait();
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const float a = __uint_as_float(oa[u]), b = __uint_as_float(ob[u]);
                        dot = fmaf(a, b, dot);
                        na = fmaf(a, a, na);
                        nb = fmaf(b, b, nb);
                    }
                }
            }
            if (valid) {
                const float den = sqrtf(na) * sqrtf(nb);
                const int hq = kh * g + grow / P.Tq;
                P.cos_out[(static_cast<int64_t>(l) * P.Hq + hq) * P.Tq + grow % P.Tq] = den > 0.f ? dot / den : 0.f;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

bool encode_cache(CUtensorMap* m, const void* base, int64_t slabs, int64_t T, uint32_t box_x, bool swizzle,
                  std::string* why) {
    EncodeTiledFn enc = get_encode_tiled();
    if (!enc) {
        if (why) *why = "cuTensorMapEncodeTiled unavailable from the driver";
        return false;
    }
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(slabs)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(HD) * 2, static_cast<cuuint64_t>(T) * HD * 2};
    cuuint32_t box[3] = {box_x, static_cast<cuuint32_t>(TK), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        if (why) *why = "cuTensorMapEncodeTiled failed with code " + std::to_string(static_cast<int>(r));
        return false;
    }
    return true;
}

}  // namespace

bool attn_tc_supported(kvb_dtype dtype, int d, int64_t T) { return dtype == KVB_BF16 && d == HD && T >= 1; }

cudaError_t launch_attn_cosine_tc(const void* q, const int* q_pos, const void* k_a, const void* v_a, const void* k_b,
                                  const void* v_b, const int* kv_pos, float* cos_out, int L, int H, int Hq, int Tq,
                                  int64_t T, DevErr err, cudaStream_t s, std::string* why) {
    Maps mp;
    const void* ks[2] = {k_a, k_b};
    const void* vs[2] = {v_a, v_b};
    for (int x = 0; x < 2; ++x) {
        if (!encode_cache(&mp.k[x], ks[x], static_cast<int64_t>(L) * H, T, 64, true, why) ||
            !encode_cache(&mp.v[x], vs[x], static_cast<int64_t>(L) * H, T, HD, false, why))
            return cudaErrorInvalidValue;
    }
    Params P{};
    P.q = static_cast<const __nv_bfloat16*>(q);
    P.q_pos = q_pos;
    P.kv_pos = kv_pos;
    P.cos_out = cos_out;
    P.L = L;
    P.H = H;
    P.Hq = Hq;
    P.Tq = Tq;
    P.T = static_cast<int>(T);
    P.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(HD));
    P.err = err;
    cudaError_t e = cudaFuncSetAttribute(attn_cosine_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int64_t rows = static_cast<int64_t>(Hq / H) * Tq;
    dim3 grid(static_cast<unsigned>((rows + TR - 1) / TR), static_cast<unsigned>(L * H));
    attn_cosine_tc_kernel<<<grid, NUM_THREADS, SMEM_BYTES, s>>>(mp, P);
    return cudaGetLastError();
}

}  // namespace kvb

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
// CTA per SM (all 512 TMEM columns).  The two caches run side by side, each
// with its own producer, MMA issuer and softmax warpgroup; for every 128-key
// tile that some row of the CTA may see (and always the first, whose copies
// start at entry):
//   warps 0, 1   TMA (cache a, b): the key tile and the value tile, each as two
//                64-wide 128-byte-swizzled boxes;
//   warps 2, 3   tcgen05.mma (cache a, b): S = Q K^T into TMEM (M 128, N 128,
//                K 128), then, once the probabilities are written,
//                O += P_hi V + P_lo V with V read MN-major straight from the
//                TMA tile;
//   warps 4..11 / 12..19  softmax of cache a / b, two threads per query row
//                (64 keys and 64 output dims each): S from TMEM (two passes:
//                the masked tile maximum, exchanged between the row's two
//                threads, then the probabilities), P as a bf16 pair (hi, lo:
//                ~16 significant bits) into shared memory in the operand
//                layout (hi over the consumed key tile).
// Exponentials are taken against a running reference maximum that is only
// raised (and O rescaled in TMEM) when a tile's maximum exceeds it by more than
// 2^8, so most tiles need no rescale; the softmax denominators cancel in the
// cosine, which is taken at the end straight from TMEM.  Every wait is bounded
// (DevErr); the softmax warps agree on a failed wait across the warp before
// leaving, so the warp-wide TMEM instructions are never divergent.
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
constexpr int NUM_THREADS = 640;
constexpr int MAX_FLAG_TILES = 1024;
constexpr int SMEM_BYTES = 7 * TILE + 1024 + 256 + MAX_FLAG_TILES;
constexpr uint64_t DRAIN_NS = 200ull * 1000 * 1000;
constexpr float RESCALE_LOG2 = 8.f;      // raise the reference maximum past this margin
// TMEM columns: S of cache x at 128 x, O of cache x at 256 + 128 x

struct Params {
    const __nv_bfloat16* q;  // [L][Hq][Tq][128]
    const int* q_pos;
    const int* kv_pos;
    float* cos_out;  // [L][Hq][Tq]
    int L, H, Hq, Tq, T;
    int kv_pos_vec;    // kv_pos is 16-byte aligned
    float scale_log2;  // log2(e) / sqrt(d)
    DevErr err;
};

struct Maps {
    CUtensorMap k[2], v[2];
    CUtensorMap q;  // queries as [L * Hq * Tq rows][128]
};

// Byte offset of 16-byte chunk c (0..15) of row r in a 128 x 128 bf16
// tile with the 128-byte swizzle (two 64-element blocks).
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
    return static_cast<uint32_t>((c >> 3) * ATOM + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint64_t desc_k(const uint8_t* tile, int kk) {  // 16-wide K step kk of 8
    return sdesc_k_sw128(smem_u32(tile) + (kk >> 2) * ATOM + (kk & 3) * 32);
}
// value tile [key][dim] as the MN-major B operand of O += P V: keys 16 kk .. 16 kk + 15
__device__ __forceinline__ uint64_t desc_v(const uint8_t* tile, int kk) {
    return sdesc_mn_sw128(smem_u32(tile) + kk * 16 * 128, ATOM);
}

// 2^x by the hardware approximation (relative error about 2^-22; subnormal results flush to 0)
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// positions of keys j .. j+3 (INT_MAX past the end)
__device__ __forceinline__ int4 key_pos4(const Params& P, int j) {
    if (P.kv_pos_vec && j + 3 < P.T) return __ldg(reinterpret_cast<const int4*>(P.kv_pos + j));
    int4 p = make_int4(INT_MAX, INT_MAX, INT_MAX, INT_MAX);
    if (j < P.T) p.x = __ldg(P.kv_pos + j);
    if (j + 1 < P.T) p.y = __ldg(P.kv_pos + j + 1);
    if (j + 2 < P.T) p.z = __ldg(P.kv_pos + j + 2);
    if (j + 3 < P.T) p.w = __ldg(P.kv_pos + j + 3);
    return p;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_cosine_tc_kernel(const __grid_constant__ Maps Mp, const __grid_constant__ Params P) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sQ = smem;
    // per cache x: key tile (then P hi), value tile, P lo
    auto sK = [&](int x) { return sQ + (1 + 3 * x) * TILE; };
    auto sV = [&](int x) { return sQ + (2 + 3 * x) * TILE; };
    auto sPl = [&](int x) { return sQ + (3 + 3 * x) * TILE; };
    uint64_t* bar = reinterpret_cast<uint64_t*>(sQ + 7 * TILE);
    uint64_t* kv_full = bar;       // [2]
    uint64_t* kv_empty = bar + 2;  // [2] committed after O += P V
    uint64_t* s_full = bar + 4;    // [2]
    uint64_t* p_full = bar + 6;    // [2]
    uint64_t* drain = bar + 8;     // [2]
    uint64_t* b_done = bar + 10;   // cache b's output is final
    uint64_t* q_full = bar + 11;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 12);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* qmax_s = reinterpret_cast<int*>(tmem_slot + 2);
    volatile int* b_ok = reinterpret_cast<volatile int*>(tmem_slot + 3);
    int* qmin_s = reinterpret_cast<int*>(tmem_slot + 4);
    uint8_t* flags = reinterpret_cast<uint8_t*>(bar) + 256;

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
        for (int x = 0; x < 2; ++x) {
            mbar_init(&kv_full[x], 1);
            mbar_init(&kv_empty[x], 1);
            mbar_init(&s_full[x], 1);
            mbar_init(&p_full[x], 256);
            mbar_init(&drain[x], 1);
        }
        mbar_init(b_done, 256);
        mbar_init(q_full, 1);
        *abort_flag = 0;
        *qmax_s = INT_MIN;
        *qmin_s = INT_MAX;
        *b_ok = 0;
        fence_mbar_init();
        // the CTA's 128 query rows are consecutive rows of the [L * Hq * Tq][128] view
        // (the Hq / H heads of KV head kh are adjacent); rows past the group are loaded
        // but never used
        const int qrow0 = (l * P.Hq + kh * g) * P.Tq + r0;
        mbar_arrive_expect_tx(q_full, TILE);
        tma_load_2d(sQ, &Mp.q, q_full, 0, qrow0);
        tma_load_2d(sQ + ATOM, &Mp.q, q_full, 64, qrow0);
        // key tile 0 counts as live for every row block (a tile that no row sees only
        // adds zero probabilities), so both caches' first key and value tiles are copied
        // now, while TMEM is allocated and the other tiles are flagged
        for (int x = 0; x < 2; ++x) {
            mbar_arrive_expect_tx(&kv_full[x], 2 * TILE);
            tma_load_3d(sK(x), &Mp.k[x], &kv_full[x], 0, 0, slab);
            tma_load_3d(sK(x) + ATOM, &Mp.k[x], &kv_full[x], 64, 0, slab);
            tma_load_3d(sV(x), &Mp.v[x], &kv_full[x], 0, 0, slab);
            tma_load_3d(sV(x) + ATOM, &Mp.v[x], &kv_full[x], 64, 0, slab);
        }
    }
    if (warp == 2) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    __syncthreads();

    // the rows' positions and the CTA's smallest and largest
    const int gx = (warp - 4) >> 3;          // softmax warps: cache index
    const int hf = ((warp - 4) >> 2) & 1;    // softmax warps: which 64 keys / output dims of the row
    const int row = 32 * (warp & 3) + lane;  // softmax warps: TMEM lane = tile row
    const int grow = r0 + row;
    const bool valid = warp >= 4 && grow < rows;
    const int qp = valid ? __ldg(P.q_pos + grow % P.Tq) : INT_MIN;
    if (valid && gx == 0 && hf == 0) {
        atomicMax(qmax_s, qp);
        atomicMin(qmin_s, qp);
    }
    __syncthreads();
    // per key tile: 0 no row of the CTA sees a key of it (skipped by every role
    // alike), 2 every row sees every key of it (no per-key test), 1 otherwise
    if (use_flags) {
        const int qmax = *qmax_s, qmin = *qmin_s;
        for (int t = warp; t < ntiles; t += NUM_THREADS / 32) {
            const int4 p4 = key_pos4(P, t * TK + 4 * lane);
            const bool any = __any_sync(0xffffffffu, p4.x <= qmax || p4.y <= qmax || p4.z <= qmax || p4.w <= qmax);
            const bool all = __all_sync(0xffffffffu, p4.x <= qmin && p4.y <= qmin && p4.z <= qmin && p4.w <= qmin) &&
                             (t + 1) * TK <= P.T;
            if (lane == 0) flags[t] = all ? 2 : (any ? 1 : 0);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    auto live = [&](int t) { return t == 0 || !use_flags || flags[t] != 0; };

    if (warp < 2) {
        if (lane == 0) {
            // ------------------------------------------------------- producer, cache x
            const int x = warp;
            int it = 0, last = -1;
            for (int t = 0; t < ntiles; ++t) {
                if (!live(t)) continue;
                if (t == 0) {  // copied at entry
                    last = it++;
                    continue;
                }
                if (!mbar_wait(&kv_empty[x], (it & 1) ^ 1u, P.err, abort_flag)) break;
                mbar_arrive_expect_tx(&kv_full[x], 2 * TILE);
                tma_load_3d(sK(x), &Mp.k[x], &kv_full[x], 0, t * TK, slab);
                tma_load_3d(sK(x) + ATOM, &Mp.k[x], &kv_full[x], 64, t * TK, slab);
                tma_load_3d(sV(x), &Mp.v[x], &kv_full[x], 0, t * TK, slab);
                tma_load_3d(sV(x) + ATOM, &Mp.v[x], &kv_full[x], 64, t * TK, slab);
                last = it++;
            }
            if (last >= 0) mbar_wait_drain(&kv_full[x], static_cast<uint32_t>(last & 1), DRAIN_NS);
            if (x == 0) mbar_wait_drain(q_full, 0, DRAIN_NS);  // the query copy issued at entry
        }
    } else if (warp < 4) {
        if (lane == 0) {
            // ------------------------------------------------------- MMA issuer, cache x
            const int x = warp - 2;
            constexpr uint32_t idesc_s = idesc_bf16_f32(TR, TK);
            constexpr uint32_t idesc_o = idesc_bf16_f32(TR, HD) | IDESC_B_MN;
            const uint32_t tS = tmem_base + 128u * x, tO = tmem_base + 256u + 128u * x;
            int it = 0;
            const bool have_q = mbar_wait(q_full, 0, P.err, abort_flag);
            for (int t = 0; have_q && t < ntiles; ++t) {
                if (!live(t)) continue;
                if (!mbar_wait(&kv_full[x], it & 1, P.err, abort_flag)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) umma_bf16(tS, desc_k(sQ, kk), desc_k(sK(x), kk), idesc_s, kk != 0);
                umma_commit(&s_full[x]);
                if (!mbar_wait(&p_full[x], it & 1, P.err, abort_flag)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < TK / 16; ++kk)
                    umma_bf16(tO, desc_k(sK(x), kk), desc_v(sV(x), kk), idesc_o, (it | kk) != 0);
#pragma unroll
                for (int kk = 0; kk < TK / 16; ++kk) umma_bf16(tO, desc_k(sPl(x), kk), desc_v(sV(x), kk), idesc_o, 1);
                umma_commit(&kv_empty[x]);  // tiles consumed and O updated
                ++it;
            }
            umma_commit(&drain[x]);  // every MMA issued here completes before TMEM is released
            mbar_wait_drain(&drain[x], 0, DRAIN_NS);
        }
    } else {
        // ----------------------------------------------------------- softmax, cache gx
        // Two threads per row (warps w and w + 4 share a TMEM lane quarter): this one
        // takes keys kh0 .. kh0+63 of every tile and output dims kh0 .. kh0+63.  The two
        // halves exchange tile maxima (and, at the end, the cosine's sums) through the
        // cache's P-lo tile, which no MMA reads at those points.  A thread's maximum goes
        // into the first 16 bytes of its partner's own P-lo chunks of the row: the partner
        // reads it before its pass 2 overwrites them, and the next maximum is written
        // only once the next S is ready, after O += P V has read P lo.  The eight warps of a
        // cache meet at named barrier 1 + x; whether to go on is agreed there first
        // (every wait before it is bounded), so no warp leaves while others wait.
        const int x = gx;
        const int kh0 = 64 * hf;
        const int bar_id = 1 + x;
        const uint32_t tl = tmem_base + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
        const uint32_t cS = 128u * x + kh0, cO = 256u + 128u * x + kh0;
        float* xch = reinterpret_cast<float*>(sPl(x));  // [3][128] cosine-sum slots (at the end)
        float* slot_in = reinterpret_cast<float*>(sPl(x) + sw_off(row, 8 * hf));         // the partner's maximum
        float* slot_out = reinterpret_cast<float*>(sPl(x) + sw_off(row, 8 * (1 - hf)));  // this thread's
        auto wait_all = [&](uint64_t* b, uint32_t parity) {  // warp-uniform outcome
            const bool got = mbar_wait(b, parity, P.err, abort_flag);
            return __all_sync(0xffffffffu, got);
        };
        float m_ref = -INFINITY;  // reference maximum of this row (base 2)
        int it = 0;
        bool ok = true;
        for (int t = 0; t < ntiles; ++t) {
            if (!live(t)) continue;
            const int j0 = t * TK + kh0;
            // visibility of this thread's 64 keys, while the MMA computes S:
            // bit u of vis[w] is key j0 + 32 w + u
            uint32_t vis[2] = {0u, 0u};
            if (use_flags && flags[t] == 2) {
                if (valid) vis[0] = vis[1] = 0xffffffffu;
            } else {
#pragma unroll
                for (int u = 0; u < 64; u += 4) {
                    const int4 p4 = key_pos4(P, j0 + u);
                    const int pa[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
                    for (int w = 0; w < 4; ++w)
                        // positions past the end are INT_MAX; a query at INT_MAX is
                        // excluded from them by the index test
                        if (valid && pa[w] <= qp && j0 + u + w < P.T) vis[u >> 5] |= 1u << ((u + w) & 31);
                }
            }
            ok = named_bar_and(bar_id, 256, wait_all(&s_full[x], it & 1));
            if (!ok) break;
            tc_fence_after();
            // pass 1: the masked maximum of this half row
            float mt = -INFINITY;
#pragma unroll 1
            for (int c0 = 0; c0 < 64; c0 += 32) {
                uint32_t sv[2][16];
                tmem_ld16(tl + cS + c0, sv[0]);
                tmem_ld16(tl + cS + c0 + 16, sv[1]);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const int kk = c0 + 16 * c + u;
                        if ((vis[kk >> 5] >> (kk & 31)) & 1u) mt = fmaxf(mt, __uint_as_float(sv[c][u]));
                    }
            }
            *slot_out = mt;
            named_bar_sync(bar_id, 256);
            mt = fmaxf(mt, *slot_in) * P.scale_log2;  // scale > 0: commutes with the maximum
            const bool raise = mt > m_ref + RESCALE_LOG2;  // also the first visible tile of the row
            if (__any_sync(0xffffffffu, raise && it > 0 && m_ref > -INFINITY)) {
                // O was accumulated against the old reference: rescale this half in TMEM
                const float f = (raise && m_ref > -INFINITY) ? ex2_approx(m_ref - mt) : 1.f;
#pragma unroll 1
                for (int c0 = 0; c0 < 64; c0 += 16) {
                    uint32_t o[16];
                    tmem_ld16(tl + cO + c0, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int u = 0; u < 16; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * f);
                    tmem_st16(tl + cO + c0, o);
                }
                tmem_st_wait();
            }
            if (raise) m_ref = mt;
            // pass 2: probabilities as bf16 (hi, lo) in the operand layout; keys that every
            // row of the warp sees need no per-key test
            const bool all_vis = __all_sync(0xffffffffu, (vis[0] & vis[1]) == 0xffffffffu);
#pragma unroll 1
            for (int c0 = 0; c0 < 64; c0 += 32) {
                uint32_t sv[2][16];
                tmem_ld16(tl + cS + c0, sv[0]);
                tmem_ld16(tl + cS + c0 + 16, sv[1]);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    float p[16];
                    if (all_vis) {
#pragma unroll
                        for (int u = 0; u < 16; ++u)
                            p[u] = ex2_approx(fmaf(__uint_as_float(sv[c][u]), P.scale_log2, -m_ref));
                    } else {
#pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            const int kk = c0 + 16 * c + u;
                            p[u] = ((vis[kk >> 5] >> (kk & 31)) & 1u)
                                       ? ex2_approx(fmaf(__uint_as_float(sv[c][u]), P.scale_log2, -m_ref))
                                       : 0.f;
                        }
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
                        const uint32_t off = sw_off(row, ((kh0 + c0) >> 3) + 2 * c + h);
                        *reinterpret_cast<uint4*>(sK(x) + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        *reinterpret_cast<uint4*>(sPl(x) + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&p_full[x]);
            ++it;
        }
        // the cache's last O += P V is complete (every warp waits; the outcome is agreed below)
        bool fin = ok && (it == 0 || wait_all(&kv_empty[x], static_cast<uint32_t>((it - 1) & 1)));
        if (x == 1) {
            fin = named_bar_and(bar_id, 256, fin);
            if (fin && lane == 0 && warp == 12) *b_ok = 1;  // read by cache a's warps after b_done
            __syncwarp();
            tc_fence_before();
            mbar_arrive(b_done);  // also on failure, so that cache a's warps do not wait it out
        } else {
            fin = fin && wait_all(b_done, 0);
            fin = named_bar_and(bar_id, 256, fin && *b_ok);
            if (fin) {
                tc_fence_after();
                float dot = 0.f, na = 0.f, nb = 0.f;
                if (it > 0) {
#pragma unroll 1
                    for (int c0 = 0; c0 < 64; c0 += 16) {
                        uint32_t oa[16], ob[16];
                        tmem_ld16(tl + 256u + kh0 + c0, oa);
                        tmem_ld16(tl + 384u + kh0 + c0, ob);
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
                // the upper half's sums to the lower half (the P-lo tile is idle now)
                if (hf == 1) {
                    xch[row] = dot;
                    xch[128 + row] = na;
                    xch[256 + row] = nb;
                }
                named_bar_sync(bar_id, 256);
                if (hf == 0 && valid) {
                    dot += xch[row];
                    na += xch[128 + row];
                    nb += xch[256 + row];
                    const float den = sqrtf(na) * sqrtf(nb);
                    const int hq = kh * g + grow / P.Tq;
                    const int64_t oi = (static_cast<int64_t>(l) * P.Hq + hq) * P.Tq + grow % P.Tq;
                    if (KVB_IN_BOUNDS(P.err, oi, 1, static_cast<int64_t>(P.L) * P.Hq * P.Tq))
                        P.cos_out[oi] = den > 0.f ? dot / den : 0.f;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
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

bool attn_tc_supported(kvb_dtype dtype, int d, int64_t T, int64_t q_rows) {
    return dtype == KVB_BF16 && d == HD && T >= 1 && T <= 0x7fffffffLL && q_rows <= 0x7fffffffLL;
}

cudaError_t launch_attn_cosine_tc(const void* q, const int* q_pos, const void* k_a, const void* v_a, const void* k_b,
                                  const void* v_b, const int* kv_pos, float* cos_out, int L, int H, int Hq, int Tq,
                                  int64_t T, DevErr err, cudaStream_t s, std::string* why) {
    Maps mp;
    {
        EncodeTiledFn enc = get_encode_tiled();
        if (!enc) {
            if (why) *why = "cuTensorMapEncodeTiled unavailable from the driver";
            return cudaErrorInvalidValue;
        }
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(L) * Hq * Tq};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(HD) * 2};
        cuuint32_t box[2] = {64, static_cast<cuuint32_t>(TR)};
        cuuint32_t estr[2] = {1, 1};
        CUresult r = enc(&mp.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            if (why) *why = "cuTensorMapEncodeTiled (queries) failed with code " + std::to_string(static_cast<int>(r));
            return cudaErrorInvalidValue;
        }
    }
    const void* ks[2] = {k_a, k_b};
    const void* vs[2] = {v_a, v_b};
    for (int x = 0; x < 2; ++x) {
        if (!encode_cache(&mp.k[x], ks[x], static_cast<int64_t>(L) * H, T, 64, true, why) ||
            !encode_cache(&mp.v[x], vs[x], static_cast<int64_t>(L) * H, T, 64, true, why))
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
    P.kv_pos_vec = (reinterpret_cast<uintptr_t>(kv_pos) & 15u) == 0;
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

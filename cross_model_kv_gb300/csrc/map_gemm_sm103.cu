// Mapper apply on the 5th-generation tensor cores (sm_103a).
//
// For every target layer t and kv in {K, V}:
//     Y = X_t . W_t^T,   X_t[token][(j*H + h)*d + e] = A_kv[sel[kv][t][j]][h][token][e]
// ("Cross-Model KV Transfer" (VeloxQuant-MLX), "The mapping"; the features are
// the top-k selected source layers across all KV heads, "KVBridge", "What
// ships").  The feature matrix is never materialised: each 64-wide K-block of
// X_t is one token-block x 64-dim box of one (layer, head) slab of the source
// cache, fetched by TMA at coordinates (e0, token0, sel*H + h).  For K the
// source operand is the RoPE-stripped copy of the keys, which the kernel's own
// epilogue warps write while the value tiles run (or a separate strip pass).
//
// Two persistent, warp-specialised kernels share the epilogue:
//   map_gemm_pair_kernel clusters of 2 CTAs on 2 SMs, tiles of 256 tokens x
//                        256 outputs, tcgen05.mma cta_group::2 (M=256 N=256):
//                        each CTA stages its own 128 token rows and half of
//                        the 256 output rows of W, so a stage is 32 KB per SM
//                        instead of 48 KB and six stages fit instead of four;
//                        tiles are claimed in order from a global counter.
//                        The default.
//   map_gemm_kernel      one CTA per SM, tiles of 128 tokens x 256 outputs,
//                        tcgen05.mma cta_group::1 (M=128 N=256 K=16), tiles
//                        assigned round-robin; with KVB_MAP_PAIR=0.
// Roles: warp 0 TMA producer (one lane), warp 1 MMA issuer (one lane; in the
// pair kernel only the even CTA issues), warps 2..5 epilogue: TMEM ->
// registers, + bias, target RoPE for K (pairs (e, e+64) of one head are in the
// same tile), round to bf16, store straight into the target cache
// [t][h][token][e].  Accumulators are double buffered in TMEM (2 x 256 columns).
// fp32 caches run through the same kernels with each operand carried as a
// bf16 (hi, lo) pair and an fp32 output (SPLIT = true).
// Every wait is bounded (DevErr::timeout_ns); on expiry the CTA records
// DEV_ERR_TIMEOUT, stops, drains its copies and MMAs and frees TMEM.
#include <cstdlib>
#include <cstring>

#include "kvb_internal.h"

namespace kvb {

namespace {

constexpr int BN = 256;  // outputs per tile (two heads of 128)
constexpr int BK = 64;   // one 128-byte swizzle atom of bf16
constexpr int NUM_THREADS = 192;
constexpr int TMEM_COLS = 512;
constexpr uint64_t DRAIN_NS = 200ull * 1000 * 1000;

// single-CTA kernel
constexpr int BM = 128;
#ifndef KVB_MAP_STAGES
#define KVB_MAP_STAGES 4
#endif
constexpr int STAGES = KVB_MAP_STAGES;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;

// CTA-pair kernel: per CTA 128 token rows and 128 of the 256 output rows
constexpr int PM = 256;
#ifndef KVB_MAP_PAIR_STAGES
#define KVB_MAP_PAIR_STAGES 6
#endif
constexpr int PSTAGES = KVB_MAP_PAIR_STAGES;
constexpr int PA_BYTES = 128 * BK * 2;
constexpr int PB_BYTES = 128 * BK * 2;
constexpr int PSTAGE_BYTES = PA_BYTES + PB_BYTES;
constexpr int PSMEM_BYTES = PSTAGES * PSTAGE_BYTES + 1024 + 512;

struct Params {
    int L_t, H, d, T, num_m, num_n, nk, total_tiles, max_pos;
    const int* pos;
    const float* bias[2];
    void* out[2];          // bf16, or fp32 for the split (fp32-operand) kernel
    const float2* tab_t;
    DevErr err;
    SelTable sel;
    // strip fused into the kernel (bf16 single-CTA kernel): value tiles run
    // first while the epilogue warps strip the source keys chunk by chunk
    int fuse_strip;
    const __nv_bfloat16* k_raw;  // [L_s*H][T][d] source keys as stored
    __nv_bfloat16* k_strip;      // same layout, stripped: the key tiles' A operand
    const float2* tab_s;
    int* strip_ctr;              // [0] next chunk to claim, [1] chunks finished
    int strip_chunks;            // chunks of 128 tokens per (layer, head) slab
    int strip_items;             // all chunks
    int* tile_ctr;               // CTA-pair kernel: next tile to claim (zeroed before the launch), or null
};

struct TileCoord {
    int kv, t, m, n;
};

__device__ __forceinline__ TileCoord decode_tile(const Params& P, int tile) {
    TileCoord c;
    c.n = tile % P.num_n;
    int r = tile / P.num_n;
    c.m = r % P.num_m;
    r /= P.num_m;
    c.t = r % P.L_t;
    c.kv = r / P.L_t;
    if (P.fuse_strip) c.kv = 1 - c.kv;  // value tiles first: their operand needs no strip
    return c;
}

// One warp strips 128 tokens of one (layer, head) slab of the source keys:
// eight lanes per row, each owning 8 RoPE pairs (two 16-byte loads and stores,
// the (cos, sin) of its pairs from the table), rotation by -angle.  A position
// outside the table is recorded and its row written as zeros.
__device__ __forceinline__ void strip_chunk(const Params& P, int item, int lane) {
    const int slab = item / P.strip_chunks;
    const int t0 = (item - slab * P.strip_chunks) * 128;
    const int half = P.d >> 1;
    const int c8 = (lane & 7) * 8;  // first pair of this lane
#pragma unroll 2
    for (int r = lane >> 3; r < 128; r += 4) {
        const int tok = t0 + r;
        if (tok >= P.T) break;
        const int64_t o = (static_cast<int64_t>(slab) * P.T + tok) * P.d + c8;
        const int64_t strip_size = static_cast<int64_t>(P.strip_items / P.strip_chunks) * P.T * P.d;
        if (!KVB_IN_BOUNDS(P.err, o, 8, strip_size) || !KVB_IN_BOUNDS(P.err, o + half, 8, strip_size)) continue;
        const int p = __ldg(P.pos + tok);
        uint4 olo = make_uint4(0, 0, 0, 0), ohi = make_uint4(0, 0, 0, 0);
        if (p < 0 || p >= P.max_pos) {
            dev_err_set(P.err, DEV_ERR_BAD_POS);
        } else {
            const uint4 vlo = __ldcs(reinterpret_cast<const uint4*>(P.k_raw + o));
            const uint4 vhi = __ldcs(reinterpret_cast<const uint4*>(P.k_raw + o + half));
            const float4* tp = reinterpret_cast<const float4*>(P.tab_s + static_cast<int64_t>(p) * half + c8);
            const __nv_bfloat162* lo2 = reinterpret_cast<const __nv_bfloat162*>(&vlo);
            const __nv_bfloat162* hi2 = reinterpret_cast<const __nv_bfloat162*>(&vhi);
            uint32_t wl[4], wh[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 cs = __ldg(tp + q);  // (c, s) of pairs 2q and 2q+1
                const float2 l = __bfloat1622float2(lo2[q]);
                const float2 h = __bfloat1622float2(hi2[q]);
                wl[q] = pack_bf16x2(fmaf(l.x, cs.x, h.x * cs.y), fmaf(l.y, cs.z, h.y * cs.w));
                wh[q] = pack_bf16x2(fmaf(h.x, cs.x, -(l.x * cs.y)), fmaf(h.y, cs.z, -(l.y * cs.w)));
            }
            olo = make_uint4(wl[0], wl[1], wl[2], wl[3]);
            ohi = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        }
        *reinterpret_cast<uint4*>(P.k_strip + o) = olo;
        *reinterpret_cast<uint4*>(P.k_strip + o + half) = ohi;
    }
}

// Producer, before the first key tile: every chunk of the stripped keys has been
// written (by any CTA), bounded like every other wait; then the TMA loads see the
// generic-proxy writes.  False on timeout or abort.
__device__ __forceinline__ bool wait_strip_done(const Params& P, volatile int* abort_flag) {
    const uint64_t t0 = global_timer_ns();
    while (ld_acquire_gpu(P.strip_ctr + 1) < P.strip_items) {
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > P.err.timeout_ns) {
            dev_err_set(P.err, DEV_ERR_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
        __nanosleep(256);
    }
    fence_proxy_async_global();
    return true;
}

// Epilogue warp: while the accumulator is not ready, strip chunks of the source
// keys.  Returns false once no chunk is left to claim (warp-uniform).
__device__ __forceinline__ bool strip_while_waiting(const Params& P, uint64_t* tfull, uint32_t parity, int lane,
                                                    volatile int* abort_flag) {
    while (!__any_sync(0xffffffffu, mbar_try_wait(tfull, parity))) {
        int item = 0;
        if (lane == 0) item = *abort_flag ? P.strip_items : atomicAdd(P.strip_ctr, 1);
        item = __shfl_sync(0xffffffffu, item, 0);
        if (item >= P.strip_items) return false;
        strip_chunk(P, item, lane);
        fence_proxy_async_global();  // for the TMA loads of other CTAs
        __syncwarp();
        if (lane == 0) {
            __threadfence();  // the warp's stores before the count (release)
            atomicAdd(P.strip_ctr + 1, 1);
        }
    }
    return true;
}

// K-block kb of target layer t: (source layer, head, first dim) of its box.
// Source of consecutive K blocks of one (kv, target layer) problem: feature
// (j * H + h) * d + e is dim e of head h of the j-th selected source layer.  The
// producer steps it BK features at a time (BK divides d), without divisions.
struct KSrc {
    int j, h, e0, slab;  // slab: the source layer's first (layer, head) slab
    __device__ __forceinline__ void start(const Params& P, int kv, int t) {
        j = h = e0 = 0;
        slab = P.sel.s[kv][t][0] * P.H;
    }
    __device__ __forceinline__ void next(const Params& P, int kv, int t) {
        e0 += BK;
        if (e0 == P.d) {
            e0 = 0;
            if (++h == P.H) {
                h = 0;
                ++j;
                slab = P.sel.s[kv][t][j < MAX_K ? j : MAX_K - 1] * P.H;  // past the last: never used
            }
        }
    }
};

// One thread's row of one accumulator tile (256 columns = two heads): bias,
// target RoPE for keys, bf16 rounding (or fp32 as is), store into [t][h][tok][e].
template <bool F32OUT>
__device__ __forceinline__ void epilogue_row(const Params& P, const TileCoord& c, int tok, uint32_t tbase, int q) {
    const bool valid = tok < P.T;
    int p = valid ? __ldg(P.pos + tok) : 0;
    bool bad_pos = false;
    if (valid && (p < 0 || p >= P.max_pos)) {  // recorded; the row is written as zeros
        dev_err_set(P.err, DEV_ERR_BAD_POS);
        bad_pos = true;
        p = 0;
    }
    const int half = P.d >> 1;  // 64
    const int heads_per_tile = BN / P.d;
    const float* bias = P.bias[c.kv] + static_cast<int64_t>(c.t) * q + c.n * BN;
    const float2* tab = P.tab_t + static_cast<int64_t>(p) * half;
    // 16 RoPE pairs at a time; their (cos, sin) serve every head of the tile
#pragma unroll 1
    for (int e0 = 0; e0 < half; e0 += 16) {
        float4 cs[8];
        if (c.kv == 0) {
            const float4* tp = reinterpret_cast<const float4*>(tab + e0);
#pragma unroll
            for (int v = 0; v < 8; ++v) cs[v] = __ldg(tp + v);  // (c, s) of pairs 2v and 2v+1
        }
#pragma unroll 1
        for (int hh = 0; hh < heads_per_tile; ++hh) {
            const int h = c.n * heads_per_tile + hh;
            const int64_t orow = ((static_cast<int64_t>(c.t) * P.H + h) * P.T + tok) * P.d;
            // checked build: the bias reads and the row's stores stay inside their
            // buffers (the TMEM loads below are warp-wide and always run)
            const int64_t out_size = static_cast<int64_t>(P.L_t) * P.H * P.T * P.d;
            const int64_t boff = static_cast<int64_t>(c.t) * q + c.n * BN + hh * P.d + e0;
            const bool inb = KVB_IN_BOUNDS(P.err, boff, 16, static_cast<int64_t>(P.L_t) * q) &&
                             KVB_IN_BOUNDS(P.err, boff + half, 16, static_cast<int64_t>(P.L_t) * q) &&
                             (!valid || (KVB_IN_BOUNDS(P.err, orow + e0, 16, out_size) &&
                                         KVB_IN_BOUNDS(P.err, orow + half + e0, 16, out_size)));
            uint32_t lo[16], hi[16];
            tmem_ld16(tbase + hh * P.d + e0, lo);
            tmem_ld16(tbase + hh * P.d + half + e0, hi);
            tmem_ld_wait();
            float xl[16], xh[16];
            const float4* bl = reinterpret_cast<const float4*>(bias + hh * P.d + e0);
            const float4* bh = reinterpret_cast<const float4*>(bias + hh * P.d + half + e0);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const float4 a = inb ? __ldg(bl + v) : make_float4(0.f, 0.f, 0.f, 0.f);
                const float4 b = inb ? __ldg(bh + v) : make_float4(0.f, 0.f, 0.f, 0.f);
                xl[4 * v + 0] = __uint_as_float(lo[4 * v + 0]) + a.x;
                xl[4 * v + 1] = __uint_as_float(lo[4 * v + 1]) + a.y;
                xl[4 * v + 2] = __uint_as_float(lo[4 * v + 2]) + a.z;
                xl[4 * v + 3] = __uint_as_float(lo[4 * v + 3]) + a.w;
                xh[4 * v + 0] = __uint_as_float(hi[4 * v + 0]) + b.x;
                xh[4 * v + 1] = __uint_as_float(hi[4 * v + 1]) + b.y;
                xh[4 * v + 2] = __uint_as_float(hi[4 * v + 2]) + b.z;
                xh[4 * v + 3] = __uint_as_float(hi[4 * v + 3]) + b.w;
            }
            if (c.kv == 0) {
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    const float l0 = xl[2 * v], h0 = xh[2 * v];
                    const float l1 = xl[2 * v + 1], h1 = xh[2 * v + 1];
                    xl[2 * v] = fmaf(l0, cs[v].x, -(h0 * cs[v].y));
                    xh[2 * v] = fmaf(h0, cs[v].x, l0 * cs[v].y);
                    xl[2 * v + 1] = fmaf(l1, cs[v].z, -(h1 * cs[v].w));
                    xh[2 * v + 1] = fmaf(h1, cs[v].z, l1 * cs[v].w);
                }
            }
            if (valid && inb && F32OUT) {
                float* o = static_cast<float*>(P.out[c.kv]) + orow;
#pragma unroll
                for (int v = 0; v < 2; ++v) {  // 8 outputs = one 32-byte sector per store
                    uint32_t a[8], b[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        a[u] = bad_pos ? 0u : __float_as_uint(xl[8 * v + u]);
                        b[u] = bad_pos ? 0u : __float_as_uint(xh[8 * v + u]);
                    }
                    st_global_v8(o + e0 + 8 * v, a);
                    st_global_v8(o + half + e0 + 8 * v, b);
                }
            } else if (valid && inb) {
                __nv_bfloat16* o = static_cast<__nv_bfloat16*>(P.out[c.kv]) + orow;
                uint32_t pl[8], ph[8];
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    pl[v] = bad_pos ? 0u : pack_bf16x2(xl[2 * v], xl[2 * v + 1]);
                    ph[v] = bad_pos ? 0u : pack_bf16x2(xh[2 * v], xh[2 * v + 1]);
                }
                st_global_v8(o + e0, pl);  // 16 outputs = one 32-byte sector
                st_global_v8(o + half + e0, ph);
            }
        }
    }
}

// ============================================================ single CTA
// SPLIT: the operands are fp32 values carried as bf16 (hi, lo) pairs; each
// 64-wide K block is issued three times (A hi x W hi, A hi x W lo, A lo x W
// hi) into the same accumulator and the output is fp32.
template <bool SPLIT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    map_gemm_kernel(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_a1,
                    const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                    const __grid_constant__ CUtensorMap tm_a0l, const __grid_constant__ CUtensorMap tm_a1l,
                    const __grid_constant__ CUtensorMap tm_w0l, const __grid_constant__ CUtensorMap tm_w1l,
                    const __grid_constant__ Params P) {
    constexpr int NSEG = SPLIT ? 3 : 1;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_a0);
        tma_prefetch_desc(&tm_a1);
        tma_prefetch_desc(&tm_w0);
        tma_prefetch_desc(&tm_w1);
        if (SPLIT) {
            tma_prefetch_desc(&tm_a0l);
            tma_prefetch_desc(&tm_a1l);
            tma_prefetch_desc(&tm_w0l);
            tma_prefetch_desc(&tm_w1l);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int q = P.H * P.d;
    const int nk_issue = P.nk * NSEG;  // K blocks issued per tile

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------- producer
            int stage = 0;
            uint32_t phase = 0;
            int issued_phase[STAGES];
            for (int s = 0; s < STAGES; ++s) issued_phase[s] = -1;
            bool ok = true;
            bool stripped = !P.fuse_strip;
            for (int tile = blockIdx.x; ok && tile < P.total_tiles; tile += gridDim.x) {
                const TileCoord c = decode_tile(P, tile);
                if (c.kv == 0 && !stripped) {
                    if (!wait_strip_done(P, abort_flag)) break;
                    stripped = true;
                }
                KSrc src;
                src.start(P, c.kv, c.t);
                int kb = 0, seg = 0;  // seg 0: hi x hi, 1: hi x lo, 2: lo x hi
                for (int ki = 0; ki < nk_issue; ++ki) {
                    const CUtensorMap* ta = seg == 2 ? (c.kv ? &tm_a1l : &tm_a0l) : (c.kv ? &tm_a1 : &tm_a0);
                    const CUtensorMap* tw = seg == 1 ? (c.kv ? &tm_w1l : &tm_w0l) : (c.kv ? &tm_w1 : &tm_w0);
                    if (!mbar_wait(&empty[stage], phase ^ 1u, P.err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
                    tma_load_3d(sA + stage * A_BYTES, ta, &full[stage], src.e0, c.m * BM, src.slab + src.h);
                    tma_load_3d(sB + stage * B_BYTES, tw, &full[stage], kb * BK, c.n * BN, c.t);
                    if (!SPLIT || seg == 2) {
                        src.next(P, c.kv, c.t);
                        ++kb;
                        seg = 0;
                    } else {
                        ++seg;
                    }
                    issued_phase[stage] = static_cast<int>(phase);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Never leave the CTA with a copy still landing in its shared memory.
            for (int s = 0; s < STAGES; ++s)
                if (issued_phase[s] >= 0) mbar_wait_drain(&full[s], static_cast<uint32_t>(issued_phase[s]), DRAIN_NS);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------------------------------------------- MMA issuer
            constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < P.total_tiles; tile += gridDim.x) {
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, P.err, abort_flag)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < nk_issue; ++kb) {
                    if (!mbar_wait(&full[stage], phase, P.err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + stage * A_BYTES);
                    const uint32_t b0 = smem_u32(sB + stage * B_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        umma_bf16(d_tmem, sdesc_k_sw128(a0 + k * 32), sdesc_k_sw128(b0 + k * 32), idesc,
                                  (kb | k) != 0);
                    }
                    umma_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(&tfull[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            // All MMAs issued by this thread complete before TMEM is released.
            umma_commit(drain);
            mbar_wait_drain(drain, 0, DRAIN_NS);
        }
    } else {
        // -------------------------------------------------------- epilogue
        const int sub = warp & 3;  // TMEM lane quarter this warp may access
        const int row = sub * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool strip_left = P.fuse_strip != 0;  // warp-uniform
        for (int tile = blockIdx.x; tile < P.total_tiles; tile += gridDim.x) {
            const TileCoord c = decode_tile(P, tile);
            if (strip_left) strip_left = strip_while_waiting(P, &tfull[acc], acc_phase, lane, abort_flag);
            if (!mbar_wait(&tfull[acc], acc_phase, P.err, abort_flag)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(sub * 32) << 16) + static_cast<uint32_t>(acc * BN);
            epilogue_row<SPLIT>(P, c, c.m * BM + row, tbase, q);
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ============================================================ CTA pair
// Cluster of two CTAs (ranks 0 and 1).  Tile (kv, t, m, n) covers tokens
// [256m, 256m + 256) and outputs [256n, 256n + 256); CTA r stages tokens
// 256m + 128r .. +128 (A) and outputs 256n + 128r .. +128 (B) and owns the
// accumulator rows of its tokens.  Both CTAs' copies complete on rank 0's
// `full` barrier; rank 0 issues the pair MMAs and commits to both CTAs'
// `empty` / `tfull` barriers; both CTAs' epilogues arrive on rank 0's `tempty`.
//
// Tiles are handed out in index order from a global counter (P.tile_ctr):
// rank 0's producer claims the next tile and passes its index through a ring
// of PRING slots in both CTAs' shared memory (sfull / sempty barriers) to the
// MMA issuer, both epilogues and rank 1's producer.  The four tiles of one
// token block (consecutive indices) therefore start together on four pairs,
// which read the block's source rows while they are in L2; a fixed
// tile-per-pair assignment lets the pairs drift apart by several tiles over a
// launch and re-read them from DRAM.  With tile_ctr == nullptr the same ring
// carries the fixed assignment pair, pair + npairs, ...
constexpr int PRING = 4;
constexpr int SCHED_CONSUMERS = 1 + 4 + 1 + 4;  // MMA, epilogue warps of rank 0, producer and epilogue warps of rank 1

// SPLIT as in the single-CTA kernel: fp32 operands as bf16 (hi, lo) pairs, three
// products per 64-wide K block, fp32 output.
template <bool SPLIT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    map_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_a1,
                         const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                         const __grid_constant__ CUtensorMap tm_a0l, const __grid_constant__ CUtensorMap tm_a1l,
                         const __grid_constant__ CUtensorMap tm_w0l, const __grid_constant__ CUtensorMap tm_w1l,
                         const __grid_constant__ Params P) {
    constexpr int NSEG = SPLIT ? 3 : 1;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sA = smem;
    uint8_t* sB = smem + PSTAGES * PA_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + PSTAGES * PSTAGE_BYTES);
    uint64_t* empty = full + PSTAGES;
    uint64_t* tfull = empty + PSTAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint64_t* sfull = drain + 1;
    uint64_t* sempty = sfull + PRING;
    volatile int* ring = reinterpret_cast<volatile int*>(sempty + PRING);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(const_cast<int*>(ring + PRING));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < PSTAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 2 * 128);
        }
        mbar_init(drain, 1);
        for (int r = 0; r < PRING; ++r) {
            mbar_init(&sfull[r], 1);
            mbar_init(&sempty[r], SCHED_CONSUMERS);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_a0);
        tma_prefetch_desc(&tm_a1);
        tma_prefetch_desc(&tm_w0);
        tma_prefetch_desc(&tm_w1);
        if (SPLIT) {
            tma_prefetch_desc(&tm_a0l);
            tma_prefetch_desc(&tm_a1l);
            tma_prefetch_desc(&tm_w0l);
            tma_prefetch_desc(&tm_w1l);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();  // both CTAs' barriers are initialised before any remote signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int q = P.H * P.d;
    // a consumer's release of a ring slot, on rank 0's sempty
    auto release_slot = [&](int slot) { mbar_arrive_cluster(mapa_shared(smem_u32(&sempty[slot]), 0)); };

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------- producer (both CTAs)
            int stage = 0;
            uint32_t phase = 0;
            int issued_phase[PSTAGES];
            for (int s = 0; s < PSTAGES; ++s) issued_phase[s] = -1;
            int slot = 0;
            uint32_t sphase = 0;
            bool ok = true;
            bool stripped = !P.fuse_strip;
            for (int claim = 0; ok; ++claim) {
                int tile;
                if (leader) {
                    // claim the next tile and publish it to both CTAs
                    if (!mbar_wait<true>(&sempty[slot], sphase ^ 1u, P.err, abort_flag)) break;
                    tile = P.tile_ctr ? atomicAdd(P.tile_ctr, 1) : pair + claim * npairs;
                    if (tile > P.total_tiles) tile = P.total_tiles;  // every index past the end is the stop mark
                    ring[slot] = tile;
                    st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(ring + slot)), 1),
                                          static_cast<uint32_t>(tile));
                    mbar_arrive(&sfull[slot]);
                    mbar_arrive_cluster(mapa_shared(smem_u32(&sfull[slot]), 1));
                } else {
                    if (!mbar_wait<true>(&sfull[slot], sphase, P.err, abort_flag)) break;
                    tile = ring[slot];
                    release_slot(slot);
                }
                if (++slot == PRING) {
                    slot = 0;
                    sphase ^= 1u;
                }
                if (tile >= P.total_tiles) break;
                const TileCoord c = decode_tile(P, tile);
                if (c.kv == 0 && !stripped) {
                    if (!wait_strip_done(P, abort_flag)) break;
                    stripped = true;
                }
                KSrc src;
                src.start(P, c.kv, c.t);
                int kb = 0, seg = 0;  // seg 0: hi x hi, 1: hi x lo, 2: lo x hi
                for (int ki = 0; ki < P.nk * NSEG; ++ki) {
                    const CUtensorMap* ta = seg == 2 ? (c.kv ? &tm_a1l : &tm_a0l) : (c.kv ? &tm_a1 : &tm_a0);
                    const CUtensorMap* tw = seg == 1 ? (c.kv ? &tm_w1l : &tm_w0l) : (c.kv ? &tm_w1 : &tm_w0);
                    if (!mbar_wait(&empty[stage], phase ^ 1u, P.err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full_leader = mapa_shared(smem_u32(&full[stage]), 0);
                    if (leader) mbar_arrive_expect_tx(&full[stage], 2 * PSTAGE_BYTES);
                    tma_load_3d_pair(sA + stage * PA_BYTES, ta, full_leader, src.e0, c.m * PM + 128 * rank,
                                     src.slab + src.h);
                    tma_load_3d_pair(sB + stage * PB_BYTES, tw, full_leader, kb * BK, c.n * BN + 128 * rank, c.t);
                    if (!SPLIT || seg == 2) {
                        src.next(P, c.kv, c.t);
                        ++kb;
                        seg = 0;
                    } else {
                        ++seg;
                    }
                    issued_phase[stage] = static_cast<int>(phase);
                    if (++stage == PSTAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // The leader's full barriers count both CTAs' bytes: drain there.
            if (leader)
                for (int s = 0; s < PSTAGES; ++s)
                    if (issued_phase[s] >= 0)
                        mbar_wait_drain(&full[s], static_cast<uint32_t>(issued_phase[s]), DRAIN_NS);
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------------------------------------------- MMA issuer (rank 0)
            constexpr uint32_t idesc = idesc_bf16_f32(PM, BN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            int slot = 0;
            uint32_t sphase = 0;
            bool ok = true;
            while (ok) {
                if (!mbar_wait<true>(&sfull[slot], sphase, P.err, abort_flag)) break;
                const int tile = ring[slot];
                release_slot(slot);
                if (++slot == PRING) {
                    slot = 0;
                    sphase ^= 1u;
                }
                if (tile >= P.total_tiles) break;
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, P.err, abort_flag)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < P.nk * NSEG; ++kb) {
                    if (!mbar_wait(&full[stage], phase, P.err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + stage * PA_BYTES);
                    const uint32_t b0 = smem_u32(sB + stage * PB_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        umma_bf16_pair(d_tmem, sdesc_k_sw128(a0 + k * 32), sdesc_k_sw128(b0 + k * 32), idesc,
                                       (kb | k) != 0);
                    }
                    umma_commit_pair(&empty[stage], 0x3);
                    if (++stage == PSTAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair(&tfull[acc], 0x3);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            umma_commit_pair(drain, 0x1);
            mbar_wait_drain(drain, 0, DRAIN_NS);
        }
    } else {
        // -------------------------------------------------------- epilogue (both CTAs)
        const int sub = warp & 3;
        const int row = sub * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        int slot = 0;
        uint32_t sphase = 0;
        bool strip_left = P.fuse_strip != 0;  // warp-uniform
        for (;;) {
            if (!mbar_wait<true>(&sfull[slot], sphase, P.err, abort_flag)) break;
            const int tile = ring[slot];
            __syncwarp();
            if (lane == 0) release_slot(slot);
            if (++slot == PRING) {
                slot = 0;
                sphase ^= 1u;
            }
            if (tile >= P.total_tiles) break;
            const TileCoord c = decode_tile(P, tile);
            if (strip_left) strip_left = strip_while_waiting(P, &tfull[acc], acc_phase, lane, abort_flag);
            if (!mbar_wait(&tfull[acc], acc_phase, P.err, abort_flag)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(sub * 32) << 16) + static_cast<uint32_t>(acc * BN);
            epilogue_row<SPLIT>(P, c, c.m * PM + 128 * static_cast<int>(rank) + row, tbase, q);
            tc_fence_before();
            mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    cluster_sync_all();  // no CTA leaves while its pair may still read its shared memory or TMEM
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

bool encode_3d_bf16(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box0,
                    uint32_t box1, std::string* why) {
    EncodeTiledFn enc = get_encode_tiled();
    if (!enc) {
        if (why) *why = "cuTensorMapEncodeTiled unavailable from the driver";
        return false;
    }
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    cuuint32_t box[3] = {box0, box1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        if (why) *why = "cuTensorMapEncodeTiled failed with code " + std::to_string(static_cast<int>(r));
        return false;
    }
    return true;
}

// The CTA-pair kernel serves bf16 caches unless KVB_MAP_PAIR=0 (single-CTA kernel).
bool use_pair_kernel() {
    const char* s = std::getenv("KVB_MAP_PAIR");
    return !(s && std::strcmp(s, "0") == 0);
}

}  // namespace

bool map_gemm_tc_supported(const Shape& sh) {
    const int q = sh.H * sh.d;
    return sh.d == 128 && q % BN == 0 && sh.L_t <= MAX_LT && sh.T <= 0x7fffffffLL;
}

bool map_gemm_fused_strip_supported(const Shape& sh) {
    return map_gemm_tc_supported(sh) &&
           static_cast<int64_t>(sh.L_s) * sh.H * ((sh.T + 127) / 128) < 0x7fffffffLL;
}

cudaError_t launch_map_gemm_tc(const MapGemmArgs& a, cudaStream_t s, std::string* why) {
    const Shape& sh = a.sh;
    const int q = sh.H * sh.d;
    const int p = sh.k * q;
    const bool pair = use_pair_kernel() && a.num_sms >= 2;
    const int tm = pair ? PM : BM;
    Params P{};
    P.L_t = sh.L_t;
    P.H = sh.H;
    P.d = sh.d;
    P.T = static_cast<int>(sh.T);
    P.num_m = static_cast<int>((sh.T + tm - 1) / tm);
    P.num_n = q / BN;
    P.nk = p / BK;
    const int64_t total = 2LL * sh.L_t * P.num_m * P.num_n;
    if (total > 0x7fffffffLL - 4096) {  // the pair kernel's claims run a few past the last tile
        if (why) *why = "too many tiles";
        return cudaErrorInvalidValue;
    }
    P.total_tiles = static_cast<int>(total);
    P.max_pos = sh.max_pos;
    P.pos = a.pos;
    P.tab_t = a.tab_t;
    P.err = a.err;
    P.sel = a.sel;
    if (a.fuse_strip && !a.split) {
        P.fuse_strip = 1;
        P.k_raw = static_cast<const __nv_bfloat16*>(a.k_raw);
        P.k_strip = static_cast<__nv_bfloat16*>(const_cast<void*>(a.a_src[0]));
        P.tab_s = a.tab_s;
        P.strip_ctr = a.strip_ctr;
        P.strip_chunks = static_cast<int>((sh.T + 127) / 128);
        P.strip_items = static_cast<int>(static_cast<int64_t>(sh.L_s) * sh.H * P.strip_chunks);
    }
    P.tile_ctr = pair ? a.tile_ctr : nullptr;
    for (int kv = 0; kv < 2; ++kv) {
        P.bias[kv] = a.bias[kv];
        P.out[kv] = a.out[kv];
    }
    CUtensorMap tma[2], tmw[2], tmal[2], tmwl[2];
    for (int kv = 0; kv < 2; ++kv) {
        if (!encode_3d_bf16(&tma[kv], a.a_src[kv], sh.d, sh.T, static_cast<uint64_t>(sh.L_s) * sh.H, BK, 128, why))
            return cudaErrorInvalidValue;
        if (!encode_3d_bf16(&tmw[kv], a.w[kv], p, q, sh.L_t, BK, pair ? 128 : BN, why)) return cudaErrorInvalidValue;
        if (a.split) {
            if (!encode_3d_bf16(&tmal[kv], a.a_lo[kv], sh.d, sh.T, static_cast<uint64_t>(sh.L_s) * sh.H, BK, 128,
                                why))
                return cudaErrorInvalidValue;
            if (!encode_3d_bf16(&tmwl[kv], a.w_lo[kv], p, q, sh.L_t, BK, pair ? 128 : BN, why))
                return cudaErrorInvalidValue;
        } else {
            tmal[kv] = tma[kv];  // unused by the bf16 kernel
            tmwl[kv] = tmw[kv];
        }
    }
    if (!pair) {
        auto kern = a.split ? map_gemm_kernel<true> : map_gemm_kernel<false>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        const int grid = static_cast<int>(total < a.num_sms ? total : a.num_sms);
        kern<<<grid, NUM_THREADS, SMEM_BYTES, s>>>(tma[0], tma[1], tmw[0], tmw[1], tmal[0], tmal[1], tmwl[0], tmwl[1],
                                                   P);
        return cudaGetLastError();
    }
    auto pkern = a.split ? map_gemm_pair_kernel<true> : map_gemm_pair_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(pkern, cudaFuncAttributeMaxDynamicSharedMemorySize, PSMEM_BYTES);
    if (e != cudaSuccess) return e;
    int pairs = a.num_sms / 2;
    if (total < pairs) pairs = static_cast<int>(total);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = PSMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, pkern, tma[0], tma[1], tmw[0], tmw[1], tmal[0], tmal[1], tmwl[0], tmwl[1], P);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace kvb

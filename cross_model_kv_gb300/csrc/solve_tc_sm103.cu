// fp32-accurate updates of the batched Cholesky solver on the 5th-generation
// tensor cores (sm_103a).
//
// The ridge systems of the fit ("KVBridge" README, "Loading": W = (M +
// lambda I)^-1 C) and of the single-source R^2 ("What ships") are solved in
// float32 by a blocked Cholesky whose work is rank-256 (and smaller) updates
//     C = alpha * A B^T + beta * C      (A: M x K, B: N x K, K <= 256, C fp32)
// of the trailing matrix and of the right-hand sides.  Here every fp32
// operand x is carried as three bf16 parts, x1 = bf16(x), x2 = bf16(x - x1),
// x3 = bf16(x - x1 - x2) (24 significant bits in all), and the product is
// accumulated in fp32 TMEM from the six part products whose weight is at
// least 2^-16 of the leading one: x1y1, x1y2, x2y1, x1y3, x2y2, x3y1.  The
// dropped terms are below 2^-23 of |x||y|, the rounding of an fp32 FMA.
//
// solve_gemm_kernel: one CTA per 128 x 256 output tile (grid N-tiles x
// M-tiles x batch), two CTAs per SM (solve_gemm_persistent_kernel below is
// the default): warp 0 issues TMA (A and B parts, 3-D maps over [batch][rows]
// [64]), warp 1 issues tcgen05.mma kind::f16 (M 128, N 256, K 16) into a
// 256-column TMEM accumulator, warps 2..5 read it back (through the then idle
// pipeline shared memory, so that C is updated with coalesced row accesses)
// and write alpha * acc + beta * C.  With `lower`, tiles wholly above the
// diagonal are skipped.
// Every wait is bounded (DevErr::timeout_ns) like the mapper kernel's.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <string>

#include "kvb_internal.h"
#include "stats_internal.h"

namespace kvb {

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;  // one 128-byte swizzle atom of bf16
constexpr int KMAX = 256;  // largest update rank
constexpr int STAGES = 2;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 192;
constexpr int TMEM_COLS = 256;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
constexpr uint64_t DRAIN_NS = 200ull * 1000 * 1000;
constexpr int NPROD = 6;
// part of A and of B in each of the six products, largest first, four bits per
// product (A 0,0,1,0,1,2 and B 0,1,0,2,1,0), so that the producer needs no table
constexpr uint32_t kPartsA = 0x210100u, kPartsB = 0x012010u;
__device__ __forceinline__ int part_a(int pr) { return static_cast<int>((kPartsA >> (4 * pr)) & 3u); }
__device__ __forceinline__ int part_b(int pr) { return static_cast<int>((kPartsB >> (4 * pr)) & 3u); }

struct Params {
    float* C;
    int64_t ldc, strideC;
    int M, N, lower, nkb;  // nkb: 64-wide K blocks (1 to 4)
    float alpha, beta;
    DevErr err;
    // persistent kernel: tiles per system and in all
    int nn, tiles_per_sys, total;
};

struct Maps {
    CUtensorMap a[3], b[3];
};

__global__ void __launch_bounds__(NUM_THREADS, 2) solve_gemm_kernel(const __grid_constant__ Maps Mp,
                                                                    const __grid_constant__ Params P) {
    const int n0 = blockIdx.x * BN;
    const int m0 = blockIdx.y * BM;
    const int bz = blockIdx.z;
    if (P.lower && n0 > m0 + BM - 1) return;  // wholly above the diagonal

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* drain = tfull + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tfull, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------- producer
            int issued_phase[STAGES];
            for (int s = 0; s < STAGES; ++s) issued_phase[s] = -1;
            uint32_t phase = 0;
            int stage = 0;
            for (int it = 0; it < P.nkb * NPROD; ++it) {
                const int kb = it / NPROD, pr = it - kb * NPROD;
                if (!mbar_wait(&empty[stage], phase ^ 1u, P.err, abort_flag)) break;
                mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
                tma_load_3d(sA + stage * A_BYTES, &Mp.a[part_a(pr)], &full[stage], kb * BK, m0, bz);
                tma_load_3d(sB + stage * B_BYTES, &Mp.b[part_b(pr)], &full[stage], kb * BK, n0, bz);
                issued_phase[stage] = static_cast<int>(phase);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            // never leave with a copy still landing in shared memory
            for (int s = 0; s < STAGES; ++s)
                if (issued_phase[s] >= 0) mbar_wait_drain(&full[s], static_cast<uint32_t>(issued_phase[s]), DRAIN_NS);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------- MMA issuer
            constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
            uint32_t phase = 0;
            int stage = 0;
            bool ok = true;
            for (int it = 0; it < P.nkb * NPROD; ++it) {
                if (!mbar_wait(&full[stage], phase, P.err, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = smem_u32(sA + stage * A_BYTES);
                const uint32_t b0 = smem_u32(sB + stage * B_BYTES);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    umma_bf16(tmem_base, sdesc_k_sw128(a0 + k * 32), sdesc_k_sw128(b0 + k * 32), idesc, (it | k) != 0);
                umma_commit(&empty[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (ok) umma_commit(tfull);
            // every MMA issued here completes before TMEM is released
            umma_commit(drain);
            mbar_wait_drain(drain, 0, DRAIN_NS);
        }
    } else {
        // ----------------------------------------------------------- epilogue
        const int sub = warp & 3;  // TMEM lane quarter this warp may access
        if (mbar_wait(tfull, 0, P.err, abort_flag)) {
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(sub * 32) << 16);
            // The pipeline's shared memory is free once the accumulator is
            // complete: each warp stages its 32 rows x 128 columns there (row
            // stride 129 floats, conflict-free both ways) and then updates C
            // one row at a time with 128-byte coalesced accesses.
            float* stg = reinterpret_cast<float*>(smem) + sub * (32 * 129);
            const int rbase = m0 + sub * 32;
#pragma unroll 1
            for (int h0 = 0; h0 < BN && n0 + h0 < P.N; h0 += 128) {
                const int ncol = P.N - (n0 + h0) < 128 ? P.N - (n0 + h0) : 128;  // multiple of 16
#pragma unroll 1
                for (int c = 0; c < ncol; c += 16) {
                    uint32_t v[16];
                    tmem_ld16(tbase + h0 + c, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) stg[lane * 129 + c + j] = __uint_as_float(v[j]);
                }
                __syncwarp();
#pragma unroll 1
                for (int r0 = 0; r0 < 32; r0 += 8) {  // 8 rows x 4 columns per lane in flight
                    float old[8][4];
#pragma unroll
                    for (int rr = 0; rr < 8; ++rr) {
                        const int r = rbase + r0 + rr;
                        const float* crow = P.C + bz * P.strideC + static_cast<int64_t>(r) * P.ldc + n0 + h0;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int col = lane + 32 * j;
                            old[rr][j] = (r < P.M && col < ncol && P.beta != 0.f) ? crow[col] : 0.f;
                        }
                    }
#pragma unroll
                    for (int rr = 0; rr < 8; ++rr) {
                        const int r = rbase + r0 + rr;
                        if (r >= P.M) continue;
                        float* crow = P.C + bz * P.strideC + static_cast<int64_t>(r) * P.ldc + n0 + h0;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int col = lane + 32 * j;
                            if (col < ncol)
                                crow[col] = fmaf(P.beta, old[rr][j], P.alpha * stg[(r0 + rr) * 129 + col]);
                        }
                    }
                }
                __syncwarp();  // the staging rows are rewritten by the next half
            }
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

// Persistent form of the same update: one CTA per SM walks the tiles (system,
// row block, column block; with `lower`, only tiles touching the lower
// triangle), four 48 KB stages, the accumulator double buffered in TMEM (2 x
// 256 columns) so that one tile's read-modify-write of C overlaps the next
// tile's products.  Epilogue: eight warps, two threads per row (128 columns
// each), 16 columns per step as two 32-byte (one-sector) accesses, C loaded
// two steps ahead of the accumulator.  Needs C, ldc and strideC 32-byte aligned.
constexpr int PSTAGES = 4;
constexpr int PEPI_WARPS = 8;
constexpr int PNUM_THREADS = 64 + 32 * PEPI_WARPS;
constexpr int PSMEM_BYTES = PSTAGES * STAGE_BYTES + 1024 + 256;

__device__ __forceinline__ void decode_tile(const Params& P, int t, int& bz, int& mi, int& nj) {
    bz = t / P.tiles_per_sys;
    int r = t - bz * P.tiles_per_sys;
    if (!P.lower) {
        mi = r / P.nn;
        nj = r - mi * P.nn;
        return;
    }
    for (mi = 0;; ++mi) {  // row block mi holds the column blocks nj with nj * BN <= mi * BM + BM - 1
        const int cnt = min(P.nn, (mi * BM + BM - 1) / BN + 1);
        if (r < cnt) break;
        r -= cnt;
    }
    nj = r;
}

__global__ void __launch_bounds__(PNUM_THREADS, 1) solve_gemm_persistent_kernel(const __grid_constant__ Maps Mp,
                                                                                const __grid_constant__ Params P) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sA = smem;
    uint8_t* sB = smem + PSTAGES * A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + PSTAGES * STAGE_BYTES);
    uint64_t* empty = full + PSTAGES;
    uint64_t* tfull = empty + PSTAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < PSTAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 32 * PEPI_WARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 2 * TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int iters = P.nkb * NPROD;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------- producer
            int issued_phase[PSTAGES];
            for (int s = 0; s < PSTAGES; ++s) issued_phase[s] = -1;
            uint32_t phase = 0;
            int stage = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < P.total; t += gridDim.x) {
                int bz, mi, nj;
                decode_tile(P, t, bz, mi, nj);
                for (int it = 0; it < iters; ++it) {
                    const int kb = it / NPROD, pr = it - kb * NPROD;
                    if (!mbar_wait(&empty[stage], phase ^ 1u, P.err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
                    tma_load_3d(sA + stage * A_BYTES, &Mp.a[part_a(pr)], &full[stage], kb * BK, mi * BM, bz);
                    tma_load_3d(sB + stage * B_BYTES, &Mp.b[part_b(pr)], &full[stage], kb * BK, nj * BN, bz);
                    issued_phase[stage] = static_cast<int>(phase);
                    if (++stage == PSTAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (int s = 0; s < PSTAGES; ++s)
                if (issued_phase[s] >= 0) mbar_wait_drain(&full[s], static_cast<uint32_t>(issued_phase[s]), DRAIN_NS);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------- MMA issuer
            constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
            uint32_t phase = 0;
            int stage = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < P.total; t += gridDim.x) {
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, P.err, abort_flag)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * TMEM_COLS);
                for (int it = 0; it < iters; ++it) {
                    if (!mbar_wait(&full[stage], phase, P.err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + stage * A_BYTES);
                    const uint32_t b0 = smem_u32(sB + stage * B_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        umma_bf16(d_tmem, sdesc_k_sw128(a0 + k * 32), sdesc_k_sw128(b0 + k * 32), idesc,
                                  (it | k) != 0);
                    umma_commit(&empty[stage]);
                    if (++stage == PSTAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(&tfull[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            umma_commit(drain);  // every MMA issued here completes before TMEM is released
            mbar_wait_drain(drain, 0, DRAIN_NS);
        }
    } else {
        // ----------------------------------------------------------- epilogue
        const int sub = warp & 3;              // TMEM lane quarter this warp may access
        const int half = (warp - 2) >> 2;      // columns [0,128) or [128,256) of the tile
        const int row = sub * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < P.total; t += gridDim.x) {
            int bz, mi, nj;
            decode_tile(P, t, bz, mi, nj);
            const int r = mi * BM + row;
            const int n0 = nj * BN + 128 * half;
            const int ncol = max(0, min(128, P.N - n0));  // multiple of 16
            const bool live = r < P.M;
            const bool rd = live && P.beta != 0.f;
            float* crow = P.C + bz * P.strideC + static_cast<int64_t>(r) * P.ldc + n0;
            // C two steps ahead: cur = step c0, nxt = step c0 + 16
            uint32_t cur[2][8] = {}, nxt[2][8] = {};
            if (rd && ncol > 0) {
                ld_global_v8(crow, cur[0]);
                ld_global_v8(crow + 8, cur[1]);
            }
            if (rd && ncol > 16) {
                ld_global_v8(crow + 16, nxt[0]);
                ld_global_v8(crow + 24, nxt[1]);
            }
            if (!mbar_wait(&tfull[acc], acc_phase, P.err, abort_flag)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(sub * 32) << 16) +
                                   static_cast<uint32_t>(acc * TMEM_COLS + 128 * half);
#pragma unroll 1
            for (int c0 = 0; c0 < ncol; c0 += 16) {
                uint32_t nn2[2][8] = {};
                if (rd && c0 + 32 < ncol) {
                    ld_global_v8(crow + c0 + 32, nn2[0]);
                    ld_global_v8(crow + c0 + 40, nn2[1]);
                }
                uint32_t v[16];
                tmem_ld16(tbase + c0, v);
                tmem_ld_wait();
                if (live) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t o[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            o[e] = __float_as_uint(
                                fmaf(P.beta, __uint_as_float(cur[h][e]), P.alpha * __uint_as_float(v[8 * h + e])));
                        st_global_v8(crow + c0 + 8 * h, o);
                    }
                }
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        cur[h][e] = nxt[h][e];
                        nxt[h][e] = nn2[h][e];
                    }
            }
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
        tmem_dealloc(tmem_base, 2 * TMEM_COLS);
    }
}

// Three bf16 parts of a rows x K fp32 operand (K <= kp), written K-major as
// [batch][rows][kp] with zeros beyond K.  Element (r, k) of batch item b is
// src[b * s_batch + r * s_row + k * s_k]; 32 x 32 tiles through shared
// memory so that both K-contiguous and row-contiguous sources read coalesced.
__global__ void __launch_bounds__(256) split3_kernel(const float* __restrict__ src, int64_t rows, int K,
                                                     int64_t s_row, int64_t s_k, int64_t s_batch,
                                                     __nv_bfloat16* __restrict__ p0, __nv_bfloat16* __restrict__ p1,
                                                     __nv_bfloat16* __restrict__ p2, int64_t ld) {
    __shared__ float tile[32][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * 32;
    const int k0 = blockIdx.y * 32;
    const int b = blockIdx.z;
    const float* s = src + b * s_batch;
    if (s_k == 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t r = r0 + ty + 8 * i;
            const int k = k0 + tx;
            tile[ty + 8 * i][tx] = (r < rows && k < K) ? s[r * s_row + k] : 0.f;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t r = r0 + tx;
            const int k = k0 + ty + 8 * i;
            tile[tx][ty + 8 * i] = (r < rows && k < K) ? s[r * s_row + k * s_k] : 0.f;
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t r = r0 + ty + 8 * i;
        if (r >= rows) continue;
        const float x = tile[ty + 8 * i][tx];
        const __nv_bfloat16 x1 = __float2bfloat16_rn(x);
        const float e1 = x - __bfloat162float(x1);
        const __nv_bfloat16 x2 = __float2bfloat16_rn(e1);
        const __nv_bfloat16 x3 = __float2bfloat16_rn(e1 - __bfloat162float(x2));
        const int64_t o = (static_cast<int64_t>(b) * rows + r) * ld + k0 + tx;
        p0[o] = x1;
        p1[o] = x2;
        p2[o] = x3;
    }
}

// kp columns of rows `ld` elements apart (systems rows * ld apart)
bool encode_parts(CUtensorMap* m, const void* base, int64_t rows, int batch, int kp, int64_t ld, uint32_t box_rows,
                  std::string* why) {
    EncodeTiledFn enc = get_encode_tiled();
    if (!enc) {
        if (why) *why = "cuTensorMapEncodeTiled unavailable from the driver";
        return false;
    }
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kp), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, static_cast<cuuint64_t>(rows) * ld * 2};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        if (why) *why = "cuTensorMapEncodeTiled failed with code " + std::to_string(static_cast<int>(r));
        return false;
    }
    return true;
}

cudaError_t split3(const TcOperand& o, int K, int kp, int batch, __nv_bfloat16* dst, cudaStream_t s) {
    const int64_t part = static_cast<int64_t>(batch) * o.rows * kp;
    dim3 grid(static_cast<unsigned>((o.rows + 31) / 32), static_cast<unsigned>(kp / 32), static_cast<unsigned>(batch));
    split3_kernel<<<grid, 256, 0, s>>>(o.src, o.rows, K, o.s_row, o.s_k, o.s_batch, dst, dst + part, dst + 2 * part,
                                       kp);
    return cudaGetLastError();
}

}  // namespace

cudaError_t tc_split_into(const TcOperand& o, int K, int batch, const TcPreSplit& dst, cudaStream_t s) {
    if (K < 1 || K > BK) return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>((o.rows + 31) / 32), static_cast<unsigned>(BK / 32), static_cast<unsigned>(batch));
    split3_kernel<<<grid, 256, 0, s>>>(o.src, o.rows, K, o.s_row, o.s_k, o.s_batch, dst.base, dst.base + dst.part,
                                       dst.base + 2 * dst.part, dst.ld);
    return cudaGetLastError();
}

size_t tc_update_ws_bytes(int64_t rows_a, int64_t rows_b, int batch) {
    return 3ull * static_cast<size_t>(batch) * static_cast<size_t>(rows_a + rows_b) * KMAX * 2 + 1024;
}

bool tc_update_supported(const TcSolve* tc, int64_t M, int64_t N, int K, const float* C, int64_t ldc) {
    // worth a launch when the update is large: many rows, or a few rows across many columns
    const bool large = (M >= 256 && N >= 256) || (M >= 64 && N >= 8192);
    return tc && tc->ws && tc->num_sms > 0 && K >= 1 && K <= KMAX && large && N % 16 == 0 && ldc % 4 == 0 &&
           (reinterpret_cast<uintptr_t>(C) & 15u) == 0 && M <= 0x7fffffffLL && N <= 0x7fffffffLL;
}

cudaError_t launch_tc_update(const TcSolve& tc, const TcOperand& A, const TcOperand* B, int K, float* C, int64_t ldc,
                             int64_t strideC, float alpha, float beta, bool lower, int batch, cudaStream_t s,
                             std::string* why, const TcPreSplit* pre_b) {
    const int64_t rows_b = B && !pre_b ? B->rows : 0;
    if (tc_update_ws_bytes(A.rows, rows_b, batch) > tc.ws_bytes) {
        if (why) *why = "tensor-core update workspace too small";
        return cudaErrorInvalidValue;
    }
    const int kp = ((K + BK - 1) / BK) * BK;
    __nv_bfloat16* wa = tc.ws;
    __nv_bfloat16* wb = wa + 3 * static_cast<int64_t>(batch) * A.rows * kp;
    cudaError_t e = split3(A, K, kp, batch, wa, s);
    if (e == cudaSuccess && B && !pre_b) e = split3(*B, K, kp, batch, wb, s);
    if (e != cudaSuccess) return e;
    const int64_t N = B ? B->rows : A.rows;
    const __nv_bfloat16* bb = B ? wb : wa;
    Maps mp;
    for (int i = 0; i < 3; ++i) {
        const bool ok_a = encode_parts(&mp.a[i], wa + i * static_cast<int64_t>(batch) * A.rows * kp, A.rows, batch, kp,
                                       kp, BM, why);
        const bool ok_b = pre_b ? encode_parts(&mp.b[i], pre_b->base + i * pre_b->part, N, batch, kp, pre_b->ld, BN, why)
                                : encode_parts(&mp.b[i], bb + i * static_cast<int64_t>(batch) * N * kp, N, batch, kp, kp,
                                               BN, why);
        if (!ok_a || !ok_b) return cudaErrorInvalidValue;
    }
    Params P{};
    P.C = C;
    P.ldc = ldc;
    P.strideC = strideC;
    P.M = static_cast<int>(A.rows);
    P.N = static_cast<int>(N);
    P.lower = lower ? 1 : 0;
    P.nkb = kp / BK;
    P.alpha = alpha;
    P.beta = beta;
    P.err = tc.err;
    // the persistent kernel's 32-byte accesses need C, ldc and strideC 32-byte aligned
    const char* env = std::getenv("KVB_SOLVE_PERSIST");
    const bool persist = !(env && std::strcmp(env, "0") == 0) && (reinterpret_cast<uintptr_t>(C) & 31u) == 0 &&
                         ldc % 8 == 0 && strideC % 8 == 0;
    const int nm = static_cast<int>((A.rows + BM - 1) / BM), nn = static_cast<int>((N + BN - 1) / BN);
    if (persist) {
        int64_t per_sys = 0;
        for (int mi = 0; mi < nm; ++mi)
            per_sys += lower ? std::min<int64_t>(nn, (int64_t(mi) * BM + BM - 1) / BN + 1) : nn;
        const int64_t total = per_sys * batch;
        if (total > 0 && total <= 0x7fffffffLL) {
            P.nn = nn;
            P.tiles_per_sys = static_cast<int>(per_sys);
            P.total = static_cast<int>(total);
            e = cudaFuncSetAttribute(solve_gemm_persistent_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     PSMEM_BYTES);
            if (e != cudaSuccess) return e;
            const int grid = static_cast<int>(total < tc.num_sms ? total : tc.num_sms);
            solve_gemm_persistent_kernel<<<grid, PNUM_THREADS, PSMEM_BYTES, s>>>(mp, P);
            return cudaGetLastError();
        }
    }
    e = cudaFuncSetAttribute(solve_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid(static_cast<unsigned>(nn), static_cast<unsigned>(nm), static_cast<unsigned>(batch));
    solve_gemm_kernel<<<grid, NUM_THREADS, SMEM_BYTES, s>>>(mp, P);
    return cudaGetLastError();
}

}  // namespace kvb

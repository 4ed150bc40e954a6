// Calibration-statistics GEMM on the 5th-generation tensor cores (sm_103a).
//
// Every job is a centered cross-product over the observations of one batch,
// merged into the running statistics with Chan's update ("KVBridge" README,
// "Loading"):
//     out[i][j] += sum_r A[i][r] B[j][r] - g za[i] zb[j] + f da[i] db[j]
// with A, B the shifted, transposed batch ([feature][observation], K-major),
// g za zb the rank-1 term that centers it on the batch mean and f da db the
// rank-1 Chan term between the running and the batch means.  The operands are bf16 pairs
// (hi + lo) of the float32 centered values; the product is accumulated as
// hi.hi + hi.lo + lo.hi in one fp32 TMEM accumulator, three K-passes over the
// same tile, which keeps ~16 significant bits per operand.
//
// Persistent, warp-specialised, one CTA per SM, 128 x 256 tiles from a tile
// list (Gram jobs list only tiles touching the lower triangle; tiles are
// grouped 16 row-blocks at a time so a group's A rows stay in L2):
//   warp 0      TMA producer (one lane)
//   warp 1      MMA issuer (one lane), TMEM double buffered (2 x 256 columns)
//   warps 2..9  epilogue: TMEM -> registers, read-modify-write of the fp32
//               statistics with the merge term.
// Waits are bounded like the mapper kernel's.
#include <cstring>
#include <string>
#include <vector>

#include "stats_internal.h"

namespace kvb {

struct StatsGemmPlan {
    uint32_t* tiles = nullptr;
    int n_tiles = 0;
};

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 8;
constexpr int NUM_THREADS = 64 + EPI_WARPS * 32;
constexpr int TMEM_COLS = 512;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
constexpr uint64_t DRAIN_NS = 200ull * 1000 * 1000;
constexpr int GROUP = 16;

struct JobP {
    float* out;
    const float* da;
    const float* db;
    const float* za;
    const float* zb;
    int64_t ldo;
};

struct Params {
    const uint32_t* tiles;
    int n_tiles;
    const int* nb;
    const float* coef;  // {f, g}
    DevErr err;
    JobP job[4];
};

struct Maps {
    CUtensorMap a_hi[4], a_lo[4], b_hi[4], b_lo[4];
};

__device__ __forceinline__ void decode(uint32_t e, int& job, int& bi, int& bj) {
    job = static_cast<int>(e >> 30);
    bi = static_cast<int>((e >> 15) & 0x7FFFu);
    bj = static_cast<int>(e & 0x7FFFu);
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    stats_gemm_kernel(const __grid_constant__ Maps M, const __grid_constant__ Params P) {
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
            mbar_init(&tempty[a], EPI_WARPS * 32);
        }
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
    const int nk = (*P.nb + BK - 1) / BK;  // K-blocks per pass (zero padding beyond n_b)
    const int iters = 3 * nk;

    if (warp == 0) {
        if (lane == 0 && iters > 0) {
            int stage = 0;
            uint32_t phase = 0;
            int issued_phase[STAGES];
            for (int s = 0; s < STAGES; ++s) issued_phase[s] = -1;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < P.n_tiles; t += gridDim.x) {
                int job, bi, bj;
                decode(P.tiles[t], job, bi, bj);
                for (int it = 0; it < iters; ++it) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, P.err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const int seg = it / nk;
                    const int kb = it - seg * nk;
                    const CUtensorMap* ma = seg == 2 ? &M.a_lo[job] : &M.a_hi[job];
                    const CUtensorMap* mb = seg == 1 ? &M.b_lo[job] : &M.b_hi[job];
                    mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
                    tma_load_2d(sA + stage * A_BYTES, ma, &full[stage], kb * BK, bi * BM);
                    tma_load_2d(sB + stage * B_BYTES, mb, &full[stage], kb * BK, bj * BN);
                    issued_phase[stage] = static_cast<int>(phase);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (int s = 0; s < STAGES; ++s)
                if (issued_phase[s] >= 0) mbar_wait_drain(&full[s], static_cast<uint32_t>(issued_phase[s]), DRAIN_NS);
        }
    } else if (warp == 1) {
        if (lane == 0 && iters > 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < P.n_tiles; t += gridDim.x) {
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, P.err, abort_flag)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
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
            umma_commit(drain);
            mbar_wait_drain(drain, 0, DRAIN_NS);
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int ew = warp - 2;
        const int sub = warp & 3;          // TMEM lane quarter
        const int colhalf = ew >> 2;       // columns [0,128) or [128,256)
        const int row = sub * 32 + lane;
        const float ff = P.coef[0], gg = P.coef[1];
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < P.n_tiles; t += gridDim.x) {
            int job, bi, bj;
            decode(P.tiles[t], job, bi, bj);
            const JobP J = P.job[job];
            const int64_t i = static_cast<int64_t>(bi) * BM + row;
            const int64_t j0 = static_cast<int64_t>(bj) * BN + colhalf * 128;
            float* orow = J.out + i * J.ldo + j0;
            const float fda = ff * __ldg(J.da + i);
            const float gza = gg * __ldg(J.za + i);
            const float* dbp = J.db + j0;
            const float* zbp = J.zb + j0;
            if (iters > 0) {
                if (!mbar_wait(&tfull[acc], acc_phase, P.err, abort_flag)) break;
                tc_fence_after();
            }
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(sub * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN + colhalf * 128);
            // 16 statistics per step as two 32-byte (one-sector) accesses; the next step's
            // values are loaded before this step's accumulator is read
            uint32_t cur[2][8];
            ld_global_v8(orow, cur[0]);
            ld_global_v8(orow + 8, cur[1]);
#pragma unroll 1
            for (int c0 = 0; c0 < 128; c0 += 16) {
                uint32_t nxt[2][8];
                if (c0 + 16 < 128) {
                    ld_global_v8(orow + c0 + 16, nxt[0]);
                    ld_global_v8(orow + c0 + 24, nxt[1]);
                }
                uint32_t r[16];
                if (iters > 0) {
                    tmem_ld16(tbase + c0, r);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int v = 0; v < 16; ++v) r[v] = 0u;
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t o[8];
#pragma unroll
                    for (int v = 0; v < 2; ++v) {
                        const float4 d = __ldg(reinterpret_cast<const float4*>(dbp + c0 + 8 * h + 4 * v));
                        const float4 z = __ldg(reinterpret_cast<const float4*>(zbp + c0 + 8 * h + 4 * v));
                        const float dd[4] = {d.x, d.y, d.z, d.w}, zz[4] = {z.x, z.y, z.z, z.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int e = 4 * v + u;
                            o[e] = __float_as_uint(__uint_as_float(cur[h][e]) + __uint_as_float(r[8 * h + e]) +
                                                   fda * dd[u] - gza * zz[u]);
                        }
                    }
                    st_global_v8(orow + c0 + 8 * h, o);
                }
                if (c0 + 16 < 128) {
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int e = 0; e < 8; ++e) cur[h][e] = nxt[h][e];
                }
            }
            if (iters > 0) {
                tc_fence_before();
                mbar_arrive(&tempty[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
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

bool encode_2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows, std::string* why) {
    EncodeTiledFn enc = get_encode_tiled();
    if (!enc) {
        if (why) *why = "cuTensorMapEncodeTiled unavailable from the driver";
        return false;
    }
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {BK, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        if (why) *why = "cuTensorMapEncodeTiled failed with code " + std::to_string(static_cast<int>(r));
        return false;
    }
    return true;
}

}  // namespace

bool stats_gemm_tc_supported(const StatsJob* jobs, int n_jobs) {
    if (n_jobs < 1 || n_jobs > 4) return false;
    for (int j = 0; j < n_jobs; ++j) {
        if (jobs[j].Ma % BM || jobs[j].Nb % BN) return false;
        if (jobs[j].Ma / BM > 0x7FFF || jobs[j].Nb / BN > 0x7FFF) return false;
    }
    return true;
}

cudaError_t stats_gemm_tc_plan(const StatsJob* jobs, int n_jobs, StatsGemmPlan** plan) {
    std::vector<uint32_t> tiles;
    for (int j = 0; j < n_jobs; ++j) {
        const int64_t nI = jobs[j].Ma / BM, nJ = jobs[j].Nb / BN;
        for (int64_t g0 = 0; g0 < nI; g0 += GROUP) {
            const int64_t g1 = g0 + GROUP < nI ? g0 + GROUP : nI;
            for (int64_t bj = 0; bj < nJ; ++bj)
                for (int64_t bi = g0; bi < g1; ++bi) {
                    if (jobs[j].lower && bj * BN > bi * BM + BM - 1) continue;
                    tiles.push_back((static_cast<uint32_t>(j) << 30) | (static_cast<uint32_t>(bi) << 15) |
                                    static_cast<uint32_t>(bj));
                }
        }
    }
    StatsGemmPlan* p = new StatsGemmPlan();
    p->n_tiles = static_cast<int>(tiles.size());
    cudaError_t e = cudaMalloc(&p->tiles, tiles.size() * sizeof(uint32_t) + 16);
    if (e == cudaSuccess)
        e = cudaMemcpy(p->tiles, tiles.data(), tiles.size() * sizeof(uint32_t), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        cudaFree(p->tiles);
        delete p;
        *plan = nullptr;
        return e;
    }
    *plan = p;
    return cudaSuccess;
}

void stats_gemm_tc_free(StatsGemmPlan* plan) {
    if (!plan) return;
    cudaFree(plan->tiles);
    delete plan;
}

cudaError_t launch_stats_gemm_tc(StatsGemmPlan* plan, const StatsJob* jobs, int n_jobs, int64_t ld,
                                 const float* coef, const int* nb, DevErr err, int num_sms, cudaStream_t s,
                                 std::string* why) {
    if (!plan || plan->n_tiles == 0) return cudaSuccess;
    Maps M;
    std::memset(&M, 0, sizeof(M));
    Params P{};
    P.tiles = plan->tiles;
    P.n_tiles = plan->n_tiles;
    P.nb = nb;
    P.coef = coef;
    P.err = err;
    for (int j = 0; j < n_jobs; ++j) {
        const StatsJob& J = jobs[j];
        if (!encode_2d(&M.a_hi[j], J.A, ld, J.Ma, BM, why) || !encode_2d(&M.a_lo[j], J.A_lo, ld, J.Ma, BM, why) ||
            !encode_2d(&M.b_hi[j], J.B, ld, J.Nb, BN, why) || !encode_2d(&M.b_lo[j], J.B_lo, ld, J.Nb, BN, why))
            return cudaErrorInvalidValue;
        P.job[j] = JobP{J.out, J.da, J.db, J.za, J.zb, J.ldo};
    }
    cudaError_t e = cudaFuncSetAttribute(stats_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int grid = plan->n_tiles < num_sms ? plan->n_tiles : num_sms;
    stats_gemm_kernel<<<grid, NUM_THREADS, SMEM_BYTES, s>>>(M, P);
    return cudaGetLastError();
}

}  // namespace kvb

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
// lo.hi + hi.lo + hi.hi (smallest first) in one fp32 TMEM accumulator, three
// K-passes over the same tile, which keeps ~16 significant bits per operand.
//
// Persistent, warp-specialised, 128 x 256 tiles on one CTA per SM, or 256 x
// 256 tiles on CTA pairs (stats_gemm_pair_kernel, the default when the sizes
// are multiples of 256), from a tile list (Gram jobs list only tiles touching
// the lower triangle; tiles are grouped 2048 rows at a time so a group's A
// rows stay in L2):
//   warp 0      TMA producer (one lane)
//   warp 1      MMA issuer (one lane), TMEM double buffered (2 x 256 columns)
//   warps 2..9  epilogue: TMEM -> registers, read-modify-write of the fp32
//               statistics with the merge term.
// Waits are bounded like the mapper kernel's.
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "stats_internal.h"

namespace kvb {

struct StatsGemmPlan {
    uint32_t* tiles = nullptr;
    int n_tiles = 0;
    bool pair = false;   // 256 x 256 tiles on CTA pairs
    int* ctr = nullptr;  // pair kernel: next tile to claim (after the tile list)
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
// CTA-pair kernel: per CTA 128 of the 256 rows of A and of B
constexpr int PM = 256;
constexpr int PSTAGES = 6;
constexpr int PA_BYTES = 128 * BK * 2;
constexpr int PSTAGE_BYTES = 2 * PA_BYTES;
constexpr int PSMEM_BYTES = PSTAGES * PSTAGE_BYTES + 1024 + 512;
constexpr int PGROUP = 8;  // 256-row blocks per group (2048 rows, as GROUP x 128)
constexpr int PRING = 4;
constexpr int PRING_CONSUMERS = 1 + EPI_WARPS + 1 + EPI_WARPS;  // MMA, rank 0 epilogue, rank 1 producer and epilogue

struct JobP {
    float* out;
    const float* da;
    const float* db;
    const float* za;
    const float* zb;
    int64_t ldo;
    int64_t rows, cols;  // out is [rows][ldo]; da, za have rows entries, db, zb cols
};

struct Params {
    const uint32_t* tiles;
    int n_tiles;
    int* ctr;  // pair kernel: tile claim counter (zeroed before the launch)
    const int* nb;
    const float* coef;  // {f, g}
    DevErr err;
    int nprod;  // 3 (operands as two bf16 parts) or 6 (three parts)
    JobP job[4];
};

struct Maps {
    CUtensorMap a[3][4], b[3][4];  // [part: hi, lo, third][job]
};

// Operand parts of product `seg` in order of size: two-part operands take
// hi.hi, hi.lo, lo.hi; three-part operands add hi.3, lo.lo, 3.hi (every product
// down to 2^-16 of the leading one).  The part indices are packed four bits per
// product so that the single producer thread computes them in registers.  The
// products are issued smallest first (product nprod - 1 down to 0): the small
// ones then add into a small accumulator instead of losing their low bits
// against the full-size sum, which leaves the statistics (and W on
// ill-conditioned systems) measurably closer to float64 at the same cost.
__device__ __forceinline__ void product_maps(const Maps& M, int job, int seg, const CUtensorMap*& ma,
                                             const CUtensorMap*& mb) {
    constexpr uint32_t PA = 0x210100u, PB = 0x012010u;  // parts of A and B for products 0..5
    ma = &M.a[(PA >> (4 * seg)) & 3u][job];
    mb = &M.b[(PB >> (4 * seg)) & 3u][job];
}

__device__ __forceinline__ void decode(uint32_t e, int& job, int& bi, int& bj) {
    job = static_cast<int>(e >> 30);
    bi = static_cast<int>((e >> 15) & 0x7FFFu);
    bj = static_cast<int>(e & 0x7FFFu);
}

// One thread's 128 statistics of row i, columns j0 .. j0+127: out += acc + f da db - g za zb,
// 16 per step as two 32-byte (one-sector) accesses; the next step's values are loaded
// before this step's accumulator is read.  acc is read from TMEM at tbase (zero if !have_acc).
// fda = f da[i], gza = g za[i] (loaded by the caller before it waits for the accumulator).
__device__ __forceinline__ void merge_row(const Params& P, int job, int64_t i, int64_t j0, uint32_t tbase,
                                          bool have_acc, float fda, float gza) {
    const JobP J = P.job[job];
    // checked build: the row's statistics and merge vectors stay inside their buffers
    // (the TMEM loads below are warp-wide and always run)
    const bool inb = KVB_IN_BOUNDS(P.err, i * J.ldo + j0, 128, J.rows * J.ldo) && KVB_IN_BOUNDS(P.err, j0, 128, J.cols);
    float* orow = J.out + i * J.ldo + j0;
    const float* dbp = J.db + j0;
    const float* zbp = J.zb + j0;
    uint32_t cur[2][8] = {};
    if (inb) {
        ld_global_v8(orow, cur[0]);
        ld_global_v8(orow + 8, cur[1]);
    }
#pragma unroll 1
    for (int c0 = 0; c0 < 128; c0 += 16) {
        uint32_t nxt[2][8] = {};
        if (inb && c0 + 16 < 128) {
            ld_global_v8(orow + c0 + 16, nxt[0]);
            ld_global_v8(orow + c0 + 24, nxt[1]);
        }
        uint32_t r[16];
        if (have_acc) {
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
                const float4 d = inb ? __ldg(reinterpret_cast<const float4*>(dbp + c0 + 8 * h + 4 * v))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                const float4 z = inb ? __ldg(reinterpret_cast<const float4*>(zbp + c0 + 8 * h + 4 * v))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                const float dd[4] = {d.x, d.y, d.z, d.w}, zz[4] = {z.x, z.y, z.z, z.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int e = 4 * v + u;
                    o[e] = __float_as_uint(__uint_as_float(cur[h][e]) + __uint_as_float(r[8 * h + e]) +
                                           fda * dd[u] - gza * zz[u]);
                }
            }
            if (inb) st_global_v8(orow + c0 + 8 * h, o);
        }
        if (c0 + 16 < 128) {
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int e = 0; e < 8; ++e) cur[h][e] = nxt[h][e];
        }
    }
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
    const int iters = P.nprod * nk;

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
                const CUtensorMap *ma, *mb;
                product_maps(M, job, P.nprod - 1, ma, mb);
                for (int it = 0, seg = 0, kb = 0; it < iters; ++it) {  // it = seg * nk + kb
                    if (!mbar_wait(&empty[stage], phase ^ 1u, P.err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
                    tma_load_2d(sA + stage * A_BYTES, ma, &full[stage], kb * BK, bi * BM);
                    tma_load_2d(sB + stage * B_BYTES, mb, &full[stage], kb * BK, bj * BN);
                    if (++kb == nk && ++seg < P.nprod) {
                        kb = 0;
                        product_maps(M, job, P.nprod - 1 - seg, ma, mb);
                    }
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
            const int64_t i = static_cast<int64_t>(bi) * BM + row;
            const float fda = ff * __ldg(P.job[job].da + i);
            const float gza = gg * __ldg(P.job[job].za + i);
            if (iters > 0) {
                if (!mbar_wait(&tfull[acc], acc_phase, P.err, abort_flag)) break;
                tc_fence_after();
            }
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(sub * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN + colhalf * 128);
            merge_row(P, job, i, static_cast<int64_t>(bj) * BN + colhalf * 128, tbase, iters > 0, fda, gza);
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

// CTA-pair kernel: clusters of two CTAs, 256 x 256 tiles, tcgen05.mma cta_group::2
// (M 256, N 256).  CTA r stages rows 256 bi + 128 r of A and 256 bj + 128 r of B
// (a 32 KB stage per SM instead of 48 KB, six stages) and merges the accumulator
// rows of its A rows.  Both CTAs' copies complete on rank 0's full barrier; rank 0
// issues the MMAs and commits to both CTAs' barriers; both epilogues arrive on
// rank 0's tempty.  Tiles are claimed in list order from a counter by rank 0's
// producer and passed through a ring in both CTAs' shared memory, so the pairs
// that share a group's rows run together (a fixed tile per pair lets them drift
// apart and re-read the rows from DRAM).
__global__ void __launch_bounds__(NUM_THREADS, 1)
    stats_gemm_pair_kernel(const __grid_constant__ Maps M, const __grid_constant__ Params P) {
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

    if (threadIdx.x == 0) {
        for (int s = 0; s < PSTAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 2 * EPI_WARPS * 32);
        }
        mbar_init(drain, 1);
        for (int r = 0; r < PRING; ++r) {
            mbar_init(&sfull[r], 1);
            mbar_init(&sempty[r], PRING_CONSUMERS);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();  // both CTAs' barriers are initialised before any remote signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int nk = (*P.nb + BK - 1) / BK;  // K-blocks per pass (zero padding beyond n_b)
    const int iters = P.nprod * nk;
    // a consumer's release of a ring slot, on rank 0's sempty
    auto release_slot = [&](int slot) { mbar_arrive_cluster(mapa_shared(smem_u32(&sempty[slot]), 0)); };
    int slot = 0;
    uint32_t sphase = 0;
    // the next tile from the ring (all consumers); the stop mark is n_tiles
    auto next_tile = [&](bool warp_wide) {
        int tile = P.n_tiles;
        bool got = mbar_wait<true>(&sfull[slot], sphase, P.err, abort_flag);
        if (warp_wide) got = __all_sync(0xffffffffu, got);
        if (got) tile = ring[slot];
        if (warp_wide) __syncwarp();
        if (got && (!warp_wide || lane == 0)) release_slot(slot);
        if (++slot == PRING) {
            slot = 0;
            sphase ^= 1u;
        }
        return got ? tile : P.n_tiles;
    };

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------- producer (both CTAs; rank 0 claims)
            int stage = 0;
            uint32_t phase = 0;
            int issued_phase[PSTAGES];
            for (int s = 0; s < PSTAGES; ++s) issued_phase[s] = -1;
            bool ok = true;
            while (ok) {
                int t;
                if (leader) {
                    if (!mbar_wait<true>(&sempty[slot], sphase ^ 1u, P.err, abort_flag)) break;
                    t = (*abort_flag || iters == 0) ? P.n_tiles : atomicAdd(P.ctr, 1);
                    if (t > P.n_tiles) t = P.n_tiles;
                    ring[slot] = t;
                    st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(ring + slot)), 1),
                                          static_cast<uint32_t>(t));
                    mbar_arrive(&sfull[slot]);
                    mbar_arrive_cluster(mapa_shared(smem_u32(&sfull[slot]), 1));
                    if (++slot == PRING) {
                        slot = 0;
                        sphase ^= 1u;
                    }
                } else {
                    t = next_tile(false);
                }
                if (t >= P.n_tiles) break;
                int job, bi, bj;
                decode(P.tiles[t], job, bi, bj);
                const CUtensorMap *ma, *mb;
                product_maps(M, job, P.nprod - 1, ma, mb);
                for (int it = 0, seg = 0, kb = 0; it < iters; ++it) {  // it = seg * nk + kb
                    if (!mbar_wait(&empty[stage], phase ^ 1u, P.err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full_leader = mapa_shared(smem_u32(&full[stage]), 0);
                    if (leader) mbar_arrive_expect_tx(&full[stage], 2 * PSTAGE_BYTES);
                    tma_load_2d_pair(sA + stage * PA_BYTES, ma, full_leader, kb * BK, bi * PM + 128 * rank);
                    tma_load_2d_pair(sB + stage * PA_BYTES, mb, full_leader, kb * BK, bj * PM + 128 * rank);
                    if (++kb == nk && ++seg < P.nprod) {
                        kb = 0;
                        product_maps(M, job, P.nprod - 1 - seg, ma, mb);
                    }
                    issued_phase[stage] = static_cast<int>(phase);
                    if (++stage == PSTAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // the leader's full barriers count both CTAs' bytes: drain there
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
            bool ok = true;
            while (ok) {
                const int t = next_tile(false);
                if (t >= P.n_tiles) break;
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, P.err, abort_flag)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int it = 0; it < iters; ++it) {
                    if (!mbar_wait(&full[stage], phase, P.err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + stage * PA_BYTES);
                    const uint32_t b0 = smem_u32(sB + stage * PA_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        umma_bf16_pair(d_tmem, sdesc_k_sw128(a0 + k * 32), sdesc_k_sw128(b0 + k * 32), idesc,
                                       (it | k) != 0);
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
        // ---------------------------------------------------------- epilogue (both CTAs)
        const int ew = warp - 2;
        const int sub = warp & 3;          // TMEM lane quarter
        const int colhalf = ew >> 2;       // columns [0,128) or [128,256)
        const int row = sub * 32 + lane;
        const float ff = P.coef[0], gg = P.coef[1];
        int acc = 0;
        uint32_t acc_phase = 0;
        for (;;) {
            const int t = next_tile(true);
            if (t >= P.n_tiles) break;
            int job, bi, bj;
            decode(P.tiles[t], job, bi, bj);
            const int64_t i = static_cast<int64_t>(bi) * PM + 128 * static_cast<int>(rank) + row;
            const float fda = ff * __ldg(P.job[job].da + i);
            const float gza = gg * __ldg(P.job[job].za + i);
            if (!mbar_wait(&tfull[acc], acc_phase, P.err, abort_flag)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(sub * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN + colhalf * 128);
            merge_row(P, job, i, static_cast<int64_t>(bj) * BN + colhalf * 128, tbase, true, fda, gza);
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
    // CTA pairs (256 x 256 tiles) when every job's sizes allow it, unless KVB_STATS_PAIR=0
    const char* env = std::getenv("KVB_STATS_PAIR");
    bool pair = !(env && std::strcmp(env, "0") == 0);
    for (int j = 0; j < n_jobs; ++j)
        if (jobs[j].Ma % PM || jobs[j].Nb % PM) pair = false;
    const int tm = pair ? PM : BM, tn = pair ? PM : BN, group = pair ? PGROUP : GROUP;
    std::vector<uint32_t> tiles;
    for (int j = 0; j < n_jobs; ++j) {
        const int64_t nI = jobs[j].Ma / tm, nJ = jobs[j].Nb / tn;
        for (int64_t g0 = 0; g0 < nI; g0 += group) {
            const int64_t g1 = g0 + group < nI ? g0 + group : nI;
            for (int64_t bj = 0; bj < nJ; ++bj)
                for (int64_t bi = g0; bi < g1; ++bi) {
                    if (jobs[j].lower && bj * tn > bi * tm + tm - 1) continue;
                    tiles.push_back((static_cast<uint32_t>(j) << 30) | (static_cast<uint32_t>(bi) << 15) |
                                    static_cast<uint32_t>(bj));
                }
        }
    }
    StatsGemmPlan* p = new StatsGemmPlan();
    p->n_tiles = static_cast<int>(tiles.size());
    p->pair = pair;
    cudaError_t e = cudaMalloc(&p->tiles, tiles.size() * sizeof(uint32_t) + 16);
    p->ctr = reinterpret_cast<int*>(p->tiles + tiles.size());
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
    P.ctr = plan->ctr;
    const bool pair = plan->pair && num_sms >= 2;
    P.nb = nb;
    P.coef = coef;
    P.err = err;
    P.nprod = jobs[0].A_3 ? 6 : 3;
    for (int j = 0; j < n_jobs; ++j) {
        const StatsJob& J = jobs[j];
        if (J.A_3 && (!encode_2d(&M.a[2][j], J.A_3, ld, J.Ma, BM, why) ||
                      !encode_2d(&M.b[2][j], J.B_3, ld, J.Nb, pair ? 128 : BN, why)))
            return cudaErrorInvalidValue;
        if (!encode_2d(&M.a[0][j], J.A, ld, J.Ma, BM, why) || !encode_2d(&M.a[1][j], J.A_lo, ld, J.Ma, BM, why) ||
            !encode_2d(&M.b[0][j], J.B, ld, J.Nb, pair ? 128 : BN, why) ||
            !encode_2d(&M.b[1][j], J.B_lo, ld, J.Nb, pair ? 128 : BN, why))
            return cudaErrorInvalidValue;
        P.job[j] = JobP{J.out, J.da, J.db, J.za, J.zb, J.ldo, J.Ma, J.Nb};
    }
    if (pair) {
        cudaError_t e = cudaMemsetAsync(plan->ctr, 0, sizeof(int), s);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(stats_gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PSMEM_BYTES);
        if (e != cudaSuccess) return e;
        const int pairs = plan->n_tiles < num_sms / 2 ? plan->n_tiles : num_sms / 2;
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
        e = cudaLaunchKernelEx(&cfg, stats_gemm_pair_kernel, M, P);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    cudaError_t e = cudaFuncSetAttribute(stats_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int grid = plan->n_tiles < num_sms ? plan->n_tiles : num_sms;
    stats_gemm_kernel<<<grid, NUM_THREADS, SMEM_BYTES, s>>>(M, P);
    return cudaGetLastError();
}

}  // namespace kvb
